"""The product path and the oracle are independent: the package neither
imports nor names the oracle (so no call can fall back to it), the oracle's C
source shares no file with the CUDA sources, and the package raises instead
of computing when its library is missing."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "bit_quantized_moe_bias_b300")


def _files(top, exts):
    for d, _, fs in os.walk(top):
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(d, f)


def test_package_source_never_names_the_oracle():
    for f in list(_files(PKG, (".py", ".cu", ".cuh", ".h", ".c"))) + [os.path.join(ROOT, "include", "ds4g.h")]:
        text = open(f, encoding="utf-8").read().lower()
        assert "oracle" not in text, f


def test_importing_the_package_loads_no_oracle():
    code = ("import sys; sys.path.insert(0, %r); import bit_quantized_moe_bias_b300 as B; B.lib(); "
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))" % ROOT)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "False"


def test_oracle_includes_nothing_from_the_cuda_sources():
    # the oracle's C files include system headers and their own header only
    odir = os.path.join(ROOT, "oracle")
    for f in _files(odir, (".c", ".h")):
        for ln in open(f, encoding="utf-8").read().splitlines():
            if ln.strip().startswith("#include") and '"' in ln:
                name = ln.split('"')[1]
                assert "/" not in name and os.path.exists(os.path.join(odir, name)), (f, ln)


def test_missing_library_raises(monkeypatch):
    import bit_quantized_moe_bias_b300 as B
    monkeypatch.setattr(B, "_SO", os.path.join(ROOT, "no_such_libds4g.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError):
        B.lib()
