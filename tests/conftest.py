import os
import subprocess
import sys
import warnings

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size oracle comparisons (tens of seconds)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        _report_other_gpu_processes(config, items)
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def _report_other_gpu_processes(config, items):
    """The fused decode kernel keeps one CTA on every SM and its CTAs wait on
    each other (bounded): kernels of another process on the same GPU make its
    tests end in DS4G_ETIMEOUT.  Say so up front instead of after a timeout."""
    if not any("gpu" in it.keywords for it in items):
        return
    try:
        q = subprocess.run(["nvidia-smi", "-i", "0", "--query-compute-apps=pid", "--format=csv,noheader"],
                           capture_output=True, text=True, timeout=30)
    except (OSError, subprocess.SubprocessError):
        return
    others = sorted({int(v) for v in q.stdout.split() if v.isdigit() and int(v) != os.getpid()})
    if others:
        warnings.warn(f"other compute processes on GPU 0: {others}; the fused decode tests need the whole GPU")
