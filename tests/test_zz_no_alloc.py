"""ds4g_moe_forward_noalloc: the variant of the MoE forward for callers that
cannot allocate device memory (allocator callbacks, real-time loops that must
not stall on the allocator, plugins given fixed buffers).  Its scratch is a
static device array inside the library, shared by every call.

This file is named so that pytest collects it last: the test must pass both
in a fresh process and after every other test has used the library."""
import ctypes as C

import numpy as np
import pytest

import oracle
import synth
from helpers import FWD_TOL, H, device_layer

import bit_quantized_moe_bias_b300 as B


def test_noalloc_rejects_bad_sizes_before_any_cuda_call():
    L = B.lib()
    fake = 0x10000000            # aligned fake device address, never dereferenced
    lay = B.ds4g_layer(0, 1, fake, fake, fake, fake, fake, fake, fake)
    f = L.ds4g_moe_forward_noalloc
    assert f(fake, 0, C.byref(lay), fake, fake, fake, None) == 1                    # T < 1
    assert f(fake, 65, C.byref(lay), fake, fake, fake, None) == 3                   # T > max
    assert f(None, 1, C.byref(lay), fake, fake, fake, None) == 1                    # NULL
    assert f(fake + 4, 1, C.byref(lay), fake, fake, fake, None) == 2                # misaligned
    bad = B.ds4g_layer(0, 2, fake, fake, fake, fake, fake, fake, fake)
    assert f(fake, 1, C.byref(bad), fake, fake, fake, None) == 5                    # IQ2 + Q4_K


@pytest.mark.gpu
@pytest.mark.parametrize("T", [1, 5])
def test_noalloc_matches_workspace_forward_twice(T):
    torch = pytest.importorskip("torch")
    dev = "cuda"
    x = synth.hidden(6, 0, T)
    ids, w, _, _ = oracle.route(x, synth.router(6, 0), synth.bias_normal(6, 0))
    layer, _, _, _ = device_layer(6, 0, 0, ids.reshape(-1))
    xd, idd, wd = (torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in (x, ids, w))
    ref = torch.empty(T, H, dtype=torch.float32, device=dev)
    ws = B.workspace(B.ds4g_forward_workspace(T))
    B.ds4g_moe_forward(xd, layer.struct, idd, wd, ref, ws)
    assert B.ds4g_last_error(ws) == 0
    r = ref.cpu().numpy().astype(np.float64)
    scale = float(np.max(np.abs(r)))
    for _ in range(2):                               # the second call reuses the array
        out = torch.full((T, H), float("nan"), dtype=torch.float32, device=dev)
        B.ds4g_moe_forward_noalloc(xd, layer.struct, idd, wd, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - r))) <= FWD_TOL * scale
