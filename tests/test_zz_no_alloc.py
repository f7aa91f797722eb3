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
from helpers import H, assert_close_fwd, device_layer, oracle_forward

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
@pytest.mark.parametrize("T", [1, 5, 64])
def test_noalloc_matches_workspace_forward_twice(T):
    """Two calls in a row: each equals, bit for bit, the workspace forward
    run on the same chunks of up to three tokens (the kernels the call
    uses), and both are within the block's tolerance of the oracle (at
    T = 64 the workspace forward of the whole batch takes the tensor-core
    prefill path, so the oracle is the reference there)."""
    torch = pytest.importorskip("torch")
    dev = "cuda"
    x = synth.hidden(6, 0, T)
    ids, w, _, _ = oracle.route(x, synth.router(6, 0), synth.bias_normal(6, 0))
    layer, hx, shared, grid = device_layer(6, 0, 0, ids.reshape(-1))
    xd, idd, wd = (torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in (x, ids, w))
    ref = torch.empty(T, H, dtype=torch.float32, device=dev)
    ws = B.workspace(B.ds4g_forward_workspace(3))
    for t0 in range(0, T, 3):
        t1 = min(T, t0 + 3)
        # fresh (16-byte aligned) copies of the chunk's rows, as the C ABI requires
        oc = torch.empty(t1 - t0, H, dtype=torch.float32, device=dev)
        B.ds4g_moe_forward(xd[t0:t1].clone(), layer.struct, idd[t0:t1].clone(), wd[t0:t1].clone(), oc, ws)
        ref[t0:t1] = oc
    assert B.ds4g_last_error(ws) == 0
    r = ref.cpu().numpy()
    ro = oracle_forward(x, ids, w, hx, shared, grid)
    for _ in range(2):                               # the second call reuses the array
        out = torch.full((T, H), float("nan"), dtype=torch.float32, device=dev)
        B.ds4g_moe_forward_noalloc(xd, layer.struct, idd, wd, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.array_equal(got, r)
        assert_close_fwd(got, ro)
