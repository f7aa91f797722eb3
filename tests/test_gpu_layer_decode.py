"""GPU parity of the fused single-token layer (rmsnorm + router + top-6 +
routed and shared experts in one launch) against the CPU oracle, through the
C ABI: expert ids exact (up to certified near-ties), weights within 1e-6,
output within max-abs 2e-3 * max|ref| (fp32 accumulation)."""
import numpy as np
import pytest

import oracle
import synth
from helpers import H, K, assert_close_fwd, check_route, device_layer, oracle_forward

torch = pytest.importorskip("torch")
import bit_quantized_moe_bias_b300 as B  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _run(x, R, b, L, ws, normalize=True):
    ids = torch.full((K,), -1, dtype=torch.int32, device=DEV)
    w = torch.zeros(K, dtype=torch.float32, device=DEV)
    out = torch.full((H,), float("nan"), dtype=torch.float32, device=DEV)
    B.ds4g_moe_layer_decode(_t(x), _t(R), _t(b), L.struct, ids, w, out, ws, normalize=normalize)
    st = B.ds4g_last_error(ws)
    return ids.cpu().numpy(), w.cpu().numpy(), out.cpu().numpy(), st


@pytest.mark.parametrize("seed,zipf", [(0, False), (1, False), (2, True)])
def test_layer_decode_matches_oracle(seed, zipf):
    xraw = synth.hidden(seed, 1, 1, layer=7, normalise=False)
    R = synth.router(seed, 1)
    b = synth.bias_zipf(seed, 1) if zipf else synth.bias_normal(seed, 1)
    xn = oracle.rmsnorm(xraw)
    ids_r, w_r, keys, margin = oracle.route(xn, R, b)
    L, hx, shared, grid = device_layer(seed, 1, 0, ids_r.reshape(-1))
    ws = B.workspace(B.ds4g_layer_decode_workspace())
    ids, w, out, st = _run(xraw[0], R, b, L, ws)
    assert st == 0
    check_route(ids[None], w[None], ids_r, w_r, keys, margin)
    assert_close_fwd(out[None], oracle_forward(xn, ids[None], w[None], hx, shared, grid))


def test_layer_decode_repeatable_and_unnormalised():
    """Counters reset at the end of every launch: repeated calls on one
    workspace give identical results; normalize=0 uses hidden as given."""
    x = synth.hidden(3, 1, 1)                 # already unit RMS
    R, b = synth.router(3, 1), synth.bias_normal(3, 1)
    ids_r, w_r, keys, margin = oracle.route(x, R, b)
    L, hx, shared, grid = device_layer(3, 1, 0, ids_r.reshape(-1))
    ws = B.workspace(B.ds4g_layer_decode_workspace())
    first = _run(x[0], R, b, L, ws, normalize=False)
    assert first[3] == 0
    for _ in range(3):
        again = _run(x[0], R, b, L, ws, normalize=False)
        assert again[3] == 0
        assert np.array_equal(again[0], first[0]) and np.array_equal(again[2], first[2])
    check_route(first[0][None], first[1][None], ids_r, w_r, keys, margin)
    assert_close_fwd(first[2][None], oracle_forward(x, first[0][None], first[1][None], hx, shared, grid))


def test_layer_decode_flags_missing_expert():
    x = synth.hidden(4, 1, 1)
    R, b = synth.router(4, 1), synth.bias_normal(4, 1)
    ids_r, _, _, _ = oracle.route(x, R, b)
    present = [int(e) for e in ids_r[0][:5]]               # the 6th selected expert is not loaded
    L, _, _, _ = device_layer(4, 1, 0, present)
    ws = B.workspace(B.ds4g_layer_decode_workspace())
    ids, _, out, st = _run(x[0], R, b, L, ws, normalize=False)
    assert st == 7
    assert np.all(np.isfinite(out))
    # the workspace is usable again afterwards
    L2, hx, shared, grid = device_layer(4, 1, 0, ids_r.reshape(-1))
    ids, w, out, st = _run(x[0], R, b, L2, ws, normalize=False)
    assert st == 0
    assert_close_fwd(out[None], oracle_forward(x, ids[None], w[None], hx, shared, grid))
