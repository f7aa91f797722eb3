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


def test_decode_stack_equals_layer_calls_and_oracle():
    """Three chained layers through ds4g_moe_decode_stack (programmatic
    dependent launches) equal three ds4g_moe_layer_decode calls bit for bit,
    and follow the oracle's chain (rmsnorm between layers, no residual)."""
    NL, seed = 3, 5
    x = synth.hidden(seed, 1, 1, layer=11, normalise=False)
    h = oracle.rmsnorm(x)
    refs, layers = [], []
    for l in range(NL):
        R, b = synth.router(seed, 1, l), synth.bias_normal(seed, 1, l)
        ids_r, w_r, keys, margin = oracle.route(h, R, b)
        assert margin[0] > 1e-4     # the seed keeps every layer clear of near-ties
        L, hx, shared, grid = device_layer(seed, 1, l, ids_r.reshape(-1))
        out_r = oracle_forward(h, ids_r, w_r, hx, shared, grid)
        refs.append((ids_r, w_r, keys, margin, out_r))
        layers.append((L, _t(R), _t(b)))
        h = oracle.rmsnorm(out_r)
    stack = B.DecodeStack([(L.struct, R, b) for L, R, b in layers])
    ids = torch.full((NL, K), -1, dtype=torch.int32, device=DEV)
    w = torch.zeros(NL, K, dtype=torch.float32, device=DEV)
    hbuf = torch.zeros(2, H, dtype=torch.float32, device=DEV)
    out = torch.full((H,), float("nan"), dtype=torch.float32, device=DEV)
    ws = B.workspace(B.ds4g_layer_decode_workspace())
    xd = _t(x[0])
    for _ in range(2):                               # the workspace is reusable call after call
        B.ds4g_moe_decode_stack(xd, stack, ids, w, hbuf, out, ws)
        assert B.ds4g_last_error(ws) == 0
    ids_s, w_s, out_s = ids.cpu().numpy(), w.cpu().numpy(), out.cpu().numpy()
    for l in range(NL):
        ids_r, w_r, keys, margin, _ = refs[l]
        check_route(ids_s[l][None], w_s[l][None], ids_r, w_r, keys, margin)
    assert_close_fwd(out_s[None], refs[-1][4])
    # the same layers one call at a time
    xl = xd
    for l, (L, R, b) in enumerate(layers):
        i1 = torch.full((K,), -1, dtype=torch.int32, device=DEV)
        w1 = torch.zeros(K, dtype=torch.float32, device=DEV)
        o1 = torch.empty(H, dtype=torch.float32, device=DEV)
        B.ds4g_moe_layer_decode(xl, R, b, L.struct, i1, w1, o1, ws)
        assert np.array_equal(i1.cpu().numpy(), ids_s[l]) and np.array_equal(w1.cpu().numpy(), w_s[l])
        xl = o1
    assert np.array_equal(xl.cpu().numpy(), out_s)
    assert B.ds4g_last_error(ws) == 0


def test_decode_stack_rejects_bad_arguments():
    L, _, _, _ = device_layer(0, 1, 0, range(6))
    R, b = _t(synth.router(0, 1)), _t(synth.bias_normal(0, 1))
    stack = B.DecodeStack([(L.struct, R, b)])
    x = torch.zeros(H, device=DEV)
    ids = torch.zeros(1, K, dtype=torch.int32, device=DEV)
    w = torch.zeros(1, K, device=DEV)
    hbuf = torch.zeros(2, H, device=DEV)
    out = torch.zeros(H, device=DEV)
    small = B.workspace(1024)
    with pytest.raises(B.DS4GError) as e:
        B.ds4g_moe_decode_stack(x, stack, ids, w, hbuf, out, small)
    assert e.value.code == 3
    ws = B.workspace(B.ds4g_layer_decode_workspace())
    with pytest.raises(B.DS4GError) as e:
        B.ds4g_moe_decode_stack(x, stack, ids, w, hbuf[0, 1:], out, ws)   # misaligned scratch
    assert e.value.code == 2
    stack.n = 0
    with pytest.raises(B.DS4GError) as e:
        B.ds4g_moe_decode_stack(x, stack, ids, w, hbuf, out, ws)
    assert e.value.code == 1


def test_decode_stack_q2_q4_layers():
    """A stack of IQ2_XXS/Q2_K and Q4_K layers (the q2-q4 model keeps its
    last layers at Q4_K), every layer on the fused kernel (Q4_K tile-blocks
    in its routed pieces).  Equal bit for bit to single-layer calls made one
    at a time, and following the oracle's chain (chained Q4_K layers drive h
    far beyond the fp16 range)."""
    seed, cfg = 5, 4
    kinds = [(synth.IQ2_XXS, synth.Q2_K), (synth.Q4_K, synth.Q4_K), (synth.Q4_K, synth.Q4_K),
             (synth.IQ2_XXS, synth.Q2_K)]
    NL = len(kinds)
    x = synth.hidden(seed, cfg, 1, layer=11, normalise=False)
    h = oracle.rmsnorm(x)
    refs, layers = [], []
    for l, (gut, dt) in enumerate(kinds):
        R, b = synth.router(seed, cfg, l), synth.bias_normal(seed, cfg, l)
        ids_r, w_r, keys, margin = oracle.route(h, R, b)
        assert margin[0] > 1e-3
        L, hx, shared, grid = device_layer(seed, cfg, l, ids_r.reshape(-1), gut, dt)
        out_r = oracle_forward(h, ids_r, w_r, hx, shared, grid, gut, dt)
        refs.append((ids_r, w_r, keys, margin, out_r))
        layers.append((L, _t(R), _t(b)))
        h = oracle.rmsnorm(out_r)
    stack = B.DecodeStack([(L.struct, R, b) for L, R, b in layers])
    ids = torch.full((NL, K), -1, dtype=torch.int32, device=DEV)
    w = torch.zeros(NL, K, dtype=torch.float32, device=DEV)
    hbuf = torch.zeros(2, H, dtype=torch.float32, device=DEV)
    out = torch.full((H,), float("nan"), dtype=torch.float32, device=DEV)
    xd = _t(x[0])
    assert B.ds4g_decode_stack_workspace() == B.ds4g_layer_decode_workspace()
    ws = B.workspace(B.ds4g_decode_stack_workspace())
    for _ in range(2):                               # the workspace is reusable call after call
        B.ds4g_moe_decode_stack(xd, stack, ids, w, hbuf, out, ws)
        assert B.ds4g_last_error(ws) == 0
    ids_s, w_s, out_s = ids.cpu().numpy(), w.cpu().numpy(), out.cpu().numpy()
    for l in range(NL):
        ids_r, w_r, keys, margin, _ = refs[l]
        check_route(ids_s[l][None], w_s[l][None], ids_r, w_r, keys, margin)
    assert_close_fwd(out_s[None], refs[-1][4])
    # the same layers one call at a time
    wsl = B.workspace(B.ds4g_layer_decode_workspace())
    xl = xd[None]
    for l, (L, R, b) in enumerate(layers):
        i1 = torch.full((1, K), -1, dtype=torch.int32, device=DEV)
        w1 = torch.zeros(1, K, dtype=torch.float32, device=DEV)
        o1 = torch.empty(1, H, dtype=torch.float32, device=DEV)
        B.ds4g_moe_layer_decode(xl[0], R, b, L.struct, i1[0], w1[0], o1[0], wsl)
        assert np.array_equal(i1.cpu().numpy()[0], ids_s[l]) and np.array_equal(w1.cpu().numpy()[0], w_s[l])
        xl = o1
    assert np.array_equal(xl.cpu().numpy()[0], out_s)
    assert B.ds4g_last_error(wsl) == 0


@pytest.mark.parametrize("seed,zipf", [(8, False), (9, True)])
def test_layer_decode_q4k_matches_oracle(seed, zipf):
    """One Q4_K layer (gate/up/down) on the fused kernel: routed gate/up
    pieces of 8 Q4_K tile-blocks, routed down in halves of h (16 output
    parts per tile), against the oracle; repeatable on one workspace."""
    xraw = synth.hidden(seed, 4, 1, layer=3, normalise=False)
    R = synth.router(seed, 4)
    b = synth.bias_zipf(seed, 4) if zipf else synth.bias_normal(seed, 4)
    xn = oracle.rmsnorm(xraw)
    ids_r, w_r, keys, margin = oracle.route(xn, R, b)
    L, hx, shared, grid = device_layer(seed, 4, 0, ids_r.reshape(-1), synth.Q4_K, synth.Q4_K)
    ws = B.workspace(B.ds4g_layer_decode_workspace())
    ids, w, out, st = _run(xraw[0], R, b, L, ws)
    assert st == 0
    check_route(ids[None], w[None], ids_r, w_r, keys, margin)
    assert_close_fwd(out[None], oracle_forward(xn, ids[None], w[None], hx, shared, grid, synth.Q4_K, synth.Q4_K))
    again = _run(xraw[0], R, b, L, ws)
    assert again[3] == 0 and np.array_equal(again[2], out)


def test_layer_decode_h_beyond_fp16_range():
    """An input for which h = silu(g) * u reaches ~3e6 (far beyond fp16):
    the fused kernel carries h with a power-of-two scale per 16 entries, so
    no flag and oracle parity."""
    rng = np.random.default_rng(11)
    x = (60.0 * rng.standard_normal((1, H))).astype(np.float32)
    R, b = synth.router(6, 4), synth.bias_normal(6, 4)
    ids_r, w_r, keys, margin = oracle.route(x, R, b)
    assert margin[0] > 1e-3
    L, hx, shared, grid = device_layer(6, 4, 5, ids_r.reshape(-1))
    ws = B.workspace(B.ds4g_layer_decode_workspace())
    ids, w, out, st = _run(x[0], R, b, L, ws, normalize=False)
    assert st == 0
    check_route(ids[None], w[None], ids_r, w_r, keys, margin)
    assert_close_fwd(out[None], oracle_forward(x, ids[None], w[None], hx, shared, grid))


def test_layer_decode_bounded_wait_times_out_and_recovers():
    """The control warps' wait for the router logits is bounded: under the test
    hook they wait for a router row that does not exist, give up after ~130 us, abort
    the launch (every CTA drains its copies) and record DS4G_ETIMEOUT; the
    same workspace then gives the normal result, bit for bit equal to a
    fresh workspace's."""
    x = synth.hidden(9, 1, 1)
    R, b = synth.router(9, 1), synth.bias_normal(9, 1)
    ids_r, w_r, keys, margin = oracle.route(x, R, b)
    L, hx, shared, grid = device_layer(9, 1, 0, ids_r.reshape(-1))
    ws = B.workspace(B.ds4g_layer_decode_workspace())
    B.ds4g_test_force_timeout(True)
    try:
        _, _, _, st = _run(x[0], R, b, L, ws, normalize=False)
    finally:
        B.ds4g_test_force_timeout(False)
    assert st == 6                                    # DS4G_ETIMEOUT
    ids, w, out, st = _run(x[0], R, b, L, ws, normalize=False)
    assert st == 0
    fresh = _run(x[0], R, b, L, B.workspace(B.ds4g_layer_decode_workspace()), normalize=False)
    assert fresh[3] == 0 and np.array_equal(out, fresh[2]) and np.array_equal(ids, fresh[0])
    check_route(ids[None], w[None], ids_r, w_r, keys, margin)
    assert_close_fwd(out[None], oracle_forward(x, ids[None], w[None], hx, shared, grid))
