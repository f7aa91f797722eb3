"""GPU parity: every kernel, called through the C ABI, against the CPU oracle
on the same seeded inputs.  Bit-exact for dequantisation, bucketing and
packing; routing ids exact except within 1e-5 of a flip (then checked to be a
valid top-6), weights within 1e-6; block outputs within max-abs
2e-3 * max|ref| (fp32 accumulation)."""
import numpy as np
import pytest

import oracle
import synth
from helpers import (E, H, K, FullLayer, assert_close_fwd, check_route, device_layer, grid_u64,
                     oracle_forward)

torch = pytest.importorskip("torch")
import bit_quantized_moe_bias_b300 as B  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def grid():
    g, g64 = grid_u64(0)
    return g, torch.from_numpy(g64.view(np.int64)).to(DEV)


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


# --------------------------------------------------------------- dequant/pack
@pytest.mark.parametrize("qt,rows,cols", [(0, 64, 512), (1, 64, 512), (2, 64, 512),
                                          (0, 2048, 4096), (1, 4096, 2048), (2, 2048, 4096)])
def test_dequant_bit_exact(qt, rows, cols, grid):
    g = synth.gguf_matrix(qt, rows, cols, 7, 100 + qt + rows)
    p = _t(B.ds4g_quantize_pack(qt, rows, cols, g))
    of = torch.empty(rows, cols, dtype=torch.float32, device=DEV)
    ob = torch.empty(rows, cols, dtype=torch.int16, device=DEV)
    B.ds4g_dequantize(qt, p, rows, cols, grid[1], of, ob)
    torch.cuda.synchronize()
    rf, rb = oracle.dequantize(qt, g, rows, cols, grid[0], bf16=True)
    assert np.array_equal(of.cpu().numpy().view(np.uint32), rf.view(np.uint32))
    assert np.array_equal(ob.cpu().numpy().view(np.uint16), rb)


@pytest.mark.parametrize("qt", [0, 1, 2])
def test_pack_device_equals_host(qt):
    rows, cols = 256, 1024
    g = synth.gguf_matrix(qt, rows, cols, 2, 55)
    n = B.ds4g_packed_size(qt, rows, cols)
    out = torch.empty(n, dtype=torch.uint8, device=DEV)
    B.ds4g_quantize_pack_device(qt, rows, cols, _t(g), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), B.ds4g_quantize_pack(qt, rows, cols, g))


@pytest.mark.parametrize("qt", [0, 1, 2])
def test_synth_device_twin_matches_host(qt):
    rows, cols = 2048, 4096
    n = rows * cols // 256 * synth.BLOCK_BYTES[qt]
    out = torch.empty(n, dtype=torch.uint8, device=DEV)
    synth.gguf_matrix_device(qt, rows, cols, 5, 1234, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    got, ref = out.cpu().numpy(), synth.gguf_matrix(qt, rows, cols, 5, 1234)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:8]}: {got[bad[:8]]} vs {ref[bad[:8]]}"


# -------------------------------------------------------------------- router
def _route_gpu(x, R, b):
    T = x.shape[0]
    ids = torch.empty(T, K, dtype=torch.int32, device=DEV)
    w = torch.empty(T, K, dtype=torch.float32, device=DEV)
    ws = B.workspace(B.ds4g_route_workspace(T))
    B.ds4g_moe_route(_t(x), _t(R), _t(b), ids, w, ws)
    assert B.ds4g_last_error(ws) == 0
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T,zipf", [(1, False), (2, False), (8, False), (9, False), (33, True), (64, True),
                                    (65, False), (300, False), (2048, False)])
def test_route_parity(T, zipf):
    x = synth.hidden(0, 3, T)
    R = synth.router(0, 3)
    b = synth.bias_zipf(0, 3) if zipf else synth.bias_normal(0, 3)
    ids_g, w_g = _route_gpu(x, R, b)
    ids_r, w_r, keys, margin = oracle.route(x, R, b)
    near = check_route(ids_g, w_g, ids_r, w_r, keys, margin)
    assert near <= max(2, T // 100)


def test_route_repeatable_and_ties():
    """Identical router rows give identical keys: the lower id comes first,
    on every call (the workspace counters reset themselves)."""
    x = synth.hidden(1, 3, 4)
    R = synth.router(1, 3)
    R[17] = 0.05
    R[200] = 0.05
    b = np.zeros(E, np.float32)
    b[17] = b[200] = 2.0
    for _ in range(3):
        ids, w = _route_gpu(x, R, b)
        assert np.all(ids[:, 0] == 17) and np.all(ids[:, 1] == 200)
        assert np.all(w[:, 0] == w[:, 1])


# -------------------------------------------------------------------- bucket
@pytest.mark.parametrize("T,mode", [(1, "rand"), (7, "rand"), (33, "one"), (2048, "rand"),
                                    (4096, "zipf"), (1000, "empty")])
def test_bucket_bit_exact(T, mode):
    rng = np.random.default_rng(T)
    if mode == "one":
        ids = np.full((T, K), 200, np.int32)
    elif mode == "zipf":
        ids = np.minimum(rng.zipf(1.3, (T, K)) - 1, 255).astype(np.int32)
    elif mode == "empty":   # only 3 experts used: 253 empty buckets
        ids = rng.choice([0, 128, 255], (T, K)).astype(np.int32)
    else:
        ids = rng.integers(0, E, (T, K)).astype(np.int32)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * K, dtype=torch.int32, device=DEV)
    inv = torch.empty(T * K, dtype=torch.int32, device=DEV)
    ws = B.workspace(B.ds4g_bucket_workspace(T))
    B.ds4g_moe_bucket(_t(ids), counts, offsets, perm, inv, ws)
    assert B.ds4g_last_error(ws) == 0
    rc, ro, rp, ri = oracle.bucket(ids)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)
    assert np.array_equal(inv.cpu().numpy(), ri)


def test_bucket_flags_bad_id():
    ids = np.zeros((3, K), np.int32)
    ids[1, 2] = 300
    ws = B.workspace(B.ds4g_bucket_workspace(3))
    bufs = [torch.empty(n, dtype=torch.int32, device=DEV) for n in (E, E + 1, 18, 18)]
    B.ds4g_moe_bucket(_t(ids), *bufs, ws)
    assert B.ds4g_last_error(ws) == 7
    assert B.ds4g_last_error(ws) == 0   # cleared after reading


def test_rmsnorm_parity():
    x = synth.normal(0, 77, (37, H), 3.0)
    y = torch.empty(37, H, device=DEV)
    B.ds4g_rmsnorm(_t(x), y)
    ref = oracle.rmsnorm(x)
    assert np.max(np.abs(y.cpu().numpy() - ref)) <= 1e-5 * np.max(np.abs(ref))


# ------------------------------------------------------------------- forward
def _forward_gpu(x, ids, w, L, phased=False):
    T = x.shape[0]
    out = torch.empty(T, H, dtype=torch.float32, device=DEV)
    ws = B.workspace(B.ds4g_forward_workspace(T))
    if phased:
        B.ds4g_moe_gate_up(_t(x), L.struct, _t(ids), _t(w), out, ws)
        B.ds4g_moe_down(_t(x), L.struct, _t(ids), _t(w), out, ws)
    else:
        B.ds4g_moe_forward(_t(x), L.struct, _t(ids), _t(w), out, ws)
    st = B.ds4g_last_error(ws)
    return out.cpu().numpy(), st


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 32, 33, 63])
def test_forward_decode_q2(T):
    """T <= 3: the per-slot decode kernels; 4 <= T < 64: the batched path
    (slots grouped by expert, chunks of up to 32 tokens: 33 and 63 end in a
    ragged chunk)."""
    x = synth.hidden(0, 0, T)
    ids, w, _, _ = oracle.route(x, synth.router(0, 0), synth.bias_normal(0, 0))
    L, hx, shared, grid = device_layer(0, 0, 0, ids.reshape(-1))
    got, st = _forward_gpu(x, ids, w, L)
    assert st == 0
    assert_close_fwd(got, oracle_forward(x, ids, w, hx, shared, grid))


def test_forward_phases_equal_forward_and_deterministic():
    x = synth.hidden(0, 0, 1)
    ids, w, _, _ = oracle.route(x, synth.router(0, 0), synth.bias_normal(0, 0))
    L, hx, shared, grid = device_layer(0, 0, 0, ids.reshape(-1))
    a, _ = _forward_gpu(x, ids, w, L)
    b, _ = _forward_gpu(x, ids, w, L)
    c, st = _forward_gpu(x, ids, w, L, phased=True)
    assert st == 0
    assert np.array_equal(a, b)   # fixed reduction order: deterministic
    assert np.array_equal(a, c)


def test_forward_duplicate_ids_and_shared_experts():
    """A repeated id within a token is summed twice; tokens may share experts."""
    x = synth.hidden(2, 0, 3)
    ids = np.array([[5, 5, 9, 9, 9, 12], [12, 5, 77, 1, 2, 3], [5, 5, 5, 5, 5, 5]], np.int32)
    w = np.array([[0.3, 0.2, 0.1, 0.1, 0.1, 0.2]] * 3, np.float32)
    L, hx, shared, grid = device_layer(2, 0, 0, ids.reshape(-1))
    got, st = _forward_gpu(x, ids, w, L)
    assert st == 0
    assert_close_fwd(got, oracle_forward(x, ids, w, hx, shared, grid))


def test_forward_batched_duplicates_flags_and_determinism():
    """The batched path (T = 8): a repeated id within a token is summed twice,
    tokens share experts, and the result is bit for bit repeatable; an expert
    whose matrices are missing, or an id out of range, is flagged and the
    other tokens are still correct."""
    T = 8
    x = synth.hidden(2, 0, T)
    ids = np.array([[5, 5, 9, 9, 9, 12], [12, 5, 77, 1, 2, 3], [5, 5, 5, 5, 5, 5], [1, 2, 3, 4, 5, 6],
                    [200, 5, 9, 77, 12, 1], [6, 6, 6, 5, 5, 5], [9, 12, 77, 200, 3, 2], [1, 1, 2, 2, 3, 3]],
                   np.int32)
    w = np.array([[0.3, 0.2, 0.1, 0.1, 0.1, 0.2]] * T, np.float32)
    L, hx, shared, grid = device_layer(2, 0, 0, ids.reshape(-1))
    a, st = _forward_gpu(x, ids, w, L)
    assert st == 0
    b, st = _forward_gpu(x, ids, w, L)
    assert st == 0 and np.array_equal(a, b)
    assert_close_fwd(a, oracle_forward(x, ids, w, hx, shared, grid))
    bad = ids.copy()
    bad[3, 4] = 999                                            # token 3: an id out of range
    got, st = _forward_gpu(x, bad, w, L)
    assert st == 7
    ok = [t for t in range(T) if t != 3]
    assert_close_fwd(got[ok], oracle_forward(x[ok], ids[ok], w[ok], hx, shared, grid))


def test_forward_batched_single_hot_expert():
    """The largest buckets of the batched path: every slot of every token
    selects expert 7 (T = 40: a 192-slot bucket in the first 32-token chunk,
    48 slots in the ragged second one), plus a token whose six slots are six
    different experts next to it."""
    T = 40
    x = synth.hidden(4, 0, T)
    ids = np.full((T, K), 7, np.int32)
    ids[17] = [7, 1, 2, 3, 4, 5]
    w = np.tile(np.array([0.25, 0.15, 0.2, 0.1, 0.2, 0.1], np.float32), (T, 1))
    L, hx, shared, grid = device_layer(4, 0, 0, ids.reshape(-1))
    got, st = _forward_gpu(x, ids, w, L)
    assert st == 0
    assert_close_fwd(got, oracle_forward(x, ids, w, hx, shared, grid))


def test_forward_flags_missing_expert():
    x = synth.hidden(3, 0, 1)
    ids = np.array([[1, 2, 3, 4, 5, 6]], np.int32)
    w = np.full((1, K), 1 / 6, np.float32)
    L, _, _, _ = device_layer(3, 0, 0, [1, 2, 3, 4, 5])        # expert 6 not loaded
    _, st = _forward_gpu(x, ids, w, L)
    assert st == 7
    ids[0, 5] = 999                                            # id out of range
    _, st = _forward_gpu(x, ids, w, L)
    assert st == 7


@pytest.mark.parametrize("T", [1, 2])
def test_forward_decode_q4k(T):
    x = synth.hidden(4, 4, T)
    ids, w, _, _ = oracle.route(x, synth.router(4, 4), synth.bias_zipf(4, 4))
    L, hx, shared, grid = device_layer(4, 4, 3, ids.reshape(-1), synth.Q4_K, synth.Q4_K)
    got, st = _forward_gpu(x, ids, w, L)
    assert st == 0
    assert_close_fwd(got, oracle_forward(x, ids, w, hx, shared, grid, synth.Q4_K, synth.Q4_K))


def test_forward_large_activation_flagged():
    """fp16 hi/lo activations need |x| < 65504; larger inputs are flagged."""
    x = synth.hidden(0, 0, 1) * np.float32(1e5)
    ids = np.array([[0, 1, 2, 3, 4, 5]], np.int32)
    w = np.full((1, K), 1 / 6, np.float32)
    L, _, _, _ = device_layer(0, 0, 0, range(6))
    _, st = _forward_gpu(x, ids, w, L)
    assert st == 7


@pytest.mark.parametrize("gut,dt", [(synth.IQ2_XXS, synth.Q2_K), (synth.Q4_K, synth.Q4_K)])
def test_forward_decode_h_beyond_fp16_range(gut, dt):
    """h = silu(g) * u far beyond the fp16 range (inputs with a large common
    mode, as a chain of layers produces) is carried by a power-of-two scale
    per 16 entries: no flag, oracle parity."""
    rng = np.random.default_rng(11)
    if gut == synth.Q4_K:   # Q4_K weights have a positive mean: a near-constant x adds up
        x = oracle.rmsnorm((1.0 + 0.1 * rng.standard_normal((2, H))).astype(np.float32))
    else:
        x = (60.0 * rng.standard_normal((2, H))).astype(np.float32)
    ids, w, _, _ = oracle.route(x, synth.router(6, 4), synth.bias_normal(6, 4))
    L, hx, shared, grid = device_layer(6, 4, 5, ids.reshape(-1), gut, dt)
    g, u, _ = hx[int(ids[0, 0])]
    G = oracle.dequantize(gut, g, 2048, H, grid).astype(np.float64)
    U = oracle.dequantize(gut, u, 2048, H, grid).astype(np.float64)
    gg, uu = G @ x[0].astype(np.float64), U @ x[0].astype(np.float64)
    assert np.abs(gg * 0.5 * (1.0 + np.tanh(0.5 * gg)) * uu).max() > 1e5   # the case this test is about
    got, st = _forward_gpu(x, ids, w, L)
    assert st == 0
    assert_close_fwd(got, oracle_forward(x, ids, w, hx, shared, grid, gut, dt))


def test_workspace_reused_across_T_and_paths():
    """One zeroed workspace serves forward calls of any T (decode chunks and
    the prefill path) and the fused layer kernel, in any order: each result
    equals the same call on a fresh workspace bit for bit (the counters sit
    at fixed offsets that no call uses as scratch)."""
    experts = [2, 9, 31, 64, 100, 150, 151, 199, 230, 255]
    rng = np.random.default_rng(8)
    Tmax = 64
    x = synth.hidden(5, 0, Tmax)
    ids = np.stack([rng.choice(experts, K, replace=False) for _ in range(Tmax)]).astype(np.int32)
    w = rng.dirichlet(np.ones(K), Tmax).astype(np.float32)
    L = FullLayer(5, 0, 0).L            # all 256 experts, generated on the device
    xd, idd, wd = _t(x), _t(ids), _t(w)
    R, b = synth.router(5, 0), synth.bias_normal(5, 0)
    ws = B.workspace(max(B.ds4g_forward_workspace(Tmax), B.ds4g_layer_decode_workspace()))

    def fwd(T, wsp):
        out = torch.full((T, H), float("nan"), device=DEV)
        B.ds4g_moe_forward(xd[:T], L.struct, idd[:T], wd[:T], out, wsp)
        assert B.ds4g_last_error(wsp) == 0
        return out.cpu().numpy()

    def layer(wsp):
        i1 = torch.full((K,), -1, dtype=torch.int32, device=DEV)
        w1 = torch.zeros(K, device=DEV)
        o1 = torch.full((H,), float("nan"), device=DEV)
        B.ds4g_moe_layer_decode(xd[0], _t(R), _t(b), L.struct, i1, w1, o1, wsp)
        assert B.ds4g_last_error(wsp) == 0
        return i1.cpu().numpy(), w1.cpu().numpy(), o1.cpu().numpy()

    for T in [1, 2, 3, 64, 2, 5, 1, 64, 3]:
        got = fwd(T, ws)
        ref = fwd(T, B.workspace(B.ds4g_forward_workspace(T)))
        assert np.array_equal(got, ref), f"T={T}"
        if T == 64:
            # the fused layer kernel on the same workspace, then forward again
            a, c = layer(ws), layer(B.workspace(B.ds4g_layer_decode_workspace()))
            assert all(np.array_equal(u, v) for u, v in zip(a, c))
    # the router's workspace across T, past 64 tiles of 32 tokens
    xr = _t(synth.hidden(5, 0, 2100))
    Rd, bd = _t(R), _t(b)
    rws = B.workspace(B.ds4g_route_workspace(2100))
    for T in [1, 2100, 5, 40, 2100, 1]:
        outs = []
        for wsp in (rws, B.workspace(B.ds4g_route_workspace(T))):
            i = torch.full((T, K), -1, dtype=torch.int32, device=DEV)
            ww = torch.zeros(T, K, device=DEV)
            B.ds4g_moe_route(xr[:T], Rd, bd, i, ww, wsp)
            outs.append((i.cpu().numpy(), ww.cpu().numpy()))
        assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1]), f"route T={T}"
