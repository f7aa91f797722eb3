"""Pins of the CPU oracle against things other than itself.

Expected values here are hand-derived literals (from the block structs of the
juejin ds4 article, §2.3, and the inner-layout reading stated in oracle.c),
closed forms, brute force, or independent numpy / Python routines.  None is
produced by the oracle.
"""
import math
import struct

import numpy as np
import pytest

import oracle
import synth

ONE_F16 = 0x3C00


# ------------------------------------------------------------ scalar conversions
@pytest.mark.parametrize("bits,val", [
    (0x3C00, 1.0), (0x0001, 2.0 ** -24), (0x03FF, 1023 * 2.0 ** -24), (0x0400, 2.0 ** -14),
    (0x7BFF, 65504.0), (0xC000, -2.0), (0x3555, 0.333251953125), (0x8000, -0.0), (0x1400, 2.0 ** -10),
])
def test_fp16_to_f32_literals(bits, val):
    got = oracle.fp16_to_f32(bits)
    assert got == val and math.copysign(1, got) == math.copysign(1, val)


def test_fp16_to_f32_all_finite_match_numpy():
    bits = np.arange(0x10000, dtype=np.uint32)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float32)
    for b in range(0, 0x10000, 97):
        r = ref[b]
        g = oracle.fp16_to_f32(int(b))
        if np.isnan(r):
            assert math.isnan(g)
        else:
            assert g == r


@pytest.mark.parametrize("val,bits", [
    (1.0, 0x3F80),
    (1.0 + 2.0 ** -8, 0x3F80),             # tie -> even (down)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),         # tie -> even (up)
    (1.0 + 2.0 ** -8 + 2.0 ** -20, 0x3F81),  # above the tie
    (-1.5, 0xBFC0),
    (3.4028234663852886e38, 0x7F80),       # max float rounds to inf
    (0.0, 0x0000),
])
def test_bf16_rounding_literals(val, bits):
    assert oracle.f32_to_bf16(val) == bits


# ---------------------------------------------------------------- IQ2_XXS
def _grid():
    g = np.zeros((256, 8), np.uint8)
    for r in range(256):
        g[r] = [(8, 25, 43)[(r + j) % 3] for j in range(8)]
    g[0] = [8] * 8
    g[1] = [25] * 8
    g[2] = [43] * 8
    g[3] = [8, 25, 43, 8, 25, 43, 8, 25]
    g[5] = [43, 25, 8, 43, 25, 8, 43, 25]
    return g


def _iq2_block(d_bits, subblocks):
    """subblocks: 8 x (four grid indices, word v) -> 66 bytes."""
    out = struct.pack("<H", d_bits)
    for idx, v in subblocks:
        out += bytes(idx) + struct.pack("<I", v)
    assert len(out) == 66
    return np.frombuffer(out, np.uint8)


def test_iq2_xxs_hand_built_blocks():
    grid = _grid()
    v1 = 1 | (3 << 7) | (0x7F << 14) | (0x40 << 21) | (15 << 28)
    blk_a = _iq2_block(ONE_F16, [((0, 1, 2, 3), 0), ((5, 5, 5, 5), v1)] + [((2, 2, 2, 2), 1 << 28)] * 6)
    blk_b = _iq2_block(0x3800, [((1, 1, 1, 1), 3 << 28)] + [((0, 0, 0, 0), 0)] * 7)
    w = oracle.dequantize(oracle.IQ2_XXS, np.concatenate([blk_a, blk_b]), 1, 512, grid)[0]
    # block a, sub-block 0: d = 1, ls = 0 -> db = 1 * 0.5 * 0.25 = 0.125
    assert list(w[0:8]) == [1.0] * 8                         # 8 * 0.125
    assert list(w[8:16]) == [3.125] * 8                      # 25 * 0.125
    assert list(w[16:24]) == [5.375] * 8                     # 43 * 0.125
    assert list(w[24:32]) == [1.0, 3.125, 5.375, 1.0, 3.125, 5.375, 1.0, 3.125]
    # sub-block 1: ls = 15 -> db = 15.5 * 0.25 = 3.875; row 5 * 3.875
    p = [166.625, 96.875, 31.0, 166.625, 96.875, 31.0, 166.625, 96.875]
    # sign index 1 -> parity 1 -> weights 0 and 7 negative
    assert list(w[32:40]) == [-p[0], p[1], p[2], p[3], p[4], p[5], p[6], -p[7]]
    # sign index 3 -> parity 0 -> weights 0, 1 negative
    assert list(w[40:48]) == [-p[0], -p[1], p[2], p[3], p[4], p[5], p[6], p[7]]
    # sign index 127 -> parity 1 -> all eight negative
    assert list(w[48:56]) == [-x for x in p]
    # sign index 64 (bit 6) -> parity 1 -> weights 6 and 7 negative
    assert list(w[56:64]) == [p[0], p[1], p[2], p[3], p[4], p[5], -p[6], -p[7]]
    # sub-blocks 2..7: ls = 1 -> db = 1.5 * 0.25 = 0.375; 43 * 0.375
    assert np.all(w[64:256] == 16.125)
    # block b: d = 0.5, ls = 3 -> db = 0.5 * 3.5 * 0.25 = 0.4375; 25 * 0.4375
    assert np.all(w[256:288] == 10.9375)
    assert np.all(w[288:512] == 0.5)                         # 8 * 0.5 * 0.5 * 0.25


def test_iq2_xxs_sign_parity_every_pattern():
    """For every 7-bit sign index the number of negative weights is even and
    the first seven follow the index bits."""
    grid = _grid()
    blocks = []
    for s7 in range(128):
        sb = [((1, 1, 1, 1), s7)] + [((1, 1, 1, 1), 0)] * 7
        blocks.append(_iq2_block(ONE_F16, sb))
    w = oracle.dequantize(oracle.IQ2_XXS, np.concatenate(blocks), 1, 256 * 128, grid)[0]
    for s7 in range(128):
        neg = w[256 * s7: 256 * s7 + 8] < 0
        assert neg.sum() % 2 == 0
        assert [bool((s7 >> j) & 1) for j in range(7)] == list(neg[:7])


# ------------------------------------------------------------------- Q2_K
def _q2k_block(scales, qs, d_bits, dmin_bits):
    out = bytes(scales) + bytes(qs) + struct.pack("<HH", d_bits, dmin_bits)
    assert len(out) == 84
    return np.frombuffer(out, np.uint8)


def test_q2_k_single_bit_moves_one_weight():
    blocks = []
    where = []
    for bi in range(64):
        for j in range(4):
            qs = [0] * 64
            qs[bi] = 1 << (2 * j)
            blocks.append(_q2k_block([0x01] * 16, qs, ONE_F16, 0))
            where.append(128 * (bi // 32) + 32 * j + bi % 32)
    w = oracle.dequantize(oracle.Q2_K, np.concatenate(blocks), len(blocks), 256)
    for r, n in enumerate(where):
        nz = np.nonzero(w[r])[0]
        assert list(nz) == [n] and w[r, n] == 1.0
    assert sorted(where) == list(range(256))       # the map is a bijection


def test_q2_k_subblock_is_n_div_16():
    # q = 1 everywhere (0b01010101), sc = sub-block index, m = 0
    w = oracle.dequantize(oracle.Q2_K, _q2k_block(list(range(16)), [0x55] * 64, ONE_F16, 0), 1, 256)[0]
    assert np.array_equal(w, (np.arange(256) // 16).astype(np.float32))
    # d = 0, dmin = 1, m = sub-block index: w = -m
    w = oracle.dequantize(oracle.Q2_K, _q2k_block([s << 4 for s in range(16)], [0x55] * 64, 0, ONE_F16), 1, 256)[0]
    assert np.array_equal(w, -(np.arange(256) // 16).astype(np.float32))


def test_q2_k_scale_min_combination():
    # d = 0.5, dmin = 0.25, sc = 1, m = 2, q = 3: 0.5*1*3 - 0.25*2 = 1.0
    w = oracle.dequantize(oracle.Q2_K, _q2k_block([0x21] * 16, [0xFF] * 64, 0x3800, 0x3400), 1, 256)[0]
    assert np.all(w == 1.0)
    # q = 0 -> -dmin*m = -0.5
    w = oracle.dequantize(oracle.Q2_K, _q2k_block([0x21] * 16, [0x00] * 64, 0x3800, 0x3400), 1, 256)[0]
    assert np.all(w == -0.5)


# ------------------------------------------------------------------- Q4_K
Q4_SCALES = [0x41, 0x82, 0xC3, 0x04, 0x45, 0x86, 0xC7, 0x08, 0x9A, 0xBC, 0xDE, 0xF0]
Q4_SC = [1, 2, 3, 4, 26, 44, 62, 0]      # derived by hand from the 6-bit packing
Q4_M = [5, 6, 7, 8, 25, 43, 61, 15]


def _q4k_block(d_bits, dmin_bits, scales, qs):
    out = struct.pack("<HH", d_bits, dmin_bits) + bytes(scales) + bytes(qs)
    assert len(out) == 144
    return np.frombuffer(out, np.uint8)


def test_q4_k_scale_unpack_both_branches():
    w = oracle.dequantize(oracle.Q4_K, _q4k_block(ONE_F16, 0, Q4_SCALES, [0x11] * 128), 1, 256)[0]
    assert np.array_equal(w, np.repeat(np.array(Q4_SC, np.float32), 32))
    w = oracle.dequantize(oracle.Q4_K, _q4k_block(0, ONE_F16, Q4_SCALES, [0x11] * 128), 1, 256)[0]
    assert np.array_equal(w, -np.repeat(np.array(Q4_M, np.float32), 32))


def test_q4_k_single_nibble_map():
    blocks, where = [], []
    for bi in range(128):
        for hi in (0, 1):
            qs = [0] * 128
            qs[bi] = 0x10 if hi else 0x01
            s = [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1]   # sc = 1, m = 0 for all eight
            blocks.append(_q4k_block(ONE_F16, 0, s, qs))
            c, l = bi // 32, bi % 32
            where.append(64 * c + 32 * hi + l)
    w = oracle.dequantize(oracle.Q4_K, np.concatenate(blocks), len(blocks), 256)
    for r, n in enumerate(where):
        assert list(np.nonzero(w[r])[0]) == [n] and w[r, n] == 1.0
    assert sorted(where) == list(range(256))


def test_dequant_bf16_is_rne_of_f32():
    g = synth.gguf_matrix(oracle.Q2_K, 16, 512, 3, 77)
    f, b = oracle.dequantize(oracle.Q2_K, g, 16, 512, bf16=True)
    ref = synth.to_bf16_bits(f)          # independent numpy rounding
    assert np.array_equal(b, ref)


# ----------------------------------------------------------------- router
def _route_brute(x, R, bias, K):
    keys = 1.0 / (1.0 + np.exp(-(x.astype(np.float64) @ R.astype(np.float64).T))) + bias.astype(np.float64)
    s = keys - bias.astype(np.float64)
    ids = []
    for t in range(x.shape[0]):
        order = sorted(range(R.shape[0]), key=lambda e: (-keys[t, e], e))
        ids.append(order[:K])
    ids = np.array(ids)
    w = np.take_along_axis(s, ids, 1)
    return ids, w / w.sum(1, keepdims=True), keys


def test_route_matches_brute_force_sort():
    x = synth.hidden(1, 9, 12)
    R = synth.router(1, 9)
    b = synth.bias_normal(1, 9)
    ids, w, keys, margin = oracle.route(x, R, b)
    rid, rw, rkeys = _route_brute(x, R, b, 6)
    assert np.allclose(keys, rkeys, rtol=0, atol=1e-12)
    for t in range(12):
        assert margin[t] > 1e-9
        assert list(ids[t]) == list(rid[t])
    assert np.allclose(w, rw, atol=1e-7)
    assert np.allclose(w.sum(1), 1.0, atol=1e-6) and np.all(w > 0)
    for t in range(12):
        kk = keys[t, ids[t]]
        assert np.all(np.diff(kk) <= 0)


def test_route_exact_ties_go_to_lower_id():
    H, E = 256, 16
    x = np.ones((1, H), np.float32) / 16
    R = np.zeros((E, H), np.float32)
    R[[3, 10, 12]] = 0.05          # three identical top rows
    b = np.zeros(E, np.float32)
    ids, w, keys, _ = oracle.route(x, R, b, K=2)
    assert list(ids[0]) == [3, 10]
    assert w[0, 0] == w[0, 1] == np.float32(0.5)


def test_route_zero_router_uses_bias_order_and_equal_weights():
    E = 256
    x = synth.hidden(0, 9, 1)
    R = np.zeros((E, 4096), np.float32)
    b = synth.bias_zipf(0, 9)
    ids, w, _, _ = oracle.route(x, R, b)
    assert list(ids[0]) == list(np.argsort(-b, kind="stable")[:6])
    assert np.allclose(w, 1.0 / 6, atol=1e-7)


# ----------------------------------------------------------------- bucket
@pytest.mark.parametrize("T,mode", [(1, "rand"), (7, "rand"), (33, "one"), (64, "zipf")])
def test_bucket_matches_stable_sort(T, mode):
    rng = np.random.default_rng(T)
    if mode == "one":
        ids = np.full((T, 6), 17, np.int32)
    elif mode == "zipf":
        ids = np.minimum(rng.zipf(1.5, (T, 6)) - 1, 255).astype(np.int32)
    else:
        ids = rng.integers(0, 256, (T, 6)).astype(np.int32)
    counts, offsets, perm, inv = oracle.bucket(ids)
    flat = ids.reshape(-1)
    ref_perm = sorted(range(flat.size), key=lambda i: flat[i])   # Python sort is stable
    assert list(perm) == ref_perm
    assert np.array_equal(counts, np.bincount(flat, minlength=256))
    assert offsets[0] == 0 and offsets[-1] == flat.size
    assert np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(perm[inv], np.arange(flat.size))


def test_rmsnorm_closed_form():
    x = np.full((2, 4096), 3.0, np.float32)
    x[1] = -0.5
    y = oracle.rmsnorm(x)
    assert np.allclose(y[0], 3.0 / math.sqrt(9.0 + 1e-6), rtol=1e-7)
    assert np.allclose(y[1], -0.5 / math.sqrt(0.25 + 1e-6), rtol=1e-7)


# ------------------------------------------------------------- MoE block
def _tiny_layer(seed, H, F, E, gut=oracle.IQ2_XXS, dt=oracle.Q2_K):
    gate = [synth.gguf_matrix(gut, F, H, seed, 100 + e) for e in range(E)]
    up = [synth.gguf_matrix(gut, F, H, seed, 200 + e) for e in range(E)]
    down = [synth.gguf_matrix(dt, H, F, seed, 300 + e) for e in range(E)]
    shg = synth.to_bf16_bits(synth.normal(seed, 1, (F, H), 0.02))
    shu = synth.to_bf16_bits(synth.normal(seed, 2, (F, H), 0.02))
    shd = synth.to_bf16_bits(synth.normal(seed, 3, (H, F), 0.02))
    return gate, up, down, shg, shu, shd


def _bf16_to_f64(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _dense_numpy(x, wmask, gate, up, down, shg, shu, shd, grid, H, F, gut, dt):
    """sum over ALL experts of mask*w*expert(x) + shared, with numpy fp64."""
    silu = lambda v: v / (1.0 + np.exp(-v))
    x64 = x.astype(np.float64)
    out = np.zeros((x.shape[0], H))
    for e in range(len(gate)):
        if not np.any(wmask[:, e]):
            continue
        G = oracle.dequantize(gut, gate[e], F, H, grid).astype(np.float64)
        U = oracle.dequantize(gut, up[e], F, H, grid).astype(np.float64)
        D = oracle.dequantize(dt, down[e], H, F, grid).astype(np.float64)
        y = (silu(x64 @ G.T) * (x64 @ U.T)) @ D.T
        out += wmask[:, e:e + 1] * y
    Sg, Su, Sd = _bf16_to_f64(shg), _bf16_to_f64(shu), _bf16_to_f64(shd)
    out += (silu(x64 @ Sg.T) * (x64 @ Su.T)) @ Sd.T
    return out


@pytest.mark.parametrize("gut,dt", [(oracle.IQ2_XXS, oracle.Q2_K), (oracle.Q4_K, oracle.Q4_K)])
def test_sparse_equals_dense_masked(gut, dt):
    H, F, E, K, T = 512, 256, 8, 3, 5
    grid = synth.iq2_grid(0)
    gate, up, down, shg, shu, shd = _tiny_layer(4, H, F, E, gut, dt)
    x = synth.unit_rms(synth.normal(4, 9, (T, H)))
    R = synth.normal(4, 10, (E, H), 1 / 16)
    ids, w, _, _ = oracle.route(x, R, synth.normal(4, 11, (E,), 0.1), K=K)
    out = oracle.moe_forward(x, ids, w, gate, up, down, shg, shu, shd, grid, gut, dt, F=F)
    wmask = np.zeros((T, E))
    for t in range(T):
        for k in range(K):
            wmask[t, ids[t, k]] += w[t, k]
    ref = _dense_numpy(x, wmask, gate, up, down, shg, shu, shd, grid, H, F, gut, dt)
    assert np.max(np.abs(out - ref)) <= 1e-6 * np.max(np.abs(ref))


def test_token_permutation_equivariance_bit_exact():
    H, F, E, K, T = 256, 256, 8, 3, 6
    grid = synth.iq2_grid(0)
    gate, up, down, shg, shu, shd = _tiny_layer(5, H, F, E)
    x = synth.unit_rms(synth.normal(5, 9, (T, H)))
    ids = np.random.default_rng(0).integers(0, E, (T, K)).astype(np.int32)
    w = np.random.default_rng(1).random((T, K)).astype(np.float32)
    out = oracle.moe_forward(x, ids, w, gate, up, down, shg, shu, shd, grid, F=F)
    p = np.random.default_rng(2).permutation(T)
    out_p = oracle.moe_forward(x[p], ids[p], w[p], gate, up, down, shg, shu, shd, grid, F=F)
    assert np.array_equal(out_p, out[p])


def test_identical_selected_experts_reduce_to_one():
    H, F, E, K = 256, 256, 8, 3
    grid = synth.iq2_grid(0)
    gate, up, down, shg, shu, shd = _tiny_layer(6, H, F, E)
    for e in (4, 6):
        gate[e], up[e], down[e] = gate[1], up[1], down[1]
    x = synth.unit_rms(synth.normal(6, 9, (1, H)))
    ids = np.array([[1, 4, 6]], np.int32)
    w = np.array([[0.5, 0.3, 0.2]], np.float32)
    out = oracle.moe_forward(x, ids, w, gate, up, down, shg, shu, shd, grid, F=F)
    zero_sh = [np.zeros_like(a) for a in (shg, shu, shd)]
    routed = oracle.moe_forward(x, ids, w, gate, up, down, *zero_sh, grid, F=F)
    y1 = oracle.expert_mlp(x[0], gate[1], up[1], down[1], grid, H, F)
    assert np.allclose(routed[0], y1 * (0.5 + 0.3 + 0.2), rtol=1e-6, atol=1e-6 * np.abs(y1).max())
    sh_only = out - routed
    assert np.all(np.isfinite(sh_only))


def test_constant_weights_closed_form_full_dims():
    """All routed and shared weights equal 1.0 and x = 1/4096: every gate/up
    row sums x to S = 1, h = silu(1), every down row sums h to 2048*silu(1);
    routed weights sum to 1, so out = 2 * 2048 * silu(1) everywhere."""
    H, F, E = 4096, 2048, 256
    grid = np.tile(np.array([8], np.uint8), (256, 8))
    iq2 = np.tile(np.frombuffer(struct.pack("<H", ONE_F16) + bytes(64), np.uint8), F * H // 256)
    q2k = np.tile(_q2k_block([0x01] * 16, [0x55] * 64, ONE_F16, 0), H * F // 256)
    gate = [None] * E
    up = [None] * E
    down = [None] * E
    for e in (0, 7, 100, 255, 3, 42):
        gate[e], up[e], down[e] = iq2, iq2, q2k
    ones = np.full((F, H), 0x3F80, np.uint16)
    x = np.full((1, H), 1.0 / 4096, np.float32)
    ids = np.array([[0, 7, 100, 255, 3, 42]], np.int32)
    w = np.array([[0.25, 0.25, 0.125, 0.125, 0.125, 0.125]], np.float32)
    out = oracle.moe_forward(x, ids, w, gate, up, down, ones, ones, ones.T.copy(), grid)
    silu1 = 1.0 / (1.0 + math.exp(-1.0))
    assert np.allclose(out, 2 * 2048 * silu1, rtol=1e-6)


def test_full_dims_single_token_matches_numpy():
    """Real dims, one token, synthetic weights: oracle vs numpy fp64 dense."""
    H, F = 4096, 2048
    seed, cfg = 0, 0
    grid = synth.iq2_grid(seed)
    x = synth.hidden(seed, cfg, 1)
    ids, w, _, _ = oracle.route(x, synth.router(seed, cfg), synth.bias_normal(seed, cfg))
    gate, up, down = [None] * 256, [None] * 256, [None] * 256
    for e in ids[0]:
        gate[e], up[e], down[e] = synth.expert(seed, cfg, 0, int(e))
    shg, shu, shd = synth.shared(seed, cfg)
    out = oracle.moe_forward(x, ids, w, gate, up, down, shg, shu, shd, grid)
    wmask = np.zeros((1, 256))
    for k in range(6):
        wmask[0, ids[0, k]] += w[0, k]
    ref = _dense_numpy(x, wmask, gate, up, down, shg, shu, shd, grid, H, F, oracle.IQ2_XXS, oracle.Q2_K)
    assert np.max(np.abs(out - ref)) <= 1e-6 * np.max(np.abs(ref))
