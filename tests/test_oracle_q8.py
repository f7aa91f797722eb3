"""Pins of the oracle's q8 mode (int8 activations: chenxutan ds4 article
§2.4, dot_iq2_pair_16, int8 grid values against int8 activations).  The
quantiser is a reading (blocks of 256, d = max|x| / 127, nearest with ties to
even, clamp to +-127); it is pinned by hand-worked blocks and invariants, and
the q8 forward is pinned to the (separately pinned) fp forward: where the
activations are exactly representable in q8, the two are the same sum of the
same exact products."""
import numpy as np
import pytest

import oracle
import synth
from helpers import H, K, host_experts, grid_u64, oracle_forward, oracle_forward_q8


def test_quantiser_hand_worked_blocks():
    # block 0: max 127 -> d = 1 exactly, so q = the value rounded, ties to even
    b0 = np.zeros(256, np.float32)
    b0[:8] = [127.0, 2.5, 3.5, -2.5, 0.5, -0.5, 1.5, -126.6]
    # block 1: max 254 -> d = 2 exactly: 5 -> 2.5 -> 2, 7 -> 3.5 -> 4, -9 -> -4.5 -> -4
    b1 = np.zeros(256, np.float32)
    b1[:4] = [254.0, 5.0, 7.0, -9.0]
    # block 2: all zero -> d = 0, q = 0
    b2 = np.zeros(256, np.float32)
    q, d = oracle.quantize_q8(np.concatenate([b0, b1, b2]))
    assert d.tolist() == [1.0, 2.0, 0.0]
    assert q[:8].tolist() == [127, 2, 4, -2, 0, 0, 2, -127]
    assert q[256:260].tolist() == [127, 2, 4, -4]
    assert not q[8:256].any() and not q[260:].any()


def test_quantiser_invariants():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(4096) * np.repeat(rng.uniform(0.01, 50, 16), 256)).astype(np.float32)
    q, d = oracle.quantize_q8(x)
    assert np.abs(q.astype(np.int32)).max() <= 127
    for b in range(16):
        blk = x[256 * b:256 * b + 256].astype(np.float64)
        assert d[b] == np.float32(np.float32(np.abs(blk).max()) / np.float32(127.0))
        assert np.abs(q[256 * b:256 * b + 256]).max() == 127        # the largest entry maps to +-127
        err = np.abs(blk - q[256 * b:256 * b + 256].astype(np.float64) * d[b])
        assert err.max() <= 0.5 * d[b] * (1 + 1e-6)              # nearest: within half a step
    q2, d2 = oracle.quantize_q8(-x)
    assert np.array_equal(q2, -q) and np.array_equal(d2, d)      # symmetric rounding


def _layer(seed, ids_row):
    grid, _ = grid_u64(seed)
    experts = sorted(set(int(e) for e in ids_row))
    hx = host_experts(seed, 1, 0, experts)
    shared = synth.shared(seed, 1, 0)
    return hx, shared, grid


def test_q8_forward_equals_fp_forward_on_exact_activations():
    """Integer activations with each block's max = 127 quantise losslessly
    (d = 1, q = x): the q8 forward is then the same sum of the same exact
    products (IQ2 weights are exact rationals d_sub * (+-g)) as the fp
    forward, up to fp64 summation order."""
    rng = np.random.default_rng(7)
    x = rng.integers(-127, 128, size=(1, H)).astype(np.float32)
    x[0, ::256] = 127.0
    ids = np.array([[3, 40, 77, 128, 200, 255]], np.int32)
    w = rng.dirichlet(np.ones(K), 1).astype(np.float32)
    hx, shared, grid = _layer(2, ids[0])
    ref = oracle_forward(x, ids, w, hx, shared, grid)
    got = oracle_forward_q8(x, ids, w, hx, shared, grid)
    assert np.max(np.abs(got - ref)) <= 1e-9 * np.max(np.abs(ref))


def test_q8_forward_close_to_fp_forward_on_general_activations():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((2, H)).astype(np.float32)
    ids = np.array([[1, 2, 3, 4, 5, 6], [6, 7, 8, 9, 10, 11]], np.int32)
    w = rng.dirichlet(np.ones(K), 2).astype(np.float32)
    hx, shared, grid = _layer(4, ids.reshape(-1))
    ref = oracle_forward(x, ids, w, hx, shared, grid)
    got = oracle_forward_q8(x, ids, w, hx, shared, grid)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert 0 < rel < 3e-2            # the activation rounding shows (a step of max|x|/127 per block), and stays small


def test_q8_forward_refuses_non_iq2():
    with pytest.raises(ValueError):
        oracle.moe_forward_q8(np.zeros((1, 256), np.float32), np.zeros((1, 1), np.int32),
                              np.ones((1, 1), np.float32), [None], [None], [None],
                              np.zeros((256, 256), np.uint16), np.zeros((256, 256), np.uint16),
                              np.zeros((256, 256), np.uint16), np.zeros(2048, np.uint8),
                              gate_up_type=synth.Q4_K, down_type=synth.Q4_K)
