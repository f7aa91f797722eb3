"""Property tests of the packed device layout (host packer, no GPU): for any
shape the layout admits and any block bytes, unpacking inverts packing, and
packing only moves bits (a permutation that depends on the shape, not on
the values: Q2_K quants are regrouped within bytes)."""
import numpy as np
from hypothesis import given, settings, strategies as st

import bit_quantized_moe_bias_b300 as B

BLOCK = {0: 66, 1: 84, 2: 144}


@st.composite
def matrices(draw):
    qt = draw(st.sampled_from([0, 1, 2]))
    rows = 16 * draw(st.integers(1, 6))
    cols = 256 * draw(st.integers(1, 4))
    seed = draw(st.integers(0, 2**32 - 1))
    data = np.random.default_rng(seed).integers(0, 256, rows * (cols // 256) * BLOCK[qt], dtype=np.uint8)
    return qt, rows, cols, data


@settings(max_examples=60, deadline=None)
@given(matrices())
def test_unpack_inverts_pack(m):
    qt, rows, cols, g = m
    p = B.ds4g_quantize_pack(qt, rows, cols, g)
    assert p.nbytes == g.nbytes == B.ds4g_packed_size(qt, rows, cols)
    assert np.array_equal(B.ds4g_unpack(qt, rows, cols, p), g)


@settings(max_examples=30, deadline=None)
@given(st.sampled_from([0, 1, 2]), st.integers(1, 4), st.integers(1, 3))
def test_pack_is_a_fixed_bit_permutation(qt, rt, ct):
    rows, cols = 16 * rt, 256 * ct
    n = rows * (cols // 256) * BLOCK[qt]
    nbits = 8 * n

    def pack_bits(bits):
        src = np.packbits(bits.astype(np.uint8), bitorder="little")
        return np.unpackbits(B.ds4g_quantize_pack(qt, rows, cols, src), bitorder="little").astype(np.int64)

    # input bit i carries bit k of its own index i; the packed bit j then
    # carries bit k of the index it came from
    idx = np.arange(nbits, dtype=np.int64)
    perm = np.zeros(nbits, np.int64)
    for k in range(int(nbits - 1).bit_length()):
        perm |= pack_bits((idx >> k) & 1) << k
    assert np.array_equal(np.sort(perm), idx)                 # every source bit lands exactly once
    data = np.random.default_rng(rt * 7 + ct + 100 * qt).integers(0, 256, n, dtype=np.uint8)
    bits = np.unpackbits(data, bitorder="little")
    got = np.unpackbits(B.ds4g_quantize_pack(qt, rows, cols, data), bitorder="little")
    assert np.array_equal(got, bits[perm])                    # values only move
