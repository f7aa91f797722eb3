"""Bit-level identities the decode kernels rest on, checked on the host by
emulating each device formula in numpy (no GPU): the operands the tensor
cores receive are exact, the scales are powers of two in range, and the
integer keys used for the top-6 order floats like the floats."""
import numpy as np

RNG = np.random.default_rng(2024)


def f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def test_q2k_scale_class_masks_give_exact_subnormals():
    # A Q2_K word holds 2-bit quants in slots s = 0..3 of each 16-bit half;
    # masking slot s in place leaves the fp16 subnormal q * 4^s * 2^-24.
    words = np.concatenate([RNG.integers(0, 2**32, 20000, dtype=np.uint64),
                            np.arange(2**16, dtype=np.uint64) * 0x10001]).astype(np.uint32)
    for shift in (0, 8):                       # slots s and s + 4 (the word shifted by 8)
        w = words >> np.uint32(shift)
        for s in range(4):
            m = np.uint32(0x00030003 << (2 * s))
            v = w & m
            for half in (0, 16):
                bits = (v >> np.uint32(half)) & np.uint32(0xFFFF)
                q = (w >> np.uint32(half + 2 * s)) & np.uint32(3)
                assert np.array_equal(f16(bits), q.astype(np.float64) * 4.0**s * 2.0**-24)


def prmt(a, b, sel):
    """PTX prmt.b32 default mode: result byte i = byte (sel nibble i & 7) of
    the 8-byte value {b, a} (a is bytes 0-3)."""
    src = [(a >> (8 * i)) & 255 for i in range(4)] + [(b >> (8 * i)) & 255 for i in range(4)]
    return sum(src[(sel >> (4 * i)) & 7] << (8 * i) for i in range(4))


def test_iq2_value_bytes_and_sign_merge():
    vals = 0x002B1908                          # value bytes 8, 25, 43 and a zero byte
    for code, want in enumerate([8, 25, 43, 0]):
        assert prmt(vals, 0, code) & 255 == want
    # an fp16 assembled as [sign byte 0x80 or 0][value byte] is +-value * 2^-24
    for value in (8, 25, 43):
        for sign in (0, 1):
            bits = (0x80 * sign) << 8 | value
            assert f16(bits) == (-1.0 if sign else 1.0) * value * 2.0**-24
    # the kernel builds two fp16 per register: value bytes (x, y) from a
    # value register, sign bytes from a sign register, selectors 0x5140/0x7362
    for _ in range(200):
        codes = RNG.integers(0, 3, 4)
        vreg = prmt(vals, 0, int(sum(int(c) << (4 * i) for i, c in enumerate(codes))))
        signs = RNG.integers(0, 2, 4)
        sreg = sum((0x80 if sg else 0) << (8 * i) for i, sg in enumerate(signs))
        for sel, pair in ((0x5140, (0, 1)), (0x7362, (2, 3))):
            r = prmt(vreg, sreg, sel)
            got = f16([r & 0xFFFF, r >> 16])
            want = [(-1.0 if signs[i] else 1.0) * [8, 25, 43][codes[i]] * 2.0**-24 for i in pair]
            assert np.array_equal(got, want)


def h_group_exp(m):
    E = ((np.asarray(m, np.float32).view(np.uint32) >> 23) & 255).astype(np.int64) - 126
    return np.where(E > 15, E - 15, 0)


def test_h_scale_is_minimal_and_keeps_fp16_in_range():
    m = np.float32(10.0) ** RNG.uniform(-30, 38.5, 200000).astype(np.float32)
    m = np.concatenate([m, np.float32([0.0, 1e-45, 32767.99, 32768.0, 65503.0, 65504.0, 3.4e38])])
    m = m[np.isfinite(m)]
    e = h_group_exp(m)
    scaled = m.astype(np.float64) * 2.0 ** (-e)
    assert np.all(scaled < 32768.0)                                 # fits fp16 with room
    big = e > 0
    assert np.all(m[big].astype(np.float64) * 2.0 ** (-(e[big] - 1)) >= 32768.0)   # no smaller e works
    assert np.all(e[m < 32768.0] == 0)                              # small groups are untouched
    # the fp16 hi/lo pair of a scaled value keeps ~22 bits of the group's largest value
    x = scaled.astype(np.float32)
    hi = x.astype(np.float16)
    lo = (x - hi.astype(np.float32)).astype(np.float16)
    err = np.abs(x.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
    assert np.all(err <= np.maximum(x.astype(np.float64), 1.0) * 2.0**-21)


def order_key(f):
    u = np.asarray(f, np.float32).view(np.uint32)
    return np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)


def test_order_key_orders_like_the_floats():
    f = np.concatenate([RNG.standard_normal(100000) * 10.0**RNG.integers(-8, 8, 100000),
                        [0.0, 1e-45, -1e-45, 1.0, -1.0, 3.4e38, -3.4e38]]).astype(np.float32)
    k = order_key(f + np.float32(0.0))          # the kernel adds +0 so that -0 keys as +0
    o = np.argsort(f, kind="stable")
    assert np.all(np.diff(k[o].astype(np.int64)) >= 0)
    strictly = np.diff(f[o]) > 0
    assert np.all(np.diff(k[o].astype(np.int64))[strictly] > 0)
    assert order_key(np.float32(-0.0) + np.float32(0.0)) == order_key(np.float32(0.0))


def test_small_integer_conversions():
    # small_u2f(n) = float(n) and half_plus(n) = n + 0.5 for the 4-bit and 8-bit fields
    n = np.arange(256, dtype=np.uint32)
    as_f = (np.uint32(0x4B000000) | n).view(np.float32)
    assert np.array_equal(as_f - np.float32(8388608.0), n.astype(np.float32))
    assert np.array_equal(as_f - np.float32(8388607.5), n.astype(np.float32) + np.float32(0.5))


def test_q4k_nibble_masks_give_exact_subnormals():
    # The per-slot Q4_K down takes nibbles (w >> s0) & 0x000F000F and
    # (w >> (s0 + 4)) & 0x000F000F, s0 in {0, 8}: each half is the fp16
    # subnormal q * 2^-24 of one 4-bit quant.
    words = np.concatenate([RNG.integers(0, 2**32, 20000, dtype=np.uint64),
                            np.arange(2**16, dtype=np.uint64) * 0x10001]).astype(np.uint32)
    for sh in (0, 4, 8, 12):
        v = (words >> np.uint32(sh)) & np.uint32(0x000F000F)
        for half in (0, 16):
            q = (words >> np.uint32(half + sh)) & np.uint32(15)
            assert np.array_equal(f16((v >> np.uint32(half)) & np.uint32(0xFFFF)), q * 2.0**-24)
