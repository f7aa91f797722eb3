"""Pins of the oracle's fp32 dequantisation arithmetic against exact rational
arithmetic (Python ``fractions.Fraction``), with non-trivial fp16 scales.

The block formats are those of the juejin ds4 article, §2.3 (``block_q2_K``,
``block_iq2_xxs``), with the inner layout and formulas read as the GGUF
convention:
  IQ2_XXS: w = ((d * (0.5 + ls)) * 0.25) * (+-g)
  Q2_K/Q4_K: w = d*sc*q - dmin*m with the multiply-subtract rounded once.

What these pins establish (each is asserted below, not assumed):
* Every product in these formulas is EXACT in fp32: an fp16 scale has at most
  11 significant bits, (0.5 + ls) at most 5, a grid value at most 6, a Q2_K
  scale/min 4 and quant 2, a Q4_K scale/min 6 and quant 4, so no product has
  more than 24 significant bits (the fp16 subnormal range included).  Hence
  the fused (fmaf) and unfused evaluation orders, and any re-association of
  the products, give the same bits; the order is not a free choice that a
  test could get wrong.
* The one rounding is the final subtraction of Q2_K/Q4_K: the oracle must
  return the exact rational d*sc*q - dmin*m rounded ONCE to the nearest fp32
  (ties to even).  The hand-built blocks below make that subtraction inexact
  for a large share of weights, so a truncating subtraction, an fp16 or bf16
  intermediate, or a dropped/doubled term fails.
* IQ2_XXS values are the exact rationals d*(0.5+ls)/4*(+-g) for fp16 d over
  the whole finite range, subnormals included.

Expected values come from Fraction arithmetic and an integer
round-to-nearest-even written here; fp16 bit patterns are decoded by numpy.
Nothing here calls the oracle to produce an expected value.
"""
from fractions import Fraction
import math
import struct

import numpy as np

import oracle


def f16(bits: int) -> Fraction:
    """Exact value of an fp16 bit pattern (numpy's decode, exact in float64)."""
    return Fraction(float(np.array([bits], np.uint16).view(np.float16)[0]))


def round_f32(x: Fraction) -> float:
    """x rounded once to the nearest binary32 value, ties to even (normal and
    subnormal range; the values here never overflow)."""
    if x == 0:
        return 0.0
    s = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()   # 2^e <= a < 2^(e+2)
    if a < Fraction(2) ** e:
        e -= 1
    while a >= Fraction(2) ** (e + 1):
        e += 1
    q = max(e, -126) - 23                 # exponent of one unit in the last place
    m = a / Fraction(2) ** q
    n = m.numerator // m.denominator
    r = m - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return s * math.ldexp(n, q)


def representable(x: Fraction) -> bool:
    return Fraction(round_f32(x)) == x


def truncate_f32(x: Fraction) -> float:
    """x truncated toward zero to binary32 (a plausible wrong rounding)."""
    if x == 0:
        return 0.0
    s = -1 if x < 0 else 1
    a = abs(x)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = max(e, -126) - 23
    m = a / Fraction(2) ** q
    return s * math.ldexp(m.numerator // m.denominator, q)


def test_round_f32_helper_against_known_values():
    # 1 + 2^-24 is a tie between 1 and 1 + 2^-23: even -> 1
    assert round_f32(Fraction(1) + Fraction(1, 2 ** 24)) == 1.0
    # 1 + 3*2^-24 ties between 1+2^-23 and 1+2^-22: even -> 1 + 2^-22
    assert round_f32(Fraction(1) + Fraction(3, 2 ** 24)) == 1.0 + 2.0 ** -22
    assert round_f32(Fraction(1, 3)) == float(np.float32(1 / 3))
    assert round_f32(Fraction(-7, 10)) == float(np.float32(-0.7))
    assert round_f32(Fraction(1, 2 ** 149)) == 2.0 ** -149            # smallest subnormal
    assert round_f32(Fraction(1, 2 ** 150)) == 0.0                    # tie -> even (0)
    for v in np.random.default_rng(0).standard_normal(2000):
        assert round_f32(Fraction(float(v))) == float(np.float32(v))


# ------------------------------------------------------------------ Q2_K
def _q2k_block(scales, qs, d_bits, dmin_bits):
    out = bytes(scales) + bytes(qs) + struct.pack("<HH", d_bits, dmin_bits)
    return np.frombuffer(out, np.uint8)


def _q2k_fields(n):
    """(qs byte index, shift, sub-block) of weight n: the GGUF element map."""
    h, j, l = n // 128, (n % 128) // 32, n % 32
    return 32 * h + l, 2 * j, 8 * h + 2 * j + (1 if l >= 16 else 0)


# fp16 (d, dmin) pairs chosen so that d*sc*q and dmin*m have many significant
# bits and differ in exponent: the subtraction then has to round.
Q2K_SCALES = [(0x3555, 0x0123), (0x1A3F, 0x3BFF), (0x13FF, 0x0001), (0x7BFF, 0x3C01), (0x2E66, 0x1A9B),
              (0x0155, 0x03FF)]


def test_q2_k_final_subtraction_rounds_once():
    rng = np.random.default_rng(11)
    blocks, expect, trunc = [], [], []
    inexact = 0
    for d_bits, dmin_bits in Q2K_SCALES:
        d, dmin = f16(d_bits), f16(dmin_bits)
        for base in range(0, 256, 16):            # every (sc, m) byte value once per scale pair
            scales = list(range(base, base + 16))
            qs = list(rng.integers(0, 256, 64))
            blocks.append(_q2k_block(scales, qs, d_bits, dmin_bits))
            for n in range(256):
                bi, sh, sb = _q2k_fields(n)
                q = (qs[bi] >> sh) & 3
                sc, m = scales[sb] & 15, scales[sb] >> 4
                # lemma: both products exact in fp32, so no evaluation order matters
                assert representable(d * sc * q) and representable(d * sc) and representable(dmin * m)
                x = d * sc * q - dmin * m
                inexact += not representable(x)
                expect.append(round_f32(x))
                trunc.append(truncate_f32(x))
    w = oracle.dequantize(oracle.Q2_K, np.concatenate(blocks), len(blocks), 256).reshape(-1)
    assert [float(v) for v in w] == expect
    assert inexact > 2000                         # the subtraction really rounds, often
    assert sum(a != b for a, b in zip(expect, trunc)) > 500   # a truncating oracle would fail


def test_q2_k_fp16_intermediate_would_fail():
    """An fp16 product d*sc (what half-precision arithmetic would give) is
    not the format's value: this pin separates the two."""
    d_bits, dmin_bits = 0x3555, 0x0123
    scales, qs = list(range(16)), [0xE4] * 64
    w = oracle.dequantize(oracle.Q2_K, _q2k_block(scales, qs, d_bits, dmin_bits), 1, 256)[0]
    d, dmin = f16(d_bits), f16(dmin_bits)
    differs = 0
    for n in range(256):
        bi, sh, sb = _q2k_fields(n)
        q = (qs[bi] >> sh) & 3
        sc, m = scales[sb] & 15, scales[sb] >> 4
        half = Fraction(float(np.float16(float(d * sc)))) * q - dmin * m
        differs += round_f32(half) != float(w[n])
        assert float(w[n]) == round_f32(d * sc * q - dmin * m)
    assert differs > 0


# ------------------------------------------------------------------ Q4_K
def _q4k_block(d_bits, dmin_bits, scales, qs):
    out = struct.pack("<HH", d_bits, dmin_bits) + bytes(scales) + bytes(qs)
    return np.frombuffer(out, np.uint8)


def _q4k_scale_min(s, i):
    if i < 4:
        return s[i] & 63, s[i + 4] & 63
    return (s[i + 4] & 15) | ((s[i - 4] >> 6) << 4), (s[i + 4] >> 4) | ((s[i] >> 6) << 4)


def test_q4_k_final_subtraction_rounds_once():
    rng = np.random.default_rng(12)
    blocks, expect = [], []
    inexact = 0
    for d_bits, dmin_bits in Q2K_SCALES:
        d, dmin = f16(d_bits), f16(dmin_bits)
        for _ in range(24):
            scales = list(rng.integers(0, 256, 12))
            qs = list(rng.integers(0, 256, 128))
            blocks.append(_q4k_block(d_bits, dmin_bits, scales, qs))
            for n in range(256):
                c, r = n // 64, n % 64
                q = (qs[32 * c + r] & 15) if r < 32 else (qs[32 * c + r - 32] >> 4)
                sc, m = _q4k_scale_min(scales, 2 * c + (r >= 32))
                assert representable(d * sc * q) and representable(dmin * m)
                x = d * sc * q - dmin * m
                inexact += not representable(x)
                expect.append(round_f32(x))
    w = oracle.dequantize(oracle.Q4_K, np.concatenate(blocks), len(blocks), 256).reshape(-1)
    assert [float(v) for v in w] == expect
    assert inexact > 2000


# --------------------------------------------------------------- IQ2_XXS
def _iq2_block(d_bits, subblocks):
    out = struct.pack("<H", d_bits)
    for idx, v in subblocks:
        out += bytes(idx) + struct.pack("<I", v)
    return np.frombuffer(out, np.uint8)


def test_iq2_xxs_values_are_exact_rationals_any_d():
    """Random fp16 d over the whole finite range (subnormals included), every
    scale nibble, random grid rows and sign indices: the oracle's weight is
    exactly d * (0.5 + ls) / 4 * (+-g), which is always representable."""
    rng = np.random.default_rng(13)
    grid = np.array([[(8, 25, 43)[(r * 7 + j * 3 + r // 5) % 3] for j in range(8)] for r in range(256)], np.uint8)
    d_list = [0x3555, 0x0001, 0x03FF, 0x0400, 0x7BFF, 0x1A3F] + [int(b) for b in rng.integers(1, 0x7C00, 26)]
    blocks, expect = [], []
    for d_bits in d_list:
        d = f16(d_bits)
        sbs = []
        for b in range(8):
            idx = [int(v) for v in rng.integers(0, 256, 4)]
            s7 = [int(v) for v in rng.integers(0, 128, 4)]
            ls = (2 * b + (d_bits & 1)) % 16
            v = s7[0] | (s7[1] << 7) | (s7[2] << 14) | (s7[3] << 21) | (ls << 28)
            sbs.append((idx, v))
            db = d * (Fraction(1, 2) + ls) / 4
            for l in range(4):
                signs = s7[l] | ((bin(s7[l]).count("1") & 1) << 7)
                for j in range(8):
                    g = int(grid[idx[l], j]) * (-1 if (signs >> j) & 1 else 1)
                    x = db * g
                    assert representable(x) and representable(d * (Fraction(1, 2) + ls))
                    expect.append(float(x))
        blocks.append(_iq2_block(d_bits, sbs))
    w = oracle.dequantize(oracle.IQ2_XXS, np.concatenate(blocks), len(blocks), 256, grid).reshape(-1)
    assert [float(v) for v in w] == expect
