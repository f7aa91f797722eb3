"""Seeded synthetic inputs for the routed-MoE block (shared by the oracle side
and the CUDA side; holds none of the block's arithmetic).

Recipe (all draws are reproducible from ``seed``):

* Integer byte streams (the quantised blocks' code bytes): byte ``8*i + b`` of
  stream ``s`` is byte ``b`` (little-endian) of ``h(seed, s, i)`` with
  ``h(seed, s, i) = splitmix64((seed ^ splitmix64(s)) + i)`` (splitmix64 as
  published by S. Vigna).  ``synth_dev.cu`` is a CUDA twin that writes the
  same bytes directly into device memory for the multi-GB stacks.
* fp16 scale fields (``d``, ``dmin``) of every block are overwritten with
  ``fp16(1e-3 + 3e-3 * u)``, ``u = (h(seed, s | 2^63, n) >> 40) * 2^-24`` where
  ``n`` counts the fp16 fields of the matrix in order; the multiply and add are
  separate fp32 roundings, then fp16 round-to-nearest-even.
* The IQ2_XXS codebook stand-in: 256 distinct rows of 8 values in {8, 25, 43}
  (the real codebook is not available); candidate row ``n`` takes value
  index ``((h(seed, GRID, n) >> 8j) & 0xff) % 3`` for entry ``j``, duplicates
  rejected.
* Gaussian tensors (hidden, router, bias, shared expert) come from numpy's
  PCG64 seeded with ``(seed, stream)``: hidden ~ N(0,1) scaled to unit RMS per
  token, router ~ N(0, 1/4096) (std 1/64), bias ~ N(0, 0.1^2), shared expert
  ~ N(0, 0.02^2) rounded to bf16 (nearest even).  Zipf-skewed bias (s = 1.1):
  a seeded permutation gives each expert a rank r in 1..256 and
  bias = r^-1.1.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

M64 = (1 << 64) - 1
GRID_STREAM = 0x6772696400000000  # "grid"
IQ2_XXS, Q2_K, Q4_K, BF16 = 0, 1, 2, 3
BLOCK_BYTES = {IQ2_XXS: 66, Q2_K: 84, Q4_K: 144}
# byte offsets of the fp16 scale fields inside a GGUF block
FP16_FIELDS = {IQ2_XXS: (0,), Q2_K: (80, 82), Q4_K: (0, 2)}

H, F, E, K = 4096, 2048, 256, 6

# tensor kinds inside a stream id
KIND_GATE, KIND_UP, KIND_DOWN = 1, 2, 3
KIND_HIDDEN, KIND_ROUTER, KIND_BIAS, KIND_SH_GATE, KIND_SH_UP, KIND_SH_DOWN = 4, 5, 6, 7, 8, 9


def stream_id(cfg: int, layer: int, kind: int, expert: int = 0) -> int:
    """Pack (config, layer, tensor kind, expert) into one 63-bit stream id."""
    return ((cfg & 0xff) << 48) | ((layer & 0xffff) << 32) | ((kind & 0xffff) << 16) | (expert & 0xffff)


def splitmix64(x):
    """Vectorised splitmix64 finaliser on uint64 numpy arrays (wraps mod 2^64)."""
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + np.uint64(0x9E3779B97F4A7C15)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def h(seed: int, stream: int, i):
    base = np.uint64(seed & M64) ^ splitmix64(np.uint64(stream & M64))
    with np.errstate(over="ignore"):
        return splitmix64(base + np.asarray(i, dtype=np.uint64))


def byte_stream(seed: int, stream: int, nbytes: int) -> np.ndarray:
    n64 = (nbytes + 7) // 8
    words = h(seed, stream, np.arange(n64, dtype=np.uint64))
    return words.astype("<u8").view(np.uint8)[:nbytes].copy()


def scale_fp16(seed: int, stream: int, n: int) -> np.ndarray:
    """n fp16 scale values in [1e-3, 4e-3] as uint16 bits."""
    u = (h(seed, stream | (1 << 63), np.arange(n, dtype=np.uint64)) >> np.uint64(40)).astype(np.float32)
    t = u * np.float32(2.0 ** -24)            # exact
    t = np.float32(3e-3) * t                   # one rounding
    d = np.float32(1e-3) + t                   # one rounding
    return d.astype(np.float16).view(np.uint16)


def gguf_matrix(qtype: int, rows: int, cols: int, seed: int, stream: int) -> np.ndarray:
    """Random GGUF-format blocks for a [rows][cols] matrix (uint8, flat)."""
    bb = BLOCK_BYTES[qtype]
    nblk = rows * (cols // 256)
    raw = byte_stream(seed, stream, nblk * bb).reshape(nblk, bb)
    fields = FP16_FIELDS[qtype]
    sc = scale_fp16(seed, stream, nblk * len(fields)).reshape(nblk, len(fields))
    for fi, off in enumerate(fields):
        raw[:, off] = (sc[:, fi] & 0xff).astype(np.uint8)
        raw[:, off + 1] = (sc[:, fi] >> 8).astype(np.uint8)
    return raw.reshape(-1)


def iq2_grid(seed: int = 0) -> np.ndarray:
    """256 distinct rows of 8 values in {8, 25, 43} (uint8 [256, 8])."""
    vals = np.array([8, 25, 43], np.uint8)
    rows, seen, n = [], set(), 0
    while len(rows) < 256:
        u = int(h(seed, GRID_STREAM, np.uint64(n)))
        n += 1
        row = tuple(int(vals[((u >> (8 * j)) & 0xff) % 3]) for j in range(8))
        if row in seen:
            continue
        seen.add(row)
        rows.append(row)
    return np.array(rows, np.uint8)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed & M64, stream & M64])))


def normal(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    return (_rng(seed, stream).standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def unit_rms(a: np.ndarray) -> np.ndarray:
    """Scale each row to unit root-mean-square (input recipe, done in fp64)."""
    a64 = a.astype(np.float64)
    return (a64 / np.sqrt((a64 * a64).mean(axis=-1, keepdims=True) + 1e-6)).astype(np.float32)


def hidden(seed: int, cfg: int, T: int, layer: int = 0, normalise: bool = True) -> np.ndarray:
    x = normal(seed, stream_id(cfg, layer, KIND_HIDDEN), (T, H))
    return unit_rms(x) if normalise else x


def router(seed: int, cfg: int, layer: int = 0) -> np.ndarray:
    return normal(seed, stream_id(cfg, layer, KIND_ROUTER), (E, H), std=1.0 / 64.0)


def bias_normal(seed: int, cfg: int, layer: int = 0) -> np.ndarray:
    return normal(seed, stream_id(cfg, layer, KIND_BIAS), (E,), std=0.1)


def bias_zipf(seed: int, cfg: int, layer: int = 0, s: float = 1.1) -> np.ndarray:
    rank = _rng(seed, stream_id(cfg, layer, KIND_BIAS)).permutation(E) + 1
    return (rank.astype(np.float64) ** (-s)).astype(np.float32)


def shared(seed: int, cfg: int, layer: int = 0):
    """bf16 bits: gate [F,H], up [F,H], down [H,F]."""
    g = to_bf16_bits(normal(seed, stream_id(cfg, layer, KIND_SH_GATE), (F, H), 0.02))
    u = to_bf16_bits(normal(seed, stream_id(cfg, layer, KIND_SH_UP), (F, H), 0.02))
    d = to_bf16_bits(normal(seed, stream_id(cfg, layer, KIND_SH_DOWN), (H, F), 0.02))
    return g, u, d


def expert(seed: int, cfg: int, layer: int, e: int, gate_up_type=IQ2_XXS, down_type=Q2_K):
    """GGUF bytes of expert e: gate [F,H], up [F,H], down [H,F]."""
    g = gguf_matrix(gate_up_type, F, H, seed, stream_id(cfg, layer, KIND_GATE, e))
    u = gguf_matrix(gate_up_type, F, H, seed, stream_id(cfg, layer, KIND_UP, e))
    d = gguf_matrix(down_type, H, F, seed, stream_id(cfg, layer, KIND_DOWN, e))
    return g, u, d


# ------------------------------------------------------------- device twin
_HERE = os.path.dirname(os.path.abspath(__file__))
_DEV_SO = os.path.join(_HERE, "libsynth.so")
_DEV_SRC = os.path.join(_HERE, "synth_dev.cu")


def build_device(force: bool = False) -> str:
    if not force and os.path.exists(_DEV_SO) and os.path.getmtime(_DEV_SO) >= os.path.getmtime(_DEV_SRC):
        return _DEV_SO
    subprocess.check_call(["nvcc", "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                           "-Xcompiler", "-fPIC", "-shared", "-o", _DEV_SO, _DEV_SRC])
    return _DEV_SO


_dev = None


def _devlib():
    global _dev
    if _dev is None:
        if not os.path.exists(_DEV_SO):
            raise RuntimeError("synth/libsynth.so is not built (run __graft_entry__.build())")
        L = C.CDLL(_DEV_SO)
        L.synth_fill_gguf.argtypes = [C.c_int, C.c_int, C.c_int, C.c_uint64, C.c_uint64, C.c_void_p,
                                      C.c_void_p]
        L.synth_fill_gguf.restype = C.c_int
        _dev = L
    return _dev


def gguf_matrix_device(qtype: int, rows: int, cols: int, seed: int, stream: int, dev_ptr: int,
                       cuda_stream: int = 0) -> None:
    """Write the same bytes as gguf_matrix() into device memory at dev_ptr."""
    rc = _devlib().synth_fill_gguf(qtype, rows, cols, seed & M64, stream & M64, C.c_void_p(dev_ptr),
                                   C.c_void_p(cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill_gguf failed rc={rc}")
