"""CPU oracle of the routed-MoE block — TEST INFRASTRUCTURE.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg (and
its ``--impl reference`` arm, which times this oracle) may import this
package.  It wraps ``oracle.c`` (plain C11, fp64 accumulation, no code shared
with the CUDA library) through ctypes and numpy.

Parity status: real-model numerics: parity unpinned (no real IQ2_XXS
codebook, weights or test vectors are available); every function is pinned by
tests/test_oracle_pins.py against hand-derived values, closed forms,
brute force and independent numpy computations.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = [os.path.join(_HERE, "oracle.c"), os.path.join(_HERE, "oracle.h")]

IQ2_XXS, Q2_K, Q4_K, BF16 = 0, 1, 2, 3
BLOCK_BYTES = {IQ2_XXS: 66, Q2_K: 84, Q4_K: 144}


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (-O2 -ffp-contract=off -fopenmp)."""
    if not force and os.path.exists(_SO):
        so_t = os.path.getmtime(_SO)
        if all(os.path.getmtime(s) <= so_t for s in _SRC):
            return _SO
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", _SO, _SRC[0], "-lm"]
    subprocess.check_call(cmd)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_SO)
        vp, i32, f32p = C.c_void_p, C.c_int, C.c_void_p
        L.oracle_fp16_to_f32.argtypes = [C.c_uint16]
        L.oracle_fp16_to_f32.restype = C.c_float
        L.oracle_f32_to_bf16.argtypes = [C.c_float]
        L.oracle_f32_to_bf16.restype = C.c_uint16
        L.oracle_dequantize.argtypes = [i32, vp, i32, i32, vp, vp, vp]
        L.oracle_route.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.oracle_bucket.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
        L.oracle_rmsnorm.argtypes = [vp, i32, i32, C.c_double, vp]
        L.oracle_rmsnorm.restype = None
        L.oracle_moe_forward.argtypes = [vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp,
                                         vp, vp, vp, vp, vp, vp, vp, i32]
        L.oracle_expert_mlp.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, i32]
        L.oracle_quantize_q8.argtypes = [vp, i32, vp, vp]
        L.oracle_moe_forward_q8.argtypes = L.oracle_moe_forward.argtypes
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def fp16_to_f32(h: int) -> float:
    return float(lib().oracle_fp16_to_f32(int(h)))


def f32_to_bf16(f: float) -> int:
    return int(lib().oracle_f32_to_bf16(float(f)))


def dequantize(qtype: int, gguf: np.ndarray, rows: int, cols: int, grid=None, bf16=False):
    """GGUF-format bytes -> fp32 [rows, cols] (and bf16 bits if bf16=True)."""
    gguf = _c(gguf, np.uint8)
    assert gguf.size >= rows * cols // 256 * BLOCK_BYTES[qtype]
    g = None if grid is None else _c(grid, np.uint8)
    out = np.empty((rows, cols), np.float32)
    ob = np.empty((rows, cols), np.uint16) if bf16 else None
    rc = lib().oracle_dequantize(qtype, _p(gguf), rows, cols, _p(g), _p(out), _p(ob))
    if rc:
        raise ValueError(f"oracle_dequantize rc={rc}")
    return (out, ob) if bf16 else out


def route(hidden: np.ndarray, router: np.ndarray, bias: np.ndarray, K: int = 6):
    """-> ids [T,K] int32, w [T,K] f32, keys [T,E] f64, margin [T] f64."""
    hidden = _c(hidden, np.float32)
    router = _c(router, np.float32)
    bias = _c(bias, np.float32)
    T, H = hidden.shape
    E = router.shape[0]
    ids = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    keys = np.empty((T, E), np.float64)
    margin = np.empty((T,), np.float64)
    rc = lib().oracle_route(_p(hidden), T, H, E, K, _p(router), _p(bias), _p(ids), _p(w),
                            _p(keys), _p(margin))
    if rc:
        raise ValueError(f"oracle_route rc={rc}")
    return ids, w, keys, margin


def bucket(ids: np.ndarray, E: int = 256):
    ids = _c(ids, np.int32)
    T, K = ids.shape
    counts = np.empty((E,), np.int32)
    offsets = np.empty((E + 1,), np.int32)
    perm = np.empty((T * K,), np.int32)
    inv = np.empty((T * K,), np.int32)
    rc = lib().oracle_bucket(_p(ids), T, K, E, _p(counts), _p(offsets), _p(perm), _p(inv))
    if rc:
        raise ValueError(f"oracle_bucket rc={rc}")
    return counts, offsets, perm, inv


def rmsnorm(x: np.ndarray, eps: float = 1e-6):
    x = _c(x, np.float32)
    y = np.empty_like(x)
    lib().oracle_rmsnorm(_p(x), x.shape[0], x.shape[1], eps, _p(y))
    return y


def _ptr_array(mats):
    arr = (C.c_void_p * len(mats))()
    for i, m in enumerate(mats):
        arr[i] = None if m is None else m.ctypes.data
    return arr


def moe_forward(hidden, ids, w, gate, up, down, sh_gate, sh_up, sh_down, grid,
                gate_up_type=IQ2_XXS, down_type=Q2_K, F=None, nthreads=0):
    """gate/up/down: lists of E GGUF-byte arrays (or None for unused experts);
    sh_*: uint16 bf16 bits arrays; returns out [T,H] f32."""
    hidden = _c(hidden, np.float32)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    T, H = hidden.shape
    K = ids.shape[1]
    E = len(gate)
    F = F if F is not None else sh_gate.shape[0]
    keep = [None if m is None else _c(m, np.uint8) for m in gate + up + down]
    ga, ua, da = (_ptr_array(keep[0:E]), _ptr_array(keep[E:2 * E]), _ptr_array(keep[2 * E:]))
    shg, shu, shd = (_c(a, np.uint16) for a in (sh_gate, sh_up, sh_down))
    g = None if grid is None else _c(grid, np.uint8)
    out = np.empty((T, H), np.float32)
    rc = lib().oracle_moe_forward(_p(hidden), T, H, F, E, K, gate_up_type, down_type, ga, ua, da,
                                  _p(shg), _p(shu), _p(shd), _p(g), _p(ids), _p(w), _p(out),
                                  nthreads)
    if rc:
        raise ValueError(f"oracle_moe_forward rc={rc}")
    return out


def quantize_q8(x: np.ndarray):
    """q8 activations of one row (blocks of 256): (int8 q [n], f32 d [n/256])."""
    x = _c(x, np.float32).reshape(-1)
    q = np.empty(x.size, np.int8)
    d = np.empty(x.size // 256, np.float32)
    if lib().oracle_quantize_q8(_p(x), x.size, _p(q), _p(d)):
        raise ValueError("oracle_quantize_q8: n must be a positive multiple of 256")
    return q, d


def moe_forward_q8(hidden, ids, w, gate, up, down, sh_gate, sh_up, sh_down, grid,
                   gate_up_type=IQ2_XXS, down_type=Q2_K, F=None, nthreads=0):
    """moe_forward with the routed IQ2_XXS gate/up on q8 activations."""
    hidden = _c(hidden, np.float32)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    T, H = hidden.shape
    K = ids.shape[1]
    E = len(gate)
    F = F if F is not None else sh_gate.shape[0]
    keep = [None if m is None else _c(m, np.uint8) for m in gate + up + down]
    ga, ua, da = (_ptr_array(keep[0:E]), _ptr_array(keep[E:2 * E]), _ptr_array(keep[2 * E:]))
    shg, shu, shd = (_c(a, np.uint16) for a in (sh_gate, sh_up, sh_down))
    g = _c(grid, np.uint8)
    out = np.empty((T, H), np.float32)
    rc = lib().oracle_moe_forward_q8(_p(hidden), T, H, F, E, K, gate_up_type, down_type, ga, ua, da,
                                     _p(shg), _p(shu), _p(shd), _p(g), _p(ids), _p(w), _p(out), nthreads)
    if rc:
        raise ValueError(f"oracle_moe_forward_q8 rc={rc}")
    return out


def expert_mlp(x, G, U, D, grid, H, F, gate_up_type=IQ2_XXS, down_type=Q2_K, nthreads=0):
    """One expert on one token: fp64 [H]."""
    x = _c(x, np.float32)
    y = np.empty((H,), np.float64)
    Gc, Uc, Dc = (_c(a, np.uint8 if a.dtype != np.uint16 else np.uint16) for a in (G, U, D))
    g = None if grid is None else _c(grid, np.uint8)
    rc = lib().oracle_expert_mlp(_p(x), H, F, gate_up_type, down_type, _p(Gc), _p(Uc), _p(Dc),
                                 _p(g), _p(y), nthreads)
    if rc:
        raise ValueError(f"oracle_expert_mlp rc={rc}")
    return y
