"""Python binding of libds4g.so — the B300 routed-MoE block of DeepSeek V4
Flash with 2-bit experts (IQ2_XXS gate/up, Q2_K down; Q4_K for q4 layers).

Argument marshalling only: every step of the block runs in the library's
CUDA kernels.  Function names match the C ABI in include/ds4g.h; device
buffers are torch tensors (``data_ptr()``), streams default to torch's current
stream.  There is no fallback: if libds4g.so is missing or a call fails, an
exception is raised.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libds4g.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "ds4g.h")

DS4G_IQ2_XXS, DS4G_Q2_K, DS4G_Q4_K, DS4G_BF16 = 0, 1, 2, 3
N_EMBD, N_FF_EXP, N_EXPERT, N_EXPERT_USED = 4096, 2048, 256, 6
STATUS = {0: "DS4G_OK", 1: "DS4G_EINVAL", 2: "DS4G_EALIGN", 3: "DS4G_ENOSPACE", 4: "DS4G_ECUDA",
          5: "DS4G_EUNSUPPORTED", 6: "DS4G_ETIMEOUT", 7: "DS4G_EDEVICE"}


class DS4GError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code


class ds4g_layer(C.Structure):
    _fields_ = [("gate_up_type", C.c_int), ("down_type", C.c_int), ("gate", C.c_void_p),
                ("up", C.c_void_p), ("down", C.c_void_p), ("sh_gate", C.c_void_p),
                ("sh_up", C.c_void_p), ("sh_down", C.c_void_p), ("iq2_grid", C.c_void_p)]


class ds4g_host_experts(C.Structure):
    _fields_ = [("gate_up_type", C.c_int), ("down_type", C.c_int), ("gate", C.c_void_p),
                ("up", C.c_void_p), ("down", C.c_void_p)]


_lib = None


def lib():
    """Load libds4g.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_SO):
            raise RuntimeError(f"{_SO} is not built; run bit_quantized_moe_bias_b300/build.py")
        L = C.CDLL(_SO)
        vp, i, sz = C.c_void_p, C.c_int, C.c_size_t
        fwd = [vp, i, C.POINTER(ds4g_layer), vp, vp, vp, vp, sz, vp]
        sig = {
            "ds4g_status_str": ([i], C.c_char_p),
            "ds4g_block_bytes": ([i], sz),
            "ds4g_packed_size": ([i, i, i], sz),
            "ds4g_quantize_pack": ([i, i, i, vp, sz, vp, sz], i),
            "ds4g_unpack": ([i, i, i, vp, sz, vp, sz], i),
            "ds4g_quantize_pack_device": ([i, i, i, vp, vp, vp], i),
            "ds4g_dequantize": ([i, vp, i, i, vp, vp, vp, vp], i),
            "ds4g_route_workspace": ([i], sz),
            "ds4g_moe_route": ([vp, i, vp, vp, vp, vp, vp, sz, vp], i),
            "ds4g_bucket_workspace": ([i], sz),
            "ds4g_moe_bucket": ([vp, i, vp, vp, vp, vp, vp, sz, vp], i),
            "ds4g_forward_workspace": ([i], sz),
            "ds4g_moe_forward": (fwd, i),
            "ds4g_moe_forward_q8": (fwd, i),
            "ds4g_moe_gate_up": (fwd, i),
            "ds4g_moe_down": (fwd, i),
            "ds4g_layer_decode_workspace": ([], sz),
            "ds4g_decode_stack_workspace": ([], sz),
            "ds4g_moe_layer_decode": ([vp, i, vp, vp, C.POINTER(ds4g_layer), vp, vp, vp, vp, sz, vp], i),
            "ds4g_moe_decode_stack": ([vp, i, C.POINTER(vp), C.POINTER(vp), C.POINTER(ds4g_layer), vp, vp, vp, vp,
                                       vp, sz, vp], i),
            "ds4g_moe_forward_noalloc": ([vp, i, C.POINTER(ds4g_layer), vp, vp, vp, vp], i),
            "ds4g_test_force_timeout": ([i], None),
            "ds4g_expert_cache_pool_bytes": ([i, i, i], sz),
            "ds4g_expert_cache_create": ([i, i, i, i, vp, sz, C.POINTER(vp)], i),
            "ds4g_expert_cache_destroy": ([vp], i),
            "ds4g_expert_cache_stats": ([vp, C.POINTER(C.c_uint64), C.POINTER(C.c_uint64),
                                         C.POINTER(C.c_uint64)], i),
            "ds4g_moe_forward_streamed": ([vp, i, i, C.POINTER(ds4g_host_experts), vp, vp, vp, vp, vp, vp, vp, vp,
                                           vp, sz, vp], i),
            "ds4g_expert_lru_simulate": ([i, i, vp, vp, vp, vp], i),
            "ds4g_expert_file_write": ([C.c_char_p, C.POINTER(ds4g_host_experts)], i),
            "ds4g_expert_file_open": ([C.c_char_p, C.POINTER(vp)], i),
            "ds4g_expert_file_close": ([vp], i),
            "ds4g_moe_forward_streamed_file": ([vp, i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i),
            "ds4g_rmsnorm": ([vp, i, vp, vp], i),
            "ds4g_last_error": ([vp, vp], i),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions declared in include/ds4g.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(ds4g_[a-z_0-9]+)\s*\(", text)))


def _check(fn: str, rc: int):
    if rc != 0:
        raise DS4GError(fn, rc)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def ds4g_status_str(code: int) -> str:
    return lib().ds4g_status_str(code).decode()


def ds4g_block_bytes(qtype: int) -> int:
    return lib().ds4g_block_bytes(qtype)


def ds4g_packed_size(qtype: int, rows: int, cols: int) -> int:
    return lib().ds4g_packed_size(qtype, rows, cols)


def ds4g_quantize_pack(qtype: int, rows: int, cols: int, gguf: np.ndarray) -> np.ndarray:
    """Host: GGUF-format bytes -> packed device-layout bytes (numpy uint8)."""
    gguf = np.ascontiguousarray(gguf, np.uint8)
    n = ds4g_packed_size(qtype, rows, cols)
    out = np.empty(max(n, 1), np.uint8)
    _check("ds4g_quantize_pack", lib().ds4g_quantize_pack(qtype, rows, cols, _ptr(gguf), gguf.nbytes,
                                                          _ptr(out), out.nbytes))
    return out[:n]


def ds4g_unpack(qtype: int, rows: int, cols: int, packed: np.ndarray) -> np.ndarray:
    packed = np.ascontiguousarray(packed, np.uint8)
    n = ds4g_packed_size(qtype, rows, cols)
    out = np.empty(max(n, 1), np.uint8)
    _check("ds4g_unpack", lib().ds4g_unpack(qtype, rows, cols, _ptr(packed), packed.nbytes, _ptr(out),
                                            out.nbytes))
    return out[:n]


def ds4g_quantize_pack_device(qtype, rows, cols, gguf_dev, packed_dev, stream=None):
    _check("ds4g_quantize_pack_device",
           lib().ds4g_quantize_pack_device(qtype, rows, cols, _ptr(gguf_dev), _ptr(packed_dev),
                                           _stream(stream)))


def ds4g_dequantize(qtype, packed_dev, rows, cols, grid_dev=None, out_f32=None, out_bf16=None, stream=None):
    _check("ds4g_dequantize", lib().ds4g_dequantize(qtype, _ptr(packed_dev), rows, cols, _ptr(grid_dev),
                                                    _ptr(out_f32), _ptr(out_bf16), _stream(stream)))


def ds4g_route_workspace(T: int) -> int:
    return lib().ds4g_route_workspace(T)


def ds4g_moe_route(hidden, router, bias, ids, w, workspace, stream=None):
    T = hidden.shape[0]
    _check("ds4g_moe_route", lib().ds4g_moe_route(_ptr(hidden), T, _ptr(router), _ptr(bias), _ptr(ids),
                                                  _ptr(w), _ptr(workspace), workspace.numel(),
                                                  _stream(stream)))


def ds4g_bucket_workspace(T: int) -> int:
    return lib().ds4g_bucket_workspace(T)


def ds4g_moe_bucket(ids, counts, offsets, perm, inv, workspace, stream=None):
    T = ids.shape[0]
    _check("ds4g_moe_bucket", lib().ds4g_moe_bucket(_ptr(ids), T, _ptr(counts), _ptr(offsets), _ptr(perm),
                                                    _ptr(inv), _ptr(workspace), workspace.numel(),
                                                    _stream(stream)))


def ds4g_forward_workspace(T: int) -> int:
    return lib().ds4g_forward_workspace(T)


def _fwd(name, hidden, layer, ids, w, out, workspace, stream):
    T = hidden.shape[0]
    _check(name, getattr(lib(), name)(_ptr(hidden), T, C.byref(layer), _ptr(ids), _ptr(w), _ptr(out),
                                      _ptr(workspace), workspace.numel(), _stream(stream)))


def ds4g_moe_forward(hidden, layer: ds4g_layer, ids, w, out, workspace, stream=None):
    _fwd("ds4g_moe_forward", hidden, layer, ids, w, out, workspace, stream)


def ds4g_moe_forward_q8(hidden, layer: ds4g_layer, ids, w, out, workspace, stream=None):
    """ds4g_moe_forward (T <= 3) with the routed IQ2_XXS gate/up on int8 activations."""
    _fwd("ds4g_moe_forward_q8", hidden, layer, ids, w, out, workspace, stream)


def ds4g_moe_gate_up(hidden, layer: ds4g_layer, ids, w, out, workspace, stream=None):
    _fwd("ds4g_moe_gate_up", hidden, layer, ids, w, out, workspace, stream)


def ds4g_moe_down(hidden, layer: ds4g_layer, ids, w, out, workspace, stream=None):
    _fwd("ds4g_moe_down", hidden, layer, ids, w, out, workspace, stream)


def ds4g_layer_decode_workspace() -> int:
    return lib().ds4g_layer_decode_workspace()


def ds4g_decode_stack_workspace() -> int:
    return lib().ds4g_decode_stack_workspace()


def ds4g_moe_layer_decode(hidden, router, bias, layer: ds4g_layer, ids, w, out, workspace, normalize=True,
                          stream=None):
    """rmsnorm (optional) + route + forward of one token in one launch."""
    _check("ds4g_moe_layer_decode",
           lib().ds4g_moe_layer_decode(_ptr(hidden), 1 if normalize else 0, _ptr(router), _ptr(bias), C.byref(layer),
                                       _ptr(ids), _ptr(w), _ptr(out), _ptr(workspace), workspace.numel(),
                                       _stream(stream)))


class DecodeStack:
    """Marshalled arguments of ds4g_moe_decode_stack for a fixed list of
    layers: (ds4g_layer struct, router tensor, bias tensor) per layer."""

    def __init__(self, layers):
        n = len(layers)
        self.n = n
        self.structs = (ds4g_layer * n)(*[l[0] for l in layers])
        self.routers = (C.c_void_p * n)(*[_ptr(l[1]) for l in layers])
        self.biases = (C.c_void_p * n)(*[_ptr(l[2]) for l in layers])
        self.keep = layers


def ds4g_moe_decode_stack(hidden, stack: DecodeStack, ids, w, hbuf, out, workspace, stream=None):
    """One token through stack.n chained layers (IQ2_XXS/Q2_K layers fused,
    programmatic dependent launches between them; Q4_K layers as rmsnorm +
    route + forward); ids, w: [n][6]; hbuf: [2][4096] scratch."""
    _check("ds4g_moe_decode_stack",
           lib().ds4g_moe_decode_stack(_ptr(hidden), stack.n, stack.routers, stack.biases, stack.structs, _ptr(ids),
                                       _ptr(w), _ptr(hbuf), _ptr(out), _ptr(workspace), workspace.numel(),
                                       _stream(stream)))


def ds4g_moe_forward_noalloc(hidden, layer: ds4g_layer, ids, w, out, stream=None):
    """ds4g_moe_forward with the library's own static scratch (no workspace)."""
    T = hidden.shape[0]
    _check("ds4g_moe_forward_noalloc",
           lib().ds4g_moe_forward_noalloc(_ptr(hidden), T, C.byref(layer), _ptr(ids), _ptr(w), _ptr(out),
                                          _stream(stream)))


def ds4g_test_force_timeout(on: bool):
    """Test hook: while on, fused layer launches wait for logits that never
    arrive and give up after ~130 us with DS4G_ETIMEOUT."""
    lib().ds4g_test_force_timeout(1 if on else 0)


class HostExperts:
    """Routed experts of one layer in host memory for ds4g_moe_forward_streamed:
    gate/up/down map expert id -> packed bytes (uint8 tensors or arrays in
    pinned host memory); missing ids are NULL."""

    def __init__(self, gate, up, down, gate_up_type=DS4G_IQ2_XXS, down_type=DS4G_Q2_K):
        self.keep = (gate, up, down)
        tabs = []
        for m in (gate, up, down):
            arr = (C.c_void_p * N_EXPERT)()
            for e, t in m.items():
                arr[int(e)] = _ptr(t)
            tabs.append(arr)
        self.tabs = tabs
        self.struct = ds4g_host_experts(gate_up_type, down_type, C.cast(tabs[0], C.c_void_p).value,
                                        C.cast(tabs[1], C.c_void_p).value, C.cast(tabs[2], C.c_void_p).value)


class ExpertCache:
    """An HBM expert cache of n_slots slots (pool allocated here as a torch
    tensor) for ds4g_moe_forward_streamed."""

    def __init__(self, n_slots, max_tokens=1, gate_up_type=DS4G_IQ2_XXS, down_type=DS4G_Q2_K, device="cuda"):
        import torch
        nbytes = lib().ds4g_expert_cache_pool_bytes(gate_up_type, down_type, n_slots)
        if nbytes == 0:
            raise DS4GError("ds4g_expert_cache_pool_bytes", 1)
        self.pool = torch.empty(nbytes, dtype=torch.uint8, device=device)
        h = C.c_void_p()
        _check("ds4g_expert_cache_create",
               lib().ds4g_expert_cache_create(gate_up_type, down_type, n_slots, max_tokens, self.pool.data_ptr(),
                                              nbytes, C.byref(h)))
        self.handle = h

    def stats(self):
        hits, misses, nbytes = C.c_uint64(), C.c_uint64(), C.c_uint64()
        _check("ds4g_expert_cache_stats",
               lib().ds4g_expert_cache_stats(self.handle, C.byref(hits), C.byref(misses), C.byref(nbytes)))
        return hits.value, misses.value, nbytes.value

    def close(self):
        if self.handle is not None and self.handle.value:
            _check("ds4g_expert_cache_destroy", lib().ds4g_expert_cache_destroy(self.handle))
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def ds4g_moe_forward_streamed(hidden, layer_key, src: HostExperts, sh_gate, sh_up, sh_down, grid, ids, w, out,
                              cache: ExpertCache, workspace, stream=None):
    """ds4g_moe_forward whose routed experts are copied on demand from host
    memory into the cache (blocks until the stream drains: ids are read back)."""
    T = hidden.shape[0]
    _check("ds4g_moe_forward_streamed",
           lib().ds4g_moe_forward_streamed(_ptr(hidden), T, layer_key, C.byref(src.struct), _ptr(sh_gate),
                                           _ptr(sh_up), _ptr(sh_down), _ptr(grid), _ptr(ids), _ptr(w), _ptr(out),
                                           cache.handle, _ptr(workspace), workspace.numel(), _stream(stream)))


def ds4g_expert_file_write(path, src: HostExperts):
    """Writes the layer's experts of src (host memory) to an expert file."""
    _check("ds4g_expert_file_write", lib().ds4g_expert_file_write(os.fsencode(path), C.byref(src.struct)))


class ExpertFile:
    """An open expert file (ds4g_expert_file_open) for ds4g_moe_forward_streamed_file."""

    def __init__(self, path):
        h = C.c_void_p()
        _check("ds4g_expert_file_open", lib().ds4g_expert_file_open(os.fsencode(path), C.byref(h)))
        self.handle = h

    def close(self):
        if self.handle is not None and self.handle.value:
            _check("ds4g_expert_file_close", lib().ds4g_expert_file_close(self.handle))
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def ds4g_moe_forward_streamed_file(hidden, layer_key, src: ExpertFile, sh_gate, sh_up, sh_down, grid, ids, w, out,
                                   cache: ExpertCache, workspace, stream=None):
    """ds4g_moe_forward_streamed with the missing experts read from an expert file."""
    T = hidden.shape[0]
    _check("ds4g_moe_forward_streamed_file",
           lib().ds4g_moe_forward_streamed_file(_ptr(hidden), T, layer_key, src.handle, _ptr(sh_gate), _ptr(sh_up),
                                                _ptr(sh_down), _ptr(grid), _ptr(ids), _ptr(w), _ptr(out),
                                                cache.handle, _ptr(workspace), workspace.numel(), _stream(stream)))


def ds4g_expert_lru_simulate(n_slots, calls):
    """The cache's slot policy on the host: calls = list of key lists; returns
    (slots, misses) lists of the same shape."""
    sizes = np.array([len(c) for c in calls], np.int32)
    keys = np.array([k for c in calls for k in c], np.int64)
    slot = np.zeros(len(keys), np.int32)
    miss = np.zeros(len(keys), np.uint8)
    _check("ds4g_expert_lru_simulate",
           lib().ds4g_expert_lru_simulate(n_slots, len(calls), sizes.ctypes.data, keys.ctypes.data,
                                          slot.ctypes.data, miss.ctypes.data))
    out_s, out_m, o = [], [], 0
    for n in sizes:
        out_s.append(slot[o:o + n].tolist())
        out_m.append(miss[o:o + n].astype(bool).tolist())
        o += n
    return out_s, out_m


def ds4g_rmsnorm(x, y, stream=None):
    _check("ds4g_rmsnorm", lib().ds4g_rmsnorm(_ptr(x), x.shape[0], _ptr(y), _stream(stream)))


def ds4g_last_error(workspace, stream=None) -> int:
    return lib().ds4g_last_error(_ptr(workspace), _stream(stream))


# --------------------------------------------------------------- conveniences
def workspace(nbytes: int, device="cuda"):
    """Zero-filled device workspace (the kernels keep their counters at zero
    between calls, so a workspace needs zeroing only once)."""
    import torch
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


class MoELayer:
    """Device-resident weights of one MoE layer and its ds4g_layer struct.

    gate/up/down: one uint8 tensor each of shape [n_experts, packed_bytes]
    (packed layout); ``expert_ids`` maps row i of those tensors to an expert
    id (experts absent from the list get NULL pointers, which the kernels
    reject if selected).  sh_*: bf16-bits 16-bit tensors.  grid: 64-bit [256].
    """

    def __init__(self, gate, up, down, sh_gate, sh_up, sh_down, grid=None,
                 gate_up_type=DS4G_IQ2_XXS, down_type=DS4G_Q2_K, expert_ids=None):
        import torch
        dev = gate.device
        n = gate.shape[0]
        ids = list(range(n)) if expert_ids is None else list(expert_ids)
        self.tensors = (gate, up, down, sh_gate, sh_up, sh_down, grid)
        ptrs = np.zeros((3, N_EXPERT), np.int64)
        for row, e in enumerate(ids):
            ptrs[0, e] = gate[row].data_ptr()
            ptrs[1, e] = up[row].data_ptr()
            ptrs[2, e] = down[row].data_ptr()
        self.ptrs = torch.from_numpy(ptrs).to(dev)
        self.struct = ds4g_layer(gate_up_type, down_type, self.ptrs[0].data_ptr(), self.ptrs[1].data_ptr(),
                                 self.ptrs[2].data_ptr(), sh_gate.data_ptr(), sh_up.data_ptr(),
                                 sh_down.data_ptr(), 0 if grid is None else grid.data_ptr())
