"""CPU-side checks of the C-ABI library: it loads, exports every function the
header declares, packs/unpacks losslessly into the documented layout, and
rejects bad arguments before touching the GPU."""
import ctypes as C
import os

import numpy as np
import pytest

import bit_quantized_moe_bias_b300 as B
import synth


def test_library_exports_every_header_function():
    L = B.lib()
    names = B.header_functions()
    assert len(names) >= 17
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


@pytest.mark.parametrize("qt,bb", [(0, 66), (1, 84), (2, 144), (3, 512)])
def test_block_bytes(qt, bb):
    assert B.ds4g_block_bytes(qt) == bb


def test_packed_size_rules():
    assert B.ds4g_packed_size(0, 2048, 4096) == 2048 * 16 * 66
    assert B.ds4g_packed_size(1, 4096, 2048) == 4096 * 8 * 84
    assert B.ds4g_packed_size(2, 16, 256) == 144 * 16
    assert B.ds4g_packed_size(0, 15, 256) == 0       # rows not a multiple of 16
    assert B.ds4g_packed_size(0, 16, 300) == 0       # cols not a multiple of 256
    assert B.ds4g_packed_size(3, 16, 256) == 0       # bf16 is not packed


@pytest.mark.parametrize("qt", [0, 1, 2])
@pytest.mark.parametrize("rows,cols", [(16, 256), (48, 768), (64, 4096)])
def test_pack_unpack_round_trip(qt, rows, cols):
    g = synth.gguf_matrix(qt, rows, cols, 11, 1000 + rows + qt)
    p = B.ds4g_quantize_pack(qt, rows, cols, g)
    assert p.nbytes == g.nbytes and not np.array_equal(p, g)
    assert np.array_equal(B.ds4g_unpack(qt, rows, cols, p), g)


def test_iq2_layout_matches_documentation():
    """Packed IQ2_XXS: record of GGUF sub-block j of tile row rr sits at
    512*hrow + 16*(4g + t) + 8*jj (g = rr&7, hrow = rr>>3, t = j&3, jj = j>>2);
    d at 1024 + 4g + 2*hrow."""
    g = synth.gguf_matrix(0, 16, 256, 3, 9).reshape(16, 66)
    p = B.ds4g_quantize_pack(0, 16, 256, g.reshape(-1))
    for rr in range(16):
        gg, hrow = rr & 7, rr >> 3
        for j in range(8):
            off = 512 * hrow + 16 * (4 * gg + (j & 3)) + 8 * (j >> 2)
            assert np.array_equal(p[off:off + 8], g[rr, 2 + 8 * j: 10 + 8 * j])
        assert np.array_equal(p[1024 + 4 * gg + 2 * hrow: 1026 + 4 * gg + 2 * hrow], g[rr, 0:2])


def test_q2k_layout_matches_documentation():
    """Packed Q2_K: quant of weight n (sub-block sb = n//16, i = n%16 = 4c+p)
    at bit 16*(p&1) + 2*(2c + (p>>1)) of the word at 512*hrow + 16*(4g+t) + 4G
    (t = sb&3, G = sb>>2); GGUF field of n = 128h + 32jq + l is bits 2jq of
    qs[32h + l]."""
    g = synth.gguf_matrix(1, 16, 256, 4, 10).reshape(16, 84)
    p = B.ds4g_quantize_pack(1, 16, 256, g.reshape(-1))
    words = p.view("<u4")
    for rr in (0, 5, 8, 15):
        gg, hrow = rr & 7, rr >> 3
        for n in range(256):
            h, jq, l = n // 128, (n % 128) // 32, n % 32
            q_ref = (int(g[rr, 16 + 32 * h + l]) >> (2 * jq)) & 3
            sb, i = n // 16, n % 16
            c, pp = i // 4, i % 4
            wi = (512 * hrow + 16 * (4 * gg + (sb & 3)) + 4 * (sb >> 2)) // 4
            q = (int(words[wi]) >> (16 * (pp & 1) + 2 * (2 * c + (pp >> 1)))) & 3
            assert q == q_ref
        for sb in range(16):
            assert p[1024 + 128 * hrow + 4 * (4 * gg + (sb & 3)) + (sb >> 2)] == g[rr, sb]


def test_q4k_layout_matches_documentation():
    """Packed Q4_K: weight n (sub-block j = n//32, i = n%32 = 4c+p) at bit
    16*(p&1) + 4*(2*(c&1) + (p>>1)) of the word at
    1024*hrow + 32*(4g+t) + 4*(4jj + (c>>1)) (t = j&3, jj = j>>2); GGUF: weight
    64c4 + l is the low nibble of qs[32c4 + l], 64c4 + 32 + l the high one."""
    g = synth.gguf_matrix(2, 16, 256, 4, 12).reshape(16, 144)
    p = B.ds4g_quantize_pack(2, 16, 256, g.reshape(-1))
    words = p.view("<u4")
    for rr in (1, 7, 9, 14):
        gg, hrow = rr & 7, rr >> 3
        for n in range(256):
            c4, r = n // 64, n % 64
            q_ref = (int(g[rr, 16 + 32 * c4 + (r % 32)]) >> (0 if r < 32 else 4)) & 15
            j, i = n // 32, n % 32
            c, pp = i // 4, i % 4
            wi = (1024 * hrow + 32 * (4 * gg + (j & 3)) + 4 * (4 * (j >> 2) + (c >> 1))) // 4
            q = (int(words[wi]) >> (16 * (pp & 1) + 4 * (2 * (c & 1) + (pp >> 1)))) & 15
            assert q == q_ref
        assert np.array_equal(p[2048 + 12 * rr: 2060 + 12 * rr], g[rr, 4:16])


def test_pack_rejects_bad_arguments():
    L = B.lib()
    buf = np.zeros(1 << 16, np.uint8)
    ptr = buf.ctypes.data
    assert L.ds4g_quantize_pack(0, 16, 256, None, 0, ptr, buf.nbytes) == 1            # EINVAL
    assert L.ds4g_quantize_pack(7, 16, 256, ptr, buf.nbytes, ptr, buf.nbytes) == 1    # bad type
    assert L.ds4g_quantize_pack(0, 17, 256, ptr, buf.nbytes, ptr, buf.nbytes) == 5    # EUNSUPPORTED
    assert L.ds4g_quantize_pack(0, 16, 256, ptr, 100, ptr, buf.nbytes) == 3           # ENOSPACE
    assert L.ds4g_quantize_pack(0, 16, 256, ptr, buf.nbytes, ptr, 100) == 3


def test_gpu_entry_points_validate_before_launch():
    """Bad arguments come back as status codes without any CUDA call."""
    L = B.lib()
    fake = 0x10000000           # aligned fake device address (never dereferenced)
    odd = fake + 4
    big = 1 << 30
    lay = B.ds4g_layer(0, 1, fake, fake, fake, fake, fake, fake, fake)
    for f in (L.ds4g_moe_forward, L.ds4g_moe_gate_up, L.ds4g_moe_down):
        assert f(None, 1, C.byref(lay), fake, fake, fake, fake, big, None) == 1        # NULL hidden
        assert f(fake, 0, C.byref(lay), fake, fake, fake, fake, big, None) == 1        # T < 1
        assert f(odd, 1, C.byref(lay), fake, fake, fake, fake, big, None) == 2         # misaligned
        assert f(fake, 1, C.byref(lay), fake, fake, fake, fake, 16, None) == 3         # workspace
        bad = B.ds4g_layer(0, 2, fake, fake, fake, fake, fake, fake, fake)             # IQ2 + Q4_K
        assert f(fake, 1, C.byref(bad), fake, fake, fake, fake, big, None) == 5
        nogrid = B.ds4g_layer(0, 1, fake, fake, fake, fake, fake, fake, None)
        assert f(fake, 1, C.byref(nogrid), fake, fake, fake, fake, big, None) == 1
    assert L.ds4g_moe_gate_up(fake, 4, C.byref(lay), fake, fake, fake, fake, big, None) == 5  # phases: T <= 3
    r = L.ds4g_moe_route
    assert r(fake, 1, fake, fake, fake, fake, fake, 8, None) == 3
    assert r(fake, 1, fake, odd, fake, fake, fake, big, None) == 2
    assert r(None, 1, fake, fake, fake, fake, fake, big, None) == 1
    assert L.ds4g_moe_bucket(fake, 0, fake, fake, fake, fake, fake, big, None) == 1
    assert L.ds4g_dequantize(0, fake, 16, 256, None, fake, None, None) == 1           # IQ2 needs grid
    assert L.ds4g_dequantize(1, fake, 16, 300, None, fake, None, None) == 5
    assert L.ds4g_rmsnorm(odd, 1, fake, None) == 2
    assert L.ds4g_quantize_pack_device(1, 16, 256, odd, fake, None) == 2


def test_decode_stack_validates_layer_types_and_workspace():
    """The stack checks every layer before any CUDA call: IQ2_XXS/Q2_K and
    Q4_K layers share the fused kernel's workspace; mixed IQ2/Q4_K types in
    one layer, a misaligned pointer and a missing router are refused."""
    L = B.lib()
    fake = 0x10000000
    q2 = B.ds4g_layer(0, 1, fake, fake, fake, fake, fake, fake, fake)
    q4 = B.ds4g_layer(2, 2, fake, fake, fake, fake, fake, fake, None)   # Q4_K layers need no grid
    mix = B.ds4g_layer(0, 2, fake, fake, fake, fake, fake, fake, fake)
    q4_odd = B.ds4g_layer(2, 2, fake, fake, fake, fake + 8, fake, fake, None)
    q2_nogrid = B.ds4g_layer(0, 1, fake, fake, fake, fake, fake, fake, None)
    ws = B.ds4g_decode_stack_workspace()
    assert ws == B.ds4g_layer_decode_workspace()

    def stack(layers, ws_bytes, routers=True):
        n = len(layers)
        structs = (B.ds4g_layer * n)(*layers)
        ptrs = (C.c_void_p * n)(*([fake] * n))
        return L.ds4g_moe_decode_stack(fake, n, ptrs if routers else None, ptrs, structs, fake, fake, fake, fake,
                                       fake, ws_bytes, None)

    assert stack([q2, q4], ws - 1) == 3
    assert stack([q2, mix], ws) == 5
    assert stack([q4_odd], ws) == 2
    assert stack([q2_nogrid], ws) == 1
    assert stack([q2, q4], ws, routers=False) == 1


def test_workspace_sizes_grow_with_T():
    """A workspace sized for T tokens serves every call with 1..T tokens: both
    size queries are non-decreasing in T, across the paths' boundaries (per-slot
    decode / batched / prefill for the forward; small / mid / tiled router)."""
    assert B.ds4g_route_workspace(0) == 0
    assert B.ds4g_route_workspace(1) < B.ds4g_route_workspace(2048)
    assert 0 < B.ds4g_forward_workspace(1) <= B.ds4g_forward_workspace(3)
    assert B.ds4g_bucket_workspace(1) >= 256
    L = B.lib()
    Ts = list(range(1, 140)) + [255, 256, 1000, 2048, 4096, 16383, 16384, 16385, 20000, 65536, 65537]
    for f in (L.ds4g_forward_workspace, L.ds4g_route_workspace):
        sizes = [f(T) for T in Ts]
        assert all(b >= a for a, b in zip(sizes, sizes[1:])), f


def test_status_strings():
    assert B.ds4g_status_str(0) == "ok"
    assert "bad data" in B.ds4g_status_str(7)


def test_expert_file_layout_and_header_checks(tmp_path):
    """ds4g_expert_file_write stores the documented layout (no GPU needed);
    ds4g_expert_file_open refuses a bad header before any CUDA call."""
    import struct
    gate = {3: np.arange(B.ds4g_packed_size(0, 2048, 4096), dtype=np.uint64).astype(np.uint8)}
    up = {3: np.full(B.ds4g_packed_size(0, 2048, 4096), 7, np.uint8)}
    down = {3: np.full(B.ds4g_packed_size(1, 4096, 2048), 9, np.uint8)}
    src = B.HostExperts(gate, up, down, 0, 1)
    path = tmp_path / "e.ds4gexp"
    B.ds4g_expert_file_write(path, src)
    raw = path.read_bytes()
    magic, gut, dt, n, zero, gb, db, stride = struct.unpack_from("<8sIIIIQQQ", raw, 0)
    assert (magic, gut, dt, n, zero) == (b"DS4GEXP1", 0, 1, 256, 0)
    assert gb == B.ds4g_packed_size(0, 2048, 4096) and db == B.ds4g_packed_size(1, 4096, 2048)
    assert stride % 4096 == 0 and stride >= 2 * gb + db
    bitmap = raw[48:80]
    assert bitmap[0] == 1 << 3 and not any(bitmap[1:])
    assert len(raw) == 4096 + 256 * stride
    base = 4096 + 3 * stride
    assert raw[base:base + gb] == gate[3].tobytes()
    assert raw[base + gb:base + 2 * gb] == up[3].tobytes()
    assert raw[base + 2 * gb:base + 2 * gb + db] == down[3].tobytes()
    # a partial expert is refused
    with pytest.raises(B.DS4GError) as e:
        B.ds4g_expert_file_write(tmp_path / "p.ds4gexp", B.HostExperts(gate, up, {}, 0, 1))
    assert e.value.code == 1
    # headers that open must refuse before any CUDA call
    L = B.lib()
    h = C.c_void_p()
    bad = bytearray(raw[:4096])
    bad[0:8] = b"XXXXXXXX"
    (tmp_path / "bad.ds4gexp").write_bytes(bytes(bad))
    assert L.ds4g_expert_file_open(os.fsencode(tmp_path / "bad.ds4gexp"), C.byref(h)) == 1
    (tmp_path / "short.ds4gexp").write_bytes(raw[:4096 + stride])   # truncated
    assert L.ds4g_expert_file_open(os.fsencode(tmp_path / "short.ds4gexp"), C.byref(h)) == 1
    assert L.ds4g_expert_file_open(os.fsencode(tmp_path / "none.ds4gexp"), C.byref(h)) == 1

