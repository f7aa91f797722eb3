"""Shared test helpers: building device layers from the seeded generator and
comparing GPU results with the oracle (tolerances from the statement of the
block: fp32-accumulate paths within max-abs 2e-3 * max|ref|)."""
from __future__ import annotations

import numpy as np

import synth

H, F, E, K = 4096, 2048, 256, 6
FWD_TOL = 2e-3       # max-abs error / max|ref| for fp32-accumulate outputs
ROUTE_MARGIN = 1e-5  # tokens closer than this to a routing flip may differ
W_TOL = 1e-6


def grid_u64(seed=0):
    g = synth.iq2_grid(seed)
    return g, np.ascontiguousarray(g).view("<u8").reshape(256)


def host_experts(seed, cfg, layer, experts, gut=synth.IQ2_XXS, dt=synth.Q2_K):
    """GGUF bytes per expert id: {e: (gate, up, down)}."""
    return {int(e): synth.expert(seed, cfg, layer, int(e), gut, dt) for e in experts}


def device_layer(seed, cfg, layer, experts, gut=synth.IQ2_XXS, dt=synth.Q2_K, device="cuda"):
    """Packs the listed experts on the host, uploads them and returns
    (MoELayer, host GGUF dict, shared bf16 triple, grid uint8)."""
    import torch
    import bit_quantized_moe_bias_b300 as B
    experts = sorted(set(int(e) for e in experts))
    hx = host_experts(seed, cfg, layer, experts, gut, dt)
    pk = {k: [] for k in ("g", "u", "d")}
    for e in experts:
        g, u, d = hx[e]
        pk["g"].append(B.ds4g_quantize_pack(gut, F, H, g))
        pk["u"].append(B.ds4g_quantize_pack(gut, F, H, u))
        pk["d"].append(B.ds4g_quantize_pack(dt, H, F, d))
    dev = {k: torch.from_numpy(np.stack(v)).to(device) for k, v in pk.items()}
    shg, shu, shd = synth.shared(seed, cfg, layer)
    sh = [torch.from_numpy(a.view(np.int16)).to(device) for a in (shg, shu, shd)]
    grid, g64 = grid_u64(seed)
    gridt = torch.from_numpy(g64.view(np.int64)).to(device)
    L = B.MoELayer(dev["g"], dev["u"], dev["d"], *sh, gridt, gut, dt, expert_ids=experts)
    return L, hx, (shg, shu, shd), grid


def oracle_forward(x, ids, w, hx, shared, grid, gut=synth.IQ2_XXS, dt=synth.Q2_K, nthreads=0):
    import oracle
    gate, up, down = [None] * E, [None] * E, [None] * E
    for e, (g, u, d) in hx.items():
        gate[e], up[e], down[e] = g, u, d
    return oracle.moe_forward(x, ids, w, gate, up, down, *shared, grid, gut, dt, nthreads=nthreads)


def assert_close_fwd(got, ref, tol=FWD_TOL):
    err = float(np.max(np.abs(got.astype(np.float64) - ref.astype(np.float64))))
    scale = float(np.max(np.abs(ref)))
    assert np.all(np.isfinite(got)), "non-finite output"
    assert err <= tol * scale, f"max-abs err {err:.3e} > {tol} * {scale:.3e}"
    return err / scale


def check_route(ids_gpu, w_gpu, ids_ref, w_ref, keys, margin):
    """ids bit-exact where the oracle margin exceeds ROUTE_MARGIN; elsewhere the
    GPU set must be a valid top-6 within that slack.  Returns #near-ties."""
    near = 0
    for t in range(ids_ref.shape[0]):
        if margin[t] > ROUTE_MARGIN:
            assert list(ids_gpu[t]) == list(ids_ref[t]), f"token {t}: {ids_gpu[t]} vs {ids_ref[t]}"
            assert np.max(np.abs(w_gpu[t] - w_ref[t])) <= W_TOL, f"token {t} weights"
        else:
            near += 1
            kth = np.sort(keys[t])[::-1][K - 1]
            assert len(set(ids_gpu[t].tolist())) == K
            assert np.all(keys[t][ids_gpu[t]] >= kth - ROUTE_MARGIN)
        assert abs(float(w_gpu[t].sum()) - 1.0) <= 1e-5
    return near


class FullLayer:
    """All 256 experts of one layer, generated and packed on the device with
    the seeded generator's CUDA twin (host bytes regenerated on demand)."""

    def __init__(self, seed, cfg, layer, gut=synth.IQ2_XXS, dt=synth.Q2_K, device="cuda"):
        import torch
        import bit_quantized_moe_bias_b300 as B
        self.seed, self.cfg, self.lay, self.gut, self.dt = seed, cfg, layer, gut, dt
        sizes = {gut: B.ds4g_packed_size(gut, F, H), dt: B.ds4g_packed_size(dt, H, F)}
        tmp = torch.empty(max(sizes.values()), dtype=torch.uint8, device=device)
        mats = {}
        st = torch.cuda.current_stream().cuda_stream
        for kind, qt, rows, cols in ((synth.KIND_GATE, gut, F, H), (synth.KIND_UP, gut, F, H),
                                     (synth.KIND_DOWN, dt, H, F)):
            t = torch.empty(E, sizes[qt], dtype=torch.uint8, device=device)
            for e in range(E):
                synth.gguf_matrix_device(qt, rows, cols, seed, synth.stream_id(cfg, layer, kind, e), tmp.data_ptr(), st)
                B.ds4g_quantize_pack_device(qt, rows, cols, tmp, t[e])
            mats[kind] = t
        self.shared = synth.shared(seed, cfg, layer)
        sh = [torch.from_numpy(a.view(np.int16)).to(device) for a in self.shared]
        self.grid, g64 = grid_u64(seed)
        gridt = torch.from_numpy(g64.view(np.int64)).to(device)
        self.L = B.MoELayer(mats[synth.KIND_GATE], mats[synth.KIND_UP], mats[synth.KIND_DOWN], *sh, gridt, gut, dt)
        torch.cuda.synchronize()

    def oracle(self, x, ids, w):
        import oracle
        gate, up, down = [None] * E, [None] * E, [None] * E
        for e in sorted(set(int(v) for v in ids.reshape(-1))):
            gate[e], up[e], down[e] = synth.expert(self.seed, self.cfg, self.lay, e, self.gut, self.dt)
        return oracle.moe_forward(x, ids, w, gate, up, down, *self.shared, self.grid, self.gut, self.dt)


def oracle_forward_q8(x, ids, w, hx, shared, grid, gut=synth.IQ2_XXS, dt=synth.Q2_K, nthreads=0):
    """The oracle's q8 mode (routed IQ2_XXS gate/up on int8 activations)."""
    import oracle
    gate, up, down = [None] * E, [None] * E, [None] * E
    for e, (g, u, d) in hx.items():
        gate[e], up[e], down[e] = g, u, d
    return oracle.moe_forward_q8(x, ids, w, gate, up, down, *shared, grid, gut, dt, nthreads=nthreads)
