"""Streamed forward (routed experts in pinned host memory, an HBM expert
cache): bit-identical to the resident forward on the same experts, hit and
miss counts as the cache's policy predicts, refusal when a call needs more
experts than slots, and oracle parity."""
import numpy as np
import pytest

import oracle
import synth
from helpers import F, H, K, assert_close_fwd, device_layer, oracle_forward

torch = pytest.importorskip("torch")
import bit_quantized_moe_bias_b300 as B  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _host_experts(hx, experts, gut, dt):
    packed = {k: {} for k in "gud"}
    for e in experts:
        g, u, d = hx[e]
        packed["g"][e] = torch.from_numpy(B.ds4g_quantize_pack(gut, F, H, g)).pin_memory()
        packed["u"][e] = torch.from_numpy(B.ds4g_quantize_pack(gut, F, H, u)).pin_memory()
        packed["d"][e] = torch.from_numpy(B.ds4g_quantize_pack(dt, H, F, d)).pin_memory()
    return B.HostExperts(packed["g"], packed["u"], packed["d"], gut, dt)


def _run_both(x, ids, w, L, src, cache, layer_key, ws):
    T = x.shape[0]
    xd, idd, wd = (torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in (x, ids, w))
    out_s = torch.full((T, H), float("nan"), device=DEV)
    out_r = torch.full((T, H), float("nan"), device=DEV)
    sg, su, sd, grid = L.tensors[3], L.tensors[4], L.tensors[5], L.tensors[6]
    B.ds4g_moe_forward_streamed(xd, layer_key, src, sg, su, sd, grid, idd, wd, out_s, cache, ws)
    assert B.ds4g_last_error(ws) == 0
    B.ds4g_moe_forward(xd, L.struct, idd, wd, out_r, ws)
    assert B.ds4g_last_error(ws) == 0
    return out_s.cpu().numpy(), out_r.cpu().numpy()


@pytest.mark.parametrize("gut,dt", [(synth.IQ2_XXS, synth.Q2_K), (synth.Q4_K, synth.Q4_K)])
def test_streamed_equals_resident_and_policy(gut, dt):
    seed, cfg, lay = 3, 1, 2
    experts = [3, 17, 40, 41, 77, 90, 128, 200, 201, 255]
    L, hx, shared, grid = device_layer(seed, cfg, lay, experts, gut, dt)
    src = _host_experts(hx, experts, gut, dt)
    cache = B.ExpertCache(8, max_tokens=2, gate_up_type=gut, down_type=dt)
    ws = B.workspace(B.ds4g_forward_workspace(2))
    rng = np.random.default_rng(1)
    calls = [[3, 17, 40, 41, 77, 90], [3, 17, 128, 200, 201, 255], [40, 41, 77, 90, 3, 17],
             [255, 255, 3, 3, 17, 17], [[200, 201, 3, 17, 40, 41], [3, 17, 40, 41, 200, 201]]]
    keys_per_call = []
    for c in calls:
        ids = np.array(c if isinstance(c[0], list) else [c], np.int32)
        T = ids.shape[0]
        x = synth.hidden(seed, cfg, T, layer=50 + len(keys_per_call))
        w = rng.dirichlet(np.ones(K), T).astype(np.float32)
        got, ref = _run_both(x, ids, w, L, src, cache, lay, ws)
        assert np.array_equal(got, ref)      # same kernels, experts read from the cache's slots
        keys_per_call.append([lay * 256 + int(e) for e in ids.reshape(-1)])
    slots, miss = B.ds4g_expert_lru_simulate(8, keys_per_call)
    n_miss = sum(sum(m) for m in miss)
    n_hit = sum(len(set(k)) for k in keys_per_call) - n_miss
    hits, misses, nbytes = cache.stats()
    assert (hits, misses) == (n_hit, n_miss)
    per = 2 * B.ds4g_packed_size(gut, F, H) + B.ds4g_packed_size(dt, H, F)
    assert nbytes == n_miss * per
    # the last call against the oracle
    ids = np.array(calls[-1], np.int32)
    x = synth.hidden(seed, cfg, 2, layer=60)
    w = np.full((2, K), 1.0 / K, np.float32)
    got, _ = _run_both(x, ids, w, L, src, cache, lay, ws)
    assert_close_fwd(got, oracle_forward(x, ids, w, hx, shared, grid, gut, dt))
    cache.close()


def test_streamed_refusals_and_recovery():
    seed, cfg, lay = 4, 1, 0
    experts = list(range(12))
    L, hx, shared, grid = device_layer(seed, cfg, lay, experts)
    src = _host_experts(hx, experts[:11], synth.IQ2_XXS, synth.Q2_K)     # expert 11 not provided
    cache = B.ExpertCache(8, max_tokens=2)
    ws = B.workspace(B.ds4g_forward_workspace(2))
    x = synth.hidden(seed, cfg, 2, layer=70)
    w = np.full((2, K), 1.0 / K, np.float32)
    # nine distinct experts for eight slots: refused
    with pytest.raises(B.DS4GError) as e:
        _run_both(x, np.array([[0, 1, 2, 3, 4, 5], [6, 7, 8, 0, 1, 2]], np.int32), w, L, src, cache, lay, ws)
    assert e.value.code == 3
    # an expert with no host copy: refused
    with pytest.raises(B.DS4GError) as e:
        _run_both(x[:1], np.array([[0, 1, 2, 3, 4, 11]], np.int32), w[:1], L, src, cache, lay, ws)
    assert e.value.code == 1
    # more tokens than the cache was made for
    with pytest.raises(B.DS4GError) as e:
        _run_both(synth.hidden(seed, cfg, 3, layer=71), np.zeros((3, K), np.int32), np.full((3, K), 1 / 6, np.float32),
                  L, src, cache, lay, ws)
    assert e.value.code == 1
    # the cache still serves correct results afterwards
    got, ref = _run_both(x, np.array([[0, 1, 2, 3, 4, 5], [5, 6, 7, 0, 1, 2]], np.int32), w, L, src, cache, lay,
                         ws)
    assert np.array_equal(got, ref)
    # an id outside [0, 256) reaches the kernels, which flag it
    xd = torch.from_numpy(x[:1]).to(DEV)
    bad = torch.tensor([[0, 1, 2, 3, 4, 999]], dtype=torch.int32, device=DEV)
    wd = torch.from_numpy(w[:1]).to(DEV)
    out = torch.empty(1, H, device=DEV)
    sg, su, sd, gr = L.tensors[3], L.tensors[4], L.tensors[5], L.tensors[6]
    B.ds4g_moe_forward_streamed(xd, lay, src, sg, su, sd, gr, bad, wd, out, cache, ws)
    assert B.ds4g_last_error(ws) == 7
    cache.close()


@pytest.mark.parametrize("gut,dt", [(synth.IQ2_XXS, synth.Q2_K), (synth.Q4_K, synth.Q4_K)])
def test_streamed_from_file_equals_host_and_resident(gut, dt, tmp_path):
    """Experts read from an expert file (pread into pinned staging, then
    copied): bit-identical to the host-memory source and to the resident
    forward, the same hit/miss counts, and an expert absent from the file is
    refused."""
    seed, cfg, lay = 7, 1, 1
    experts = [1, 2, 5, 8, 13, 21, 34, 55, 89, 144]
    L, hx, shared, grid = device_layer(seed, cfg, lay, experts, gut, dt)
    src = _host_experts(hx, experts, gut, dt)
    path = tmp_path / "layer1.ds4gexp"
    B.ds4g_expert_file_write(path, src)
    f = B.ExpertFile(path)
    cache_f = B.ExpertCache(10, max_tokens=2, gate_up_type=gut, down_type=dt)
    cache_h = B.ExpertCache(10, max_tokens=2, gate_up_type=gut, down_type=dt)
    ws = B.workspace(B.ds4g_forward_workspace(2))
    sg, su, sd, gridt = L.tensors[3], L.tensors[4], L.tensors[5], L.tensors[6]
    rng = np.random.default_rng(5)
    # 10 slots: the last call needs all ten experts, so each earlier miss is evicted at most once
    calls = [[[1, 2, 5, 8, 13, 21]], [[34, 55, 89, 144, 1, 2]], [[5, 8, 13, 21, 34, 55], [89, 144, 1, 2, 5, 8]],
             [[21, 34, 55, 89, 144, 13]]]
    for i, c in enumerate(calls):
        ids = np.array(c, np.int32)
        T = ids.shape[0]
        x = synth.hidden(seed, cfg, T, layer=70 + i)
        w = rng.dirichlet(np.ones(K), T).astype(np.float32)
        xd, idd, wd = (torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in (x, ids, w))
        outs = []
        for mode in ("file", "host", "resident"):
            o = torch.full((T, H), float("nan"), device=DEV)
            if mode == "file":
                B.ds4g_moe_forward_streamed_file(xd, lay, f, sg, su, sd, gridt, idd, wd, o, cache_f, ws)
            elif mode == "host":
                B.ds4g_moe_forward_streamed(xd, lay, src, sg, su, sd, gridt, idd, wd, o, cache_h, ws)
            else:
                B.ds4g_moe_forward(xd, L.struct, idd, wd, o, ws)
            assert B.ds4g_last_error(ws) == 0
            outs.append(o.cpu().numpy())
        assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    assert cache_f.stats() == cache_h.stats()
    ids = np.array([[1, 2, 3, 5, 8, 13]], np.int32)       # expert 3 is not in the file
    idd = torch.from_numpy(ids).to(DEV)
    o = torch.empty(1, H, device=DEV)
    with pytest.raises(B.DS4GError) as e:
        B.ds4g_moe_forward_streamed_file(torch.zeros(1, H, device=DEV), lay, f, sg, su, sd, gridt, idd,
                                         torch.full((1, K), 1.0 / K, device=DEV), o, cache_f, ws)
    assert e.value.code == 1
    f.close()
    cache_f.close()
    cache_h.close()
