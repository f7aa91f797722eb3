"""GPU parity on the two remaining workload shapes, everything computed by the
library (router, bucketing, experts, norm) and compared with the oracle run
on the same seeded inputs.

* Batched decode: one layer, T = 32 independent tokens, Zipf(1.1)-ranked
  router bias so that the top-6 sets overlap (the T < 64 decode path).
* q2-q4 prefill: T = 4096 tokens through 8 chained layers (2 IQ2_XXS/Q2_K
  layers, then 6 Q4_K layers), Zipf bias, each layer's output RMS-normalised
  as the next layer's input (the "q2-q4" mixed model: 2-bit body, last
  layers at 4 bits, per the ds4 deep-dive's quantisation policy section).

The stacked case is compared layer by layer, not end to end: with the
synthetic Q4_K weights some tokens' outputs come from the exponential tail of
SiLU (gate values near -20 against row norms of ~7000), and a CPU emulation
of the tensor-core path's roundings (fp16/bf16 operands) turns the 6e-3 drift
of two IQ2 layers into a 97 % change of such a token's third-layer output.
That is the arithmetic, not a fault, so each layer gets the oracle's input."""
import numpy as np
import pytest

import oracle
import synth
from helpers import H, K, ROUTE_MARGIN, FullLayer, assert_close_fwd, check_route

torch = pytest.importorskip("torch")
import bit_quantized_moe_bias_b300 as B  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"
REL_L2 = 1e-2        # tensor-core path bound, per token and per layer


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _route(h, R, b):
    T = h.shape[0]
    ids = torch.empty(T, K, dtype=torch.int32, device=DEV)
    w = torch.empty(T, K, dtype=torch.float32, device=DEV)
    ws = B.workspace(B.ds4g_route_workspace(T))
    B.ds4g_moe_route(h, R, b, ids, w, ws)
    assert B.ds4g_last_error(ws) == 0
    return ids, w


def _forward(h, L, ids, w):
    T = h.shape[0]
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    ws = B.workspace(B.ds4g_forward_workspace(T))
    B.ds4g_moe_forward(h, L.L.struct, ids, w, out, ws)
    assert B.ds4g_last_error(ws) == 0
    return out


def test_batched_decode_T32_zipf():
    L = FullLayer(0, 2, 0)
    T = 32
    x = synth.hidden(0, 2, T)
    R, b = synth.router(0, 2), synth.bias_zipf(0, 2)
    ids_g, w_g = _route(_t(x), _t(R), _t(b))
    out = _forward(_t(x), L, ids_g, w_g).cpu().numpy()
    ids_r, w_r, keys, margin = oracle.route(x, R, b)
    check_route(ids_g.cpu().numpy(), w_g.cpu().numpy(), ids_r, w_r, keys, margin)
    ok = margin > ROUTE_MARGIN
    assert ok.sum() >= T - 2
    # heavy overlap: far fewer distinct experts than 6T slots
    assert len(set(ids_r.reshape(-1).tolist())) < K * T
    assert_close_fwd(out[ok], L.oracle(x[ok], ids_r[ok], w_r[ok]))


def _rel_l2(got, ref):
    return float(np.linalg.norm(got.astype(np.float64) - ref) / np.linalg.norm(ref))


def test_q2q4_prefill_layers_T4096():
    """Every layer of the 8-layer q2-q4 stack at T = 4096 with Zipf routing.
    The library runs the whole chain (route, forward, rmsnorm on the device);
    before each layer the sampled tokens' rows are replaced by the oracle
    chain's hidden state, so the oracle and the library see the same input
    for the compared rows while the other 4096 - n rows keep the library's own
    chain and so its bucket sizes (up to all 4096 tokens on one expert).
    256 seeded tokens per layer are compared."""
    T, NL, NS = 4096, 8, 256
    layers = [FullLayer(0, 4, l) if l < 2 else FullLayer(0, 4, l, synth.Q4_K, synth.Q4_K) for l in range(NL)]
    rng = np.random.default_rng(4)
    s = np.array(sorted(set(rng.choice(T, NS, replace=False).tolist()) | {0, T - 1}))
    sd = torch.from_numpy(s).to(DEV)
    x = synth.hidden(0, 4, T)
    h = _t(x)
    hs = x[s]
    worst, big = 0.0, 0
    for l, L in enumerate(layers):
        h[sd] = _t(hs)
        R, b = synth.router(0, 4, l), synth.bias_zipf(0, 4, l)
        ids, w = _route(h, _t(R), _t(b))
        big = max(big, int(torch.bincount(ids.reshape(-1).long(), minlength=256).max()))
        out = _forward(h, L, ids, w)
        ids_g, w_g, out_g = ids.cpu().numpy()[s], w.cpu().numpy()[s], out.cpu().numpy()[s]
        ids_r, w_r, keys, margin = oracle.route(hs, R, b)
        check_route(ids_g, w_g, ids_r, w_r, keys, margin)
        ok = margin > ROUTE_MARGIN
        assert ok.sum() >= len(s) - 2
        out_r = L.oracle(hs[ok], ids_r[ok], w_r[ok])
        assert np.all(np.isfinite(out_g))
        for i, t in enumerate(np.nonzero(ok)[0]):
            e = _rel_l2(out_g[t], out_r[i])
            worst = max(worst, e)
            assert e <= REL_L2, f"layer {l} token {s[t]}: rel L2 {e:.3e}"
        hs = oracle.rmsnorm(L.oracle(hs, ids_r, w_r)) if not ok.all() else oracle.rmsnorm(out_r)
        if l + 1 < NL:
            hn = torch.empty_like(out)
            B.ds4g_rmsnorm(out, hn)
            h = hn
    assert big >= 1024   # the Zipf ranking does concentrate the load
    print(f"q2-q4 layers: worst rel L2 {worst:.2e}, largest bucket {big}")
