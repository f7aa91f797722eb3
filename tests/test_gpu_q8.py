"""The int8-activation decode path (ds4g_moe_forward_q8) against the
oracle's q8 mode on the same seeded inputs: the q8 activations and the
integer sub-block sums are exact on both sides, so the outputs differ by fp32
rounding only (bound: max-abs 2e-3 * max|ref|, the decode bound)."""
import numpy as np
import pytest

import synth
from helpers import H, K, assert_close_fwd, device_layer, oracle_forward, oracle_forward_q8

torch = pytest.importorskip("torch")
import bit_quantized_moe_bias_b300 as B  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("T", [1, 2, 3])
def test_q8_forward_matches_oracle_q8(T):
    seed = 10 + T
    rng = np.random.default_rng(seed)
    x = synth.hidden(seed, 1, T, layer=3)
    ids = np.stack([rng.choice(256, K, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.dirichlet(np.ones(K), T).astype(np.float32)
    L, hx, shared, grid = device_layer(seed, 1, 0, ids.reshape(-1))
    xd, idd, wd = (torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in (x, ids, w))
    ws = B.workspace(B.ds4g_forward_workspace(T))
    out = torch.full((T, H), float("nan"), device=DEV)
    B.ds4g_moe_forward_q8(xd, L.struct, idd, wd, out, ws)
    assert B.ds4g_last_error(ws) == 0
    got = out.cpu().numpy()
    ref = oracle_forward_q8(x, ids, w, hx, shared, grid)
    assert_close_fwd(got, ref)
    # against the fp path: the activation rounding shows, by about as much
    # on the GPU as in the oracle
    fp = oracle_forward(x, ids, w, hx, shared, grid)
    d_gpu = np.linalg.norm(got - fp) / np.linalg.norm(fp)
    d_orc = np.linalg.norm(ref - fp) / np.linalg.norm(fp)
    # 8-bit activations per 256-block: a step of max|x|/127, about 0.7 % of a unit-RMS entry
    assert 0 < d_gpu < 3e-2 and abs(d_gpu - d_orc) <= 0.1 * d_orc
    # repeatable
    out2 = torch.empty_like(out)
    B.ds4g_moe_forward_q8(xd, L.struct, idd, wd, out2, ws)
    assert np.array_equal(out2.cpu().numpy(), got)


def test_q8_forward_refusals():
    seed = 20
    x = synth.hidden(seed, 1, 4)
    ids = np.tile(np.arange(K, dtype=np.int32), (4, 1))
    w = np.full((4, K), 1.0 / K, np.float32)
    L, hx, shared, grid = device_layer(seed, 1, 0, ids.reshape(-1))
    xd, idd, wd = (torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in (x, ids, w))
    ws = B.workspace(B.ds4g_forward_workspace(4))
    out = torch.empty(4, H, device=DEV)
    with pytest.raises(B.DS4GError) as e:          # T > 3
        B.ds4g_moe_forward_q8(xd, L.struct, idd, wd, out, ws)
    assert e.value.code == 5
    L4, _, _, _ = device_layer(seed, 1, 0, ids.reshape(-1), synth.Q4_K, synth.Q4_K)
    with pytest.raises(B.DS4GError) as e:          # not IQ2_XXS
        B.ds4g_moe_forward_q8(xd[:1], L4.struct, idd[:1], wd[:1], out[:1], ws)
    assert e.value.code == 5
