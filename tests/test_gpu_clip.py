"""QK-Clip parity: bit-exact against the oracle (one rounding of the exact
product per weight), gamma bit-exact from the GPU's own S_max, untouched
heads / components bit-unchanged."""
import numpy as np
import pytest
import torch

import mc_inputs
import oracle
from gpu_helpers import bits16, dev, lib

pytestmark = pytest.mark.gpu

S_CASES = np.array([50.0, 150.0, 1000.0, 100.0, 100.0001, 0.0, -5.0, np.nan, np.inf, 3.7e5],
                   np.float32)


def _weights(rows, cols, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, cols, generator=g) * 0.02).to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("dh", [64, 24, 5])
def test_mha_clip_bit_exact(dtype, dh):
    lib()
    from muonclip_mc_max_gb300 import api
    H = len(S_CASES)
    D = 96
    wq, wk = _weights(D, H * dh, dtype, 1), _weights(D, H * dh, dtype, 2)
    wq_d, wk_d = wq.to(dev()), wk.to(dev())
    s = torch.tensor(S_CASES, device=dev())
    g = api.mc_qk_clip_mha(wq_d, wk_d, H, dh, s, 100.0)
    torch.cuda.synchronize()
    rq, rk, rg = oracle.qk_clip_mha(wq, wk, H, dh, S_CASES, 100.0)
    assert np.array_equal(g.cpu().numpy().view(np.uint32), rg.view(np.uint32))
    if dtype == torch.bfloat16:
        assert np.array_equal(bits16(wq_d), bits16(rq))
        assert np.array_equal(bits16(wk_d), bits16(rk))
    else:
        assert np.array_equal(wq_d.cpu().numpy().view(np.uint32), rq.numpy().view(np.uint32))
        assert np.array_equal(wk_d.cpu().numpy().view(np.uint32), rk.numpy().view(np.uint32))
    # heads with gamma == 1 keep their bits
    for h in np.nonzero(rg == 1.0)[0]:
        assert torch.equal(wq_d[:, h * dh:(h + 1) * dh].cpu(), wq[:, h * dh:(h + 1) * dh])


def test_bf16_rounding_ties_exact():
    """Weights and factors chosen so the float product lands near bf16 ties:
    a single rounding of the exact product must still be reproduced."""
    lib()
    from muonclip_mc_max_gb300 import api
    H, dh, D = 4, 8, 512
    rng = np.random.default_rng(3)
    bits = rng.integers(0x3C00, 0x4100, size=(D, H * dh)).astype(np.uint16)
    w = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    # tau / S with many mantissa bits so w * sqrt(gamma) is rarely exact
    s = np.array([100.0 / 0.7000001, 100.0 / 0.33333334, 100.0 / 0.9999999, 401.0], np.float32)
    wd = w.to(dev())
    wk = w.clone().to(dev())
    api.mc_qk_clip_mha(wd, wk, H, dh, torch.tensor(s, device=dev()), 100.0)
    torch.cuda.synchronize()
    rq, _, _ = oracle.qk_clip_mha(w, w.clone(), H, dh, s, 100.0)
    assert np.array_equal(bits16(wd), bits16(rq))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_mla_clip_bit_exact(dtype):
    lib()
    from muonclip_mc_max_gb300 import api
    H, nope, rope, ql, kvl = len(S_CASES), 128, 64, 96, 64
    w_qb = _weights(ql, H * (nope + rope), dtype, 3)
    w_kb = _weights(kvl, H * nope, dtype, 4)
    w_kva = _weights(64, kvl + rope, dtype, 5)
    qb_d, kb_d, kva_d = w_qb.to(dev()), w_kb.to(dev()), w_kva.to(dev())
    s = torch.tensor(S_CASES, device=dev())
    g = api.mc_qk_clip_mla(qb_d, kb_d, H, nope, rope, s, 100.0)
    torch.cuda.synchronize()
    rqb, rkb, rg = oracle.qk_clip_mla(w_qb, w_kb, H, nope, rope, S_CASES, 100.0)
    assert np.array_equal(g.cpu().numpy().view(np.uint32), rg.view(np.uint32))
    if dtype == torch.bfloat16:
        assert np.array_equal(bits16(qb_d), bits16(rqb))
        assert np.array_equal(bits16(kb_d), bits16(rkb))
    else:
        assert np.array_equal(qb_d.cpu().numpy().view(np.uint32), rqb.numpy().view(np.uint32))
        assert np.array_equal(kb_d.cpu().numpy().view(np.uint32), rkb.numpy().view(np.uint32))
    assert torch.equal(kva_d.cpu(), w_kva)  # k^R lives in W_kva: never touched


def test_gamma_from_gpu_smax_bit_exact():
    """Scan on the GPU, then gamma: equal to the oracle's gamma computed
    from the GPU's own S_max, bit for bit; clipped heads land at <= tau."""
    lib()
    from muonclip_mc_max_gb300 import api
    inp = mc_inputs.mha_layer(B=2, T=256, D=128, H=4, dh=64, n_hot=2, hot_scale=60.0, seed=91,
                              muon=False, w_std=0.05)
    x, wq, wk = inp["x"].to(dev()), inp["wq"].to(dev()), inp["wk"].to(dev())
    s = api.mc_max_logits_mha(x, wq, wk, 4, 64)
    g = api.mc_qk_clip_mha(wq, wk, 4, 64, s, 100.0)
    torch.cuda.synchronize()
    s_np = s.cpu().numpy()
    rg, _ = oracle.gamma(s_np, 100.0)
    assert np.array_equal(g.cpu().numpy().view(np.uint32), rg.view(np.uint32))
    assert (rg < 1).sum() >= 1
    after = oracle.max_logits_mha(inp["x"], wq.cpu(), wk.cpu(), 4, 64).max(0)
    assert np.all(after[rg < 1] <= 100.0 * (1 + 2 ** -7))  # bf16 storage: one rounding per weight


def test_global_clip():
    lib()
    from muonclip_mc_max_gb300 import api
    w = _weights(64, 96, torch.float32, 9)
    wq, wk = w.clone().to(dev()), (w * 2).to(dev())
    s = np.array([50.0, 400.0, 120.0], np.float32)
    g = api.mc_qk_clip_global(wq, wk, torch.tensor(s, device=dev()), 100.0, alpha=0.5)
    torch.cuda.synchronize()
    rq, rk, rg = oracle.qk_clip_global(w, w * 2, s, 100.0, 0.5)
    assert float(g.cpu()[0]) == rg
    np.testing.assert_allclose(wq.cpu().numpy(), rq.numpy(), rtol=2 ** -23)
    np.testing.assert_allclose(wk.cpu().numpy(), rk.numpy(), rtol=2 ** -23)
