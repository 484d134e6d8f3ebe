"""Degenerate cases of the method on the CUDA path: Newton-Schulz of a zero
matrix and of vectors, a Muon step with no gradient (weight decay only), a
single-token causal scan, and a head whose weights are zero (S = 0, so
gamma = 1 and the clip leaves it alone)."""
import numpy as np
import pytest
import torch

import mc_inputs
import oracle
from gpu_helpers import NS_RTOL, dev, lib, rel_fro

pytestmark = pytest.mark.gpu


def test_newton_schulz_zero_matrix_is_zero():
    """X0 = 0 / (0 + eps) = 0, and every quintic step maps 0 to 0."""
    lib()
    from muonclip_mc_max_gb300 import api
    z = torch.zeros(200, 300, device=dev())
    out = api.mc_newton_schulz([z, z.t().contiguous()])
    torch.cuda.synchronize()
    for o in out:
        assert bool((o == 0).all())


@pytest.mark.parametrize("shape", [(1, 300), (300, 1), (2, 3), (3, 2), (37, 13)])
def test_newton_schulz_vectors_and_tiny(shape):
    """Rank-1, 2 x 3 and odd widths (columns not a multiple of 4: the
    element-by-element path) against the oracle; a vector maps to
    phi^5(1 / (1 + eps / |v|)) v / |v|."""
    lib()
    from muonclip_mc_max_gb300 import api
    g = mc_inputs.matrix(*shape, seed=900 + shape[0] * 7 + shape[1])
    out = api.mc_newton_schulz([g.to(dev())])[0]
    torch.cuda.synchronize()
    assert rel_fro(out.cpu().numpy(), oracle.newton_schulz(g)) < NS_RTOL


def test_muon_step_without_gradient_is_weight_decay():
    """G = 0 and M = 0: M stays 0, O = NS(0) = 0, W <- (1 - lr wd) W."""
    lib()
    from muonclip_mc_max_gb300 import api
    shapes = [(256, 128), (96, 512)]
    W = [mc_inputs.matrix(r, c, seed=930 + i, std=0.02) for i, (r, c) in enumerate(shapes)]
    wd_ = [t.to(dev()) for t in W]
    g = [torch.zeros(r, c, device=dev()) for r, c in shapes]
    m = [torch.zeros(r, c, device=dev()) for r, c in shapes]
    lr, wd = 2e-4, 0.1
    api.mc_muon_step(wd_, g, m, lr=lr, wd=wd)
    torch.cuda.synchronize()
    for w0, w1, mm in zip(W, wd_, m):
        assert bool((mm == 0).all())
        ref = (1.0 - lr * wd) * w0.double().numpy()
        assert rel_fro(w1.cpu().numpy(), ref) < 1e-6


def test_causal_single_token_scan():
    """T = 1 causal: each sequence has one logit q_0 . k_0.  A single dot
    product can cancel, so the bound is on its terms: fp16 rounding of q and
    k moves q.k by at most about 2 * 2^-11 * sum_f |q_f k_f| / sqrt(d)."""
    lib()
    from muonclip_mc_max_gb300 import api
    inp = mc_inputs.mha_layer(B=3, T=1, D=128, H=2, dh=64, n_hot=1, seed=941, muon=False,
                              w_std=0.05)
    s_bh = torch.empty(3, 2, dtype=torch.float32, device=dev())
    s = api.mc_max_logits_mha(inp["x"].to(dev()), inp["wq"].to(dev()), inp["wk"].to(dev()), 2, 64,
                              causal=True, s_max_bh=s_bh)
    torch.cuda.synchronize()
    ref = oracle.max_logits_mha(inp["x"], inp["wq"], inp["wk"], 2, 64, True)
    x0 = inp["x"][:, 0].double().numpy()
    q = x0 @ inp["wq"].double().numpy()
    k = x0 @ inp["wk"].double().numpy()
    mag = np.abs(q * k).reshape(3, 2, 64).sum(-1) / 8.0  # sum_f |q_f k_f| / sqrt(64)
    err = np.abs(s_bh.cpu().numpy() - ref)
    assert np.all(err <= 4 * 2.0 ** -11 * mag + 1e-6), (err, mag)
    assert np.array_equal(s.cpu().numpy(), s_bh.cpu().numpy().max(0))


def test_zero_weight_head_gives_gamma_one():
    """A head whose W_q block is zero has only zero logits: S = 0, gamma = 1,
    and the clip writes none of its weights; the hot head is clipped."""
    lib()
    from muonclip_mc_max_gb300 import api
    H, dh = 3, 64
    inp = mc_inputs.mha_layer(B=2, T=256, D=128, H=H, dh=dh, n_hot=1, hot_scale=60.0, seed=951,
                              muon=False, w_std=0.05)
    wq = inp["wq"].clone()
    cold = [h for h in range(H) if h not in inp["hot"]][0]
    wq[:, cold * dh:(cold + 1) * dh] = 0
    wq_d, wk_d = wq.to(dev()), inp["wk"].to(dev())
    s = api.mc_max_logits_mha(inp["x"].to(dev()), wq_d, wk_d, H, dh)
    torch.cuda.synchronize()
    assert float(s[cold]) == 0.0
    wk_before = wk_d.clone()
    g = api.mc_qk_clip_mha(wq_d, wk_d, H, dh, s, 100.0)
    torch.cuda.synchronize()
    assert float(g[cold]) == 1.0
    assert torch.equal(wk_d[:, cold * dh:(cold + 1) * dh], wk_before[:, cold * dh:(cold + 1) * dh])
    assert float(g[inp["hot"][0]]) < 1.0


def test_muon_step_odd_widths():
    """Widths that are not a multiple of 4 (element-by-element momentum,
    cast and update), tall and wide, against the oracle."""
    lib()
    from muonclip_mc_max_gb300 import api
    shapes = [(37, 13), (13, 37), (130, 70)]
    W = [mc_inputs.matrix(r, c, seed=960 + i, std=0.02) for i, (r, c) in enumerate(shapes)]
    G = [mc_inputs.matrix(r, c, seed=970 + i, std=1e-3) for i, (r, c) in enumerate(shapes)]
    M = [mc_inputs.matrix(r, c, seed=980 + i, std=1e-3) for i, (r, c) in enumerate(shapes)]
    wd_ = [t.to(dev()) for t in W]
    md = [t.to(dev()) for t in M]
    api.mc_muon_step(wd_, [t.to(dev()) for t in G], md, lr=2e-4)
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        rw, rm, _ = oracle.muon_step(W[i], G[i], M[i], lr=2e-4)
        assert rel_fro(md[i].cpu().numpy(), rm) < 1e-6
        assert rel_fro(wd_[i].cpu().double().numpy() - W[i].double().numpy(),
                       rw - W[i].double().numpy()) < NS_RTOL
