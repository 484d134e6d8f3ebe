"""Parity of the composed MuonClip step (Kimi K2 section 2.1, "MuonClip";
the K2 review's note that QK-Clip runs after the optimizer update with the
max logit of this step) for MHA and MLA layers at test sizes where some
heads clip and others do not.

For each layer the composed call (``muonclip_step_mha`` / ``_mla``) is
checked four ways:

  * S_max per head against the fp64 oracle (relative error <= 1e-3), and
    gamma bit-exact against the oracle's gamma of the GPU's S_max;
  * the post-Muon, pre-clip masters -- taken by running the scan, the Muon
    step and the clip as three separate calls on the same inputs -- against
    the oracle's Muon step, on the update over all columns (relative
    Frobenius error <= 2e-2);
  * every column of the composed step's final masters bit-exact against the
    oracle's clip applied to those pre-clip masters with the GPU's S_max
    (clipped heads rescaled, the rest bit-unchanged);
  * the whole composition against the oracle's own composition (its Muon
    step, then its clip with its own S_max) on the change of the masters.

For MLA, W_qa and W_kva (which holds the shared k^R) must come out of the
clip bit-identical to their post-Muon values.
"""
import numpy as np
import pytest
import torch

import mc_inputs
import oracle
from gpu_helpers import NS_RTOL, SMAX_RTOL, dev, lib, rel_err, rel_fro

pytestmark = pytest.mark.gpu

LR = mc_inputs.LR


def _bits32(t) -> np.ndarray:
    a = t.detach().cpu().contiguous().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def _to_dev(inp, names):
    return {n: inp[n].to(dev()) for n in names}


def _state(inp):
    return ([t.to(dev()).clone() for t in inp["w_master"]],
            [t.to(dev()) for t in inp["grad"]],
            [t.to(dev()).clone() for t in inp["m_prev"]])


@pytest.mark.parametrize("dims", [
    dict(B=2, T=300, D=192, H=4, dh=64, seed=21),     # ragged T, 2 hot heads of 4
    dict(B=1, T=1030, D=256, H=6, dh=64, seed=22),    # several query tiles, 2 hot of 6
])
def test_muonclip_step_mha_composition(dims):
    lib()
    from muonclip_mc_max_gb300 import api, muonclip_step_mha
    H, dh = dims["H"], dims["dh"]
    inp = mc_inputs.mha_layer(n_hot=2, w_std=0.05, **dims)
    tau = inp["tau"]
    d = _to_dev(inp, ("x", "wq", "wk"))

    # (1) the composed step
    masters, grads, moms = _state(inp)
    s_max, gamma = muonclip_step_mha(d["x"], d["wq"], d["wk"], H, dh, masters, grads, moms,
                                     lr=LR, tau=tau)
    torch.cuda.synchronize()
    s_np = s_max.cpu().numpy()
    g_np = gamma.cpu().numpy()

    # (2) the same three calls separately, keeping the pre-clip masters
    masters2, grads2, moms2 = _state(inp)
    s2 = api.mc_max_logits_mha(d["x"], d["wq"], d["wk"], H, dh)
    api.mc_muon_step(masters2, grads2, moms2, lr=LR)
    torch.cuda.synchronize()
    pre = [t.cpu().clone() for t in masters2]
    g2 = api.mc_qk_clip_mha(masters2[0], masters2[1], H, dh, s2, tau)
    torch.cuda.synchronize()
    assert np.array_equal(_bits32(s2), _bits32(s_np))
    assert np.array_equal(_bits32(g2), _bits32(g_np))
    assert api.mc_read_device_status(clear=True) == 0

    # S_max and gamma
    ref_s = oracle.max_logits_mha(inp["x"], inp["wq"], inp["wk"], H, dh, False).max(0)
    assert rel_err(s_np, ref_s).max() < SMAX_RTOL
    ref_g, _ = oracle.gamma(s_np, tau)
    assert np.array_equal(_bits32(g_np), _bits32(ref_g))
    clipped = ref_g < 1
    assert clipped.sum() == 2 and (~clipped).sum() == H - 2

    # post-Muon, pre-clip masters against the oracle's Muon step (all columns)
    w_muon = []
    for i in range(2):
        w0 = inp["w_master"][i].double().numpy()
        rw, _, _ = oracle.muon_step(inp["w_master"][i], inp["grad"][i], inp["m_prev"][i], lr=LR)
        assert rel_fro(pre[i].double().numpy() - w0, rw - w0) < NS_RTOL
        w_muon.append(rw)

    # final masters: every column bit-exact to the oracle's clip of the
    # GPU's pre-clip masters with the GPU's S_max
    rq, rk, rg = oracle.qk_clip_mha(pre[0], pre[1], H, dh, s_np, tau)
    assert np.array_equal(_bits32(rg), _bits32(g_np))
    assert np.array_equal(_bits32(masters[0]), _bits32(rq))
    assert np.array_equal(_bits32(masters[1]), _bits32(rk))
    assert np.array_equal(_bits32(masters2[0]), _bits32(rq))
    cols = np.repeat(~clipped, dh)
    assert np.array_equal(_bits32(masters[0])[:, cols], _bits32(pre[0])[:, cols])

    # the composition against the oracle's own composition
    oq, ok, _ = oracle.qk_clip_mha(w_muon[0].astype(np.float32), w_muon[1].astype(np.float32),
                                   H, dh, ref_s.astype(np.float32), tau)
    for i, ref in enumerate((oq, ok)):
        w0 = inp["w_master"][i].double().numpy()
        got = masters[i].cpu().double().numpy() - w0
        assert rel_fro(got, ref.double().numpy() - w0) < NS_RTOL


@pytest.mark.parametrize("dims", [
    dict(B=1, T=520, D=256, H=4, q_lora=128, kv_lora=64, w_std=0.035),
    dict(B=2, T=200, D=128, H=5, q_lora=192, kv_lora=128, w_std=0.04),
])
def test_muonclip_step_mla_composition(dims):
    """The K2-shaped MLA parity recipe (1% heavy-tailed token rows x20, hot
    heads' q^C/q^R blocks x30) at test size: the hot heads clip, the cold
    ones stay below tau."""
    lib()
    from muonclip_mc_max_gb300 import api, muonclip_step_mla
    H, nope, rope = dims["H"], 128, 64
    inp = mc_inputs.c3b(muon=True, n_hot=2, heavy_frac=0.02, **dims)
    tau = inp["tau"]
    base = inp["rope_base"]
    names = ("x", "w_qa", "w_qb", "w_kva", "w_kb")
    d = _to_dev(inp, names)

    masters, grads, moms = _state(inp)
    s_max, gamma = muonclip_step_mla(d["x"], d["w_qa"], d["w_qb"], d["w_kva"], d["w_kb"], H, nope,
                                     rope, base, masters, grads, moms, lr=LR, tau=tau)
    torch.cuda.synchronize()
    s_np, g_np = s_max.cpu().numpy(), gamma.cpu().numpy()

    masters2, grads2, moms2 = _state(inp)
    s2 = api.mc_max_logits_mla(d["x"], d["w_qa"], d["w_qb"], d["w_kva"], d["w_kb"], H, nope, rope,
                               base, causal=True)
    api.mc_muon_step(masters2, grads2, moms2, lr=LR)
    torch.cuda.synchronize()
    pre = [t.cpu().clone() for t in masters2]
    api.mc_qk_clip_mla(masters2[1], masters2[3], H, nope, rope, s2, tau)
    torch.cuda.synchronize()
    assert np.array_equal(_bits32(s2), _bits32(s_np))
    assert api.mc_read_device_status(clear=True) == 0

    ref_s = oracle.max_logits_mla(inp["x"], inp["w_qa"], inp["w_qb"], inp["w_kva"], inp["w_kb"],
                                  H, nope, rope, base, True).max(0)
    assert rel_err(s_np, ref_s).max() < SMAX_RTOL
    ref_g, _ = oracle.gamma(s_np, tau)
    assert np.array_equal(_bits32(g_np), _bits32(ref_g))
    clipped = ref_g < 1
    assert clipped.any() and (~clipped).any()

    w_muon = []
    for i in range(4):
        w0 = inp["w_master"][i].double().numpy()
        rw, _, _ = oracle.muon_step(inp["w_master"][i], inp["grad"][i], inp["m_prev"][i], lr=LR)
        assert rel_fro(pre[i].double().numpy() - w0, rw - w0) < NS_RTOL, i
        w_muon.append(rw)

    rqb, rkb, rg = oracle.qk_clip_mla(pre[1], pre[3], H, nope, rope, s_np, tau)
    assert np.array_equal(_bits32(rg), _bits32(g_np))
    assert np.array_equal(_bits32(masters[1]), _bits32(rqb))
    assert np.array_equal(_bits32(masters[3]), _bits32(rkb))
    # W_qa and W_kva (latent projections and the shared k^R) are left alone
    assert np.array_equal(_bits32(masters[0]), _bits32(pre[0]))
    assert np.array_equal(_bits32(masters[2]), _bits32(pre[2]))
    for i in range(4):
        assert np.array_equal(_bits32(masters2[i]), _bits32(masters[i])), i

    oqb, okb, _ = oracle.qk_clip_mla(w_muon[1].astype(np.float32), w_muon[3].astype(np.float32),
                                     H, nope, rope, ref_s.astype(np.float32), tau)
    for i, ref in ((1, oqb), (3, okb)):
        w0 = inp["w_master"][i].double().numpy()
        got = masters[i].cpu().double().numpy() - w0
        assert rel_fro(got, ref.double().numpy() - w0) < NS_RTOL, i
