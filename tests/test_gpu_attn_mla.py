"""MLA attention forward with the max logit taken along (Kimi K2's
attention: per-head q^C, k^C, q^R and the shared k^R of the K2 review's MLA
table, d = 192 for the logits, dv = 128), against the fp64 oracle on the
same bf16 inputs, element by element.

Bounds as for the MHA forward: P.v uses the softmax weights rounded once to
bf16 and O is rounded once to bf16, so |O - O_ref| <= 2^-9 max_j |v_j| +
2^-9 |O_ref| up to fp32 terms; the tests allow twice that.  S_max comes from
bf16 q.k with fp32 accumulation over 192 products: relative error below
1e-4 at the maximum logit."""
import numpy as np
import pytest
import torch

import mc_inputs
import oracle
from gpu_helpers import dev, lib

pytestmark = pytest.mark.gpu

NOPE, ROPE, DV = 128, 64, 128


def _check(inp, causal, kr_in_latent=False):
    lib()
    from muonclip_mc_max_gb300 import api
    q, kc, kr, v, H = inp["q"], inp["k_c"], inp["k_r"], inp["v"], inp["H"]
    B, T, _ = q.shape
    kr_dev, kr_col = kr.to(dev()), 0
    if kr_in_latent:
        # k^R as the rope part of a [c_KV | k^R] buffer (576 columns, k^R from 512)
        buf = torch.zeros(B, T, 576, dtype=torch.bfloat16)
        buf[..., 512:] = kr
        kr_dev, kr_col = buf.to(dev()), 512
    s_bh = torch.empty(B, H, dtype=torch.float32, device=dev())
    o, s = api.mc_attention_mla(q.to(dev()), kc.to(dev()), kr_dev, v.to(dev()), H, causal=causal,
                                kr_col=kr_col, s_max_bh=s_bh)
    torch.cuda.synchronize()
    assert api.mc_read_device_status(clear=True) == 0
    o_ref, s_ref = oracle.attention_mla_np(q, kc, kr, v, H, NOPE, ROPE, DV, causal)
    got = o.cpu().double().numpy().reshape(B, T, H, DV)
    vmax = np.abs(v.double().numpy()).reshape(B, T, H, DV).max(axis=(1, 3))  # [B, H]
    tol = 2.0 ** -8 * vmax[:, None, :, None] + 2.0 ** -8 * np.abs(o_ref)
    bad = np.abs(got - o_ref) > tol
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} outputs off; max err {np.abs(got - o_ref).max()}"
    rel = np.abs(s_bh.cpu().numpy() - s_ref) / np.abs(s_ref)
    assert rel.max() < 1e-4, rel
    assert np.array_equal(s.cpu().numpy(), s_bh.cpu().numpy().max(0))
    return o, s


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", [
    (1, 300, 2),    # three query tiles, ragged key tail
    (2, 128, 1),    # exactly one tile
    (2, 77, 3),     # T below one tile
    (1, 1030, 1),   # nine key blocks, tail of 6
    (3, 1, 2),      # a single token
    (1, 129, 2),    # one row past the first tile
    (1, 256, 1),    # exactly one pair of tiles
])
def test_attention_mla_vs_oracle(shape, causal):
    B, T, H = shape
    inp = mc_inputs.attention_mla_qkv(B, T, H, seed=1500 + T + H)
    _check(inp, causal)


def test_attention_mla_rope_key_inside_the_latent_buffer():
    """k^R read from columns 512..575 of a [c_KV | k^R] buffer."""
    inp = mc_inputs.attention_mla_qkv(2, 260, 2, seed=1601)
    _check(inp, True, kr_in_latent=True)


def test_attention_mla_peaked_softmax_rescales():
    """Large logits: the running max grows block after block, so O is
    rescaled in TMEM many times, with P stored over the S columns."""
    inp = mc_inputs.attention_mla_qkv(1, 640, 2, seed=1602, q_std=6.0)
    _check(inp, False)
    _check(inp, True)


def test_attention_mla_max_logit_matches_the_mla_scan():
    """The forward's max logit on the MLA layer's own projections (q^C, q^R,
    k^C, k^R with RoPE, as the scan forms them) equals the scan's S_max."""
    lib()
    from muonclip_mc_max_gb300 import api
    H = 3
    inp = mc_inputs.mla_layer(B=1, T=384, D=256, H=H, q_lora=128, kv_lora=64, n_hot=1, w_std=0.04,
                              seed=1603, heavy_frac=0.02)
    x = inp["x"].double().numpy()[0]
    qa, qb, kva, kb = (inp[n].double().numpy() for n in ("w_qa", "w_qb", "w_kva", "w_kb"))
    cq, ckv = x @ qa, x @ kva
    q = np.empty((384, H * 192))
    kc = np.empty((384, H * 128))
    for h in range(H):
        qh = cq @ qb[:, h * 192:(h + 1) * 192]
        q[:, h * 192:h * 192 + 128] = qh[:, :128]
        q[:, h * 192 + 128:(h + 1) * 192] = oracle._rope_np(qh[:, 128:], 0, inp["rope_base"])
        kc[:, h * 128:(h + 1) * 128] = ckv[:, :64] @ kb[:, h * 128:(h + 1) * 128]
    kr = oracle._rope_np(ckv[:, 64:], 0, inp["rope_base"])

    def bf(a):
        return torch.from_numpy(a).float().to(torch.bfloat16).reshape(1, 384, -1).to(dev())

    v = torch.randn(1, 384, H * 128).to(torch.bfloat16).to(dev())
    _, s = api.mc_attention_mla(bf(q), bf(kc), bf(kr), v, H, causal=True)
    s_scan = api.mc_max_logits_mla(*(inp[n].to(dev()) for n in ("x", "w_qa", "w_qb", "w_kva", "w_kb")),
                                   H, 128, 64, inp["rope_base"], causal=True)
    torch.cuda.synchronize()
    ref = oracle.max_logits_mla(inp["x"], inp["w_qa"], inp["w_qb"], inp["w_kva"], inp["w_kb"], H, 128,
                                64, inp["rope_base"], True).max(0)
    # both within the scan tolerance of the exact value (the forward's q and k
    # are the fp64 projections rounded once to bf16)
    assert (np.abs(s.cpu().numpy() - ref) / ref).max() < 1e-2
    assert (np.abs(s_scan.cpu().numpy() - ref) / ref).max() < 1e-3


def test_attention_mla_rejects_unsupported_shapes():
    lib()
    from muonclip_mc_max_gb300 import api
    inp = mc_inputs.attention_mla_qkv(1, 64, 1, seed=1604)
    q, kc, kr, v = (inp[n].to(dev()) for n in ("q", "k_c", "k_r", "v"))
    with pytest.raises(api.MCError) as e:
        api.mc_attention_mla(q[..., :160].contiguous(), kc[..., :96].contiguous(), kr, v[..., :96].contiguous(),
                             1, nope=96, rope=64, dv=96)
    assert e.value.status == 2  # MC_ERR_UNSUPPORTED
    with pytest.raises(api.MCError):
        api.mc_attention_mla(q, kc, kr, v, 1, kr_col=4)  # rope columns past the row
