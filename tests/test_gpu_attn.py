"""Attention forward with the max logit taken along, against the fp64
oracle on the same bf16 q, k, v.

Bounds: P.v uses the softmax weights rounded once to bf16 (relative error
<= 2^-9 each, the sum l from the unrounded weights) and O is rounded once to
bf16, so |O - O_ref| <= 2^-9 max_j |v_j| + 2^-9 |O_ref| up to fp32 terms;
the tests allow twice that.  S_max comes from bf16 q.k with fp32
accumulation: relative error well below 1e-4 at the maximum logit."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import dev, lib

pytestmark = pytest.mark.gpu


def _qkv(B, T, H, dh, seed, q_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, T, H * dh, generator=g) * q_scale).to(torch.bfloat16)
    k = torch.randn(B, T, H * dh, generator=g).to(torch.bfloat16)
    v = torch.randn(B, T, H * dh, generator=g).to(torch.bfloat16)
    return q, k, v


def _check(q, k, v, H, dh, causal):
    lib()
    from muonclip_mc_max_gb300 import api
    B, T, _ = q.shape
    s_bh = torch.empty(B, H, dtype=torch.float32, device=dev())
    o, s = api.mc_attention_mha(q.to(dev()), k.to(dev()), v.to(dev()), H, dh, causal=causal, s_max_bh=s_bh)
    torch.cuda.synchronize()
    assert api.mc_read_device_status(clear=True) == 0
    o_ref, s_ref = oracle.attention_mha_np(q, k, v, H, dh, causal)
    got = o.cpu().double().numpy().reshape(B, T, H, dh)
    vmax = np.abs(v.double().numpy()).reshape(B, T, H, dh).max(axis=(1, 3))  # [B, H]
    tol = 2.0 ** -8 * vmax[:, None, :, None] + 2.0 ** -8 * np.abs(o_ref)
    bad = np.abs(got - o_ref) > tol
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} outputs off; max err {np.abs(got - o_ref).max()}"
    rel = np.abs(s_bh.cpu().numpy() - s_ref) / np.abs(s_ref)
    assert rel.max() < 1e-4, rel
    assert np.array_equal(s.cpu().numpy(), s_bh.cpu().numpy().max(0))
    return o, s


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [
    (2, 200, 2, 64),    # two query tiles, ragged key tail
    (1, 300, 3, 128),   # dh = 128 (two 64-column blocks), three tiles
    (1, 128, 1, 64),    # exactly one tile
    (2, 77, 2, 64),     # T below one tile
    (1, 1030, 1, 64),   # nine key blocks, tail of 6
    (2, 77, 2, 128),    # dh = 128 below one tile
    (2, 200, 2, 128),   # dh = 128, two query tiles, ragged key tail
    (1, 1030, 1, 128),  # dh = 128, nine key blocks through its two K stages
    (3, 1, 2, 64),      # a single token
    (2, 1, 1, 128),     # a single token, dh = 128
    (1, 129, 2, 64),    # one row past the first tile
    (1, 257, 1, 128),   # one row past a pair of tiles, dh = 128
])
def test_attention_vs_oracle(shape, causal):
    B, T, H, dh = shape
    q, k, v = _qkv(B, T, H, dh, seed=1200 + T + dh)
    _check(q, k, v, H, dh, causal)


@pytest.mark.parametrize("dh", [64, 128])
def test_attention_peaked_softmax_rescales(dh):
    """Large logits: the running max grows block after block, so O is
    rescaled in TMEM many times."""
    q, k, v = _qkv(1, 640, 2, dh, seed=1300 + dh, q_scale=6.0)
    _check(q, k, v, 2, dh, False)
    _check(q, k, v, 2, dh, True)


def test_attention_accumulate_and_max_logit_semantics():
    """accumulate max-merges into s_max, like the scan."""
    lib()
    from muonclip_mc_max_gb300 import api
    q, k, v = _qkv(2, 150, 2, 64, seed=1400)
    q2, k2, v2 = _qkv(2, 150, 2, 64, seed=1401, q_scale=3.0)
    _, s1 = api.mc_attention_mha(q.to(dev()), k.to(dev()), v.to(dev()), 2, 64)
    _, s2 = api.mc_attention_mha(q2.to(dev()), k2.to(dev()), v2.to(dev()), 2, 64, accumulate=True,
                                 s_max=s1.clone())
    torch.cuda.synchronize()
    _, r1 = oracle.attention_mha_np(q, k, v, 2, 64)
    _, r2 = oracle.attention_mha_np(q2, k2, v2, 2, 64)
    ref = np.maximum(r1.max(0), r2.max(0))
    assert np.all(np.abs(s2.cpu().numpy() - ref) / np.abs(ref) < 1e-4)


def test_attention_negative_max_logit():
    """Every logit of a head below zero (its keys are the negated queries,
    all rows parallel): S_max is negative and goes through the sign-bit
    path of the merge; a second head with k = q stays positive."""
    g = torch.Generator().manual_seed(1500)
    B, T, H, dh = 2, 200, 2, 64
    u = torch.randn(H * dh, generator=g)
    a = torch.rand(B, T, 1, generator=g) + 0.5
    q = (a * u).to(torch.bfloat16)
    k = q.clone()
    k[:, :, :dh] = -q[:, :, :dh]
    v = torch.randn(B, T, H * dh, generator=g).to(torch.bfloat16)
    for causal in (False, True):
        _, s = _check(q, k, v, H, dh, causal)
        s = s.cpu().numpy()
        assert s[0] < 0 < s[1]
