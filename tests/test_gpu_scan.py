"""Max-logit scan parity: the CUDA path (tcgen05 for bf16, CUDA cores for
fp32 / small shapes) against the fp64 oracle on the same seeded inputs,
per (sequence, head), with causal and ragged sequence lengths."""
import numpy as np
import pytest
import torch

import mc_inputs
import oracle
from gpu_helpers import SMAX_RTOL, dev, lib, rel_err

pytestmark = pytest.mark.gpu


def _run_mha(x, wq, wk, H, dh, causal, accumulate=False, s_max=None):
    lib()
    from muonclip_mc_max_gb300 import api
    B = x.shape[0]
    s_bh = torch.empty(B, H, dtype=torch.float32, device=dev())
    s = api.mc_max_logits_mha(x.to(dev()), wq.to(dev()), wk.to(dev()), H, dh, causal=causal,
                              accumulate=accumulate, s_max=s_max, s_max_bh=s_bh)
    torch.cuda.synchronize()
    return s.cpu().numpy(), s_bh.cpu().numpy()


def test_c1_fp32_page_example():
    """The seed-7 example of the MHA semantic reference (fp32, CUDA cores)."""
    inp = mc_inputs.c1()
    s, s_bh = _run_mha(inp["x"], inp["wq"], inp["wk"], inp["H"], inp["dh"], False)
    ref = oracle.max_logits_mha(inp["x"], inp["wq"], inp["wk"], inp["H"], inp["dh"])
    assert rel_err(s_bh, ref).max() < 1e-5
    assert rel_err(s, ref.max(0)).max() < 1e-5


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [
    (2, 300, 192, 3, 64),    # ragged T (not a multiple of 128 or 256), several key tiles
    (1, 128, 64, 1, 64),     # exactly one query tile
    (3, 77, 128, 2, 128),    # dh = 128: two K blocks per head, T < one tile
    (1, 1030, 256, 2, 64),   # many tiles, ragged tail of 6
    (1, 257, 128, 1, 64),    # one key past a 256-key tile, one row past two query tiles
])
def test_mha_bf16_tensor_path(shape, causal):
    B, T, D, H, dh = shape
    inp = mc_inputs.mha_layer(B=B, T=T, D=D, H=H, dh=dh, n_hot=1, causal=causal, seed=50 + T,
                              muon=False, w_std=0.05)
    s, s_bh = _run_mha(inp["x"], inp["wq"], inp["wk"], H, dh, causal)
    ref = oracle.max_logits_mha(inp["x"], inp["wq"], inp["wk"], H, dh, causal)
    err = rel_err(s_bh, ref)
    assert err.max() < SMAX_RTOL, (err.max(), s_bh, ref)
    assert np.array_equal(s, s_bh.max(0))


def test_fp32_small_shapes_simt():
    inp = mc_inputs.mha_layer(B=2, T=37, D=20, H=3, dh=6, n_hot=1, seed=61, muon=False)
    x, wq, wk = inp["x"].float(), inp["wq"].float(), inp["wk"].float()
    for causal in (False, True):
        s, s_bh = _run_mha(x, wq, wk, 3, 6, causal)
        ref = oracle.max_logits_mha(x, wq, wk, 3, 6, causal)
        assert rel_err(s_bh, ref).max() < 1e-5


def test_accumulate_is_max_over_microbatches():
    a = mc_inputs.mha_layer(B=2, T=200, D=128, H=2, dh=64, n_hot=1, seed=71, muon=False)
    b = mc_inputs.mha_layer(B=2, T=200, D=128, H=2, dh=64, n_hot=1, seed=72, muon=False)
    wq, wk = a["wq"], a["wk"]
    s1, _ = _run_mha(a["x"], wq, wk, 2, 64, True)
    s_dev = torch.tensor(s1, device=dev())
    s2, s_bh2 = _run_mha(b["x"], wq, wk, 2, 64, True, accumulate=True, s_max=s_dev)
    ref_b = oracle.max_logits_mha(b["x"], wq, wk, 2, 64, True)
    ref = np.maximum(oracle.max_logits_mha(a["x"], wq, wk, 2, 64, True).max(0), ref_b.max(0))
    assert rel_err(s2, ref).max() < SMAX_RTOL
    # the per-sequence maxima are this call's alone (only s_max accumulates)
    assert rel_err(s_bh2, ref_b).max() < SMAX_RTOL


def test_nonfinite_input_sets_status_and_gamma_one():
    lib()
    from muonclip_mc_max_gb300 import api
    api.mc_read_device_status(clear=True)
    inp = mc_inputs.mha_layer(B=1, T=64, D=64, H=2, dh=64, n_hot=0, seed=81, muon=False)
    x = inp["x"].clone()
    x[0, 5, 3] = float("nan")
    s, _ = _run_mha(x, inp["wq"], inp["wk"], 2, 64, False)
    assert np.isnan(s).all()
    assert api.mc_read_device_status(clear=True) & api.MC_DEV_NONFINITE
    wq = inp["wq"].to(dev())
    before = wq.clone()
    g = api.mc_qk_clip_mha(wq, inp["wk"].to(dev()), 2, 64, torch.tensor(s, device=dev()), 100.0)
    assert torch.equal(g.cpu(), torch.ones(2))
    assert torch.equal(wq, before)


@pytest.mark.parametrize("causal", [False, True])
def test_negative_and_positive_maxima_merge(causal):
    """The per-item maxima are merged into S_max with integer atomics whose
    order depends on the sign bit.  Activations that are positive multiples
    of one vector make every row's projections parallel: with W_k = -W_q a
    head's logits are all negative, with W_k = W_q all positive.  Head 0 is
    negative and head 1 positive; S_max and the per-sequence maxima must
    match the oracle, and accumulating keeps the larger of old and new."""
    rng = np.random.default_rng(91)
    B, T, D, H, dh = 2, 300, 128, 2, 64
    vdir = rng.standard_normal(D)
    a = rng.uniform(0.5, 1.5, size=(B, T, 1))
    x = torch.tensor(a * vdir[None, None, :], dtype=torch.float32).to(torch.bfloat16)
    wq = torch.tensor(rng.standard_normal((D, H * dh)) * 0.1, dtype=torch.float32).to(torch.bfloat16)
    wk = wq.clone()
    wk[:, :dh] = -wq[:, :dh]
    s, s_bh = _run_mha(x, wq, wk, H, dh, causal)
    ref = oracle.max_logits_mha(x, wq, wk, H, dh, causal)
    assert (ref[:, 0] < 0).all() and (ref[:, 1] > 0).all()
    assert rel_err(s_bh, ref).max() < SMAX_RTOL
    assert np.array_equal(s, s_bh.max(0))
    # accumulate: an old S_max below the new one on head 0, above it on head 1
    old = torch.tensor([2.0 * s[0], 2.0 * s[1]], dtype=torch.float32, device=dev())
    s2, _ = _run_mha(x, wq, wk, H, dh, causal, accumulate=True, s_max=old)
    assert s2[0] == s[0] and s2[1] == np.float32(2.0 * s[1])
