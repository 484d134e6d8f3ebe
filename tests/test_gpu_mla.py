"""MLA max-logit scan parity (four tcgen05 projections with the RoPE in the
epilogue, then the three-block scan) against the fp64 oracle, and the MLA
clip of a GPU-measured S_max."""
import numpy as np
import pytest
import torch

import mc_inputs
import oracle
from gpu_helpers import SMAX_RTOL, bits16, dev, lib, rel_err

pytestmark = pytest.mark.gpu


def _mla(inp, causal):
    lib()
    from muonclip_mc_max_gb300 import api
    B = inp["x"].shape[0]
    H = inp["H"]
    s_bh = torch.empty(B, H, dtype=torch.float32, device=dev())
    d = {k: inp[k].to(dev()) for k in ("x", "w_qa", "w_qb", "w_kva", "w_kb")}
    s = api.mc_max_logits_mla(d["x"], d["w_qa"], d["w_qb"], d["w_kva"], d["w_kb"], H,
                              inp["nope"], inp["rope"], inp["rope_base"], causal=causal,
                              s_max_bh=s_bh)
    torch.cuda.synchronize()
    return s.cpu().numpy(), s_bh.cpu().numpy(), d


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("dims", [
    dict(B=2, T=200, D=256, H=2, q_lora=128, kv_lora=64),
    dict(B=1, T=520, D=128, H=3, q_lora=192, kv_lora=128),
    dict(B=1, T=257, D=128, H=2, q_lora=128, kv_lora=64),   # one key past a 256-key tile
])
def test_mla_scan_vs_oracle(dims, causal):
    inp = mc_inputs.mla_layer(**dims, n_hot=1, w_std=0.05, seed=31 + dims["T"], causal=causal)
    s, s_bh, _ = _mla(inp, causal)
    ref = oracle.max_logits_mla(inp["x"], inp["w_qa"], inp["w_qb"], inp["w_kva"], inp["w_kb"],
                                inp["H"], inp["nope"], inp["rope"], inp["rope_base"], causal)
    err = rel_err(s_bh, ref)
    assert err.max() < SMAX_RTOL, (err.max(), s_bh, ref)


def test_mla_long_positions_rope():
    """Positions up to 4100: the RoPE table must keep angles accurate."""
    inp = mc_inputs.mla_layer(B=1, T=4100, D=64, H=1, q_lora=64, kv_lora=64, n_hot=0,
                              w_std=0.1, seed=41, heavy_frac=0.01)
    s, s_bh, _ = _mla(inp, True)
    ref = oracle.max_logits_mla(inp["x"], inp["w_qa"], inp["w_qb"], inp["w_kva"], inp["w_kb"],
                                1, 128, 64, inp["rope_base"], True)
    assert rel_err(s_bh, ref).max() < SMAX_RTOL


def test_mla_clip_after_scan():
    lib()
    from muonclip_mc_max_gb300 import api
    inp = mc_inputs.mla_layer(B=1, T=256, D=128, H=4, q_lora=64, kv_lora=64, n_hot=2,
                              hot_scale=30.0, w_std=0.05, seed=43, heavy_frac=0.02)
    s, _, d = _mla(inp, True)
    qb0, kb0 = d["w_qb"].clone(), d["w_kb"].clone()
    g = api.mc_qk_clip_mla(d["w_qb"], d["w_kb"], 4, 128, 64, torch.tensor(s, device=dev()), 10.0)
    torch.cuda.synchronize()
    rqb, rkb, rg = oracle.qk_clip_mla(qb0.cpu(), kb0.cpu(), 4, 128, 64, s, 10.0)
    assert np.array_equal(g.cpu().numpy().view(np.uint32), rg.view(np.uint32))
    assert (rg < 1).any()
    assert np.array_equal(bits16(d["w_qb"]), bits16(rqb))
    assert np.array_equal(bits16(d["w_kb"]), bits16(rkb))
