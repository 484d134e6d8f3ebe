"""Parity at the full workload sizes, in the launch configurations bench.py
times: the CUDA path runs the whole workload, the fp64 oracle (its
library-GEMM restatement) recomputes sampled outputs one by one, and
properties that hold at any size cover the rest.

  MHA layer   x [8,1024,1024], 16 heads of 64: S_max of every head of two
              sequences and one rotating head of each other sequence, gamma
              and the clip bit-exact, both Muon matrices.
  K2 MLA      x [16,4096,7168] causal: every head of two sequences and one
              rotating head of each of the other 14.
  expert batch 96 matrices of 7168x2048 / 2048x7168: eight matrices (four
              tall, four wide) against the oracle, every matrix's update
              RMS checked.
  long MLA    x [1,32768,7168] causal + heavy rows: the 8 planted heads and
              8 cold ones, the MLA clip bit-exact, Muon on W_kva and W_kb
              against the oracle.
  attention   the forwards of the three attention workloads ([8,1024,16x64],
              [2,8192,16x128] causal, MLA [2,8192,64 heads] causal): O of
              four (sequence, head) pairs element by element and
              S_max of their heads.
"""
import gc

import numpy as np
import pytest
import torch

import mc_inputs
import oracle
from gpu_helpers import NS_RTOL, SMAX_RTOL, bits16, dev, lib, rel_err, rel_fro

pytestmark = pytest.mark.gpu


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def _phi5_band():
    a, b, c = oracle.NS_COEFFS
    s = np.linspace(1e-4, 1.0, 20001)
    for _ in range(5):
        s = a * s + b * s ** 3 + c * s ** 5
    return s.min(), s.max()


def test_mha_layer_fullsize():
    lib()
    from muonclip_mc_max_gb300 import api
    inp = mc_inputs.c2(device=dev())
    H, dh, B = inp["H"], inp["dh"], 8
    x, wq, wk = inp["x"], inp["wq"], inp["wk"]
    s_bh = torch.empty(B, H, dtype=torch.float32, device=dev())
    s = api.mc_max_logits_mha(x, wq, wk, H, dh, s_max_bh=s_bh)
    torch.cuda.synchronize()
    # every head of two sequences (the first and the last scheduling band)
    ref = oracle.max_logits_mha_np(x.cpu(), wq.cpu(), wk.cpu(), H, dh, False, batches=[0, 7])
    got = s_bh.cpu().numpy()[[0, 7]]
    assert rel_err(got, ref).max() < SMAX_RTOL
    # and one head of every other sequence, rotating through the heads
    for b in range(1, 7):
        h = (5 * b) % H
        ref = oracle.max_logits_mha_np(x.cpu(), wq.cpu(), wk.cpu(), H, dh, False, heads=[h],
                                       batches=[b])
        assert rel_err(s_bh.cpu().numpy()[b, h], ref[0, 0]) < SMAX_RTOL, (b, h)
    assert np.array_equal(s.cpu().numpy(), s_bh.cpu().numpy().max(0))
    # Muon on both 1024 x 1024 masters
    w0 = [t.cpu() for t in inp["w_master"]]
    masters = [t.clone() for t in inp["w_master"]]
    moms = [t.clone() for t in inp["m_prev"]]
    api.mc_muon_step(masters, inp["grad"], moms, lr=mc_inputs.LR)
    torch.cuda.synchronize()
    for i in range(2):
        rw, rm, _ = oracle.muon_step_np(w0[i], inp["grad"][i].cpu(), inp["m_prev"][i].cpu(),
                                        lr=mc_inputs.LR)
        assert rel_fro(moms[i].cpu().numpy(), rm) < 1e-6
        d_gpu = masters[i].cpu().double().numpy() - w0[i].double().numpy()
        assert rel_fro(d_gpu, rw - w0[i].double().numpy()) < NS_RTOL
    # clip of the layer's bf16 weights with the GPU's S_max: bit-exact
    s_np = s.cpu().numpy()
    wq0, wk0 = wq.cpu().clone(), wk.cpu().clone()
    g = api.mc_qk_clip_mha(wq, wk, H, dh, s, inp["tau"])
    torch.cuda.synchronize()
    rq, rk, rg = oracle.qk_clip_mha(wq0, wk0, H, dh, s_np, inp["tau"])
    assert np.array_equal(g.cpu().numpy().view(np.uint32), rg.view(np.uint32))
    assert (rg < 1).sum() == len(inp["hot"])
    assert np.array_equal(bits16(wq), bits16(rq)) and np.array_equal(bits16(wk), bits16(rk))
    del inp, x, wq, wk, masters, moms
    _free()


def test_k2_mla_layer_fullsize():
    lib()
    from muonclip_mc_max_gb300 import api
    inp = mc_inputs.c3(device=dev())
    H, B = inp["H"], 16
    d = {k: inp[k] for k in ("x", "w_qa", "w_qb", "w_kva", "w_kb")}
    s_bh = torch.empty(B, H, dtype=torch.float32, device=dev())
    api.mc_max_logits_mla(d["x"], d["w_qa"], d["w_qb"], d["w_kva"], d["w_kb"], H, 128, 64,
                          inp["rope_base"], causal=True, s_max_bh=s_bh)
    torch.cuda.synchronize()
    got_all = s_bh.cpu().numpy()
    w = [d[k].cpu() for k in ("w_qa", "w_qb", "w_kva", "w_kb")]
    x_cpu = d["x"].cpu()
    # every head of two sequences (first and last scheduling band)
    for b in (0, 15):
        ref = oracle.max_logits_mla_np(x_cpu[b:b + 1], *w, H, 128, 64, inp["rope_base"], True)
        assert rel_err(got_all[b:b + 1], ref).max() < SMAX_RTOL, b
    # one head of every other sequence, rotating through the heads (hot ones included)
    for b in range(1, 15):
        h = inp["hot"][b % len(inp["hot"])] if b % 4 == 0 else (9 * b + 1) % H
        ref = oracle.max_logits_mla_np(x_cpu[b:b + 1], *w, H, 128, 64, inp["rope_base"], True,
                                       heads=[h])
        assert rel_err(got_all[b, h], ref[0, 0]) < SMAX_RTOL, (b, h)
    assert api.mc_read_device_status(clear=True) == 0
    del inp, d, s_bh
    _free()


def test_expert_batch_fullsize():
    lib()
    from muonclip_mc_max_gb300 import api
    inp = mc_inputs.c4(device=dev())
    # four tall (7168 x 2048) and four wide (2048 x 7168) matrices, spread
    # over the batch and so over the tiles and phases of the launch
    picks = [0, 17, 31, 47, 48, 63, 80, 95]
    w0 = {i: inp["w"][i].cpu() for i in picks}
    m0 = {i: inp["m_prev"][i].cpu() for i in picks + [1, 50]}
    wcopy = [t.clone() for t in inp["w"]]
    api.mc_muon_step(inp["w"], inp["grad"], inp["m_prev"], lr=mc_inputs.LR)
    torch.cuda.synchronize()
    for i in picks:
        rw, rm, _ = oracle.muon_step_np(w0[i], inp["grad"][i].cpu(), m0[i], lr=mc_inputs.LR)
        assert rel_fro(inp["m_prev"][i].cpu().numpy(), rm) < 1e-6
        d_gpu = inp["w"][i].cpu().double().numpy() - w0[i].double().numpy()
        assert rel_fro(d_gpu, rw - w0[i].double().numpy()) < NS_RTOL
    # momentum of other matrices: mu M + G in fp32 (one fma rounding)
    for i in (1, 50):
        ref = 0.95 * m0[i].double() + inp["grad"][i].cpu().double()
        assert rel_fro(inp["m_prev"][i].cpu().numpy(), ref.numpy()) < 1e-6
    # every matrix: finite, and the orthogonalised part of the update has the
    # RMS the lemma gives for singular values inside the phi^5 band
    lo, hi = _phi5_band()
    for i in range(96):
        w_new = inp["w"][i]
        assert bool(torch.isfinite(w_new).all())
        o = (wcopy[i] * (1 - mc_inputs.LR * mc_inputs.WD) - w_new).double() / (
            mc_inputs.LR * mc_inputs.RMS * np.sqrt(7168))
        rms_o = float(o.pow(2).mean().sqrt()) * np.sqrt(7168)  # = sqrt(sum s_i^2 / 2048)
        assert lo * 0.95 <= rms_o <= hi * 1.05, (i, rms_o)
    del inp, wcopy
    _free()


def test_long_mla_fullsize():
    lib()
    from muonclip_mc_max_gb300 import api
    inp = mc_inputs.c5(device=dev())
    H = inp["H"]
    d = {k: inp[k] for k in ("x", "w_qa", "w_qb", "w_kva", "w_kb")}
    s_bh = torch.empty(1, H, dtype=torch.float32, device=dev())
    s = api.mc_max_logits_mla(d["x"], d["w_qa"], d["w_qb"], d["w_kva"], d["w_kb"], H, 128, 64,
                              inp["rope_base"], causal=True, s_max_bh=s_bh)
    torch.cuda.synchronize()
    # all 8 planted heads and 8 cold ones spread over the head range
    cold = [h for h in range(H) if h not in inp["hot"]][::7][:8]
    heads = inp["hot"] + cold
    assert len(heads) == 16
    ref = oracle.max_logits_mla_np(d["x"].cpu(), d["w_qa"].cpu(), d["w_qb"].cpu(),
                                   d["w_kva"].cpu(), d["w_kb"].cpu(), H, 128, 64,
                                   inp["rope_base"], True, heads=heads)
    got = s_bh.cpu().numpy()[:, heads]
    assert rel_err(got, ref).max() < SMAX_RTOL, (got, ref)
    s_np = s.cpu().numpy()
    assert (s_np > inp["tau"]).sum() >= len(inp["hot"])  # the planted heads clip
    # MLA clip of the bf16 weights with the GPU's S_max: bit-exact
    qb0, kb0, kva0 = d["w_qb"].cpu(), d["w_kb"].cpu(), d["w_kva"].cpu()
    g = api.mc_qk_clip_mla(d["w_qb"], d["w_kb"], H, 128, 64, s, inp["tau"])
    torch.cuda.synchronize()
    rqb, rkb, rg = oracle.qk_clip_mla(qb0, kb0, H, 128, 64, s_np, inp["tau"])
    assert np.array_equal(g.cpu().numpy().view(np.uint32), rg.view(np.uint32))
    assert np.array_equal(bits16(d["w_qb"]), bits16(rqb))
    assert np.array_equal(bits16(d["w_kb"]), bits16(rkb))
    assert torch.equal(d["w_kva"].cpu(), kva0)
    # Muon on the layer's four projections; W_kva and W_kb against the oracle
    w0 = [t.cpu() for t in inp["w_master"]]
    m0 = [t.cpu() for t in inp["m_prev"]]
    api.mc_muon_step(inp["w_master"], inp["grad"], inp["m_prev"], lr=mc_inputs.LR)
    torch.cuda.synchronize()
    for i in (2, 3):
        rw, rm, _ = oracle.muon_step_np(w0[i], inp["grad"][i].cpu(), m0[i], lr=mc_inputs.LR)
        assert rel_fro(inp["m_prev"][i].cpu().numpy(), rm) < 1e-6
        d_gpu = inp["w_master"][i].cpu().double().numpy() - w0[i].double().numpy()
        assert rel_fro(d_gpu, rw - w0[i].double().numpy()) < NS_RTOL
    for t in inp["w_master"]:
        assert bool(torch.isfinite(t).all())
    assert api.mc_read_device_status(clear=True) == 0
    del inp, d
    _free()


def _attn_check(o_dev, v_cols, s_max_h, o_ref, s_ref_b):
    """o_dev [T, d] of one (sequence, head) against the oracle's o_ref
    [T, d] (bounds of the attention tests: P and O each rounded once to
    bf16); s_max_h against the max of the oracle's per-sequence maxima."""
    got = o_dev.double().numpy()
    vmax = np.abs(v_cols.double().numpy()).max()
    tol = 2.0 ** -8 * vmax + 2.0 ** -8 * np.abs(o_ref)
    bad = np.abs(got - o_ref) > tol
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} outputs off; max err {np.abs(got - o_ref).max()}"
    ref = max(s_ref_b)
    assert abs(s_max_h - ref) / abs(ref) < 1e-4, (s_max_h, ref)


@pytest.mark.parametrize("name,picks", [
    ("attn", [(0, 0), (7, 15), (3, 8), (5, 3)]),   # [8, 1024, 16 x 64] non-causal
    ("attnl", [(1, 5), (0, 12), (0, 0), (1, 15)]),  # [2, 8192, 16 x 128] causal
])
def test_attention_mha_fullsize(name, picks):
    """The attention forward of the bench's MHA workloads in the bench's
    launch: O of the picked (sequence, head) pairs element by element and
    S_max of their heads (every sequence of the head) against the oracle."""
    lib()
    import bench
    from muonclip_mc_max_gb300 import api
    wl = bench.AttnLayer(name)
    s = wl.make(dev())
    wl.step_part(s, api, "scan")
    torch.cuda.synchronize()
    assert api.mc_read_device_status(clear=True) == 0
    H, dh, B = wl.H, wl.dh, wl.B
    q, k, v = s["q"].cpu(), s["k"].cpu(), s["v"].cpu()
    o, s_max = s["o"].cpu(), s["s_max"].cpu().numpy()
    del s
    _free()
    for b, h in picks:
        cols = slice(h * dh, (h + 1) * dh)
        hq, hk, hv = (t[:, :, cols].contiguous() for t in (q, k, v))
        o_ref, s_ref = oracle.attention_mha_np(hq, hk, hv, 1, dh, wl.causal, batches=range(B), heads=[0])
        _attn_check(o[b, :, cols], hv[b], s_max[h], o_ref[b, :, 0], s_ref[:, 0])


def test_attention_mla_fullsize():
    """The K2-shaped MLA attention forward of the bench ([2, 8192], 64 heads,
    causal) in the bench's launch: O of four (sequence, head) pairs and S_max
    of their heads against the oracle."""
    lib()
    import bench
    from muonclip_mc_max_gb300 import api
    wl = bench.AttnMlaLayer()
    s = wl.make(dev())
    wl.step_part(s, api, "scan")
    torch.cuda.synchronize()
    assert api.mc_read_device_status(clear=True) == 0
    H, B = wl.H, wl.B
    q, kc, kr, v = s["q"].cpu(), s["k_c"].cpu(), s["k_r"].cpu(), s["v"].cpu()
    o, s_max = s["o"].cpu(), s["s_max"].cpu().numpy()
    del s
    _free()
    for b, h in [(0, 37), (1, 2), (0, 0), (1, 63)]:
        hq = q[:, :, h * 192:(h + 1) * 192].contiguous()
        hkc = kc[:, :, h * 128:(h + 1) * 128].contiguous()
        hv = v[:, :, h * 128:(h + 1) * 128].contiguous()
        o_ref, s_ref = oracle.attention_mla_np(hq, hkc, kr, hv, 1, 128, 64, 128, True, batches=range(B),
                                               heads=[0])
        _attn_check(o[b, :, h * 128:(h + 1) * 128], hv[b], s_max[h], o_ref[b, :, 0], s_ref[:, 0])
