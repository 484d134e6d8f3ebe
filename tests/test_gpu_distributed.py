"""The library kernels behind the data-parallel MuonClip step, on the GPU.

  * S_max <-> int32 keys: the keys order like the floats (NaN largest, -0
    below +0, subnormals and infinities in place) and decode bit for bit;
  * momentum and update on flat shards reproduce mc_muon_step bit for bit
    when composed with mc_newton_schulz (plain and Nesterov momentum, 16-byte
    vectors and the element-by-element tail);
  * the ZeRO-1 step of ``distributed`` on one NCCL rank reproduces the
    single-GPU composed MuonClip step (MHA and MLA) bit for bit.  Runs with
    more ranks need more GPUs than one call here has; the exchange logic on
    2 and 3 ranks is covered on the CPU (test_distributed_cpu.py).
"""
import socket

import numpy as np
import pytest
import torch

import mc_inputs
from gpu_helpers import dev, lib

pytestmark = pytest.mark.gpu

LR = mc_inputs.LR


def _u32(t):
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


def _ref_keys(s: np.ndarray) -> np.ndarray:
    b = s.astype(np.float32).view(np.int32).copy()
    b[b < 0] ^= 0x7FFFFFFF
    b[np.isnan(s)] = 0x7FFFFFFF
    return b


def test_smax_keys_order_and_round_trip():
    lib()
    from muonclip_mc_max_gb300 import api
    g = torch.Generator().manual_seed(5)
    vals = torch.cat([torch.randn(1000, generator=g) * 1e3,
                      torch.tensor([float("nan"), float("inf"), float("-inf"), 0.0, -0.0, 1e-42,
                                    -1e-42, 3.4e38, -3.4e38, 1.0, -1.0])]).float()
    s = vals.to(dev())
    keys = api.mc_smax_to_keys(s)
    back = api.mc_smax_from_keys(keys)
    torch.cuda.synchronize()
    k = keys.cpu().numpy()
    v = vals.numpy()
    assert np.array_equal(k, _ref_keys(v))
    fin = ~np.isnan(v)
    vf = v[fin]
    order = np.lexsort((~np.signbit(vf), vf))  # by value, -0 before +0
    assert (np.diff(k[fin][order]) > 0).all()
    assert (k[~fin] == 0x7FFFFFFF).all() and (k[fin] < 0x7FFFFFFF).all()
    b = back.cpu().numpy()
    assert np.array_equal(b[fin].view(np.uint32), v[fin].view(np.uint32))
    assert np.isnan(b[~fin]).all()


@pytest.mark.parametrize("nesterov", [False, True])
@pytest.mark.parametrize("shape", [(256, 192), (130, 77)])  # float4 path; odd width (scalar tail)
def test_flat_shard_passes_match_muon_step(shape, nesterov):
    lib()
    from muonclip_mc_max_gb300 import api
    rows, cols = shape
    w0 = mc_inputs.matrix(rows, cols, seed=11, std=0.02).to(dev())
    m0 = mc_inputs.matrix(rows, cols, seed=12, std=1e-3).to(dev())
    g0 = mc_inputs.matrix(rows, cols, seed=13, std=1e-3).to(dev())
    # whole-matrix step
    w1, m1 = w0.clone(), m0.clone()
    api.mc_muon_step([w1], [g0], [m1], lr=LR, nesterov=nesterov)
    # flat passes around a stand-alone Newton-Schulz
    w2, m2 = w0.clone(), m0.clone()
    u = torch.empty_like(m2)
    api.mc_muon_momentum(m2, g0, u, mu=mc_inputs.MU, grad_scale=1.0, nesterov=nesterov)
    o = api.mc_newton_schulz([u])[0]
    api.mc_muon_apply(w2, o, rows, cols, LR, rms=mc_inputs.RMS, wd=mc_inputs.WD)
    torch.cuda.synchronize()
    assert np.array_equal(_u32(m1), _u32(m2))
    assert np.array_equal(_u32(w1), _u32(w2))
    # an unaligned shard (offset by one element) takes the scalar path
    w3, m3 = w0.clone().view(-1), m0.clone().view(-1)
    api.mc_muon_momentum(m3[1:], g0.view(-1)[1:], None, mu=mc_inputs.MU)
    api.mc_muon_apply(w3[1:], o.view(-1)[1:], rows, cols, LR)
    torch.cuda.synchronize()
    assert np.array_equal(_u32(m3[1:]), _u32(m2.view(-1)[1:]))
    assert np.array_equal(_u32(w3[1:]), _u32(w2.view(-1)[1:]))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.fixture
def one_rank_group():
    import torch.distributed as dist
    if dist.is_initialized():
        pytest.skip("a process group is already initialised")
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0,
                            world_size=1)
    try:
        yield
    finally:
        dist.destroy_process_group()


def test_distributed_step_mha_one_rank_matches_single_gpu(one_rank_group):
    lib()
    from muonclip_mc_max_gb300 import muonclip_step_mha
    from muonclip_mc_max_gb300.distributed import DistributedMuon, distributed_muonclip_step_mha
    inp = mc_inputs.mha_layer(B=2, T=300, D=192, H=4, dh=64, n_hot=2, w_std=0.05, seed=21)
    x, wq, wk = (inp[k].to(dev()) for k in ("x", "wq", "wk"))
    grads = [t.to(dev()) for t in inp["grad"]]
    masters = [t.to(dev()).clone() for t in inp["w_master"]]
    moms = [t.to(dev()).clone() for t in inp["m_prev"]]
    s1, g1 = muonclip_step_mha(x, wq, wk, 4, 64, masters, grads, moms, lr=LR, tau=inp["tau"])
    opt = DistributedMuon([t.to(dev()) for t in inp["w_master"]], [t.to(dev()) for t in inp["m_prev"]],
                          lr=LR)
    s2, g2 = distributed_muonclip_step_mha(opt, x, wq, wk, 4, 64, grads, inp["tau"])
    torch.cuda.synchronize()
    assert (g1.cpu() < 1).sum() == 2
    assert np.array_equal(_u32(s1), _u32(s2)) and np.array_equal(_u32(g1), _u32(g2))
    for i in range(2):
        assert np.array_equal(_u32(masters[i]), _u32(opt.gather_params(i))), i
        assert np.array_equal(_u32(moms[i]), _u32(opt.mats[i].m)), i
    from muonclip_mc_max_gb300 import api
    assert api.mc_read_device_status(clear=True) == 0


def test_distributed_step_mla_one_rank_matches_single_gpu(one_rank_group):
    lib()
    from muonclip_mc_max_gb300 import muonclip_step_mla
    from muonclip_mc_max_gb300.distributed import DistributedMuon, distributed_muonclip_step_mla
    inp = mc_inputs.c3b(B=1, T=520, D=256, H=4, q_lora=128, kv_lora=64, w_std=0.035, n_hot=2,
                        heavy_frac=0.02, muon=True)
    names = ("x", "w_qa", "w_qb", "w_kva", "w_kb")
    d = {k: inp[k].to(dev()) for k in names}
    grads = [t.to(dev()) for t in inp["grad"]]
    masters = [t.to(dev()).clone() for t in inp["w_master"]]
    moms = [t.to(dev()).clone() for t in inp["m_prev"]]
    args = (d["x"], d["w_qa"], d["w_qb"], d["w_kva"], d["w_kb"], 4, 128, 64, inp["rope_base"])
    s1, g1 = muonclip_step_mla(*args, masters, grads, moms, lr=LR, tau=inp["tau"])
    opt = DistributedMuon([t.to(dev()) for t in inp["w_master"]], [t.to(dev()) for t in inp["m_prev"]],
                          lr=LR)
    s2, g2 = distributed_muonclip_step_mla(opt, *args, grads, inp["tau"])
    torch.cuda.synchronize()
    assert (g1.cpu() < 1).any() and (g1.cpu() == 1).any()
    assert np.array_equal(_u32(s1), _u32(s2)) and np.array_equal(_u32(g1), _u32(g2))
    for i in range(4):
        assert np.array_equal(_u32(masters[i]), _u32(opt.gather_params(i))), i
