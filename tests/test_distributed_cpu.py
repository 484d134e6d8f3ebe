"""Data-parallel MuonClip ("Notes on Moonlight", "Distributed Muon"; the
S_max of Kimi K2 section 2.1 as a max over the whole batch) on gloo ranks
on the CPU.

The exchange logic of ``muonclip_mc_max_gb300.distributed`` -- the ZeRO-1
row blocks, the owner map, the int32-key max-all-reduce of S_max, the
reduce-scatter of the gradients, the DP gather to each matrix's owner, the
scatter of O and the clip of the local blocks -- runs here on 2 and 3 gloo
ranks with the arithmetic done by the fp64 oracle (``OracleKernels``
below) instead of the CUDA library.  Checked:

  * S_max on every rank equals the oracle's maximum over the whole batch;
  * each matrix is orthogonalised exactly once, by its owner, and the
    owners cover every matrix;
  * the gathered masters equal, bit for bit, the same code run on one rank
    with the mean gradient, and match the oracle's Muon step followed by
    its clip;
  * NaN, +-inf and -0 survive the key all-reduce.
"""
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LR = 2e-4


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleKernels:
    """The methods of distributed.LibraryKernels on CPU tensors, computed by
    the fp64 oracle (rounded to fp32 where the library stores fp32)."""

    def __init__(self):
        import oracle
        self.oracle = oracle
        self.ns_calls = []

    @staticmethod
    def smax_to_keys(s):
        b = s.detach().numpy().astype(np.float32).view(np.int32).copy()
        neg = b < 0
        b[neg] ^= 0x7FFFFFFF
        b[np.isnan(s.numpy())] = 0x7FFFFFFF
        return torch.from_numpy(b)

    @staticmethod
    def smax_from_keys(keys, out):
        b = keys.numpy().copy()
        neg = b < 0
        b[neg] ^= 0x7FFFFFFF
        out.copy_(torch.from_numpy(b.view(np.float32)))
        return out

    @staticmethod
    def momentum(m, g, u, mu, grad_scale, nesterov):
        gv = (g.double() * grad_scale).float()
        mv = (np.float32(mu) * m.double() + gv.double()).float()
        m.copy_(mv)
        if u is not None:
            u.copy_((np.float32(mu) * mv.double() + gv.double()).float() if nesterov else mv)

    def newton_schulz(self, ins, outs, steps, coeffs, eps):
        for a, o in zip(ins, outs):
            self.ns_calls.append(tuple(a.shape))
            o.copy_(torch.from_numpy(self.oracle.newton_schulz(a, steps, coeffs, eps)).float())

    @staticmethod
    def apply(w, o, rows, cols, lr, rms, wd):
        scale = rms * np.sqrt(max(rows, cols))
        w.copy_((w.double() - lr * (scale * o.double() + wd * w.double())).float())

    def max_logits_mha(self, x, wq, wk, H, dh, causal):
        s = self.oracle.max_logits_mha(x, wq, wk, H, dh, causal).max(0)
        return torch.from_numpy(s.astype(np.float32))

    def max_logits_mla(self, x, w_qa, w_qb, w_kva, w_kb, H, nope, rope, rope_base, causal):
        s = self.oracle.max_logits_mla(x, w_qa, w_qb, w_kva, w_kb, H, nope, rope, rope_base, causal)
        return torch.from_numpy(s.max(0).astype(np.float32))

    def qk_clip_mha(self, wq, wk, H, dh, s_max, tau):
        rq, rk, g = self.oracle.qk_clip_mha(wq, wk, H, dh, s_max.numpy(), tau)
        wq.copy_(rq)
        wk.copy_(rk)
        return torch.from_numpy(g)

    def qk_clip_mla(self, w_qb, w_kb, H, nope, rope, s_max, tau):
        rq, rk, g = self.oracle.qk_clip_mla(w_qb, w_kb, H, nope, rope, s_max.numpy(), tau)
        w_qb.copy_(rq)
        w_kb.copy_(rk)
        return torch.from_numpy(g)


def _layer(kind, world):
    """The seeded layer shared by every rank, and every rank's gradients."""
    import mc_inputs
    if kind == "mha":
        # 47 rows: ragged ZeRO-1 blocks on 2 and 3 ranks
        inp = mc_inputs.mha_layer(B=world, T=7, D=47, H=3, dh=4, n_hot=1, hot_scale=6.0,
                                  w_std=0.15, seed=71)
        inp["tau"] = 10.0
        names = ("wq", "wk")
    else:
        inp = mc_inputs.mla_layer(B=world, T=6, D=16, H=2, q_lora=12, kv_lora=10, nope=4, rope=4,
                                  n_hot=1, hot_scale=5.0, w_std=0.3, seed=73, muon=True)
        inp["tau"] = 10.0
        names = ("w_qa", "w_qb", "w_kva", "w_kb")
    shapes = [tuple(inp[n].shape) for n in names]
    # gradients on a grid of 2^-8 so that their sum over ranks is exact in
    # fp32 whatever order the reduce-scatter adds them in
    g = torch.Generator().manual_seed(1234)
    grads = [[torch.randint(-512, 512, s, generator=g).float() / 256 for s in shapes]
             for _ in range(world)]
    return inp, grads


def _mean(grads, i, world):
    """The mean gradient as the reduce-scatter path forms it: the fp32 sum
    (exact here) times 1/world, rounded once to fp32."""
    return (sum(g[i] for g in grads).double() * (1.0 / world)).float()


def _run_rank(rank, world, port, kind, out_dir, mean_grads_world1):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    from muonclip_mc_max_gb300.distributed import (DistributedMuon, distributed_muonclip_step_mha,
                                                   distributed_muonclip_step_mla)
    from test_distributed_cpu import OracleKernels, _layer, _mean
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        layers = mean_grads_world1 or world
        inp, grads = _layer(kind, layers)
        if mean_grads_world1:
            # one rank standing in for `layers` ranks: the whole batch and the
            # mean gradient, summed and scaled as the reduce-scatter path does
            my_grads = [_mean(grads, i, layers) for i in range(len(grads[0]))]
            x = inp["x"]
        else:
            my_grads = grads[rank]
            x = inp["x"][rank:rank + 1]
        k = OracleKernels()
        opt = DistributedMuon([t.clone() for t in inp["w_master"]],
                              [t.clone() for t in inp["m_prev"]], lr=LR, kernels=k)
        if kind == "mha":
            s, gam = distributed_muonclip_step_mha(opt, x, inp["wq"], inp["wk"], inp["H"], inp["dh"],
                                                   my_grads, inp["tau"])
        else:
            s, gam = distributed_muonclip_step_mla(opt, x, inp["w_qa"], inp["w_qb"], inp["w_kva"],
                                                   inp["w_kb"], inp["H"], inp["nope"], inp["rope"],
                                                   inp["rope_base"], my_grads, inp["tau"])
        full = [opt.gather_params(i) for i in range(len(opt.mats))]
        res = {"s_max": s.numpy().view(np.uint32).tolist(), "gamma": gam.numpy().view(np.uint32).tolist(),
               "owned": opt.owned, "ns_calls": len(k.ns_calls),
               "w": [t.numpy().view(np.uint32).ravel().tolist() for t in full]}
        tag = f"w{world}" + ("m" if mean_grads_world1 else "")
        with open(os.path.join(out_dir, f"{kind}_{tag}_r{rank}.json"), "w") as f:
            json.dump(res, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _spawn(world, kind, out_dir, mean_grads_world1=0):
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_run_rank, args=(r, world, port, kind, out_dir, mean_grads_world1))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    tag = f"w{world}" + ("m" if mean_grads_world1 else "")
    out = []
    for r in range(world):
        with open(os.path.join(out_dir, f"{kind}_{tag}_r{r}.json")) as f:
            out.append(json.load(f))
    return out


@pytest.mark.parametrize("kind,world", [("mha", 2), ("mha", 3), ("mla", 2)])
def test_distributed_muonclip_on_gloo_ranks(tmp_path, kind, world):
    sys.path.insert(0, ROOT)
    import oracle
    ranks = _spawn(world, kind, str(tmp_path))
    one = _spawn(1, kind, str(tmp_path), mean_grads_world1=world)[0]
    inp, grads = _layer(kind, world)
    n_mats = len(inp["w_master"])
    # owners: every matrix exactly once, one Newton-Schulz per owned matrix
    owned = sorted(i for r in ranks for i in r["owned"])
    assert owned == list(range(n_mats))
    assert all(r["ns_calls"] == len(r["owned"]) for r in ranks)
    assert one["ns_calls"] == n_mats
    # S_max: the max over the whole batch on every rank
    if kind == "mha":
        ref_s = oracle.max_logits_mha(inp["x"], inp["wq"], inp["wk"], inp["H"], inp["dh"]).max(0)
    else:
        ref_s = oracle.max_logits_mla(inp["x"], inp["w_qa"], inp["w_qb"], inp["w_kva"], inp["w_kb"],
                                      inp["H"], inp["nope"], inp["rope"], inp["rope_base"],
                                      True).max(0)
    for r in ranks:
        assert r["s_max"] == ranks[0]["s_max"] == one["s_max"]
        assert r["gamma"] == ranks[0]["gamma"] == one["gamma"]
    s = np.array(ranks[0]["s_max"], dtype=np.uint32).view(np.float32)
    assert np.array_equal(s, ref_s.astype(np.float32))
    g = np.array(ranks[0]["gamma"], dtype=np.uint32).view(np.float32)
    assert (g < 1).any() and (g == 1).any(), g  # some heads clip, some do not
    # the gathered masters: identical on every rank and to the one-rank run
    for i in range(n_mats):
        for r in ranks:
            assert r["w"][i] == one["w"][i], (kind, world, i)
    # and the oracle's own composition: Muon with the mean gradient, then
    # the clip with the whole batch's S_max
    names_clip = (0, 1) if kind == "mha" else (1, 3)
    w_ref = []
    for i in range(n_mats):
        rw, _, _ = oracle.muon_step(inp["w_master"][i], _mean(grads, i, world), inp["m_prev"][i],
                                    lr=LR)
        w_ref.append(rw.astype(np.float32))
    a, b = names_clip
    if kind == "mha":
        ra, rb, _ = oracle.qk_clip_mha(w_ref[a], w_ref[b], inp["H"], inp["dh"], s, inp["tau"])
    else:
        ra, rb, _ = oracle.qk_clip_mla(w_ref[a], w_ref[b], inp["H"], inp["nope"], inp["rope"], s,
                                       inp["tau"])
    w_ref[a], w_ref[b] = ra.numpy(), rb.numpy()
    for i in range(n_mats):
        got = np.array(ranks[0]["w"][i], dtype=np.uint32).view(np.float32).reshape(w_ref[i].shape)
        w0 = inp["w_master"][i].double().numpy()
        d_got, d_ref = got.astype(np.float64) - w0, w_ref[i].astype(np.float64) - w0
        assert np.linalg.norm(d_got - d_ref) <= 1e-5 * np.linalg.norm(d_ref) + 1e-12, (kind, i)


def _keys_rank(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    from muonclip_mc_max_gb300.distributed import allreduce_smax
    from test_distributed_cpu import OracleKernels
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        vals = [[float("nan"), -3.0, -0.0, 5.0, float("-inf"), 1e-40],
                [2.0, -7.0, 0.0, float("inf"), -1.0, -1e-40]][rank]
        s = torch.tensor(vals, dtype=torch.float32)
        allreduce_smax(s, kernels=OracleKernels())
        with open(os.path.join(out_dir, f"keys_r{rank}.json"), "w") as f:
            json.dump(s.numpy().view(np.uint32).tolist(), f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_smax_key_allreduce_keeps_nan_inf_and_signed_zero(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_keys_rank, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = []
    for r in range(2):
        with open(os.path.join(tmp_path, f"keys_r{r}.json")) as f:
            res.append(np.array(json.load(f), dtype=np.uint32).view(np.float32))
    assert np.array_equal(res[0].view(np.uint32), res[1].view(np.uint32))
    s = res[0]
    assert np.isnan(s[0])
    assert s[1] == -3.0 and s[3] == np.inf and s[4] == -1.0
    assert s[2] == 0.0 and not np.signbit(s[2])       # max(-0, +0) is +0
    assert s[5] == np.float32(1e-40)                  # subnormals keep their order


def test_owner_map_balances_cost():
    sys.path.insert(0, ROOT)
    from muonclip_mc_max_gb300.distributed import assign_owners, block_rows, ns_cost, shard_range
    shapes = [(7168, 2048)] * 48 + [(2048, 7168)] * 48
    own = assign_owners(shapes, 8)
    assert [own.count(r) for r in range(8)] == [12] * 8
    mixed = [(7168, 1536), (1536, 12288), (7168, 576), (512, 8192)]
    own = assign_owners(mixed, 2)
    load = [sum(ns_cost(*mixed[i]) for i in range(4) if own[i] == r) for r in range(2)]
    assert max(load) == max(ns_cost(*s) for s in mixed)  # the largest alone, the rest together
    assert block_rows(45, 2) == 23 and shard_range(45, 2, 1) == (23, 45)
    assert shard_range(2, 3, 2) == (2, 2)  # an empty block on the last rank
