"""Data-parallel MuonClip: Distributed Muon over ZeRO-1 shards and the
per-head max logit over ranks.

"Notes on Moonlight", section "Distributed Muon": ZeRO-1 partitions the
optimizer state across the data-parallel (DP) ranks; Muon, which needs the
whole matrix, adds a DP gather of the partitions and a full Newton-Schulz
update on the gathered matrix.  Kimi K2 section 2.1 (S_max equation): the
max logit of a head is a max over every X of the global batch, so each rank
scans its own micro-batch and the ranks combine their maxima.

Layout.  Matrix i of shape [rows_i, cols_i] is cut into ``world`` blocks of
``ceil(rows_i / world)`` whole rows; rank r holds block r of the fp32 master
W_i and momentum M_i, zero-padded past the last row.  A block of whole rows
holds every column of every head, so momentum, the update and QK-Clip run
on it unchanged.

One step on rank r (every arithmetic step is a library kernel; this module
only sequences them and issues the collectives):

  1. S_max:   the scan of this rank's micro-batch -> s_max[H]; encoded as
              order-preserving int32 keys (NaN largest), all_reduce(MAX),
              decoded: every rank holds the global per-head maximum.
  2. grads:   reduce_scatter(SUM) of each full local gradient; the momentum
              kernel scales the sum by 1/world (the mean gradient).
  3. momentum on the local block: M_r <- mu M_r + G_r.
  4. DP gather: the owner of matrix i gathers the blocks of its
              Newton-Schulz input into the full matrix.
  5. full update: the owner runs Newton-Schulz on its matrices (one batched
              call), so every matrix is orthogonalised exactly once.
  6. scatter: the owner returns block r of O_i to rank r, which applies
              W_r <- W_r - lr (0.2 sqrt(max(A, B)) O_r + wd W_r).
  7. QK-Clip of the local blocks of W_q / W_k (MLA: W_qb / W_kb) with the
              global gamma (padding rows are zero and stay zero throughout).
  8. ``gather_params`` all-gathers the blocks into full matrices for the
              next forward (ZeRO-1's parameter all-gather).

Owners: matrices are dealt in decreasing Newton-Schulz cost to the rank
with the least work so far (ties to the lower rank), which is round-robin
for equal shapes.  Moonlight's own description gathers the full matrix on
every rank and computes the update redundantly; giving each matrix one
owner computes it once and sends each rank only its block of O back.

Where several ranks share one GPU nothing here waits on another rank
inside a kernel: each collective is a separate NCCL (or gloo) call between
library launches.

``kernels`` is the CUDA library binding by default.  Tests pass an object
with the same methods to run the exchange logic on CPU ranks.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.distributed as dist

from .api import NS_COEFFS


# ---------------------------------------------------------------------------
# partitioning
# ---------------------------------------------------------------------------

def block_rows(rows: int, world: int) -> int:
    """Rows per ZeRO-1 block (every rank's block has this many, padded)."""
    return -(-rows // world)


def shard_range(rows: int, world: int, rank: int) -> tuple[int, int]:
    """[r0, r1) of the real rows in rank ``rank``'s block (may be empty)."""
    rp = block_rows(rows, world)
    r0 = min(rows, rank * rp)
    return r0, min(rows, r0 + rp)


def ns_cost(rows: int, cols: int) -> int:
    """Algorithmic flops of one quintic iteration on a rows x cols matrix
    (m = min, n = max): Gram m(m+1)n, A A m^2(m+1), B X 2 m^2 n."""
    m, n = min(rows, cols), max(rows, cols)
    return m * (m + 1) * n + m * m * (m + 1) + 2 * m * m * n


def assign_owners(shapes, world: int) -> list[int]:
    """Owner rank of each matrix: decreasing cost to the least-loaded rank."""
    load = [0] * world
    owner = [0] * len(shapes)
    order = sorted(range(len(shapes)), key=lambda i: (-ns_cost(*shapes[i]), i))
    for i in order:
        r = min(range(world), key=lambda k: (load[k], k))
        owner[i] = r
        load[r] += ns_cost(*shapes[i])
    return owner


# ---------------------------------------------------------------------------
# the library kernels this module sequences
# ---------------------------------------------------------------------------

class LibraryKernels:
    """The CUDA library (``api``) behind the exchange."""

    def __init__(self):
        from . import api
        self.api = api

    def smax_to_keys(self, s):
        return self.api.mc_smax_to_keys(s)

    def smax_from_keys(self, keys, out):
        return self.api.mc_smax_from_keys(keys, out)

    def momentum(self, m, g, u, mu, grad_scale, nesterov):
        self.api.mc_muon_momentum(m, g, u, mu=mu, grad_scale=grad_scale, nesterov=nesterov)

    def newton_schulz(self, ins, outs, steps, coeffs, eps):
        self.api.mc_newton_schulz(ins, steps=steps, coeffs=coeffs, eps=eps, out=outs)

    def apply(self, w, o, rows, cols, lr, rms, wd):
        self.api.mc_muon_apply(w, o, rows, cols, lr, rms=rms, wd=wd)

    def max_logits_mha(self, x, wq, wk, H, dh, causal):
        return self.api.mc_max_logits_mha(x, wq, wk, H, dh, causal=causal)

    def max_logits_mla(self, x, w_qa, w_qb, w_kva, w_kb, H, nope, rope, rope_base, causal):
        return self.api.mc_max_logits_mla(x, w_qa, w_qb, w_kva, w_kb, H, nope, rope, rope_base,
                                          causal=causal)

    def qk_clip_mha(self, wq, wk, H, dh, s_max, tau):
        return self.api.mc_qk_clip_mha(wq, wk, H, dh, s_max, tau)

    def qk_clip_mla(self, w_qb, w_kb, H, nope, rope, s_max, tau):
        return self.api.mc_qk_clip_mla(w_qb, w_kb, H, nope, rope, s_max, tau)


# ---------------------------------------------------------------------------
# S_max over ranks
# ---------------------------------------------------------------------------

def allreduce_smax(s_max: torch.Tensor, group=None, kernels=None) -> torch.Tensor:
    """Replace this rank's per-head S_max with the maximum over the group's
    ranks (in place; returns it).  NaN on any rank gives NaN everywhere."""
    k = kernels or LibraryKernels()
    keys = k.smax_to_keys(s_max)
    dist.all_reduce(keys, op=dist.ReduceOp.MAX, group=group)
    k.smax_from_keys(keys, s_max)
    return s_max


# ---------------------------------------------------------------------------
# Distributed Muon
# ---------------------------------------------------------------------------

@dataclass
class _Mat:
    rows: int
    cols: int
    owner: int
    rp: int                   # rows per block
    w: torch.Tensor           # [rp, cols] this rank's block of the master
    m: torch.Tensor           # [rp, cols] this rank's block of the momentum
    g: torch.Tensor           # [rp, cols] reduce-scattered gradient block
    u: torch.Tensor | None    # [rp, cols] Nesterov input block (else the momentum is sent)
    o: torch.Tensor           # [rp, cols] this rank's block of O
    full_u: torch.Tensor | None  # owner: [world * rp, cols] gathered input
    full_o: torch.Tensor | None  # owner: [world * rp, cols] Newton-Schulz output
    pad_g: torch.Tensor | None   # [world * rp, cols] padded gradient when rows % world


class DistributedMuon:
    """ZeRO-1 Muon over the ranks of ``group``.

    ``masters`` and ``moms``: the full fp32 matrices (identical on every
    rank at construction); each rank keeps only its own blocks.  The
    hyper-parameters follow ``mc_muon_step``."""

    def __init__(self, masters, moms, group=None, lr=2e-4, mu=0.95, wd=0.1, rms=0.2, steps=5,
                 coeffs=NS_COEFFS, eps=1e-7, nesterov=False, kernels=None):
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.kernels = kernels or LibraryKernels()
        self.lr, self.mu, self.wd, self.rms = lr, mu, wd, rms
        self.steps, self.coeffs, self.eps, self.nesterov = steps, coeffs, eps, nesterov
        shapes = [tuple(t.shape) for t in masters]
        self.owners = assign_owners(shapes, self.world)
        self.mats: list[_Mat] = []
        for i, (wf, mf) in enumerate(zip(masters, moms)):
            rows, cols = shapes[i]
            rp = block_rows(rows, self.world)
            r0, r1 = shard_range(rows, self.world, self.rank)
            dev = wf.device

            def block(full):
                b = torch.zeros((rp, cols), dtype=torch.float32, device=dev)
                b[:r1 - r0].copy_(full[r0:r1])
                return b

            own = self.owners[i] == self.rank
            full_o = torch.zeros((self.world * rp, cols), dtype=torch.float32, device=dev) if own else None
            self.mats.append(_Mat(
                rows=rows, cols=cols, owner=self.owners[i], rp=rp, w=block(wf), m=block(mf),
                g=torch.empty((rp, cols), dtype=torch.float32, device=dev),
                u=torch.empty((rp, cols), dtype=torch.float32, device=dev) if nesterov else None,
                o=torch.empty((rp, cols), dtype=torch.float32, device=dev),
                full_u=torch.zeros_like(full_o) if own else None, full_o=full_o,
                pad_g=torch.zeros((self.world * rp, cols), dtype=torch.float32, device=dev)
                if rows % self.world else None))

    @property
    def owned(self) -> list[int]:
        """Indices of the matrices this rank orthogonalises."""
        return [i for i, r in enumerate(self.owners) if r == self.rank]

    def local_block(self, i: int) -> torch.Tensor:
        """This rank's real rows of master i (a view of its block)."""
        r0, r1 = shard_range(self.mats[i].rows, self.world, self.rank)
        return self.mats[i].w[:r1 - r0]

    def step(self, grads):
        """One Muon step from this rank's full local gradients (summed over
        ranks and scaled to their mean).  Updates this rank's blocks."""
        k, world = self.kernels, self.world
        # 2-3. reduce-scatter of the gradients, momentum on the blocks
        for mat, gf in zip(self.mats, grads):
            src = gf
            if mat.pad_g is not None:
                mat.pad_g[:mat.rows].copy_(gf)
                src = mat.pad_g
            dist.reduce_scatter_tensor(mat.g, src.reshape(world * mat.rp, mat.cols),
                                       op=dist.ReduceOp.SUM, group=self.group)
            k.momentum(mat.m, mat.g, mat.u, self.mu, 1.0 / world, self.nesterov)
        # 4. DP gather of each matrix's Newton-Schulz input to its owner
        for mat in self.mats:
            send = mat.u if self.nesterov else mat.m
            recv = list(mat.full_u.chunk(world)) if mat.full_u is not None else None
            dist.gather(send, recv, dst=self._global(mat.owner), group=self.group)
        # 5. one batched Newton-Schulz over the owned matrices
        own = self.owned
        if own:
            ins = [self.mats[i].full_u[:self.mats[i].rows] for i in own]
            outs = [self.mats[i].full_o[:self.mats[i].rows] for i in own]
            k.newton_schulz(ins, outs, self.steps, self.coeffs, self.eps)
        # 6. scatter of O's blocks and the update of the local blocks
        for mat in self.mats:
            chunks = list(mat.full_o.chunk(world)) if mat.full_o is not None else None
            dist.scatter(mat.o, chunks, src=self._global(mat.owner), group=self.group)
            k.apply(mat.w, mat.o, mat.rows, mat.cols, self.lr, self.rms, self.wd)

    def gather_params(self, i: int, out: torch.Tensor | None = None) -> torch.Tensor:
        """All-gather master i's blocks into the full [rows, cols] matrix."""
        mat = self.mats[i]
        full = torch.empty((self.world * mat.rp, mat.cols), dtype=torch.float32, device=mat.w.device)
        dist.all_gather_into_tensor(full, mat.w, group=self.group)
        if out is None:
            return full[:mat.rows]
        out.copy_(full[:mat.rows])
        return out

    def _global(self, group_rank: int) -> int:
        if self.group is None:
            return group_rank
        return dist.get_global_rank(self.group, group_rank)


# ---------------------------------------------------------------------------
# the data-parallel MuonClip step
# ---------------------------------------------------------------------------

def distributed_muonclip_step_mha(opt: DistributedMuon, x, wq, wk, H: int, dh: int, grads,
                                  tau: float, causal: bool = False):
    """Data-parallel MuonClip step of an MHA layer whose Muon matrices are
    [W_q, W_k] (in that order in ``opt``): this rank's micro-batch x, the
    current forward weights wq, wk, and this rank's full gradients.  Returns
    (s_max, gamma), identical on every rank."""
    k = opt.kernels
    s_max = k.max_logits_mha(x, wq, wk, H, dh, causal)
    allreduce_smax(s_max, opt.group, k)
    opt.step(grads)
    # the whole padded blocks: padding rows are zero and stay zero
    gamma = k.qk_clip_mha(opt.mats[0].w, opt.mats[1].w, H, dh, s_max, tau)
    return s_max, gamma


def distributed_muonclip_step_mla(opt: DistributedMuon, x, w_qa, w_qb, w_kva, w_kb, H: int,
                                  nope: int, rope: int, rope_base: float, grads, tau: float,
                                  causal: bool = True):
    """As the MHA step for an MLA layer whose Muon matrices are [W_qa, W_qb,
    W_kva, W_kb]; the clip scales this rank's blocks of W_qb and W_kb."""
    k = opt.kernels
    s_max = k.max_logits_mla(x, w_qa, w_qb, w_kva, w_kb, H, nope, rope, rope_base, causal)
    allreduce_smax(s_max, opt.group, k)
    opt.step(grads)
    gamma = k.qk_clip_mla(opt.mats[1].w, opt.mats[3].w, H, nope, rope, s_max, tau)
    return s_max, gamma


__all__ = ["block_rows", "shard_range", "ns_cost", "assign_owners", "LibraryKernels",
           "allreduce_smax", "DistributedMuon", "distributed_muonclip_step_mha",
           "distributed_muonclip_step_mla"]
