"""The composed MuonClip step (Kimi K2 section 2.1, "MuonClip: the new
optimizer"; the K2 review's note that the clip runs after the optimizer
update with the max logit observed in this step, leaving the current
forward/backward unchanged):

  (i)   S_max from the forward's inputs and the current (bf16) weights;
  (ii)  Muon with weight decay and RMS matching on every 2-D matrix (the
        fp32 master weights), W_{t-1} -> W_t;
  (iii) QK-Clip of W_t with gamma from (i).

Pure orchestration of library calls on one stream; every step runs in the
CUDA library."""
from __future__ import annotations

from .api import (NS_COEFFS, mc_max_logits_mha, mc_max_logits_mla, mc_muon_step,
                  mc_qk_clip_mha, mc_qk_clip_mla)


def muonclip_step_mha(x, wq, wk, H, dh, masters, grads, moms, lr, tau, causal=False, mu=0.95,
                      wd=0.1, rms=0.2, steps=5, coeffs=NS_COEFFS, eps=1e-7, nesterov=False,
                      workspace=None, stream=None):
    """x [B,T,D]; wq, wk [D,H*dh] forward weights; masters = [W_q, W_k] fp32
    (updated in place, then clipped).  Returns (s_max, gamma)."""
    s_max = mc_max_logits_mha(x, wq, wk, H, dh, causal=causal, workspace=workspace, stream=stream)
    mc_muon_step(masters, grads, moms, lr, mu=mu, wd=wd, rms=rms, steps=steps, coeffs=coeffs,
                 eps=eps, nesterov=nesterov, workspace=workspace, stream=stream)
    gamma = mc_qk_clip_mha(masters[0], masters[1], H, dh, s_max, tau, stream=stream)
    return s_max, gamma


def muonclip_step_mla(x, w_qa, w_qb, w_kva, w_kb, H, nope, rope, rope_base, masters, grads, moms,
                      lr, tau, causal=True, mu=0.95, wd=0.1, rms=0.2, steps=5, coeffs=NS_COEFFS,
                      eps=1e-7, nesterov=False, workspace=None, stream=None):
    """MLA layer: masters = [W_qa, W_qb, W_kva, W_kb] fp32 (each its own
    Muon matrix); the clip touches W_qb (q^C, q^R) and W_kb (k^C) only.
    Returns (s_max, gamma)."""
    s_max = mc_max_logits_mla(x, w_qa, w_qb, w_kva, w_kb, H, nope, rope, rope_base, causal=causal,
                              workspace=workspace, stream=stream)
    mc_muon_step(masters, grads, moms, lr, mu=mu, wd=wd, rms=rms, steps=steps, coeffs=coeffs,
                 eps=eps, nesterov=nesterov, workspace=workspace, stream=stream)
    gamma = mc_qk_clip_mla(masters[1], masters[3], H, nope, rope, s_max, tau, stream=stream)
    return s_max, gamma


class CapturedStep:
    """Captures a sequence of library calls (``fn``, launched on the current
    stream) into one CUDA graph and replays it: the whole step costs one
    graph launch on the host instead of one launch per kernel.

    The calls are capture-safe: they only enqueue kernels and memsets on the
    caller's stream and read device pointers that stay fixed, so inputs are
    refreshed by copying into the same tensors before ``replay``.  ``fn`` is
    run ``warmup`` times eagerly first (sizing workspaces outside capture)."""

    def __init__(self, fn, warmup: int = 2):
        import torch
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fn()
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()

    __call__ = replay
