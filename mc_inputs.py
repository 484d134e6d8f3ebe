"""Seeded synthetic inputs for the MuonClip step (shared by tests, oracle
checks, smoke and the benchmark).

This module only DRAWS inputs: it holds none of the method's arithmetic
(no projection, logit, clip or Muon math).  The shapes follow the workloads
of the pages (Kimi K2: hidden 7168, 64 MLA heads, expert hidden 2048, tau 100)
and the five workload recipes:

  c1  tiny MHA + 64x32 Newton-Schulz, fp32, seed 7, in the draw order of the
      MHA semantic reference printed in "Kimi K2: 1T MoE, MuonClip and
      Agentic training system" (x = randn(2,5,4); W_q, W_k = 8 randn(3,4,2)).
  c2  MHA layer in bf16: x [8,1024,1024], H=16, dh=64, W ~ N(0, 0.02^2),
      3 planted hot heads x40, tau=100, Muon on the 1024x1024 projections.
  c3  K2-shaped MLA layer in bf16: hidden 7168, 64 heads, q_lora 1536,
      kv_lora 512, nope 128, rope 64 (base 50000), x [16,4096], W ~ N(0,
      0.006^2), 4 hot heads' q^C/q^R blocks x30, causal.
  c4  Muon batch: 48 up-projections 7168x2048 + 48 down-projections
      2048x7168, fp32 W ~ N(0, 0.006^2), momentum and grads ~ N(0, 1e-3^2).
  c5  long-context MLA: c3 shapes with B=1, T=32768, 1% of tokens x20,
      8 hot heads x30, causal, then a MuonClip step on W_qa/W_qb/W_kva/W_kb.

Every generator takes size overrides so tests can draw the same recipe at
sizes the oracle finishes in seconds.  Real K2 activations / checkpoints are
not available; these synthetic tensors stand in for them.
"""
from __future__ import annotations

import torch

TAU = 100.0
ROPE_BASE = 50000.0
NS_STEPS = 5
MU = 0.95
LR = 2e-4
WD = 0.1
RMS = 0.2
EPS = 1e-7


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, std=1.0, dtype=torch.float32):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def heads_to_cols(w_hdf: torch.Tensor) -> torch.Tensor:
    """[H, D, dh] (per-head layout of the semantic reference) -> [D, H*dh]
    (x @ W layout, head h = column block h).  A pure relayout."""
    H, D, dh = w_hdf.shape
    return w_hdf.permute(1, 0, 2).reshape(D, H * dh).contiguous()


# ---------------------------------------------------------------------------
# c1
# ---------------------------------------------------------------------------

def c1():
    """Tiny fp32 case.  Draw order: x, W_q, W_k (as in the printed MHA
    reference, seed 7), then the 64x32 momentum, then for the full Muon step
    a gradient and a weight of the same shape."""
    torch.manual_seed(7)
    x = torch.randn(2, 5, 4)
    wq_hdf = torch.randn(3, 4, 2) * 8
    wk_hdf = torch.randn(3, 4, 2) * 8
    m_prev = torch.randn(64, 32)
    grad = torch.randn(64, 32)
    w = torch.randn(64, 32)
    return dict(x=x, wq_hdf=wq_hdf, wk_hdf=wk_hdf, wq=heads_to_cols(wq_hdf),
                wk=heads_to_cols(wk_hdf), H=3, dh=2, tau=10.0, causal=False,
                m_prev=m_prev, grad=grad, w=w)


# ---------------------------------------------------------------------------
# MHA layer (c2 and test-sized variants)
# ---------------------------------------------------------------------------

def mha_layer(B=8, T=1024, D=1024, H=16, dh=64, w_std=0.02, n_hot=3, hot_scale=40.0,
              causal=False, seed=1002, device="cpu", muon=True, state_std=1e-3):
    g = _gen(seed, device)
    x = _randn((B, T, D), g, device, dtype=torch.bfloat16)
    wq = _randn((D, H * dh), g, device, std=w_std)
    wk = _randn((D, H * dh), g, device, std=w_std)
    hot = torch.randperm(H, generator=g, device=device)[:n_hot].sort().values.tolist()
    for h in hot:
        wq[:, h * dh:(h + 1) * dh] *= hot_scale
        wk[:, h * dh:(h + 1) * dh] *= hot_scale
    out = dict(x=x, wq=wq.to(torch.bfloat16), wk=wk.to(torch.bfloat16), H=H, dh=dh,
               hot=hot, tau=TAU, causal=causal)
    if muon:
        # fp32 master weights are the exact up-cast of the bf16 forward copies
        out["w_master"] = [out["wq"].float(), out["wk"].float()]
        out["m_prev"] = [_randn((D, H * dh), g, device, std=state_std) for _ in range(2)]
        out["grad"] = [_randn((D, H * dh), g, device, std=state_std) for _ in range(2)]
    return out


def c2(device="cpu", **kw):
    return mha_layer(seed=1002, device=device, **kw)


# ---------------------------------------------------------------------------
# MLA layer (c3, c5 and test-sized variants)
# ---------------------------------------------------------------------------

def mla_layer(B=16, T=4096, D=7168, H=64, q_lora=1536, kv_lora=512, nope=128, rope=64,
              w_std=0.006, n_hot=4, hot_scale=30.0, hot_k=False, heavy_frac=0.0,
              heavy_scale=20.0, causal=True, seed=1003, device="cpu", muon=False,
              state_std=1e-3):
    g = _gen(seed, device)
    x = _randn((B, T, D), g, device)
    w_qa = _randn((D, q_lora), g, device, std=w_std)
    w_qb = _randn((q_lora, H * (nope + rope)), g, device, std=w_std)
    w_kva = _randn((D, kv_lora + rope), g, device, std=w_std)
    w_kb = _randn((kv_lora, H * nope), g, device, std=w_std)
    hot = torch.randperm(H, generator=g, device=device)[:n_hot].sort().values.tolist()
    qk = nope + rope
    for h in hot:
        w_qb[:, h * qk:(h + 1) * qk] *= hot_scale       # q^C and q^R blocks
        if hot_k:
            w_kb[:, h * nope:(h + 1) * nope] *= hot_scale
    heavy = []
    if heavy_frac > 0:
        n_heavy = int(round(heavy_frac * T))
        for b in range(B):
            rows = torch.randperm(T, generator=g, device=device)[:n_heavy]
            x[b, rows] *= heavy_scale
            heavy.append(rows.sort().values)
    out = dict(x=x.to(torch.bfloat16), w_qa=w_qa.to(torch.bfloat16),
               w_qb=w_qb.to(torch.bfloat16), w_kva=w_kva.to(torch.bfloat16),
               w_kb=w_kb.to(torch.bfloat16), H=H, q_lora=q_lora, kv_lora=kv_lora,
               nope=nope, rope=rope, rope_base=ROPE_BASE, hot=hot, heavy=heavy,
               tau=TAU, causal=causal)
    if muon:
        names = ["w_qa", "w_qb", "w_kva", "w_kb"]
        out["w_master"] = [out[n].float() for n in names]
        out["m_prev"] = [_randn(tuple(out[n].shape), g, device, std=state_std) for n in names]
        out["grad"] = [_randn(tuple(out[n].shape), g, device, std=state_std) for n in names]
    return out


def c3(device="cpu", **kw):
    return mla_layer(seed=1003, device=device, **kw)


def c3b(device="cpu", **kw):
    """c3 shapes with 1% heavy-tailed token rows (x20) so the MLA clip fires
    (c3 as written keeps every head below tau)."""
    kw.setdefault("heavy_frac", 0.01)
    return mla_layer(seed=1013, device=device, **kw)


def c5(device="cpu", **kw):
    kw.setdefault("B", 1)
    kw.setdefault("T", 32768)
    kw.setdefault("n_hot", 8)
    kw.setdefault("heavy_frac", 0.01)
    kw.setdefault("muon", True)
    return mla_layer(seed=1005, device=device, **kw)


# ---------------------------------------------------------------------------
# Muon expert batch (c4 and test-sized variants)
# ---------------------------------------------------------------------------

def expert_batch(n_up=48, n_down=48, hidden=7168, expert=2048, w_std=0.006, state_std=1e-3,
                 seed=1004, device="cpu"):
    g = _gen(seed, device)
    shapes = [(hidden, expert)] * n_up + [(expert, hidden)] * n_down
    w = [_randn(s, g, device, std=w_std) for s in shapes]
    m_prev = [_randn(s, g, device, std=state_std) for s in shapes]
    grad = [_randn(s, g, device, std=state_std) for s in shapes]
    return dict(w=w, m_prev=m_prev, grad=grad, shapes=shapes)


def c4(device="cpu", **kw):
    return expert_batch(seed=1004, device=device, **kw)


def matrix(rows, cols, seed, device="cpu", std=1.0):
    """One N(0, std^2) fp32 matrix (Newton-Schulz and GEMM test inputs)."""
    g = _gen(seed, device)
    return _randn((rows, cols), g, device, std=std)


def attention_qkv(B, T, H, dh, seed, device="cpu", q_std=1.0):
    """bf16 q, k, v [B, T, H*dh], N(0, 1) (q scaled by q_std): the inputs of
    the attention forward with the max logit taken along."""
    g = _gen(seed, device)
    q = _randn((B, T, H * dh), g, device, std=q_std).to(torch.bfloat16)
    k = _randn((B, T, H * dh), g, device).to(torch.bfloat16)
    v = _randn((B, T, H * dh), g, device).to(torch.bfloat16)
    return {"q": q, "k": k, "v": v, "H": H, "dh": dh}


def attention_mla_qkv(B, T, H, seed, device="cpu", q_std=1.0, nope=128, rope=64, dv=128):
    """bf16 inputs of the MLA attention forward, N(0, 1) (q scaled by q_std):
    q [B, T, H*(nope+rope)] (per head q^C then q^R), k_c [B, T, H*nope], the
    shared k_r [B, T, rope] and v [B, T, H*dv]."""
    g = _gen(seed, device)
    q = _randn((B, T, H * (nope + rope)), g, device, std=q_std).to(torch.bfloat16)
    k_c = _randn((B, T, H * nope), g, device).to(torch.bfloat16)
    k_r = _randn((B, T, rope), g, device).to(torch.bfloat16)
    v = _randn((B, T, H * dv), g, device).to(torch.bfloat16)
    return {"q": q, "k_c": k_c, "k_r": k_r, "v": v, "H": H}
