#!/usr/bin/env python
"""MuonClip step benchmark: prints ONE JSON line.

A step is one pass of the whole hot path on one batch of synthetic input,
through the library's C ABI.  The default line measures the two K2-scale
workloads in one process:

  * the headline: Muon on the MoE expert batch -- 48 up-projections
    7168 x 2048 and 48 down-projections 2048 x 7168, fp32 masters, momentum
    0.95, 5 quintic Newton-Schulz iterations (16-bit operands, fp32
    accumulation), RMS matching 0.2 sqrt(max(A,B)), weight decay 0.1
    (``value``, ``ms_per_step``, ``roofline``, ``e2e``, ``cpu_baseline``);
  * beside it, the long-context K2 MLA MuonClip step -- x [1, 32768, 7168],
    64 heads, causal max-logit scan, Muon on W_qa, W_qb, W_kva, W_kb, then
    the MLA QK-Clip (``muonclip_step_ms``, ``scan_tflops``,
    ``scan_frac_bf16_peak`` and the object ``long_mla`` with its own
    roofline and kernel breakdown).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload c4|c2|c3|c5|attn|attnl|attn_mla] [--no-long-mla]

value     = algorithmic TFLOP/s of the step (scan + Newton-Schulz flops per
            step / device time per step, inputs resident, L2 flushed between
            timed steps);
e2e       = the same through the public API with the step's inputs copied
            host->device from pinned memory and the results read back;
roofline  = the dominant kernel's algorithmic work per launch / its
            event-timed duration against the measured peak (the sustained
            bf16 figure for a contraction inside a step of milliseconds that
            repeats back to back, the burst figure otherwise);
cpu_baseline = the fp64 oracle on this host's cores on a bounded sample.
--impl reference times that oracle (the only reference this method has).

c2 is the MHA layer (x [8,1024,1024], 16 heads of 64, Muon on W_q and W_k).
attn / attnl time the attention forward that takes the max logit along
(value = its algorithmic TFLOP/s: 4 flops per allowed (i, j) pair and head
dimension), attn_mla the MLA forward (2 (192 + 128) flops per allowed pair
and head); they are extra lines, not the default workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import mc_inputs  # noqa: E402

METRIC = "max-logit scan & Newton-Schulz TFLOP/s (% bf16 peak); MuonClip step ms"
L2_FLUSH_BYTES = 256 << 20  # > 129 MB L2


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------

def ns_flops_per_iter(m: int, n: int) -> dict:
    """Per quintic iteration on an m x n (m <= n) matrix, counting the
    symmetric products once: Gram m(m+1)n, A A m^2(m+1), B X 2 m^2 n."""
    return {"gram": m * (m + 1) * n, "poly": m * m * (m + 1), "apply": 2 * m * m * n}


def scan_pairs(B, T, causal):
    return B * (T * (T + 1) // 2 if causal else T * T)


# DRAM bytes (read + write) per launch of each kernel kind, from the ncu
# captures summarised in profiles/ (cold-cache replays), all taken on the
# bench workloads themselves (1-pass metric sets on the large ones).  The
# expert-batch Newton-Schulz launch (cooperative, on CTA pairs) cannot be
# captured by ncu and has no entry.  Drop an entry whenever the kernel changes.
TRAFFIC = {
    ("c2", "gemm:ns"): 4281856 + 20736,
    ("c2", "scan"): 33608448 + 0,
    ("c3", "scan"): 2750955008 + 2818816,
    ("c5", "scan"): 1391011840 + 3112960,
    ("attn", "attn"): 50578176 + 762624,
    ("attnl", "attn"): 537211136 + 46925568,
    ("attn_mla", "attn_mla"): 1069263616 + 249915392,
}


def _twin_state(s, ins):
    """A copy of workload state s whose per-step input tensors (ins) are
    fresh device buffers; everything else (weights, optimizer state,
    workspaces) is shared."""
    ids = {id(t): t.clone() for t in ins}

    def twin(v):
        if id(v) in ids:
            return ids[id(v)]
        if isinstance(v, list):
            return [twin(u) for u in v]
        if isinstance(v, tuple):
            return tuple(twin(u) for u in v)
        return v
    out = {k: twin(v) for k, v in s.items()}
    for k in ("s_max", "gamma"):
        if k in out and hasattr(out[k], "clone"):
            out[k] = out[k].clone()
    return out


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

class Workload:
    name = ""
    desc = ""
    # a contraction inside a step of milliseconds, repeated back to back,
    # runs under the power cap: its roofline takes the sustained bf16 peak
    sustained = False

    def make(self, device):
        raise NotImplementedError

    def cpu_state(self):
        """Host-side inputs of the oracle sample (the reference arm)."""
        return self.make("cpu")

    def step(self, s, api):
        raise NotImplementedError

    def step_part(self, s, api, part):
        raise NotImplementedError


class MhaLayer(Workload):
    """c2: MHA layer + Muon on the W_q / W_k masters + clip."""

    def __init__(self, B=8, T=1024, D=1024, H=16, dh=64):
        self.B, self.T, self.D, self.H, self.dh = B, T, D, H, dh
        self.name = "c2"
        self.desc = (f"MHA layer bf16 x[{B},{T},{D}] H={H} dh={dh} tau=100 non-causal; "
                     f"Muon (5 NS steps, mu 0.95, lr 2e-4, wd 0.1, rms 0.2) on fp32 W_q, W_k "
                     f"[{D},{H * dh}]; QK-Clip of both")
        N = H * dh
        m, n = min(D, N), max(D, N)
        ns = ns_flops_per_iter(m, n)
        self.units = {
            "gemm:proj": ("tensor", 2 * 2 * B * T * D * N),
            "scan": ("tensor", 2 * scan_pairs(B, T, False) * H * dh),
            # all 5 quintic iterations (15 GEMM phases) run as one launch
            "gemm:ns": ("tensor", 5 * 2 * (ns["gram"] + ns["poly"] + ns["apply"])),
            "muon_momentum": ("hbm", 2 * D * N * 14),
            "muon_update": ("hbm", 2 * D * N * 10),
        }
        self.scan_flops = self.units["gemm:proj"][1] + self.units["scan"][1]
        self.ns_flops = self.units["gemm:ns"][1]

    def make(self, device):
        inp = mc_inputs.c2(device=device, B=self.B, T=self.T, D=self.D, H=self.H, dh=self.dh)
        import torch
        s = dict(inp)
        s["masters"] = [t.clone() for t in inp["w_master"]]
        s["moms"] = [t.clone() for t in inp["m_prev"]]
        s["s_max"] = torch.empty(self.H, dtype=torch.float32, device=device)
        s["gamma"] = torch.empty(self.H, dtype=torch.float32, device=device)
        return s

    def inputs(self, s):
        """Per-step inputs a trainer would hand over: activations, grads."""
        return [s["x"]] + s["grad"]

    def outputs(self, s):
        return [s["s_max"], s["gamma"]]

    def step(self, s, api):
        self.step_part(s, api, "scan")
        self.step_part(s, api, "muon")
        self.step_part(s, api, "clip")

    def step_part(self, s, api, part):
        if part == "scan":
            api.mc_max_logits_mha(s["x"], s["wq"], s["wk"], self.H, self.dh, s_max=s["s_max"])
        elif part == "muon":
            api.mc_muon_step(s["masters"], s["grad"], s["moms"], lr=mc_inputs.LR, mu=mc_inputs.MU,
                             wd=mc_inputs.WD, rms=mc_inputs.RMS, steps=mc_inputs.NS_STEPS)
        else:
            api.mc_qk_clip_mha(s["masters"][0], s["masters"][1], self.H, self.dh, s["s_max"],
                               s["tau"], gamma=s["gamma"])

    # --- oracle sample for the CPU baseline ---------------------------------
    def oracle_sample(self, s):
        import oracle
        x = s["x"][:1].cpu()
        wq, wk = s["wq"].cpu(), s["wk"].cpu()
        w0, g0, m0 = (t[0].cpu() for t in (s["w_master"], s["grad"], s["m_prev"]))
        heads = [0, 1]
        t0 = time.perf_counter()
        oracle.max_logits_mha(x, wq, wk, self.H, self.dh, False, heads=heads)
        oracle.muon_step(w0, g0, m0, lr=mc_inputs.LR)
        dt = time.perf_counter() - t0
        N = self.H * self.dh
        m, n = min(self.D, N), max(self.D, N)
        flops = len(heads) * (2 * 2 * self.T * self.D * self.dh + 2 * self.T * self.T * self.dh)
        flops += 5 * sum(ns_flops_per_iter(m, n).values())
        return flops, dt, (f"2 of {self.B * self.H} (sequence, head) scans and 1 of 2 "
                           f"Muon steps ({self.D}x{N}), fp64")


class ExpertBatch(Workload):
    """c4: Muon on 48 up + 48 down expert matrices (no scan)."""

    def __init__(self, n_up=48, n_down=48):
        self.n_up, self.n_down = n_up, n_down
        self.name = "c4"
        self.sustained = True
        self.desc = (f"Muon batch: {n_up} x 7168x2048 + {n_down} x 2048x7168 fp32, 5 NS steps "
                     "(bf16 operands, fp32 accumulation)")
        ns = ns_flops_per_iter(2048, 7168)
        cnt = n_up + n_down
        self.units = {
            "gemm:ns": ("tensor", 5 * (ns["gram"] + ns["poly"] + ns["apply"]) * cnt),
            "muon_momentum": ("hbm", cnt * 2048 * 7168 * 14),
            "muon_update": ("hbm", cnt * 2048 * 7168 * 10),
        }
        self.scan_flops = 0
        self.ns_flops = self.units["gemm:ns"][1]

    def make(self, device):
        return mc_inputs.c4(device=device, n_up=self.n_up, n_down=self.n_down)

    def cpu_state(self):
        """The oracle sample reads one up-projection's momentum: draw the
        recipe with that one matrix instead of all 96 (17 GB on the host)."""
        return mc_inputs.c4(device="cpu", n_up=1, n_down=0)

    def inputs(self, s):
        return s["grad"]

    def outputs(self, s):
        """The step's result is the updated weights; read back one row of the
        first matrix."""
        return [s["w"][0][0, :64]]

    def step(self, s, api):
        self.step_part(s, api, "muon")

    def step_part(self, s, api, part):
        if part == "muon":
            api.mc_muon_step(s["w"], s["grad"], s["m_prev"], lr=mc_inputs.LR)

    def oracle_sample(self, s):
        import oracle
        t0 = time.perf_counter()
        oracle.newton_schulz(s["m_prev"][0][:512].cpu(), 5)
        dt = time.perf_counter() - t0
        m, n = 512, 2048
        flops = 5 * sum(ns_flops_per_iter(m, n).values())
        return flops, dt, "Newton-Schulz of one 512x2048 slice of an expert momentum, fp64"


class MlaLayer(Workload):
    """c3 / c5: MLA layer scan (+ Muon on its 4 projections for c5) + clip."""

    def __init__(self, which="c5", B=None, T=None):
        self.which = which
        self.name = which
        self.B = B if B is not None else (1 if which == "c5" else 16)
        self.T = T if T is not None else (32768 if which == "c5" else 4096)
        self.muon = which == "c5"
        self.sustained = True
        self.desc = (f"K2-shaped MLA layer bf16 x[{self.B},{self.T},7168] H=64 q_lora 1536 "
                     f"kv_lora 512 nope 128 rope 64 causal"
                     + ("; Muon on W_qa, W_qb, W_kva, W_kb; MLA clip" if self.muon else ""))
        BT = self.B * self.T
        proj = 2 * BT * (7168 * 1536 + 7168 * 576 + 1536 * 64 * 192 + 512 * 64 * 128)
        self.units = {"gemm:proj": ("tensor", proj),
                      "scan": ("tensor", 2 * scan_pairs(self.B, self.T, True) * 64 * 192)}
        self.scan_flops = proj + self.units["scan"][1]
        self.ns_flops = 0
        if self.muon:
            for r, c in [(7168, 1536), (1536, 12288), (7168, 576), (512, 8192)]:
                m, n = min(r, c), max(r, c)
                self.ns_flops += 5 * sum(ns_flops_per_iter(m, n).values())

    def make(self, device):
        fn = mc_inputs.c5 if self.which == "c5" else mc_inputs.c3
        inp = fn(device=device, B=self.B, T=self.T)
        import torch
        s = dict(inp)
        if self.muon:
            s["masters"] = [t.clone() for t in inp["w_master"]]
            s["moms"] = [t.clone() for t in inp["m_prev"]]
        s["s_max"] = torch.empty(64, dtype=torch.float32, device=device)
        s["gamma"] = torch.empty(64, dtype=torch.float32, device=device)
        return s

    def inputs(self, s):
        return [s["x"]] + (s["grad"] if self.muon else [])

    def outputs(self, s):
        return [s["s_max"], s["gamma"]]

    def step(self, s, api):
        self.step_part(s, api, "scan")
        self.step_part(s, api, "muon")
        self.step_part(s, api, "clip")

    def step_part(self, s, api, part):
        if part == "scan":
            api.mc_max_logits_mla(s["x"], s["w_qa"], s["w_qb"], s["w_kva"], s["w_kb"], 64, 128, 64,
                                  s["rope_base"], causal=True, s_max=s["s_max"])
            return
        if part == "muon":
            if self.muon:
                api.mc_muon_step(s["masters"], s["grad"], s["moms"], lr=mc_inputs.LR)
            return
        if self.muon:
            api.mc_qk_clip_mla(s["masters"][1], s["masters"][3], 64, 128, 64, s["s_max"], s["tau"],
                               gamma=s["gamma"])
        else:
            api.mc_qk_clip_mla(s["w_qb"], s["w_kb"], 64, 128, 64, s["s_max"], s["tau"],
                               gamma=s["gamma"])

    def oracle_sample(self, s):
        import oracle
        T = min(self.T, 512)
        t0 = time.perf_counter()
        oracle.max_logits_mla(s["x"][:1, :T].cpu(), s["w_qa"].cpu(), s["w_qb"].cpu(),
                              s["w_kva"].cpu(), s["w_kb"].cpu(), 64, 128, 64, s["rope_base"],
                              True, heads=[0])
        dt = time.perf_counter() - t0
        flops = 2 * T * (7168 * 1536 + 7168 * 576) + 2 * T * (1536 * 192 + 512 * 128)
        flops += 2 * (T * (T + 1) // 2) * 192
        return flops, dt, f"one head of the MLA scan over the first {T} tokens, fp64"


class AttnLayer(Workload):
    """attn / attnl: the attention forward with the max logit taken along."""

    def __init__(self, which="attn"):
        self.name = which
        if which == "attn":
            self.B, self.T, self.H, self.dh, self.causal = 8, 1024, 16, 64, False
        else:
            self.B, self.T, self.H, self.dh, self.causal = 2, 8192, 16, 128, True
        self.desc = (f"MHA attention forward bf16 q,k,v [{self.B},{self.T},{self.H}x{self.dh}] "
                     f"{'causal' if self.causal else 'non-causal'}, O bf16 and the per-head max logit")
        pairs = scan_pairs(self.B, self.T, self.causal)
        self.units = {"attn": ("tensor", 4 * pairs * self.H * self.dh)}
        self.metric = "attention forward with the max logit taken along, TFLOP/s (% bf16 peak)"
        self.scan_flops = self.units["attn"][1]
        self.ns_flops = 0

    def make(self, device):
        import torch
        s = mc_inputs.attention_qkv(self.B, self.T, self.H, self.dh, seed=1500, device=device)
        s["o"] = torch.empty_like(s["q"])
        s["s_max"] = torch.empty(self.H, dtype=torch.float32, device=device)
        return s

    def inputs(self, s):
        return [s["q"], s["k"], s["v"]]

    def outputs(self, s):
        return [s["s_max"]]

    def step(self, s, api):
        self.step_part(s, api, "scan")

    def step_part(self, s, api, part):
        if part == "scan":
            api.mc_attention_mha(s["q"], s["k"], s["v"], self.H, self.dh, causal=self.causal, out=s["o"],
                                 s_max=s["s_max"])

    def oracle_sample(self, s):
        import oracle
        T = min(self.T, 512)
        cols = slice(0, self.dh)
        q, k, v = (s[n][:1, :T, cols].cpu() for n in ("q", "k", "v"))
        t0 = time.perf_counter()
        oracle.attention_mha(q, k, v, 1, self.dh, self.causal)
        dt = time.perf_counter() - t0
        return (4 * scan_pairs(1, T, self.causal) * self.dh, dt,
                f"one head of one sequence over the first {T} tokens, fp64")


class AttnMlaLayer(Workload):
    """attn_mla: the MLA attention forward (K2 shapes: 64 heads, q^C/k^C 128,
    q^R/k^R 64 with k^R shared, dv 128) with the max logit taken along."""

    def __init__(self, B=2, T=8192, H=64):
        self.name = "attn_mla"
        self.B, self.T, self.H, self.causal = B, T, H, True
        self.desc = (f"MLA attention forward bf16 q [{B},{T},{H}x192], k^C [{B},{T},{H}x128], shared "
                     f"k^R [{B},{T},64], v [{B},{T},{H}x128] causal, O bf16 and the per-head max logit")
        pairs = scan_pairs(B, T, True)
        # 2 flops per multiply-add: q.k over 192 and p.v over 128 per allowed pair and head
        self.units = {"attn_mla": ("tensor", 2 * pairs * H * (192 + 128))}
        self.metric = "MLA attention forward with the max logit taken along, TFLOP/s (% bf16 peak)"
        self.scan_flops = self.units["attn_mla"][1]
        self.ns_flops = 0

    def make(self, device):
        import torch
        s = mc_inputs.attention_mla_qkv(self.B, self.T, self.H, seed=1700, device=device)
        s["o"] = torch.empty((self.B, self.T, self.H * 128), dtype=torch.bfloat16, device=device)
        s["s_max"] = torch.empty(self.H, dtype=torch.float32, device=device)
        return s

    def inputs(self, s):
        return [s["q"], s["k_c"], s["k_r"], s["v"]]

    def outputs(self, s):
        return [s["s_max"]]

    def step(self, s, api):
        self.step_part(s, api, "scan")

    def step_part(self, s, api, part):
        if part == "scan":
            api.mc_attention_mla(s["q"], s["k_c"], s["k_r"], s["v"], self.H, causal=True, out=s["o"],
                                 s_max=s["s_max"])

    def oracle_sample(self, s):
        import oracle
        T = min(self.T, 512)
        q = s["q"][:1, :T, :192].cpu()
        kc, kr, v = s["k_c"][:1, :T, :128].cpu(), s["k_r"][:1, :T].cpu(), s["v"][:1, :T, :128].cpu()
        t0 = time.perf_counter()
        oracle.attention_mla(q, kc, kr, v, 1, 128, 64, 128, True)
        dt = time.perf_counter() - t0
        return (2 * scan_pairs(1, T, True) * (192 + 128), dt,
                f"one head of one sequence over the first {T} tokens, fp64")


WORKLOADS = {"c2": lambda: MhaLayer(), "c4": lambda: ExpertBatch(), "c3": lambda: MlaLayer("c3"),
             "c5": lambda: MlaLayer("c5"), "attn": lambda: AttnLayer("attn"),
             "attnl": lambda: AttnLayer("attnl"), "attn_mla": lambda: AttnMlaLayer()}


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples (the JSON line carries their summary)
        self.path = os.path.join(os.environ.get("MC_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"mc_clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        busy = [v for v in sm if v > 0.5 * max(sm)] if sm else []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def clip_summary(s) -> dict | None:
    """S_max, gamma and the number of clipped heads (gamma < 1) that the last
    step left in workload state s; None for a workload without a scan."""
    if "s_max" not in s:
        return None
    sm = s["s_max"].detach().float().cpu()
    res = {"heads": int(sm.numel()), "s_max_max": float(sm.max()), "s_max_min": float(sm.min())}
    if s.get("tau") is not None:
        res["tau"] = float(s["tau"])
    if "gamma" in s:
        g = s["gamma"].detach().float().cpu()
        res["clipped_heads"] = int((g < 1).sum())
        res["gamma_min"] = float(g.min())
    if s.get("hot") is not None:
        res["planted_hot_heads"] = [int(h) for h in s["hot"]]
    return res


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of the ranks' values: in a replica job the slowest rank
    sets the job's time.  One rank returns x itself."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_rank: float, seconds: float) -> float:
    """Whole-job throughput: every rank's algorithmic flops over the job's time."""
    return world * flops_per_rank / seconds / 1e12


def line_config(wl, world: int) -> dict:
    """The workload description both arms print in ``config``."""
    return {"workload": wl.desc, "l2": "flushed between timed steps (256 MiB write)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args, wl):
    """The fp64 oracle on the host cores: each step is one bounded sample of
    the workload (inputs drawn on the CPU)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    s = wl.cpu_state() if hasattr(wl, "cpu_state") else wl.make("cpu")
    for _ in range(min(args.warmup, 1)):
        wl.oracle_sample(s)
    times, flops, sample = [], 0, ""
    for _ in range(args.steps):
        f, dt, sample = wl.oracle_sample(s)
        times.append(dt)
        flops = f
    tot = sum(times)
    value = flops * len(times) / tot / 1e12
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    line = {"metric": getattr(wl, "metric", METRIC), "value": value, "unit": "TFLOP/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / len(times), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": line_config(wl, world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def roofline_entry(wl, name, trace, K, peaks) -> dict:
    """Roofline of kernel kind ``name``: its algorithmic work per launch over
    its mean event-timed launch duration, against the measured peak."""
    hbm_peak, bf16_peak, bf16_sus, peak_src = peaks
    kind, work = wl.units[name]
    n_launch = trace[name][0] / K
    dur = trace[name][1] / trace[name][0] * 1e-3      # s per launch
    if kind == "tensor":
        achieved = work / n_launch / dur / 1e12
        sus = wl.sustained and bf16_sus is not None
        peak = bf16_sus if sus else bf16_peak
        return {"kernel": name, "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "frac_of_burst_peak": achieved / bf16_peak,
                "traffic": TRAFFIC.get((wl.name, name)),
                "peak_kind": f"{peak_src} bf16 dense ({'sustained' if sus else 'burst'})"}
    achieved = work / n_launch / dur / 1e9
    return {"kernel": name, "bound": "hbm", "achieved": achieved, "peak": hbm_peak,
            "unit": "GB/s", "frac": achieved / hbm_peak,
            "traffic": TRAFFIC.get((wl.name, name)),
            "peak_kind": f"{peak_src} HBM copy"}


def measure(wl, args, api, device, world, flush, e2e: bool = True) -> dict:
    """Everything the line reports for workload ``wl`` on this rank: the
    device time per step (whole step as one CUDA graph, L2 flushed between
    timed steps), the scan and Muon halves alone, per-kernel event times, the
    dominant kernel's roofline and, if ``e2e``, the end-to-end rate through
    the public API with host copies inside the timed region."""
    import torch
    from muonclip_mc_max_gb300.step import CapturedStep

    s = wl.make(device)
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # the whole step as one CUDA graph (launch-bound at small sizes); the
    # scan and Muon halves are also captured alone for the breakdown
    n0 = api.mc_launch_count()
    graph = CapturedStep(lambda: wl.step(s, api), warmup=2)
    per_step_launches = (api.mc_launch_count() - n0) // 3  # 2 warm-up runs + the capture
    g_scan = CapturedStep(lambda: wl.step_part(s, api, "scan"), warmup=1) if wl.scan_flops else None
    g_muon = CapturedStep(lambda: wl.step_part(s, api, "muon"), warmup=1) if wl.ns_flops else None
    for _ in range(max(args.warmup, 3)):
        graph.replay()
    assert api.mc_read_device_status(clear=True) == 0, "device status set during warm-up"

    # ---- timed region: device time per step, L2 flushed between steps ----
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    clocks = ClockSampler(device.index or 0)
    clocks.start()
    barrier()
    for k in range(K):
        flush.zero_()
        ev[k][0].record(stream)
        graph.replay()
        ev[k][1].record(stream)
    barrier()
    clk = clocks.stop()
    clip = clip_summary(s)  # the last timed step's S_max and gamma
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(sum(step_ms), world, device) / K
    flops = wl.scan_flops + wl.ns_flops
    peaks = load_peaks()
    bf16_peak = peaks[1]

    def part_ms(g):
        if g is None:
            return None
        e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(K)]
        for k in range(K):
            flush.zero_()
            e[k][0].record(stream)
            g.replay()
            e[k][1].record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in e)

    scan_t, muon_t = part_ms(g_scan), part_ms(g_muon)

    # ---- per-kernel times: a graph captured with event nodes around every
    # launch (on the launching stream), read back after each replay ----
    api.mc_trace_collect()  # drop anything recorded so far
    api.mc_trace_enable(True)
    traced = CapturedStep(lambda: wl.step(s, api), warmup=0)
    api.mc_trace_enable(False)
    trace = {}
    for k in range(K):
        flush.zero_()
        traced.replay()
        torch.cuda.synchronize()
        for name, (n, tms) in api.mc_trace_collect(keep=True).items():
            a = trace.setdefault(name, [0, 0.0])
            a[0] += n
            a[1] += tms
    api.mc_trace_collect(keep=False)
    kernels = {}
    tot_k = sum(v[1] for v in trace.values()) or 1.0
    for name, (n, tms) in trace.items():
        entry = {"launches_per_step": n / K, "ms_per_launch": tms / n, "ms_per_step": tms / K,
                 "share": tms / tot_k}
        if name in wl.units:
            kind, work = wl.units[name]  # algorithmic work per step
            if kind == "tensor":
                entry["achieved_tflops"] = work / (tms / K * 1e-3) / 1e12
            else:
                entry["achieved_gbs"] = work / (tms / K * 1e-3) / 1e9
        kernels[name] = entry
    dominant = max((k for k in kernels if k in wl.units), key=lambda k: trace[k][1])
    roof = roofline_entry(wl, dominant, trace, K, peaks)
    # every HBM-bound pass gets its own entry too
    hbm_roofs = {k: roofline_entry(wl, k, trace, K, peaks) for k in kernels
                 if k in wl.units and wl.units[k][0] == "hbm"}
    assert api.mc_read_device_status(clear=True) == 0, "device status set during timing"
    del traced, g_scan, g_muon

    res = {"wl": wl, "ms": ms, "value": job_tflops(world, flops, ms * 1e-3), "clk": clk,
           "clip": clip, "launches": per_step_launches * K, "scan_ms": scan_t, "muon_ms": muon_t,
           "scan_tflops": (wl.scan_flops / (scan_t * 1e-3) / 1e12) if scan_t else None,
           "ns_tflops": (wl.ns_flops / (muon_t * 1e-3) / 1e12) if muon_t else None,
           "roof": roof, "hbm_roofs": hbm_roofs, "kernels": kernels, "state": s}
    res["scan_frac_bf16_peak"] = res["scan_tflops"] / bf16_peak if scan_t else None
    res["ns_frac_bf16_peak"] = res["ns_tflops"] / bf16_peak if muon_t else None
    if not e2e:
        del graph
        return res

    # ---- end to end through the public API: every step uploads its inputs
    # from pinned host memory and reads its results back.  Two input buffer
    # sets, each with its own captured step, let the upload of step k+1
    # overlap the compute of step k, as a training loop would.  The steps run
    # on a stream of their own and the uploads are spread over four copy
    # streams: the legacy default stream would serialise with every copy. ----
    ins = wl.inputs(s)
    outs = wl.outputs(s)
    s_twin = _twin_state(s, ins)
    graph_twin = CapturedStep(lambda: wl.step(s_twin, api), warmup=1)
    ins_sets = [ins, wl.inputs(s_twin)]
    outs_sets = [outs, wl.outputs(s_twin)]
    graphs = [graph, graph_twin]
    host_in = [t.detach().cpu().pin_memory() for t in ins]
    host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    run_stream = torch.cuda.Stream()
    copy_streams = [torch.cuda.Stream() for _ in range(4)]
    ev_in = [[torch.cuda.Event() for _ in copy_streams] for _ in range(2)]
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]

    def upload(k):
        j = k & 1
        for c, cs in enumerate(copy_streams):
            with torch.cuda.stream(cs):
                if k >= 2:
                    cs.wait_event(ev_done[j])  # step k-2 has finished with buffer set j
                for hd, dv in list(zip(host_in, ins_sets[j]))[c::len(copy_streams)]:
                    dv.copy_(hd, non_blocking=True)
                ev_in[j][c].record(cs)

    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    upload(0)
    with torch.cuda.stream(run_stream):
        for k in range(K):
            j = k & 1
            if k + 1 < K:
                upload(k + 1)
            for e in ev_in[j]:
                run_stream.wait_event(e)
            graphs[j].replay()
            for hd, dv in zip(host_out[j], outs_sets[j]):
                hd.copy_(dv, non_blocking=True)
            ev_done[j].record(run_stream)
    run_stream.synchronize()
    for cs in copy_streams:
        cs.synchronize()
    barrier()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, device)
    res["e2e"] = {"value": job_tflops(world, flops * K, e2e_s), "unit": "TFLOP/s",
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    del graph, graph_twin, graphs, s_twin, ins_sets, outs_sets, host_in, host_out
    return res


def cpu_baseline(wl, s) -> dict:
    """The oracle on this host's cores, repeated for about 10 s of CPU work."""
    f_tot, dt_tot, sample, reps = 0, 0.0, "", 0
    while dt_tot < 10.0 and reps < 50:
        f, dt, sample = wl.oracle_sample(s)
        f_tot += f
        dt_tot += dt
        reps += 1
    return {"value": f_tot / dt_tot / 1e12, "unit": "TFLOP/s",
            "cores": int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)),
            "kind": "oracle", "sample": f"{sample}; {reps} repetitions, {dt_tot:.1f} s"}


def run_ours(args, wl, extra=None):
    """Times ``wl`` (the line's headline) and, if given, ``extra`` (the long
    MLA MuonClip step, reported beside it) on this rank."""
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl")

    from muonclip_mc_max_gb300 import api, build
    build.build()
    api.load_library()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    K = args.steps

    r = measure(wl, args, api, device, world, flush, e2e=True)
    cpu = cpu_baseline(wl, r["state"]) if rank == 0 else None
    r.pop("state")
    torch.cuda.empty_cache()
    rx = None
    if extra is not None:
        rx = measure(extra, args, api, device, world, flush, e2e=False)
        rx.pop("state")
        torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": getattr(wl, "metric", METRIC), "value": r["value"], "unit": "TFLOP/s",
            "n_gpus": world, "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": r["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16/fp16",
            "data": "synthetic", "config": line_config(wl, world),
            "muonclip_step_ms": r["ms"] if r["scan_ms"] is not None else None,
            "scan_tflops": r["scan_tflops"], "scan_frac_bf16_peak": r["scan_frac_bf16_peak"],
            "ns_tflops": r["ns_tflops"], "ns_frac_bf16_peak": r["ns_frac_bf16_peak"],
            "scan_ms": r["scan_ms"], "muon_ms": r["muon_ms"],
            "roofline": r["roof"], "hbm_passes": r["hbm_roofs"], "kernels": r["kernels"],
            "gpu_launches": int(r["launches"]), "clocks": r["clk"], "e2e": r["e2e"],
            "cpu_baseline": cpu,
        }
        if r["clip"] is not None:
            line["clip"] = r["clip"]
        if rx is not None:
            xw = rx["wl"]
            line["muonclip_step_ms"] = rx["ms"]
            line["scan_tflops"] = rx["scan_tflops"]
            line["scan_frac_bf16_peak"] = rx["scan_frac_bf16_peak"]
            line["scan_ms"] = rx["scan_ms"]
            line["long_mla"] = {
                "workload": xw.desc, "muonclip_step_ms": rx["ms"], "value": rx["value"],
                "unit": "TFLOP/s", "scan_tflops": rx["scan_tflops"],
                "scan_frac_bf16_peak": rx["scan_frac_bf16_peak"], "scan_ms": rx["scan_ms"],
                "ns_tflops": rx["ns_tflops"], "muon_ms": rx["muon_ms"],
                "roofline": rx["roof"], "kernels": rx["kernels"], "clip": rx["clip"],
                "gpu_launches": int(rx["launches"]), "clocks": rx["clk"]}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="c4")
    ap.add_argument("--experts", type=int, default=48,
                    help="c4: up- and down-projections each (smaller for profiling)")
    ap.add_argument("--seqs", type=int, default=None, help="c3/c5: sequences (smaller for profiling)")
    ap.add_argument("--tokens", type=int, default=None, help="c3/c5: tokens per sequence")
    ap.add_argument("--no-long-mla", action="store_true",
                    help="c4: leave out the long-context MLA MuonClip step reported beside it")
    args = ap.parse_args()
    extra = None
    if args.workload == "c4":
        wl = ExpertBatch(args.experts, args.experts)
        if not args.no_long_mla:
            extra = MlaLayer("c5", B=args.seqs, T=args.tokens)
    elif args.workload in ("c3", "c5"):
        wl = MlaLayer(args.workload, B=args.seqs, T=args.tokens)
    else:
        wl = WORKLOADS[args.workload]()
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl, extra)


if __name__ == "__main__":
    main()
