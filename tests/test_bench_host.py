"""Host logic of the benchmark, on the CPU.

The method's path needs no exchange between GPUs here: N GPUs run N
independent replicas of the step, and the job's time is the slowest rank's.
Two gloo ranks check that reduction, the whole-job throughput, and that only
rank 0 runs and prints the oracle (reference) arm; the oracle arm's line is
checked for the contract's keys, and the S_max / gamma report of the bench
line is checked on known values.
"""
import io
import json
import os
import socket
import sys
import types
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _FakeWorkload:
    """Stands in for a workload in the reference arm: one 'sample' is 2e9
    flops in 0.5 s.  make() counts its calls so a rank that should do no work
    can be seen to have done none."""
    metric = "test metric"
    desc = "fake workload"

    def __init__(self):
        self.made = 0

    def make(self, device):
        self.made += 1
        return {}

    def oracle_sample(self, s):
        return 2e9, 0.5, "fake sample"


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        args = types.SimpleNamespace(gpus=world, steps=3, warmup=1)
        wl = _FakeWorkload()
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.run_reference(args, wl)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"t": t, "made": wl.made, "stdout": buf.getvalue()}, f)
    finally:
        dist.destroy_process_group()


def test_replica_timing_and_reference_arm_on_two_gloo_ranks(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            p.join()
    assert [p.exitcode for p in procs] == [0, 0]
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    # the slowest rank sets the time on every rank
    assert [r["t"] for r in res] == [15.0, 15.0]
    # rank 0 alone draws inputs, runs the oracle and prints one JSON line
    assert res[0]["made"] == 1 and res[1]["made"] == 0
    assert res[1]["stdout"] == ""
    lines = res[0]["stdout"].strip().splitlines()
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 3
    assert line["value"] == pytest.approx(2e9 / 0.5 / 1e12)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # two replicas of 1e12 flops each in the job's 0.5 s: 4 TFLOP/s
    assert bench.job_tflops(2, 1e12, 0.5) == pytest.approx(4.0)
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_prints_one_contract_line():
    """The oracle arm of the benchmark on the default workload, one bounded
    sample: one JSON line with the keys the benchmark contract names."""
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "impl"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 1
    assert line["config"]["workload"].startswith("Muon batch: 48 x 7168x2048")
    assert line["cpu_baseline"]["value"] == line["value"]


def test_clip_summary_of_the_last_step():
    """The bench line's S_max / gamma report: heads whose gamma < 1 are
    counted as clipped; a workload without a scan reports nothing."""
    import torch
    sys.path.insert(0, ROOT)
    import bench
    s = {"s_max": torch.tensor([1.6, 2409.8, 1.4, 2540.7]),
         "gamma": torch.tensor([1.0, 0.0415, 1.0, 0.0394]), "tau": 100.0, "hot": [1, 3]}
    r = bench.clip_summary(s)
    assert r["heads"] == 4 and r["clipped_heads"] == 2 and r["planted_hot_heads"] == [1, 3]
    assert r["s_max_max"] == pytest.approx(2540.7) and r["gamma_min"] == pytest.approx(0.0394)
    assert r["tau"] == 100.0
    json.dumps(r)
    assert bench.clip_summary({"w": [torch.zeros(2)]}) is None
    only_smax = bench.clip_summary({"s_max": torch.tensor([3.0, 1.0])})
    assert only_smax == {"heads": 2, "s_max_max": 3.0, "s_max_min": 1.0}


def test_newton_schulz_flop_accounting():
    """The bench's Newton-Schulz flop count against the FLOP formula of the
    Muon blog's "Analysis" section: 2T(2nm^2 + m^3) for T iterations on an
    m x n matrix counts every product densely.  The algorithmic count of the
    roofline takes the symmetric Gram and A.A once (m(m+1)n and m^2(m+1));
    for the expert batch (96 matrices 2048 x 7168, T = 5) the two totals are
    65.97 and 47.43 TFLOP."""
    sys.path.insert(0, ROOT)
    import bench
    m, n, T = 2048, 7168, 5
    f = bench.ns_flops_per_iter(m, n)
    dense = 2 * m * m * n + 2 * m ** 3 + 2 * m * m * n
    assert T * dense == 2 * T * (2 * n * m * m + m ** 3)
    assert f["gram"] == m * (m + 1) * n and f["poly"] == m * m * (m + 1) and f["apply"] == 2 * m * m * n
    assert 96 * T * dense / 1e12 == pytest.approx(65.97, abs=0.01)
    assert 96 * T * sum(f.values()) / 1e12 == pytest.approx(47.43, abs=0.01)


def test_workload_flop_accounting():
    """Algorithmic work of each bench workload from first principles: a
    projection is 2 M N K flops, a logit 2 d flops per (i, j) pair (T^2 per
    sequence, T(T+1)/2 when causal), Newton-Schulz as above (two 1024 x 1024
    matrices for the MHA layer; W_qa, W_qb, W_kva, W_kb for the long MLA)."""
    sys.path.insert(0, ROOT)
    import bench
    c2 = bench.WORKLOADS["c2"]()
    assert c2.units["gemm:proj"][1] == 2 * 2 * 8 * 1024 * 1024 * 1024           # 34.4 GF
    assert c2.units["scan"][1] == 2 * 8 * 1024 * 1024 * 16 * 64                  # 17.2 GF
    assert c2.ns_flops == 2 * 5 * (2 * 1024 * 1025 * 1024 + 2 * 1024 ** 3)       # 2 x 21.5 GF
    c3 = bench.WORKLOADS["c3"]()
    assert c3.scan_flops / 1e12 == pytest.approx(8.307, abs=1e-3)                # 5.008 + 3.299
    assert c3.units["scan"][1] == 2 * 16 * (4096 * 4097 // 2) * 64 * 192
    c5 = bench.WORKLOADS["c5"]()
    assert c5.scan_flops / 1e12 == pytest.approx(15.699, abs=1e-3)               # 2.504 + 13.195
    assert c5.ns_flops / 1e12 == pytest.approx(0.7945, abs=1e-4)
