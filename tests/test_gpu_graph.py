"""The step as the benchmark times it -- every library call of one step
captured into one CUDA graph and replayed -- computes exactly what the same
calls compute when launched one by one.

The parity tests call the library eagerly; the benchmark replays a captured
graph of the same calls.  For each benchmark workload (at full size where it
is small, else at a reduced size that keeps its launch shapes: the expert
batch on CTA pairs, the MLA scan over several rounds of items), two eager
steps and two graph replays start from the same state, and every tensor of
the state -- activations, forward weights, fp32 masters, momenta, S_max,
gamma, attention outputs -- must agree bit for bit after each step.  The
library's kernels are deterministic (no floating-point atomics; maxima are
combined as order-preserving integer keys; tiles and reductions in a fixed
order), so any difference is a capture fault: a workspace or pointer baked
into the graph that the eager calls do not use, or a launch that was left
out of the capture.
"""
import pytest
import torch

from gpu_helpers import dev, lib

pytestmark = pytest.mark.gpu


def _tensors(v, out):
    if isinstance(v, torch.Tensor):
        out.append(v)
    elif isinstance(v, (list, tuple)):
        for u in v:
            _tensors(u, out)
    return out


def _state_tensors(s):
    return [(k, t) for k in sorted(s) for t in _tensors(s[k], [])]


def _snapshot(s):
    return [(k, t.clone()) for k, t in _state_tensors(s)]


def _restore(s, snap):
    for (k, t), (k2, c) in zip(_state_tensors(s), snap):
        assert k == k2
        t.copy_(c)


def _same(s, snap, what):
    for (k, t), (k2, c) in zip(_state_tensors(s), snap):
        assert k == k2
        a, b = t.reshape(-1).view(torch.uint8), c.reshape(-1).view(torch.uint8)
        assert torch.equal(a, b), f"{what}: '{k}' differs"


def _workloads():
    import bench
    return {
        "mha_layer": lambda: bench.MhaLayer(),                       # the full MHA layer
        "expert_batch_16": lambda: bench.ExpertBatch(n_up=8, n_down=8),
        "mla_long_t2048": lambda: bench.MlaLayer("c5", B=1, T=2048),
        "mla_layer_b2": lambda: bench.MlaLayer("c3", B=2, T=1024),
        "attn": lambda: bench.AttnLayer("attn"),                     # full size
        "attn_mla_small": lambda: bench.AttnMlaLayer(B=1, T=1024, H=8),
    }


@pytest.mark.parametrize("name", list(_workloads()))
def test_graph_replay_matches_eager_steps(name):
    lib()
    from muonclip_mc_max_gb300 import api
    from muonclip_mc_max_gb300.step import CapturedStep

    wl = _workloads()[name]()
    s = wl.make(dev())
    torch.cuda.synchronize()
    init = _snapshot(s)

    # two eager steps
    wl.step(s, api)
    torch.cuda.synchronize()
    after1 = _snapshot(s)
    wl.step(s, api)
    torch.cuda.synchronize()
    after2 = _snapshot(s)
    assert api.mc_read_device_status(clear=True) == 0

    # the captured step (its eager warm-up runs move the state on: reset it)
    graph = CapturedStep(lambda: wl.step(s, api), warmup=1)
    _restore(s, init)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    _same(s, after1, "first replay")
    graph.replay()
    torch.cuda.synchronize()
    _same(s, after2, "second replay")
    assert api.mc_read_device_status(clear=True) == 0
    del graph
