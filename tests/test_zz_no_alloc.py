"""The allocation-free scan entry point, mc_max_logits_mha_noalloc.

It serves callers that may not allocate device memory when they run the
scan (a plugin inside a framework that owns every device allocation, or code
running while its stream is captured into a CUDA graph): instead of a
caller workspace it uses the library's own static device scratch.  Called
here straight through the C ABI (ctypes) and checked against the
workspace-taking entry point on the same inputs, twice in a row (the
scratch keeps the previous call's contents, so the second call shows that
what must start at zero is cleared).  Collected last on purpose."""
import ctypes

import pytest
import torch

import mc_inputs
from gpu_helpers import SMAX_RTOL, dev, lib, rel_err

pytestmark = pytest.mark.gpu


def _vp(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point():
    L = lib()
    from muonclip_mc_max_gb300 import api
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for causal, seed in ((False, 301), (True, 302)):
        inp = mc_inputs.mha_layer(B=2, T=300, D=192, H=3, dh=64, n_hot=1, seed=seed,
                                  causal=causal, muon=False, w_std=0.05)
        x, wq, wk = (inp[k].to(dev()) for k in ("x", "wq", "wk"))
        B, T, D, H, dh = 2, 300, 192, 3, 64
        ref = torch.empty(H, dtype=torch.float32, device=dev())
        ref_bh = torch.empty(B, H, dtype=torch.float32, device=dev())
        api.mc_max_logits_mha(x, wq, wk, H, dh, causal=causal, s_max=ref, s_max_bh=ref_bh)
        for _ in range(2):  # two calls in a row share (and reuse) the static scratch
            got = torch.full((H,), -1.0, dtype=torch.float32, device=dev())
            got_bh = torch.full((B, H), -1.0, dtype=torch.float32, device=dev())
            st = L.mc_max_logits_mha_noalloc(_vp(x), _vp(wq), _vp(wk), api.MC_BF16, B, T, D, H,
                                             dh, int(causal), 0, _vp(got), _vp(got_bh), stream)
            assert st == 0, api.mc_status_string(st)
            torch.cuda.synchronize()
            assert rel_err(got.cpu().numpy(), ref.cpu().numpy()).max() < SMAX_RTOL
            assert rel_err(got_bh.cpu().numpy(), ref_bh.cpu().numpy()).max() < SMAX_RTOL
    assert api.mc_read_device_status(clear=True) == 0


def test_noalloc_rejects_sizes_beyond_the_scratch():
    L = lib()
    from muonclip_mc_max_gb300 import api
    B, T, D, H, dh = 16, 4096, 1024, 16, 64  # needs 4 GiB of scratch
    assert api.mc_max_logits_mha_workspace_size(B, T, D, H, dh) > api.MC_NOALLOC_SCRATCH_BYTES
    dummy = torch.empty(16, device=dev())
    st = L.mc_max_logits_mha_noalloc(_vp(dummy), _vp(dummy), _vp(dummy), api.MC_BF16, B, T, D, H,
                                     dh, 0, 0, _vp(dummy), None,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 4  # MC_ERR_WORKSPACE, nothing enqueued
