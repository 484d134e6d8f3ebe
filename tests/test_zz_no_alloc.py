"""The allocation-free scan entry point, mc_max_logits_mha_noalloc.

It serves callers that may not allocate device memory when they run the
scan (a plugin inside a framework that owns every device allocation, or code
running while its stream is captured into a CUDA graph): instead of a
caller workspace it uses the library's own static device scratch.  Called
here straight through the C ABI (ctypes) and through its Python wrapper,
and checked against the fp64 oracle and the workspace-taking entry point on
the same inputs.
Two calls in a row use different inputs, the second with logits 100 times
smaller: the scratch keeps the first call's maximum keys, so the second
result is only right if each call clears what must start at zero.
Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import mc_inputs
import oracle
from gpu_helpers import SMAX_RTOL, dev, lib, rel_err

pytestmark = pytest.mark.gpu


def _vp(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point():
    L = lib()
    from muonclip_mc_max_gb300 import api
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    B, T, D, H, dh = 2, 300, 192, 3, 64
    for causal, seed in ((False, 301), (True, 302)):
        inp = mc_inputs.mha_layer(B=B, T=T, D=D, H=H, dh=dh, n_hot=1, seed=seed,
                                  causal=causal, muon=False, w_std=0.05)
        x, wq, wk = (inp[k].to(dev()) for k in ("x", "wq", "wk"))
        prev = None
        # second call: W_q scaled by 0.01 and rounded to bf16, so every
        # head's S_max drops about 100-fold
        for wq_call in (wq, (wq.float() * 0.01).to(torch.bfloat16)):
            ref = torch.empty(H, dtype=torch.float32, device=dev())
            ref_bh = torch.empty(B, H, dtype=torch.float32, device=dev())
            api.mc_max_logits_mha(x, wq_call, wk, H, dh, causal=causal, s_max=ref, s_max_bh=ref_bh)
            got = torch.full((H,), -1.0, dtype=torch.float32, device=dev())
            got_bh = torch.full((B, H), -1.0, dtype=torch.float32, device=dev())
            st = L.mc_max_logits_mha_noalloc(_vp(x), _vp(wq_call), _vp(wk), api.MC_BF16, B, T, D,
                                             H, dh, int(causal), 0, _vp(got), _vp(got_bh), stream)
            assert st == 0, api.mc_status_string(st)
            torch.cuda.synchronize()
            r = ref.cpu().numpy()
            ref_o = oracle.max_logits_mha(inp["x"], wq_call.cpu(), inp["wk"], H, dh, causal)
            assert rel_err(got_bh.cpu().numpy(), ref_o).max() < SMAX_RTOL
            assert rel_err(got.cpu().numpy(), ref_o.max(0)).max() < SMAX_RTOL
            assert rel_err(got.cpu().numpy(), r).max() < SMAX_RTOL
            assert rel_err(got_bh.cpu().numpy(), ref_bh.cpu().numpy()).max() < SMAX_RTOL
            if prev is not None:
                assert (r < 0.05 * prev).all()  # stale keys would have kept the first maxima
            prev = r
            # the Python wrapper of the same entry point, without s_max_bh
            w = api.mc_max_logits_mha_noalloc(x, wq_call, wk, H, dh, causal=causal)
            torch.cuda.synchronize()
            assert np.array_equal(w.cpu().numpy(), got.cpu().numpy())
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
