"""Failure detection on the GPU without a fault.

Every on-chip wait of the library is bounded: when it expires it sets
MC_DEV_TIMEOUT in the device status word and raises its CTA's abort flag, so
the CTA's other waits end too and the kernel returns.  The self-test entry
point runs that same wait on barriers that nothing completes (one waiter
with a short limit, one with the normal 1 s limit).  Nothing faults, traps or
hangs; the host reads the status and the context goes on working."""
import time

import numpy as np
import pytest
import torch

import mc_inputs
import oracle
from gpu_helpers import SMAX_RTOL, dev, lib

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_the_context_stays_usable():
    lib()
    from muonclip_mc_max_gb300 import api
    api.mc_read_device_status(clear=True)
    limit_us = 20000
    t0 = time.perf_counter()
    out = api.mc_selftest_wait_timeout(limit_us)
    bits = api.mc_read_device_status(clear=True)
    wall = time.perf_counter() - t0
    short_ns, normal_ns, short_done, normal_done = out.cpu().tolist()
    assert bits & api.MC_DEV_TIMEOUT
    assert short_done == 0 and normal_done == 0
    # the short-limit waiter gave up just after its limit ...
    assert limit_us * 1000 <= short_ns < limit_us * 1000 + 50_000_000
    # ... and the other left on the abort flag, long before its own 1 s
    assert normal_ns < 500_000_000
    assert wall < 0.9

    # the context still works: a scan matches the oracle and sets no status
    inp = mc_inputs.mha_layer(B=2, T=200, D=128, H=2, dh=64, n_hot=1, seed=951, muon=False,
                              w_std=0.05)
    s_bh = torch.empty(2, 2, dtype=torch.float32, device=dev())
    api.mc_max_logits_mha(inp["x"].to(dev()), inp["wq"].to(dev()), inp["wk"].to(dev()), 2, 64,
                          s_max_bh=s_bh)
    assert api.mc_read_device_status(clear=True) == 0
    ref = oracle.max_logits_mha(inp["x"], inp["wq"], inp["wk"], 2, 64, False)
    np.testing.assert_allclose(s_bh.cpu().numpy(), ref, rtol=SMAX_RTOL, atol=0)
