"""Newton-Schulz and Muon-step parity against the fp64 oracle: relative
Frobenius error <= 2e-2 for the orthogonalised update (bf16 operands, fp32
accumulation), momentum to fp32 rounding, weights bit-unchanged at lr = 0."""
import numpy as np
import pytest
import torch

import mc_inputs
import oracle
from gpu_helpers import NS_RTOL, dev, lib, rel_fro

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(64, 32), (32, 64), (256, 256), (200, 520), (520, 200),
                                   (1024, 1024), (576, 1024)])
def test_newton_schulz_vs_oracle(shape):
    lib()
    from muonclip_mc_max_gb300 import api
    g = mc_inputs.matrix(*shape, seed=shape[0] * 3 + shape[1])
    out = api.mc_newton_schulz([g.to(dev())])[0]
    torch.cuda.synchronize()
    ref = oracle.newton_schulz(g)
    assert rel_fro(out.cpu().numpy(), ref) < NS_RTOL


def test_newton_schulz_mixed_batch():
    """Several shapes in one call (grouped by padded shape, one launch per
    phase)."""
    lib()
    from muonclip_mc_max_gb300 import api
    shapes = [(64, 32), (300, 128), (128, 300), (256, 512), (512, 256), (96, 96)]
    mats = [mc_inputs.matrix(r, c, seed=100 + i) for i, (r, c) in enumerate(shapes)]
    outs = api.mc_newton_schulz([m.to(dev()) for m in mats])
    torch.cuda.synchronize()
    for m, o in zip(mats, outs):
        assert rel_fro(o.cpu().numpy(), oracle.newton_schulz(m)) < NS_RTOL


@pytest.mark.parametrize("steps", [0, 1, 5])
def test_newton_schulz_steps(steps):
    lib()
    from muonclip_mc_max_gb300 import api
    g = mc_inputs.matrix(128, 384, seed=7)
    out = api.mc_newton_schulz([g.to(dev())], steps=steps)[0]
    torch.cuda.synchronize()
    assert rel_fro(out.cpu().numpy(), oracle.newton_schulz(g, steps)) < NS_RTOL


@pytest.mark.parametrize("nesterov", [False, True])
def test_c1_muon_step(nesterov):
    """The tiny workload: 64 x 32 momentum, lr 2e-4, wd 0.1, RMS 0.2."""
    lib()
    from muonclip_mc_max_gb300 import api
    inp = mc_inputs.c1()
    w, g, m = inp["w"], inp["grad"], inp["m_prev"]
    wd_, gd, md = w.to(dev()), g.to(dev()), m.to(dev())
    api.mc_muon_step([wd_], [gd], [md], lr=2e-4, mu=0.95, wd=0.1, rms=0.2, nesterov=nesterov)
    torch.cuda.synchronize()
    rw, rm, ro = oracle.muon_step(w, g, m, lr=2e-4, mu=0.95, wd=0.1, rms=0.2, nesterov=nesterov)
    assert rel_fro(md.cpu().numpy(), rm) < 1e-6
    upd = (wd_.cpu().double().numpy() - w.double().numpy())
    assert rel_fro(upd, rw - w.double().numpy()) < NS_RTOL
    assert rel_fro(wd_.cpu().numpy(), rw) < 1e-5


def test_muon_batch_mixed_and_resume():
    lib()
    from muonclip_mc_max_gb300 import api
    shapes = [(256, 128), (128, 256), (384, 384)]
    W = [mc_inputs.matrix(r, c, seed=200 + i, std=0.006) for i, (r, c) in enumerate(shapes)]
    G1 = [mc_inputs.matrix(r, c, seed=300 + i, std=1e-3) for i, (r, c) in enumerate(shapes)]
    G2 = [mc_inputs.matrix(r, c, seed=400 + i, std=1e-3) for i, (r, c) in enumerate(shapes)]
    M = [mc_inputs.matrix(r, c, seed=500 + i, std=1e-3) for i, (r, c) in enumerate(shapes)]
    wd_ = [t.to(dev()) for t in W]
    md = [t.to(dev()) for t in M]
    api.mc_muon_step(wd_, [t.to(dev()) for t in G1], md, lr=2e-4)
    # save, reload, second step == continuing (the library keeps no state)
    saved_w = [t.clone() for t in wd_]
    saved_m = [t.clone() for t in md]
    api.mc_muon_step(wd_, [t.to(dev()) for t in G2], md, lr=2e-4)
    api.mc_muon_step(saved_w, [t.to(dev()) for t in G2], saved_m, lr=2e-4)
    torch.cuda.synchronize()
    for a, b in zip(wd_ + md, saved_w + saved_m):
        assert torch.equal(a, b)
    for i in range(3):
        rw, rm, _ = oracle.muon_step(W[i], G1[i], M[i], lr=2e-4)
        rw, rm, _ = oracle.muon_step(rw, G2[i], rm, lr=2e-4)
        assert rel_fro(md[i].cpu().numpy(), rm) < 1e-6
        assert rel_fro(wd_[i].cpu().double().numpy() - W[i].double().numpy(),
                       rw - W[i].double().numpy()) < NS_RTOL


def test_muon_step_many_groups_and_matrices():
    """42 matrices in seven padded-shape groups: more groups than one
    Newton-Schulz launch holds (the launch is split by group) and more
    matrices than one elementwise pass holds (the passes are split by
    matrix); every matrix against the oracle.  Beside the 2e-2 contract,
    matrices with min(rows, cols) >= 8 must stay within 6e-3: the fp16
    iterates measure at most 4.5e-3 there, where bf16 iterates gave 1-2.2%
    (990 x 40 broke the contract)."""
    lib()
    from muonclip_mc_max_gb300 import api
    groups = [
        [(32, 64), (64, 32), (50, 60), (60, 50), (10, 20), (64, 64), (1, 64)],          # 256 x 64
        [(100, 130), (130, 100), (129, 191), (191, 129), (70, 180), (180, 70), (2, 150)],  # 256 x 192
        [(60, 600), (600, 60), (90, 580), (580, 90), (5, 640), (640, 5), (200, 590)],   # 256 x 640
        [(17, 1000), (1000, 17), (40, 990), (990, 40), (8, 1024), (1024, 8), (3, 970)],  # 256 x 1024
        [(250, 260), (260, 250), (256, 300), (300, 256), (200, 290), (290, 200), (256, 320)],  # 256 x 320
        [(300, 320), (320, 300), (270, 300), (300, 270), (260, 310), (310, 260)],  # 512 x 320
        [(400, 300)],                                                                      # 512 x 448
    ]
    shapes = [s for g in groups for s in g]
    assert len(shapes) == 42
    W = [mc_inputs.matrix(r, c, seed=700 + i, std=0.02) for i, (r, c) in enumerate(shapes)]
    G = [mc_inputs.matrix(r, c, seed=800 + i, std=1e-3) for i, (r, c) in enumerate(shapes)]
    M = [mc_inputs.matrix(r, c, seed=900 + i, std=1e-3) for i, (r, c) in enumerate(shapes)]
    wd_ = [t.to(dev()) for t in W]
    md = [t.to(dev()) for t in M]
    api.mc_muon_step(wd_, [t.to(dev()) for t in G], md, lr=2e-4)
    torch.cuda.synchronize()
    assert api.mc_read_device_status(clear=True) == 0
    for i in range(len(shapes)):
        rw, rm, _ = oracle.muon_step(W[i], G[i], M[i], lr=2e-4)
        assert rel_fro(md[i].cpu().numpy(), rm) < 1e-6, shapes[i]
        err = rel_fro(wd_[i].cpu().double().numpy() - W[i].double().numpy(), rw - W[i].double().numpy())
        assert err < NS_RTOL, shapes[i]
        if min(shapes[i]) >= 8:
            assert err < 6e-3, (shapes[i], err)


def test_lr_zero_leaves_weights_bit_unchanged():
    lib()
    from muonclip_mc_max_gb300 import api
    w = mc_inputs.matrix(128, 256, seed=9)
    wd_ = w.to(dev())
    api.mc_muon_step([wd_], [mc_inputs.matrix(128, 256, seed=10).to(dev())],
                     [torch.zeros(128, 256, device=dev())], lr=0.0)
    torch.cuda.synchronize()
    assert torch.equal(wd_.cpu(), w)


def test_newton_schulz_pair_tiles_symmetric():
    """A batch large enough for 256 x 256 CTA-pair tiles whose Gram and A.A
    use the symmetric upper-tile schedule (192 symmetric against 280 full
    Gram tiles), in two shape groups: 16 wide 512 x 1024 matrices and 24 tall
    1024 x 768 ones (iterated transposed)."""
    lib()
    from muonclip_mc_max_gb300 import api
    shapes = [(512, 1024)] * 16 + [(1024, 768)] * 24
    mats = [mc_inputs.matrix(r, c, seed=700 + i) for i, (r, c) in enumerate(shapes)]
    outs = api.mc_newton_schulz([m.to(dev()) for m in mats])
    torch.cuda.synchronize()
    # several waves of pair tiles per phase: every matrix is checked
    for i in range(len(shapes)):
        assert rel_fro(outs[i].cpu().numpy(), oracle.newton_schulz_np(mats[i])) < NS_RTOL, i


def test_newton_schulz_single_cta_two_waves():
    """Three 1024 x 1024 matrices: 128 x 128 tiles on single CTAs, whose
    apply phase has 192 tiles, more than there are SMs (a second wave), while
    the symmetric Gram and A.A phases (108 tiles) fit in one.  Every matrix
    against the oracle, and a second run bit-identical to the first."""
    lib()
    from muonclip_mc_max_gb300 import api
    mats = [mc_inputs.matrix(1024, 1024, seed=950 + i) for i in range(3)]
    outs = api.mc_newton_schulz([m.to(dev()) for m in mats])
    again = api.mc_newton_schulz([m.to(dev()) for m in mats])
    torch.cuda.synchronize()
    for i in range(3):
        assert rel_fro(outs[i].cpu().numpy(), oracle.newton_schulz_np(mats[i])) < NS_RTOL, i
        assert torch.equal(outs[i], again[i]), i
