"""Pins for the fp64 oracle: each check ties it to something other than
itself -- a library routine (numpy GEMM / SVD / complex rotation), a closed
form, brute force on tiny inputs, or the checks the pages print.  A dropped
term, a wrong sign, index or transposed operand in the oracle fails one of
these.  CPU only."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import mc_inputs
import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def _bf16_grid_neighbors(x: float):
    """All bf16 values around x, by stepping the bf16 bit pattern."""
    f = np.float32(x)
    b = int(np.array([f]).view(np.uint32)[0] >> 16)
    cands = []
    for d in range(-2, 3):
        bb = (b + d) & 0xFFFF
        v = float(np.array([bb << 16], dtype=np.uint32).view(np.float32)[0])
        if math.isfinite(v):
            cands.append((bb, v))
    return cands


def _bf16_nearest_even(x: float) -> int:
    """Brute-force round-to-nearest-even onto the bf16 grid with exact
    rational distances."""
    best = None
    for bb, v in _bf16_grid_neighbors(x):
        d = abs(Fraction(v) - Fraction(x))
        key = (d, bb & 1)  # ties -> even mantissa bit
        if best is None or key < best[0]:
            best = (key, bb)
    return best[1]


def test_bf16_rounding_against_brute_force():
    rng = np.random.default_rng(0)
    vals = list(rng.standard_normal(400) * 10.0 ** rng.integers(-6, 6, 400))
    # exact ties and near-ties: bf16 midpoints +- one double ulp
    for _ in range(200):
        b = int(rng.integers(0x0080, 0x7F00)) | (int(rng.integers(0, 2)) << 15)
        lo = float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0])
        hi = float(np.array([(b + 1) << 16], dtype=np.uint32).view(np.float32)[0])
        mid = (lo + hi) / 2
        vals += [mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf)]
    for v in vals:
        got = int(oracle.f64_to_bf16_bits(np.array([v]))[0])
        assert got == _bf16_nearest_even(float(v)), v


def test_bf16_roundtrip_exact():
    bits = np.arange(0, 0x7F80, 7, dtype=np.uint16)
    vals = oracle.bf16_to_f64(bits)
    assert np.array_equal(oracle.f64_to_bf16_bits(vals), bits)


# ---------------------------------------------------------------------------
# (1) max logits -- MHA
# ---------------------------------------------------------------------------

def _np_max_logits_mha(x, wq, wk, H, dh, causal):
    """Independent formulation with library GEMMs: per (b, h) the whole
    score matrix (x Wq_h)(x Wk_h)^T, masked, then its max."""
    B, T, D = x.shape
    out = np.empty((B, H))
    for b in range(B):
        for h in range(H):
            q = x[b] @ wq[:, h * dh:(h + 1) * dh]
            k = x[b] @ wk[:, h * dh:(h + 1) * dh]
            s = q @ k.T
            if causal:
                s = np.where(np.tril(np.ones((T, T), bool)), s, -np.inf)
            out[b, h] = s.max() / math.sqrt(dh)
    return out


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(2, 7, 12, 3, 4), (1, 33, 16, 2, 8), (3, 1, 5, 4, 2)])
def test_mha_max_logits_vs_library_gemm(shape, causal):
    B, T, D, H, dh = shape
    rng = np.random.default_rng(B * 100 + T)
    x = rng.standard_normal((B, T, D))
    wq = rng.standard_normal((D, H * dh))
    wk = rng.standard_normal((D, H * dh))
    got = oracle.max_logits_mha(x, wq, wk, H, dh, causal)
    ref = _np_max_logits_mha(x, wq, wk, H, dh, causal)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_mha_subset_selection_matches_full():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 9, 8))
    wq = rng.standard_normal((8, 5 * 4))
    wk = rng.standard_normal((8, 5 * 4))
    full = oracle.max_logits_mha(x, wq, wk, 5, 4, True)
    sub = oracle.max_logits_mha(x, wq, wk, 5, 4, True, heads=[4, 1], batches=[2])
    np.testing.assert_array_equal(sub, full[[2]][:, [4, 1]])


def test_causal_single_token_is_self_dot():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 1, 6))
    wq = rng.standard_normal((6, 2 * 3))
    wk = rng.standard_normal((6, 2 * 3))
    got = oracle.max_logits_mha(x, wq, wk, 2, 3, True)
    for b in range(3):
        for h in range(2):
            q = x[b, 0] @ wq[:, 3 * h:3 * h + 3]
            k = x[b, 0] @ wk[:, 3 * h:3 * h + 3]
            assert got[b, h] == pytest.approx(q @ k / math.sqrt(3), rel=1e-13)


def test_nan_logit_propagates():
    x = np.ones((1, 3, 2))
    x[0, 1, 0] = np.nan
    w = np.ones((2, 2))
    assert np.isnan(oracle.max_logits_mha(x, w, w, 1, 2, False)[0, 0])


# ---------------------------------------------------------------------------
# (2) gamma and clip
# ---------------------------------------------------------------------------

def test_gamma_special_cases():
    tau = 100.0
    s = np.array([100.0, 200.0, -3.0, 0.0, np.nan, np.inf, 300.0, 50.0, 1e-30], np.float32)
    g, sg = oracle.gamma(s, tau)
    assert g[0] == 1.0 and g[1] == 0.5 and g[2] == 1.0 and g[3] == 1.0
    assert g[4] == 1.0 and g[5] == 0.0 and g[7] == 1.0 and g[8] == 1.0
    assert g[6] == np.float32(1.0) / np.float32(3.0)
    assert sg[1] == np.float32(math.sqrt(0.5))


def test_gamma_is_ieee_float_division():
    """RN32(tau / S) computed through double equals IEEE float division
    (numpy float32 divide and sqrt are correctly rounded)."""
    rng = np.random.default_rng(5)
    s = (rng.random(20000) * 1e4 + 1e-3).astype(np.float32)
    for tau in (100.0, 10.0, 3.3):
        g, sg = oracle.gamma(s, tau)
        ref = np.minimum(np.float32(1), np.float32(tau) / s)
        assert np.array_equal(g, ref)
        assert np.array_equal(sg, np.sqrt(ref))


def test_c1_page_checks():
    """The checks printed under the MHA semantic reference, on its own
    inputs (seed 7): after == before * gamma, after <= 10.0001, gamma <= 1."""
    ref = _gold("c1_reference.json")
    inp = mc_inputs.c1()
    assert list(inp["x"].shape) == ref["x_shape"]
    H, dh, tau = inp["H"], inp["dh"], ref["tau"]
    before = oracle.max_logits_mha(inp["x"], inp["wq"], inp["wk"], H, dh).max(axis=0)
    s32 = before.astype(np.float32)
    wq2, wk2, g = oracle.qk_clip_mha(inp["wq"], inp["wk"], H, dh, s32, tau)
    after = oracle.max_logits_mha(inp["x"], wq2, wk2, H, dh).max(axis=0)
    assert np.all(g <= ref["checks"]["gamma_upper_bound"])
    np.testing.assert_allclose(after, before * g.astype(np.float64), rtol=2e-6)
    assert np.all(after <= ref["checks"]["after_upper_bound"])
    assert np.any(g < 1.0)  # this example does clip


def test_clip_single_rounding_bf16():
    """Each scaled bf16 weight equals the exact rational product rounded
    once to bf16 (brute force)."""
    rng = np.random.default_rng(6)
    w = torch.from_numpy(rng.standard_normal((6, 2 * 5)).astype(np.float32)).to(torch.bfloat16)
    s = np.array([400.0, 50.0], np.float32)
    wq2, _, g = oracle.qk_clip_mha(w, w, 2, 5, s, 100.0)
    sg = np.float32(math.sqrt(np.float64(g[0])))
    wb = w.view(torch.int16).numpy().view(np.uint16)
    out = wq2.view(torch.int16).numpy().view(np.uint16)
    for r in range(6):
        for c in range(10):
            x = float(oracle.bf16_to_f64(wb[r, c]))
            if c < 5:
                exact = Fraction(x) * Fraction(float(sg))
                assert float(exact) == exact  # 8 x 24 bits: exact in a double
                assert out[r, c] == _bf16_nearest_even(float(exact))
            else:
                assert out[r, c] == wb[r, c]  # gamma == 1 head: untouched bits


def test_clip_fp32_matches_numpy_float32_multiply():
    rng = np.random.default_rng(7)
    w = rng.standard_normal((5, 3 * 4)).astype(np.float32)
    s = np.array([250.0, 90.0, 1000.0], np.float32)
    wq2, wk2, g = oracle.qk_clip_mha(torch.from_numpy(w), torch.from_numpy(w * 2), 3, 4, s, 100.0)
    sg = np.sqrt(g)
    ref = w.copy()
    for h in range(3):
        if g[h] != 1:
            ref[:, 4 * h:4 * h + 4] = ref[:, 4 * h:4 * h + 4] * sg[h]
    assert np.array_equal(wq2.numpy(), ref)


def test_global_clip_variant():
    rng = np.random.default_rng(8)
    w = rng.standard_normal((4, 6)).astype(np.float32)
    s = np.array([50.0, 400.0, 120.0], np.float32)
    wq2, wk2, g = oracle.qk_clip_global(torch.from_numpy(w), torch.from_numpy(w), s, 100.0, 0.25)
    assert g == np.float32(0.25)
    np.testing.assert_allclose(wq2.numpy(), w * 0.25 ** 0.25, rtol=1e-6)
    np.testing.assert_allclose(wk2.numpy(), w * 0.25 ** 0.75, rtol=1e-6)


# ---------------------------------------------------------------------------
# (1') max logits -- MLA
# ---------------------------------------------------------------------------

def _np_rope(v, base):
    """RoPE as a complex rotation: z_f = v[f] + i v[f + r/2] turned by
    exp(i t theta_f), theta_f = base^(-2f/r)."""
    T, r = v.shape
    h = r // 2
    z = v[:, :h] + 1j * v[:, h:]
    theta = base ** (-2.0 * np.arange(h) / r)
    z = z * np.exp(1j * np.arange(T)[:, None] * theta[None, :])
    return np.concatenate([z.real, z.imag], axis=1)


def _np_max_logits_mla(x, qa, qb, kva, kb, H, nope, rope, base, causal):
    B, T, D = x.shape
    kvl = kva.shape[1] - rope
    qk = nope + rope
    out = np.empty((B, H))
    for b in range(B):
        cq = x[b] @ qa
        ckv = x[b] @ kva
        kr = _np_rope(ckv[:, kvl:], base) if rope else np.zeros((T, 0))
        for h in range(H):
            qh = cq @ qb[:, h * qk:(h + 1) * qk]
            qc, qr = qh[:, :nope], qh[:, nope:]
            if rope:
                qr = _np_rope(qr, base)
            kc = ckv[:, :kvl] @ kb[:, h * nope:(h + 1) * nope]
            s = qc @ kc.T + qr @ kr.T
            if causal:
                s = np.where(np.tril(np.ones((T, T), bool)), s, -np.inf)
            out[b, h] = s.max() / math.sqrt(qk)
    return out


def _mla_rand(seed, B, T, D, H, ql, kvl, nope, rope):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, T, D)), rng.standard_normal((D, ql)) * 0.3,
            rng.standard_normal((ql, H * (nope + rope))) * 0.3,
            rng.standard_normal((D, kvl + rope)) * 0.3,
            rng.standard_normal((kvl, H * nope)) * 0.3)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("dims", [(2, 11, 10, 3, 6, 5, 4, 4), (1, 40, 8, 2, 4, 3, 2, 6)])
def test_mla_max_logits_vs_complex_rope(dims, causal):
    B, T, D, H, ql, kvl, nope, rope = dims
    x, qa, qb, kva, kb = _mla_rand(11, B, T, D, H, ql, kvl, nope, rope)
    got = oracle.max_logits_mla(x, qa, qb, kva, kb, H, nope, rope, 50000.0, causal)
    ref = _np_max_logits_mla(x, qa, qb, kva, kb, H, nope, rope, 50000.0, causal)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-11)


def test_mla_without_rope_reduces_to_mha():
    B, T, D, H, ql, kvl, nope = 2, 9, 8, 3, 5, 4, 4
    x, qa, qb, kva, kb = _mla_rand(12, B, T, D, H, ql, kvl, nope, 0)
    got = oracle.max_logits_mla(x, qa, qb, kva, kb, H, nope, 0, 50000.0, True)
    wq_eff = qa @ qb
    wk_eff = kva @ kb
    ref = oracle.max_logits_mha(x, wq_eff, wk_eff, H, nope, True)
    np.testing.assert_allclose(got, ref, rtol=1e-12)


def test_rope_logit_depends_on_relative_position_only():
    """With identical tokens, q^R_i . k^R_j depends on i - j only, and at
    position 0 the rotation is the identity."""
    T, D, H, ql, kvl, nope, rope = 12, 6, 1, 5, 3, 0, 8
    rng = np.random.default_rng(13)
    row = rng.standard_normal(D)
    x = np.tile(row, (1, T, 1))
    qa = rng.standard_normal((D, ql))
    qb = rng.standard_normal((ql, H * (nope + rope)))
    kva = rng.standard_normal((D, kvl + rope))
    kb = np.zeros((kvl, 0))
    # the max over i, j of a function of (i - j) only: every diagonal offset
    # is present at T and at T-1 with j<=i, so the causal max over the first
    # k tokens is nondecreasing in k and equal for shifted windows.
    s_full = oracle.max_logits_mla(x, qa, qb, kva, kb, H, nope, rope, 10.0, True)
    cq = row @ qa
    qr = cq @ qb
    kr = row @ kva[:, kvl:]
    h = rope // 2
    theta = 10.0 ** (-2.0 * np.arange(h) / rope)
    best = -np.inf
    for delta in range(T):
        ang = delta * theta
        zq = qr[:h] + 1j * qr[h:]
        zk = kr[:h] + 1j * kr[h:]
        best = max(best, float(np.real(np.sum(zq * np.conj(zk) * np.exp(1j * ang)))))
    assert s_full[0, 0] == pytest.approx(best / math.sqrt(rope), rel=1e-12)


def test_mla_clip_component_rules():
    """After the MLA clip every head's S scales by exactly its gamma (fp32
    storage: up to one float rounding per weight), q^R by gamma, q^C and
    k^C by sqrt(gamma), k^R (inside W_kva) and W_qa untouched; a head whose
    blocks are zero has S = 0 and gamma = 1."""
    table = _gold("mla_scaling.json")["components"]
    assert table == {"q_C": "sqrt_gamma", "k_C": "sqrt_gamma", "q_R": "gamma", "k_R": "unchanged"}
    B, T, D, H, ql, kvl, nope, rope = 2, 10, 8, 4, 6, 5, 4, 4
    x, qa, qb, kva, kb = _mla_rand(14, B, T, D, H, ql, kvl, nope, rope)
    qb[:, 1 * 8:2 * 8] *= 30.0
    kb[:, 1 * 4:2 * 4] *= 30.0
    qb[:, 3 * 8:4 * 8] = 0.0
    kb[:, 3 * 4:4 * 4] = 0.0
    qb32, kb32 = qb.astype(np.float32), kb.astype(np.float32)
    x = x * 3
    before = oracle.max_logits_mla(x, qa, qb32, kva, kb32, H, nope, rope, 50000.0, True).max(0)
    tau = float(np.float32(before[1]) / 4)
    qb2, kb2, g = oracle.qk_clip_mla(torch.from_numpy(qb32), torch.from_numpy(kb32), H, nope,
                                    rope, before.astype(np.float32), tau)
    assert before[3] == 0.0 and g[3] == 1.0
    assert g[1] < 1.0
    after = oracle.max_logits_mla(x, qa, qb2.numpy(), kva, kb2.numpy(), H, nope, rope,
                                  50000.0, True).max(0)
    np.testing.assert_allclose(after, before * g, rtol=1e-6, atol=1e-12)
    assert np.all(after <= np.maximum(before, tau) * (1 + 1e-6))
    sg = np.sqrt(g)
    for h in range(H):
        blk = qb32[:, h * 8:(h + 1) * 8]
        new = qb2.numpy()[:, h * 8:(h + 1) * 8]
        if g[h] == 1.0:
            assert np.array_equal(new, blk)
            continue
        assert np.array_equal(new[:, :nope], blk[:, :nope] * sg[h])
        assert np.array_equal(new[:, nope:], blk[:, nope:] * g[h])
        assert np.array_equal(kb2.numpy()[:, h * 4:(h + 1) * 4], kb32[:, h * 4:(h + 1) * 4] * sg[h])


# ---------------------------------------------------------------------------
# (3) Newton-Schulz and Muon
# ---------------------------------------------------------------------------

def _phi_n(s, n, coeffs):
    a, b, c = coeffs
    for _ in range(n):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def test_ns_coefficient_sign():
    gold = _gold("ns_coefficients.json")
    coeffs = (gold["a"], gold["b"], gold["c"])
    assert coeffs == oracle.NS_COEFFS
    x = np.linspace(1e-3, 1.0, 2001)
    lo, hi = gold["band_stated"]
    y = _phi_n(x, 30, coeffs)
    assert y.min() > lo - 0.03 and y.max() < hi  # stays in the stated band
    with np.errstate(over="ignore", invalid="ignore"):
        y_pos = _phi_n(x, 30, (gold["a"], -gold["b"], gold["c"]))
    assert not np.all(np.isfinite(y_pos) & (y_pos < hi))  # the + sign diverges


@pytest.mark.parametrize("shape", [(8, 20), (20, 8), (16, 16), (64, 32)])
def test_ns_equals_svd_closed_form(shape):
    """N quintic steps act on singular values: U phi^N(S / (||G||_F + eps)) V^T."""
    gold = _gold("ns_coefficients.json")
    rng = np.random.default_rng(shape[0] * 7 + shape[1])
    g = rng.standard_normal(shape)
    got = oracle.newton_schulz(g, gold["steps"], oracle.NS_COEFFS, gold["eps"])
    u, s, vt = np.linalg.svd(g, full_matrices=False)
    sn = s / (np.linalg.norm(g) + gold["eps"])
    ref = (u * _phi_n(sn, gold["steps"], oracle.NS_COEFFS)) @ vt
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-11 * np.abs(ref).max())


def test_ns_rank_one():
    rng = np.random.default_rng(21)
    u, v = rng.standard_normal(6), rng.standard_normal(15)
    g = np.outer(u, v)
    got = oracle.newton_schulz(g)
    nrm = np.linalg.norm(g)
    ref = _phi_n(nrm / (nrm + 1e-7), 5, oracle.NS_COEFFS) * g / nrm
    np.testing.assert_allclose(got, ref, atol=1e-12)


def test_ns_orthonormal_rows():
    rng = np.random.default_rng(22)
    q, _ = np.linalg.qr(rng.standard_normal((24, 9)))
    m = q.T  # 9 x 24, orthonormal rows
    got = oracle.newton_schulz(m)
    ref = _phi_n(1.0 / (3.0 + 1e-7), 5, oracle.NS_COEFFS) * m
    np.testing.assert_allclose(got, ref, atol=1e-12)


def test_ns_of_zero_is_zero():
    assert np.array_equal(oracle.newton_schulz(np.zeros((4, 6))), np.zeros((4, 6)))


def test_muon_weight_decay_only():
    rng = np.random.default_rng(23)
    w = rng.standard_normal((5, 7))
    z = np.zeros((5, 7))
    w2, m2, o = oracle.muon_step(w, z, z, lr=0.01, wd=0.1)
    np.testing.assert_allclose(w2, w * (1 - 0.01 * 0.1), rtol=1e-15)
    assert np.array_equal(m2, z) and np.array_equal(o, z)


@pytest.mark.parametrize("nesterov", [False, True])
@pytest.mark.parametrize("shape", [(12, 30), (30, 12)])
def test_muon_step_closed_form(shape, nesterov):
    """M_t = mu M + G; O = U phi^5(S) V^T of the (Nesterov) momentum;
    W_t = W - lr (0.2 sqrt(max) O + wd W)."""
    rng = np.random.default_rng(24)
    w, g, m = (rng.standard_normal(shape) for _ in range(3))
    lr, mu, wd = 2e-4, 0.95, 0.1
    w2, m2, o = oracle.muon_step(w, g, m, lr=lr, mu=mu, wd=wd, nesterov=nesterov)
    m_ref = mu * m + g
    np.testing.assert_allclose(m2, m_ref, rtol=1e-15)
    upd = g + mu * m_ref if nesterov else m_ref
    u, s, vt = np.linalg.svd(upd, full_matrices=False)
    o_ref = (u * _phi_n(s / (np.linalg.norm(upd) + 1e-7), 5, oracle.NS_COEFFS)) @ vt
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    w_ref = w - lr * (0.2 * math.sqrt(max(shape)) * o_ref + wd * w)
    np.testing.assert_allclose(w2, w_ref, rtol=1e-12, atol=1e-15)


def test_muon_update_rms_matches_lemma():
    """RMS lemma: the polar factor of a full-rank A x B matrix has RMS
    sqrt(1/max(A,B)), so 0.2 sqrt(max) O has RMS 0.2 x (singular values of
    O, which lie in the phi^5 band)."""
    rng = np.random.default_rng(25)
    A, Bc = 40, 100
    g = rng.standard_normal((A, Bc))
    w = np.zeros((A, Bc))
    w2, _, o = oracle.muon_step(w, g, np.zeros_like(g), lr=1.0, mu=0.0, wd=0.0)
    s_o = np.linalg.svd(o, compute_uv=False)
    rms = np.sqrt(np.mean(w2 ** 2))
    np.testing.assert_allclose(rms, 0.2 * math.sqrt(max(A, Bc)) * math.sqrt(np.sum(s_o ** 2) / (A * Bc)),
                               rtol=1e-12)
    band = _phi_n(np.linspace(1e-4, 1, 10001), 5, oracle.NS_COEFFS)
    u, _, vt = np.linalg.svd(g, full_matrices=False)
    polar = u @ vt
    assert np.sqrt(np.mean((0.2 * math.sqrt(max(A, Bc)) * polar) ** 2)) == pytest.approx(0.2, rel=1e-12)
    assert s_o.min() >= band.min() - 1e-9 and s_o.max() <= band.max() + 1e-9


def test_muon_two_steps_equal_save_reload():
    rng = np.random.default_rng(26)
    w, g1, g2, m = (rng.standard_normal((10, 6)) for _ in range(4))
    wa, ma, _ = oracle.muon_step(w, g1, m, lr=1e-2)
    wb, mb, _ = oracle.muon_step(wa, g2, ma, lr=1e-2)
    saved_w, saved_m = wa.copy(), ma.copy()
    wc, mc, _ = oracle.muon_step(saved_w, g2, saved_m, lr=1e-2)
    assert np.array_equal(wb, wc) and np.array_equal(mb, mc)


# ---------------------------------------------------------------------------
# the library-GEMM restatements used for full-size sampled checks
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_np_mha_matches_c_oracle(causal):
    rng = np.random.default_rng(31)
    x = rng.standard_normal((3, 70, 12))
    wq, wk = rng.standard_normal((12, 4 * 5)), rng.standard_normal((12, 4 * 5))
    a = oracle.max_logits_mha(x, wq, wk, 4, 5, causal, heads=[3, 0], batches=[2, 1])
    b = oracle.max_logits_mha_np(x, wq, wk, 4, 5, causal, heads=[3, 0], batches=[2, 1])
    np.testing.assert_allclose(b, a, rtol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_np_mla_matches_c_oracle(causal):
    x, qa, qb, kva, kb = _mla_rand(32, 2, 1100, 10, 3, 6, 5, 4, 8)  # > one 1024-row block
    a = oracle.max_logits_mla(x, qa, qb, kva, kb, 3, 4, 8, 50000.0, causal, heads=[2, 1])
    b = oracle.max_logits_mla_np(x, qa, qb, kva, kb, 3, 4, 8, 50000.0, causal, heads=[2, 1])
    np.testing.assert_allclose(b, a, rtol=1e-11)


@pytest.mark.parametrize("shape", [(40, 24), (24, 40)])
def test_np_muon_matches_c_oracle(shape):
    rng = np.random.default_rng(33)
    w, g, m = (rng.standard_normal(shape) for _ in range(3))
    for nesterov in (False, True):
        a = oracle.muon_step(w, g, m, lr=1e-3, nesterov=nesterov)
        b = oracle.muon_step_np(w, g, m, lr=1e-3, nesterov=nesterov)
        for u, v in zip(a, b):
            np.testing.assert_allclose(v, u, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(oracle.newton_schulz_np(g, 3), oracle.newton_schulz(g, 3),
                               rtol=1e-10, atol=1e-13)


# ---------------------------------------------------------------------------
# attention forward with the max logit taken along
# ---------------------------------------------------------------------------

def _qkv(B, T, H, dh, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((B, T, H * dh)) * scale for _ in range(3)]


@pytest.mark.parametrize("causal", [False, True])
def test_attention_c_matches_library_gemm_formulation(causal):
    q, k, v = _qkv(2, 13, 3, 8, 1101)
    o, s = oracle.attention_mha(q, k, v, 3, 8, causal)
    o2, s2 = oracle.attention_mha_np(q, k, v, 3, 8, causal)
    assert np.abs(o.reshape(2, 13, 3, 8) - o2).max() < 1e-12
    assert np.abs(s - s2).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_attention_zero_queries_average_the_values(causal):
    """q = 0: every logit is 0, the softmax is uniform over the allowed keys,
    so O_i is the mean of v_0..v_{i} (causal) or of all v (not causal)."""
    _, k, v = _qkv(1, 11, 2, 4, 1102)
    q = np.zeros_like(k)
    o, s = oracle.attention_mha(q, k, v, 2, 4, causal)
    for i in range(11):
        n = i + 1 if causal else 11
        assert np.allclose(o[0, i], v[0, :n].mean(axis=0), atol=1e-14)
    assert np.all(s == 0.0)


def test_attention_single_key_returns_its_value():
    q, k, v = _qkv(3, 1, 2, 8, 1103)
    o, s = oracle.attention_mha(q, k, v, 2, 8, True)
    assert np.array_equal(o, v)
    ref = (q.reshape(3, 1, 2, 8) * k.reshape(3, 1, 2, 8)).sum(-1)[:, 0] / np.sqrt(8)
    assert np.allclose(s, ref, atol=1e-14)


def test_attention_is_invariant_to_key_order():
    """Without a mask, permuting the (key, value) pairs leaves O and S alone."""
    q, k, v = _qkv(1, 9, 1, 8, 1104)
    perm = np.random.default_rng(5).permutation(9)
    o, s = oracle.attention_mha(q, k, v, 1, 8, False)
    o2, s2 = oracle.attention_mha(q, k[:, perm], v[:, perm], 1, 8, False)
    assert np.allclose(o, o2, atol=1e-13) and np.allclose(s, s2, atol=1e-13)


def test_attention_dominant_key_selects_its_value():
    """A logit 60 above all others puts weight > 1 - 1e-20 on its key."""
    q, k, v = _qkv(1, 6, 1, 4, 1105, scale=0.01)
    k[0, 3] = 0.0
    k[0, 3, 0] = 1.0
    q[0, :, :] = 0.0
    q[0, :, 0] = 60.0 * 2.0   # q.k_3 / sqrt(4) = 60; every other logit is ~0
    o, _ = oracle.attention_mha(q, k, v, 1, 4, False)
    assert np.allclose(o[0], np.broadcast_to(v[0, 3], (6, 4)), atol=1e-20 * np.abs(v).max() + 1e-24)


def test_attention_max_logit_equals_the_scan_oracle():
    """S from the attention oracle on q = x W_q, k = x W_k is the max logit
    of oracle_max_logits_mha on (x, W_q, W_k)."""
    inp = mc_inputs.mha_layer(B=2, T=40, D=24, H=3, dh=8, n_hot=1, seed=1106, muon=False,
                              w_std=0.3)
    x = inp["x"].double().numpy()
    wq, wk = inp["wq"].double().numpy(), inp["wk"].double().numpy()
    q, k = x @ wq, x @ wk
    for causal in (False, True):
        _, s = oracle.attention_mha(q, k, np.zeros_like(q), 3, 8, causal)
        ref = oracle.max_logits_mha(inp["x"], inp["wq"], inp["wk"], 3, 8, causal)
        assert np.allclose(s, ref, rtol=1e-12, atol=0)


def test_attention_nan_logit_propagates():
    q, k, v = _qkv(1, 5, 1, 4, 1107)
    q[0, 2, 1] = np.nan
    o, s = oracle.attention_mha(q, k, v, 1, 4, True)
    assert np.isnan(s).all() and np.isnan(o[0, 2]).all() and np.isfinite(o[0, 1]).all()


# ---------------------------------------------------------------------------
# MLA attention forward with the max logit taken along
# ---------------------------------------------------------------------------

def _mla_qkv(B, T, H, nope, rope, dv, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H * (nope + rope))) * scale
    kc = rng.standard_normal((B, T, H * nope))
    kr = rng.standard_normal((B, T, rope))
    v = rng.standard_normal((B, T, H * dv))
    return q, kc, kr, v


@pytest.mark.parametrize("causal", [False, True])
def test_attention_mla_reduces_to_mha_with_shared_rope_keys(causal):
    """MLA attention is MHA attention over d = nope + rope once every head's
    key is [k^C_h | k^R] (the shared k^R repeated per head) and the values
    are padded with zeros to d: the MHA output's first dv columns of each
    head, and its max logit, are the MLA ones."""
    B, T, H, nope, rope, dv = 2, 9, 3, 6, 4, 7
    q, kc, kr, v = _mla_qkv(B, T, H, nope, rope, dv, 1201)
    dq = nope + rope
    k_full = np.concatenate([np.concatenate([kc[..., h * nope:(h + 1) * nope], kr], axis=-1)
                             for h in range(H)], axis=-1)
    v_pad = np.concatenate([np.concatenate([v[..., h * dv:(h + 1) * dv],
                                            np.zeros((B, T, dq - dv))], axis=-1) for h in range(H)],
                           axis=-1)
    o, s = oracle.attention_mla(q, kc, kr, v, H, nope, rope, dv, causal)
    o2, s2 = oracle.attention_mha(q, k_full, v_pad, H, dq, causal)
    o2 = o2.reshape(B, T, H, dq)
    assert np.allclose(o.reshape(B, T, H, dv), o2[..., :dv], rtol=1e-13, atol=1e-14)
    assert np.all(o2[..., dv:] == 0.0)
    assert np.allclose(s, s2, rtol=1e-14, atol=0)


def test_attention_mla_c_matches_library_gemm_formulation():
    q, kc, kr, v = _mla_qkv(2, 11, 2, 8, 4, 5, 1202)
    for causal in (False, True):
        o, s = oracle.attention_mla(q, kc, kr, v, 2, 8, 4, 5, causal)
        o2, s2 = oracle.attention_mla_np(q, kc, kr, v, 2, 8, 4, 5, causal)
        assert np.abs(o.reshape(2, 11, 2, 5) - o2).max() < 1e-12
        assert np.abs(s - s2).max() < 1e-12


def test_attention_mla_without_query_rope_ignores_the_shared_key_rope():
    """q^R = 0: the rope term vanishes, so replacing k^R changes nothing."""
    q, kc, kr, v = _mla_qkv(1, 8, 2, 6, 4, 3, 1203)
    q = q.reshape(1, 8, 2, 10)
    q[..., 6:] = 0.0
    q = q.reshape(1, 8, 20)
    o, s = oracle.attention_mla(q, kc, kr, v, 2, 6, 4, 3, True)
    o2, s2 = oracle.attention_mla(q, kc, 5.0 * kr + 3.0, v, 2, 6, 4, 3, True)
    assert np.array_equal(o, o2) and np.array_equal(s, s2)


def test_attention_mla_single_key_returns_its_value():
    q, kc, kr, v = _mla_qkv(2, 1, 3, 4, 2, 5, 1204)
    o, s = oracle.attention_mla(q, kc, kr, v, 3, 4, 2, 5, True)
    assert np.array_equal(o, v)
    qh, kch = q.reshape(2, 3, 6), kc.reshape(2, 3, 4)
    ref = ((qh[..., :4] * kch).sum(-1) + (qh[..., 4:] * kr.reshape(2, 1, 2)).sum(-1)) / np.sqrt(6)
    assert np.allclose(s, ref, atol=1e-14)


def test_attention_mla_max_logit_equals_the_scan_oracle():
    """S from the MLA attention oracle on the layer's projections (q^C, q^R,
    k^C, k^R with RoPE) is the max logit of oracle_max_logits_mla on (x, W)."""
    inp = mc_inputs.mla_layer(B=2, T=24, D=32, H=2, q_lora=16, kv_lora=12, nope=8, rope=4, n_hot=1,
                              w_std=0.3, seed=1205)
    x = inp["x"].double().numpy()
    qa, qb, kva, kb = (inp[n].double().numpy() for n in ("w_qa", "w_qb", "w_kva", "w_kb"))
    H, nope, rope, base = 2, 8, 4, inp["rope_base"]
    q = np.empty((2, 24, H * 12))
    kc = np.empty((2, 24, H * nope))
    kr = np.empty((2, 24, rope))
    for b in range(2):
        cq, ckv = x[b] @ qa, x[b] @ kva
        kr[b] = oracle._rope_np(ckv[:, 12:], 0, base)
        for h in range(H):
            qh = cq @ qb[:, h * 12:(h + 1) * 12]
            q[b, :, h * 12:h * 12 + nope] = qh[:, :nope]
            q[b, :, h * 12 + nope:(h + 1) * 12] = oracle._rope_np(qh[:, nope:], 0, base)
            kc[b, :, h * nope:(h + 1) * nope] = ckv[:, :12] @ kb[:, h * nope:(h + 1) * nope]
    for causal in (True, False):
        _, s = oracle.attention_mla(q, kc, kr, np.zeros((2, 24, H)), H, nope, rope, 1, causal)
        ref = oracle.max_logits_mla(inp["x"], inp["w_qa"], inp["w_qb"], inp["w_kva"], inp["w_kb"], H,
                                    nope, rope, base, causal)
        assert np.allclose(s, ref, rtol=1e-12, atol=0)
