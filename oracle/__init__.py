"""fp64 CPU oracle for the MuonClip optimizer step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``mc_oracle.c`` (plain C,
double precision, OpenMP) through ctypes and converts torch / numpy inputs
to float64 exactly (bf16 and fp32 up-cast without rounding).  It shares no
code with the CUDA library under ``muonclip_mc_max_gb300/``.

Definitions followed (see the header of ``mc_oracle.c`` for the full list):
  * S_max^h = max_{X,i,j} Q_i^h K_j^h / sqrt(d) -- "Kimi K2: 1T MoE, MuonClip
    and Agentic training system", section on attention-logit growth; Kimi K2
    section 2.1 "MuonClip".
  * gamma_h = min(1, tau / S_max^h), MHA sqrt(gamma) clip, MLA table -- same
    review, sections on the MHA clip and "MLA asymmetric scaling".
  * Muon momentum, quintic Newton-Schulz, RMS matching 0.2*sqrt(max(A,B)),
    decoupled weight decay -- "Notes on Moonlight" ("Background",
    "Scaling up Muon"), "Notes on Muon blog" ("Newton-Schulz", "Algorithm").
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build as _build, library_path

__all__ = [
    "NS_COEFFS", "load", "bf16_to_f64", "f64_to_bf16_bits", "max_logits_mha",
    "max_logits_mla", "gamma", "qk_clip_mha", "qk_clip_mla", "qk_clip_global",
    "newton_schulz", "muon_step", "max_logits_mha_np", "max_logits_mla_np", "newton_schulz_np",
    "muon_step_np", "attention_mha", "attention_mha_np", "attention_mla", "attention_mla_np",
]

# Quintic coefficients (a, b, c) of "Notes on Muon blog", section "Algorithm";
# the sign of b follows the printed pseudocode (negative) -- the positive
# sign printed in the prose diverges (phi(1) = 10.25), see the pins.
NS_COEFFS = (3.4445, -4.7750, 2.0315)

_lib = None
_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_ip = ctypes.POINTER(ctypes.c_int)
_u16p = ctypes.POINTER(ctypes.c_uint16)


def load():
    """Build (if needed) and load the oracle shared library."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        _build()
    lib = ctypes.CDLL(path)
    I, D, L, F, V = ctypes.c_int, ctypes.c_double, ctypes.c_long, ctypes.c_float, ctypes.c_void_p
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = D
    lib.oracle_f64_to_bf16.argtypes = [D]
    lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
    lib.oracle_max_logits_mha.argtypes = [_dp, I, I, I, _dp, _dp, I, I, I, _ip, I, _ip, I, _dp]
    lib.oracle_max_logits_mha.restype = I
    lib.oracle_max_logits_mla.argtypes = [_dp, I, I, I, _dp, I, _dp, _dp, I, _dp,
                                          I, I, I, D, I, _ip, I, _ip, I, _dp]
    lib.oracle_max_logits_mla.restype = I
    lib.oracle_attention_mha.argtypes = [_dp, _dp, _dp, I, I, I, I, I, _dp, _dp]
    lib.oracle_attention_mha.restype = I
    lib.oracle_attention_mla.argtypes = [_dp, _dp, _dp, _dp, I, I, I, I, I, I, I, _dp, _dp]
    lib.oracle_attention_mla.restype = I
    lib.oracle_gamma.argtypes = [_fp, I, F, _fp, _fp]
    lib.oracle_gamma.restype = None
    lib.oracle_qk_clip_mha.argtypes = [V, V, I, I, I, I, _fp, F, _fp]
    lib.oracle_qk_clip_mha.restype = None
    lib.oracle_qk_clip_mla.argtypes = [V, V, I, I, I, I, I, I, _fp, F, _fp]
    lib.oracle_qk_clip_mla.restype = None
    lib.oracle_qk_clip_global.argtypes = [V, V, I, I, I, _fp, I, F, F, _fp]
    lib.oracle_qk_clip_global.restype = None
    lib.oracle_newton_schulz.argtypes = [_dp, I, I, I, D, D, D, D, _dp]
    lib.oracle_newton_schulz.restype = I
    lib.oracle_muon_step.argtypes = [_dp, _dp, _dp, I, I, D, D, D, D, I, D, D, D, D, I, _dp]
    lib.oracle_muon_step.restype = I
    _lib = lib
    return lib


# ---------------------------------------------------------------------------
# conversions
# ---------------------------------------------------------------------------

def _to_f64(a) -> np.ndarray:
    """Exact up-cast of a torch tensor (bf16/fp16/fp32/fp64) or array to a
    C-contiguous float64 numpy array."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return np.ascontiguousarray(a.detach().to("cpu").double().numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray, typ=_dp):
    return a.ctypes.data_as(typ)


def _intlist(v):
    if v is None:
        return None, 0
    arr = np.ascontiguousarray(np.asarray(v, dtype=np.int32))
    return arr, len(arr)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns with a single round-to-nearest-even."""
    lib = load()
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    flat, oflat = x.ravel(), out.ravel()
    for i in range(flat.size):
        oflat[i] = lib.oracle_f64_to_bf16(float(flat[i]))
    return out


# ---------------------------------------------------------------------------
# (1) max logits
# ---------------------------------------------------------------------------

def max_logits_mha(x, wq, wk, H: int, dh: int, causal: bool = False,
                   heads=None, batches=None) -> np.ndarray:
    """Per-(batch, head) S = max_{i,j} q_i.k_j / sqrt(dh) in fp64.

    x [B, T, D]; wq, wk [D, H*dh].  Returns [len(batches), len(heads)]
    (all batches / heads when None).  S_max^h is the max over axis 0."""
    lib = load()
    X, WQ, WK = _to_f64(x), _to_f64(wq), _to_f64(wk)
    B, T, D = X.shape
    assert WQ.shape == (D, H * dh) and WK.shape == (D, H * dh)
    hs, nh = _intlist(heads)
    bs, nb = _intlist(batches)
    out = np.empty(((nb if bs is not None else B), (nh if hs is not None else H)))
    rc = lib.oracle_max_logits_mha(_ptr(X), B, T, D, _ptr(WQ), _ptr(WK), H, dh, int(causal),
                                   None if hs is None else _ptr(hs, _ip), nh,
                                   None if bs is None else _ptr(bs, _ip), nb, _ptr(out))
    if rc:
        raise RuntimeError(f"oracle_max_logits_mha failed ({rc})")
    return out


def max_logits_mla(x, w_qa, w_qb, w_kva, w_kb, H: int, nope: int, rope: int,
                   rope_base: float, causal: bool = True, heads=None, batches=None) -> np.ndarray:
    """Per-(batch, head) MLA S = max (q^C.k^C + q^R.k^R) / sqrt(nope+rope).

    x [B, T, D]; w_qa [D, q_lora]; w_qb [q_lora, H*(nope+rope)];
    w_kva [D, kv_lora+rope]; w_kb [kv_lora, H*nope]."""
    lib = load()
    X = _to_f64(x)
    QA, QB, KVA, KB = _to_f64(w_qa), _to_f64(w_qb), _to_f64(w_kva), _to_f64(w_kb)
    B, T, D = X.shape
    q_lora = QA.shape[1]
    kv_lora = KVA.shape[1] - rope
    assert QA.shape == (D, q_lora) and QB.shape == (q_lora, H * (nope + rope))
    assert KVA.shape == (D, kv_lora + rope) and KB.shape == (kv_lora, H * nope)
    hs, nh = _intlist(heads)
    bs, nb = _intlist(batches)
    out = np.empty(((nb if bs is not None else B), (nh if hs is not None else H)))
    rc = lib.oracle_max_logits_mla(_ptr(X), B, T, D, _ptr(QA), q_lora, _ptr(QB), _ptr(KVA),
                                   kv_lora, _ptr(KB), H, nope, rope, float(rope_base),
                                   int(causal), None if hs is None else _ptr(hs, _ip), nh,
                                   None if bs is None else _ptr(bs, _ip), nb, _ptr(out))
    if rc:
        raise RuntimeError(f"oracle_max_logits_mla failed ({rc})")
    return out


# ---------------------------------------------------------------------------
# (2) gamma and QK-Clip
# ---------------------------------------------------------------------------

def attention_mha(q, k, v, H: int, dh: int, causal: bool = False):
    """Softmax attention forward in fp64 with the max logit taken along.

    q, k, v [B, T, H*dh] (head h = column block h).  Returns (o [B, T, H*dh],
    s_bh [B, H]) with s_bh = max_{i,j} q_i.k_j / sqrt(dh) over allowed pairs."""
    lib = load()
    Q, K, V = _to_f64(q), _to_f64(k), _to_f64(v)
    B, T, W = Q.shape
    assert W == H * dh and K.shape == Q.shape and V.shape == Q.shape
    o = np.empty_like(Q)
    s = np.empty((B, H))
    rc = lib.oracle_attention_mha(_ptr(Q), _ptr(K), _ptr(V), B, T, H, dh, int(causal), _ptr(o),
                                  _ptr(s))
    if rc:
        raise RuntimeError(f"oracle_attention_mha failed ({rc})")
    return o, s


def attention_mla(q, k_c, k_r, v, H: int, nope: int, rope: int, dv: int, causal: bool = True):
    """MLA softmax attention forward in fp64 with the max logit taken along.

    q [B, T, H*(nope+rope)] (per head q^C then q^R, RoPE applied), k_c
    [B, T, H*nope], k_r [B, T, rope] (shared by every head), v [B, T, H*dv].
    Returns (o [B, T, H*dv], s_bh [B, H]) with s_bh = max_{i,j} (q^C_i.k^C_j
    + q^R_i.k^R_j) / sqrt(nope + rope) over allowed pairs."""
    lib = load()
    Q, KC, KR, V = _to_f64(q), _to_f64(k_c), _to_f64(k_r), _to_f64(v)
    B, T, W = Q.shape
    assert W == H * (nope + rope) and KC.shape == (B, T, H * nope) and KR.shape == (B, T, rope)
    assert V.shape == (B, T, H * dv)
    o = np.empty((B, T, H * dv))
    s = np.empty((B, H))
    rc = lib.oracle_attention_mla(_ptr(Q), _ptr(KC), _ptr(KR), _ptr(V), B, T, H, nope, rope, dv,
                                  int(causal), _ptr(o), _ptr(s))
    if rc:
        raise RuntimeError(f"oracle_attention_mla failed ({rc})")
    return o, s


def gamma(s_max, tau: float):
    """(gamma, sqrt_gamma) as float32 arrays from float32 S_max."""
    lib = load()
    s = np.ascontiguousarray(np.asarray(s_max, dtype=np.float32))
    g = np.empty_like(s)
    sg = np.empty_like(s)
    lib.oracle_gamma(_ptr(s, _fp), s.size, float(tau), _ptr(g, _fp), _ptr(sg, _fp))
    return g, sg


def _weight_buf(w):
    """A writable contiguous numpy buffer of the storage format (bf16 bits
    as uint16, or float32) plus a flag telling which."""
    import torch
    if isinstance(w, torch.Tensor):
        w = w.detach().to("cpu").contiguous()
        if w.dtype == torch.bfloat16:
            return w.view(torch.int16).numpy().view(np.uint16).copy(), 1
        if w.dtype == torch.float32:
            return w.numpy().copy(), 0
        raise TypeError(f"unsupported weight dtype {w.dtype}")
    arr = np.asarray(w)
    if arr.dtype == np.uint16:
        return np.ascontiguousarray(arr).copy(), 1
    return np.ascontiguousarray(arr, dtype=np.float32).copy(), 0


def _weight_out(buf, is_bf16):
    import torch
    t = torch.from_numpy(buf)
    return t.view(torch.bfloat16) if is_bf16 else t


def qk_clip_mha(wq, wk, H: int, dh: int, s_max, tau: float):
    """Returns (wq', wk', gamma): new weights in the input storage format."""
    lib = load()
    bq, fq = _weight_buf(wq)
    bk, fk = _weight_buf(wk)
    assert fq == fk
    D = bq.shape[0]
    s = np.ascontiguousarray(np.asarray(s_max, dtype=np.float32))
    g = np.empty(H, dtype=np.float32)
    lib.oracle_qk_clip_mha(bq.ctypes.data, bk.ctypes.data, fq, D, H, dh, _ptr(s, _fp),
                           float(tau), _ptr(g, _fp))
    return _weight_out(bq, fq), _weight_out(bk, fk), g


def qk_clip_mla(w_qb, w_kb, H: int, nope: int, rope: int, s_max, tau: float):
    """Returns (w_qb', w_kb', gamma).  W_qa and W_kva are never changed."""
    lib = load()
    bq, fq = _weight_buf(w_qb)
    bk, fk = _weight_buf(w_kb)
    assert fq == fk
    s = np.ascontiguousarray(np.asarray(s_max, dtype=np.float32))
    g = np.empty(H, dtype=np.float32)
    lib.oracle_qk_clip_mla(bq.ctypes.data, bk.ctypes.data, fq, bq.shape[0], bk.shape[0], H,
                           nope, rope, _ptr(s, _fp), float(tau), _ptr(g, _fp))
    return _weight_out(bq, fq), _weight_out(bk, fk), g


def qk_clip_global(wq, wk, s_max, tau: float, alpha: float = 0.5):
    """All-heads variant: one gamma from max_h S^h, W_q x gamma^alpha,
    W_k x gamma^(1-alpha).  Returns (wq', wk', gamma)."""
    lib = load()
    bq, fq = _weight_buf(wq)
    bk, fk = _weight_buf(wk)
    s = np.ascontiguousarray(np.asarray(s_max, dtype=np.float32))
    g = np.empty(1, dtype=np.float32)
    lib.oracle_qk_clip_global(bq.ctypes.data, bk.ctypes.data, fq, bq.shape[0], bq.shape[1],
                              _ptr(s, _fp), s.size, float(tau), float(alpha), _ptr(g, _fp))
    return _weight_out(bq, fq), _weight_out(bk, fk), float(g[0])


# ---------------------------------------------------------------------------
# (3) Muon
# ---------------------------------------------------------------------------

def newton_schulz(g, steps: int = 5, coeffs=NS_COEFFS, eps: float = 1e-7) -> np.ndarray:
    lib = load()
    G = _to_f64(g)
    rows, cols = G.shape
    out = np.empty_like(G)
    a, b, c = coeffs
    rc = lib.oracle_newton_schulz(_ptr(G), rows, cols, steps, a, b, c, eps, _ptr(out))
    if rc:
        raise RuntimeError(f"oracle_newton_schulz failed ({rc})")
    return out


def muon_step(w, g, m, lr: float, mu: float = 0.95, wd: float = 0.1, rms: float = 0.2,
              steps: int = 5, coeffs=NS_COEFFS, eps: float = 1e-7, nesterov: bool = False):
    """One Muon step in fp64.  Returns (w_new, m_new, o) as float64 arrays."""
    lib = load()
    W, G, M = _to_f64(w).copy(), _to_f64(g), _to_f64(m).copy()
    rows, cols = W.shape
    O = np.empty_like(W)
    a, b, c = coeffs
    rc = lib.oracle_muon_step(_ptr(W), _ptr(G), _ptr(M), rows, cols, lr, mu, wd, rms, steps,
                              a, b, c, eps, int(nesterov), _ptr(O))
    if rc:
        raise RuntimeError(f"oracle_muon_step failed ({rc})")
    return W, M, O


# ---------------------------------------------------------------------------
# Library-GEMM restatements (numpy fp64 BLAS) for full-size sampled checks.
# Same definitions, steps in the same order; the matrix products run in a
# library routine so the large workloads finish in seconds.  Pinned against
# the plain-loop C functions above (tests/test_oracle_pins.py).
# ---------------------------------------------------------------------------

def _rope_np(v: np.ndarray, pos0: int, base: float) -> np.ndarray:
    """Rotate-half RoPE of rows v[t] at positions pos0 + t (fp64)."""
    T, r = v.shape
    h = r // 2
    theta = base ** (-2.0 * np.arange(h) / r)
    ang = (pos0 + np.arange(T))[:, None].astype(np.float64) * theta[None, :]
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = v[:, :h], v[:, h:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=1)


def _pair_max(q: np.ndarray, k: np.ndarray, causal: bool, block: int = 1024) -> float:
    """max over i, j (j <= i if causal) of q_i . k_j, computed in row blocks."""
    T = q.shape[0]
    best = -np.inf
    for i0 in range(0, T, block):
        i1 = min(T, i0 + block)
        jend = i1 if causal else T
        s = q[i0:i1] @ k[:jend].T
        if causal:
            s = np.where(np.arange(jend)[None, :] <= np.arange(i0, i1)[:, None], s, -np.inf)
        if np.isnan(s).any():
            return float("nan")
        best = max(best, float(s.max()))
    return best


def max_logits_mha_np(x, wq, wk, H, dh, causal=False, heads=None, batches=None) -> np.ndarray:
    """As max_logits_mha, with library GEMMs (fp64)."""
    heads = list(range(H)) if heads is None else list(heads)
    B = x.shape[0]
    batches = list(range(B)) if batches is None else list(batches)
    WQ, WK = _to_f64(wq), _to_f64(wk)
    out = np.empty((len(batches), len(heads)))
    for ib, b in enumerate(batches):
        xb = _to_f64(x[b])
        for ih, h in enumerate(heads):
            q = xb @ WQ[:, h * dh:(h + 1) * dh]
            k = xb @ WK[:, h * dh:(h + 1) * dh]
            out[ib, ih] = _pair_max(q, k, causal) / np.sqrt(dh)
    return out


def max_logits_mla_np(x, w_qa, w_qb, w_kva, w_kb, H, nope, rope, rope_base, causal=True,
                      heads=None, batches=None) -> np.ndarray:
    """As max_logits_mla, with library GEMMs (fp64)."""
    heads = list(range(H)) if heads is None else list(heads)
    B = x.shape[0]
    batches = list(range(B)) if batches is None else list(batches)
    QA, QB, KVA, KB = _to_f64(w_qa), _to_f64(w_qb), _to_f64(w_kva), _to_f64(w_kb)
    kvl = KVA.shape[1] - rope
    qk = nope + rope
    out = np.empty((len(batches), len(heads)))
    for ib, b in enumerate(batches):
        xb = _to_f64(x[b])
        cq = xb @ QA
        ckv = xb @ KVA
        kr = _rope_np(ckv[:, kvl:], 0, rope_base)
        for ih, h in enumerate(heads):
            qh = cq @ QB[:, h * qk:(h + 1) * qk]
            q = np.concatenate([qh[:, :nope], _rope_np(qh[:, nope:], 0, rope_base)], axis=1)
            kc = ckv[:, :kvl] @ KB[:, h * nope:(h + 1) * nope]
            k = np.concatenate([kc, kr], axis=1)
            out[ib, ih] = _pair_max(q, k, causal) / np.sqrt(qk)
    return out


def attention_mha_np(q, k, v, H: int, dh: int, causal: bool = False, batches=None, heads=None):
    """As attention_mha, with library GEMMs (fp64), for the listed
    (batch, head) pairs: returns (o [nb, T, nh, dh], s_bh [nb, nh])."""
    Q, K, V = _to_f64(q), _to_f64(k), _to_f64(v)
    B, T, _ = Q.shape
    batches = list(range(B)) if batches is None else list(batches)
    heads = list(range(H)) if heads is None else list(heads)
    o = np.empty((len(batches), T, len(heads), dh))
    s_bh = np.empty((len(batches), len(heads)))
    mask = np.tril(np.ones((T, T), dtype=bool)) if causal else np.ones((T, T), dtype=bool)
    for ib, b in enumerate(batches):
        for ih, h in enumerate(heads):
            cols = slice(h * dh, (h + 1) * dh)
            s = (Q[b][:, cols] @ K[b][:, cols].T) / np.sqrt(dh)
            s = np.where(mask, s, -np.inf)
            s_bh[ib, ih] = s.max()
            p = np.exp(s - s.max(axis=1, keepdims=True))
            o[ib, :, ih] = (p @ V[b][:, cols]) / p.sum(axis=1, keepdims=True)
    return o, s_bh


def attention_mla_np(q, k_c, k_r, v, H: int, nope: int, rope: int, dv: int, causal: bool = True,
                     batches=None, heads=None):
    """As attention_mla, with library GEMMs (fp64), for the listed
    (batch, head) pairs: returns (o [nb, T, nh, dv], s_bh [nb, nh])."""
    Q, KC, KR, V = _to_f64(q), _to_f64(k_c), _to_f64(k_r), _to_f64(v)
    B, T, _ = Q.shape
    batches = list(range(B)) if batches is None else list(batches)
    heads = list(range(H)) if heads is None else list(heads)
    dq = nope + rope
    o = np.empty((len(batches), T, len(heads), dv))
    s_bh = np.empty((len(batches), len(heads)))
    mask = np.tril(np.ones((T, T), dtype=bool)) if causal else np.ones((T, T), dtype=bool)
    for ib, b in enumerate(batches):
        for ih, h in enumerate(heads):
            qh = Q[b][:, h * dq:(h + 1) * dq]
            s = (qh[:, :nope] @ KC[b][:, h * nope:(h + 1) * nope].T + qh[:, nope:] @ KR[b].T) / np.sqrt(dq)
            s = np.where(mask, s, -np.inf)
            s_bh[ib, ih] = s.max()
            p = np.exp(s - s.max(axis=1, keepdims=True))
            o[ib, :, ih] = (p @ V[b][:, h * dv:(h + 1) * dv]) / p.sum(axis=1, keepdims=True)
    return o, s_bh


def newton_schulz_np(g, steps: int = 5, coeffs=NS_COEFFS, eps: float = 1e-7) -> np.ndarray:
    """As newton_schulz, with library GEMMs (fp64)."""
    G = _to_f64(g)
    tr = G.shape[0] > G.shape[1]
    X = G.T.copy() if tr else G.copy()
    X /= np.sqrt(np.sum(X * X)) + eps
    a, b, c = coeffs
    for _ in range(steps):
        A = X @ X.T
        Bm = b * A + c * (A @ A)
        X = a * X + Bm @ X
    return X.T.copy() if tr else X


def muon_step_np(w, g, m, lr: float, mu: float = 0.95, wd: float = 0.1, rms: float = 0.2,
                 steps: int = 5, coeffs=NS_COEFFS, eps: float = 1e-7, nesterov: bool = False):
    """As muon_step, with library GEMMs (fp64).  Returns (w_new, m_new, o)."""
    W, G, M = _to_f64(w), _to_f64(g), _to_f64(m)
    M = mu * M + G
    U = G + mu * M if nesterov else M
    O = newton_schulz_np(U, steps, coeffs, eps)
    W = W - lr * (rms * np.sqrt(max(W.shape)) * O + wd * W)
    return W, M, O
