"""Thin ctypes binding of ``include/mc_max.h``.

Every function carries the C entry point's name and only marshals
arguments: torch tensors supply device pointers, the caller's current CUDA
stream is passed through, and workspaces are torch-allocated byte buffers.
All arithmetic runs in the CUDA library; if ``libmc_max.so`` is missing this
module raises instead of computing anything elsewhere.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from .build import library_path

__all__ = [
    "MCError", "load_library", "header_symbols", "Workspace",
    "mc_status_string", "mc_read_device_status",
    "mc_max_logits_mha", "mc_max_logits_mha_workspace_size", "mc_max_logits_mha_noalloc",
    "mc_attention_mha", "mc_attention_mha_workspace_size", "mc_attention_mla",
    "MC_NOALLOC_SCRATCH_BYTES",
    "mc_max_logits_mla", "mc_max_logits_mla_workspace_size",
    "mc_qk_clip_mha", "mc_qk_clip_mla", "mc_qk_clip_global",
    "mc_newton_schulz", "mc_newton_schulz_workspace_size",
    "mc_muon_step", "mc_muon_workspace_size", "mc_gemm_bf16",
    "mc_smax_to_keys", "mc_smax_from_keys", "mc_muon_momentum", "mc_muon_apply",
    "mc_launch_count", "mc_trace_enable", "mc_trace_collect", "mc_selftest_wait_timeout",
    "MC_F32", "MC_BF16", "MC_DEV_NONFINITE", "MC_DEV_TIMEOUT", "MC_DEV_RANGE", "NS_COEFFS",
]

MC_F32, MC_BF16 = 0, 1
MC_DEV_NONFINITE, MC_DEV_TIMEOUT, MC_DEV_RANGE = 0x1, 0x2, 0x4
MC_NOALLOC_SCRATCH_BYTES = 64 << 20  # static scratch of mc_max_logits_mha_noalloc
# quintic Newton-Schulz coefficients ("Notes on Muon blog", "Algorithm")
NS_COEFFS = (3.4445, -4.7750, 2.0315)

_HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                       "include", "mc_max.h")


class MCError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


class TraceEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_longlong),
                ("total_ms", ctypes.c_double)]


class MlaLayer(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int), ("q_lora", ctypes.c_int), ("kv_lora", ctypes.c_int),
                ("H", ctypes.c_int), ("nope", ctypes.c_int), ("rope", ctypes.c_int),
                ("rope_base", ctypes.c_float), ("wtype", ctypes.c_int),
                ("w_qa", ctypes.c_void_p), ("w_qb", ctypes.c_void_p),
                ("w_kva", ctypes.c_void_p), ("w_kb", ctypes.c_void_p)]


_lib = None


def header_symbols() -> list[str]:
    """Names of every function declared in include/mc_max.h."""
    with open(_HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(mc_\w+)\s*\(", text, re.M)))


def load_library():
    """Load libmc_max.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with muonclip_mc_max_gb300.build.build()")
    lib = ctypes.CDLL(path)
    V, I, F, S, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint
    IP = ctypes.POINTER(ctypes.c_int)
    VP = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "mc_status_string": ([I], ctypes.c_char_p),
        "mc_read_device_status": ([V, ctypes.POINTER(U), I], I),
        "mc_max_logits_mha_workspace_size": ([I, I, I, I, I, I], S),
        "mc_max_logits_mha": ([V, V, V, I, I, I, I, I, I, I, I, V, V, V, S, V], I),
        "mc_max_logits_mha_noalloc": ([V, V, V, I, I, I, I, I, I, I, I, V, V, V], I),
        "mc_max_logits_mla_workspace_size": ([ctypes.POINTER(MlaLayer), I, I], S),
        "mc_max_logits_mla": ([ctypes.POINTER(MlaLayer), V, I, I, I, I, V, V, V, S, V], I),
        "mc_attention_mha_workspace_size": ([I, I], S),
        "mc_attention_mha": ([V, V, V, I, I, I, I, I, I, V, V, V, V, S, V], I),
        "mc_attention_mla": ([V, V, V, I, I, V, I, I, I, I, I, I, I, I, V, V, V, V, S, V], I),
        "mc_qk_clip_mha": ([V, V, I, I, I, I, V, F, V, V], I),
        "mc_qk_clip_mla": ([ctypes.POINTER(MlaLayer), V, F, V, V], I),
        "mc_qk_clip_global": ([V, V, I, I, I, V, I, F, F, V, V], I),
        "mc_newton_schulz_workspace_size": ([IP, IP, I], S),
        "mc_muon_workspace_size": ([IP, IP, I], S),
        "mc_newton_schulz": ([VP, VP, IP, IP, I, I, F, F, F, F, V, S, V], I),
        "mc_muon_step": ([VP, VP, VP, IP, IP, I, F, F, F, F, I, F, F, F, F, I, V, S, V], I),
        "mc_gemm_bf16": ([V, V, V, I, I, I, I, I, I, V], I),
        "mc_smax_to_keys": ([V, V, I, V], I),
        "mc_smax_from_keys": ([V, V, I, V], I),
        "mc_muon_momentum": ([V, V, V, S, F, F, I, V], I),
        "mc_muon_apply": ([V, V, S, I, I, F, F, F, V], I),
        "mc_selftest_wait_timeout": ([U, V, V], I),
        "mc_launch_count": ([], ctypes.c_ulonglong),
        "mc_trace_enable": ([I], I),
        "mc_trace_collect": ([ctypes.POINTER(TraceEntry), I, I], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def mc_status_string(status: int) -> str:
    return load_library().mc_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != 0:
        raise MCError(fn, status, mc_status_string(status))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MC_BF16
    if t.dtype == torch.float32:
        return MC_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensor must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")


class Workspace:
    """A growable device byte buffer handed to the library as scratch."""

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, nbytes: int, device) -> torch.Tensor:
        nbytes = max(int(nbytes), 256)
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != device:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        return self.buf


# One default scratch buffer per device, used by every call that passes no
# workspace.  Calls are stream-ordered on it, so calls issued concurrently on
# different streams must each pass their own Workspace; a buffer grows (and
# its old storage returns to torch's allocator) only between calls, never
# while a CUDA graph is being captured once the graph's calls have run once.
_default_ws: dict = {}


def _ws(workspace, nbytes, device):
    if nbytes == 0:
        return ctypes.c_void_p(None), 0
    if workspace is None:
        workspace = _default_ws.setdefault(str(device), Workspace())
    buf = workspace.get(nbytes, device)
    return ctypes.c_void_p(buf.data_ptr()), buf.numel()


def mc_read_device_status(clear: bool = True, stream=None) -> int:
    bits = ctypes.c_uint(0)
    _check("mc_read_device_status",
           load_library().mc_read_device_status(_stream(stream), ctypes.byref(bits), int(clear)))
    return bits.value


# ---------------------------------------------------------------------------
# (1) max logits
# ---------------------------------------------------------------------------

def mc_max_logits_mha_workspace_size(B, T, D, H, dh, dtype=MC_BF16) -> int:
    return load_library().mc_max_logits_mha_workspace_size(B, T, D, H, dh, dtype)


def mc_max_logits_mha(x, wq, wk, H: int, dh: int, causal: bool = False, accumulate: bool = False,
                      s_max=None, s_max_bh=None, workspace=None, stream=None):
    """x [B,T,D], wq/wk [D,H*dh] (bf16 or f32).  Returns s_max [H] f32."""
    lib = load_library()
    _need_cuda(x, wq, wk, s_max, s_max_bh)
    B, T, D = x.shape
    if wq.shape != (D, H * dh) or wk.shape != (D, H * dh):
        raise ValueError("wq, wk must be [D, H*dh]")
    dt = _dtype(x)
    if s_max is None:
        s_max = torch.empty(H, dtype=torch.float32, device=x.device)
    ws, nb = _ws(workspace, lib.mc_max_logits_mha_workspace_size(B, T, D, H, dh, dt), x.device)
    _check("mc_max_logits_mha", lib.mc_max_logits_mha(
        _ptr(x), _ptr(wq), _ptr(wk), dt, B, T, D, H, dh, int(causal), int(accumulate),
        _ptr(s_max), _ptr(s_max_bh), ws, nb, _stream(stream)))
    return s_max


def mc_attention_mha_workspace_size(B: int, H: int) -> int:
    return load_library().mc_attention_mha_workspace_size(B, H)


def mc_attention_mha(q, k, v, H: int, dh: int, causal: bool = False, accumulate: bool = False,
                     out=None, s_max=None, s_max_bh=None, workspace=None, stream=None):
    """q, k, v [B,T,H*dh] bf16.  Returns (o [B,T,H*dh] bf16, s_max [H] f32):
    softmax attention with the per-head max logit taken along.  The forward
    needs no workspace (``workspace`` is accepted and not used)."""
    lib = load_library()
    _need_cuda(q, k, v, out, s_max, s_max_bh)
    B, T, W = q.shape
    if W != H * dh or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all be [B, T, H*dh]")
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise ValueError("q, k, v must be bf16")
    if out is None:
        out = torch.empty_like(q)
    if s_max is None:
        s_max = torch.empty(H, dtype=torch.float32, device=q.device)
    ws, nb = _ws(workspace, lib.mc_attention_mha_workspace_size(B, H), q.device)
    _check("mc_attention_mha", lib.mc_attention_mha(
        _ptr(q), _ptr(k), _ptr(v), B, T, H, dh, int(causal), int(accumulate), _ptr(out), _ptr(s_max),
        _ptr(s_max_bh), ws, nb, _stream(stream)))
    return out, s_max


def mc_attention_mla(q, k_c, k_r, v, H: int, nope: int = 128, rope: int = 64, dv: int = 128,
                     causal: bool = True, accumulate: bool = False, kr_col: int = 0, out=None,
                     s_max=None, s_max_bh=None, workspace=None, stream=None):
    """q [B,T,H*(nope+rope)], k_c [B,T,H*nope], k_r [B,T,>= kr_col+rope]
    (the shared k^R at columns kr_col..), v [B,T,H*dv], all bf16.  Returns
    (o [B,T,H*dv] bf16, s_max [H] f32): MLA attention with the per-head max
    logit taken along."""
    lib = load_library()
    _need_cuda(q, k_c, k_r, v, out, s_max, s_max_bh)
    B, T, W = q.shape
    if W != H * (nope + rope) or k_c.shape != (B, T, H * nope) or v.shape != (B, T, H * dv):
        raise ValueError("q, k_c, v must be [B, T, H*(nope+rope)], [B, T, H*nope], [B, T, H*dv]")
    if k_r.dim() != 3 or k_r.shape[:2] != (B, T):
        raise ValueError("k_r must be [B, T, kr_ld]")
    for t in (q, k_c, k_r, v):
        if t.dtype != torch.bfloat16:
            raise ValueError("q, k_c, k_r, v must be bf16")
    if out is None:
        out = torch.empty((B, T, H * dv), dtype=torch.bfloat16, device=q.device)
    if s_max is None:
        s_max = torch.empty(H, dtype=torch.float32, device=q.device)
    ws, nb = _ws(workspace, lib.mc_attention_mha_workspace_size(B, H), q.device)
    _check("mc_attention_mla", lib.mc_attention_mla(
        _ptr(q), _ptr(k_c), _ptr(k_r), k_r.shape[2], kr_col, _ptr(v), B, T, H, nope, rope, dv,
        int(causal), int(accumulate), _ptr(out), _ptr(s_max), _ptr(s_max_bh), ws, nb,
        _stream(stream)))
    return out, s_max


def mc_max_logits_mha_noalloc(x, wq, wk, H: int, dh: int, causal: bool = False,
                              accumulate: bool = False, s_max=None, s_max_bh=None, stream=None):
    """mc_max_logits_mha without a workspace: the library's static scratch
    (MC_NOALLOC_SCRATCH_BYTES, shared by every call) is used instead, for
    callers that may not allocate.  Pass s_max (and s_max_bh) preallocated
    to allocate nothing here either."""
    lib = load_library()
    _need_cuda(x, wq, wk, s_max, s_max_bh)
    B, T, D = x.shape
    if wq.shape != (D, H * dh) or wk.shape != (D, H * dh):
        raise ValueError("wq, wk must be [D, H*dh]")
    if s_max is None:
        s_max = torch.empty(H, dtype=torch.float32, device=x.device)
    _check("mc_max_logits_mha_noalloc", lib.mc_max_logits_mha_noalloc(
        _ptr(x), _ptr(wq), _ptr(wk), _dtype(x), B, T, D, H, dh, int(causal), int(accumulate),
        _ptr(s_max), _ptr(s_max_bh), _stream(stream)))
    return s_max


def _mla_layer(w_qa, w_qb, w_kva, w_kb, H, nope, rope, rope_base, D=None, q_lora=None,
               kv_lora=None, wtype=None):
    L = MlaLayer()
    L.D = D if D is not None else (w_qa.shape[0] if w_qa is not None else 0)
    L.q_lora = q_lora if q_lora is not None else w_qb.shape[0]
    L.kv_lora = kv_lora if kv_lora is not None else w_kb.shape[0]
    L.H, L.nope, L.rope = H, nope, rope
    L.rope_base = rope_base
    L.wtype = wtype if wtype is not None else _dtype(w_qb)
    L.w_qa = None if w_qa is None else w_qa.data_ptr()
    L.w_qb = w_qb.data_ptr()
    L.w_kva = None if w_kva is None else w_kva.data_ptr()
    L.w_kb = w_kb.data_ptr()
    return L


def mc_max_logits_mla_workspace_size(layer: MlaLayer, B: int, T: int) -> int:
    return load_library().mc_max_logits_mla_workspace_size(ctypes.byref(layer), B, T)


def mc_max_logits_mla(x, w_qa, w_qb, w_kva, w_kb, H: int, nope: int, rope: int,
                      rope_base: float = 50000.0, causal: bool = True, accumulate: bool = False,
                      s_max=None, s_max_bh=None, workspace=None, stream=None):
    """MLA per-head max logit; shapes as in mc_mla_layer.  Returns s_max [H]."""
    lib = load_library()
    _need_cuda(x, w_qa, w_qb, w_kva, w_kb, s_max, s_max_bh)
    B, T, D = x.shape
    L = _mla_layer(w_qa, w_qb, w_kva, w_kb, H, nope, rope, rope_base)
    if s_max is None:
        s_max = torch.empty(H, dtype=torch.float32, device=x.device)
    ws, nb = _ws(workspace, lib.mc_max_logits_mla_workspace_size(ctypes.byref(L), B, T), x.device)
    _check("mc_max_logits_mla", lib.mc_max_logits_mla(
        ctypes.byref(L), _ptr(x), B, T, int(causal), int(accumulate), _ptr(s_max),
        _ptr(s_max_bh), ws, nb, _stream(stream)))
    return s_max


# ---------------------------------------------------------------------------
# (2) QK-Clip
# ---------------------------------------------------------------------------

def mc_qk_clip_mha(wq, wk, H: int, dh: int, s_max, tau: float, gamma=None, stream=None):
    """In-place MHA clip; returns gamma [H]."""
    lib = load_library()
    _need_cuda(wq, wk, s_max, gamma)
    if gamma is None:
        gamma = torch.empty(H, dtype=torch.float32, device=wq.device)
    D = wq.shape[0]
    _check("mc_qk_clip_mha", lib.mc_qk_clip_mha(_ptr(wq), _ptr(wk), _dtype(wq), D, H, dh,
                                                _ptr(s_max), float(tau), _ptr(gamma),
                                                _stream(stream)))
    return gamma


def mc_qk_clip_mla(w_qb, w_kb, H: int, nope: int, rope: int, s_max, tau: float, gamma=None,
                   stream=None):
    """In-place MLA clip of W_qb (q^C, q^R) and W_kb (k^C); returns gamma."""
    lib = load_library()
    _need_cuda(w_qb, w_kb, s_max, gamma)
    if gamma is None:
        gamma = torch.empty(H, dtype=torch.float32, device=w_qb.device)
    L = _mla_layer(None, w_qb, None, w_kb, H, nope, rope, 0.0, D=1)
    _check("mc_qk_clip_mla", lib.mc_qk_clip_mla(ctypes.byref(L), _ptr(s_max), float(tau),
                                                _ptr(gamma), _stream(stream)))
    return gamma


def mc_qk_clip_global(wq, wk, s_max, tau: float, alpha: float = 0.5, gamma=None, stream=None):
    lib = load_library()
    _need_cuda(wq, wk, s_max, gamma)
    if gamma is None:
        gamma = torch.empty(1, dtype=torch.float32, device=wq.device)
    rows, cols = wq.shape
    _check("mc_qk_clip_global", lib.mc_qk_clip_global(
        _ptr(wq), _ptr(wk), _dtype(wq), rows, cols, _ptr(s_max), s_max.numel(), float(tau),
        float(alpha), _ptr(gamma), _stream(stream)))
    return gamma


# ---------------------------------------------------------------------------
# (3) Muon
# ---------------------------------------------------------------------------

def _shapes(mats):
    n = len(mats)
    rows = (ctypes.c_int * n)(*[m.shape[0] for m in mats])
    cols = (ctypes.c_int * n)(*[m.shape[1] for m in mats])
    return rows, cols


def _ptrs(mats):
    return (ctypes.c_void_p * len(mats))(*[m.data_ptr() for m in mats])


def mc_newton_schulz_workspace_size(shapes) -> int:
    n = len(shapes)
    rows = (ctypes.c_int * n)(*[s[0] for s in shapes])
    cols = (ctypes.c_int * n)(*[s[1] for s in shapes])
    return load_library().mc_newton_schulz_workspace_size(rows, cols, n)


def mc_muon_workspace_size(shapes) -> int:
    n = len(shapes)
    rows = (ctypes.c_int * n)(*[s[0] for s in shapes])
    cols = (ctypes.c_int * n)(*[s[1] for s in shapes])
    return load_library().mc_muon_workspace_size(rows, cols, n)


def mc_newton_schulz(mats, steps: int = 5, coeffs=NS_COEFFS, eps: float = 1e-7, out=None,
                     workspace=None, stream=None):
    """Newton-Schulz of each f32 matrix; returns a list of f32 outputs."""
    lib = load_library()
    _need_cuda(*mats)
    if out is None:
        out = [torch.empty_like(m) for m in mats]
    _need_cuda(*out)
    rows, cols = _shapes(mats)
    n = len(mats)
    ws, nb = _ws(workspace, lib.mc_newton_schulz_workspace_size(rows, cols, n), mats[0].device)
    a, b, c = coeffs
    _check("mc_newton_schulz", lib.mc_newton_schulz(
        _ptrs(mats), _ptrs(out), rows, cols, n, steps, a, b, c, eps, ws, nb, _stream(stream)))
    return out


def mc_muon_step(w, g, m, lr: float, mu: float = 0.95, wd: float = 0.1, rms: float = 0.2,
                 steps: int = 5, coeffs=NS_COEFFS, eps: float = 1e-7, nesterov: bool = False,
                 workspace=None, stream=None):
    """One in-place Muon step over lists of f32 weights, grads, momenta."""
    lib = load_library()
    _need_cuda(*w, *g, *m)
    rows, cols = _shapes(w)
    n = len(w)
    ws, nb = _ws(workspace, lib.mc_muon_workspace_size(rows, cols, n), w[0].device)
    a, b, c = coeffs
    _check("mc_muon_step", lib.mc_muon_step(
        _ptrs(w), _ptrs(g), _ptrs(m), rows, cols, n, lr, mu, wd, rms, steps, a, b, c, eps,
        int(nesterov), ws, nb, _stream(stream)))


# ---------------------------------------------------------------------------
# (4) data-parallel exchange helpers
# ---------------------------------------------------------------------------

def mc_smax_to_keys(s_max, keys=None, stream=None):
    """f32 S_max [n] -> order-preserving int32 keys [n] (NaN largest)."""
    lib = load_library()
    _need_cuda(s_max, keys)
    if s_max.dtype != torch.float32:
        raise ValueError("s_max must be float32")
    if keys is None:
        keys = torch.empty(s_max.shape, dtype=torch.int32, device=s_max.device)
    elif keys.dtype != torch.int32 or keys.numel() != s_max.numel():
        raise ValueError("keys must be int32 with one entry per head")
    _check("mc_smax_to_keys", lib.mc_smax_to_keys(_ptr(s_max), _ptr(keys), s_max.numel(),
                                                  _stream(stream)))
    return keys


def mc_smax_from_keys(keys, s_max=None, stream=None):
    """int32 keys [n] -> f32 S_max [n] (the inverse of mc_smax_to_keys)."""
    lib = load_library()
    _need_cuda(keys, s_max)
    if keys.dtype != torch.int32:
        raise ValueError("keys must be int32")
    if s_max is None:
        s_max = torch.empty(keys.shape, dtype=torch.float32, device=keys.device)
    elif s_max.dtype != torch.float32 or s_max.numel() != keys.numel():
        raise ValueError("s_max must be float32 with one entry per key")
    _check("mc_smax_from_keys", lib.mc_smax_from_keys(_ptr(keys), _ptr(s_max), keys.numel(),
                                                      _stream(stream)))
    return s_max


def mc_muon_momentum(m, g, u=None, mu: float = 0.95, grad_scale: float = 1.0,
                     nesterov: bool = False, stream=None):
    """In-place m <- mu m + grad_scale g on one f32 shard; u (optional, same
    size) receives the Newton-Schulz input (m, or the Nesterov input)."""
    lib = load_library()
    _need_cuda(m, g, u)
    for t in (m, g, u):
        if t is not None and (t.dtype != torch.float32 or t.numel() != m.numel()):
            raise ValueError("m, g, u must be float32 of equal size")
    _check("mc_muon_momentum", lib.mc_muon_momentum(_ptr(m), _ptr(g), _ptr(u), m.numel(), mu,
                                                    grad_scale, int(nesterov), _stream(stream)))
    return u if u is not None else m


def mc_muon_apply(w, o, rows: int, cols: int, lr: float, rms: float = 0.2, wd: float = 0.1,
                  stream=None):
    """In-place w <- w - lr (rms sqrt(max(rows, cols)) o + wd w) on one f32
    shard of a [rows, cols] matrix."""
    lib = load_library()
    _need_cuda(w, o)
    if w.dtype != torch.float32 or o.dtype != torch.float32 or o.numel() != w.numel():
        raise ValueError("w and o must be float32 of equal size")
    _check("mc_muon_apply", lib.mc_muon_apply(_ptr(w), _ptr(o), w.numel(), int(rows), int(cols),
                                              lr, rms, wd, _stream(stream)))


# ---------------------------------------------------------------------------
# tensor-core GEMM
# ---------------------------------------------------------------------------

def mc_gemm_bf16(a, b, b_kmajor: bool = True, out_dtype=torch.float32, out=None, stream=None):
    """a [(Z,)M,K] bf16; b [(Z,)N,K] (b_kmajor) or [(Z,)K,N]; returns [(Z,)M,N]."""
    lib = load_library()
    _need_cuda(a, b)
    batched = a.dim() == 3
    A = a if batched else a.unsqueeze(0)
    Bt = b if batched else b.unsqueeze(0)
    Z, M, K = A.shape
    N = Bt.shape[1] if b_kmajor else Bt.shape[2]
    if out is None:
        out = torch.empty((Z, M, N), dtype=out_dtype, device=a.device)
    _need_cuda(out)
    ct = MC_F32 if out.dtype == torch.float32 else MC_BF16
    _check("mc_gemm_bf16", lib.mc_gemm_bf16(_ptr(A), _ptr(Bt), _ptr(out), ct, M, N, K, Z,
                                            int(b_kmajor), _stream(stream)))
    return out if batched else out[0]


# ---------------------------------------------------------------------------
# tracing
# ---------------------------------------------------------------------------

def mc_selftest_wait_timeout(limit_us: int = 20000, out=None, stream=None):
    """Bounded-wait self-test: one CTA whose warps wait on barriers nothing
    completes; returns the device int64[4] result (the two warps' waits in
    ns, then two completion flags).  Read MC_DEV_TIMEOUT with
    mc_read_device_status afterwards."""
    lib = load_library()
    _need_cuda(out)
    if out is None:
        out = torch.zeros(4, dtype=torch.int64, device=torch.device("cuda", torch.cuda.current_device()))
    elif out.dtype != torch.int64 or out.numel() < 4:
        raise ValueError("out must hold 4 int64 values")
    _check("mc_selftest_wait_timeout", lib.mc_selftest_wait_timeout(int(limit_us), _ptr(out), _stream(stream)))
    return out


def mc_launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(load_library().mc_launch_count())


def mc_trace_enable(on: bool = True):
    _check("mc_trace_enable", load_library().mc_trace_enable(int(on)))


def mc_trace_collect(keep: bool = False) -> dict:
    """{kernel kind: (launches, total_ms)} of the launches traced since the
    last collect (event-timed on their launch streams).  keep=True leaves
    the records in place (for replays of a captured graph)."""
    lib = load_library()
    cap = 64
    buf = (TraceEntry * cap)()
    n = lib.mc_trace_collect(buf, cap, int(keep))
    if n < 0:
        raise MCError("mc_trace_collect", 3, "CUDA error while reading trace events")
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms))
            for i in range(min(n, cap))}
