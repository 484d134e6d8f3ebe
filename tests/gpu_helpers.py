"""Shared helpers of the GPU parity tests (imported by tests only)."""
import numpy as np
import torch

_built = False


def lib():
    """Build (once) and load the CUDA library; fail loudly if it is absent."""
    global _built
    from muonclip_mc_max_gb300 import api, build
    if not _built:
        build.build()
        _built = True
    return api.load_library()


def dev():
    return torch.device("cuda:0")


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy()


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def rel_err(got, ref) -> np.ndarray:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.abs(got - ref) / np.maximum(np.abs(ref), 1e-30)


# S_max and scaled weights: relative error <= 1e-3 from bf16 inputs with
# fp32 accumulation; Newton-Schulz: relative Frobenius error <= 2e-2 against
# the fp64 oracle with the same coefficients.
SMAX_RTOL = 1e-3
NS_RTOL = 2e-2
