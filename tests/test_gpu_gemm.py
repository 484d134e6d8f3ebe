"""The tcgen05 contraction core on its own: mc_gemm_bf16 against an fp64
CPU product of the same bf16 inputs, for K-major and MN-major B operands,
batched, with tiles that are full and ragged in M, N and K."""
import pytest
import torch

from gpu_helpers import dev, lib

pytestmark = pytest.mark.gpu


def _case(M, N, K, Z, kmajor, out_dtype, seed):
    lib()
    from muonclip_mc_max_gb300 import api
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(Z, M, K, generator=g).to(torch.bfloat16)
    b = (torch.randn(Z, N, K, generator=g) if kmajor else torch.randn(Z, K, N, generator=g)).to(torch.bfloat16)
    out = api.mc_gemm_bf16(a.to(dev()), b.to(dev()), b_kmajor=kmajor, out_dtype=out_dtype)
    torch.cuda.synchronize()
    A, Bm = a.double(), b.double()
    ref = A @ (Bm.transpose(1, 2) if kmajor else Bm)
    mag = A.abs() @ (Bm.abs().transpose(1, 2) if kmajor else Bm.abs())
    got = out.double().cpu()
    # fp32 accumulation over K terms; bf16 output adds one rounding
    tol = K * 2.0 ** -23 * mag + 1e-30
    if out_dtype == torch.bfloat16:
        tol = tol + 2.0 ** -8 * ref.abs()
    bad = (got - ref).abs() > tol
    assert not bool(bad.any()), f"{int(bad.sum())} elements off; max err {(got - ref).abs().max()}"


@pytest.mark.parametrize("kmajor", [True, False])
def test_single_tile(kmajor):
    _case(128, 256, 64, 1, kmajor, torch.float32, 1)


@pytest.mark.parametrize("kmajor", [True, False])
def test_multi_tile_k_loop(kmajor):
    _case(256, 512, 512, 1, kmajor, torch.float32, 2)


@pytest.mark.parametrize("kmajor", [True, False])
def test_ragged_batched(kmajor):
    _case(300, 520, 200, 3, kmajor, torch.float32, 3)


@pytest.mark.parametrize("kmajor", [True, False])
def test_bf16_output(kmajor):
    _case(384, 768, 1024, 1, kmajor, torch.bfloat16, 4)


def test_many_tiles_persistent():
    # more tiles than SMs: every CTA walks several tiles and both TMEM buffers
    _case(2048, 2048, 256, 2, True, torch.float32, 5)


def test_tiny():
    _case(8, 8, 16, 1, False, torch.float32, 6)
