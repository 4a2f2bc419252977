"""Tensor-core prefill: the tcgen05 GEMM against float64 numpy on the same 16-bit operands."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    assert torch.cuda.is_available(), "a CUDA GPU is required"
    from autoregressive_decode_persistent_gb300 import adp, build
    build.build()
    return adp


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 300, 100), (5, 17, 8), (384, 1024, 2560), (130, 512, 704)])
@pytest.mark.parametrize("bf16", [False, True])
def test_tc_gemm_matches_float64(lib, M, N, K, bf16):
    """fp32 accumulation of exact 16-bit products: every entry within 2^-20 of the row's sum of
    |a_k w_k| (fp32 rounding of K partial sums) of the float64 product."""
    import torch
    dt = torch.bfloat16 if bf16 else torch.float16
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K)
    a = torch.randn(M, K, generator=g).to(dt)
    w = torch.randn(N, K, generator=g).to(dt)
    ref = a.double() @ w.double().T
    bound = (a.double().abs() @ w.double().abs().T) * 2.0 ** -20 + 1e-30
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    lib.adp_debug_tc_gemm(bf16, a.cuda(), w.cuda(), c)
    err = (c.cpu().double() - ref).abs()
    assert torch.isfinite(c).all()
    assert (err <= bound).all(), float((err / bound).max())
