"""Tensor-core building blocks on the GPU: a 128 x N x K bf16 product through
the descriptor forms (K-major / MN-major operands, swizzled panels, TMA)
the fused backward uses, against torch's fp32 product of the same bf16
values."""
import ctypes

import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K,a_mn,b_mn,tma", [
    (128, 128, 0, 0, 0), (128, 64, 0, 0, 0), (64, 128, 0, 0, 0),
    (64, 128, 1, 1, 0), (128, 64, 0, 1, 0), (128, 128, 1, 1, 0), (64, 128, 1, 0, 0),
    (128, 128, 0, 0, 1), (64, 128, 1, 1, 1), (128, 64, 0, 1, 1),
])
def test_umma_product(N, K, a_mn, b_mn, tma):
    L = ssd.lib()
    f = L.mamba2_ssd_selftest_umma
    g = torch.Generator().manual_seed(N * 1000 + K * 10 + a_mn * 2 + b_mn)
    A = torch.randn(128, K, generator=g).bfloat16()
    B = torch.randn(N, K, generator=g).bfloat16()
    want = A.float() @ B.float().T
    a_store = (A.T if a_mn else A).contiguous().cuda()
    b_store = (B.T if b_mn else B).contiguous().cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    rc = f(a_store.data_ptr(), b_store.data_ptr(), D.data_ptr(), 128, N, K, a_mn, b_mn, tma,
           torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    err = (D.cpu() - want).abs().max().item()
    assert err < 1e-3 * want.abs().max().item(), err
