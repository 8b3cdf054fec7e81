"""The tcgen05 GEMM building block (foak_gemm_bf16) against a float64 product.

Covers every operand layout the chunked linear+CE uses (K-major and MN-major A
and B), the three output modes, several tiles per CTA, and ragged M, N and K
(TMA zero-fill and epilogue masking).  Reference: numpy float64 matmul of the
same bf16 values; fp32 accumulation over K terms bounds the error by about
K * 2^-24 * sum|a*b|, far inside the tolerances below.
"""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


def _bf16(rows, cols, seed, sigma=1.0):
    bits = wl.normal_matrix(rows, cols, seed=seed, sigma=sigma, dtype=wl.BF16)
    return bits, wl.bf16_bits_to_f64(bits)


def _dev(bits):
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def _pad8(n):
    return (n + 7) // 8 * 8


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (384, 512, 320), (200, 300, 136), (1000, 776, 1032)])
def test_gemm_layouts_and_shapes(cuda_lib, a_mn, b_mn, M, N, K):
    ce = cuda_lib
    # stored shapes: K-major A [M][K], MN-major A [K][M]; same for B with N
    a_bits, a64 = _bf16(K if a_mn else M, _pad8(M if a_mn else K), seed=M + K + 1)
    b_bits, b64 = _bf16(K if b_mn else N, _pad8(N if b_mn else K), seed=N + K + 2)
    A = a64[:, :M].T if a_mn else a64[:, :K]  # logical [M][K]
    B = b64[:, :N].T if b_mn else b64[:, :K]  # logical [N][K]
    ref = A @ B.T
    ad, bd = _dev(a_bits), _dev(b_bits)
    ldo = _pad8(N)
    out = torch.full((M, ldo), 7.0, dtype=torch.float32, device="cuda")
    ce.foak_gemm_bf16(ad, bd, out, a_mn_major=bool(a_mn), b_mn_major=bool(b_mn), mode=ce.FOAK_GEMM_F32, M=M, N=N,
                      K=K)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    scale = np.abs(A) @ np.abs(B).T
    np.testing.assert_allclose(got[:, :N], ref, rtol=0, atol=1e-5 * scale.max() + 1e-6)
    assert np.all(got[:, N:] == 7.0), "columns past N must be untouched"


def test_gemm_bf16_out_and_accumulate(cuda_lib):
    ce = cuda_lib
    M, N, K = 256, 512, 192
    a_bits, A = _bf16(M, K, seed=5)
    b_bits, B = _bf16(N, K, seed=6)
    ref = A @ B.T
    ad, bd = _dev(a_bits), _dev(b_bits)
    o16 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ce.foak_gemm_bf16(ad, bd, o16, mode=ce.FOAK_GEMM_BF16)
    acc = torch.ones(M, N, dtype=torch.float32, device="cuda")
    ce.foak_gemm_bf16(ad, bd, acc, mode=ce.FOAK_GEMM_F32_ACC)
    ce.foak_gemm_bf16(ad, bd, acc, mode=ce.FOAK_GEMM_F32_ACC)
    torch.cuda.synchronize()
    g16 = o16.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(g16 - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-3)
    np.testing.assert_allclose(acc.cpu().numpy(), 1.0 + 2.0 * ref, rtol=1e-5, atol=1e-3)


def test_gemm_rejects_misaligned(cuda_lib):
    ce = cuda_lib
    a = torch.zeros(64, 72, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(64, 68, dtype=torch.bfloat16, device="cuda")  # row stride 136 B: not 16-byte aligned
    with pytest.raises(ce.FoakError):
        ce.foak_gemm_bf16(a, a, out, mode=ce.FOAK_GEMM_BF16)
