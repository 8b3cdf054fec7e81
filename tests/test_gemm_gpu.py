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


def _operand(rows, K, mn, seed, sigma=1.0):
    """bf16 operand of logical shape [rows][K]: stored [rows][K] (K-major) or [K][rows] (MN-major)."""
    bits, v = _bf16(K if mn else rows, _pad8(rows if mn else K), seed=seed, sigma=sigma)
    return _dev(bits), (v[:, :rows].T if mn else v[:, :K])


def _group_case():
    """Three products of different shapes, layouts and output modes, all on CTA pairs
    (M > 128): ragged M, N and K; one with a long K (many k-blocks per unit, as dH of
    the chunked call) next to short ones, so the balanced list mixes unit sizes."""
    specs = [  # (M, N, K, a_mn, b_mn, mode)
        (384, 520, 1000, 0, 0, "bf16"),
        (512, 256, 4096, 0, 1, "f32"),
        (300, 700, 192, 1, 0, "acc"),
    ]
    probs, refs = [], []
    for i, (M, N, K, amn, bmn, mode) in enumerate(specs):
        ad, A = _operand(M, K, amn, seed=100 + i)
        bd, B = _operand(N, K, bmn, seed=200 + i)
        ldo = _pad8(N)
        if mode == "bf16":
            out = torch.full((M, ldo), 3.0, dtype=torch.bfloat16, device="cuda")
        else:
            out = torch.full((M, ldo), 0.5 if mode == "acc" else 7.0, dtype=torch.float32, device="cuda")
        probs.append(dict(a=ad, b=bd, out=out, a_mn_major=bool(amn), b_mn_major=bool(bmn), M=M, N=N, K=K))
        refs.append((mode, A, B))
    return probs, refs


def test_gemm_group_matches_float64(cuda_lib):
    ce = cuda_lib
    probs, refs = _group_case()
    modes = {"bf16": ce.FOAK_GEMM_BF16, "f32": ce.FOAK_GEMM_F32, "acc": ce.FOAK_GEMM_F32_ACC}
    for q, (mode, _, _) in zip(probs, refs):
        q["mode"] = modes[mode]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ce.foak_gemm_bf16_group(probs, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    for q, (mode, A, B) in zip(probs, refs):
        N = q["N"]
        ref = A @ B.T
        got = q["out"].float().cpu().numpy().astype(np.float64)
        if mode == "bf16":
            assert np.all(np.abs(got[:, :N] - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-3)
            assert np.all(got[:, N:] == 3.0), "columns past N must be untouched"
        else:
            base = 0.5 if mode == "acc" else 0.0
            scale = np.abs(A) @ np.abs(B).T
            np.testing.assert_allclose(got[:, :N], base + ref, rtol=0, atol=1e-5 * scale.max() + 1e-6)
            assert np.all(got[:, N:] == (0.5 if mode == "acc" else 7.0))


def test_gemm_group_bit_identical_to_separate_launches(cuda_lib):
    """Each output unit is computed the same way whichever launch and SM pair takes it."""
    ce = cuda_lib
    probs, refs = _group_case()
    modes = {"bf16": ce.FOAK_GEMM_BF16, "f32": ce.FOAK_GEMM_F32, "acc": ce.FOAK_GEMM_F32_ACC}
    sep = []
    for q, (mode, _, _) in zip(probs, refs):
        q["mode"] = modes[mode]
        s = dict(q, out=q["out"].clone())
        ce.foak_gemm_bf16(s["a"], s["b"], s["out"], a_mn_major=s["a_mn_major"], b_mn_major=s["b_mn_major"],
                          mode=s["mode"], M=s["M"], N=s["N"], K=s["K"])
        sep.append(s["out"])
    ce.foak_gemm_bf16_group(probs)
    torch.cuda.synchronize()
    for q, s in zip(probs, sep):
        assert torch.equal(q["out"], s)


def test_gemm_group_with_single_cta_product_runs_in_order(cuda_lib):
    """A product with M <= 128 sends the group down the one-after-another path; the
    results are the same products."""
    ce = cuda_lib
    ad0, A0 = _operand(96, 256, 0, seed=301)
    bd0, B0 = _operand(264, 256, 0, seed=302)
    ad1, A1 = _operand(256, 128, 0, seed=303)
    bd1, B1 = _operand(512, 128, 1, seed=304)
    o0 = torch.zeros(96, 264, dtype=torch.float32, device="cuda")
    o1 = torch.zeros(256, 512, dtype=torch.float32, device="cuda")
    ce.foak_gemm_bf16_group([dict(a=ad0, b=bd0, out=o0, mode=ce.FOAK_GEMM_F32),
                             dict(a=ad1, b=bd1, out=o1, b_mn_major=True, mode=ce.FOAK_GEMM_F32)])
    torch.cuda.synchronize()
    for o, A, B in ((o0, A0, B0), (o1, A1, B1)):
        scale = np.abs(A) @ np.abs(B).T
        np.testing.assert_allclose(o.cpu().numpy().astype(np.float64), A @ B.T, rtol=0,
                                   atol=1e-5 * scale.max() + 1e-6)
