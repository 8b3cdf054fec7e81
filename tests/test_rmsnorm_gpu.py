"""GPU parity of the RMSNorm kernels and of the decoder tail (final RMSNorm ->
chunked LM head -> cross-entropy) against the float64 oracle.

Bars: Y within one bf16 ulp (fp32: 1e-5 relative) of the oracle, rstd 1e-5
relative; dX within 4e-3 relative Frobenius error for bf16 storage (1e-5 for
fp32), dgamma 1e-4 (fp32 sums); the decoder tail: loss 2e-3 relative, dX, dgamma
and dW 1e-2 relative Frobenius (the chunked linear + CE bars), n_valid and the
error word exact.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from ce_helpers import assert_grad_close, to_f64

pytestmark = pytest.mark.gpu


def _dev(a, dtype):
    if dtype == wl.BF16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _frob(got, ref):
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def _bf16_round(a):
    return wl.bf16_bits_to_f64(wl.f64_to_bf16_bits(a))


def _inputs(N, D, dtype, seed, ld=None):
    X = wl.normal_matrix(N, D, seed=seed, sigma=2.0, dtype=dtype, ld=ld, stream=wl.S_X)
    gz = wl.normal_matrix(1, D, seed=seed, sigma=0.1, dtype=wl.F32, stream=wl.S_GAMMA)[0].astype(np.float64) + 1.0
    gamma = wl.f64_to_bf16_bits(gz) if dtype == wl.BF16 else gz.astype(np.float32)
    return X, gamma


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
@pytest.mark.parametrize("N,D,ld", [(1, 8, None), (37, 4096, None), (513, 1000, None), (64, 8192, None),
                                    (100, 2048, 2056), (1500, 4096, None), (700, 3000, 3016)])
def test_rmsnorm_forward(cuda_lib, dtype, N, D, ld):
    X, gamma = _inputs(N, D, dtype, seed=N + D, ld=ld)
    ref_y, ref_r = oracle.rmsnorm(X[:, :D], gamma, 1e-5)
    x = _dev(X, dtype)[:, :D]
    y, rstd = cuda_lib.foak_rmsnorm_forward(x, _dev(gamma, dtype), eps=1e-5)
    torch.cuda.synchronize()
    np.testing.assert_allclose(to_f64(rstd), ref_r, rtol=1e-5)
    if dtype == wl.BF16:
        assert_grad_close(to_f64(y), ref_y, what="rmsnorm Y")
    else:
        np.testing.assert_allclose(to_f64(y), ref_y, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
@pytest.mark.parametrize("N,D", [(1, 8), (77, 4096), (1024, 1000), (300, 8192), (2000, 4096), (1500, 2304), (9, 64), (611, 2048)])
def test_rmsnorm_backward(cuda_lib, dtype, N, D):
    X, gamma = _inputs(N, D, dtype, seed=3 * N + D)
    dY = wl.normal_matrix(N, D, seed=N + 7, sigma=1.0, dtype=dtype, stream=wl.S_H)
    ref_dx, ref_dg = oracle.rmsnorm_backward(dY, X, gamma, 1e-5)
    x, g = _dev(X, dtype), _dev(gamma, dtype)
    _, rstd = cuda_lib.foak_rmsnorm_forward(x, g, eps=1e-5)
    dx, dg = cuda_lib.foak_rmsnorm_backward(_dev(dY, dtype), x, g, rstd)
    torch.cuda.synchronize()
    assert _frob(to_f64(dx), ref_dx) < (4e-3 if dtype == wl.BF16 else 1e-5)
    assert _frob(to_f64(dg), ref_dg) < (1e-4 if dtype == wl.BF16 else 1e-5)


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
def test_rmsnorm_backward_padded_rows(cuda_lib, dtype):
    """dY, X and dX as views of wider row-major buffers (three different row strides)."""
    N, D = 700, 1024
    X, gamma = _inputs(N, D, dtype, seed=41, ld=D + 24)
    dY = wl.normal_matrix(N, D, seed=43, sigma=1.0, dtype=dtype, ld=D + 8, stream=wl.S_H)
    ref_dx, ref_dg = oracle.rmsnorm_backward(dY[:, :D], X[:, :D], gamma, 1e-5)
    x, g = _dev(X, dtype)[:, :D], _dev(gamma, dtype)
    _, rstd = cuda_lib.foak_rmsnorm_forward(x, g, eps=1e-5)
    dx_buf = torch.full((N, D + 40), 7.0, device="cuda").to(x.dtype)
    dx, dg = cuda_lib.foak_rmsnorm_backward(_dev(dY, dtype)[:, :D], x, g, rstd, dX=dx_buf[:, :D])
    torch.cuda.synchronize()
    assert _frob(to_f64(dx), ref_dx) < (4e-3 if dtype == wl.BF16 else 1e-5)
    assert _frob(to_f64(dg), ref_dg) < (1e-4 if dtype == wl.BF16 else 1e-5)
    assert bool((dx_buf[:, D:] == 7.0).all()), "a write past the rows' D elements"


def test_rmsnorm_backward_empty_batch_zero_dgamma(cuda_lib):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    r = torch.empty(0, dtype=torch.float32, device="cuda")
    dx, dg = cuda_lib.foak_rmsnorm_backward(x, x, g, r)
    torch.cuda.synchronize()
    assert dx.numel() == 0 and int(dg.count_nonzero().item()) == 0


def _tail_case(N, V, D, seed, n_ignore):
    X, gamma = _inputs(N, D, wl.BF16, seed=seed)
    W = wl.normal_matrix(V, D, seed=seed, sigma=0.05, dtype=wl.BF16, stream=wl.S_W)
    y = wl.uniform_labels(N, V, seed=seed)
    y[wl.pick_rows(N, n_ignore, seed=seed)] = -100
    return X, gamma, W, y


def _run_tail(ce, X, gamma, W, y, chunk, eps=1e-5, g=1.0, denom=0.0):
    out = ce.foak_rmsnorm_linear_ce_chunked(_dev(X, wl.BF16), _dev(gamma, wl.BF16), _dev(W, wl.BF16),
                                            torch.from_numpy(y).cuda(), eps=eps, chunk=chunk, g=g, denom=denom)
    torch.cuda.synchronize()
    return out


def _check_tail(out, ref):
    assert abs(out["loss"].item() - ref["loss"]) <= 2e-3 * abs(ref["loss"])
    assert out["n_valid"].item() == ref["n_valid"]
    assert _frob(to_f64(out["dX"]), ref["dX"]) < 1e-2
    assert _frob(to_f64(out["dgamma"]), ref["dgamma"]) < 1e-2
    assert _frob(out["dW"].cpu().numpy().astype(np.float64), ref["dW"]) < 1e-2


@pytest.mark.parametrize("N,V,D,chunk", [(300, 1000, 256, 128), (129, 520, 64, 1024), (1024, 4096, 512, 256)])
def test_decoder_tail_small(cuda_lib, N, V, D, chunk):
    X, gamma, W, y = _tail_case(N, V, D, seed=N + V + D, n_ignore=N // 10)
    ref = oracle.rmsnorm_linear_ce(X, gamma, W, y, eps=1e-5, g=1.5, round_h=_bf16_round)
    out = _run_tail(cuda_lib, X, gamma, W, y, chunk, g=1.5)
    _check_tail(out, ref)
    assert out["err"].item() == 0


def test_decoder_tail_bad_label_and_denominator(cuda_lib):
    X, gamma, W, y = _tail_case(200, 300, 64, seed=9, n_ignore=20)
    y[5] = 300
    ref = oracle.rmsnorm_linear_ce(X, gamma, W, y, eps=1e-6, denom=1000.0, round_h=_bf16_round)
    out = _run_tail(cuda_lib, X, gamma, W, y, 64, eps=1e-6, denom=1000.0)
    _check_tail(out, ref)
    assert out["err"].item() == 1


def test_decoder_tail_full_size(cuda_lib):
    """The decoder tail at the chunked workload's sizes: X 8192x4096, W 32000x4096, chunks of 1024."""
    c = wl.norm_chunked()
    ref = oracle.rmsnorm_linear_ce(c["X"], c["gamma"], c["W"], c["labels"], eps=c["eps"], round_h=_bf16_round)
    out = _run_tail(cuda_lib, c["X"], c["gamma"], c["W"], c["labels"], c["chunk"], eps=c["eps"])
    _check_tail(out, ref)
    assert out["n_valid"].item() == 8192 - 819 and out["err"].item() == 0


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
@pytest.mark.parametrize("N,D", [(301, 4096), (50, 16384)])
def test_rmsnorm_backward_without_dgamma(cuda_lib, dtype, N, D):
    """dX alone (no dgamma wanted): the ring without its dgamma partials up to 1024
    vectors a row, the warp-per-row two-pass kernel beyond."""
    X, gamma = _inputs(N, D, dtype, seed=17)
    dY = wl.normal_matrix(N, D, seed=19, sigma=1.0, dtype=dtype, stream=wl.S_H)
    ref_dx, _ = oracle.rmsnorm_backward(dY, X, gamma, 1e-5)
    x, g = _dev(X, dtype), _dev(gamma, dtype)
    _, rstd = cuda_lib.foak_rmsnorm_forward(x, g, eps=1e-5)
    dx, dg = cuda_lib.foak_rmsnorm_backward(_dev(dY, dtype), x, g, rstd, want_dgamma=False)
    torch.cuda.synchronize()
    assert dg is None
    assert _frob(to_f64(dx), ref_dx) < (4e-3 if dtype == wl.BF16 else 1e-5)
