"""GPU parity of the rotary position embedding (table build and in-place apply,
forward and inverse) against the float64 oracle.

Bars: the table within fp32 rounding of cos/sin (6e-8 absolute); rotated values
within one bf16 ulp of the oracle for bf16 (the grad bar: max(2^(e-7), 1e-6)), and
within 1e-6 of the largest magnitude for fp32; out-of-range positions flagged in
the error word and their tokens left bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from ce_helpers import assert_grad_close, bits, to_f64

pytestmark = pytest.mark.gpu


def _dev(a, dtype):
    a = np.ascontiguousarray(a)
    if dtype == wl.BF16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def _close(got, ref, dtype):
    if dtype == wl.BF16:
        assert_grad_close(got, ref, what="rope")
    else:
        np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-6 * max(1.0, float(np.abs(ref).max())))


def _x(T, H, d, dtype, seed):
    return wl.normal_matrix(T, H * d, seed=seed, sigma=1.0, dtype=dtype, stream=wl.S_X).reshape(T, H, d)


def test_rope_table_matches_cos_sin(cuda_lib):
    cache = cuda_lib.foak_rope_cache(4096, 128, base=500000.0)
    torch.cuda.synchronize()
    half = 64
    tab = cache.view(torch.float32).cpu().numpy().astype(np.float64)
    plane = (4096 * half * 4 + 255) // 256 * 256 // 4
    th = oracle.rope_angles(np.arange(4096), 128, 500000.0)
    np.testing.assert_allclose(tab[: 4096 * half].reshape(4096, half), np.cos(th), rtol=0, atol=6e-8)
    np.testing.assert_allclose(tab[plane: plane + 4096 * half].reshape(4096, half), np.sin(th), rtol=0, atol=6e-8)


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
@pytest.mark.parametrize("T,H,d,base", [(1, 1, 16, 10000.0), (5, 3, 32, 10000.0), (77, 4, 128, 500000.0),
                                        (300, 8, 64, 10000.0)])
@pytest.mark.parametrize("inverse", [False, True])
def test_rope_matches_oracle(cuda_lib, dtype, T, H, d, base, inverse):
    X = _x(T, H, d, dtype, seed=T + H + d)
    pos = np.random.default_rng(T).integers(0, 4096, size=T).astype(np.int64)
    ref = oracle.rope(X, pos, base, inverse=inverse)
    cache = cuda_lib.foak_rope_cache(4096, d, base=base)
    x = _dev(X, dtype)
    err = cuda_lib.foak_rope_apply(x, torch.from_numpy(pos).cuda(), cache, inverse=inverse)
    torch.cuda.synchronize()
    assert err.item() == 0
    _close(to_f64(x), ref, dtype)


def test_rope_round_trip_and_qkv_views(cuda_lib):
    """Q and K as views of a fused QKV buffer (token stride (32 + 2*8) * 128): the
    rotation touches only its view; forward then inverse gives the input back."""
    T, d = 64, 128
    qkv = torch.randn(T, 48, d, device="cuda", dtype=torch.float32)
    ref = qkv.clone()
    q, k = qkv[:, :32], qkv[:, 32:40]
    pos = torch.arange(T, device="cuda", dtype=torch.int64) * 37
    cache = cuda_lib.foak_rope_cache(4096, d, base=500000.0)
    cuda_lib.foak_rope_apply(q, pos, cache)
    cuda_lib.foak_rope_apply(k, pos, cache)
    torch.cuda.synchronize()
    assert torch.equal(qkv[:, 40:], ref[:, 40:])  # V untouched
    want = oracle.rope(ref[:, :32].cpu().numpy(), pos.cpu().numpy(), 500000.0)
    _close(q.cpu().numpy().astype(np.float64), want, wl.F32)
    cuda_lib.foak_rope_apply(q, pos, cache, inverse=True)
    cuda_lib.foak_rope_apply(k, pos, cache, inverse=True)
    torch.cuda.synchronize()
    np.testing.assert_allclose(qkv.cpu().numpy(), ref.cpu().numpy(), rtol=0, atol=2e-6)


def test_rope_out_of_range_positions_flagged(cuda_lib):
    X = _x(6, 2, 32, wl.BF16, seed=4)
    pos = np.array([0, 5, -1, 100, 4096, 7], dtype=np.int64)
    cache = cuda_lib.foak_rope_cache(4096, 32)
    x = _dev(X, wl.BF16)
    err = cuda_lib.foak_rope_apply(x, torch.from_numpy(pos).cuda(), cache)
    torch.cuda.synchronize()
    assert err.item() == cuda_lib.FOAK_ERRBIT_LABEL_RANGE
    got = bits(x)
    np.testing.assert_array_equal(got[[2, 4]], X[[2, 4]].view(np.int16))  # untouched, bit-exact
    ok = np.array([0, 1, 3, 5])
    assert_grad_close(to_f64(x)[ok], oracle.rope(X[ok], pos[ok], 10000.0), what="rope")


def test_rope_empty(cuda_lib):
    cache = cuda_lib.foak_rope_cache(16, 16)
    x = torch.empty(0, 4, 16, dtype=torch.bfloat16, device="cuda")
    err = cuda_lib.foak_rope_apply(x, torch.empty(0, dtype=torch.int64, device="cuda"), cache)
    torch.cuda.synchronize()
    assert err.item() == 0


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
def test_rope_llama3_full_size(cuda_lib, dtype):
    """Llama-3-8B shapes: Q 8192 x 32 x 128 and K 8192 x 8 x 128, packed positions, base 500000."""
    w = wl.rope_llama3(dtype=dtype)
    cache = cuda_lib.foak_rope_cache(w["max_pos"], w["d"], base=w["base"])
    pos = torch.from_numpy(w["positions"]).cuda()
    for name in ("Q", "K"):
        x = _dev(w[name], dtype)
        err = cuda_lib.foak_rope_apply(x, pos, cache)
        torch.cuda.synchronize()
        assert err.item() == 0
        _close(to_f64(x), oracle.rope(w[name], w["positions"], w["base"]), dtype)


@pytest.mark.parametrize("inverse", [False, True])
def test_rope_qk_one_launch_matches_separate_calls(cuda_lib, inverse):
    """Q and K views of a fused QKV buffer rotated in one launch give the same bits as two calls."""
    T, d = 333, 128
    qkv = torch.randn(T, 48, d, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    two = qkv.clone()
    pos = torch.from_numpy(wl.packed_positions(T, seed=5, max_len=100)).cuda()
    cache = cuda_lib.foak_rope_cache(2048, d, base=500000.0)
    err = cuda_lib.foak_rope_apply_qk(qkv[:, :32], qkv[:, 32:40], pos, cache, inverse=inverse)
    cuda_lib.foak_rope_apply(two[:, :32], pos, cache, inverse=inverse)
    cuda_lib.foak_rope_apply(two[:, 32:40], pos, cache, inverse=inverse)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(qkv.view(torch.int16), two.view(torch.int16))
