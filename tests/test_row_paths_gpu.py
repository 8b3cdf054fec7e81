"""Every row kernel on the same inputs: the one-pass kernel (one CTA per row in
step, or a cluster of 2-8 CTAs when the row is longer than a 64 KB slice), the
two-pass streaming kernel (one CTA per row, the row loaded twice in 64 KB chunks)
and the independent-warp kernel (aligned rows of one slice; each warp streams a
4 KB region of every row).  The automatic choice takes the independent-warp
kernel for aligned rows of one slice, the one-pass kernel for other rows of one
slice and the two-pass kernel beyond; here each is forced through the row-path
test hook (the independent-warp hook falls back to the automatic choice where
it does not apply) and checked against the oracle with the same bars as the
other fused tests.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from ce_helpers import assert_grad_close, assert_loss_close, bits, to_device, to_f64
from test_ce_gpu import _check_fused, _rand

pytestmark = pytest.mark.gpu

ONE_PASS, TWO_PASS, WARPS = 1, 2, 3


@pytest.fixture
def row_path(cuda_lib, request):
    cuda_lib.lib.foak_test_set_row_path(request.param)
    yield request.param
    cuda_lib.lib.foak_test_set_row_path(0)


@pytest.mark.parametrize("row_path", [ONE_PASS, TWO_PASS, WARPS], indirect=True)
@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
@pytest.mark.parametrize("N,V", [(1, 1), (5, 7), (9, 8), (64, 1000), (33, 4097), (13, 32003), (6, 40000),
                                 (7, 70001), (5, 128256), (3, 200003), (2, 300007)])
def test_fused_both_paths(cuda_lib, row_path, dtype, N, V):
    """Rows past the one-pass plans' reach (fp32 from 131073, bf16 from 262145) take the
    two-pass kernel whatever path is asked for."""
    x, y = _rand(N, V, dtype, seed=300 + N + V, sigma=3.0, n_ignore=1, spikes=1e-4)
    _check_fused(cuda_lib, x, y, V, dtype)


@pytest.mark.parametrize("row_path", [ONE_PASS, TWO_PASS], indirect=True)
@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
@pytest.mark.parametrize("V,ld,off", [(999, 1008, 1), (40001, 40001, 0), (70003, 70016, 5), (128256, 128263, 3)])
def test_unaligned_rows_both_paths(cuda_lib, row_path, dtype, V, ld, off):
    N = 9
    x = wl.normal_matrix(N, ld, seed=V + ld + off, sigma=2.0, dtype=dtype)
    y = wl.uniform_labels(N, V, seed=V + 1)
    y[3] = -100
    y[0] = 0       # label in the scalar head
    y[1] = V - 1   # label in the scalar tail
    y[2] = min(V - 1, 4096 * (16 // (4 if dtype == wl.F32 else 2)) + 5)  # label past the first 64 KB chunk
    _check_fused(cuda_lib, x, y, V, dtype, col_offset=off)


@pytest.mark.parametrize("row_path", [TWO_PASS], indirect=True)
@pytest.mark.parametrize("g,denom", [(0.37, 123.0), (-1.5, 0.0), (0.0, 0.0)])
def test_two_pass_scale_signs(cuda_lib, row_path, g, denom):
    # scale > 0 is folded into the exponent; zero and negative scales are multiplied
    x, y = _rand(12, 70001, wl.BF16, seed=41, n_ignore=2)
    _check_fused(cuda_lib, x, y, 70001, wl.BF16, g=g, denom=denom)


@pytest.mark.parametrize("row_path", [TWO_PASS], indirect=True)
@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
def test_two_pass_forward_only(cuda_lib, row_path, dtype):
    N, V = 10, 128256
    x, y = _rand(N, V, dtype, seed=43, n_ignore=2)
    ref = oracle.ce(x, y)
    t = to_device(x, dtype)
    f = cuda_lib.foak_ce_forward(t, torch.from_numpy(y).cuda(), want_lse=True, want_row_loss=True)
    torch.cuda.synchronize()
    assert_loss_close(f["loss"].item(), ref["loss"], dtype)
    valid = ref["state"] == oracle.VALID
    np.testing.assert_allclose(to_f64(f["lse"])[valid], ref["lse"][valid], rtol=2e-6, atol=2e-6)
    np.testing.assert_allclose(to_f64(f["row_loss"]), ref["row_loss"], rtol=1e-5, atol=1e-5)
    np.testing.assert_array_equal(bits(t), bits(to_device(x, dtype)))  # logits not written


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
def test_paths_agree_on_llama3_rows(cuda_lib, dtype):
    """The two kernels on 300 rows of the Llama-3 batch (V = 128256): losses agree
    to fp32 summation order, gradients to one bf16 ulp, ignored rows both +0.0."""
    cfg = wl.llama3(dtype=dtype, rows=300)
    x, y = cfg["logits"], cfg["labels"]
    outs = []
    try:
        for path in (ONE_PASS, TWO_PASS):
            cuda_lib.lib.foak_test_set_row_path(path)
            t = to_device(x, dtype)
            out = cuda_lib.foak_ce_fwd_bwd(t, torch.from_numpy(y).cuda(), want_lse=True)
            torch.cuda.synchronize()
            outs.append((out["loss"].item(), to_f64(out["lse"]), to_f64(t), out["n_valid"].item()))
    finally:
        cuda_lib.lib.foak_test_set_row_path(0)
    (l1, lse1, g1, n1), (l2, lse2, g2, n2) = outs
    assert n1 == n2
    assert l2 == pytest.approx(l1, rel=2e-6)
    np.testing.assert_allclose(lse2, lse1, rtol=2e-6, atol=2e-6)
    assert_grad_close(g2, g1)


def test_two_pass_timeout_is_reported_and_recovers(cuda_lib):
    """The two-pass kernel's load of one row never completes (test hook): the wait
    runs out its short limit, the call reports FOAK_ERRBIT_TIMEOUT, and the next
    call on the same workspace is correct."""
    ce = cuda_lib
    x, y = _rand(400, 70001, wl.BF16, seed=47, n_ignore=20)
    try:
        ce.lib.foak_test_set_row_path(TWO_PASS)
        ce.lib.foak_test_set_wait_limit_ns(100_000_000)
        ce.lib.foak_test_skip_row_load(int(np.nonzero(y != -100)[0][160]))
        out = ce.foak_ce_fwd_bwd(to_device(x, wl.BF16), torch.from_numpy(y).cuda())
        torch.cuda.synchronize()
        assert out["err"].item() & ce.FOAK_ERRBIT_TIMEOUT
        ce.lib.foak_test_skip_row_load(-1)
        ce.lib.foak_test_set_wait_limit_ns(0)
        _check_fused(cuda_lib, x, y, 70001, wl.BF16)
    finally:
        ce.lib.foak_test_skip_row_load(-1)
        ce.lib.foak_test_set_wait_limit_ns(0)
        ce.lib.foak_test_set_row_path(0)


def test_two_pass_all_ignored_and_empty(cuda_lib):
    ce = cuda_lib
    try:
        ce.lib.foak_test_set_row_path(TWO_PASS)
        x = wl.normal_matrix(3, 70001, seed=2, sigma=1.0, dtype=wl.BF16)
        t = to_device(x, wl.BF16)
        out = ce.foak_ce_fwd_bwd(t, torch.full((3,), -100, dtype=torch.int64, device="cuda"))
        torch.cuda.synchronize()
        assert math.isnan(out["loss"].item()) and out["n_valid"].item() == 0
        assert np.all(bits(t) == 0)
        e = torch.empty(0, 70001, dtype=torch.bfloat16, device="cuda")
        out = ce.foak_ce_fwd_bwd(e, torch.empty(0, dtype=torch.int64, device="cuda"))
        torch.cuda.synchronize()
        assert math.isnan(out["loss"].item()) and out["err"].item() == 0
    finally:
        ce.lib.foak_test_set_row_path(0)


@pytest.mark.parametrize("row_path", [WARPS, ONE_PASS], indirect=True)
@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
@pytest.mark.parametrize("g,denom", [(0.37, 123.0), (-1.5, 0.0), (0.0, 0.0)])
def test_aligned_rows_scale_signs(cuda_lib, row_path, dtype, g, denom):
    # aligned rows of one slice: a positive scale is folded into the exponent, zero
    # and negative scales multiply; several rows per CTA so the row rings wrap
    x, y = _rand(700, 4096, dtype, seed=43, n_ignore=60)
    _check_fused(cuda_lib, x, y, 4096, dtype, g=g, denom=denom)


@pytest.mark.parametrize("row_path", [WARPS], indirect=True)
@pytest.mark.parametrize("V", [8, 1024, 8000, 16384, 32768])
def test_independent_warps_region_edges(cuda_lib, row_path, V):
    # rows that end inside, or exactly at the end of, a warp's 4 KB region and a
    # 64 KB stage; labels at the first and last column and at a region boundary
    dtype = wl.BF16
    x, y = _rand(400, V, dtype, seed=V + 7, n_ignore=37, spikes=1e-3)
    y[0], y[1], y[2] = 0, V - 1, min(V - 1, 2048)
    _check_fused(cuda_lib, x, y, V, dtype)
    f = cuda_lib.foak_ce_forward(to_device(x, dtype), torch.from_numpy(y).cuda(), want_lse=True,
                                 want_row_loss=True)
    torch.cuda.synchronize()
    ref = oracle.ce(x, y, V)
    assert_loss_close(f["loss"].item(), ref["loss"], dtype)
    valid = ref["state"] == oracle.VALID
    np.testing.assert_allclose(to_f64(f["lse"])[valid], ref["lse"][valid], rtol=2e-6, atol=2e-6)


@pytest.mark.parametrize("row_path", [WARPS], indirect=True)
def test_independent_warps_wait_timeout(cuda_lib, row_path, monkeypatch):
    """A row load that never happens makes the independent-warp kernel's waits run out
    (fused and forward): the call reports FOAK_ERRBIT_TIMEOUT without faulting, every
    warp winds down, and the next call is correct."""
    ce = cuda_lib
    x, y = _rand(400, 4096, wl.BF16, seed=19, n_ignore=20)
    row = int(np.nonzero(y != -100)[0][200])
    try:
        ce.lib.foak_test_set_wait_limit_ns(100_000_000)
        ce.lib.foak_test_skip_row_load(row)
        out = ce.foak_ce_fwd_bwd(to_device(x, wl.BF16), torch.from_numpy(y).cuda())
        f = ce.foak_ce_forward(to_device(x, wl.BF16), torch.from_numpy(y).cuda())
        torch.cuda.synchronize()
        assert out["err"].item() & ce.FOAK_ERRBIT_TIMEOUT
        assert f["err"].item() & ce.FOAK_ERRBIT_TIMEOUT
    finally:
        ce.lib.foak_test_skip_row_load(-1)
        ce.lib.foak_test_set_wait_limit_ns(0)
    _check_fused(cuda_lib, x, y, 4096, wl.BF16)
    f = ce.foak_ce_forward(to_device(x, wl.BF16), torch.from_numpy(y).cuda())
    torch.cuda.synchronize()
    assert f["err"].item() == 0
    assert_loss_close(f["loss"].item(), oracle.ce(x, y, 4096)["loss"], wl.BF16)
