"""GPU parity of the row kernels (forward, backward, fused fwd+bwd) against the oracle.

Every call goes through the C ABI (via the ctypes binding).  Bars: loss within 1e-5
relative (fp32 logits) or 2e-3 (bf16); dlogits within one bf16 ulp of the oracle or
1e-6 absolute, whichever is larger; ignored rows bit-exact +0.0 and excluded from
n_valid; n_valid and the error word exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from ce_helpers import (assert_grad_close, assert_grad_rows, assert_loss_close, bits, to_device, to_f64)

pytestmark = pytest.mark.gpu


def _rand(N, V, dtype, seed, ld=None, sigma=2.0, n_ignore=None, spikes=0.0):
    x = wl.normal_matrix(N, V, seed=seed, sigma=sigma, dtype=dtype, ld=ld, spike_p=spikes, spike_lo=20.0,
                         spike_hi=30.0)
    y = wl.uniform_labels(N, V, seed=seed)
    k = N // 7 if n_ignore is None else n_ignore
    y[wl.pick_rows(N, min(k, N), seed=seed)] = -100
    return x, y


def _device_logits(x, dtype, V, col_offset=0):
    """Device N x V view (row stride = x's ld); col_offset shifts the base by whole elements."""
    t = to_device(x, dtype)
    return t[:, col_offset:col_offset + V]


def _check_fused(ce, x, y, V, dtype, g=1.0, denom=0.0, ii=-100, col_offset=0):
    xv = x[:, col_offset:col_offset + V] if col_offset else x
    ref = oracle.ce(np.ascontiguousarray(xv) if col_offset else x, y, V, ignore_index=ii, g=g, denom=denom)
    t = _device_logits(x, dtype, V, col_offset)
    out = ce.foak_ce_fwd_bwd(t, torch.from_numpy(y).cuda(), g=g, denom=denom, ignore_index=ii, want_lse=True)
    torch.cuda.synchronize()
    assert_loss_close(out["loss"].item(), ref["loss"], dtype)
    assert out["n_valid"].item() == ref["n_valid"]
    assert out["err"].item() == (1 if ref["n_bad"] else 0)
    got = to_f64(t)
    assert_grad_close(got, ref["grad"])
    valid = ref["state"] == oracle.VALID
    np.testing.assert_allclose(to_f64(out["lse"])[valid], ref["lse"][valid], rtol=2e-6, atol=2e-6)
    assert np.all(bits(t)[~valid] == 0), "ignored rows must be +0.0 bit-exact"
    return out, ref


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
@pytest.mark.parametrize("N,V", [(1, 1), (3, 2), (5, 7), (9, 8), (17, 9), (64, 1000), (33, 4097),
                                 (40, 32000), (13, 32003)])
def test_fused_small_shapes(cuda_lib, dtype, N, V):
    x, y = _rand(N, V, dtype, seed=100 + N + V)
    _check_fused(cuda_lib, x, y, V, dtype)


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
@pytest.mark.parametrize("N,V", [(6, 40000), (7, 70001), (5, 128256)])
def test_fused_cluster_rows(cuda_lib, dtype, N, V):
    # rows longer than one CTA's 64 KB slice: by default one CTA streams the row twice
    x, y = _rand(N, V, dtype, seed=200 + V, sigma=3.0, n_ignore=1, spikes=1e-4)
    _check_fused(cuda_lib, x, y, V, dtype)


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
@pytest.mark.parametrize("V,ld,off", [(1000, 1024, 0), (1001, 1001, 0), (999, 1008, 1), (5003, 5011, 3),
                                      (40001, 40001, 0), (70003, 70016, 5)])
def test_fused_padded_and_unaligned_rows(cuda_lib, dtype, V, ld, off):
    N = 11
    x = wl.normal_matrix(N, ld, seed=V + ld, sigma=2.0, dtype=dtype)
    y = wl.uniform_labels(N, V, seed=V)
    y[3] = -100
    y[0] = 0
    y[1] = V - 1  # label in the scalar head / tail
    _check_fused(cuda_lib, x, y, V, dtype, col_offset=off)
    # padding columns untouched by the in-place call? (only the N x V view is written)


def test_fused_padding_columns_untouched(cuda_lib):
    N, V, ld = 8, 3001, 3072
    x = wl.normal_matrix(N, ld, seed=3, sigma=2.0, dtype=wl.BF16)
    y = wl.uniform_labels(N, V, seed=3)
    y[2] = -100
    full = to_device(x, wl.BF16)
    before = bits(full)[:, V:].copy()
    cuda_lib.foak_ce_fwd_bwd(full[:, :V], torch.from_numpy(y).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(full)[:, V:], before)


def test_tiny_config_all_entry_points(cuda_lib):
    c = wl.tiny()
    x, y, V = c["logits"], c["labels"], c["V"]
    ref = oracle.ce(x, y, g=1.0)
    yd = torch.from_numpy(y).cuda()
    # fused
    _check_fused(cuda_lib, x, y, V, wl.F32)
    # forward
    t = to_device(x, wl.F32)
    f = cuda_lib.foak_ce_forward(t, yd, want_lse=True, want_row_loss=True)
    torch.cuda.synchronize()
    assert_loss_close(f["loss"].item(), ref["loss"], wl.F32)
    np.testing.assert_allclose(to_f64(f["row_loss"]), ref["row_loss"], rtol=1e-5, atol=1e-5)
    np.testing.assert_array_equal(to_f64(t), x.astype(np.float64))  # forward does not write logits
    # backward (out of place, then in place), g as a device scalar
    g = torch.tensor([2.5], dtype=torch.float32, device="cuda")
    d, err = cuda_lib.foak_ce_backward(t, yd, f["lse"], g)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert_grad_close(to_f64(d), 2.5 * ref["grad"])
    d2, _ = cuda_lib.foak_ce_backward(t, yd, f["lse"], g, dlogits=t)
    torch.cuda.synchronize()
    assert_grad_close(to_f64(t), 2.5 * ref["grad"])


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
def test_vocabulary_past_the_one_pass_plans(cuda_lib, dtype):
    """V = 600011: past what 8 CTAs x 64 KB hold in either dtype, so every call streams
    the rows twice; fused, forward and backward against the oracle."""
    N, V = 3, 600011
    assert cuda_lib.foak_ce_max_vocab(cuda_lib.FOAK_F32 if dtype == wl.F32 else cuda_lib.FOAK_BF16) >= V
    x, y = _rand(N, V, dtype, seed=61, sigma=3.0, n_ignore=1, spikes=1e-4)
    y[0] = V - 1
    ref = oracle.ce(x, y, g=1.0)
    _check_fused(cuda_lib, x, y, V, dtype)
    t, yd = to_device(x, dtype), torch.from_numpy(y).cuda()
    f = cuda_lib.foak_ce_forward(t, yd, want_lse=True)
    d, err = cuda_lib.foak_ce_backward(t, yd, f["lse"])
    torch.cuda.synchronize()
    assert err.item() == 0
    assert_loss_close(f["loss"].item(), ref["loss"], dtype)
    assert_grad_close(to_f64(d), ref["grad"])


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
def test_forward_backward_padded_unaligned(cuda_lib, dtype):
    N, V, ld, off = 21, 33001, 33013, 1
    x = wl.normal_matrix(N, ld, seed=9, sigma=2.0, dtype=dtype)
    y = wl.uniform_labels(N, V, seed=9)
    y[[4, 5]] = -100
    xv = np.ascontiguousarray(x[:, off:off + V])
    ref = oracle.ce(xv, y)
    t = to_device(x, dtype)[:, off:off + V]
    yd = torch.from_numpy(y).cuda()
    f = cuda_lib.foak_ce_forward(t, yd)
    d, _ = cuda_lib.foak_ce_backward(t, yd, f["lse"])
    torch.cuda.synchronize()
    assert_loss_close(f["loss"].item(), ref["loss"], dtype)
    assert_grad_close(to_f64(d), ref["grad"])
    assert np.all(bits(d)[[4, 5]] == 0)


def test_g_denom_and_ignore_index(cuda_lib):
    x, y = _rand(50, 3000, wl.BF16, seed=77)
    y[y == -100] = -1
    _check_fused(cuda_lib, x, y, 3000, wl.BF16, g=0.37, denom=123.0, ii=-1)


def test_all_rows_ignored_and_empty(cuda_lib):
    x = wl.normal_matrix(4, 500, seed=1, sigma=1.0, dtype=wl.F32)
    y = np.full(4, -100, dtype=np.int64)
    t = to_device(x, wl.F32)
    out = cuda_lib.foak_ce_fwd_bwd(t, torch.from_numpy(y).cuda())
    torch.cuda.synchronize()
    assert math.isnan(out["loss"].item()) and out["n_valid"].item() == 0
    assert np.all(bits(t) == 0)
    e = torch.empty(0, 500, dtype=torch.float32, device="cuda")
    out = cuda_lib.foak_ce_fwd_bwd(e, torch.empty(0, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert math.isnan(out["loss"].item()) and out["n_valid"].item() == 0 and out["err"].item() == 0


def test_bad_labels_flagged_and_ignored(cuda_lib):
    x, y = _rand(30, 777, wl.F32, seed=5)
    y[2] = 777
    y[9] = -5
    out, ref = _check_fused(cuda_lib, x, y, 777, wl.F32)
    assert ref["n_bad"] == 2 and out["err"].item() == 1


def test_data_parallel_shards_compose(cuda_lib):
    # per-token mean across ranks: each shard divides by the global n_valid
    x, y = _rand(96, 5000, wl.BF16, seed=31)
    n_valid = oracle.count(y, 5000)[0]
    full = to_device(x, wl.BF16)
    o = cuda_lib.foak_ce_fwd_bwd(full, torch.from_numpy(y).cuda())
    parts = []
    tot = 0.0
    for a, b in [(0, 40), (40, 96)]:
        s = to_device(np.ascontiguousarray(x[a:b]), wl.BF16)
        r = cuda_lib.foak_ce_fwd_bwd(s, torch.from_numpy(y[a:b].copy()).cuda(), denom=float(n_valid))
        tot += r["loss"].item()
        parts.append(s)
    torch.cuda.synchronize()
    assert tot == pytest.approx(o["loss"].item(), rel=1e-6)
    np.testing.assert_array_equal(bits(torch.cat(parts)), bits(full))


@pytest.mark.parametrize("dtype,V", [(wl.BF16, 5000), (wl.F32, 70001)])
def test_device_denominator_shards_compose(cuda_lib, dtype, V):
    """The data-parallel pair: foak_ce_count_valid counts each shard's labels on the
    device, the counts are summed on the device (what an all-reduce does across
    ranks), and foak_ce_fwd_bwd_devdenom divides by that total -- the shards'
    losses add up to the whole batch's and their gradients equal it bit for bit,
    and each shard equals foak_ce_fwd_bwd given the same denominator on the host."""
    ce = cuda_lib
    x, y = _rand(96, V, dtype, seed=32, sigma=2.0)
    y[7] = V + 3  # a bad label: flagged by the count and by the fused call
    n_valid, n_bad = oracle.count(y, V)
    full = to_device(x, dtype)
    o = ce.foak_ce_fwd_bwd(full, torch.from_numpy(y).cuda())
    spans = [(0, 40), (40, 96)]
    cnts, errs = [], []
    for a, b in spans:
        e = torch.empty(1, dtype=torch.int32, device="cuda")
        cnts.append(ce.foak_ce_count_valid(torch.from_numpy(y[a:b].copy()).cuda(), V, err=e))
        errs.append(e)
    total = cnts[0] + cnts[1]  # the all-reduce of two ranks, on the device
    tot_loss, parts = 0.0, []
    for a, b in spans:
        s = to_device(np.ascontiguousarray(x[a:b]), dtype)
        s2 = s.clone()
        ys = torch.from_numpy(y[a:b].copy()).cuda()
        r = ce.foak_ce_fwd_bwd_devdenom(s, ys, total)
        h = ce.foak_ce_fwd_bwd(s2, ys, denom=float(n_valid))
        torch.cuda.synchronize()
        assert r["loss"].item() == h["loss"].item()
        assert torch.equal(bits_view(s), bits_view(s2))
        tot_loss += r["loss"].item()
        parts.append(s)
    torch.cuda.synchronize()
    assert [int(c.item()) for c in cnts] == [oracle.count(y[a:b], V)[0] for a, b in spans]
    assert int(total.item()) == n_valid and n_bad == 1
    assert [int(e.item()) for e in errs] == [1, 0]
    assert tot_loss == pytest.approx(o["loss"].item(), rel=1e-6)
    np.testing.assert_array_equal(bits(torch.cat(parts)), bits(full))
    # an empty shard counts 0
    assert int(ce.foak_ce_count_valid(torch.empty(0, dtype=torch.int64, device="cuda"), V).item()) == 0


def test_deterministic_and_workspace_reuse(cuda_lib):
    x, y = _rand(300, 2048, wl.BF16, seed=8)
    losses = set()
    for n in [300, 17, 300, 1, 300]:
        t = to_device(np.ascontiguousarray(x[:n]), wl.BF16)
        o = cuda_lib.foak_ce_fwd_bwd(t, torch.from_numpy(y[:n].copy()).cuda())
        if n == 300:
            losses.add(o["loss"].item())
    torch.cuda.synchronize()
    assert len(losses) == 1
    ws = cuda_lib.workspace(300, torch.device("cuda"))
    assert int(ws[:256].count_nonzero().item()) == 0  # header back to zero


# ------------------------------------------------------------ full-size workloads

def _full_size(cuda_lib, cfg):
    """The fused call on a whole workload: loss, n_valid, lse of every valid row and
    every row of the in-place gradient against the oracle."""
    x, y, V, dtype = cfg["logits"], cfg["labels"], cfg["V"], cfg["dtype"]
    n_valid, _ = oracle.count(y, V)
    scale = oracle.scale_of(1.0, 0.0, n_valid)
    lse, rl, st, _ = oracle.rows(x, y, V, scale=scale, want_grad=False)
    ref_loss = oracle.mean(rl, st)
    t = to_device(x, dtype)
    out = cuda_lib.foak_ce_fwd_bwd(t, torch.from_numpy(y).cuda(), want_lse=True)
    torch.cuda.synchronize()
    assert_loss_close(out["loss"].item(), ref_loss, dtype)
    assert out["n_valid"].item() == n_valid and out["err"].item() == 0
    valid = st == oracle.VALID
    np.testing.assert_allclose(to_f64(out["lse"])[valid], lse[valid], rtol=2e-6, atol=2e-6)
    assert_grad_rows(t, x, y, V, scale)
    return out, lse


def test_mistral_batch_full_size(cuda_lib):
    _full_size(cuda_lib, wl.mistral())


def test_packed_batch_full_size(cuda_lib):
    _full_size(cuda_lib, wl.packed())


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
def test_llama3_vocab_full_size(cuda_lib, dtype):
    cfg = wl.llama3(dtype=dtype)
    out, lse = _full_size(cuda_lib, cfg)
    r = wl.LLAMA3_CONST_ROW
    # the all-equal row: lse = 3 + ln V exactly in the oracle
    assert lse[r] == pytest.approx(3.0 + math.log(128256), abs=1e-12)
    assert to_f64(out["lse"])[r] == pytest.approx(3.0 + math.log(128256), abs=3e-6)


_WORKLOADS = {"mistral": wl.mistral, "packed": wl.packed,
              "llama3": lambda: wl.llama3(dtype=wl.BF16), "llama3_f32": lambda: wl.llama3(dtype=wl.F32)}


@pytest.mark.parametrize("in_place", [False, True], ids=["out_of_place", "in_place"])
@pytest.mark.parametrize("name", sorted(_WORKLOADS))
def test_forward_then_backward_full_size(cuda_lib, name, in_place):
    """The separate forward and backward (FastCrossEntropyLoss as a pair) on whole
    workloads, where every persistent CTA of the forward takes many rows (its ring
    of stages wraps) and the backward's grid-stride loop runs many items per CTA:
    loss, n_valid, lse and row_loss of every row, logits left unchanged by the
    forward, and every row of the gradient (g = 0.75 from a device scalar)."""
    cfg = _WORKLOADS[name]()
    x, y, V, dtype = cfg["logits"], cfg["labels"], cfg["V"], cfg["dtype"]
    N = x.shape[0]
    g = 0.75
    n_valid, _ = oracle.count(y, V)
    scale = oracle.scale_of(g, 0.0, n_valid)
    lse, rl, st, _ = oracle.rows(x, y, V, scale=scale, want_grad=False)
    valid = st == oracle.VALID
    t = to_device(x, dtype)
    yd = torch.from_numpy(y).cuda()
    f = cuda_lib.foak_ce_forward(t, yd, want_lse=True, want_row_loss=True)
    torch.cuda.synchronize()
    assert_loss_close(f["loss"].item(), oracle.mean(rl, st), dtype)
    assert f["n_valid"].item() == n_valid and f["err"].item() == 0
    np.testing.assert_allclose(to_f64(f["lse"])[valid], lse[valid], rtol=2e-6, atol=2e-6)
    # a row term lse - x_y carries the lse's own rounding (the lse bar above) besides the
    # loss bar's relative error: a label on a spike leaves ~1e-4 after subtracting ~25
    rtol = 1e-5 if dtype == wl.F32 else 2e-3
    got_rl = to_f64(f["row_loss"])
    tol = rtol * np.abs(rl[valid]) + 2e-6 * (1.0 + np.abs(lse[valid]))
    assert np.all(np.abs(got_rl[valid] - rl[valid]) <= tol), "row_loss out of tolerance"
    assert np.all(got_rl[~valid] == 0.0)
    x_dev = to_device(x, dtype)
    assert torch.equal(bits_view(t), bits_view(x_dev)), "the forward must not write the logits"
    del x_dev
    gd = torch.tensor([g], dtype=torch.float32, device="cuda")
    d, err = cuda_lib.foak_ce_backward(t, yd, f["lse"], gd, dlogits=t if in_place else None)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert (d.data_ptr() == t.data_ptr()) == in_place
    assert_grad_rows(d, x, y, V, scale)
    assert N == d.shape[0]


def bits_view(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


# ------------------------------------------------------------ failure detection

def test_wait_timeout_is_reported_and_recovers(cuda_lib, monkeypatch):
    """A barrier wait that nothing completes runs out its short limit: the call
    reports FOAK_ERRBIT_TIMEOUT (FOAK_ERR_TIMEOUT under FOAK_SYNC_CHECK=1), nothing
    faults, and the next call on the same workspace is correct."""
    ce = cuda_lib
    cases = [_rand(300, 5000, wl.BF16, seed=4), _rand(6, 128256, wl.BF16, seed=5, n_ignore=1)]
    try:
        ce.lib.foak_test_set_wait_limit_ns(100_000_000)
        for x, y in cases:
            row = int(np.nonzero(y != -100)[0][2])
            ce.lib.foak_test_skip_row_load(row)
            t = to_device(x, wl.BF16)
            out = ce.foak_ce_fwd_bwd(t, torch.from_numpy(y).cuda())
            torch.cuda.synchronize()
            assert out["err"].item() & ce.FOAK_ERRBIT_TIMEOUT
            monkeypatch.setenv("FOAK_SYNC_CHECK", "1")
            with pytest.raises(ce.FoakError) as ei:
                ce.foak_ce_fwd_bwd(to_device(x, wl.BF16), torch.from_numpy(y).cuda())
            assert ei.value.status == ce.FOAK_ERR_TIMEOUT
            monkeypatch.delenv("FOAK_SYNC_CHECK")
    finally:
        ce.lib.foak_test_skip_row_load(-1)
        ce.lib.foak_test_set_wait_limit_ns(0)
    for x, y in cases:
        _check_fused(cuda_lib, x, y, x.shape[1], wl.BF16)


def test_sync_check_reports_bad_labels(cuda_lib, monkeypatch):
    ce = cuda_lib
    x, y = _rand(20, 300, wl.F32, seed=6)
    y[4] = 300
    monkeypatch.setenv("FOAK_SYNC_CHECK", "1")
    with pytest.raises(ce.FoakError) as ei:
        ce.foak_ce_fwd_bwd(to_device(x, wl.F32), torch.from_numpy(y).cuda())
    assert ei.value.status == ce.FOAK_ERR_LABEL_RANGE


def test_many_rows_per_cta(cuda_lib):
    # more than 1024 rows per CTA: labels past the shared-memory cache are read from global memory
    N, V = 160_000, 64
    x, y = _rand(N, V, wl.F32, seed=12, n_ignore=N // 10)
    _check_fused(cuda_lib, x, y, V, wl.F32)


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
def test_loss_sum_within_one_ulp_of_exact(cuda_lib, dtype):
    """The loss is the exact sum of the kernel's own row terms (lse - x_y in float32,
    reproduced here from the returned lse) over D, to within one float ulp.  Row 0's
    label logit is -1000 (a term near 1e3), every other row's +25 (terms near 2e-6,
    each below half an ulp of the running total): together the small terms move the
    sum by over a hundred ulps, which a float accumulation would lose entirely.  bf16
    takes the one-CTA row kernel, fp32 (125 KB rows) the two-pass one."""
    N, V = 4096, 32000
    x = wl.normal_matrix(N, V, seed=77, sigma=2.0, dtype=dtype)
    y = wl.uniform_labels(N, V, seed=77)
    r = np.arange(N)
    val = np.where(r == 0, -1000.0, 25.0)
    x[r, y] = wl.f64_to_bf16_bits(val) if dtype == wl.BF16 else val.astype(np.float32)
    y[wl.pick_rows(N, 50, seed=77, exclude=(0,))] = -100
    out = cuda_lib.foak_ce_fwd_bwd(to_device(x, dtype), torch.from_numpy(y).cuda(), want_lse=True)
    lse = out["lse"].cpu().numpy()
    valid = y != -100
    xy = x[r[valid], y[valid]]
    xy = wl.bf16_bits_to_f64(xy).astype(np.float32) if dtype == wl.BF16 else xy
    terms = lse[valid] - xy  # float32 arithmetic, as in the kernel
    n = int(valid.sum())
    want = np.float32(math.fsum(terms.astype(np.float64)) / n)
    got = np.float32(out["loss"].item())
    assert out["n_valid"].item() == n
    assert abs(int(got.view(np.int32)) - int(want.view(np.int32))) <= 1, (got, want)
    # the same terms accumulated in float32 from row 0 on land far from the exact value
    naive = np.float32(0.0)
    for t in terms:
        naive = np.float32(naive + t)
    assert abs(int(np.float32(naive / np.float32(n)).view(np.int32)) - int(want.view(np.int32))) > 50


def test_forward_counts_on_the_way_with_bad_labels(cuda_lib):
    """The forward of aligned rows counts each CTA's labels on the way and adds the counts
    at the end: n_valid, the label-range bit and the loss must come out as the oracle's
    with ignored and out-of-range labels among 700 rows (several per CTA)."""
    N, V = 700, 4000
    x, y = _rand(N, V, wl.BF16, seed=31, n_ignore=60)
    y[[3, 401]] = [V, -7]  # out of range: counted as bad, treated as ignored
    ref = oracle.ce(x, y, V)
    f = cuda_lib.foak_ce_forward(to_device(x, wl.BF16), torch.from_numpy(y).cuda(), want_lse=True)
    torch.cuda.synchronize()
    assert ref["n_bad"] == 2
    assert f["n_valid"].item() == ref["n_valid"] and f["err"].item() == 1
    assert_loss_close(f["loss"].item(), ref["loss"], wl.BF16)
    valid = ref["state"] == oracle.VALID
    np.testing.assert_allclose(to_f64(f["lse"])[valid], ref["lse"][valid], rtol=2e-6, atol=2e-6)
