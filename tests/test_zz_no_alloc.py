"""foak_ce_fwd_bwd_noalloc: the fused call for callers that may not allocate device memory.

It must give what foak_ce_fwd_bwd gives (same loss, n_valid, error word and
dlogits, within the parity tolerances used everywhere else), on consecutive calls
that share its fixed scratch, and refuse batches larger than that scratch.  The
file is named to be collected last; it needs nothing from the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from ce_helpers import assert_grad_close, assert_loss_close, to_device, to_f64

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_noalloc(ce, x, y, g=1.0):
    """Straight through the C ABI with raw device pointers."""
    N, V = x.shape
    dt = ce.FOAK_BF16 if x.dtype == torch.bfloat16 else ce.FOAK_F32
    loss = torch.empty(1, dtype=torch.float32, device=x.device)
    nv = torch.empty(1, dtype=torch.int32, device=x.device)
    err = torch.empty(1, dtype=torch.int32, device=x.device)
    lse = torch.empty(N, dtype=torch.float32, device=x.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = ce.lib.foak_ce_fwd_bwd_noalloc(_p(x), dt, x.stride(0), _p(y), N, V, -100, g, 0.0, _p(loss), _p(lse),
                                        _p(nv), _p(err), stream)
    assert st == ce.FOAK_OK, ce.status_string(st)
    return loss, nv, err, lse


def _case(N, V, dtype, seed):
    x = wl.normal_matrix(N, V, seed=seed, sigma=2.0, dtype=dtype)
    y = wl.uniform_labels(N, V, seed=seed)
    y[wl.pick_rows(N, N // 9, seed=seed)] = -100
    if N > 3:
        y[3] = V + 5  # a bad label: flagged in the error word, row ignored
    return x, y


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
def test_noalloc_matches_workspace_call_twice_in_a_row(cuda_lib, dtype):
    ce = cuda_lib
    # two consecutive calls of different shapes: the second must not see the first's leftovers
    for (N, V, seed) in [(700, 32000, 11), (129, 70001, 12)]:
        x, y = _case(N, V, dtype, seed)
        yd = torch.from_numpy(y).cuda()
        a = to_device(x, dtype)
        b = to_device(x, dtype)
        ref = ce.foak_ce_fwd_bwd(a, yd, g=1.5, want_lse=True)
        loss, nv, err, lse = _call_noalloc(ce, b, yd, g=1.5)
        torch.cuda.synchronize()
        assert_loss_close(loss.item(), ref["loss"].item(), dtype)
        assert nv.item() == ref["n_valid"].item()
        assert err.item() == ref["err"].item() == 1
        np.testing.assert_allclose(to_f64(lse), to_f64(ref["lse"]), rtol=2e-6, atol=2e-6)
        assert_grad_close(to_f64(b), to_f64(a), what="noalloc dlogits")


def test_noalloc_rejects_batches_beyond_its_scratch(cuda_lib):
    ce = cuda_lib
    n = ce.FOAK_CE_NOALLOC_MAX_ROWS + 1
    x = torch.zeros(n, 8, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(n, dtype=torch.int64, device="cuda")
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    st = ce.lib.foak_ce_fwd_bwd_noalloc(_p(x), ce.FOAK_BF16, 8, _p(y), n, 8, -100, 1.0, 0.0, _p(loss), None, None,
                                        None, None)
    assert st == ce.FOAK_ERR_WORKSPACE
    with pytest.raises(ce.FoakError):
        ce.foak_ce_fwd_bwd_noalloc(x, y)
