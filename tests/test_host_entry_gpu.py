"""GPU parity of foak_ce_fwd_bwd_host: logits and labels start in (pinned) host
memory, the call copies them in row chunks and sweeps each chunk as it lands.

Bars: the same as the fused call against the oracle (loss 1e-5 / 2e-3 relative,
dlogits one bf16 ulp or 1e-6, ignored rows +0.0, n_valid and error word exact);
against foak_ce_fwd_bwd on the same inputs the results are bit-identical (each
row is computed the same way whatever the chunking, and the loss is the same
reduction in the same order).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from ce_helpers import assert_grad_close, assert_grad_rows, assert_loss_close, bits, to_f64

pytestmark = pytest.mark.gpu


def _host_tensor(x, dtype):
    t = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) if dtype == wl.BF16 else torch.from_numpy(x)
    return t.pin_memory()


def _run_host(ce, x, y, dtype, g=1.0, denom=0.0, ii=-100):
    hx = _host_tensor(x, dtype)
    hy = torch.from_numpy(y).pin_memory()
    dx = torch.empty(hx.shape, dtype=hx.dtype, device="cuda")
    dy = torch.empty(y.shape[0], dtype=torch.int64, device="cuda")
    out = ce.foak_ce_fwd_bwd_host(hx, hy, dx, dy, g=g, denom=denom, ignore_index=ii)
    torch.cuda.synchronize()
    return out, dx, dy


def _rand(N, V, dtype, seed, n_ignore):
    x = wl.normal_matrix(N, V, seed=seed, sigma=2.0, dtype=dtype)
    y = wl.uniform_labels(N, V, seed=seed)
    y[wl.pick_rows(N, min(n_ignore, N), seed=seed)] = -100
    return x, y


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
@pytest.mark.parametrize("N,V", [(1, 7), (300, 1000), (513, 4096), (1500, 32000), (2049, 3001)])
def test_host_entry_matches_oracle(cuda_lib, dtype, N, V):
    # 513 and 1500 rows give 2 and 3 chunks with a ragged last chunk
    x, y = _rand(N, V, dtype, seed=N + V, n_ignore=N // 9)
    ref = oracle.ce(x, y, V, g=0.75)
    out, dx, dy = _run_host(cuda_lib, x, y, dtype, g=0.75)
    assert_loss_close(out["loss"].item(), ref["loss"], dtype)
    assert out["n_valid"].item() == ref["n_valid"] and out["err"].item() == 0
    assert np.array_equal(dy.cpu().numpy(), y)
    assert_grad_close(to_f64(dx), ref["grad"])
    valid = ref["state"] == oracle.VALID
    assert np.all(bits(dx)[~valid] == 0)


def test_host_entry_bit_identical_to_device_call(cuda_lib):
    cfg = wl.mistral()
    x, y = cfg["logits"], cfg["labels"]
    out, dx, _ = _run_host(cuda_lib, x, y, wl.BF16)
    t = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    ref = cuda_lib.foak_ce_fwd_bwd(t, torch.from_numpy(y).cuda())
    torch.cuda.synchronize()
    assert out["loss"].item() == ref["loss"].item()
    assert out["n_valid"].item() == ref["n_valid"].item() == 4092
    assert torch.equal(dx.view(torch.int16), t.view(torch.int16))


def test_host_entry_mistral_against_oracle(cuda_lib):
    """The headline workload through host buffers: loss, n_valid and every gradient row."""
    cfg = wl.mistral()
    x, y, V = cfg["logits"], cfg["labels"], cfg["V"]
    n_valid, _ = oracle.count(y, V)
    scale = oracle.scale_of(1.0, 0.0, n_valid)
    _, rl, st, _ = oracle.rows(x, y, V, scale=scale, want_grad=False)
    out, dx, _ = _run_host(cuda_lib, x, y, wl.BF16)
    assert_loss_close(out["loss"].item(), oracle.mean(rl, st), wl.BF16)
    assert out["n_valid"].item() == n_valid
    assert_grad_rows(dx, x, y, V, scale)


def test_host_entry_denominator_bad_label_and_ignored(cuda_lib):
    x, y = _rand(700, 2000, wl.F32, seed=5, n_ignore=50)
    y[10] = 2000  # out of range: flagged and treated as ignored
    ref = oracle.ce(x, y, 2000, denom=3000.0)
    out, dx, _ = _run_host(cuda_lib, x, y, wl.F32, denom=3000.0)
    assert_loss_close(out["loss"].item(), ref["loss"], wl.F32)
    assert out["err"].item() == 1 and out["n_valid"].item() == ref["n_valid"]
    assert_grad_close(to_f64(dx), ref["grad"])
    # every row ignored: loss 0/0 = NaN, gradient all +0.0
    y[:] = -100
    out, dx, _ = _run_host(cuda_lib, x, y, wl.F32)
    assert math.isnan(out["loss"].item()) and out["n_valid"].item() == 0
    assert int(dx.view(torch.int32).count_nonzero().item()) == 0


def test_host_entry_empty_batch(cuda_lib):
    hx = torch.empty(0, 500, dtype=torch.float32).pin_memory()
    hy = torch.empty(0, dtype=torch.int64).pin_memory()
    dx = torch.empty(0, 500, dtype=torch.float32, device="cuda")
    dy = torch.empty(0, dtype=torch.int64, device="cuda")
    out = cuda_lib.foak_ce_fwd_bwd_host(hx, hy, dx, dy)
    torch.cuda.synchronize()
    assert math.isnan(out["loss"].item()) and out["n_valid"].item() == 0 and out["err"].item() == 0
