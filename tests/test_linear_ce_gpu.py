"""GPU parity of the chunked linear + cross-entropy against the float64 oracle.

Bars: loss within 2e-3 relative (bf16 inputs), dH and dW within 1e-2 relative
Frobenius error, n_valid and the error word exact; chunking does not change
the result beyond fp32 summation order.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


def _dev(bits):
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def _frob(got, ref):
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def _case(N, V, D, seed, n_ignore):
    H = wl.normal_matrix(N, D, seed=seed, sigma=1.0, dtype=wl.BF16, stream=wl.S_H)
    W = wl.normal_matrix(V, D, seed=seed, sigma=0.05, dtype=wl.BF16, stream=wl.S_W)
    y = wl.uniform_labels(N, V, seed=seed)
    y[wl.pick_rows(N, n_ignore, seed=seed)] = -100
    return H, W, y


def _run(ce, H, W, y, chunk, g=1.0, denom=0.0):
    out = ce.foak_linear_ce_chunked(_dev(H), _dev(W), torch.from_numpy(y).cuda(), chunk=chunk, g=g, denom=denom)
    torch.cuda.synchronize()
    return (out["loss"].item(), out["dH"].float().cpu().numpy().astype(np.float64),
            out["dW"].cpu().numpy().astype(np.float64), out["n_valid"].item(), out["err"].item())


# (2600, 4096, 512, 256): 11 chunks -- dZ passes inside the grouped launches, a dW group
# launched mid-loop, Z slots reused, a partial last group and a 40-row last chunk on
# single-CTA tiles; (600, 1001, 128, 256): a vocabulary that is not a multiple of 8
# (the dZ pass runs by itself)
@pytest.mark.parametrize("N,V,D,chunk", [(300, 1000, 256, 128), (129, 520, 64, 1024), (1024, 4096, 512, 256),
                                         (2600, 4096, 512, 256), (600, 1001, 128, 256)])
def test_linear_ce_small(cuda_lib, N, V, D, chunk):
    H, W, y = _case(N, V, D, seed=N + V + D, n_ignore=N // 10)
    ref = oracle.linear_ce(H, W, y, g=1.5)
    loss, dH, dW, nv, err = _run(cuda_lib, H, W, y, chunk, g=1.5)
    assert abs(loss - ref["loss"]) <= 2e-3 * abs(ref["loss"])
    assert nv == ref["n_valid"] and err == 0
    assert _frob(dH, ref["dH"]) < 1e-2
    assert _frob(dW, ref["dW"]) < 1e-2
    ign = y == -100
    assert np.all(dH[ign] == 0.0)


def test_linear_ce_ragged_vocabulary_and_last_chunk(cuda_lib):
    """V = 40000 (a partial last 256-column tile) in chunks of 512 rows with a 300-row
    last chunk: parity with the oracle, and dH identical to a one-chunk call."""
    H, W, y = _case(1836, 40000, 256, seed=77, n_ignore=180)
    ref = oracle.linear_ce(H, W, y)
    a = _run(cuda_lib, H, W, y, chunk=512)
    assert abs(a[0] - ref["loss"]) <= 2e-3 * abs(ref["loss"])
    assert a[3] == ref["n_valid"] and a[4] == 0
    assert _frob(a[1], ref["dH"]) < 1e-2
    assert _frob(a[2], ref["dW"]) < 1e-2
    b = _run(cuda_lib, H, W, y, chunk=2048)
    np.testing.assert_array_equal(a[1], b[1])
    assert a[0] == pytest.approx(b[0], rel=1e-6)


def test_linear_ce_chunk_size_invariance(cuda_lib):
    H, W, y = _case(512, 777, 128, seed=3, n_ignore=40)
    a = _run(cuda_lib, H, W, y, chunk=512)
    b = _run(cuda_lib, H, W, y, chunk=96)
    assert a[0] == pytest.approx(b[0], rel=1e-6)
    np.testing.assert_array_equal(a[1], b[1])  # dH rows do not depend on the chunking
    assert _frob(b[2], a[2]) < 1e-5            # dW only differs by fp32 summation order


def test_linear_ce_denominator_and_bad_labels(cuda_lib):
    H, W, y = _case(200, 300, 64, seed=9, n_ignore=20)
    y[5] = 300  # out of range: flagged, treated as ignored
    ref = oracle.linear_ce(H, W, y, denom=1000.0)
    loss, dH, dW, nv, err = _run(cuda_lib, H, W, y, 64, denom=1000.0)
    assert abs(loss - ref["loss"]) <= 2e-3 * abs(ref["loss"])
    assert err == 1 and nv == ref["n_valid"]
    assert _frob(dW, ref["dW"]) < 1e-2 and np.all(dH[5] == 0.0)


def test_linear_ce_all_ignored_and_empty(cuda_lib):
    H, W, y = _case(64, 100, 64, seed=1, n_ignore=0)
    y[:] = -100
    loss, dH, dW, nv, err = _run(cuda_lib, H, W, y, 32)
    assert math.isnan(loss) and nv == 0 and err == 0
    assert np.all(dH == 0.0) and np.all(dW == 0.0)
    ce = cuda_lib
    Wd = _dev(W)
    out = ce.foak_linear_ce_chunked(torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"), Wd,
                                    torch.empty(0, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert math.isnan(out["loss"].item()) and int(out["dW"].count_nonzero().item()) == 0


def test_linear_ce_chunked_full_size(cuda_lib):
    """The chunked workload at full size: H 8192x4096, W 32000x4096, chunks of 1024."""
    c = wl.chunked()
    ref = oracle.linear_ce(c["H"], c["W"], c["labels"])
    loss, dH, dW, nv, err = _run(cuda_lib, c["H"], c["W"], c["labels"], c["chunk"])
    assert abs(loss - ref["loss"]) <= 2e-3 * abs(ref["loss"]), (loss, ref["loss"])
    assert nv == ref["n_valid"] == 8192 - 819 and err == 0
    assert _frob(dH, ref["dH"]) < 1e-2
    assert _frob(dW, ref["dW"]) < 1e-2
