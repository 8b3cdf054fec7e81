"""Shared helpers of the GPU parity tests (device transfer, tolerances, sampling)."""
import numpy as np
import torch

import workloads as wl

LOSS_RTOL = {wl.F32: 1e-5, wl.BF16: 2e-3}


def to_device(a: np.ndarray, dtype: int, device="cuda") -> torch.Tensor:
    """Upload fp32 values, or bf16 bit patterns (uint16), as a torch tensor of that dtype."""
    if dtype == wl.BF16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw element bits (int16 for bf16, int32 for fp32) of a device tensor."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy()
    return t.view(torch.int32).cpu().numpy()


def grad_tol(ref: np.ndarray) -> np.ndarray:
    """One bf16 ulp of the oracle value, or 1e-6 absolute, whichever is larger."""
    a = np.abs(ref)
    ulp = np.exp2(np.floor(np.log2(np.where(a > 0, a, 1e-300))) - 7)
    return np.maximum(ulp, 1e-6)


def assert_grad_close(got: np.ndarray, ref: np.ndarray, what: str = "dlogits"):
    err = np.abs(got - ref)
    # every element within 1e-6 passes (the bar's absolute term); only the rest need their ulp
    over = err > 1e-6
    if not over.any():
        return
    tol = np.full(err.shape, 1e-6)
    tol[over] = grad_tol(ref[over])
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at {i}: "
                             f"got {got[i]!r} oracle {ref[i]!r} tol {tol[i]!r}")


def assert_grad_rows(dl: torch.Tensor, x: np.ndarray, y: np.ndarray, V: int, scale: float,
                     ignore_index: int = -100, block: int = 256):
    """Every row of the device gradient ``dl`` (N x V) against the oracle, a block of rows at a
    time: element by element within the dlogits bar, ignored rows +0.0 bit-exact."""
    import oracle

    N = x.shape[0]
    for a in range(0, N, block):
        b = min(N, a + block)
        _, _, st, g = oracle.rows(x[a:b], y[a:b], V, ignore_index=ignore_index, scale=scale)
        got = dl[a:b]
        assert_grad_close(to_f64(got), g, f"dlogits rows {a}..{b - 1}")
        ign = np.nonzero(st != oracle.VALID)[0]
        if ign.size:
            z = bits(got[torch.from_numpy(ign).to(got.device)])
            assert not z.any(), f"ignored rows in {a}..{b - 1} must be +0.0 bit-exact"


def assert_loss_close(got: float, ref: float, dtype: int):
    if np.isnan(ref):
        assert np.isnan(got), (got, ref)
        return
    # relative bar; a loss that is (near) zero, e.g. V = 1, gets a 1e-6 absolute floor
    tol = max(LOSS_RTOL[dtype] * abs(ref), 1e-6)
    assert abs(got - ref) <= tol, f"loss {got!r} vs oracle {ref!r} (tol {tol})"
