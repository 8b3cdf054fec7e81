"""CPU oracle for the fused cross-entropy path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline and
reference legs may import this package.  The product (``cross_entropy_loss_gb300``)
never does, and the two share no code: this side is plain float64 C
(``ce_oracle.c``) plus numpy matrix products for the linear layer.

Definitions followed (the FOAK pages name the kernels but print no formula; the
reading is the textbook one, stated in ``ce_oracle.c``):

* ``ce`` -- softmax cross-entropy over the rows of an N x V logits matrix, mean
  over rows whose label is not ``ignore_index`` ("Fast Cross Entropy Triton
  Kernels", fms-acceleration-foak 0.7.4 page, list of fused operations and
  kernels; FastCrossEntropyLoss, fms-acceleration PR #79, Description item 4),
  with the gradient ``(softmax - onehot) * g / D``.
* ``linear_ce`` -- the same loss applied to ``Z = H W^T`` with the gradients
  ``dH = dZ W`` and ``dW = dZ^T H`` (the fused linear + cross-entropy the pages
  call LigerFusedLinearCrossEntropy -- "Running Liger Kernel Benchmarks" on the
  foak page -- and "chunked loss" -- PR #79, TODO list).  Chunking is a schedule,
  not a different result, so the oracle does not chunk.
* ``rmsnorm`` / ``rmsnorm_backward`` / ``rmsnorm_linear_ce`` -- the RMSNorm the
  foak page lists among its kernels ("Fast RMS LayerNorm Triton Kernels"), alone
  and as the final norm in front of the chunked linear + cross-entropy.
* ``rope`` / ``rope_angles`` -- the rotary position embedding the foak page lists
  ("Fast RoPE Triton Kernels"), with explicit position ids.

Parity pins (closed forms, invariants, finite differences, brute force, a
hand-worked example) live in ``tests/test_oracle_pins.py``; every function here
is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ce_oracle.c")
_LIB = os.path.join(_HERE, "libce_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2
IGNORED, VALID, BAD_LABEL = 0, 1, 2


def build_lib(force: bool = False) -> str:
    """Compile ce_oracle.c with the host gcc (plain -O2, no fast-math, no arch flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_lib())
            i64, dbl, vp, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            lib.oracle_ce_count.argtypes = [vp, i64, i64, i64, vp, vp]
            lib.oracle_ce_rows.argtypes = [vp, i32, i64, vp, i64, i64, i64, i64, dbl, vp, vp, vp, vp]
            lib.oracle_ce_mean.argtypes = [vp, vp, i64, dbl]
            lib.oracle_ce_mean.restype = dbl
            _lib = lib
    return _lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:  # bfloat16 bit patterns
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"oracle: unsupported logits dtype {a.dtype}")


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def count(labels: np.ndarray, V: int, ignore_index: int = -100):
    """(n_valid, n_bad): rows with a label in [0, V), rows with any other non-ignored label."""
    labels = np.ascontiguousarray(labels, dtype=np.int64)
    nv, nb = ctypes.c_int64(), ctypes.c_int64()
    _get().oracle_ce_count(labels.ctypes.data, labels.size, V, ignore_index,
                           ctypes.byref(nv), ctypes.byref(nb))
    return int(nv.value), int(nb.value)


def scale_of(g: float, denom: float, n_valid: int) -> float:
    """g / D with D = denom if denom > 0 else n_valid (inf/NaN when D == 0; no row uses it then)."""
    D = float(denom) if denom > 0 else float(n_valid)
    with np.errstate(divide="ignore", invalid="ignore"):
        return float(np.float64(g) / np.float64(D))


def rows(logits: np.ndarray, labels: np.ndarray, V: int, *, ignore_index: int = -100,
         scale: float = 1.0, want_grad: bool = True, threads: int | None = None):
    """Per-row quantities for every row of ``logits`` (shape rows x ld, ld >= V).

    Returns (lse, row_loss, state, grad) as float64 / int8 arrays; grad is rows x V
    (or None).  ``scale`` multiplies the gradient (g / D of the whole batch).
    """
    logits = np.ascontiguousarray(logits)
    labels = np.ascontiguousarray(labels, dtype=np.int64)
    n, ld = logits.shape
    assert ld >= V and labels.shape == (n,)
    dt = _dtype_code(logits)
    lse = np.zeros(n, dtype=np.float64)
    rl = np.zeros(n, dtype=np.float64)
    st = np.zeros(n, dtype=np.int8)
    grad = np.zeros((n, V), dtype=np.float64) if want_grad else None
    lib = _get()
    nt = max(1, min(threads or default_threads(), n))
    bounds = np.linspace(0, n, nt + 1).astype(np.int64)
    xp, yp = logits.ctypes.data, labels.ctypes.data

    def work(t):
        a, b = int(bounds[t]), int(bounds[t + 1])
        if b > a:
            gp = grad[a:].ctypes.data if grad is not None else None
            lib.oracle_ce_rows(xp, dt, ld, yp, a, b, V, ignore_index, scale,
                               lse[a:].ctypes.data, rl[a:].ctypes.data, st[a:].ctypes.data, gp)

    if nt == 1:
        work(0)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(work, range(nt)))
    return lse, rl, st, grad


def mean(row_loss: np.ndarray, state: np.ndarray, denom: float = 0.0) -> float:
    row_loss = np.ascontiguousarray(row_loss, dtype=np.float64)
    state = np.ascontiguousarray(state, dtype=np.int8)
    return float(_get().oracle_ce_mean(row_loss.ctypes.data, state.ctypes.data, row_loss.size,
                                       float(denom)))


def ce(logits: np.ndarray, labels: np.ndarray, V: int | None = None, *, ignore_index: int = -100,
       g: float = 1.0, denom: float = 0.0, want_grad: bool = True, threads: int | None = None):
    """The whole definition on one batch: loss, n_valid, n_bad, lse, row_loss, state, grad, scale."""
    V = logits.shape[1] if V is None else V
    n_valid, n_bad = count(labels, V, ignore_index)
    scale = scale_of(g, denom, n_valid)
    lse, rl, st, grad = rows(logits, labels, V, ignore_index=ignore_index, scale=scale,
                             want_grad=want_grad, threads=threads)
    loss = mean(rl, st, denom)
    return dict(loss=loss, n_valid=n_valid, n_bad=n_bad, lse=lse, row_loss=rl, state=st,
                grad=grad, scale=scale)


def _to_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def linear_ce(H: np.ndarray, W: np.ndarray, labels: np.ndarray, *, ignore_index: int = -100,
              g: float = 1.0, denom: float = 0.0, threads: int | None = None):
    """Loss, dH and dW of cross-entropy over Z = H W^T, all in float64.

    H: N x D, W: V x D (float32, float64 or bf16 bit patterns).  Steps: Z = H W^T;
    the ``ce`` definition on Z gives loss and dZ; dH = dZ W; dW = dZ^T H.
    """
    Hd, Wd = _to_f64(H), _to_f64(W)
    Z = Hd @ Wd.T
    r = ce(Z, labels, Z.shape[1], ignore_index=ignore_index, g=g, denom=denom, threads=threads)
    dZ = r["grad"]
    dH = dZ @ Wd
    dW = dZ.T @ Hd
    return dict(loss=r["loss"], n_valid=r["n_valid"], n_bad=r["n_bad"], dH=dH, dW=dW, Z=Z, dZ=dZ,
                lse=r["lse"], row_loss=r["row_loss"], state=r["state"], scale=r["scale"])


# --------------------------------------------------------------------- RMSNorm
# "Fast RMS LayerNorm Triton Kernels" (fms-acceleration-foak 0.7.4 page, list of
# fused operations and kernels; the patch rule there swaps the model's RMSNorm
# module for fast_rms_layernorm).  The pages print no formula; the reading taken
# is the RMSNorm of the Llama / Mistral / Granite decoders they patch:
#     r_i = 1 / sqrt(mean_j x_ij^2 + eps),   y_ij = x_ij * r_i * gamma_j.

def rmsnorm(X: np.ndarray, gamma: np.ndarray, eps: float):
    """y = x * r * gamma per row, r = 1 / sqrt(mean(x^2) + eps); float64.  Returns (Y, r)."""
    Xd, gd = _to_f64(X), _to_f64(gamma)
    ms = np.mean(Xd * Xd, axis=1)
    r = 1.0 / np.sqrt(ms + eps)
    return Xd * r[:, None] * gd[None, :], r


def rmsnorm_backward(dY: np.ndarray, X: np.ndarray, gamma: np.ndarray, eps: float):
    """Gradients of sum(dY * rmsnorm(X)) w.r.t. X and gamma, float64.

    With xh = x * r and u = gamma * dy (per row):  dx = r * (u - xh * mean(xh * u)),
    dgamma = sum over rows of dy * xh.
    """
    Xd, gd, dYd = _to_f64(X), _to_f64(gamma), _to_f64(dY)
    _, r = rmsnorm(Xd, gd, eps)
    xh = Xd * r[:, None]
    u = dYd * gd[None, :]
    dX = r[:, None] * (u - xh * np.mean(xh * u, axis=1)[:, None])
    dgamma = np.sum(dYd * xh, axis=0)
    return dX, dgamma


def rmsnorm_linear_ce(X: np.ndarray, gamma: np.ndarray, W: np.ndarray, labels: np.ndarray, *, eps: float,
                      ignore_index: int = -100, g: float = 1.0, denom: float = 0.0, threads: int | None = None,
                      round_h=None):
    """Final norm -> LM head -> cross-entropy: H = rmsnorm(X), then ``linear_ce`` on H,
    then dX, dgamma through the norm; float64 throughout.

    ``round_h`` (optional) maps H to the values the device stores (e.g. bf16 rounding)
    before the linear layer; the gradient then flows through the unrounded norm, the
    straight-through reading of a rounded activation.
    """
    H, r = rmsnorm(X, gamma, eps)
    Hq = round_h(H) if round_h is not None else H
    res = linear_ce(Hq, W, labels, ignore_index=ignore_index, g=g, denom=denom, threads=threads)
    dX, dgamma = rmsnorm_backward(res["dH"], X, gamma, eps)
    res.update(H=H, rstd=r, dX=dX, dgamma=dgamma)
    return res


# --------------------------------------------------------------------- RoPE
# "Fast RoPE Triton Kernels" (fms-acceleration-foak 0.7.4 page, list of fused
# operations and kernels; its Known Issues, and "Notes on FastKernels" of
# fms-hf-tuning PR #280, say the FOAK version takes no position_ids).  The pages
# print no formula; the reading taken is the rotary embedding of the Llama /
# Mistral decoders in the "rotate half" pairing: for head dimension d and
# i < d/2, element i pairs with element i + d/2 and the pair turns by
#     theta(p, i) = p * base^(-2i/d),   p = the token's position id.

def rope_angles(positions: np.ndarray, d: int, base: float) -> np.ndarray:
    """theta[t, i] = positions[t] * base^(-2i/d), float64, shape (T, d/2)."""
    i = np.arange(d // 2, dtype=np.float64)
    inv_freq = np.power(float(base), -2.0 * i / d)
    return np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]


def rope(X: np.ndarray, positions: np.ndarray, base: float, *, inverse: bool = False) -> np.ndarray:
    """Rotate every head vector of X (T x H x d, any float dtype or bf16 bits) by its
    token's angles; ``inverse`` turns by -theta (the backward: the rotation is
    orthogonal, so the gradient of sum(G * rope(X)) is rope(G, inverse=True))."""
    Xd = _to_f64(X)
    T, H, d = Xd.shape
    th = rope_angles(positions, d, base)
    c, s = np.cos(th)[:, None, :], np.sin(th)[:, None, :]
    if inverse:
        s = -s
    lo, hi = Xd[..., : d // 2], Xd[..., d // 2:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)
