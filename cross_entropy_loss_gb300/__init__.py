"""GB300 (sm_103a) fused cross-entropy -- Python binding of ``libfoak_ce.so``.

The library is the FastCrossEntropyLoss of the fms-acceleration FOAK plugin
(fms-acceleration PR #79, Description item 4) rebuilt as hand-written CUDA for
sm_103a behind a C ABI (``include/foak_ce.h``).  This module only marshals
arguments: it takes torch tensors for device memory and the current stream,
passes their pointers through ctypes, and raises on a non-zero status.  Every
step of the computation runs in the library's kernels; there is no CPU or
PyTorch fallback -- importing fails loudly when the library is missing.

Build it with ``python -c "import __graft_entry__ as g; g.build()"`` (or
``cross_entropy_loss_gb300._build.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

LIB_PATH = _build.LIB

FOAK_OK = 0
FOAK_ERR_INVALID_ARG = 1
FOAK_ERR_UNSUPPORTED = 2
FOAK_ERR_LABEL_RANGE = 3
FOAK_ERR_WORKSPACE = 4
FOAK_ERR_CUDA = 5
FOAK_ERR_TIMEOUT = 6
FOAK_F32 = 0
FOAK_BF16 = 1
FOAK_ERRBIT_LABEL_RANGE = 1
FOAK_ERRBIT_TIMEOUT = 2

# C entry points and their ctypes signatures (restype, argtypes).
_vp, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "foak_status_string": (ctypes.c_char_p, [_i32]),
    "foak_abi_version": (_i32, []),
    "foak_ce_max_vocab": (_i64, [_i32]),
    "foak_ce_workspace_size": (_sz, [_i64]),
    "foak_ce_forward": (_i32, [_vp, _i32, _i64, _vp, _i64, _i64, _i64, _f32, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                               _vp]),
    "foak_ce_backward": (_i32, [_vp, _vp, _i32, _i64, _vp, _i64, _i64, _i64, _vp, _vp, _f32, _vp, _vp]),
    "foak_rmsnorm_forward": (_i32, [_vp, _i32, _i64, _vp, _i64, _i64, _f32, _vp, _i64, _vp, _vp]),
    "foak_rmsnorm_workspace_size": (_sz, [_i64]),
    "foak_rmsnorm_backward": (_i32, [_vp, _i64, _vp, _i64, _vp, _vp, _i32, _i64, _i64, _vp, _i64, _vp, _vp, _sz,
                                     _vp]),
    "foak_rmsnorm_linear_ce_workspace_size": (_sz, [_i64, _i64, _i64, _i64]),
    "foak_rmsnorm_linear_ce_chunked": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _f32, _f32, _f32,
                                              _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "foak_rope_cache_size": (_sz, [_i64, _i64]),
    "foak_rope_build_cache": (_i32, [ctypes.c_double, _i64, _i64, _vp, _sz, _vp]),
    "foak_rope_apply": (_i32, [_vp, _i32, _i64, _i64, _i64, _i64, _vp, _vp, _i64, _i32, _vp, _vp]),
    "foak_rope_apply_qk": (_i32, [_vp, _i64, _i64, _vp, _i64, _i64, _i32, _i64, _i64, _vp, _vp, _i64, _i32, _vp,
                                  _vp]),
    "foak_ce_host_workspace_size": (_sz, [_i64]),
    "foak_ce_fwd_bwd_host": (_i32, [_vp, _i32, _i64, _vp, _i64, _i64, _i64, _f32, _f32, _vp, _vp, _vp, _vp, _vp, _vp,
                                    _sz, _vp]),
    "foak_ce_fwd_bwd": (_i32, [_vp, _i32, _i64, _vp, _i64, _i64, _i64, _f32, _f32, _vp, _vp, _vp, _vp, _vp, _sz,
                               _vp]),
    "foak_ce_count_valid": (_i32, [_vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "foak_ce_fwd_bwd_devdenom": (_i32, [_vp, _i32, _i64, _vp, _i64, _i64, _i64, _f32, _vp, _vp, _vp, _vp, _vp, _vp,
                                        _sz, _vp]),
    "foak_ce_fwd_bwd_noalloc": (_i32, [_vp, _i32, _i64, _vp, _i64, _i64, _i64, _f32, _f32, _vp, _vp, _vp, _vp,
                                       _vp]),
    "foak_gemm_bf16": (_i32, [_vp, _i64, _i32, _vp, _i64, _i32, _i64, _i64, _i64, _vp, _i64, _i32, _vp, _vp]),
    "foak_gemm_bf16_group": (_i32, [_vp, _i32, _vp, _vp]),
    "foak_test_gemm_group_schedule": (_i32, [_vp, _i32, _i32, _vp, _vp, _i32]),
    "foak_linear_ce_workspace_size": (_sz, [_i64, _i64, _i64, _i64]),
    "foak_linear_ce_chunked": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _f32, _f32, _vp, _vp, _vp, _vp,
                                      _vp, _vp, _sz, _vp]),
    "foak_test_fail_next_launches": (None, [_i32]),
    "foak_test_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "foak_test_skip_row_load": (None, [_i64]),
    "foak_test_set_row_path": (None, [_i32]),
}


class FoakError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"cross_entropy_loss_gb300: {LIB_PATH} is missing; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()'). There is no fallback path.")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.foak_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != FOAK_OK:
        raise FoakError(status, where)


def foak_ce_workspace_size(N: int) -> int:
    return int(lib.foak_ce_workspace_size(int(N)))


def foak_ce_max_vocab(dtype: int) -> int:
    return int(lib.foak_ce_max_vocab(int(dtype)))


# --------------------------------------------------------------------- torch glue
import torch  # noqa: E402  (device memory and streams only)

_DT = {torch.bfloat16: FOAK_BF16, torch.float32: FOAK_F32}
_ws_lock = threading.Lock()
_ws_cache: dict = {}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device, stream):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _logits_args(logits):
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be a 2-D tensor with unit column stride (N x V, row stride ld)")
    if logits.dtype not in _DT:
        raise TypeError("logits must be bfloat16 or float32")
    if not logits.is_cuda:
        raise ValueError("logits must be on a CUDA device")
    N, V = logits.shape
    ld = logits.stride(0) if N > 1 else max(V, logits.stride(0))
    return N, V, ld, _DT[logits.dtype]


def _labels_arg(labels, N, device):
    if labels.dtype != torch.int64 or labels.dim() != 1 or labels.numel() != N or not labels.is_contiguous():
        raise ValueError("labels must be a contiguous int64 vector of length N")
    if labels.device != device:
        raise ValueError("labels must live on the logits' device")
    return labels


def workspace(N: int, device) -> torch.Tensor:
    """A zero-filled, reusable workspace of at least foak_ce_workspace_size(N) bytes.

    Calls leave it zeroed again, so the cached buffer serves every stream-ordered
    call on its device.  Calls on different streams should pass their own buffer.
    """
    need = foak_ce_workspace_size(N)
    dev = torch.device(device)
    with _ws_lock:
        ws = _ws_cache.get(dev)
        if ws is None or ws.numel() < need:
            ws = torch.zeros(max(need, 4096), dtype=torch.uint8, device=dev)
            _ws_cache[dev] = ws
    return ws


def foak_ce_forward(logits, labels, *, ignore_index: int = -100, denom: float = 0.0, want_lse: bool = True,
                    want_row_loss: bool = False, workspace_tensor=None, stream=None):
    """Mean CE loss over non-ignored rows.  Returns dict(loss, lse, row_loss, n_valid, err)."""
    N, V, ld, dt = _logits_args(logits)
    dev = logits.device
    labels = _labels_arg(labels, N, dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    n_valid = torch.empty(1, dtype=torch.int32, device=dev)
    err = torch.empty(1, dtype=torch.int32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev) if want_lse else None
    row_loss = torch.empty(N, dtype=torch.float32, device=dev) if want_row_loss else None
    ws = workspace(N, dev) if workspace_tensor is None else workspace_tensor
    st = lib.foak_ce_forward(_ptr(logits), dt, ld, _ptr(labels), N, V, int(ignore_index), float(denom), _ptr(loss),
                             _ptr(lse), _ptr(row_loss), _ptr(n_valid), _ptr(err), _ptr(ws), ws.numel(),
                             _stream(dev, stream))
    _check(st, "foak_ce_forward")
    return dict(loss=loss, lse=lse, row_loss=row_loss, n_valid=n_valid, err=err)


def foak_ce_backward(logits, labels, lse, grad_out=None, *, dlogits=None, ignore_index: int = -100,
                     denom: float = 0.0, stream=None):
    """dlogits = (softmax - onehot) * g / D.  Pass ``dlogits=logits`` to overwrite in place."""
    N, V, ld, dt = _logits_args(logits)
    dev = logits.device
    labels = _labels_arg(labels, N, dev)
    if dlogits is None:
        # same row stride and the same offset modulo 16 bytes as logits (the kernels share row geometry)
        es = logits.element_size()
        shift = (logits.data_ptr() % 16) // es
        n = ((N - 1) * ld + V + shift) if N > 0 else 1
        base = torch.empty(n, dtype=logits.dtype, device=dev)
        dlogits = base.as_strided((N, V), (ld, 1), storage_offset=shift)
    if dlogits.shape != logits.shape or dlogits.stride() != logits.stride() or dlogits.dtype != logits.dtype:
        raise ValueError("dlogits must match logits in shape, strides and dtype")
    if lse.dtype != torch.float32 or lse.numel() != N or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 vector of length N")
    if grad_out is not None and (grad_out.dtype != torch.float32 or grad_out.numel() != 1):
        raise ValueError("grad_out must be a float32 scalar tensor")
    err = torch.empty(1, dtype=torch.int32, device=dev)
    st = lib.foak_ce_backward(_ptr(dlogits), _ptr(logits), dt, ld, _ptr(labels), N, V, int(ignore_index), _ptr(lse),
                              _ptr(grad_out), float(denom), _ptr(err), _stream(dev, stream))
    _check(st, "foak_ce_backward")
    return dlogits, err


def foak_ce_fwd_bwd(logits, labels, *, g: float = 1.0, ignore_index: int = -100, denom: float = 0.0,
                    want_lse: bool = False, workspace_tensor=None, stream=None):
    """Fused forward + backward in place: ``logits`` is overwritten by dlogits.

    Returns dict(loss, n_valid, err, lse).
    """
    N, V, ld, dt = _logits_args(logits)
    dev = logits.device
    labels = _labels_arg(labels, N, dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    n_valid = torch.empty(1, dtype=torch.int32, device=dev)
    err = torch.empty(1, dtype=torch.int32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev) if want_lse else None
    ws = workspace(N, dev) if workspace_tensor is None else workspace_tensor
    st = lib.foak_ce_fwd_bwd(_ptr(logits), dt, ld, _ptr(labels), N, V, int(ignore_index), float(g), float(denom),
                             _ptr(loss), _ptr(lse), _ptr(n_valid), _ptr(err), _ptr(ws), ws.numel(),
                             _stream(dev, stream))
    _check(st, "foak_ce_fwd_bwd")
    return dict(loss=loss, n_valid=n_valid, err=err, lse=lse)


def foak_ce_count_valid(labels, V: int, *, ignore_index: int = -100, out=None, err=None, stream=None):
    """Number of labels in [0, V) (not ignore_index), as an int64 device tensor of one element
    (``out`` if given), e.g. this rank's term of a data-parallel all-reduced denominator."""
    if labels.dtype != torch.int64 or labels.dim() != 1 or not labels.is_contiguous():
        raise ValueError("labels must be a contiguous int64 vector")
    dev = labels.device
    if out is None:
        out = torch.empty(1, dtype=torch.int64, device=dev)
    if out.dtype != torch.int64 or out.numel() != 1:
        raise ValueError("out must be a one-element int64 tensor")
    st = lib.foak_ce_count_valid(_ptr(labels), labels.numel(), int(V), int(ignore_index), _ptr(out), _ptr(err),
                                 _stream(dev, stream))
    _check(st, "foak_ce_count_valid")
    return out


def foak_ce_fwd_bwd_devdenom(logits, labels, denom_count, *, g: float = 1.0, ignore_index: int = -100,
                             want_lse: bool = False, workspace_tensor=None, stream=None):
    """foak_ce_fwd_bwd dividing by the int64 count in device memory ``denom_count`` (read when the
    kernel runs, e.g. after an all-reduce on the same stream).  ``loss`` is this call's share
    sum(l_i) / D.  Returns dict(loss, n_valid, err, lse)."""
    N, V, ld, dt = _logits_args(logits)
    dev = logits.device
    labels = _labels_arg(labels, N, dev)
    if denom_count.dtype != torch.int64 or denom_count.numel() != 1 or denom_count.device != dev:
        raise ValueError("denom_count must be a one-element int64 tensor on the logits' device")
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    n_valid = torch.empty(1, dtype=torch.int32, device=dev)
    err = torch.empty(1, dtype=torch.int32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev) if want_lse else None
    ws = workspace(N, dev) if workspace_tensor is None else workspace_tensor
    st = lib.foak_ce_fwd_bwd_devdenom(_ptr(logits), dt, ld, _ptr(labels), N, V, int(ignore_index), float(g),
                                      _ptr(denom_count), _ptr(loss), _ptr(lse), _ptr(n_valid), _ptr(err), _ptr(ws),
                                      ws.numel(), _stream(dev, stream))
    _check(st, "foak_ce_fwd_bwd_devdenom")
    return dict(loss=loss, n_valid=n_valid, err=err, lse=lse)


def foak_ce_host_workspace_size(N: int) -> int:
    return int(lib.foak_ce_host_workspace_size(int(N)))


def foak_ce_fwd_bwd_host(host_logits, host_labels, dev_logits, dev_labels, *, g: float = 1.0,
                         ignore_index: int = -100, denom: float = 0.0, workspace_tensor=None, out=None, stream=None):
    """Fused forward + backward on HOST logits: the call copies labels and logits to
    ``dev_logits`` / ``dev_labels`` in row chunks and sweeps each chunk as it lands;
    ``dev_logits`` ends holding dlogits.

    ``host_logits`` is a CPU bf16/fp32 tensor (pinned for a full-speed copy) with
    the shape and row stride of ``dev_logits``; ``host_labels`` a CPU int64 tensor.
    Returns dict(loss, n_valid, err) of pinned host tensors (pass ``out`` to reuse
    them), valid once the stream has been synchronised.
    """
    N, V, ld, dt = _logits_args(dev_logits)
    dev = dev_logits.device
    if host_logits.is_cuda or host_logits.dtype != dev_logits.dtype or host_logits.dim() != 2:
        raise ValueError("host_logits must be a CPU tensor of the device logits' dtype")
    if tuple(host_logits.shape) != (N, V) or host_logits.stride(1) != 1 or (N > 1 and host_logits.stride(0) != ld):
        raise ValueError("host_logits must have the shape and row stride of dev_logits")
    if host_labels.is_cuda or host_labels.dtype != torch.int64 or host_labels.numel() != N:
        raise ValueError("host_labels must be a CPU int64 tensor of N labels")
    if not host_labels.is_contiguous():
        raise ValueError("host_labels must be contiguous")
    dev_labels = _labels_arg(dev_labels, N, dev)
    if out is None:
        out = dict(loss=torch.empty(1, dtype=torch.float32).pin_memory(),
                   n_valid=torch.empty(1, dtype=torch.int32).pin_memory(),
                   err=torch.empty(1, dtype=torch.int32).pin_memory())
    need = foak_ce_host_workspace_size(N)
    ws = workspace(N + 64, dev) if workspace_tensor is None else workspace_tensor  # + 256 bytes of results
    if ws.numel() < need:
        raise ValueError("workspace_tensor smaller than foak_ce_host_workspace_size(N)")
    st = lib.foak_ce_fwd_bwd_host(_ptr(host_logits), dt, ld, _ptr(host_labels), N, V, int(ignore_index), float(g),
                                  float(denom), _ptr(dev_logits), _ptr(dev_labels), _ptr(out["loss"]),
                                  _ptr(out["n_valid"]), _ptr(out["err"]), _ptr(ws), ws.numel(), _stream(dev, stream))
    _check(st, "foak_ce_fwd_bwd_host")
    return out


FOAK_CE_NOALLOC_MAX_ROWS = 262144


def foak_ce_fwd_bwd_noalloc(logits, labels, *, g: float = 1.0, ignore_index: int = -100, denom: float = 0.0,
                            want_lse: bool = False, stream=None):
    """Fused forward + backward in place, for callers that may not allocate device memory.

    Same result as :func:`foak_ce_fwd_bwd`, but the library takes its scratch from a
    fixed array in its own device image instead of a workspace, so no workspace
    buffer is needed (this wrapper still allocates its small output tensors with
    torch; a C caller passes its own).  N is limited to FOAK_CE_NOALLOC_MAX_ROWS,
    and calls that overlap on the GPU race on the shared scratch.
    """
    N, V, ld, dt = _logits_args(logits)
    dev = logits.device
    labels = _labels_arg(labels, N, dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    n_valid = torch.empty(1, dtype=torch.int32, device=dev)
    err = torch.empty(1, dtype=torch.int32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev) if want_lse else None
    # the library uses the scratch array of the CURRENT device: make it the logits' device
    with torch.cuda.device(dev):
        st = lib.foak_ce_fwd_bwd_noalloc(_ptr(logits), dt, ld, _ptr(labels), N, V, int(ignore_index), float(g),
                                         float(denom), _ptr(loss), _ptr(lse), _ptr(n_valid), _ptr(err),
                                         _stream(dev, stream))
    _check(st, "foak_ce_fwd_bwd_noalloc")
    return dict(loss=loss, n_valid=n_valid, err=err, lse=lse)


FOAK_GEMM_BF16, FOAK_GEMM_F32, FOAK_GEMM_F32_ACC = 0, 1, 2


def foak_gemm_bf16(a, b, out, *, a_mn_major: bool = False, b_mn_major: bool = False, mode: int = FOAK_GEMM_BF16,
                   M: int | None = None, N: int | None = None, K: int | None = None, err=None, stream=None):
    """out (+)= A @ B^T on the tensor cores.  a, b: 2-D bf16 tensors with unit column stride.

    a is [M][K] (or [K][M] with a_mn_major), b is [N][K] (or [K][N] with b_mn_major);
    out is [M][N] with unit column stride, bf16 for FOAK_GEMM_BF16 else fp32.
    """
    for t in (a, b, out):
        if t.dim() != 2 or t.stride(1) != 1 or not t.is_cuda:
            raise ValueError("operands must be 2-D CUDA tensors with unit column stride")
    if a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16:
        raise TypeError("a and b must be bfloat16")
    M = (a.shape[1] if a_mn_major else a.shape[0]) if M is None else M
    K = (a.shape[0] if a_mn_major else a.shape[1]) if K is None else K
    N = (b.shape[1] if b_mn_major else b.shape[0]) if N is None else N
    st = lib.foak_gemm_bf16(_ptr(a), a.stride(0), int(a_mn_major), _ptr(b), b.stride(0), int(b_mn_major), M, N, K,
                            _ptr(out), out.stride(0), int(mode), _ptr(err), _stream(out.device, stream))
    _check(st, "foak_gemm_bf16")
    return out


class _GemmProblem(ctypes.Structure):
    """foak_gemm_problem of the C header."""
    _fields_ = [("a", ctypes.c_void_p), ("lda", ctypes.c_int64), ("a_mn_major", ctypes.c_int32),
                ("b", ctypes.c_void_p), ("ldb", ctypes.c_int64), ("b_mn_major", ctypes.c_int32),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("out", ctypes.c_void_p), ("ldo", ctypes.c_int64), ("out_mode", ctypes.c_int32)]


FOAK_GEMM_GROUP_MAX = 3


def foak_gemm_bf16_group(problems, *, err=None, stream=None):
    """Several independent products out (+)= A @ B^T in one persistent launch.

    problems: sequence of dicts with keys a, b, out and optionally a_mn_major, b_mn_major,
    mode, M, N, K -- each as for foak_gemm_bf16.  No product may write what another reads.
    """
    if len(problems) > FOAK_GEMM_GROUP_MAX:
        raise ValueError(f"at most {FOAK_GEMM_GROUP_MAX} products")
    arr = (_GemmProblem * max(1, len(problems)))()
    dev = None
    for i, q in enumerate(problems):
        a, b, out = q["a"], q["b"], q["out"]
        for t in (a, b, out):
            if t.dim() != 2 or t.stride(1) != 1 or not t.is_cuda:
                raise ValueError("operands must be 2-D CUDA tensors with unit column stride")
        if a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16:
            raise TypeError("a and b must be bfloat16")
        amn, bmn = bool(q.get("a_mn_major", False)), bool(q.get("b_mn_major", False))
        M = q.get("M", a.shape[1] if amn else a.shape[0])
        K = q.get("K", a.shape[0] if amn else a.shape[1])
        N = q.get("N", b.shape[1] if bmn else b.shape[0])
        arr[i] = _GemmProblem(_ptr(a), a.stride(0), int(amn), _ptr(b), b.stride(0), int(bmn), M, N, K, _ptr(out),
                              out.stride(0), int(q.get("mode", FOAK_GEMM_BF16)))
        dev = out.device
    st = lib.foak_gemm_bf16_group(ctypes.cast(arr, ctypes.c_void_p), len(problems), _ptr(err),
                                  _stream(dev, stream) if dev is not None else None)
    _check(st, "foak_gemm_bf16_group")


def foak_linear_ce_workspace_size(N: int, V: int, D: int, chunk: int) -> int:
    return int(lib.foak_linear_ce_workspace_size(int(N), int(V), int(D), int(chunk)))


_lin_ws: dict = {}


def foak_linear_ce_chunked(H, W, labels, *, chunk: int = 1024, g: float = 1.0, ignore_index: int = -100,
                           denom: float = 0.0, dH=None, dW=None, workspace_tensor=None, stream=None):
    """Loss, dH and dW of CE(H W^T) in chunks of rows on the tensor cores.

    H: bf16 [N][D], W: bf16 [V][D] (contiguous).  Returns dict(loss, dH, dW, n_valid, err);
    dH is bf16 [N][D], dW fp32 [V][D].
    """
    if H.dtype != torch.bfloat16 or W.dtype != torch.bfloat16 or not H.is_contiguous() or not W.is_contiguous():
        raise ValueError("H and W must be contiguous bfloat16 tensors")
    N, D = H.shape
    V, D2 = W.shape
    if D2 != D:
        raise ValueError("H and W disagree on the hidden size")
    dev = H.device
    labels = _labels_arg(labels, N, dev)
    dH = torch.empty(N, D, dtype=torch.bfloat16, device=dev) if dH is None else dH
    dW = torch.empty(V, D, dtype=torch.float32, device=dev) if dW is None else dW
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    n_valid = torch.empty(1, dtype=torch.int32, device=dev)
    err = torch.empty(1, dtype=torch.int32, device=dev)
    need = foak_linear_ce_workspace_size(N, V, D, chunk)
    ws = workspace_tensor
    if ws is None:
        with _ws_lock:
            ws = _lin_ws.get(dev)
            if ws is None or ws.numel() < need:
                ws = torch.zeros(need, dtype=torch.uint8, device=dev)
                _lin_ws[dev] = ws
    st = lib.foak_linear_ce_chunked(_ptr(H), _ptr(W), _ptr(labels), N, V, D, int(ignore_index), int(chunk), float(g),
                                    float(denom), _ptr(loss), _ptr(dH), _ptr(dW), _ptr(n_valid), _ptr(err), _ptr(ws),
                                    ws.numel(), _stream(dev, stream))
    _check(st, "foak_linear_ce_chunked")
    return dict(loss=loss, dH=dH, dW=dW, n_valid=n_valid, err=err)


# --------------------------------------------------------------------- RMSNorm
_norm_ws: dict = {}


def _rows_arg(t, name):
    if t.dim() != 2 or t.stride(1) != 1 or t.dtype not in _DT or not t.is_cuda:
        raise ValueError(f"{name} must be a 2-D bfloat16/float32 CUDA tensor with unit column stride")
    return t.shape[0], t.shape[1], (t.stride(0) if t.shape[0] > 1 else t.shape[1])


def foak_rmsnorm_forward(X, gamma, *, eps: float = 1e-5, Y=None, want_rstd: bool = True, stream=None):
    """Y = X / sqrt(mean(X^2) + eps) * gamma per row (fp32 arithmetic, one rounding).

    Returns (Y, rstd); rstd (float32 [N]) is None unless ``want_rstd``.
    """
    N, D, ldx = _rows_arg(X, "X")
    if gamma.dtype != X.dtype or gamma.numel() != D or not gamma.is_contiguous():
        raise ValueError("gamma must be a contiguous vector of D elements in X's dtype")
    Y = torch.empty_like(X) if Y is None else Y
    _, _, ldy = _rows_arg(Y, "Y")
    rstd = torch.empty(N, dtype=torch.float32, device=X.device) if want_rstd else None
    st = lib.foak_rmsnorm_forward(_ptr(X), _DT[X.dtype], ldx, _ptr(gamma), N, D, float(eps), _ptr(Y), ldy, _ptr(rstd),
                                  _stream(X.device, stream))
    _check(st, "foak_rmsnorm_forward")
    return Y, rstd


def foak_rmsnorm_backward(dY, X, gamma, rstd, *, dX=None, want_dgamma: bool = True, stream=None):
    """dX (X's dtype) and dgamma (float32 [D], or None) of sum(dY * rmsnorm(X))."""
    N, D, lddy = _rows_arg(dY, "dY")
    _, _, ldx = _rows_arg(X, "X")
    dX = torch.empty_like(X) if dX is None else dX
    _, _, lddx = _rows_arg(dX, "dX")
    dev = X.device
    dgamma = torch.empty(D, dtype=torch.float32, device=dev) if want_dgamma else None
    need = int(lib.foak_rmsnorm_workspace_size(D))
    with _ws_lock:
        ws = _norm_ws.get(dev)
        if ws is None or ws.numel() < need:
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
            _norm_ws[dev] = ws
    st = lib.foak_rmsnorm_backward(_ptr(dY), lddy, _ptr(X), ldx, _ptr(gamma), _ptr(rstd), _DT[X.dtype], N, D, _ptr(dX),
                                   lddx, _ptr(dgamma), _ptr(ws), ws.numel(), _stream(dev, stream))
    _check(st, "foak_rmsnorm_backward")
    return dX, dgamma


def foak_rmsnorm_linear_ce_chunked(X, gamma, W, labels, *, eps: float = 1e-5, chunk: int = 1024, g: float = 1.0,
                                   ignore_index: int = -100, denom: float = 0.0, dX=None, dW=None,
                                   workspace_tensor=None, stream=None):
    """Final norm -> LM head -> CE: loss, dX, dgamma, dW of CE(rmsnorm(X, gamma) W^T).

    X: bf16 [N][D], gamma: bf16 [D], W: bf16 [V][D] (contiguous).  Returns
    dict(loss, dX, dgamma, dW, n_valid, err); dX bf16, dgamma and dW float32.
    """
    for t, n in ((X, "X"), (gamma, "gamma"), (W, "W")):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous bfloat16 tensor")
    N, D = X.shape
    V = W.shape[0]
    if W.shape[1] != D or gamma.numel() != D:
        raise ValueError("X, gamma and W disagree on the hidden size")
    dev = X.device
    labels = _labels_arg(labels, N, dev)
    dX = torch.empty_like(X) if dX is None else dX
    dW = torch.empty(V, D, dtype=torch.float32, device=dev) if dW is None else dW
    dgamma = torch.empty(D, dtype=torch.float32, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    n_valid = torch.empty(1, dtype=torch.int32, device=dev)
    err = torch.empty(1, dtype=torch.int32, device=dev)
    need = int(lib.foak_rmsnorm_linear_ce_workspace_size(N, V, D, chunk))
    ws = workspace_tensor
    if ws is None:
        with _ws_lock:
            key = ("norm_lin", dev)
            ws = _norm_ws.get(key)
            if ws is None or ws.numel() < need:
                ws = torch.zeros(need, dtype=torch.uint8, device=dev)  # zero-filled before first use
                _norm_ws[key] = ws
    st = lib.foak_rmsnorm_linear_ce_chunked(_ptr(X), _ptr(gamma), _ptr(W), _ptr(labels), N, V, D, int(ignore_index),
                                            int(chunk), float(eps), float(g), float(denom), _ptr(loss), _ptr(dX),
                                            _ptr(dgamma), _ptr(dW), _ptr(n_valid), _ptr(err), _ptr(ws), ws.numel(),
                                            _stream(dev, stream))
    _check(st, "foak_rmsnorm_linear_ce_chunked")
    return dict(loss=loss, dX=dX, dgamma=dgamma, dW=dW, n_valid=n_valid, err=err)


# --------------------------------------------------------------------- RoPE
def foak_rope_cache(max_pos: int, d: int, base: float = 10000.0, device="cuda", stream=None):
    """The cos/sin table for positions [0, max_pos) and head dimension d (uint8 device tensor)."""
    need = int(lib.foak_rope_cache_size(int(max_pos), int(d)))
    if need == 0:
        raise ValueError("unsupported max_pos / d (d must be a multiple of 16)")
    dev = torch.device(device)
    cache = torch.empty(need, dtype=torch.uint8, device=dev)
    st = lib.foak_rope_build_cache(float(base), int(d), int(max_pos), _ptr(cache), need, _stream(dev, stream))
    _check(st, "foak_rope_build_cache")
    cache.max_pos, cache.head_dim = int(max_pos), int(d)
    return cache


def foak_rope_apply(x, positions, cache, *, inverse: bool = False, stream=None):
    """Rotate ``x`` (T x H x d bf16/fp32 CUDA view, heads contiguous) in place by the
    angles of ``positions`` (int64 [T]); returns the device error word."""
    if x.dim() != 3 or x.stride(2) != 1 or x.stride(1) != x.shape[2] or x.dtype not in _DT or not x.is_cuda:
        raise ValueError("x must be a T x H x d CUDA view with contiguous heads")
    T, H, d = x.shape
    if d != cache.head_dim:
        raise ValueError("cache built for another head dimension")
    if positions.dtype != torch.int64 or positions.numel() != T or not positions.is_contiguous():
        raise ValueError("positions must be a contiguous int64 vector of length T")
    ldt = x.stride(0) if T > 1 else H * d
    err = torch.empty(1, dtype=torch.int32, device=x.device)
    st = lib.foak_rope_apply(_ptr(x), _DT[x.dtype], T, H, ldt, d, _ptr(positions), _ptr(cache), cache.max_pos,
                             1 if inverse else 0, _ptr(err), _stream(x.device, stream))
    _check(st, "foak_rope_apply")
    return err


def foak_rope_apply_qk(q, k, positions, cache, *, inverse: bool = False, stream=None):
    """Rotate Q (T x Hq x d) and K (T x Hk x d) in place in one launch; returns the error word."""
    views = []
    for x in (q, k):
        if x.dim() != 3 or x.stride(2) != 1 or x.stride(1) != x.shape[2] or x.dtype not in _DT or not x.is_cuda:
            raise ValueError("q and k must be T x H x d CUDA views with contiguous heads")
        T, H, d = x.shape
        views.append((H, x.stride(0) if T > 1 else H * d))
    if q.shape[0] != k.shape[0] or q.shape[2] != k.shape[2] or q.dtype != k.dtype:
        raise ValueError("q and k disagree on tokens, head dimension or dtype")
    T, _, d = q.shape
    if d != cache.head_dim:
        raise ValueError("cache built for another head dimension")
    if positions.dtype != torch.int64 or positions.numel() != T or not positions.is_contiguous():
        raise ValueError("positions must be a contiguous int64 vector of length T")
    err = torch.empty(1, dtype=torch.int32, device=q.device)
    (hq, ldq), (hk, ldk) = views
    st = lib.foak_rope_apply_qk(_ptr(q), hq, ldq, _ptr(k), hk, ldk, _DT[q.dtype], T, d, _ptr(positions), _ptr(cache),
                                cache.max_pos, 1 if inverse else 0, _ptr(err), _stream(q.device, stream))
    _check(st, "foak_rope_apply_qk")
    return err
