"""Seeded synthetic workloads for the fused cross-entropy path.

This module only produces inputs (logits, labels, hidden states, weights); it
holds none of the loss's arithmetic, so both the CUDA path's tests/bench and the
CPU oracle can consume the very same bytes.  Numbers come from the counter-based
SplitMix64 generator in ``gen.c`` (Steele, Lea and Flood, OOPSLA 2014) and normals
from Box-Muller; see that file's header.

Workload recipes (shapes and value distributions follow the loss workloads the
FOAK pages benchmark: Mistral-7B full fine-tuning at batch 4, padding-free
packed batches, Llama-3's 128256-token vocabulary, and the chunked linear+CE
head), each with a fixed seed ``20261200 + k``:

* ``tiny``        N=64, V=1000, fp32 ~N(0,1), labels U[0,V), exactly 6 rows -100
* ``mistral``     N=4096 (4 x 1024), V=32000, bf16 ~N(0,2^2), last token of each
                  sequence -100 (rows 1023, 2047, 3071, 4095)
* ``packed``      8192 tokens of sequences with lengths U{64..1024} (last one
                  truncated), V=32000, bf16 ~N(0,2^2); per sequence the first
                  floor(u*L) tokens (u ~ U[0.3,0.6], at least one) are -100
* ``llama3``      N=8192, V=128256, bf16 or fp32 ~N(0,3^2), each entry replaced
                  with probability 1e-4 by U[20,30); row 4097 all 3.0 with a
                  valid label; exactly 410 other rows -100
* ``chunked``     H 8192x4096 bf16 ~N(0,1), W 32000x4096 bf16 ~N(0,0.02^2),
                  labels U[0,32000) with exactly 819 rows -100, chunk 1024
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libwlgen.so")
_lock = threading.Lock()
_lib = None

IGNORE_INDEX = -100
F32, BF16 = 0, 1

# stream ids (any distinct constants)
S_LOGITS, S_SPIKE, S_LABELS, S_IGNORE, S_SEQLEN, S_PROMPT, S_H, S_W, S_X, S_GAMMA = range(1, 11)


def build_lib(force: bool = False) -> str:
    """Compile gen.c with the host gcc (no architecture-specific flags)."""
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
            u64, i64, dbl, vp, i32 = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
                                      ctypes.c_void_p, ctypes.c_int)
            lib.wl_stream_key.restype = u64
            lib.wl_stream_key.argtypes = [u64, u64]
            lib.wl_u64.argtypes = [u64, u64, i64, vp]
            lib.wl_uniform.argtypes = [u64, u64, i64, vp]
            lib.wl_normal.argtypes = [u64, u64, i64, dbl, dbl, u64, dbl, dbl, dbl, i32, vp]
            lib.wl_normal_matrix.argtypes = [u64, i64, i64, i64, i64, dbl, dbl, u64, dbl, dbl,
                                             dbl, i32, vp]
            _lib = lib
    return _lib


def stream_key(seed: int, stream: int) -> int:
    return int(_get().wl_stream_key(seed, stream))


def u64(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    if n:
        _get().wl_u64(stream_key(seed, stream), start, n, out.ctypes.data)
    return out


def uniform(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    if n:
        _get().wl_uniform(stream_key(seed, stream), start, n, out.ctypes.data)
    return out


def _threads() -> int:
    return max(1, os.cpu_count() or 1)


def normal_matrix(rows: int, cols: int, *, seed: int, sigma: float, dtype: int, ld: int | None = None,
                  mean: float = 0.0, spike_p: float = 0.0, spike_lo: float = 0.0,
                  spike_hi: float = 0.0, stream: int = S_LOGITS, row0: int = 0,
                  out: np.ndarray | None = None) -> np.ndarray:
    """Rows [row0, row0+rows) of a seeded normal matrix (bf16 as uint16 bits, or float32).

    Element (r, c) is draw r*cols + c of the stream, so a row block can be generated
    alone and equals the same rows of the full matrix.  With ``ld > cols`` the padding
    columns are zero.
    """
    ld = cols if ld is None else ld
    npdt = np.float32 if dtype == F32 else np.uint16
    if out is None:
        out = np.zeros((rows, ld), dtype=npdt)
    assert out.shape == (rows, ld) and out.dtype == npdt and out.flags.c_contiguous
    if rows == 0 or cols == 0:
        return out
    lib = _get()
    key = stream_key(seed, stream)
    skey = stream_key(seed, S_SPIKE)
    es = out.itemsize
    base = out.ctypes.data
    nt = min(_threads(), rows)
    bounds = np.linspace(0, rows, nt + 1).astype(np.int64)

    def work(t):
        a, b = int(bounds[t]), int(bounds[t + 1])
        if b > a:
            lib.wl_normal_matrix(key, row0 + a, row0 + b, cols, ld, mean, sigma, skey, spike_p,
                                 spike_lo, spike_hi, dtype, base + a * ld * es)

    if nt == 1:
        work(0)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(work, range(nt)))
    return out


def uniform_labels(n: int, v: int, *, seed: int, stream: int = S_LABELS) -> np.ndarray:
    """Labels uniform in [0, v): floor(u * v) of 53-bit uniforms."""
    u = uniform(seed, stream, n)
    return np.minimum(np.floor(u * v).astype(np.int64), v - 1)


def pick_rows(n: int, k: int, *, seed: int, stream: int = S_IGNORE, exclude=()) -> np.ndarray:
    """Exactly k distinct rows of [0, n), none in ``exclude``: a seeded permutation's prefix."""
    keys = u64(seed, stream, n)
    order = np.argsort(keys, kind="stable")
    ex = set(int(e) for e in exclude)
    chosen = [int(r) for r in order if int(r) not in ex][:k]
    return np.array(sorted(chosen), dtype=np.int64)


SEED_BASE = 20261200


def tiny(seed: int = SEED_BASE + 1):
    n, v = 64, 1000
    x = normal_matrix(n, v, seed=seed, sigma=1.0, dtype=F32)
    y = uniform_labels(n, v, seed=seed)
    y[pick_rows(n, round(0.1 * n), seed=seed)] = IGNORE_INDEX
    return dict(name="tiny", logits=x, labels=y, N=n, V=v, dtype=F32, g=1.0, seed=seed)


def mistral(seed: int = SEED_BASE + 2, rows: int | None = None, row0: int = 0):
    """Mistral-7B-shaped loss batch (4 x 1024 tokens, V=32000, bf16 ~N(0, 2^2)).

    ``rows``/``row0`` restrict generation to a row block (the labels stay the full
    batch's labels for those rows), for bounded oracle samples.
    """
    n, v = 4096, 32000
    y = uniform_labels(n, v, seed=seed)
    y[[1023, 2047, 3071, 4095]] = IGNORE_INDEX
    rows = n - row0 if rows is None else rows
    x = normal_matrix(rows, v, seed=seed, sigma=2.0, dtype=BF16, row0=row0)
    return dict(name="mistral", logits=x, labels=y[row0:row0 + rows], N=rows, V=v, dtype=BF16,
                g=1.0, seed=seed, full_labels=y)


def packed_labels(n: int, v: int, *, seed: int):
    """Labels of a padding-free packed batch, and the sequence lengths used."""
    y = uniform_labels(n, v, seed=seed)
    lens = []
    pos, k = 0, 0
    while pos < n:
        L = 64 + int(np.floor(uniform(seed, S_SEQLEN, 1, start=k)[0] * (1024 - 64 + 1)))
        L = min(L, n - pos)
        u = 0.3 + 0.3 * uniform(seed, S_PROMPT, 1, start=k)[0]
        p = max(1, int(np.floor(u * L)))
        y[pos:pos + p] = IGNORE_INDEX
        lens.append(L)
        pos += L
        k += 1
    return y, lens


def packed(seed: int = SEED_BASE + 3, rows: int | None = None, row0: int = 0):
    n, v = 8192, 32000
    y, lens = packed_labels(n, v, seed=seed)
    rows = n - row0 if rows is None else rows
    x = normal_matrix(rows, v, seed=seed, sigma=2.0, dtype=BF16, row0=row0)
    return dict(name="packed", logits=x, labels=y[row0:row0 + rows], N=rows, V=v, dtype=BF16,
                g=1.0, seed=seed, seq_lens=lens, full_labels=y)


LLAMA3_CONST_ROW = 4097


def llama3_labels(n: int, v: int, *, seed: int):
    y = uniform_labels(n, v, seed=seed)
    y[pick_rows(n, round(0.05 * n), seed=seed, exclude=(LLAMA3_CONST_ROW,))] = IGNORE_INDEX
    return y


def llama3(dtype: int = BF16, seed: int = SEED_BASE + 4, rows: int | None = None, row0: int = 0,
           out: np.ndarray | None = None):
    n, v = 8192, 128256
    y = llama3_labels(n, v, seed=seed)
    rows = n - row0 if rows is None else rows
    x = normal_matrix(rows, v, seed=seed, sigma=3.0, dtype=dtype, spike_p=1e-4, spike_lo=20.0,
                      spike_hi=30.0, row0=row0, out=out)
    if row0 <= LLAMA3_CONST_ROW < row0 + rows:
        x[LLAMA3_CONST_ROW - row0, :v] = 3.0 if dtype == F32 else np.uint16(0x4040)  # bf16(3.0)
    return dict(name="llama3", logits=x, labels=y[row0:row0 + rows], N=rows, V=v, dtype=dtype,
                g=1.0, seed=seed, full_labels=y)


def chunked(seed: int = SEED_BASE + 5, n: int = 8192, v: int = 32000, d: int = 4096,
            chunk: int = 1024):
    h = normal_matrix(n, d, seed=seed, sigma=1.0, dtype=BF16, stream=S_H)
    w = normal_matrix(v, d, seed=seed, sigma=0.02, dtype=BF16, stream=S_W)
    y = uniform_labels(n, v, seed=seed)
    y[pick_rows(n, round(0.1 * n), seed=seed)] = IGNORE_INDEX
    return dict(name="chunked", H=h, W=w, labels=y, N=n, V=v, D=d, chunk=chunk, g=1.0, seed=seed)


def norm_chunked(seed: int = SEED_BASE + 6, n: int = 8192, v: int = 32000, d: int = 4096,
                 chunk: int = 1024, eps: float = 1e-5):
    """The decoder's tail -- final RMSNorm, LM head, cross-entropy -- at the chunked
    workload's sizes: X 8192x4096 bf16 ~N(0, 2^2) (pre-norm hidden states), gamma
    bf16 ~N(1, 0.1^2) (a trained norm weight near one), W and labels as ``chunked``."""
    x = normal_matrix(n, d, seed=seed, sigma=2.0, dtype=BF16, stream=S_X)
    gz = normal_matrix(1, d, seed=seed, sigma=0.1, dtype=F32, stream=S_GAMMA)[0].astype(np.float64)
    gamma = f64_to_bf16_bits(1.0 + gz)
    w = normal_matrix(v, d, seed=seed, sigma=0.02, dtype=BF16, stream=S_W)
    y = uniform_labels(n, v, seed=seed)
    y[pick_rows(n, round(0.1 * n), seed=seed)] = IGNORE_INDEX
    return dict(name="norm_chunked", X=x, gamma=gamma, W=w, labels=y, N=n, V=v, D=d, chunk=chunk, eps=eps, g=1.0,
                seed=seed)


def packed_positions(n: int, *, seed: int, max_len: int = 2048) -> np.ndarray:
    """Position ids of a padding-free packed batch: sequences of lengths U{64..max_len}
    (the last truncated) laid end to end, each counting from 0."""
    pos = np.empty(n, dtype=np.int64)
    at, k = 0, 0
    while at < n:
        L = 64 + int(np.floor(uniform(seed, S_SEQLEN, 1, start=k)[0] * (max_len - 64 + 1)))
        L = min(L, n - at)
        pos[at:at + L] = np.arange(L)
        at += L
        k += 1
    return pos


def rope_llama3(dtype: int = BF16, seed: int = SEED_BASE + 7, tokens: int = 8192):
    """Llama-3-8B attention shapes for the rotary embedding: Q (T x 32 x 128) and K
    (T x 8 x 128) ~N(0, 1) in a packed batch of sequences up to 2048 tokens, rope
    base 500000, table for 8192 positions."""
    q = normal_matrix(tokens, 32 * 128, seed=seed, sigma=1.0, dtype=dtype, stream=S_X).reshape(tokens, 32, 128)
    k = normal_matrix(tokens, 8 * 128, seed=seed, sigma=1.0, dtype=dtype, stream=S_H).reshape(tokens, 8, 128)
    return dict(name="rope_llama3", Q=q, K=k, positions=packed_positions(tokens, seed=seed), base=500000.0,
                max_pos=8192, d=128, dtype=dtype, seed=seed)


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64 (plain data conversion)."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float64 -> float32 -> bfloat16 (nearest-even) bit patterns."""
    f = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    f = f + 0x7FFF + ((f >> 16) & 1)
    return (f >> 16).astype(np.uint16)
