"""Host-side checks of the C ABI that need no GPU.

The library must load, export every function include/foak_ce.h declares, and turn
bad arguments (and an injected launch failure) into status codes before anything
is enqueued.  The pointers below are never dereferenced: every call here returns
before the first CUDA call.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "foak_ce.h")


@pytest.fixture(scope="module")
def so():
    import __graft_entry__

    __graft_entry__._build_module().build()
    import cross_entropy_loss_gb300 as ce

    return ce


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(foak_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(so):
    names = _declared()
    assert "foak_ce_fwd_bwd" in names and "foak_ce_forward" in names and "foak_ce_backward" in names
    raw = ctypes.CDLL(so.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in foak_ce.h but not exported"
    assert set(names) == set(so.SIGNATURES), "binding signatures and header drifted apart"


def test_version_vocab_and_workspace(so):
    assert so.lib.foak_abi_version() == 1
    assert so.foak_ce_max_vocab(so.FOAK_BF16) == 2 ** 31 - 1
    assert so.foak_ce_max_vocab(so.FOAK_F32) == 2 ** 31 - 1
    assert so.foak_ce_max_vocab(7) == 0
    assert so.foak_ce_workspace_size(0) == 256
    assert so.foak_ce_workspace_size(8192) == 256 + 8192 * 4
    assert so.foak_ce_workspace_size(3) == 512


FAKE = 0x10000  # 64 KB-aligned fake device address (never touched)


def _fwd_bwd(so, logits=FAKE, dtype=1, ld=32000, labels=FAKE, N=4, V=32000, loss=FAKE, ws=FAKE,
             wsb=1 << 20, lse=None, nv=None, err=None):
    return so.lib.foak_ce_fwd_bwd(logits, dtype, ld, labels, N, V, -100, 1.0, 0.0, loss, lse, nv, err, ws, wsb,
                                  None)


def test_argument_errors_return_before_launch(so):
    E = so
    assert _fwd_bwd(so, dtype=2) == E.FOAK_ERR_UNSUPPORTED           # fp16 / unknown dtype
    assert _fwd_bwd(so, ld=31999) == E.FOAK_ERR_INVALID_ARG          # ld < V
    assert _fwd_bwd(so, V=0) == E.FOAK_ERR_INVALID_ARG
    assert _fwd_bwd(so, N=-1) == E.FOAK_ERR_INVALID_ARG
    assert _fwd_bwd(so, logits=None) == E.FOAK_ERR_INVALID_ARG
    assert _fwd_bwd(so, labels=None) == E.FOAK_ERR_INVALID_ARG
    assert _fwd_bwd(so, loss=None) == E.FOAK_ERR_INVALID_ARG
    assert _fwd_bwd(so, logits=FAKE + 1) == E.FOAK_ERR_INVALID_ARG   # bf16 needs 2-byte alignment
    assert _fwd_bwd(so, labels=FAKE + 4) == E.FOAK_ERR_INVALID_ARG   # int64 labels
    assert _fwd_bwd(so, lse=FAKE + 2) == E.FOAK_ERR_INVALID_ARG
    assert _fwd_bwd(so, V=2 ** 31, ld=2 ** 31) == E.FOAK_ERR_UNSUPPORTED   # column indexes are 32-bit
    assert _fwd_bwd(so, ws=None) == E.FOAK_ERR_WORKSPACE
    assert _fwd_bwd(so, ws=FAKE + 16) == E.FOAK_ERR_WORKSPACE        # 256-byte alignment
    assert _fwd_bwd(so, wsb=256) == E.FOAK_ERR_WORKSPACE             # too small for N rows
    # data-parallel pair: count into an 8-byte aligned int64, fused call with a device denominator
    assert so.lib.foak_ce_count_valid(FAKE, 4, 32000, -100, None, None, None) == E.FOAK_ERR_INVALID_ARG
    assert so.lib.foak_ce_count_valid(FAKE, 4, 32000, -100, FAKE + 4, None, None) == E.FOAK_ERR_INVALID_ARG
    assert so.lib.foak_ce_count_valid(None, 4, 32000, -100, FAKE, None, None) == E.FOAK_ERR_INVALID_ARG
    assert so.lib.foak_ce_count_valid(FAKE, -1, 32000, -100, FAKE, None, None) == E.FOAK_ERR_INVALID_ARG
    assert so.lib.foak_ce_count_valid(FAKE, 4, 0, -100, FAKE, None, None) == E.FOAK_ERR_INVALID_ARG
    dd = so.lib.foak_ce_fwd_bwd_devdenom
    assert dd(FAKE, 1, 32000, FAKE, 4, 32000, -100, 1.0, None, FAKE, None, None, None, FAKE, 1 << 20,
              None) == E.FOAK_ERR_INVALID_ARG                          # no denominator
    assert dd(FAKE, 1, 32000, FAKE, 4, 32000, -100, 1.0, FAKE + 4, FAKE, None, None, None, FAKE, 1 << 20,
              None) == E.FOAK_ERR_INVALID_ARG                          # misaligned int64
    assert dd(FAKE, 1, 31999, FAKE, 4, 32000, -100, 1.0, FAKE, FAKE, None, None, None, FAKE, 1 << 20,
              None) == E.FOAK_ERR_INVALID_ARG                          # ld < V
    # backward: dlogits must share logits' 16-byte phase
    st = so.lib.foak_ce_backward(FAKE + 2, FAKE, 1, 32000, FAKE, 4, 32000, -100, FAKE, None, 0.0, None, None)
    assert st == E.FOAK_ERR_INVALID_ARG
    st = so.lib.foak_ce_backward(FAKE, FAKE, 1, 32000, FAKE, 4, 32000, -100, None, None, 0.0, None, None)
    assert st == E.FOAK_ERR_INVALID_ARG  # lse required


def test_injected_launch_failure(so):
    so.lib.foak_test_fail_next_launches(2)
    try:
        assert _fwd_bwd(so) == so.FOAK_ERR_CUDA
        st = so.lib.foak_ce_forward(FAKE, 0, 64, FAKE, 4, 64, -100, 0.0, FAKE, None, None, None, None, FAKE,
                                    1 << 20, None)
        assert st == so.FOAK_ERR_CUDA
    finally:
        so.lib.foak_test_fail_next_launches(0)
    # argument errors still win over the injected failure
    so.lib.foak_test_fail_next_launches(1)
    assert _fwd_bwd(so, dtype=5) == so.FOAK_ERR_UNSUPPORTED
    so.lib.foak_test_fail_next_launches(0)


def test_status_strings(so):
    for code in range(7):
        assert so.status_string(code).startswith("FOAK_")
    assert "unknown" in so.status_string(99)
    err = so.FoakError(so.FOAK_ERR_WORKSPACE, "x")
    assert "WORKSPACE" in str(err)


def _host(so, hx=FAKE, dtype=1, ld=32000, hy=FAKE, N=4, V=32000, dx=FAKE, dy=FAKE, hl=FAKE, ws=FAKE,
          wsb=1 << 20):
    return so.lib.foak_ce_fwd_bwd_host(hx, dtype, ld, hy, N, V, -100, 1.0, 0.0, dx, dy, hl, None, None, ws, wsb,
                                       None)


def test_host_entry_argument_errors(so):
    """foak_ce_fwd_bwd_host checks its host and device buffers before any copy."""
    E = so
    assert so.foak_ce_host_workspace_size(0) == 512
    assert so.foak_ce_host_workspace_size(8192) == 256 + 8192 * 4 + 256
    assert so.foak_ce_host_workspace_size(-1) == 0
    assert _host(so, dtype=3) == E.FOAK_ERR_UNSUPPORTED
    assert _host(so, ld=10) == E.FOAK_ERR_INVALID_ARG
    assert _host(so, hx=None) == E.FOAK_ERR_INVALID_ARG
    assert _host(so, hy=None) == E.FOAK_ERR_INVALID_ARG
    assert _host(so, dx=None) == E.FOAK_ERR_INVALID_ARG
    assert _host(so, dy=None) == E.FOAK_ERR_INVALID_ARG
    assert _host(so, hl=None) == E.FOAK_ERR_INVALID_ARG
    assert _host(so, dx=FAKE + 8) == E.FOAK_ERR_INVALID_ARG       # device logits 16-byte aligned
    assert _host(so, ws=None) == E.FOAK_ERR_WORKSPACE
    assert _host(so, wsb=512) == E.FOAK_ERR_WORKSPACE             # N rows need 256 + 256 + 256 bytes
    so.lib.foak_test_fail_next_launches(1)
    try:
        assert _host(so) == E.FOAK_ERR_CUDA
    finally:
        so.lib.foak_test_fail_next_launches(0)


def test_rmsnorm_entries_argument_errors(so):
    """The RMSNorm calls reject bad sizes, dtypes and alignments before any launch."""
    E = so
    L = so.lib
    assert L.foak_rmsnorm_workspace_size(4096) == 512 * 4096 * 4
    assert L.foak_rmsnorm_workspace_size(0) == 0
    fwd = lambda X=FAKE, dt=1, ldx=64, g=FAKE, N=4, D=64, eps=1e-5, Y=FAKE, ldy=64, r=FAKE: (  # noqa: E731
        L.foak_rmsnorm_forward(X, dt, ldx, g, N, D, eps, Y, ldy, r, None))
    assert fwd(dt=2) == E.FOAK_ERR_UNSUPPORTED
    assert fwd(D=60, ldx=60, ldy=60) == E.FOAK_ERR_UNSUPPORTED       # D % 8
    assert fwd(ldx=32) == E.FOAK_ERR_INVALID_ARG                     # ld < D
    assert fwd(eps=-1.0) == E.FOAK_ERR_INVALID_ARG
    assert fwd(X=FAKE + 2) == E.FOAK_ERR_INVALID_ARG                 # rows start on 16 bytes
    assert fwd(ldx=68) == E.FOAK_ERR_INVALID_ARG                     # 136-byte row stride
    assert fwd(g=None) == E.FOAK_ERR_INVALID_ARG
    bwd = lambda dY=FAKE, r=FAKE, dg=FAKE, ws=FAKE, wsb=1 << 20: (  # noqa: E731
        L.foak_rmsnorm_backward(dY, 64, FAKE, 64, FAKE, r, 1, 4, 64, FAKE, 64, dg, ws, wsb, None))
    assert bwd(dY=None) == E.FOAK_ERR_INVALID_ARG
    assert bwd(r=None) == E.FOAK_ERR_INVALID_ARG
    assert bwd(wsb=16) == E.FOAK_ERR_WORKSPACE
    assert bwd(ws=None) == E.FOAK_ERR_WORKSPACE
    assert L.foak_rmsnorm_linear_ce_workspace_size(8192, 32000, 4096, 1024) > 2 * 8192 * 4096 * 2
    tail = lambda X=FAKE, g=FAKE, D=64, eps=1e-5, dg=FAKE, wsb=1 << 30: (  # noqa: E731
        L.foak_rmsnorm_linear_ce_chunked(X, g, FAKE, FAKE, 4, 100, D, -100, 1024, eps, 1.0, 0.0, FAKE, FAKE, dg,
                                         FAKE, None, None, FAKE, wsb, None))
    assert tail(D=60) == E.FOAK_ERR_UNSUPPORTED
    assert tail(eps=-0.5) == E.FOAK_ERR_INVALID_ARG
    assert tail(g=None) == E.FOAK_ERR_INVALID_ARG
    assert tail(dg=None) == E.FOAK_ERR_INVALID_ARG
    assert tail(X=FAKE + 8) == E.FOAK_ERR_INVALID_ARG
    assert tail(wsb=1024) == E.FOAK_ERR_WORKSPACE


def test_rope_entries_argument_errors(so):
    """The RoPE calls reject bad head dimensions, strides and alignments before any launch."""
    E = so
    L = so.lib
    assert L.foak_rope_cache_size(8192, 128) == 2 * 8192 * 64 * 4
    assert L.foak_rope_cache_size(8192, 120) == 0                    # d % 16
    assert L.foak_rope_cache_size(0, 128) == 0
    assert L.foak_rope_build_cache(1e4, 120, 16, FAKE, 1 << 20, None) == E.FOAK_ERR_UNSUPPORTED
    assert L.foak_rope_build_cache(0.5, 128, 16, FAKE, 1 << 20, None) == E.FOAK_ERR_INVALID_ARG   # base > 1
    assert L.foak_rope_build_cache(1e4, 128, 16, FAKE + 16, 1 << 20, None) == E.FOAK_ERR_INVALID_ARG
    assert L.foak_rope_build_cache(1e4, 128, 16, FAKE, 64, None) == E.FOAK_ERR_WORKSPACE
    ap = lambda X=FAKE, dt=1, T=4, H=2, ldt=256, d=128, pos=FAKE, c=FAKE: (  # noqa: E731
        L.foak_rope_apply(X, dt, T, H, ldt, d, pos, c, 16, 0, None, None))
    assert ap(dt=2) == E.FOAK_ERR_UNSUPPORTED
    assert ap(d=72, ldt=144) == E.FOAK_ERR_UNSUPPORTED
    assert ap(ldt=255) == E.FOAK_ERR_INVALID_ARG                     # ldt < H * d
    assert ap(X=FAKE + 2) == E.FOAK_ERR_INVALID_ARG
    assert ap(ldt=260) == E.FOAK_ERR_INVALID_ARG                     # 520-byte token stride
    assert ap(pos=None) == E.FOAK_ERR_INVALID_ARG
    assert ap(c=FAKE + 64) == E.FOAK_ERR_INVALID_ARG                 # table 256-byte aligned
    qk = lambda Q=FAKE, K=FAKE, ldk=128: (  # noqa: E731
        L.foak_rope_apply_qk(Q, 2, 256, K, 1, ldk, 1, 4, 128, FAKE, FAKE, 16, 0, None, None))
    assert qk(K=None) == E.FOAK_ERR_INVALID_ARG
    assert qk(ldk=64) == E.FOAK_ERR_INVALID_ARG


def test_gemm_group_argument_errors(so):
    """foak_gemm_bf16_group rejects a bad count or a bad product before any launch; an
    empty group (or only empty products) is a no-op."""
    E = so
    L = so.lib

    def prob(**kw):
        f = dict(a=FAKE, lda=64, a_mn_major=0, b=FAKE, ldb=64, b_mn_major=0, M=256, N=256, K=64, out=FAKE, ldo=256,
                 out_mode=E.FOAK_GEMM_BF16)
        f.update(kw)
        return E._GemmProblem(**f)

    def group(*ps, n=None):
        arr = (E._GemmProblem * max(1, len(ps)))(*ps)
        return L.foak_gemm_bf16_group(ctypes.cast(arr, ctypes.c_void_p), len(ps) if n is None else n, None, None)

    assert group(n=-1) == E.FOAK_ERR_INVALID_ARG
    assert group(prob(), prob(), prob(), prob()) == E.FOAK_ERR_INVALID_ARG  # more than FOAK_GEMM_GROUP_MAX
    assert L.foak_gemm_bf16_group(None, 1, None, None) == E.FOAK_ERR_INVALID_ARG
    assert group(prob(), prob(out_mode=7)) == E.FOAK_ERR_INVALID_ARG
    assert group(prob(lda=32)) == E.FOAK_ERR_INVALID_ARG                   # lda < K
    assert group(prob(), prob(a=FAKE + 8)) == E.FOAK_ERR_INVALID_ARG       # 16-byte alignment
    assert group(prob(ldo=100)) == E.FOAK_ERR_INVALID_ARG                  # ldo < N
    assert group(prob(K=-1)) == E.FOAK_ERR_INVALID_ARG
    assert group(n=0) == E.FOAK_OK
    assert group(prob(M=0), prob(N=0, ldo=0)) == E.FOAK_OK


def _group_schedule(so, shapes, pairs, cap=20000):
    mnk = (ctypes.c_int64 * (3 * len(shapes)))(*[v for s in shapes for v in s])
    start = (ctypes.c_int32 * (pairs + 1))()
    ent = (ctypes.c_int32 * cap)()
    nc = so.lib.foak_test_gemm_group_schedule(mnk, len(shapes), pairs, start, ent, cap)
    if nc < 0:
        return nc, None, None
    return nc, list(start[:nc + 1]), list(ent[:start[nc]])


@pytest.mark.parametrize("shapes", [
    [(1024, 32000, 4096), (1024, 4096, 32000)],                      # {Z(c), dH(c-2)}
    [(1024, 32000, 4096), (1024, 4096, 32000), (32000, 4096, 4096)],  # ... with a group's dW
    [(300, 700, 192), (512, 256, 4096)],                             # ragged shapes
])
def test_gemm_group_schedule_every_unit_once_longest_first_balanced(so, shapes):
    """The grouped GEMM's unit list (host logic): each (product, 256 x 256 unit) exactly
    once, every SM pair's list longest first, and the estimated work per pair (k-blocks
    + 8 per unit) within 10% of the mean or one unit of the longest kind."""
    pairs = 76
    nc, start, ent = _group_schedule(so, shapes, pairs)
    units = [((M + 127) // 128 + 1) // 2 * ((N + 255) // 256) for M, N, K in shapes]
    cost = [(K + 63) // 64 + 8 for M, N, K in shapes]
    assert nc == min(pairs, sum(units)) and start[0] == 0
    assert sorted(ent) == sorted((q << 14) | u for q in range(len(shapes)) for u in range(units[q]))
    loads = []
    for c in range(nc):
        mine = [cost[e >> 14] for e in ent[start[c]:start[c + 1]]]
        assert mine == sorted(mine, reverse=True)
        loads.append(sum(mine))
    mean = sum(loads) / nc
    assert max(loads) <= max(1.10 * mean, mean + max(cost))


def test_gemm_group_schedule_argument_errors(so):
    assert _group_schedule(so, [(128, 256, 64)], 76)[0] == -1        # single-CTA tiles
    assert _group_schedule(so, [(1024, 32000, 4096)], 76, cap=10)[0] == -1
    assert so.lib.foak_test_gemm_group_schedule(None, 1, 76, None, None, 0) == -1
