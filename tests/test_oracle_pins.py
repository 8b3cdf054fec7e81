"""Pins for the CPU oracle: what the definition and the mathematics fix.

Each test compares the oracle with something other than itself -- hand-derived
fractions, closed forms, invariants, central finite differences, an independent
50-digit evaluation, or a library routine with the same definition -- so that a
dropped term, a wrong sign or index, or a transposed operand fails at least one.
The definition is the softmax cross-entropy with mean over non-ignored rows that
the FOAK pages call FastCrossEntropyLoss (fms-acceleration PR #79, Description
item 4) and its fused linear + CE form (LigerFusedLinearCrossEntropy, "Running
Liger Kernel Benchmarks" on the fms-acceleration-foak 0.7.4 page).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _frac(s: str) -> Fraction:
    if "/" in s:
        a, b = s.split("/")
        return Fraction(a) / Fraction(b)
    return Fraction(s)


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_worked(case):
    x = np.array([[math.log(float(_frac(q))) for q in row] for row in case["logits_ln"]])
    y = np.array(case["labels"], dtype=np.int64)
    r = oracle.ce(x, y, ignore_index=case["ignore_index"], g=float(_frac(case["g"])),
                  denom=float(_frac(case["denom"])))
    exp_loss = sum(c * math.log(float(_frac(q))) for q, c in case["loss_terms"])
    exp_loss /= float(_frac(case["loss_divisor"]))
    assert r["n_valid"] == case["n_valid"]
    assert r["n_bad"] == case.get("n_bad", 0)
    assert r["loss"] == pytest.approx(exp_loss, rel=1e-13, abs=1e-15)
    exp_grad = np.array([[float(_frac(q)) for q in row] for row in case["grad"]])
    np.testing.assert_allclose(r["grad"], exp_grad, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("V", [1, 7, 1000, 128256])
def test_uniform_row_gives_ln_V(V):
    x = np.full((2, V), 3.0)
    y = np.array([V - 1, 0], dtype=np.int64)
    r = oracle.ce(x, y)
    assert r["loss"] == pytest.approx(math.log(V), rel=1e-14, abs=1e-15)
    expect = np.full((2, V), 1.0 / V) / 2
    expect[0, V - 1] -= 0.5
    expect[1, 0] -= 0.5
    np.testing.assert_allclose(r["grad"], expect, rtol=1e-12, atol=1e-18)


@pytest.mark.parametrize("V", [2, 1000, 32000])
def test_dominant_label_loss_goes_to_zero(V):
    rng = np.random.default_rng(1)
    base = rng.normal(size=V) * 0.0 + 1.5  # all others equal, so the closed form is exact
    y = V // 3
    base[y] += 50.0
    r = oracle.ce(base[None, :], np.array([y]))
    exact = math.log1p((V - 1) * math.exp(-50.0))
    assert r["loss"] == pytest.approx(exact, rel=1e-9)
    assert r["loss"] < 1e-16 * V


def test_single_class_is_zero():
    x = np.array([[-4.0], [123.5]])
    r = oracle.ce(x, np.array([0, 0]))
    assert r["loss"] == 0.0
    assert np.all(r["grad"] == 0.0)


@pytest.mark.parametrize("d", [-30.0, -2.5, 0.0, 0.75, 12.0])
def test_two_classes_is_logistic_loss(d):
    # x_other - x_y = d  ->  loss = softplus(d) = ln(1 + e^d); dloss/dx_y = -sigmoid(d)
    x = np.array([[0.25, 0.25 + d]])
    r = oracle.ce(x, np.array([0]))
    sp = d + math.log1p(math.exp(-d)) if d > 0 else math.log1p(math.exp(d))
    # lse - x_y cancels: the double result is good to a few ulps of the logits' size
    assert r["loss"] == pytest.approx(sp, rel=1e-13, abs=4e-16 * (abs(d) + 1))
    sig = 1.0 / (1.0 + math.exp(-d))
    assert r["grad"][0, 0] == pytest.approx(-sig, rel=1e-13, abs=4e-16)  # p_y - 1 cancels too
    assert r["grad"][0, 1] == pytest.approx(sig, rel=1e-13, abs=1e-300)


def _rand_case(n=9, v=13, seed=5, ignore=(2, 7)):
    rng = np.random.default_rng(seed)
    x = rng.normal(scale=3.0, size=(n, v))
    y = rng.integers(0, v, size=n).astype(np.int64)
    y[list(ignore)] = -100
    return x, y


def test_shift_invariance():
    x, y = _rand_case()
    a = oracle.ce(x, y)
    shift = np.arange(x.shape[0])[:, None] * 17.25 - 40.0
    b = oracle.ce(x + shift, y)
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-13)
    np.testing.assert_allclose(b["grad"], a["grad"], rtol=1e-10, atol=1e-15)


def test_gradient_rows_sum_to_zero_and_ignored_rows_are_zero():
    x, y = _rand_case(n=40, v=257, seed=11, ignore=(0, 5, 39))
    r = oracle.ce(x, y, g=1.7)
    valid = y != -100
    sums = r["grad"].sum(axis=1)
    assert np.all(np.abs(sums[valid]) < 1e-15 * x.shape[1])
    assert np.all(r["grad"][~valid] == 0.0)
    assert np.all(np.signbit(r["grad"][~valid]) == False)  # +0.0
    assert r["n_valid"] == int(valid.sum())
    assert np.all(r["row_loss"][~valid] == 0.0)


def test_finite_differences():
    x, y = _rand_case(n=4, v=6, seed=3, ignore=(1,))
    g = 0.8
    r = oracle.ce(x, y, g=g)
    h = 1e-5
    fd = np.zeros_like(x)
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            fd[i, j] = g * (oracle.ce(xp, y)["loss"] - oracle.ce(xm, y)["loss"]) / (2 * h)
    np.testing.assert_allclose(r["grad"], fd, rtol=0, atol=1e-9)


def test_linear_in_upstream_gradient_and_denominator():
    x, y = _rand_case()
    a = oracle.ce(x, y, g=1.0)
    b = oracle.ce(x, y, g=-2.5)
    np.testing.assert_allclose(b["grad"], -2.5 * a["grad"], rtol=1e-14, atol=0)
    assert b["loss"] == a["loss"]  # g scales only the gradient
    c = oracle.ce(x, y, g=1.0, denom=1000.0)
    assert c["loss"] * 1000.0 == pytest.approx(a["row_loss"].sum(), rel=1e-14)
    np.testing.assert_allclose(c["grad"] * 1000.0, a["grad"] * a["n_valid"], rtol=1e-13)


def test_all_rows_ignored():
    x = np.ones((3, 5))
    r = oracle.ce(x, np.array([-100, -100, -100]))
    assert r["n_valid"] == 0 and math.isnan(r["loss"])
    assert np.all(r["grad"] == 0.0)


def test_matches_50_digit_evaluation():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    x, y = _rand_case(n=5, v=11, seed=9, ignore=(3,))
    x = x * 10  # spread values so an unshifted double sum would lose digits
    r = oracle.ce(x, y, g=1.0)
    valid = [i for i in range(len(y)) if y[i] != -100]
    tot = mpmath.mpf(0)
    for i in valid:
        s = mpmath.fsum(mpmath.e ** mpmath.mpf(float(v)) for v in x[i])
        lse = mpmath.log(s)
        tot += lse - mpmath.mpf(float(x[i, y[i]]))
        for j in range(x.shape[1]):
            p = mpmath.e ** (mpmath.mpf(float(x[i, j])) - lse)
            want = (p - (1 if j == y[i] else 0)) / len(valid)
            # label entries are p - 1: double cancellation leaves ~1e-16 absolute
            assert r["grad"][i, j] == pytest.approx(float(want), rel=1e-12, abs=1e-15)
    assert r["loss"] == pytest.approx(float(tot / len(valid)), rel=1e-14)


def test_matches_torch_float64_cross_entropy():
    torch = pytest.importorskip("torch")
    x, y = _rand_case(n=33, v=50, seed=21, ignore=(0, 4, 32))
    y[10] = -1  # ignore_index below is -1; the -100 rows are then out-of-range labels
    r = oracle.ce(x, y, ignore_index=-1)
    assert r["n_bad"] == int((y == -100).sum()) == 3
    # bad labels contribute like ignored rows: torch sees them as ignore_index
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    yt = torch.tensor(np.where(y >= 0, y, -1))
    lt = torch.nn.functional.cross_entropy(xt, yt, ignore_index=-1, reduction="mean")
    lt.backward()
    assert r["loss"] == pytest.approx(lt.item(), rel=1e-13)
    np.testing.assert_allclose(r["grad"], xt.grad.numpy(), rtol=1e-12, atol=1e-18)


def test_bf16_and_padded_rows_decode_exactly():
    n, v, ld = 6, 37, 48
    bits = wl.normal_matrix(n, v, seed=4, sigma=2.0, dtype=wl.BF16, ld=ld)
    bits[:, v:] = 0x7F7F  # huge padding values must never be read
    y = np.array([0, 36, -100, 5, 12, 1], dtype=np.int64)
    a = oracle.ce(bits, y, V=v)
    as64 = wl.bf16_bits_to_f64(bits[:, :v])
    b = oracle.ce(as64, y)
    assert a["loss"] == b["loss"]
    np.testing.assert_array_equal(a["grad"], b["grad"])
    f32 = as64.astype(np.float32)
    c = oracle.ce(f32, y)
    assert c["loss"] == b["loss"]


def test_row_subsets_equal_whole_batch():
    x, y = _rand_case(n=30, v=40, seed=8, ignore=(3, 4, 29))
    whole = oracle.ce(x, y, g=2.0)
    lse, rl, st, grad = oracle.rows(x[10:20], y[10:20], 40, scale=whole["scale"])
    np.testing.assert_array_equal(lse, whole["lse"][10:20])
    np.testing.assert_array_equal(grad, whole["grad"][10:20])
    t1 = oracle.ce(x, y, threads=1)
    t4 = oracle.ce(x, y, threads=4)
    assert t1["loss"] == t4["loss"]


# ---------------------------------------------------------------- linear + CE


def _lin_case(n=6, d=5, v=7, seed=2):
    rng = np.random.default_rng(seed)
    H = rng.normal(size=(n, d))
    W = rng.normal(scale=0.7, size=(v, d))
    y = rng.integers(0, v, size=n).astype(np.int64)
    y[1] = -100
    return H, W, y


def test_linear_logits_match_triple_loop():
    H, W, y = _lin_case()
    r = oracle.linear_ce(H, W, y)
    Z = np.zeros((H.shape[0], W.shape[0]))
    for i in range(H.shape[0]):
        for j in range(W.shape[0]):
            s = 0.0
            for k in range(H.shape[1]):
                s += H[i, k] * W[j, k]
            Z[i, j] = s
    np.testing.assert_allclose(r["Z"], Z, rtol=1e-13, atol=1e-13)


def test_linear_gradients_by_finite_differences():
    H, W, y = _lin_case()
    g = 1.3
    r = oracle.linear_ce(H, W, y, g=g)
    h = 1e-6

    def loss(Hx, Wx):
        return oracle.linear_ce(Hx, Wx, y)["loss"]

    for (i, k) in [(0, 0), (2, 3), (5, 4), (1, 2)]:
        Hp, Hm = H.copy(), H.copy()
        Hp[i, k] += h
        Hm[i, k] -= h
        assert g * (loss(Hp, W) - loss(Hm, W)) / (2 * h) == pytest.approx(r["dH"][i, k], abs=1e-8)
    for (j, k) in [(0, 0), (6, 4), (3, 1)]:
        Wp, Wm = W.copy(), W.copy()
        Wp[j, k] += h
        Wm[j, k] -= h
        assert g * (loss(H, Wp) - loss(H, Wm)) / (2 * h) == pytest.approx(r["dW"][j, k], abs=1e-8)
    # the ignored row contributes no hidden-state gradient
    assert np.all(r["dH"][1] == 0.0)


def test_linear_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    H, W, y = _lin_case(n=12, d=8, v=10, seed=6)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    lt = torch.nn.functional.cross_entropy(Ht @ Wt.T, torch.tensor(y), ignore_index=-100)
    lt.backward()
    r = oracle.linear_ce(H, W, y)
    assert r["loss"] == pytest.approx(lt.item(), rel=1e-13)
    np.testing.assert_allclose(r["dH"], Ht.grad.numpy(), rtol=1e-11, atol=1e-15)
    np.testing.assert_allclose(r["dW"], Wt.grad.numpy(), rtol=1e-11, atol=1e-15)


def test_linear_chunks_of_rows_compose_to_whole():
    # a global D makes chunk results add up to the whole batch's
    H, W, y = _lin_case(n=10, d=4, v=9, seed=12)
    whole = oracle.linear_ce(H, W, y)
    D = whole["n_valid"]
    dW = np.zeros_like(W)
    tot = 0.0
    for c in range(0, 10, 3):
        part = oracle.linear_ce(H[c:c + 3], W, y[c:c + 3], denom=float(D)) if (y[c:c + 3] != -100).any() \
            else None
        if part is None:
            continue
        tot += part["loss"]
        dW += part["dW"]
        np.testing.assert_allclose(part["dH"], whole["dH"][c:c + 3], rtol=1e-12, atol=1e-16)
    assert tot == pytest.approx(whole["loss"], rel=1e-13)
    np.testing.assert_allclose(dW, whole["dW"], rtol=1e-12, atol=1e-16)


# ------------------------------------------------------------------ RMSNorm pins

def test_rmsnorm_hand_worked_and_closed_forms():
    # hand-worked row: x = (3, 4), gamma = (1, 2), eps = 0: mean square 12.5, rms 3.5355339059327378
    Y, r = oracle.rmsnorm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.0)
    assert r[0] == pytest.approx(0.28284271247461906, rel=1e-15)
    np.testing.assert_allclose(Y[0], [0.8485281374238571, 2.2627416997969522], rtol=1e-15)
    # a constant row c: y_j = c / sqrt(c^2 + eps) * gamma_j
    g = np.array([0.5, -1.0, 2.0, 3.0])
    Y, _ = oracle.rmsnorm(np.full((1, 4), 2.0), g, 0.25)
    np.testing.assert_allclose(Y[0], 2.0 / math.sqrt(4.25) * g, rtol=1e-15)
    # the normalised row's mean square is ms / (ms + eps)
    rng = np.random.default_rng(7)
    X = rng.normal(size=(5, 33)) * 3.0
    Y, _ = oracle.rmsnorm(X, np.ones(33), 0.1)
    ms = (X ** 2).sum(axis=1) / 33
    np.testing.assert_allclose((Y ** 2).sum(axis=1) / 33, ms / (ms + 0.1), rtol=1e-14)
    # with eps = 0 the norm is scale invariant
    Ya, _ = oracle.rmsnorm(X, g[:1].repeat(33), 0.0)
    Yb, _ = oracle.rmsnorm(3.7 * X, g[:1].repeat(33), 0.0)
    np.testing.assert_allclose(Ya, Yb, rtol=1e-14)


def _fd(f, a, h=1e-6):
    out = np.zeros_like(a)
    for idx in np.ndindex(a.shape):
        p, m = a.copy(), a.copy()
        p[idx] += h
        m[idx] -= h
        out[idx] = (f(p) - f(m)) / (2 * h)
    return out


def test_rmsnorm_backward_matches_finite_differences():
    rng = np.random.default_rng(11)
    X, g, dY, eps = rng.normal(size=(3, 5)), rng.normal(size=5), rng.normal(size=(3, 5)), 1e-3
    dX, dg = oracle.rmsnorm_backward(dY, X, g, eps)
    fx = _fd(lambda x: float(np.sum(dY * oracle.rmsnorm(x, g, eps)[0])), X)
    fg = _fd(lambda gg: float(np.sum(dY * oracle.rmsnorm(X, gg, eps)[0])), g)
    np.testing.assert_allclose(dX, fx, rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(dg, fg, rtol=1e-7, atol=1e-9)


def test_rmsnorm_linear_ce_matches_finite_differences():
    """Final norm -> LM head -> CE on tiny sizes: dX, dgamma and dW against central
    differences of the loss (one row ignored, so the mean is over 3 rows)."""
    rng = np.random.default_rng(5)
    N, D, V, eps = 4, 6, 5, 1e-4
    X, g, W = rng.normal(size=(N, D)), rng.normal(size=D), rng.normal(size=(V, D)) * 0.5
    y = np.array([1, -100, 4, 0], dtype=np.int64)
    res = oracle.rmsnorm_linear_ce(X, g, W, y, eps=eps, g=1.3)
    L = lambda x, gg, w: oracle.rmsnorm_linear_ce(x, gg, w, y, eps=eps, g=1.3)["loss"] * 1.3  # noqa: E731
    np.testing.assert_allclose(res["dX"], _fd(lambda x: L(x, g, W), X, 1e-5), rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(res["dgamma"], _fd(lambda gg: L(X, gg, W), g, 1e-5), rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(res["dW"], _fd(lambda w: L(X, g, w), W, 1e-5), rtol=1e-6, atol=1e-9)
    assert res["n_valid"] == 3


# ------------------------------------------------------------------ RoPE pins

def test_rope_hand_worked_and_identity():
    # d = 4, base 100: angles (p, p / 10); q = e0 at p = 1 turns into (cos 1, 0, sin 1, 0)
    out = oracle.rope(np.array([[[1.0, 0.0, 0.0, 0.0]]]), np.array([1]), 100.0)
    np.testing.assert_allclose(out[0, 0], [math.cos(1.0), 0.0, math.sin(1.0), 0.0], atol=1e-16)
    # the second pair (elements 1 and 3) turns by 0.1 rad at p = 1
    out = oracle.rope(np.array([[[0.0, 2.0, 0.0, 0.0]]]), np.array([1]), 100.0)
    np.testing.assert_allclose(out[0, 0], [0.0, 2 * math.cos(0.1), 0.0, 2 * math.sin(0.1)], atol=1e-15)
    # position 0 is the identity
    X = np.random.default_rng(1).normal(size=(3, 2, 8))
    np.testing.assert_array_equal(oracle.rope(X, np.zeros(3, dtype=np.int64), 1e4), X)


def test_rope_is_a_rotation_and_relative():
    rng = np.random.default_rng(2)
    X = rng.normal(size=(5, 3, 16))
    p = np.array([0, 7, 100, 4095, 8191])
    Y = oracle.rope(X, p, 5e5)
    # each (i, i + d/2) pair keeps its length; the inverse turns it back
    half = 8
    np.testing.assert_allclose(Y[..., :half] ** 2 + Y[..., half:] ** 2, X[..., :half] ** 2 + X[..., half:] ** 2,
                               rtol=1e-12)
    np.testing.assert_allclose(oracle.rope(Y, p, 5e5, inverse=True), X, atol=1e-12)
    # the defining property: <rope(q, m), rope(k, n)> depends on m - n only
    q, k = rng.normal(size=(1, 1, 16)), rng.normal(size=(1, 1, 16))
    a = np.sum(oracle.rope(q, np.array([10]), 1e4) * oracle.rope(k, np.array([3]), 1e4))
    b = np.sum(oracle.rope(q, np.array([1007]), 1e4) * oracle.rope(k, np.array([1000]), 1e4))
    assert a == pytest.approx(b, rel=1e-10)


def test_rope_backward_matches_finite_differences():
    rng = np.random.default_rng(3)
    X, G, p = rng.normal(size=(2, 2, 6)), rng.normal(size=(2, 2, 6)), np.array([3, 11])
    dX = oracle.rope(G, p, 1e4, inverse=True)
    fd = _fd(lambda x: float(np.sum(G * oracle.rope(x, p, 1e4))), X)
    np.testing.assert_allclose(dX, fd, rtol=1e-8, atol=1e-10)
