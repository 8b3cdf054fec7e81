"""The seeded generators: determinism, block independence, and the recipes' structure."""
import numpy as np
import pytest

import workloads as wl


def test_row_blocks_equal_full_matrix_and_ld_is_irrelevant():
    full = wl.normal_matrix(37, 101, seed=7, sigma=2.0, dtype=wl.BF16)
    part = wl.normal_matrix(10, 101, seed=7, sigma=2.0, dtype=wl.BF16, row0=20)
    np.testing.assert_array_equal(full[20:30], part)
    padded = wl.normal_matrix(37, 101, seed=7, sigma=2.0, dtype=wl.BF16, ld=112)
    np.testing.assert_array_equal(padded[:, :101], full)
    assert np.all(padded[:, 101:] == 0)


def test_normal_moments_and_bf16_rounding():
    x = wl.normal_matrix(200, 1000, seed=3, sigma=2.0, dtype=wl.F32)
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 2.0) < 0.02
    b = wl.normal_matrix(200, 1000, seed=3, sigma=2.0, dtype=wl.BF16)
    np.testing.assert_array_equal(b, wl.f64_to_bf16_bits(x.astype(np.float64)))


def test_spikes_rate_and_range():
    x = wl.normal_matrix(100, 100000, seed=9, sigma=3.0, dtype=wl.F32, spike_p=1e-4,
                         spike_lo=20.0, spike_hi=30.0)
    big = x[np.abs(x) >= 20.0]
    assert 800 < big.size < 1200 and big.min() >= 20.0 and big.max() < 30.0


def test_tiny_recipe():
    c = wl.tiny()
    assert c["logits"].shape == (64, 1000) and c["logits"].dtype == np.float32
    assert int((c["labels"] == -100).sum()) == 6
    assert c["labels"].max() < 1000


def test_mistral_recipe():
    c = wl.mistral(rows=8, row0=1020)
    assert c["logits"].shape == (8, 32000) and c["logits"].dtype == np.uint16
    y = c["full_labels"]
    assert list(np.nonzero(y == -100)[0]) == [1023, 2047, 3071, 4095]
    assert c["labels"][3] == -100


def test_packed_recipe():
    y, lens = wl.packed_labels(8192, 32000, seed=wl.SEED_BASE + 3)
    assert sum(lens) == 8192 and all(1 <= L <= 1024 for L in lens)
    assert all(64 <= L for L in lens[:-1])
    pos = 0
    for L in lens:
        seg = y[pos:pos + L]
        assert seg[0] == -100
        k = int(np.argmax(seg != -100)) if (seg != -100).any() else L
        assert np.all(seg[:k] == -100) and np.all(seg[k:] != -100)
        assert 0.3 * L - 1 <= k <= 0.6 * L + 1 or L < 4
        pos += L


def test_llama3_recipe_labels_and_constant_row():
    y = wl.llama3_labels(8192, 128256, seed=wl.SEED_BASE + 4)
    assert int((y == -100).sum()) == 410 and y[wl.LLAMA3_CONST_ROW] >= 0
    c = wl.llama3(dtype=wl.F32, rows=3, row0=wl.LLAMA3_CONST_ROW - 1)
    assert np.all(c["logits"][1] == 3.0)
    assert not np.all(c["logits"][0] == 3.0)


@pytest.mark.parametrize("k", [0, 1, 5])
def test_pick_rows_exact(k):
    r = wl.pick_rows(50, k, seed=1, exclude=(3,))
    assert len(r) == k == len(set(r.tolist())) and 3 not in r
