"""Pins of the selective-scan rows oracle (CPU, no GPU).

The recurrence h_t = a_t h_{t-1} + b_t of add_selective_scan_rows ("perf(mamba):
prefill text prompts in multi-token chunks", Implementation) is pinned to
things other than itself:

* closed forms: a = 1 gives running sums, b = 0 gives running products,
  constant a and b give the geometric series, and the end state equals the
  explicit sum of products for tiny inputs (brute force);
* the page's own algorithm (chunks of at most 64 rows, ceil(log2 S) doubling
  rounds with an identity pad, then the incoming state) for every chunk size;
* the page's test shape: 75 rows as 64 + 11 with the state carried equals the
  unsplit run; empty sequences keep their state; linearity in (b, h_0).
"""

import numpy as np
import pytest

from oracle import scan_rows as sr


def _rand(seed, T, C, B=1):
    rng = np.random.default_rng(seed)
    a = np.exp(-np.log1p(np.exp(rng.normal(-1.0, 1.0, (T, C)))))
    b = rng.normal(size=(T, C))
    h0 = rng.normal(0, 0.3, (B, C))
    return a, b, h0


def test_unit_decay_is_running_sum():
    _, b, h0 = _rand(1, 40, 3)
    rows, out = sr.oracle_scan_rows(np.ones_like(b), b, [0, 40], h0)
    np.testing.assert_allclose(rows, h0 + np.cumsum(b, axis=0), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[0], rows[-1], rtol=0, atol=0)


def test_zero_input_is_running_product():
    a, _, h0 = _rand(2, 33, 4)
    rows, _ = sr.oracle_scan_rows(a, np.zeros_like(a), [0, 33], h0)
    np.testing.assert_allclose(rows, h0 * np.cumprod(a, axis=0), rtol=1e-13, atol=0)


def test_constant_coefficients_geometric_series():
    alpha, beta, h0, T = 0.9, 0.5, 2.0, 50
    rows, _ = sr.oracle_scan_rows(np.full((T, 1), alpha), np.full((T, 1), beta), [0, T], [[h0]])
    t = np.arange(1, T + 1)
    want = alpha ** t * h0 + beta * (1 - alpha ** t) / (1 - alpha)
    np.testing.assert_allclose(rows[:, 0], want, rtol=1e-13)


def test_end_state_is_explicit_sum_of_products():
    """Brute force: h_T = (prod_i a_i) h_0 + sum_j (prod_{i>j} a_i) b_j."""
    a, b, h0 = _rand(3, 9, 2)
    _, out = sr.oracle_scan_rows(a, b, [0, 9], h0)
    want = np.prod(a, axis=0) * h0[0]
    for j in range(9):
        want = want + np.prod(a[j + 1:], axis=0) * b[j]
    np.testing.assert_allclose(out[0], want, rtol=1e-13)


@pytest.mark.parametrize("chunk", [1, 2, 3, 7, 16, 63, 64])
def test_page_doubling_scan_equals_row_loop(chunk):
    a, b, h0 = _rand(4, 150, 6, B=3)
    cu = [0, 70, 70, 150]
    r1, o1 = sr.oracle_scan_rows(a, b, cu, h0)
    r2, o2 = sr.hillis_steele_rows(a, b, cu, h0, chunk=chunk)
    np.testing.assert_allclose(r2, r1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-12)


def test_75_rows_as_64_plus_11():
    a, b, h0 = _rand(5, 75, 8)
    r_all, o_all = sr.oracle_scan_rows(a, b, [0, 75], h0)
    r1, o1 = sr.oracle_scan_rows(a[:64], b[:64], [0, 64], h0)
    r2, o2 = sr.oracle_scan_rows(a[64:], b[64:], [0, 11], o1)
    np.testing.assert_array_equal(np.concatenate([r1, r2]), r_all)
    np.testing.assert_array_equal(o2, o_all)


def test_empty_sequence_and_null_state():
    a, b, h0 = _rand(6, 20, 4, B=3)
    rows, out = sr.oracle_scan_rows(a, b, [0, 10, 10, 20], h0)
    np.testing.assert_array_equal(out[1], h0[1])
    rz, oz = sr.oracle_scan_rows(a, b, [0, 10, 10, 20], None)
    rz2, oz2 = sr.oracle_scan_rows(a, b, [0, 10, 10, 20], np.zeros_like(h0))
    np.testing.assert_array_equal(rz, rz2)
    np.testing.assert_array_equal(oz, oz2)


def test_linear_in_input_and_state():
    a, b, h0 = _rand(7, 30, 5)
    _, b2, h2 = _rand(8, 30, 5)
    r1, _ = sr.oracle_scan_rows(a, b, [0, 30], h0)
    r2, _ = sr.oracle_scan_rows(a, b2, [0, 30], h2)
    r3, _ = sr.oracle_scan_rows(a, 2 * b - 3 * b2, [0, 30], 2 * h0 - 3 * h2)
    np.testing.assert_allclose(r3, 2 * r1 - 3 * r2, rtol=1e-12, atol=1e-12)


def test_decays_keep_state_bounded():
    """Every factor is a decay in (0, 1] (the page's argument for finiteness):
    |h_t| <= |h_0| + sum |b|."""
    a, b, h0 = _rand(9, 500, 4)
    rows, _ = sr.oracle_scan_rows(a, b, [0, 500], h0)
    assert np.all(np.abs(rows) <= np.abs(h0) + np.cumsum(np.abs(b), axis=0) + 1e-12)
