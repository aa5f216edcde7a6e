"""Pins of the RWKV-4 WKV rows oracle (CPU, no GPU).

The decoder recurrence of "perf(rwkv): prefill text prompts in multi-token
chunks" (Implementation) is pinned to things other than itself:

* brute force: without max shifting, in float64 on small exponents, the
  outputs are the explicit sums (A_{t-1} + e^{u+k_t} v_t) / (B_{t-1} + e^{u+k_t})
  with A_{t-1} = e^{t w} A_{-1} + sum_{i<t} e^{(t-1-i) w + k_i} v_i;
* the page's chunk form (per-row max shift over the incoming state, earlier
  rows and bonus, the 65 x 64 distance table, row S as the new state) for
  every chunk size, including the page's 64 + 11 test shape and large keys;
* closed forms: w -> -inf keeps only the previous row and the bonus; equal
  values give that value back; a huge bonus returns v_t;
* the state is a representation: (num c, den c, max - log c) gives the same
  outputs; empty sequences keep their state.
"""

import numpy as np
import pytest

from oracle import wkv_rows as wr


def _rand(seed, T, C, B=1, big=0.0):
    rng = np.random.default_rng(seed)
    k = rng.normal(size=(T, C))
    if big:
        m = rng.random((T, C)) < big
        k = np.where(m, np.sign(rng.normal(size=(T, C))) * rng.uniform(20, 40, (T, C)), k)
    v = rng.normal(size=(T, C))
    w = -np.exp(rng.uniform(-5, 3, C))
    u = rng.normal(0.5, 1.0, C)
    den = np.exp(rng.normal(size=(B, C)))
    st = np.stack([den * rng.normal(size=(B, C)), den, rng.normal(0, 2, (B, C))], axis=1)
    return k, v, w, u, st


def _close_state(s1, s2, tol=1e-12):
    for x, y in zip(wr.state_invariants(s1), wr.state_invariants(s2)):
        fin = np.isfinite(y)
        assert np.array_equal(fin, np.isfinite(x))
        np.testing.assert_allclose(x[fin], y[fin], rtol=tol, atol=tol)


def test_brute_force_sums_without_shift():
    k, v, w, u, st = _rand(1, 12, 3)
    w = -np.exp(np.random.default_rng(2).uniform(-2, 0.5, 3))
    wkv, s_out = wr.oracle_wkv_rows(k, v, w, u, [0, 12], st)
    A0 = st[0, 0] * np.exp(st[0, 2])
    B0 = st[0, 1] * np.exp(st[0, 2])
    for t in range(12):
        A = np.exp(t * w) * A0 + sum(np.exp((t - 1 - i) * w + k[i]) * v[i] for i in range(t))
        Bs = np.exp(t * w) * B0 + sum(np.exp((t - 1 - i) * w + k[i]) for i in range(t))
        want = (A + np.exp(u + k[t]) * v[t]) / (Bs + np.exp(u + k[t]))
        np.testing.assert_allclose(wkv[t], want, rtol=1e-12)
    A_end = np.exp(12 * w) * A0 + sum(np.exp((11 - i) * w + k[i]) * v[i] for i in range(12))
    B_end = np.exp(12 * w) * B0 + sum(np.exp((11 - i) * w + k[i]) for i in range(12))
    np.testing.assert_allclose(s_out[0, 0] * np.exp(s_out[0, 2]), A_end, rtol=1e-12)
    np.testing.assert_allclose(s_out[0, 1] * np.exp(s_out[0, 2]), B_end, rtol=1e-12)


@pytest.mark.parametrize("chunk", [1, 2, 5, 16, 33, 64])
def test_page_chunk_form_equals_row_loop(chunk):
    k, v, w, u, st = _rand(3, 150, 5, B=3, big=0.05)
    cu = [0, 75, 75, 150]
    a, sa = wr.oracle_wkv_rows(k, v, w, u, cu, st)
    b, sb = wr.page_chunk_rows(k, v, w, u, cu, st, chunk=chunk)
    np.testing.assert_allclose(b, a, rtol=1e-11, atol=1e-12)
    _close_state(sb, sa, tol=1e-11)


def test_75_rows_as_64_plus_11_with_state():
    k, v, w, u, st = _rand(4, 75, 8, big=0.05)
    a, sa = wr.oracle_wkv_rows(k, v, w, u, [0, 75], st)
    a1, s1 = wr.oracle_wkv_rows(k[:64], v[:64], w, u, [0, 64], st)
    a2, s2 = wr.oracle_wkv_rows(k[64:], v[64:], w, u, [0, 11], s1)
    np.testing.assert_array_equal(np.concatenate([a1, a2]), a)
    np.testing.assert_array_equal(s2, sa)


def test_no_memory_keeps_previous_row_and_bonus():
    k, v, _, u, _ = _rand(5, 20, 4)
    w = np.full(4, -1e30)
    wkv, _ = wr.oracle_wkv_rows(k, v, w, u, [0, 20], None)
    np.testing.assert_allclose(wkv[0], v[0], rtol=1e-13)
    for t in range(1, 20):
        e_prev, e_bonus = np.exp(k[t - 1]), np.exp(u + k[t])
        want = (e_prev * v[t - 1] + e_bonus * v[t]) / (e_prev + e_bonus)
        np.testing.assert_allclose(wkv[t], want, rtol=1e-12)


def test_equal_values_and_huge_bonus():
    k, _, w, u, st = _rand(6, 40, 3, big=0.1)
    st[:, 0] = 2.5 * st[:, 1]
    wkv, s_out = wr.oracle_wkv_rows(k, np.full_like(k, 2.5), w, u, [0, 40], st)
    np.testing.assert_allclose(wkv, 2.5, rtol=1e-13)
    np.testing.assert_allclose(wr.state_invariants(s_out)[0], 2.5, rtol=1e-13)
    _, v, _, _, _ = _rand(7, 40, 3)
    wkv2, _ = wr.oracle_wkv_rows(k, v, w, np.full(3, 400.0), [0, 40], st)
    np.testing.assert_allclose(wkv2, v, rtol=1e-12)


def test_state_representation_invariance():
    k, v, w, u, st = _rand(8, 50, 6)
    c = np.exp(np.random.default_rng(9).normal(0, 3, (1, 6)))
    st2 = st.copy()
    st2[:, 0] *= c
    st2[:, 1] *= c
    st2[:, 2] -= np.log(c)
    a, sa = wr.oracle_wkv_rows(k, v, w, u, [0, 50], st)
    b, sb = wr.oracle_wkv_rows(k, v, w, u, [0, 50], st2)
    np.testing.assert_allclose(b, a, rtol=1e-12)
    _close_state(sb, sa, tol=1e-12)


def test_empty_sequence_and_absent_state():
    k, v, w, u, st = _rand(10, 30, 4, B=3)
    _, s = wr.oracle_wkv_rows(k, v, w, u, [0, 10, 10, 30], st)
    np.testing.assert_array_equal(s[1], st[1])
    _, s0 = wr.oracle_wkv_rows(k, v, w, u, [0, 10, 10, 30], None)
    np.testing.assert_array_equal(s0[1], [[0.0] * 4, [0.0] * 4, [wr.EMPTY_MAX] * 4])


def test_large_keys_stay_finite():
    k, v, w, u, st = _rand(11, 500, 8, big=0.3)
    wkv, s = wr.oracle_wkv_rows(k, v, w, u, [0, 500], st)
    assert np.all(np.isfinite(wkv)) and np.all(np.isfinite(s))
    assert np.all(np.abs(wkv) <= np.abs(v).max() + np.abs(st[0, 0] / st[0, 1]).max() + 1e-9)
