"""Pins of the full-attention rows oracle (CPU, no GPU).

The attention over the cache plus the chunk's causal prefix ("perf(qwen3_5):
prefill text prompts in multi-token chunks", Implementation) is pinned to
closed forms and invariants:

* the first row of an empty cache sees only itself: o_0 = v_0;
* zero queries weight every visible key equally: o_t = mean of the visible v;
* one key scoring far above the rest returns its value;
* adding the same constant to every score of a row (an extra key dimension
  against a constant query component) changes nothing;
* the page's test shape: 11 rows as 7 + 4 with the cache appended in between
  equals one 11-row call, outputs and cache;
* causality: changing later rows leaves earlier outputs unchanged;
* GQA: query heads of one kv group with equal queries give equal outputs.
"""

import numpy as np

from oracle import attn_rows as ar


def _rand(seed, lengths, caches, Hq=4, Hkv=2, D=16, cap=64):
    rng = np.random.default_rng(seed)
    T, B = sum(lengths), len(lengths)
    q = rng.normal(size=(T, Hq, D))
    k = rng.normal(size=(T, Hkv, D))
    v = rng.normal(size=(T, Hkv, D))
    kc = np.zeros((B, Hkv, cap, D))
    vc = np.zeros((B, Hkv, cap, D))
    for n, c in enumerate(caches):
        kc[n, :, :c] = rng.normal(size=(Hkv, c, D))
        vc[n, :, :c] = rng.normal(size=(Hkv, c, D))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    return q, k, v, kc, vc, np.array(caches), cu


def test_first_row_of_empty_cache_returns_its_value():
    q, k, v, kc, vc, cl, cu = _rand(1, [5], [0])
    o, _, _ = ar.oracle_attn_rows(q, k, v, kc, vc, cl, cu)
    for h in range(4):
        np.testing.assert_allclose(o[0, h], v[0, h // 2], rtol=1e-13)


def test_zero_queries_average_the_visible_values():
    q, k, v, kc, vc, cl, cu = _rand(2, [6], [3])
    o, kco, vco = ar.oracle_attn_rows(np.zeros_like(q), k, v, kc, vc, cl, cu)
    for t in range(6):
        for h in range(4):
            want = vco[0, h // 2, :3 + t + 1].mean(axis=0)
            np.testing.assert_allclose(o[t, h], want, rtol=1e-12, atol=1e-14)


def test_dominant_key_returns_its_value():
    q, k, v, kc, vc, cl, cu = _rand(3, [4], [6], Hq=2, Hkv=2)
    q[:, 0] = 0.0
    q[:, 0, 0] = 1.0
    kc[0, 0, 2] = 0.0
    kc[0, 0, 2, 0] = 1e4                     # cache row 2 of kv head 0 dominates
    o, _, _ = ar.oracle_attn_rows(q, k, v, kc, vc, cl, cu)
    np.testing.assert_allclose(o[:, 0], np.repeat(vc[0, 0, 2][None], 4, axis=0), rtol=1e-12)


def test_constant_score_shift_changes_nothing():
    q, k, v, kc, vc, cl, cu = _rand(4, [7, 3], [2, 9])
    o, _, _ = ar.oracle_attn_rows(q, k, v, kc, vc, cl, cu, scale=0.25)
    # extra dimension: query component 1, key component c -> every score + 0.25 c
    pad = lambda x, val: np.concatenate([x, np.full(x.shape[:-1] + (1,), val)], axis=-1)
    o2, _, _ = ar.oracle_attn_rows(pad(q, 1.0), pad(k, 3.0), pad(v, 0.0), pad(kc, 3.0), pad(vc, 0.0), cl, cu,
                                   scale=0.25)
    np.testing.assert_allclose(o2[..., :-1], o, rtol=1e-12, atol=1e-13)


def test_11_rows_as_7_plus_4_with_cache_append():
    q, k, v, kc, vc, cl, cu = _rand(5, [11], [5])
    o, kco, vco = ar.oracle_attn_rows(q, k, v, kc, vc, cl, cu)
    o1, kc1, vc1 = ar.oracle_attn_rows(q[:7], k[:7], v[:7], kc, vc, cl, [0, 7])
    o2, kc2, vc2 = ar.oracle_attn_rows(q[7:], k[7:], v[7:], kc1, vc1, cl + 7, [0, 4])
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(kc2, kco)
    np.testing.assert_array_equal(vc2, vco)


def test_causal_rows_ignore_later_rows():
    q, k, v, kc, vc, cl, cu = _rand(6, [9], [4])
    o, _, _ = ar.oracle_attn_rows(q, k, v, kc, vc, cl, cu)
    k2, v2 = k.copy(), v.copy()
    k2[5:] += 3.0
    v2[5:] -= 2.0
    o2, _, _ = ar.oracle_attn_rows(q, k2, v2, kc, vc, cl, cu)
    np.testing.assert_array_equal(o2[:5], o[:5])
    assert np.abs(o2[5:] - o[5:]).max() > 1e-3


def test_gqa_group_heads_with_equal_queries_agree():
    q, k, v, kc, vc, cl, cu = _rand(7, [8], [3], Hq=4, Hkv=2)
    q[:, 1] = q[:, 0]
    o, _, _ = ar.oracle_attn_rows(q, k, v, kc, vc, cl, cu)
    np.testing.assert_array_equal(o[:, 1], o[:, 0])
    assert np.abs(o[:, 2] - o[:, 0]).max() > 1e-3
