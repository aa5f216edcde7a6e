"""Pins for the float64 oracle (CPU only).

The oracle is checked against facts that do not come from the oracle itself:
closed forms, special cases, invariants, brute force with a different
formulation, and library routines.  Each test says what it pins.  Citations
name the page and section the fact comes from:

* QWEN = "perf(qwen3_5): prefill text prompts in multi-token chunks"
  (TensorRT-Model-Connect pull request 2191);
* MAMBA = "perf(mamba): prefill text prompts in multi-token chunks"
  (pull request 2184);
* RWKV = "perf(rwkv): prefill text prompts in multi-token chunks"
  (pull request 2192).
"""

import numpy as np
import pytest

from oracle import chunk_form as cf
from oracle import oracle_l2norm, oracle_prefill, oracle_short_conv, oracle_step

RTOL = 1e-10


def _unit(a):
    return a / np.linalg.norm(a, axis=-1, keepdims=True)


def _rand_problem(rng, lengths, Hk, Hv, dk, dv, g_scale=1.0, s0=True):
    T = int(sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q = _unit(rng.standard_normal((T, Hk, dk)))
    k = _unit(rng.standard_normal((T, Hk, dk)))
    v = rng.standard_normal((T, Hv, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, Hv))))
    g = -np.log1p(np.exp(rng.standard_normal((T, Hv)))) * g_scale
    S0 = rng.standard_normal((len(lengths), Hv, dk, dv)) * 0.1 if s0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, cu=cu, S0=S0, Hk=Hk, Hv=Hv, dk=dk, dv=dv)


def _run_loop(p, **kw):
    return oracle_prefill(p["q"], p["k"], p["v"], p["g"], p["beta"], p["cu"], p["Hk"], p["Hv"],
                          p["dk"], p["dv"], state_in=p["S0"], use_l2norm=kw.pop("use_l2norm", False),
                          **kw)


def _close(a, b, rtol=RTOL):
    scale = max(np.abs(b).max(), 1e-300)
    assert np.abs(a - b).max() <= rtol * scale, (np.abs(a - b).max(), scale)


# --------------------------------------------------------------------------
# Brute force: the token loop against the matrix recurrence as the pages state it
#   S_t = exp(g_t)(I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T, o_t = S_t^T q_t
# written as dense matrix products (a different formulation of the step).
# Pins: decay placement, the sign and beta placement of the delta update, and
# that the output uses the updated state.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(4))
def test_token_loop_matches_dense_transition_products(seed):
    rng = np.random.default_rng(seed)
    dk, dv = int(rng.integers(1, 9)), int(rng.integers(1, 9))
    p = _rand_problem(rng, [13], 1, 1, dk, dv)
    res = _run_loop(p)
    S = p["S0"][0, 0].copy()
    for t in range(13):
        kt, vt, qt = p["k"][t, 0], p["v"][t, 0], p["q"][t, 0]
        M = np.exp(p["g"][t, 0]) * (np.eye(dk) - p["beta"][t, 0] * np.outer(kt, kt))
        S = M @ S + p["beta"][t, 0] * np.outer(kt, vt)
        _close(res["out"][t, 0], S.T @ qt)
    _close(res["state_out"][0, 0], S)


# --------------------------------------------------------------------------
# QWEN, Implementation: the chunked closed form equals the token loop.  Both
# triangular inverses (forward substitution; blocked 8x8 Neumann + 2x2 levels)
# and numpy.linalg.inv.  Random GQA, ragged lengths (including an empty
# sequence), several chunk sizes.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed,chunk,inverse", [
    (0, 64, "block"), (1, 64, "forward"), (2, 1, "block"), (3, 8, "numpy"),
    (4, 16, "block"), (5, 33, "forward"), (6, 64, "numpy"), (7, 5, "block")])
def test_chunk_form_equals_token_loop(seed, chunk, inverse):
    rng = np.random.default_rng(100 + seed)
    Hk = int(rng.integers(1, 3))
    Hv = Hk * int(rng.integers(1, 3))
    dk, dv = int(rng.integers(1, 17)), int(rng.integers(1, 17))
    lengths = [int(x) for x in rng.integers(1, 131, size=3)] + [0]
    p = _rand_problem(rng, lengths, Hk, Hv, dk, dv)
    res = _run_loop(p)
    out, s_out = cf.chunk_prefill(p["q"], p["k"], p["v"], p["g"], p["beta"], p["cu"], Hk, Hv,
                                  state_in=p["S0"], chunk=chunk, inverse=inverse)
    _close(out, res["out"])
    _close(s_out, res["state_out"])


def test_chunk_of_one_row_is_the_token_step():
    """With chunk = 1 the closed form is exactly one token step: A is empty,
    U = beta (v - Gamma S^T k) and S_S = exp(g) S + k U^T."""
    rng = np.random.default_rng(7)
    p = _rand_problem(rng, [9], 1, 1, 6, 5)
    S = p["S0"][0, 0]
    for t in range(9):
        sl = slice(t, t + 1)
        O, S_next = cf.chunk_step(p["q"][sl, 0], p["k"][sl, 0], p["v"][sl, 0], p["g"][sl, 0],
                                  p["beta"][sl, 0], S)
        one = dict(p, q=p["q"][sl], k=p["k"][sl], v=p["v"][sl], g=p["g"][sl],
                   beta=p["beta"][sl], cu=np.array([0, 1], np.int32), S0=S[None, None])
        ref = _run_loop(one)
        _close(O, ref["out"][:, 0])
        _close(S_next, ref["state_out"][0, 0])
        S = S_next


@pytest.mark.parametrize("chunks", [(1, 8, 16, 32, 64)])
def test_chunk_size_invariance(chunks):
    """Results do not depend on where the prompt is cut (QWEN, Notes For
    Future Readers: longer prompts run several chunks)."""
    rng = np.random.default_rng(11)
    p = _rand_problem(rng, [130], 1, 1, 8, 8)
    ref = None
    for c in chunks:
        o, s = cf.chunk_prefill_head(p["q"][:, 0], p["k"][:, 0], p["v"][:, 0], p["g"][:, 0],
                                     p["beta"][:, 0], p["S0"][0, 0], chunk=c)
        if ref is None:
            ref = (o, s)
        else:
            _close(o, ref[0])
            _close(s, ref[1])


# --------------------------------------------------------------------------
# RWKV / MAMBA Tests: a 75-token prompt prefilled as 64 + 11 rows equals the
# unsplit run; QWEN Tests: 11 tokens as 7 + 4.  Here: two chained oracle calls
# (state and conv state carried) equal one call.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("total,first", [(75, 64), (11, 7)])
def test_split_prompt_equals_unsplit(total, first):
    rng = np.random.default_rng(total)
    Hk, Hv, dk, dv, K = 1, 2, 8, 4, 4
    C = 2 * Hk * dk + Hv * dv
    x = rng.standard_normal((total, C))
    w = rng.uniform(-0.5, 0.5, (C, K))
    cs = rng.standard_normal((1, C, K - 1))
    g = -np.log1p(np.exp(rng.standard_normal((total, Hv))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((total, Hv))))
    S0 = rng.standard_normal((1, Hv, dk, dv)) * 0.1
    full = oracle_prefill(None, None, None, g, beta, [0, total], Hk, Hv, dk, dv, state_in=S0,
                          conv=dict(x=x, w=w, state_in=cs, act=1))
    a = oracle_prefill(None, None, None, g[:first], beta[:first], [0, first], Hk, Hv, dk, dv,
                       state_in=S0, conv=dict(x=x[:first], w=w, state_in=cs, act=1))
    b = oracle_prefill(None, None, None, g[first:], beta[first:], [0, total - first], Hk, Hv, dk,
                       dv, state_in=a["state_out"],
                       conv=dict(x=x[first:], w=w, state_in=a["conv_state_out"], act=1))
    _close(np.concatenate([a["out"], b["out"]]), full["out"], 1e-12)
    _close(b["state_out"], full["state_out"], 1e-12)
    _close(b["conv_state_out"], full["conv_state_out"], 0)
    # and the closed form with 64-row chunks (64 + 11 internally) agrees
    if total == 75:
        y, _ = oracle_short_conv(x, w, [0, total], cs, act=1)
        qn = oracle_l2norm(y[:, :dk].reshape(total, 1, dk))
        kn = oracle_l2norm(y[:, dk:2 * dk].reshape(total, 1, dk))
        vv = y[:, 2 * dk:].reshape(total, Hv, dv)
        out, s = cf.chunk_prefill(qn, kn, vv, g, beta, [0, total], Hk, Hv, state_in=S0, chunk=64)
        _close(out, full["out"])
        _close(s, full["state_out"])


# --------------------------------------------------------------------------
# Special cases and closed forms of the recurrence.
# --------------------------------------------------------------------------
def test_zero_decay_zero_beta_keeps_state():
    """g = 0, beta = 0: the state is unchanged and o_t = S_0^T q_t."""
    rng = np.random.default_rng(1)
    p = _rand_problem(rng, [20, 7], 2, 4, 8, 6)
    p["g"][:] = 0.0
    p["beta"][:] = 0.0
    res = _run_loop(p)
    assert np.array_equal(res["state_out"], p["S0"])
    for n, (a, e) in enumerate([(0, 20), (20, 27)]):
        for h in range(4):
            ref = p["q"][a:e, h // 2] @ p["S0"][n, h]
            _close(res["out"][a:e, h], ref)


def test_pure_decay_closed_form():
    """beta = 0: S_T = exp(sum g) S_0 and o_t = exp(sum_{i<=t} g_i) S_0^T q_t."""
    rng = np.random.default_rng(2)
    p = _rand_problem(rng, [30], 1, 1, 5, 3)
    p["beta"][:] = 0.0
    res = _run_loop(p)
    gam = np.cumsum(p["g"][:, 0])
    _close(res["state_out"][0, 0], np.exp(gam[-1]) * p["S0"][0, 0])
    _close(res["out"][:, 0], np.exp(gam)[:, None] * (p["q"][:, 0] @ p["S0"][0, 0]))


def test_delta_rule_projection():
    """beta = 1 and unit keys: after each step k_t^T S_t = v_t^T exactly (the
    delta rule overwrites the value stored under k_t), for any decay.  With
    q_t = k_t the output is therefore v_t."""
    rng = np.random.default_rng(3)
    p = _rand_problem(rng, [40], 1, 1, 7, 5)
    p["beta"][:] = 1.0
    p["q"] = p["k"].copy()
    res = _run_loop(p)
    _close(res["out"][:, 0], p["v"][:, 0], 1e-12)


def test_parallel_keys_closed_form():
    """All keys one unit vector k, beta = 1, g = 0 (the near-parallel hazard
    of QWEN, Implementation, taken to the limit):
    S_t = (I - k k^T) S_0 + k v_t^T and o_t = S_0^T (I - k k^T) q_t + (k.q_t) v_t.
    In the chunk form I + A is I plus ones below the diagonal, whose inverse is
    I minus the first subdiagonal; both inverses must give it exactly."""
    rng = np.random.default_rng(4)
    dk, dv, T = 6, 4, 64
    kvec = _unit(rng.standard_normal(dk))
    p = _rand_problem(rng, [T], 1, 1, dk, dv)
    p["k"][:] = kvec
    p["beta"][:] = 1.0
    p["g"][:] = 0.0
    res = _run_loop(p)
    P = np.eye(dk) - np.outer(kvec, kvec)
    S0 = p["S0"][0, 0]
    for t in range(T):
        ref = S0.T @ P @ p["q"][t, 0] + (kvec @ p["q"][t, 0]) * p["v"][t, 0]
        _close(res["out"][t, 0], ref, 1e-12)
    _close(res["state_out"][0, 0], P @ S0 + np.outer(kvec, p["v"][-1, 0]), 1e-12)
    L = np.eye(T) + np.tril(np.ones((T, T)), -1)
    expect = np.eye(T) - np.eye(T, k=-1)
    assert np.array_equal(cf.inv_block_neumann(L), expect)
    assert np.array_equal(cf.inv_forward_sub(L), expect)


def test_single_token_from_zero_state():
    """One token from a zero state: S = beta k v^T and o = beta (k.q) v."""
    rng = np.random.default_rng(5)
    p = _rand_problem(rng, [1], 1, 1, 9, 7, s0=False)
    res = _run_loop(p)
    b, kt, vt, qt = p["beta"][0, 0], p["k"][0, 0], p["v"][0, 0], p["q"][0, 0]
    _close(res["state_out"][0, 0], b * np.outer(kt, vt))
    _close(res["out"][0, 0], b * (kt @ qt) * vt)


def test_linearity_in_values_and_state():
    """For fixed q, k, g, beta the map (V, S_0) -> (O, S_T) is linear."""
    rng = np.random.default_rng(6)
    p1 = _rand_problem(rng, [50, 17], 1, 2, 6, 5)
    p2 = dict(p1, v=rng.standard_normal(p1["v"].shape), S0=rng.standard_normal(p1["S0"].shape))
    a, b = 0.7, -1.9
    p3 = dict(p1, v=a * p1["v"] + b * p2["v"], S0=a * p1["S0"] + b * p2["S0"])
    r1, r2, r3 = _run_loop(p1), _run_loop(p2), _run_loop(p3)
    _close(r3["out"], a * r1["out"] + b * r2["out"], 1e-12)
    _close(r3["state_out"], a * r1["state_out"] + b * r2["state_out"], 1e-12)


def test_gqa_value_head_reads_its_key_group():
    """Value head h reads key head h // (Hv / Hk): a grouped run equals single
    head runs on the matching slices."""
    rng = np.random.default_rng(8)
    p = _rand_problem(rng, [33], 2, 6, 5, 4)
    res = _run_loop(p)
    for h in range(6):
        kh = h // 3
        one = dict(p, q=p["q"][:, kh:kh + 1], k=p["k"][:, kh:kh + 1], v=p["v"][:, h:h + 1],
                   g=p["g"][:, h:h + 1], beta=p["beta"][:, h:h + 1], S0=p["S0"][:, h:h + 1],
                   Hk=1, Hv=1)
        r = _run_loop(one)
        assert np.array_equal(r["out"][:, 0], res["out"][:, h])
        assert np.array_equal(r["state_out"][:, 0], res["state_out"][:, h])


def test_empty_sequence_passes_state_through():
    """A zero-length sequence writes no rows and returns its incoming state."""
    rng = np.random.default_rng(9)
    p = _rand_problem(rng, [5, 0, 3], 1, 1, 4, 4)
    res = _run_loop(p)
    assert np.array_equal(res["state_out"][1], p["S0"][1])


def test_decode_step_is_prefill_of_one_token():
    """oracle_step on B tokens = oracle_prefill on B sequences of one token."""
    rng = np.random.default_rng(10)
    p = _rand_problem(rng, [1, 1, 1], 2, 4, 8, 8)
    step = oracle_step(p["q"], p["k"], p["v"], p["g"], p["beta"], p["S0"], 2, 4, 8, 8,
                       use_l2norm=False)
    S = p["S0"]
    for n in range(3):
        for h in range(4):
            kt, vt, qt = p["k"][n, h // 2], p["v"][n, h], p["q"][n, h // 2]
            Sn = np.exp(p["g"][n, h]) * (S[n, h] - p["beta"][n, h] * np.outer(kt, kt @ S[n, h])) \
                + p["beta"][n, h] * np.outer(kt, vt)
            _close(step["state_out"][n, h], Sn)
            _close(step["out"][n, h], Sn.T @ qt)


# --------------------------------------------------------------------------
# QWEN Tests: the batched block inverse matches NumPy on nearly parallel keys
# with beta near one.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n", [64, 40, 11, 1])
def test_block_inverse_matches_numpy_nearly_parallel(n):
    rng = np.random.default_rng(n)
    d = _unit(rng.standard_normal(32))
    perp = rng.standard_normal((n, 32))
    perp -= np.outer(perp @ d, d)
    K = _unit(d + 0.04 * rng.uniform(0, 1, (n, 1)) * _unit(perp))
    beta = 1 / (1 + np.exp(-(6 + rng.uniform(-0.5, 0.5, n))))
    g = np.where(rng.uniform(size=n) < 0.25, -rng.uniform(0, 0.01, n), -rng.uniform(0, 0.01, n))
    gam = np.cumsum(g)
    A = np.tril(beta[:, None] * np.exp(gam[:, None] - gam[None, :]) * (K @ K.T), -1)
    L = np.eye(n) + A
    ref = np.linalg.inv(L)
    for inv in (cf.inv_block_neumann, cf.inv_forward_sub):
        X = inv(L)
        assert np.abs(X - ref).max() <= 1e-9 * np.abs(ref).max()
        assert np.abs(L @ X - np.eye(n)).max() <= 1e-9


def test_neumann_block_identity():
    """(I + N)^-1 = (I - N)(I + N^2)(I + N^4) for strictly lower 8x8 N."""
    rng = np.random.default_rng(12)
    N = np.tril(rng.standard_normal((8, 8)), -1)
    X = cf.inv_block_neumann(np.eye(8) + N, pad=8, block=8)
    assert np.abs(X @ (np.eye(8) + N) - np.eye(8)).max() < 1e-12


# --------------------------------------------------------------------------
# QWEN, gamma_S commit: gamma_S is the last cumulative sum and the end-state
# exponent is clamped at zero, so states stay finite at large decays.
# --------------------------------------------------------------------------
def test_stress_large_decays_stay_finite_and_match():
    """Nearly parallel keys, beta ~ sigmoid(6), g down to -20 per token: the
    closed form (both inverses) is finite and equals the token loop."""
    rng = np.random.default_rng(13)
    H, d, L = 2, 16, 200
    dirn = _unit(rng.standard_normal((H, d)))
    perp = rng.standard_normal((L, H, d))
    perp -= (perp * dirn).sum(-1, keepdims=True) * dirn
    k = _unit(dirn + 0.04 * rng.uniform(0, 1, (L, H, 1)) * _unit(perp))
    q = _unit(rng.standard_normal((L, H, d)))
    v = rng.standard_normal((L, H, d))
    beta = 1 / (1 + np.exp(-(6 + rng.uniform(-0.5, 0.5, (L, H)))))
    g = np.where(rng.uniform(size=(L, H)) < 0.25, -rng.uniform(0, 0.01, (L, H)),
                 -rng.uniform(0, 20, (L, H)))
    S0 = rng.standard_normal((1, H, d, d)) * 0.1
    ref = oracle_prefill(q, k, v, g, beta, [0, L], H, H, d, d, state_in=S0, use_l2norm=False)
    for inv in ("block", "forward"):
        out, s = cf.chunk_prefill(q, k, v, g, beta, [0, L], H, H, state_in=S0, chunk=64,
                                  inverse=inv)
        assert np.isfinite(out).all() and np.isfinite(s).all()
        _close(out, ref["out"], 1e-9)
        _close(s, ref["state_out"], 1e-9)


def test_gamma_S_clamp_bounds_end_state_weights():
    """Negative control for the clamp.  In half precision a gamma_S reduced in
    another order (here: summed backwards) differs from the last cumulative
    sum by ulps of |gamma| ~ 10^3, so exp(gamma_S - gamma_i) exceeds one (and
    overflows once the excess passes the format's exponent range); with
    gamma_S the last cumulative sum and the exponent clamped at zero every
    weight stays in (0, 1]."""
    for seed in range(100):
        rng = np.random.default_rng(seed)
        g = (-rng.uniform(0, 20, 64)).astype(np.float16)
        gam = np.cumsum(g, dtype=np.float16)
        gS_sep = np.float16(0)
        for x in g[::-1]:
            gS_sep = np.float16(gS_sep + x)
        if gS_sep > gam[-1]:
            break
    else:
        pytest.fail("no seed where the backward sum exceeds the forward one")
    unclamped = np.exp((gS_sep - gam).astype(np.float32))
    assert unclamped.max() > 1.0                       # the separate reduction exceeds gamma_i
    clamped = cf.state_decay_weights(gam.astype(np.float64), float(gS_sep))
    assert np.isfinite(clamped).all() and clamped.max() <= 1.0
    last = cf.state_decay_weights(gam.astype(np.float64), float(gam[-1]))
    assert np.isfinite(last).all() and last.max() <= 1.0 and last[-1] == 1.0


# --------------------------------------------------------------------------
# MAMBA, Implementation (add_short_conv_rows): the depthwise causal conv over
# the previous kernel-1 conv-state columns plus the chunk; the new conv state
# is the last kernel-1 columns.
# --------------------------------------------------------------------------
def test_conv_identity_tap_and_state_out():
    rng = np.random.default_rng(15)
    T, C, K = 10, 5, 4
    x = rng.standard_normal((T, C))
    w = np.zeros((C, K))
    w[:, K - 1] = 1.0                      # tap K-1 weighs the current token
    s_in = rng.standard_normal((1, C, K - 1))
    y, s_out = oracle_short_conv(x, w, [0, T], s_in)
    assert np.array_equal(y, x)
    assert np.array_equal(s_out[0], x[-(K - 1):].T)


def test_conv_zero_input_reads_state_taps_only():
    rng = np.random.default_rng(16)
    T, C, K = 6, 3, 4
    w = rng.standard_normal((C, K))
    s_in = rng.standard_normal((1, C, K - 1))
    y, s_out = oracle_short_conv(np.zeros((T, C)), w, [0, T], s_in)
    for t in range(T):
        for c in range(C):
            ref = sum(w[c, j] * s_in[0, c, t + j] for j in range(K) if t + j < K - 1)
            assert abs(y[t, c] - ref) <= 1e-15
    assert np.array_equal(s_out, np.zeros_like(s_out)) or T < K - 1


def test_conv_matches_numpy_convolve_and_short_sequences():
    """Against numpy.convolve of [state ++ x] with the reversed taps, for
    sequence lengths shorter than, equal to and longer than K - 1 (the new
    state then mixes old state and new columns)."""
    rng = np.random.default_rng(17)
    C, K = 3, 4
    lengths = [1, 2, 3, 9, 0]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    x = rng.standard_normal((cu[-1], C))
    w = rng.standard_normal((C, K))
    s_in = rng.standard_normal((len(lengths), C, K - 1))
    y, s_out = oracle_short_conv(x, w, cu, s_in)
    for n, L in enumerate(lengths):
        for c in range(C):
            xx = np.concatenate([s_in[n, c], x[cu[n]:cu[n + 1], c]])
            if L > 0:
                ref = np.convolve(xx, w[c, ::-1], mode="valid")
                assert np.abs(y[cu[n]:cu[n + 1], c] - ref).max() <= 1e-14
            assert np.array_equal(s_out[n, c], xx[-(K - 1):])


def test_conv_silu_activation():
    """SiLU(y) = y * sigmoid(y), checked against scipy's expit."""
    from scipy.special import expit
    rng = np.random.default_rng(18)
    x = rng.standard_normal((7, 2)) * 3
    w = np.zeros((2, 4))
    w[:, 3] = 1.0
    y, _ = oracle_short_conv(x, w, [0, 7], None, act=1)
    assert np.abs(y - x * expit(x)).max() <= 1e-14


def test_l2norm_values():
    """x / sqrt(sum x^2 + eps): (3, 4) -> (3, 4)/sqrt(25 + eps); scale
    invariance for norms far above sqrt(eps)."""
    out = oracle_l2norm(np.array([[3.0, 4.0]]), eps=1e-6)
    assert np.allclose(out, np.array([[3.0, 4.0]]) / np.sqrt(25 + 1e-6), rtol=0, atol=1e-16)
    rng = np.random.default_rng(19)
    x = rng.standard_normal((5, 16))
    a, b = oracle_l2norm(x, eps=0.0), oracle_l2norm(7.5 * x, eps=0.0)
    assert np.abs(a - b).max() < 1e-15
    assert np.abs(np.linalg.norm(a, axis=1) - 1).max() < 1e-15


def test_prefill_composes_conv_then_l2norm_then_recurrence():
    """The full oracle = short conv -> L2 norm of q and k -> token loop."""
    rng = np.random.default_rng(20)
    Hk, Hv, dk, dv, K = 1, 2, 8, 4, 4
    C = 2 * Hk * dk + Hv * dv
    lengths = [9, 3]
    cu = np.array([0, 9, 12], np.int32)
    x = rng.standard_normal((12, C))
    w = rng.uniform(-0.5, 0.5, (C, K))
    cs = rng.standard_normal((2, C, K - 1))
    g = -np.log1p(np.exp(rng.standard_normal((12, Hv))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((12, Hv))))
    S0 = rng.standard_normal((2, Hv, dk, dv)) * 0.1
    full = oracle_prefill(None, None, None, g, beta, cu, Hk, Hv, dk, dv, state_in=S0,
                          conv=dict(x=x, w=w, state_in=cs, act=0), use_l2norm=True, q_scale=0.5)
    y, s_out = oracle_short_conv(x, w, cu, cs)
    q = oracle_l2norm(y[:, :dk].reshape(12, 1, dk))
    k = oracle_l2norm(y[:, dk:2 * dk].reshape(12, 1, dk))
    v = y[:, 2 * dk:].reshape(12, Hv, dv)
    ref = oracle_prefill(q, k, v, g, beta, cu, Hk, Hv, dk, dv, state_in=S0, use_l2norm=False,
                         q_scale=0.5)
    assert np.array_equal(full["conv_state_out"], s_out)
    _close(full["out"], ref["out"], 1e-14)
    _close(full["state_out"], ref["state_out"], 1e-14)
    assert len(lengths) == 2
