"""Float64 chunked closed form of the gated delta rule — TEST INFRASTRUCTURE.

This is the method of the Qwen3.5 chunked-prefill pull request ("perf(qwen3_5):
prefill text prompts in multi-token chunks", Implementation section), written
out step by step in NumPy float64 for one (sequence, head).  It exists to pin
the token-loop oracle (the two must agree to rounding) and to localise GPU
errors; it is not the parity reference for the GPU.

Per chunk of n <= 64 rows with incoming state S_0 [dk, dv]:

    gamma_t = sum_{i<=t} g_i,   Gamma_t = exp(gamma_t)
    (I + A) U = diag(beta) V - diag(beta Gamma) K S_0,
        A_ij = beta_i exp(gamma_i - gamma_j) k_i . k_j   (j < i, else 0)
    O   = diag(Gamma) Q S_0 + (exp(gamma_t - gamma_i) q_t . k_i)_{i <= t} U
    S_S = exp(gamma_S) S_0 + (K * exp(min(gamma_S - gamma, 0)))^T U

with gamma_S the last cumulative sum and the end-state exponent clamped at
zero (the page's gamma_S commit message).  I + A is inverted on a fixed 64-row
padding whose padded rows are identity: 8x8 diagonal blocks by a Neumann
product, then 2x2 block inversion level by level (Implementation section).
Exponentials are evaluated only where the triangular masks keep the entry.
"""

from __future__ import annotations

import numpy as np

PAD_ROWS = 64      # the static padding of the triangular solve
NEUMANN_BLOCK = 8  # diagonal block size of the Neumann stage


def cumulative_decay(g):
    """gamma_t = sum_{i<=t} g_i over one chunk (inclusive prefix sum)."""
    return np.cumsum(np.asarray(g, dtype=np.float64))


def inv_forward_sub(L):
    """Inverse of a unit lower-triangular matrix by forward substitution
    (textbook: solve L x = e_c column by column)."""
    L = np.asarray(L, dtype=np.float64)
    n = L.shape[0]
    X = np.zeros_like(L)
    for c in range(n):
        for i in range(n):
            acc = 1.0 if i == c else 0.0
            for j in range(i):
                acc -= L[i, j] * X[j, c]
            X[i, c] = acc
    return X


def inv_block_neumann(L, pad=PAD_ROWS, block=NEUMANN_BLOCK):
    """Inverse of a unit lower-triangular n x n matrix (n <= pad) the way the
    page describes it.

    1. Pad to ``pad`` rows; the padded rows and columns are identity.
    2. Each diagonal ``block`` x ``block`` block is I + N with N strictly lower
       triangular, so N^block = 0 and
       (I + N)^-1 = (I - N)(I + N^2)(I + N^4)   (for block = 8).
    3. Level by level (8 -> 16 -> 32 -> 64), every diagonal pair of inverted
       blocks is combined by 2x2 block inversion
       [[L11, 0], [L21, L22]]^-1 = [[L11^-1, 0], [-L22^-1 L21 L11^-1, L22^-1]],
       all blocks of a level at once.
    """
    L = np.asarray(L, dtype=np.float64)
    n = L.shape[0]
    assert n <= pad and pad % block == 0
    P = np.eye(pad)
    P[:n, :n] = L
    inv = np.zeros((pad, pad))
    eye = np.eye(block)
    nb = pad // block
    # Stage 1: Neumann product on every diagonal block (batched).
    diag = np.stack([P[b * block:(b + 1) * block, b * block:(b + 1) * block] for b in range(nb)])
    N = diag - eye
    factor = eye - N
    power = N
    k = 1
    while 2 * k < block:          # multiply in (I + N^2), (I + N^4), ...
        power = power @ power
        factor = factor @ (eye + power)
        k *= 2
    for b in range(nb):
        inv[b * block:(b + 1) * block, b * block:(b + 1) * block] = factor[b]
    # Stage 2: 2x2 block inversion, level by level.
    size = block
    while size < pad:
        for b in range(pad // (2 * size)):
            o = b * 2 * size
            top = slice(o, o + size)
            bot = slice(o + size, o + 2 * size)
            inv[bot, top] = -inv[bot, bot] @ P[bot, top] @ inv[top, top]
        size *= 2
    return inv[:n, :n]


def inv_numpy(L):
    """Library inverse (numpy.linalg.inv), the page's test comparison."""
    return np.linalg.inv(np.asarray(L, dtype=np.float64))


_INVERSES = {"forward": inv_forward_sub, "block": inv_block_neumann, "numpy": inv_numpy}


def state_decay_weights(gamma, gamma_S, clamp=True):
    """exp(gamma_S - gamma_i), clamped at exponent zero (the gamma_S commit):
    the factor by which row i's contribution reaches the chunk's end state."""
    e = np.asarray(gamma_S) - np.asarray(gamma)
    if clamp:
        e = np.minimum(e, 0)
    return np.exp(e)


def chunk_step(Q, K, V, g, beta, S0, inverse="block"):
    """Solve one chunk of n <= 64 rows in closed form.

    Q, K [n, dk]; V [n, dv]; g, beta [n]; S0 [dk, dv].  Returns (O [n, dv],
    S_S [dk, dv])."""
    Q, K, V = (np.asarray(a, dtype=np.float64) for a in (Q, K, V))
    b = np.asarray(beta, dtype=np.float64)
    S0 = np.asarray(S0, dtype=np.float64)
    n = K.shape[0]
    gam = cumulative_decay(g)
    Gam = np.exp(gam)
    # A_ij = beta_i exp(gamma_i - gamma_j) k_i . k_j on the strict lower triangle.
    A = np.zeros((n, n))
    il, jl = np.tril_indices(n, -1)
    A[il, jl] = b[il] * np.exp(gam[il] - gam[jl]) * np.einsum("pd,pd->p", K[il], K[jl])
    rhs = b[:, None] * V - (b * Gam)[:, None] * (K @ S0)
    U = _INVERSES[inverse](np.eye(n) + A) @ rhs
    # Output mask: exp(gamma_t - gamma_i) q_t . k_i for i <= t.
    Mqk = np.zeros((n, n))
    it, jt = np.tril_indices(n, 0)
    Mqk[it, jt] = np.exp(gam[it] - gam[jt]) * np.einsum("pd,pd->p", Q[it], K[jt])
    O = Gam[:, None] * (Q @ S0) + Mqk @ U
    gS = gam[-1]                      # the last cumulative sum
    S = np.exp(gS) * S0 + (K * state_decay_weights(gam, gS)[:, None]).T @ U
    return O, S


def chunk_prefill_head(q, k, v, g, beta, S0, chunk=64, inverse="block", q_scale=1.0):
    """One sequence and one head: cut into chunks of ``chunk`` rows (the last
    one partial) and carry the state from chunk to chunk.

    q, k [T, dk]; v [T, dv]; g, beta [T]; S0 [dk, dv] or None.  Returns
    (O [T, dv], S_T [dk, dv])."""
    assert 1 <= chunk <= PAD_ROWS
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    O = np.zeros((T, dv))
    for s in range(0, T, chunk):
        e = min(s + chunk, T)
        O[s:e], S = chunk_step(q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e], S, inverse)
    return q_scale * O, S


def chunk_prefill(q, k, v, g, beta, cu_seqlens, Hk, Hv, state_in=None, chunk=64,
                  inverse="block", q_scale=1.0):
    """Packed variable-length batch, GQA value head h reads key head
    h // (Hv // Hk).  Inputs are taken as given (no conv, no L2 norm).

    q, k [T, Hk, dk]; v [T, Hv, dv]; g, beta [T, Hv]; state_in [B, Hv, dk, dv]
    or None.  Returns (out [T, Hv, dv], state_out [B, Hv, dk, dv])."""
    q, k, v, g, beta = (np.asarray(a, dtype=np.float64) for a in (q, k, v, g, beta))
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    B = len(cu) - 1
    dk, dv = k.shape[2], v.shape[2]
    group = Hv // Hk
    out = np.zeros((q.shape[0], Hv, dv))
    s_out = np.zeros((B, Hv, dk, dv))
    for n in range(B):
        a, e = cu[n], cu[n + 1]
        for h in range(Hv):
            kh = h // group
            S0 = None if state_in is None else np.asarray(state_in, dtype=np.float64)[n, h]
            if e == a:
                s_out[n, h] = 0.0 if S0 is None else S0
                continue
            o, S = chunk_prefill_head(q[a:e, kh], k[a:e, kh], v[a:e, h], g[a:e, h],
                                      beta[a:e, h], S0, chunk, inverse, q_scale)
            out[a:e, h] = o
            s_out[n, h] = S
    return out, s_out
