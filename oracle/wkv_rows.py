"""RWKV-4 WKV rows oracle — TEST INFRASTRUCTURE.

The RWKV chunked-prefill pull request ("perf(rwkv): prefill text prompts in
multi-token chunks", Implementation) keeps the one-token decoder's state
(num, den, max), A = num exp(max), B = den exp(max), of

    A_t = exp(w) A_{t-1} + exp(k_t) v_t,   B_t = exp(w) B_{t-1} + exp(k_t),
    wkv_t = (A_{t-1} + exp(u + k_t) v_t) / (B_{t-1} + exp(u + k_t)).

Two float64 implementations:

``oracle_wkv_rows``  the decoder's recurrence one row at a time (C, from
                     ``gdn_oracle.c``): the GPU path is compared with it.
``page_chunk_rows``  the page's chunk form, in NumPy: the prompt cut into
                     chunks of at most ``chunk`` rows; row t of a chunk sums
                     the incoming state with exponent max_0 + t w, the earlier
                     rows i < t with exponents k_i + (t - 1 - i) w (distances
                     from a static 65 x 64 table sliced to the chunk) and its
                     own bonus u + k_t; every row subtracts its largest
                     exponent; row S (no bonus) is the state after the chunk,
                     (num, den, max) with max that largest exponent.  Used only
                     to pin the row loop.

The state is not unique ((num c, den c, max - log c) is the same A, B), so
comparisons use the unique quantities num / den and max + log(den).
An absent state is (0, 0, -1e38).
"""

from __future__ import annotations

import ctypes

import numpy as np

from .token_loop import _cu_array, _f64, _load, _ptr

EMPTY_MAX = -1e38

# t - 1 - i for rows t = 0..64 and earlier rows i = 0..63 (the page's table)
DIST = np.arange(65)[:, None] - 1 - np.arange(64)[None, :]


def _lib():
    lib = _load()
    if not getattr(lib, "_wkv_bound", False):
        dp = ctypes.POINTER(ctypes.c_double)
        lib.oracle_wkv_rows.restype = ctypes.c_int
        lib.oracle_wkv_rows.argtypes = [dp, dp, dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int32),
                                        ctypes.c_int, ctypes.c_long]
        lib._wkv_bound = True
    return lib


def oracle_wkv_rows(k, v, w, u, cu_seqlens, state_in=None):
    """k, v [T, C]; w, u [C]; state_in [B, 3, C] or None.
    Returns (wkv [T, C], state_out [B, 3, C]) in float64."""
    lib = _lib()
    cu = _cu_array(cu_seqlens)
    B = cu.shape[0] - 1
    T = int(cu[-1])
    k64, v64 = _f64(k), _f64(v)
    C = k64.shape[-1]
    k64 = np.ascontiguousarray(k64.reshape(-1, C)[:T])
    v64 = np.ascontiguousarray(v64.reshape(-1, C)[:T])
    w64, u64 = _f64(w).reshape(C), _f64(u).reshape(C)
    s_in = _f64(state_in)
    if s_in is not None:
        s_in = s_in.reshape(B, 3, C)
    wkv = np.zeros((T, C))
    s_out = np.zeros((B, 3, C))
    rc = lib.oracle_wkv_rows(_ptr(k64), _ptr(v64), _ptr(w64), _ptr(u64), _ptr(s_in), _ptr(s_out),
                             _ptr(wkv), cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), B, C)
    if rc != 0:
        raise RuntimeError(f"oracle_wkv_rows failed with code {rc}")
    return wkv, s_out


def _chunk(k, v, w, u, num0, den0, max0):
    """One chunk of S rows: outputs of rows 0..S-1 and the state after row S-1."""
    S = k.shape[0]
    D = DIST[:S + 1, :S]                                   # [S+1, S] distances
    rows = np.arange(S + 1)
    # exponents: earlier rows (masked to i < t), the incoming state, the bonus
    e_rows = k[None, :, :] + D[:, :, None] * w[None, None, :]          # [S+1, S, C]
    mask = (np.arange(S)[None, :] < rows[:, None])[:, :, None]
    e_rows = np.where(mask, e_rows, -np.inf)
    e_state = max0[None, :] + rows[:, None] * w[None, :]                # [S+1, C]
    e_bonus = np.full((S + 1, k.shape[1]), -np.inf)
    e_bonus[:S] = u[None, :] + k                                        # row S has none
    m = np.maximum(np.maximum(e_rows.max(axis=1), e_state), e_bonus)    # [S+1, C]
    p_rows = np.exp(e_rows - m[:, None, :])
    p_state = np.exp(e_state - m)
    p_bonus = np.exp(e_bonus - m)
    vb = np.zeros((S + 1, k.shape[1]))
    vb[:S] = v
    num = num0[None, :] * p_state + (p_rows * v[None, :, :]).sum(axis=1) + p_bonus * vb
    den = den0[None, :] * p_state + p_rows.sum(axis=1) + p_bonus
    return num[:S] / den[:S], (num[S], den[S], m[S])


def page_chunk_rows(k, v, w, u, cu_seqlens, state_in=None, chunk=64):
    """The page's chunk form over every sequence; same returns as
    ``oracle_wkv_rows``."""
    assert 1 <= chunk <= 64
    cu = _cu_array(cu_seqlens)
    B = cu.shape[0] - 1
    k64, v64 = _f64(k), _f64(v)
    C = k64.shape[-1]
    w64, u64 = _f64(w).reshape(C), _f64(u).reshape(C)
    T = int(cu[-1])
    wkv = np.zeros((T, C))
    s_out = np.zeros((B, 3, C))
    for n in range(B):
        if state_in is None:
            num, den, mx = np.zeros(C), np.zeros(C), np.full(C, EMPTY_MAX)
        else:
            s = _f64(state_in).reshape(B, 3, C)[n]
            num, den, mx = s[0].copy(), s[1].copy(), s[2].copy()
        for s0 in range(int(cu[n]), int(cu[n + 1]), chunk):
            e = min(s0 + chunk, int(cu[n + 1]))
            out, (num, den, mx) = _chunk(k64[s0:e], v64[s0:e], w64, u64, num, den, mx)
            wkv[s0:e] = out
        s_out[n] = np.stack([num, den, mx])
    return wkv, s_out


def state_invariants(state):
    """The unique parts of a (num, den, max) state: num / den and
    max + log(den) (rows with den = 0 give 0 and -inf)."""
    s = np.asarray(state, dtype=np.float64)
    num, den, mx = s[..., 0, :], s[..., 1, :], s[..., 2, :]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0)
        logb = np.where(den > 0, mx + np.log(np.where(den > 0, den, 1.0)), -np.inf)
    return ratio, logb
