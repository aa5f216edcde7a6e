"""Selective-scan rows oracle — TEST INFRASTRUCTURE.

The Mamba chunked-prefill pull request ("perf(mamba): prefill text prompts in
multi-token chunks", Implementation, add_selective_scan_rows) defines the
recurrence h_t = a_t h_{t-1} + b_t over the rows of a chunk, in FP32 on the
page, every a_t a decay in (0, 1], at most 64 rows per chunk (MAX_ROWS), the
chunk's incoming state h_0 applied at the end.

Two implementations, both float64:

``oracle_scan_rows``  the plain definition, one row at a time (C, compiled
                      from ``gdn_oracle.c``): the GPU path is compared with it.
``hillis_steele_rows`` the page's algorithm, in NumPy: the prompt cut into
                      chunks of at most ``chunk`` rows; in each chunk
                      ceil(log2 S) rounds of (a, b)_t <- (a_t a_{t-k},
                      a_t b_{t-k} + b_t) for k = 1, 2, 4, ..., the shifted
                      operands padded with the identity pair (1, 0); then
                      h_t = a_t h_0 + b_t with the chunk's incoming state.
                      Used only to pin the plain definition.
"""

from __future__ import annotations

import ctypes

import numpy as np

from .token_loop import _cu_array, _f64, _load, _ptr


def _lib():
    lib = _load()
    if not getattr(lib, "_scan_bound", False):
        dp = ctypes.POINTER(ctypes.c_double)
        lib.oracle_scan_rows.restype = ctypes.c_int
        lib.oracle_scan_rows.argtypes = [dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int32),
                                         ctypes.c_int, ctypes.c_long]
        lib._scan_bound = True
    return lib


def oracle_scan_rows(a, b, cu_seqlens, h_in=None):
    """a, b [T, C]; cu_seqlens [B+1]; h_in [B, C] or None (zero state).
    Returns (h_rows [T, C], h_out [B, C]) in float64."""
    lib = _lib()
    cu = _cu_array(cu_seqlens)
    B = cu.shape[0] - 1
    a64, b64 = _f64(a), _f64(b)
    T = int(cu[-1])
    C = a64.shape[-1] if a64.ndim > 1 else 1
    a64, b64 = a64.reshape(-1, C)[:T], b64.reshape(-1, C)[:T]
    a64, b64 = np.ascontiguousarray(a64), np.ascontiguousarray(b64)
    h0 = _f64(h_in)
    if h0 is not None:
        h0 = h0.reshape(B, C)
    rows = np.zeros((T, C), dtype=np.float64)
    out = np.zeros((B, C), dtype=np.float64)
    rc = lib.oracle_scan_rows(_ptr(a64), _ptr(b64), _ptr(h0), _ptr(out), _ptr(rows),
                              cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), B, C)
    if rc != 0:
        raise RuntimeError(f"oracle_scan_rows failed with code {rc}")
    return rows, out


def _chunk_scan(a, b, h0):
    """One chunk of S rows: the doubling rounds, then the incoming state."""
    A, Bv = a.copy(), b.copy()
    S = A.shape[0]
    k = 1
    while k < S:
        # (A, B)_t <- (A_t A_{t-k}, A_t B_{t-k} + B_t); rows t < k meet the
        # identity pair (1, 0) from the static pad
        A_prev = np.concatenate([np.ones_like(A[:k]), A[:-k]], axis=0)
        B_prev = np.concatenate([np.zeros_like(Bv[:k]), Bv[:-k]], axis=0)
        A, Bv = A * A_prev, A * B_prev + Bv
        k *= 2
    return A * h0[None, :] + Bv


def hillis_steele_rows(a, b, cu_seqlens, h_in=None, chunk=64):
    """The page's chunked doubling scan over every sequence; same returns as
    ``oracle_scan_rows``."""
    cu = _cu_array(cu_seqlens)
    B = cu.shape[0] - 1
    a64, b64 = _f64(a), _f64(b)
    C = a64.shape[-1]
    T = int(cu[-1])
    h0_all = np.zeros((B, C)) if h_in is None else _f64(h_in).reshape(B, C)
    rows = np.zeros((T, C), dtype=np.float64)
    out = np.zeros((B, C), dtype=np.float64)
    for n in range(B):
        h = h0_all[n].copy()
        for s in range(int(cu[n]), int(cu[n + 1]), chunk):
            e = min(s + chunk, int(cu[n + 1]))
            hr = _chunk_scan(a64[s:e], b64[s:e], h)
            rows[s:e] = hr
            h = hr[-1].copy()
        out[n] = h
    return rows, out
