"""ctypes front end of the float64 token-loop oracle — TEST INFRASTRUCTURE.

The arithmetic lives in ``gdn_oracle.c`` (plain C loops, float64).  This file
only compiles it with gcc, converts arrays to float64 and passes pointers.

Definition followed (one token at a time, per sequence and value head):
    S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
    o_t = q_scale * S_t^T q_t,
the one-token decoder step that the Qwen3.5 chunked-prefill pull request
("perf(qwen3_5): prefill text prompts in multi-token chunks", Background, Exit
Criteria) requires the chunked prefill to reproduce.  The short convolution in
front follows add_short_conv_rows ("perf(mamba): prefill text prompts in
multi-token chunks", Implementation).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` into ``oracle/_build/libgdn_oracle.so``.

    ``-ffp-contract=off`` keeps gcc from fusing multiply-adds, so the x86
    container and the Arm GPU host produce the same float64 results.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = build_oracle()
            lib = ctypes.CDLL(path)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_prefill.restype = ctypes.c_int
            lib.oracle_prefill.argtypes = [
                dp, dp, dp,                      # q, k, v
                dp, dp, dp, dp,                  # conv_x, conv_w, conv_state_in, conv_state_out
                ctypes.c_int, ctypes.c_int,      # conv_K, conv_act
                dp, dp,                          # g, beta
                dp, dp, dp,                      # state_in, state_out, out
                ctypes.POINTER(ctypes.c_int32),  # cu_seqlens
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_int,
            ]
            lib.oracle_short_conv.restype = ctypes.c_int
            lib.oracle_short_conv.argtypes = [
                dp, dp, dp, ctypes.c_int, dp, dp, ctypes.c_int,
                ctypes.POINTER(ctypes.c_int32), ctypes.c_int, ctypes.c_long]
            lib.oracle_l2norm_rows.restype = ctypes.c_int
            lib.oracle_l2norm_rows.argtypes = [dp, ctypes.c_long, ctypes.c_int,
                                               ctypes.c_long, ctypes.c_double]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def max_threads() -> int:
    """OpenMP threads the oracle uses when ``nthreads=0``."""
    return int(_load().oracle_max_threads())


def _f64(x):
    """Any array-like (NumPy, or a CPU/GPU torch tensor of any float dtype) to
    a C-contiguous float64 NumPy array.  bf16 values convert exactly."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def oracle_prefill(q, k, v, g, beta, cu_seqlens, Hk, Hv, dk, dv, state_in=None,
                   conv=None, use_l2norm=True, eps=1e-6, q_scale=1.0, nthreads=0):
    """Run the float64 token loop over a packed variable-length batch.

    q, k: [T, Hk, dk]; v: [T, Hv, dv]; g, beta: [T, Hv];
    cu_seqlens: [B+1] int; state_in: [B, Hv, dk, dv] or None (zero state).
    conv: None, or a dict with ``x`` [T, 2*Hk*dk + Hv*dv] (channels q|k|v; then
    q, k, v are ignored and may be None), ``w`` [channels, K], ``state_in``
    [B, channels, K-1] or None, ``act`` 0 (none) or 1 (SiLU).
    Returns a dict of float64 arrays: ``out`` [T, Hv, dv], ``state_out``
    [B, Hv, dk, dv] and, with conv, ``conv_state_out`` [B, channels, K-1].
    """
    lib = _load()
    cu = _cu_array(cu_seqlens)
    B = cu.shape[0] - 1
    T = int(cu[-1])
    g64, b64 = _f64(g).reshape(T, Hv), _f64(beta).reshape(T, Hv)
    s_in = _f64(state_in)
    if s_in is not None:
        s_in = s_in.reshape(B, Hv, dk, dv)
    out = np.zeros((T, Hv, dv), dtype=np.float64)
    s_out = np.zeros((B, Hv, dk, dv), dtype=np.float64)
    C = 2 * Hk * dk + Hv * dv
    if conv is not None:
        x64 = _f64(conv["x"]).reshape(T, C)
        w64 = _f64(conv["w"]).reshape(C, -1)
        K = w64.shape[1]
        cs_in = _f64(conv.get("state_in"))
        if cs_in is not None:
            cs_in = cs_in.reshape(B, C, K - 1)
        cs_out = np.zeros((B, C, max(K - 1, 0)), dtype=np.float64)
        act = int(conv.get("act", 0))
        q64 = k64 = v64 = None
    else:
        x64 = w64 = cs_in = cs_out = None
        K, act = 0, 0
        q64 = _f64(q).reshape(T, Hk, dk)
        k64 = _f64(k).reshape(T, Hk, dk)
        v64 = _f64(v).reshape(T, Hv, dv)
    rc = lib.oracle_prefill(
        _ptr(q64), _ptr(k64), _ptr(v64),
        _ptr(x64), _ptr(w64), _ptr(cs_in), _ptr(cs_out), K, act,
        _ptr(g64), _ptr(b64), _ptr(s_in), _ptr(s_out), _ptr(out),
        cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        B, Hk, Hv, dk, dv, 1 if use_l2norm else 0, float(eps), float(q_scale),
        int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_prefill failed with code {rc}")
    res = {"out": out, "state_out": s_out}
    if conv is not None:
        res["conv_state_out"] = cs_out
    return res


def _cu_array(cu_seqlens):
    return np.ascontiguousarray(np.asarray(
        cu_seqlens.detach().cpu().numpy() if hasattr(cu_seqlens, "detach") else cu_seqlens,
        dtype=np.int32))


def oracle_short_conv(x, w, cu_seqlens, state_in=None, act=0):
    """The short convolution alone (step 1 of the oracle).

    x [T, C]; w [C, K]; state_in [B, C, K-1] or None.  Returns (y [T, C],
    state_out [B, C, K-1]) in float64."""
    lib = _load()
    cu = _cu_array(cu_seqlens)
    B = cu.shape[0] - 1
    x64 = _f64(x)
    T, C = x64.shape
    w64 = _f64(w).reshape(C, -1)
    K = w64.shape[1]
    s_in = _f64(state_in)
    y = np.zeros_like(x64)
    s_out = np.zeros((B, C, K - 1), dtype=np.float64)
    rc = lib.oracle_short_conv(_ptr(x64), _ptr(y), _ptr(w64), K, _ptr(s_in), _ptr(s_out),
                               int(act), cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                               B, C)
    if rc != 0:
        raise RuntimeError(f"oracle_short_conv failed with code {rc}")
    return y, s_out


def oracle_l2norm(x, eps=1e-6):
    """Step 2 alone: every row of x [..., n] divided by sqrt(sum x^2 + eps)."""
    lib = _load()
    a = _f64(x).copy()
    n = a.shape[-1]
    rows = a.size // n
    rc = lib.oracle_l2norm_rows(_ptr(a), rows, n, n, float(eps))
    if rc != 0:
        raise RuntimeError(f"oracle_l2norm_rows failed with code {rc}")
    return a


def oracle_step(q, k, v, g, beta, state_in, Hk, Hv, dk, dv, conv=None,
                use_l2norm=True, eps=1e-6, q_scale=1.0, nthreads=0):
    """One decode token per batch entry: q, k [B, Hk, dk], v [B, Hv, dv],
    g, beta [B, Hv], state_in [B, Hv, dk, dv] (None = zero).  A decode step is
    a prefill of B sequences of length one, so it runs the same loop with
    cu_seqlens = 0, 1, ..., B."""
    if conv is not None:
        B = _f64(conv["x"]).shape[0]
    else:
        B = _f64(q).reshape(-1, Hk, dk).shape[0]
    cu = np.arange(B + 1, dtype=np.int32)
    return oracle_prefill(q, k, v, g, beta, cu, Hk, Hv, dk, dv, state_in=state_in,
                          conv=conv, use_l2norm=use_l2norm, eps=eps, q_scale=q_scale,
                          nthreads=nthreads)
