"""ctypes binding of libgdn.so — argument marshalling only.

Each function has the name of the C entry point it calls (see include/gdn.h)
and passes device pointers, sizes and the stream straight through; every step
of the computation runs in the library's CUDA kernels.  Tensors may be torch
tensors (their ``data_ptr()`` is passed) or raw integer addresses; ``None``
passes NULL.  A non-zero status raises ``GdnError``.  There is no fallback: if
the library has not been built, loading it raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

_lock = threading.Lock()
_lib = None

GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_CHUNK = 2
GDN_ERR_UNSUPPORTED = 3
GDN_ERR_ALIGN = 4
GDN_ERR_CUDA = 5
GDN_ERR_WORKSPACE = 6
GDN_ERR_TOO_LARGE = 7

GDN_BF16 = 0
GDN_FP32 = 1
GDN_ACT_NONE = 0
GDN_ACT_SILU = 1

# Every symbol include/gdn.h declares.
EXPORTED = ("gdn_prefill_desc_init", "gdn_prefill", "gdn_prefill_ex", "gdn_workspace_bytes",
            "gdn_step", "gdn_step_ex", "gdn_prefill_plan", "gdn_status_string",
            "gdn_last_cuda_error", "gdn_version", "gdn_prefill_noalloc",
            "gdn_noalloc_scratch_bytes", "gdn_launch_timer_start", "gdn_launch_timer_stop",
            "gdn_launch_timer_read", "gdn_scan_workspace_bytes", "gdn_scan_rows",
            "gdn_wait_timeouts", "gdn_wkv_workspace_bytes", "gdn_wkv_rows", "gdn_attn_rows")


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().gdn_status_string(status).decode()
        if status == GDN_ERR_CUDA:
            msg += f" (cudaError {lib().gdn_last_cuda_error()})"
        super().__init__(f"{where}: status {status}: {msg}")


class gdn_prefill_desc(ctypes.Structure):
    """Mirror of ``struct gdn_prefill_desc`` in include/gdn.h (same field order)."""
    _fields_ = [
        ("dtype", ctypes.c_int), ("B", ctypes.c_int), ("Hk", ctypes.c_int), ("Hv", ctypes.c_int),
        ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("chunk", ctypes.c_int),
        ("T_total", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("state_in", ctypes.c_void_p), ("state_out", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("cu_seqlens", ctypes.c_void_p),
        ("conv_x", ctypes.c_void_p), ("conv_w", ctypes.c_void_p),
        ("conv_state_in", ctypes.c_void_p), ("conv_state_out", ctypes.c_void_p),
        ("conv_kernel", ctypes.c_int), ("conv_act", ctypes.c_int),
        ("use_qk_l2norm", ctypes.c_int), ("l2_eps", ctypes.c_float), ("q_scale", ctypes.c_float),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("segment_chunks", ctypes.c_int), ("split_prep", ctypes.c_int),
    ]


def lib():
    """Load libgdn.so (built in-tree by ``build.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(
                    f"{LIB} is missing: build it with chunked_gated_delta_chunk_gb300.build.build()")
            L = ctypes.CDLL(LIB)
            vp, i, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
            L.gdn_prefill_desc_init.restype = None
            L.gdn_prefill_desc_init.argtypes = [ctypes.POINTER(gdn_prefill_desc)]
            L.gdn_prefill.restype = i
            L.gdn_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      i, i, i, i, i, i, st]
            L.gdn_prefill_ex.restype = i
            L.gdn_prefill_ex.argtypes = [ctypes.POINTER(gdn_prefill_desc), st]
            L.gdn_workspace_bytes.restype = ctypes.c_size_t
            L.gdn_workspace_bytes.argtypes = [ctypes.POINTER(gdn_prefill_desc)]
            L.gdn_step.restype = i
            L.gdn_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, st]
            L.gdn_step_ex.restype = i
            L.gdn_step_ex.argtypes = [ctypes.POINTER(gdn_prefill_desc), st]
            L.gdn_prefill_plan.restype = i
            L.gdn_prefill_plan.argtypes = [ctypes.POINTER(gdn_prefill_desc),
                                           ctypes.POINTER(ctypes.c_char_p), i]
            L.gdn_prefill_noalloc.restype = i
            L.gdn_prefill_noalloc.argtypes = [ctypes.POINTER(gdn_prefill_desc), st]
            L.gdn_noalloc_scratch_bytes.restype = ctypes.c_size_t
            L.gdn_noalloc_scratch_bytes.argtypes = []
            L.gdn_launch_timer_start.restype = i
            L.gdn_launch_timer_start.argtypes = [i]
            L.gdn_launch_timer_stop.restype = i
            L.gdn_launch_timer_stop.argtypes = []
            L.gdn_launch_timer_read.restype = i
            L.gdn_launch_timer_read.argtypes = [ctypes.POINTER(ctypes.c_char_p),
                                                ctypes.POINTER(ctypes.c_float), i,
                                                ctypes.POINTER(ctypes.c_int)]
            L.gdn_scan_workspace_bytes.restype = ctypes.c_size_t
            L.gdn_scan_workspace_bytes.argtypes = [i, ctypes.c_int64]
            L.gdn_scan_rows.restype = i
            L.gdn_scan_rows.argtypes = [vp, vp, vp, vp, vp, vp, i, i, ctypes.c_int64, vp,
                                        ctypes.c_size_t, st]
            L.gdn_wkv_workspace_bytes.restype = ctypes.c_size_t
            L.gdn_wkv_workspace_bytes.argtypes = [i, ctypes.c_int64]
            L.gdn_wkv_rows.restype = i
            L.gdn_wkv_rows.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, ctypes.c_int64, vp,
                                       ctypes.c_size_t, st]
            L.gdn_attn_rows.restype = i
            L.gdn_attn_rows.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_int64,
                                        ctypes.c_float, st]
            L.gdn_wait_timeouts.restype = ctypes.c_longlong
            L.gdn_wait_timeouts.argtypes = []
            L.gdn_status_string.restype = ctypes.c_char_p
            L.gdn_status_string.argtypes = [i]
            L.gdn_last_cuda_error.restype = i
            L.gdn_last_cuda_error.argtypes = []
            L.gdn_version.restype = i
            L.gdn_version.argtypes = []
            _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str):
    if status != GDN_OK:
        raise GdnError(status, where)


def gdn_prefill(q, k, v, g, beta, state_in, state_out, out, cu_seqlens, B, Hk, Hv, dk, dv,
                chunk=64, stream=None):
    _check(lib().gdn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in),
                             _ptr(state_out), _ptr(out), _ptr(cu_seqlens), int(B), int(Hk),
                             int(Hv), int(dk), int(dv), int(chunk), _stream(stream)),
           "gdn_prefill")


def make_desc(**fields) -> gdn_prefill_desc:
    """A ``gdn_prefill_desc`` with the library defaults, then ``fields``
    (tensors for pointer fields, plain numbers for the rest)."""
    d = gdn_prefill_desc()
    lib().gdn_prefill_desc_init(ctypes.byref(d))
    for name, val in fields.items():
        ctype = dict(gdn_prefill_desc._fields_)[name]
        setattr(d, name, _ptr(val) if ctype is ctypes.c_void_p else val)
    return d


def gdn_workspace_bytes(desc: gdn_prefill_desc) -> int:
    n = lib().gdn_workspace_bytes(ctypes.byref(desc))
    if n == ctypes.c_size_t(-1).value:
        raise GdnError(GDN_ERR_INVALID_ARG, "gdn_workspace_bytes")
    return int(n)


def gdn_prefill_ex(desc: gdn_prefill_desc, stream=None):
    _check(lib().gdn_prefill_ex(ctypes.byref(desc), _stream(stream)), "gdn_prefill_ex")


def gdn_step(q, k, v, g, beta, state, out, B, Hk, Hv, dk, dv, stream=None):
    _check(lib().gdn_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(out),
                          int(B), int(Hk), int(Hv), int(dk), int(dv), _stream(stream)),
           "gdn_step")


def gdn_step_ex(desc: gdn_prefill_desc, stream=None):
    _check(lib().gdn_step_ex(ctypes.byref(desc), _stream(stream)), "gdn_step_ex")


def gdn_prefill_plan(desc: gdn_prefill_desc):
    """Names of the kernels one gdn_prefill_ex call with ``desc`` launches."""
    names = (ctypes.c_char_p * 8)()
    n = lib().gdn_prefill_plan(ctypes.byref(desc), names, 8)
    if n < 0:
        raise GdnError(-n, "gdn_prefill_plan")
    return [names[i].decode() for i in range(n)]


def gdn_prefill_noalloc(desc: gdn_prefill_desc, stream=None):
    """gdn_prefill_ex without a caller workspace: for callers that cannot
    allocate device memory; uses the library's fixed scratch array."""
    _check(lib().gdn_prefill_noalloc(ctypes.byref(desc), _stream(stream)), "gdn_prefill_noalloc")


def gdn_noalloc_scratch_bytes() -> int:
    return int(lib().gdn_noalloc_scratch_bytes())


def gdn_launch_timer_start(capacity: int):
    """Record the device time of the next ``capacity`` kernel launches."""
    _check(lib().gdn_launch_timer_start(int(capacity)), "gdn_launch_timer_start")


def gdn_launch_timer_stop():
    _check(lib().gdn_launch_timer_stop(), "gdn_launch_timer_stop")


def gdn_launch_timer_read():
    """``([(kernel name, ms), ...] in launch order, dropped launches)``."""
    L = lib()
    dropped = ctypes.c_int(0)
    n = L.gdn_launch_timer_read(None, None, 0, ctypes.byref(dropped))
    if n < 0:
        raise GdnError(-n, "gdn_launch_timer_read")
    names = (ctypes.c_char_p * max(n, 1))()
    ms = (ctypes.c_float * max(n, 1))()
    m = L.gdn_launch_timer_read(names, ms, n, ctypes.byref(dropped))
    if m < 0:
        raise GdnError(-m, "gdn_launch_timer_read")
    return [(names[i].decode(), float(ms[i])) for i in range(min(n, m))], int(dropped.value)


def gdn_scan_workspace_bytes(C: int, T_total: int) -> int:
    n = lib().gdn_scan_workspace_bytes(int(C), int(T_total))
    if n == ctypes.c_size_t(-1).value:
        raise GdnError(GDN_ERR_INVALID_ARG, "gdn_scan_workspace_bytes")
    return int(n)


def gdn_scan_rows(a, b, h_in, h_out, h_rows, cu_seqlens, B, C, T_total, workspace,
                  workspace_bytes, stream=None):
    """h_t = a_t h_{t-1} + b_t per channel over every sequence (device tensors)."""
    _check(lib().gdn_scan_rows(_ptr(a), _ptr(b), _ptr(h_in), _ptr(h_out), _ptr(h_rows),
                               _ptr(cu_seqlens), int(B), int(C), int(T_total), _ptr(workspace),
                               int(workspace_bytes), _stream(stream)), "gdn_scan_rows")


def gdn_wkv_workspace_bytes(C: int, T_total: int) -> int:
    n = lib().gdn_wkv_workspace_bytes(int(C), int(T_total))
    if n == ctypes.c_size_t(-1).value:
        raise GdnError(GDN_ERR_INVALID_ARG, "gdn_wkv_workspace_bytes")
    return int(n)


def gdn_wkv_rows(k, v, w, u, state_in, state_out, wkv, cu_seqlens, B, C, T_total, workspace,
                 workspace_bytes, stream=None):
    """RWKV-4 WKV over every sequence (device tensors)."""
    _check(lib().gdn_wkv_rows(_ptr(k), _ptr(v), _ptr(w), _ptr(u), _ptr(state_in), _ptr(state_out),
                              _ptr(wkv), _ptr(cu_seqlens), int(B), int(C), int(T_total),
                              _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "gdn_wkv_rows")


def gdn_attn_rows(q, k, v, k_cache, v_cache, cache_len, o, cu_seqlens, B, Hq, Hkv, head_dim,
                  cache_capacity, T_total, scale=0.0, stream=None):
    """Attention over the KV cache plus the chunk's causal prefix; appends the
    chunk's k / v rows to the cache (device tensors)."""
    _check(lib().gdn_attn_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(cache_len),
                               _ptr(o), _ptr(cu_seqlens), int(B), int(Hq), int(Hkv), int(head_dim),
                               int(cache_capacity), int(T_total), float(scale), _stream(stream)),
           "gdn_attn_rows")


def gdn_wait_timeouts() -> int:
    """Bounded device waits that ran out since load (synchronises the device)."""
    n = int(lib().gdn_wait_timeouts())
    if n < 0:
        raise GdnError(GDN_ERR_CUDA, "gdn_wait_timeouts")
    return n


def gdn_status_string(status: int) -> str:
    return lib().gdn_status_string(int(status)).decode()


def gdn_version() -> int:
    return int(lib().gdn_version())
