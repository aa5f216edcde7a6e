"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

* libgdn.so loads and exports every function include/gdn.h declares;
* the ctypes mirror of ``gdn_prefill_desc`` has the C layout (checked against
  a small C program compiled with gcc from the header);
* argument validation returns the documented status before anything is
  enqueued (every call here is rejected, or has B = 0, so no CUDA call runs).
"""

import ctypes
import os
import re
import subprocess

import pytest

from chunked_gated_delta_chunk_gb300 import binding as B
from chunked_gated_delta_chunk_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")

A = 0x100000          # a 16- and 256-byte aligned fake device address (never dereferenced)


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 8
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(B.EXPORTED) == names


def test_desc_layout_matches_c(tmp_path, lib):
    fields = [f for f, _ in B.gdn_prefill_desc._fields_]
    src = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "gdn.h"', 'int main(void){',
             'printf("%zu\\n", sizeof(gdn_prefill_desc));']
    lines += [f'printf("%zu\\n", offsetof(gdn_prefill_desc, {f}));' for f in fields]
    lines += ["return 0;}"]
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                            check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(B.gdn_prefill_desc)
    for f, off in zip(fields, vals[1:]):
        assert getattr(B.gdn_prefill_desc, f).offset == off, f


def _prefill(lib, **kw):
    args = dict(q=A, k=A, v=A, g=A, beta=A, state_in=A, state_out=A, out=A, cu=A,
                B=1, Hk=2, Hv=4, dk=128, dv=128, chunk=64)
    args.update(kw)
    return lib.gdn_prefill(args["q"], args["k"], args["v"], args["g"], args["beta"],
                           args["state_in"], args["state_out"], args["out"], args["cu"],
                           args["B"], args["Hk"], args["Hv"], args["dk"], args["dv"],
                           args["chunk"], None)


@pytest.mark.parametrize("chunk", [0, -1, 65, 128])
def test_chunk_outside_1_to_64_is_rejected(lib, chunk):
    assert _prefill(lib, chunk=chunk) == B.GDN_ERR_CHUNK


@pytest.mark.parametrize("kw,status", [
    (dict(dk=48), B.GDN_ERR_UNSUPPORTED), (dict(dv=256), B.GDN_ERR_UNSUPPORTED),
    (dict(dk=8), B.GDN_ERR_UNSUPPORTED), (dict(Hk=3, Hv=4), B.GDN_ERR_UNSUPPORTED),
    (dict(Hk=0), B.GDN_ERR_INVALID_ARG), (dict(B=-1), B.GDN_ERR_INVALID_ARG),
    (dict(q=None), B.GDN_ERR_INVALID_ARG), (dict(g=None), B.GDN_ERR_INVALID_ARG),
    (dict(beta=None), B.GDN_ERR_INVALID_ARG), (dict(out=None), B.GDN_ERR_INVALID_ARG),
    (dict(cu=None), B.GDN_ERR_INVALID_ARG),
    (dict(q=A + 2), B.GDN_ERR_ALIGN), (dict(v=A + 8), B.GDN_ERR_ALIGN),
    (dict(out=A + 4), B.GDN_ERR_ALIGN), (dict(state_in=A + 4), B.GDN_ERR_ALIGN),
    (dict(B=70000), B.GDN_ERR_TOO_LARGE),
])
def test_invalid_prefill_arguments(lib, kw, status):
    assert _prefill(lib, **kw) == status


def test_empty_batch_is_ok_without_launch(lib):
    assert _prefill(lib, B=0) == B.GDN_OK


def _desc(**kw):
    base = dict(B=1, Hk=16, Hv=32, dk=128, dv=128, T_total=100, g=A, beta=A, out=A,
                cu_seqlens=A, conv_x=A, conv_w=A, conv_kernel=4)
    base.update(kw)
    return B.make_desc(**base)


def test_workspace_size_and_rejection(lib):
    d = _desc()
    conv = ((100 * (2 * 16 * 128 + 32 * 128) * 2 + 255) // 256) * 256
    records = 32 * (100 // 64 + 1 + 1) * 82432      # Hv x chunk slots x record bytes
    assert B.gdn_workspace_bytes(d) == conv + records
    assert B.gdn_workspace_bytes(_desc(split_prep=-1)) == conv
    assert B.gdn_workspace_bytes(_desc(dtype=B.GDN_FP32)) == ((100 * 8192 * 4 + 255) // 256) * 256
    need = conv                                      # only the convolution's output is required
    assert lib.gdn_prefill_ex(ctypes.byref(d), None) == B.GDN_ERR_WORKSPACE
    d.workspace, d.workspace_bytes = A, need - 1
    assert lib.gdn_prefill_ex(ctypes.byref(d), None) == B.GDN_ERR_WORKSPACE
    d.workspace, d.workspace_bytes = A + 16, need
    assert lib.gdn_prefill_ex(ctypes.byref(d), None) == B.GDN_ERR_WORKSPACE
    d32 = _desc(dtype=B.GDN_FP32)
    assert B.gdn_workspace_bytes(d32) == ((100 * 8192 * 4 + 255) // 256) * 256
    assert B.gdn_workspace_bytes(_desc(conv_x=None)) == records
    assert B.gdn_workspace_bytes(_desc(conv_x=None, split_prep=-1)) == 0
    assert B.gdn_workspace_bytes(_desc(conv_x=None, T_total=-1)) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(T_total=-1), B.GDN_ERR_INVALID_ARG), (dict(conv_w=None), B.GDN_ERR_INVALID_ARG),
    (dict(conv_kernel=1), B.GDN_ERR_UNSUPPORTED), (dict(conv_kernel=9), B.GDN_ERR_UNSUPPORTED),
    (dict(conv_act=2), B.GDN_ERR_UNSUPPORTED), (dict(conv_x=A + 2), B.GDN_ERR_ALIGN),
    (dict(dtype=5), B.GDN_ERR_UNSUPPORTED),
])
def test_invalid_conv_descriptions(lib, kw, status):
    d = _desc(**kw)
    d.workspace, d.workspace_bytes = A, 1 << 40
    assert lib.gdn_prefill_ex(ctypes.byref(d), None) == status


def test_step_rejects_cu_seqlens_and_bad_shapes(lib):
    d = B.make_desc(B=2, Hk=1, Hv=1, dk=16, dv=16, q=A, k=A, v=A, g=A, beta=A, out=A,
                    state_in=A, state_out=A, cu_seqlens=A)
    assert lib.gdn_step_ex(ctypes.byref(d), None) == B.GDN_ERR_INVALID_ARG
    assert lib.gdn_step(A, A, A, A, A, A, A, 1, 1, 1, 24, 16, None) == B.GDN_ERR_UNSUPPORTED
    assert lib.gdn_step(A, A, A, A, A, A, A + 4, 1, 1, 1, 16, 16, None) == B.GDN_ERR_ALIGN
    assert lib.gdn_step(A, A, A, A, A, A, A, 0, 1, 1, 16, 16, None) == B.GDN_OK


def test_status_strings_and_defaults(lib):
    for code in range(8):
        assert B.gdn_status_string(code)
    assert "chunk" in B.gdn_status_string(B.GDN_ERR_CHUNK)
    d = B.make_desc()
    assert (d.dtype, d.chunk, d.T_total, d.conv_kernel, d.use_qk_l2norm) == (B.GDN_BF16, 64, -1, 4, 1)
    assert abs(d.l2_eps - 1e-6) < 1e-12 and d.q_scale == 1.0
    assert B.gdn_version() >= 100


def test_launch_plan_names(lib):
    """Host-only launch plan: the tensor-core kernel for bf16 with
    dk = dv = 128, the SIMT kernel otherwise; conv adds its two kernels, and
    the split preparation runs first when the workspace holds its records."""
    d = B.make_desc(B=1, Hk=2, Hv=4, dk=128, dv=128, q=A, k=A, v=A, g=A, beta=A, out=A,
                    cu_seqlens=A)
    assert B.gdn_prefill_plan(d) == ["chunk_tc_kernel"]
    d32 = B.make_desc(B=1, Hk=2, Hv=4, dk=128, dv=128, q=A, k=A, v=A, g=A, beta=A, out=A,
                      cu_seqlens=A, dtype=B.GDN_FP32)
    assert B.gdn_prefill_plan(d32) == ["chunk_simt_kernel"]
    d64 = B.make_desc(B=1, Hk=2, Hv=4, dk=64, dv=128, q=A, k=A, v=A, g=A, beta=A, out=A,
                      cu_seqlens=A)
    assert B.gdn_prefill_plan(d64) == ["chunk_simt_kernel"]
    dc = _desc(conv_state_out=A)
    dc.workspace, dc.workspace_bytes = A, 1 << 40
    assert B.gdn_prefill_plan(dc) == ["conv_kernel", "chunk_prep_kernel", "chunk_state_kernel",
                                      "conv_state_kernel"]
    dc.split_prep = -1
    assert B.gdn_prefill_plan(dc) == ["conv_kernel", "chunk_tc_kernel", "conv_state_kernel"]
    dc.split_prep = 0
    dc.workspace_bytes = B.gdn_workspace_bytes(dc) - 1      # no room for the chunk records
    assert B.gdn_prefill_plan(dc) == ["conv_kernel", "chunk_tc_kernel", "conv_state_kernel"]
    bad = B.make_desc(B=1, Hk=2, Hv=4, dk=48, dv=128, q=A, k=A, v=A, g=A, beta=A, out=A,
                      cu_seqlens=A)
    with pytest.raises(B.GdnError):
        B.gdn_prefill_plan(bad)


def test_launch_timer_host_paths(lib):
    """The launch timer's argument check and its empty record need no GPU:
    capacity outside 1..1e6 is rejected before any CUDA call, and reading
    without a started timer returns no launches."""
    assert lib.gdn_launch_timer_start(0) == B.GDN_ERR_INVALID_ARG
    assert lib.gdn_launch_timer_start(1000001) == B.GDN_ERR_INVALID_ARG
    assert lib.gdn_launch_timer_stop() == B.GDN_OK
    records, dropped = B.gdn_launch_timer_read()
    assert records == [] and dropped == 0


def test_scan_rows_argument_checks(lib):
    """Selective-scan rows: every invalid call is rejected before any CUDA
    call (fake device addresses, never dereferenced)."""
    ws = B.gdn_scan_workspace_bytes(256, 1000)
    assert ws > 0 and ws % 256 == 0
    assert B.gdn_scan_workspace_bytes(256, 2000) > ws
    assert lib.gdn_scan_workspace_bytes(0, 10) == ctypes.c_size_t(-1).value
    good = dict(a=A, b=A, h_in=None, h_out=A, h_rows=A, cu=A, B=1, C=256, T=1000, ws=A, wsb=ws)

    def call(**kw):
        d = dict(good, **kw)
        return lib.gdn_scan_rows(d["a"], d["b"], d["h_in"], d["h_out"], d["h_rows"], d["cu"],
                                 d["B"], d["C"], d["T"], d["ws"], d["wsb"], None)
    assert call(B=-1) == B.GDN_ERR_INVALID_ARG
    assert call(C=0) == B.GDN_ERR_INVALID_ARG
    assert call(h_out=None) == B.GDN_ERR_INVALID_ARG
    assert call(a=None) == B.GDN_ERR_INVALID_ARG
    assert call(C=250) == B.GDN_ERR_UNSUPPORTED
    assert call(b=A + 4) == B.GDN_ERR_ALIGN
    assert call(ws=None) == B.GDN_ERR_WORKSPACE
    assert call(ws=A + 16) == B.GDN_ERR_WORKSPACE
    assert call(wsb=ws - 1) == B.GDN_ERR_WORKSPACE
    assert call(B=0, T=0) == B.GDN_OK            # nothing to do, nothing enqueued


def test_wkv_rows_argument_checks(lib):
    """RWKV-4 WKV rows: invalid calls are rejected before any CUDA call."""
    ws = B.gdn_wkv_workspace_bytes(256, 1000)
    assert ws > 0 and ws % 256 == 0
    assert B.gdn_wkv_workspace_bytes(256, 2000) > ws
    good = dict(k=A, v=A, w=A, u=A, s_in=None, s_out=A, wkv=A, cu=A, B=1, C=256, T=1000,
                ws=A, wsb=ws)

    def call(**kw):
        d = dict(good, **kw)
        return lib.gdn_wkv_rows(d["k"], d["v"], d["w"], d["u"], d["s_in"], d["s_out"], d["wkv"],
                                d["cu"], d["B"], d["C"], d["T"], d["ws"], d["wsb"], None)
    assert call(B=-1) == B.GDN_ERR_INVALID_ARG
    assert call(w=None) == B.GDN_ERR_INVALID_ARG
    assert call(s_out=None) == B.GDN_ERR_INVALID_ARG
    assert call(k=None) == B.GDN_ERR_INVALID_ARG
    assert call(C=6) == B.GDN_ERR_UNSUPPORTED
    assert call(wkv=A + 8) == B.GDN_ERR_ALIGN
    assert call(wsb=ws - 256) == B.GDN_ERR_WORKSPACE
    assert call(B=0, T=0) == B.GDN_OK


def test_attn_rows_argument_checks(lib):
    """Attention rows: invalid calls are rejected before any CUDA call."""
    good = dict(q=A, k=A, v=A, kc=A, vc=A, cl=A, o=A, cu=A, B=1, Hq=4, Hkv=2, D=128, cap=256, T=100,
                scale=0.0)

    def call(**kw):
        d = dict(good, **kw)
        return lib.gdn_attn_rows(d["q"], d["k"], d["v"], d["kc"], d["vc"], d["cl"], d["o"], d["cu"],
                                 d["B"], d["Hq"], d["Hkv"], d["D"], d["cap"], d["T"], d["scale"], None)
    assert call(B=-1) == B.GDN_ERR_INVALID_ARG
    assert call(cap=0) == B.GDN_ERR_INVALID_ARG
    assert call(scale=-1.0) == B.GDN_ERR_INVALID_ARG
    assert call(D=64) == B.GDN_ERR_UNSUPPORTED
    assert call(Hq=3) == B.GDN_ERR_UNSUPPORTED
    assert call(q=None) == B.GDN_ERR_INVALID_ARG
    assert call(cl=None) == B.GDN_ERR_INVALID_ARG
    assert call(o=A + 2) == B.GDN_ERR_ALIGN
    assert call(cap=1 << 30) == B.GDN_ERR_TOO_LARGE
    assert call(B=0, T=0) == B.GDN_OK


def test_segmented_plan_and_workspace(lib):
    """A 4096-token prompt over 16 value heads takes the segment-parallel
    scan: five segments of 13 chunks (phase 1 on 16 x 9 CTAs, one wave of the
    152 SMs), then seg_out_kernel.  Its workspace holds the segment maps (three
    128 x 128 fp32 matrices per head and slot), the output map G (bf16, one row
    of Hv x dv per token) and the chunk records."""
    d = B.make_desc(B=1, Hk=16, Hv=16, dk=128, dv=128, T_total=4096, q=A, k=A, v=A, g=A, beta=A,
                    out=A, cu_seqlens=A)
    slots = 4096 // (13 * 64) + 1 + 1
    maps = ((16 * slots * 3 * 128 * 128 * 4 + 255) // 256) * 256
    g_map = 4096 * 16 * 128 * 2
    records = 16 * (4096 // 64 + 1 + 1) * 82432
    assert B.gdn_workspace_bytes(d) == maps + g_map + records
    d.workspace, d.workspace_bytes = A, B.gdn_workspace_bytes(d)
    assert B.gdn_prefill_plan(d) == ["chunk_prep_kernel", "chunk_state_kernel", "seg_out_kernel"]
    d.workspace_bytes = maps + g_map                 # no room for the records: inline preparation
    assert B.gdn_prefill_plan(d) == ["chunk_tc_kernel", "seg_out_kernel"]
    d.workspace_bytes = maps + g_map - 1             # no room for G either: one pass
    assert B.gdn_prefill_plan(d) == ["chunk_tc_kernel"]
    d.segment_chunks = -1                            # one pass asked for
    d.workspace_bytes = 1 << 40
    assert B.gdn_prefill_plan(d) == ["chunk_prep_kernel", "chunk_state_kernel"]
    d.split_prep = 1                                 # any value >= 0: on when the records fit
    assert B.gdn_prefill_plan(d) == ["chunk_prep_kernel", "chunk_state_kernel"]
    d.workspace_bytes = 0                            # no records: the inline pass
    assert B.gdn_prefill_plan(d) == ["chunk_tc_kernel"]


def test_batch_without_tokens_needs_no_token_tensors(lib):
    """T_total == 0 (every sequence empty): the token tensors may be NULL; the
    plan launches no kernel, and with no state to return nothing is enqueued."""
    d = B.make_desc(B=3, Hk=2, Hv=4, dk=128, dv=128, T_total=0, cu_seqlens=A)
    assert B.gdn_prefill_plan(d) == []
    assert lib.gdn_prefill_ex(ctypes.byref(d), None) == B.GDN_OK
    # the rest is still validated
    assert lib.gdn_prefill_ex(ctypes.byref(B.make_desc(B=3, Hk=2, Hv=4, dk=128, dv=128, T_total=0)),
                              None) == B.GDN_ERR_INVALID_ARG                 # no cu_seqlens
    d_conv = B.make_desc(B=3, Hk=2, Hv=4, dk=128, dv=128, T_total=0, cu_seqlens=A, conv_state_out=A,
                         conv_kernel=1)
    assert lib.gdn_prefill_ex(ctypes.byref(d_conv), None) == B.GDN_ERR_UNSUPPORTED


def test_preparation_counts_items_in_32_bits(lib):
    """The split preparation numbers its items (Hv x chunk slots) in 32 bits:
    a description with 2^31 or more of them asks for no chunk records and
    runs the chain with the inline preparation, one with fewer uses them."""
    T = 1 << 30
    slots = T // 64 + 1 + 1
    for hv, records in ((127, True), (128, False)):
        assert (hv * slots < (1 << 31)) == records
        d = B.make_desc(B=1, Hk=hv, Hv=hv, dk=128, dv=128, T_total=T, segment_chunks=-1,
                        q=A, k=A, v=A, g=A, beta=A, out=A, cu_seqlens=A)
        assert B.gdn_workspace_bytes(d) == (hv * slots * 82432 if records else 0)
        d.workspace, d.workspace_bytes = A, 1 << 62
        assert B.gdn_prefill_plan(d) == (["chunk_prep_kernel", "chunk_state_kernel"] if records
                                         else ["chunk_tc_kernel"])
