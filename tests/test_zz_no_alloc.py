"""gdn_prefill_noalloc: the prefill entry point for callers that cannot
allocate device memory (a runtime whose device memory all belongs to its own
pool, or code that must not synchronise the device by allocating).  It runs
the same kernels as gdn_prefill_ex, with the convolution's scratch taken from
a fixed array inside the library instead of a caller workspace.

Checked on a GPU through the C ABI: two calls in a row (different inputs, so
the second call runs on the array the first one left behind) each match
gdn_prefill_ex on the same inputs and the float64 oracle within the parity
tolerance, with and without the short convolution; a call after the first
one on the device leaves the device's free memory unchanged; a description
whose scratch would exceed the array is rejected.  This file is collected
last so that a failure here leaves every other test already run.
"""

import pytest
import torch

from chunked_gated_delta_chunk_gb300 import binding as B
from chunked_gated_delta_chunk_gb300 import build as build_mod
from chunked_gated_delta_chunk_gb300 import inputs, runner
from tests.harness import TOL_BF16, assert_close, compare, run_oracle, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()


def _noalloc_results(call):
    """Run the same description as `call` through gdn_prefill_noalloc into
    fresh output buffers (no workspace passed)."""
    out = torch.empty_like(call.out)
    st = torch.empty_like(call.state_out)
    cs = torch.empty_like(call.cs_out) if call.cs_out is not None else None
    d = B.gdn_prefill_desc()
    import ctypes
    ctypes.memmove(ctypes.byref(d), ctypes.byref(call.desc), ctypes.sizeof(d))
    d.out, d.state_out = out.data_ptr(), st.data_ptr()
    if cs is not None:
        d.conv_state_out = cs.data_ptr()
    d.workspace, d.workspace_bytes = None, 0
    B.gdn_prefill_noalloc(d)
    res = {"out": out, "state_out": st}
    if cs is not None:
        res["conv_state_out"] = cs
    return res


@pytest.mark.parametrize("dtype,dk,conv", [(torch.bfloat16, 128, 4), (torch.float32, 32, 4),
                                           (torch.bfloat16, 128, 0)])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(dtype, dk, conv):
    problems = [inputs.make_problem(seed, lengths, 2, 4, dk, dk, dtype=dtype, conv_kernel=conv)
                for seed, lengths in ((501, [75, 40]), (502, [3, 130, 64]))]
    for p in problems:                       # two calls in a row, different inputs
        ref_call = runner.PrefillCall(p)
        ref_call.run()
        got = _noalloc_results(ref_call)
        torch.cuda.synchronize()
        tol = tol_for(p)
        assert_close(got["out"].cpu(), ref_call.out.cpu(), tol, "out")
        assert_close(got["state_out"].cpu(), ref_call.state_out.cpu(), tol, "state_out")
        if conv:
            assert_close(got["conv_state_out"].cpu(), ref_call.cs_out.cpu(), 0.0, "conv_state_out")
        compare({k: v.cpu() for k, v in got.items()}, run_oracle(p), tol)


def test_noalloc_later_calls_leave_free_memory_unchanged():
    """The array's memory is reserved by the first call on the device (module
    load and address lookup); a later call reserves nothing more."""
    p = inputs.make_problem(504, [200, 17], 2, 4, 128, 128, conv_kernel=4)
    call = runner.PrefillCall(p)
    _noalloc_results(call)                   # first call (if no earlier test made it)
    torch.cuda.synchronize()
    out = torch.empty_like(call.out)
    st = torch.empty_like(call.state_out)
    cs = torch.empty_like(call.cs_out)
    d = B.gdn_prefill_desc()
    import ctypes
    ctypes.memmove(ctypes.byref(d), ctypes.byref(call.desc), ctypes.sizeof(d))
    d.out, d.state_out, d.conv_state_out = out.data_ptr(), st.data_ptr(), cs.data_ptr()
    d.workspace, d.workspace_bytes = None, 0
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    B.gdn_prefill_noalloc(d)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    compare({"out": out.cpu(), "state_out": st.cpu(), "conv_state_out": cs.cpu()}, run_oracle(p), TOL_BF16)


def test_noalloc_rejects_scratch_beyond_its_array():
    cap = B.gdn_noalloc_scratch_bytes()
    assert cap == 32 << 20
    p = inputs.make_problem(503, [8], 2, 4, 128, 128, conv_kernel=4)
    call = runner.PrefillCall(p)
    C = p.channels
    d = B.gdn_prefill_desc()
    import ctypes
    ctypes.memmove(ctypes.byref(d), ctypes.byref(call.desc), ctypes.sizeof(d))
    d.T_total = cap // (C * 2) + 1           # scratch T_total * C * 2 bytes > the array
    with pytest.raises(B.GdnError) as e:
        B.gdn_prefill_noalloc(d)
    assert e.value.status == B.GDN_ERR_TOO_LARGE
