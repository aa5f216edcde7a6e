"""GPU parity of the selective-scan rows (h_t = a_t h_{t-1} + b_t) through the
C ABI against the float64 row-loop oracle.

Tolerance: fp32 like the page ("all in FP32"); per tensor max|gpu - oracle|
<= 1e-5 * max|oracle|.  Cases: the 75-row prompt of the page's test (and its
64 + 11 split), ragged batches with empty and one-row sequences, a NULL and
an aliased incoming state, long single sequences whose tiles chain through
the look-back, and the 4096-row, 24576-channel benchmark workload on sampled
channels.
"""

import numpy as np
import pytest
import torch

from chunked_gated_delta_chunk_gb300 import binding as B
from chunked_gated_delta_chunk_gb300 import build as build_mod
from chunked_gated_delta_chunk_gb300 import inputs, runner
from oracle import scan_rows as sr

pytestmark = pytest.mark.gpu
TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()


def _check(got, want, tol=TOL):
    got = got.double().numpy() if hasattr(got, "numpy") else got
    assert np.all(np.isfinite(got))
    scale = max(np.abs(want).max(), 1e-30)
    err = np.abs(got - want).max() / scale
    assert err <= tol, f"relative error {err:.3e} > {tol}"


def _vs_oracle(p, **kw):
    rows, out = runner.scan_rows(p, **kw)
    r_ref, o_ref = sr.oracle_scan_rows(p.a, p.b, p.cu_seqlens, p.h_in)
    _check(rows, r_ref)
    _check(out, o_ref)
    return rows, out


def test_tiny_75_rows():
    _vs_oracle(inputs.make_scan_config(1))


def test_64_plus_11_chained_equals_one_call():
    p = inputs.make_scan_config(1)
    rows, out = runner.scan_rows(p)
    p1 = inputs.ScanProblem(p.a[:64], p.b[:64], torch.tensor([0, 64], dtype=torch.int32), p.h_in)
    r1, o1 = runner.scan_rows(p1)
    p2 = inputs.ScanProblem(p.a[64:], p.b[64:], torch.tensor([0, 11], dtype=torch.int32), o1)
    r2, o2 = runner.scan_rows(p2)
    _check(torch.cat([r1, r2]), rows.double().numpy())
    _check(o2, out.double().numpy())


@pytest.mark.parametrize("lengths,C", [([1, 63, 64, 65, 0, 130, 1], 64), ([5000], 256),
                                       ([0, 0, 700, 0], 132), ([3] * 40, 128)])
def test_ragged_and_long(lengths, C):
    _vs_oracle(inputs.make_scan_problem(60 + len(lengths), lengths, C))


def test_null_state_and_aliased_state():
    p = inputs.make_scan_problem(70, [300, 0, 90], 64, h_sd=None)
    _vs_oracle(p)
    q = inputs.make_scan_problem(71, [300, 0, 90, 1], 64)
    call = runner.ScanCall(q, alias_state=True)
    call.run()
    torch.cuda.synchronize()
    r_ref, o_ref = sr.oracle_scan_rows(q.a, q.b, q.cu_seqlens, q.h_in)
    _check(call.h_rows.cpu(), r_ref)
    _check(call.h_out.cpu(), o_ref)


def test_ragged_config():
    _vs_oracle(inputs.make_scan_config(3))


def test_benchmark_workload_sampled_channels():
    """Full 4096 x 24576 call; the oracle runs on 640 sampled channels
    (channels are independent), including the first and last tiles."""
    p = inputs.make_scan_config(2)
    rows, out = runner.scan_rows(p)
    cols = np.unique(np.concatenate([np.arange(0, 128), np.arange(p.C - 128, p.C),
                                     np.random.default_rng(0).choice(p.C, 384, replace=False)]))
    r_ref, o_ref = sr.oracle_scan_rows(p.a[:, cols], p.b[:, cols], p.cu_seqlens, p.h_in[:, cols])
    _check(rows[:, cols], r_ref)
    _check(out[:, cols], o_ref)


def test_repeated_calls_reuse_workspace_and_no_wait_ran_out():
    p = inputs.make_scan_problem(72, [2000, 37], 512)
    call = runner.ScanCall(p)
    for _ in range(3):
        call.run()
    torch.cuda.synchronize()
    r_ref, o_ref = sr.oracle_scan_rows(p.a, p.b, p.cu_seqlens, p.h_in)
    _check(call.h_rows.cpu(), r_ref)
    _check(call.h_out.cpu(), o_ref)
    assert B.gdn_wait_timeouts() == 0
