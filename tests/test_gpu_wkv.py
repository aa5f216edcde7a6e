"""GPU parity of the RWKV-4 WKV rows through the C ABI against the float64
decoder-loop oracle.

fp32 like the page's unquantized builds.  Tolerance, derived from that
arithmetic: the decoder keeps `max` in fp32 and adds w to it every row, so
exp(max) carries a relative error that grows with the rows since `max` was
last reset by a dominant key (about rows x 2^-24 x |max|); on these inputs
the page's own decoder run in fp32 (``_fp32_decoder`` below) deviates from
the float64 oracle by up to 8e-5 of the output scale.  The bound is
max|gpu - oracle| <= 2e-4 * max|oracle| for outputs and num / den, the same
relative bound for max + log(den), and on the long sequence the GPU path must
also be no less accurate than 1.5 x the fp32 decoder.  The state (num, den,
max) is one representation of (A, B), so only its unique parts are compared;
the empty state is checked exactly.  Cases: the page's 75-row prompt and its 64 + 11 split,
large keys, ragged batches with empty and one-row sequences, absent and
aliased state, long sequences chained through the look-back, and the
4096-row, 4096-channel benchmark workload on sampled channels.
"""

import numpy as np
import pytest
import torch

from chunked_gated_delta_chunk_gb300 import binding as B
from chunked_gated_delta_chunk_gb300 import build as build_mod
from chunked_gated_delta_chunk_gb300 import inputs, runner
from oracle import wkv_rows as wr

pytestmark = pytest.mark.gpu
TOL = 2e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()


def _rel(got, want):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got))
    return np.abs(got - want).max() / max(np.abs(want).max(), 1e-30)


def _check_state(got, want):
    g_ratio, g_logb = wr.state_invariants(np.asarray(got, dtype=np.float64))
    w_ratio, w_logb = wr.state_invariants(want)
    assert _rel(g_ratio, w_ratio) <= TOL
    fin = np.isfinite(w_logb)
    assert np.array_equal(fin, np.isfinite(g_logb))
    if fin.any():
        assert _rel(g_logb[fin], w_logb[fin]) <= TOL


def _fp32_decoder(p):
    """The page's one-token decoder, row by row, in float32 (NumPy)."""
    k, v = p.k.numpy(), p.v.numpy()
    w, u = p.w.numpy(), p.u.numpy()
    out = np.zeros_like(k)
    for n in range(p.B):
        s = p.state_in[n].numpy() if p.state_in is not None else None
        num = s[0].copy() if s is not None else np.zeros_like(w)
        den = s[1].copy() if s is not None else np.zeros_like(w)
        mx = s[2].copy() if s is not None else np.full_like(w, -1e38)
        for t in range(int(p.cu_seqlens[n]), int(p.cu_seqlens[n + 1])):
            ww = u + k[t]
            q = np.maximum(mx, ww)
            e1, e2 = np.exp(mx - q), np.exp(ww - q)
            out[t] = (e1 * num + e2 * v[t]) / (e1 * den + e2)
            ww = mx + w
            q = np.maximum(ww, k[t])
            e1, e2 = np.exp(ww - q), np.exp(k[t] - q)
            num, den, mx = e1 * num + e2 * v[t], e1 * den + e2, q
    return out


def _vs_oracle(p, **kw):
    wkv, s_out = runner.wkv_rows(p, **kw)
    w_ref, s_ref = wr.oracle_wkv_rows(p.k, p.v, p.w, p.u, p.cu_seqlens, p.state_in)
    assert _rel(wkv.numpy(), w_ref) <= TOL
    _check_state(s_out.numpy(), s_ref)
    return wkv, s_out


def test_tiny_75_rows():
    _vs_oracle(inputs.make_wkv_config(1))


def test_64_plus_11_chained_equals_one_call():
    p = inputs.make_wkv_config(1)
    wkv, s_out = runner.wkv_rows(p)
    p1 = inputs.WkvProblem(p.k[:64], p.v[:64], p.w, p.u, torch.tensor([0, 64], dtype=torch.int32),
                           p.state_in)
    a1, s1 = runner.wkv_rows(p1)
    p2 = inputs.WkvProblem(p.k[64:], p.v[64:], p.w, p.u, torch.tensor([0, 11], dtype=torch.int32), s1)
    a2, s2 = runner.wkv_rows(p2)
    assert _rel(torch.cat([a1, a2]).numpy(), wkv.double().numpy()) <= TOL
    _check_state(s2.numpy(), s_out.double().numpy())


@pytest.mark.parametrize("lengths,C,big", [([1, 63, 64, 65, 0, 130, 1], 64, 0.05), ([5000], 256, 0.05),
                                           ([0, 700, 0], 132, 0.3), ([3] * 40, 128, 0.0)])
def test_ragged_long_and_large_keys(lengths, C, big):
    p = inputs.make_wkv_problem(80 + len(lengths), lengths, C, large_key_frac=big)
    wkv, _ = _vs_oracle(p)
    if lengths == [5000]:
        w_ref, _ = wr.oracle_wkv_rows(p.k, p.v, p.w, p.u, p.cu_seqlens, p.state_in)
        assert _rel(wkv.numpy(), w_ref) <= 1.5 * _rel(_fp32_decoder(p), w_ref)


def test_absent_and_aliased_state():
    p = inputs.make_wkv_problem(90, [300, 0, 90], 64, with_state=False)
    wkv, s_out = _vs_oracle(p)
    np.testing.assert_array_equal(s_out[1].numpy(),
                                  np.array([[0.0] * 64, [0.0] * 64, [-1e38] * 64], dtype=np.float32))
    q = inputs.make_wkv_problem(91, [300, 0, 90, 1], 64)
    call = runner.WkvCall(q, alias_state=True)
    call.run()
    torch.cuda.synchronize()
    w_ref, s_ref = wr.oracle_wkv_rows(q.k, q.v, q.w, q.u, q.cu_seqlens, q.state_in)
    assert _rel(call.wkv.cpu().numpy(), w_ref) <= TOL
    _check_state(call.state_out.cpu().numpy(), s_ref)


def test_ragged_config():
    _vs_oracle(inputs.make_wkv_config(3))


def test_benchmark_workload_sampled_channels():
    p = inputs.make_wkv_config(2)
    wkv, s_out = runner.wkv_rows(p)
    cols = np.unique(np.concatenate([np.arange(0, 128), np.arange(p.C - 128, p.C),
                                     np.random.default_rng(1).choice(p.C, 256, replace=False)]))
    w_ref, s_ref = wr.oracle_wkv_rows(p.k[:, cols], p.v[:, cols], p.w[cols], p.u[cols], p.cu_seqlens,
                                      p.state_in[:, :, cols])
    assert _rel(wkv[:, cols].numpy(), w_ref) <= TOL
    _check_state(s_out[:, :, cols].numpy(), s_ref)


def test_repeated_calls_and_no_wait_ran_out():
    p = inputs.make_wkv_problem(92, [2000, 37], 512)
    call = runner.WkvCall(p)
    for _ in range(3):
        call.run()
    torch.cuda.synchronize()
    w_ref, s_ref = wr.oracle_wkv_rows(p.k, p.v, p.w, p.u, p.cu_seqlens, p.state_in)
    assert _rel(call.wkv.cpu().numpy(), w_ref) <= TOL
    _check_state(call.state_out.cpu().numpy(), s_ref)
    assert B.gdn_wait_timeouts() == 0
