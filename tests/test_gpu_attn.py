"""GPU parity of the full-attention rows (attention over the KV cache plus
the chunk's causal prefix, the chunk's k / v appended to the cache) through
the C ABI against the float64 oracle.

Tolerance: bf16 inputs and outputs with fp32 scores, softmax and
accumulation, like the main path's bf16 workloads: max|gpu - oracle| <=
1e-2 * max|oracle| per tensor; the cache rows are copies, so the updated
caches must match bit for bit.  Cases: the page's 11-row prompt (and its
7 + 4 split with the cache carried), query tiles and key tiles cut at every
boundary, ragged batches over non-empty caches, and the 4096-row benchmark
workload on sampled heads.
"""

import numpy as np
import pytest
import torch

from chunked_gated_delta_chunk_gb300 import binding as B
from chunked_gated_delta_chunk_gb300 import build as build_mod
from chunked_gated_delta_chunk_gb300 import inputs, runner
from oracle import attn_rows as ar

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()


def _rel(got, want):
    got = got.double().numpy() if hasattr(got, "numpy") else np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got))
    return np.abs(got - want).max() / max(np.abs(want).max(), 1e-30)


def _vs_oracle(p):
    o, kc, vc = runner.attn_rows(p)
    o_ref, kc_ref, vc_ref = ar.oracle_attn_rows(p.q, p.k, p.v, p.k_cache, p.v_cache, p.cache_len,
                                                p.cu_seqlens, p.scale)
    assert _rel(o, o_ref) <= TOL
    np.testing.assert_array_equal(kc.double().numpy(), kc_ref)
    np.testing.assert_array_equal(vc.double().numpy(), vc_ref)
    return o


def test_tiny_11_rows_over_cache():
    _vs_oracle(inputs.make_attn_config(1))


def test_7_plus_4_chained_equals_one_call():
    p = inputs.make_attn_config(1)
    o_all = _vs_oracle(p)
    p1 = inputs.AttnProblem(p.q[:7], p.k[:7], p.v[:7], p.k_cache, p.v_cache, p.cache_len,
                            torch.tensor([0, 7], dtype=torch.int32), p.scale)
    o1, kc1, vc1 = runner.attn_rows(p1)
    p2 = inputs.AttnProblem(p.q[7:], p.k[7:], p.v[7:], kc1, vc1, p.cache_len + 7,
                            torch.tensor([0, 4], dtype=torch.int32), p.scale)
    o2, _, _ = runner.attn_rows(p2)
    assert _rel(torch.cat([o1, o2]), o_all.double().numpy()) <= TOL


@pytest.mark.parametrize("lengths,caches,Hq,Hkv", [([1, 127, 128, 129, 300], [0, 1, 130, 0, 255], 4, 1),
                                                   ([256, 5], [128, 383], 2, 2), ([700], [0], 8, 2)])
def test_tile_boundaries(lengths, caches, Hq, Hkv):
    _vs_oracle(inputs.make_attn_problem(90 + len(lengths), lengths, caches, Hq, Hkv))


def test_ragged_config():
    _vs_oracle(inputs.make_attn_config(3))


def test_benchmark_workload_sampled_heads():
    """The full 4096-row call; the oracle runs query heads 0, 7 (kv head 0)
    and 8, 15 (kv head 1)."""
    p = inputs.make_attn_config(2)
    o, kc, vc = runner.attn_rows(p)
    for heads in ([0, 8], [7, 15]):
        o_ref, _, _ = ar.oracle_attn_rows(p.q[:, heads], p.k, p.v, p.k_cache, p.v_cache, p.cache_len,
                                          p.cu_seqlens, p.scale)
        assert _rel(o[:, heads], o_ref) <= TOL
    assert B.gdn_wait_timeouts() == 0
