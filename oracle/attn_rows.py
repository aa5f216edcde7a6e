"""Full-attention rows over a KV cache plus the chunk's causal prefix —
TEST INFRASTRUCTURE.

The Qwen3.5 chunked-prefill pull request ("perf(qwen3_5): prefill text
prompts in multi-token chunks", Implementation) builds the full-attention
layers of a prefill chunk as attention over the cache plus the chunk's causal
prefix (an attention mask of [S, cache + S]) and appends the chunk's
present k / v rows to the KV cache after the chunk.

Readings (the page states no more): softmax attention with scores
q . k * scale, scale = 1 / sqrt(head_dim) by default; GQA maps query head h
to kv head h / (Hq / Hkv); q and k arrive with their positional encoding
already applied (the model's business); the cache of sequence n holds
cache_len[n] rows; the chunk's rows are appended at cache_len[n] ..
cache_len[n] + L_n - 1, and row t of the chunk sees cache rows 0 ..
cache_len[n] - 1 and chunk rows 0 .. t.

``oracle_attn_rows`` is that definition in float64 NumPy (a matrix product
and a softmax per (sequence, head)); library routines serve as steps, with
no blocking or rescaling.
"""

from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def oracle_attn_rows(q, k, v, k_cache, v_cache, cache_len, cu_seqlens, scale=None):
    """q [T, Hq, D]; k, v [T, Hkv, D]; k_cache, v_cache [B, Hkv, cap, D];
    cache_len [B]; cu_seqlens [B+1].  Returns (o [T, Hq, D], k_cache_out,
    v_cache_out) in float64: the outputs and the caches with the chunk's rows
    appended."""
    q64, k64, v64 = _f64(q), _f64(k), _f64(v)
    kc, vc = _f64(k_cache).copy(), _f64(v_cache).copy()
    cl = np.asarray(_f64(cache_len), dtype=np.int64)
    cu = np.asarray(_f64(cu_seqlens), dtype=np.int64)
    T, Hq, D = q64.shape
    Hkv = k64.shape[1]
    group = Hq // Hkv
    s = 1.0 / np.sqrt(D) if scale is None else float(scale)
    o = np.zeros((T, Hq, D))
    for n in range(len(cu) - 1):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        L, c0 = t1 - t0, int(cl[n])
        kc[n, :, c0:c0 + L] = k64[t0:t1].transpose(1, 0, 2)
        vc[n, :, c0:c0 + L] = v64[t0:t1].transpose(1, 0, 2)
        if L == 0:
            continue
        # row t sees keys 0 .. c0 + t
        visible = np.arange(c0 + L)[None, :] <= (c0 + np.arange(L))[:, None]
        for h in range(Hq):
            kh = h // group
            scores = (q64[t0:t1, h] @ kc[n, kh, :c0 + L].T) * s
            scores = np.where(visible, scores, -np.inf)
            w = np.exp(scores - scores.max(axis=1, keepdims=True))
            w /= w.sum(axis=1, keepdims=True)
            o[t0:t1, h] = w @ vc[n, kh, :c0 + L]
    return o, kc, vc
