"""Test helpers: run the oracle on a workload (optionally on a sample of value
heads) and compare GPU results with it, tensor by tensor, relative to each
tensor's scale (the comparison the chunked-prefill pages' tests use).

Head sampling slices inputs only (the short conv is depthwise, so a channel
subset convolves exactly as in the full tensor); no arithmetic of the method
lives here.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle

TOL_BF16 = 1e-2   # bf16 inputs, fp32 accumulation and state
TOL_FP32 = 1e-5   # fp32 end to end


def tol_for(p):
    return TOL_FP32 if p.dtype == torch.float32 else TOL_BF16


def _sel_channels(p, heads):
    """Channel indices of the sub-problem: q heads, k heads, v heads."""
    group = p.Hv // p.Hk
    kheads = [h // group for h in heads]
    q_ch = [kh * p.dk + d for kh in kheads for d in range(p.dk)]
    k_ch = [p.Hk * p.dk + kh * p.dk + d for kh in kheads for d in range(p.dk)]
    v_ch = [2 * p.Hk * p.dk + h * p.dv + d for h in heads for d in range(p.dv)]
    return q_ch + k_ch + v_ch


def run_oracle(p, heads=None, state_in="problem", conv_state_in="problem", nthreads=0):
    """Oracle results for problem ``p``.  With ``heads`` (a list of value
    heads), only those heads are computed: ``out`` [T, n, dv], ``state_out``
    [B, n, dk, dv] and ``conv_state_out`` restricted to ``channels``."""
    s_in = p.state_in if state_in == "problem" else state_in
    cs_in = (p.conv.get("state_in") if p.conv is not None else None) \
        if isinstance(conv_state_in, str) else conv_state_in
    if heads is None:
        heads = list(range(p.Hv))
        full = True
    else:
        full = False
    n = len(heads)
    group = p.Hv // p.Hk
    kheads = [h // group for h in heads]
    g = p.g[:, heads]
    beta = p.beta[:, heads]
    s_sub = None if s_in is None else s_in[:, heads]
    res_extra = {}
    if p.conv is not None:
        ch = _sel_channels(p, heads) if not full else list(range(p.channels))
        idx = torch.tensor(ch, dtype=torch.long)
        if full:
            conv = dict(x=p.conv["x"], w=p.conv["w"], state_in=cs_in, act=p.conv.get("act", 0))
            Hk, Hv = p.Hk, p.Hv
        else:
            conv = dict(x=p.conv["x"].index_select(1, idx), w=p.conv["w"].index_select(0, idx),
                        state_in=None if cs_in is None else cs_in.index_select(1, idx),
                        act=p.conv.get("act", 0))
            Hk, Hv = n, n
        r = oracle.oracle_prefill(None, None, None, g if not full else p.g,
                                  beta if not full else p.beta, p.cu_seqlens, Hk, Hv, p.dk, p.dv,
                                  state_in=s_sub if not full else s_in, conv=conv,
                                  use_l2norm=p.use_l2norm, q_scale=p.q_scale, nthreads=nthreads)
        res_extra["channels"] = ch
    else:
        if full:
            q, k, v, Hk, Hv, gg, bb, ss = p.q, p.k, p.v, p.Hk, p.Hv, p.g, p.beta, s_in
        else:
            q, k, v = p.q[:, kheads], p.k[:, kheads], p.v[:, heads]
            Hk, Hv, gg, bb, ss = n, n, g, beta, s_sub
        r = oracle.oracle_prefill(q, k, v, gg, bb, p.cu_seqlens, Hk, Hv, p.dk, p.dv,
                                  state_in=ss, use_l2norm=p.use_l2norm, q_scale=p.q_scale,
                                  nthreads=nthreads)
    r.update(res_extra)
    r["heads"] = heads
    return r


def _np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def rel_err(gpu, ref):
    g, r = _np(gpu), _np(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    scale = np.abs(r).max() if r.size else 0.0
    err = np.abs(g - r).max() if r.size else 0.0
    return err / scale if scale > 0 else err


def assert_close(gpu, ref, tol, what=""):
    g = _np(gpu)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    e = rel_err(gpu, ref)
    assert e <= tol, f"{what}: max|gpu - oracle| / max|oracle| = {e:.3e} > {tol:.1e}"
    return e


def compare(gpu: dict, ref: dict, tol: float, heads=None):
    """Compare every tensor present in both dicts; returns the errors."""
    errs = {}
    h = ref.get("heads") if heads is None else heads
    out = gpu["out"]
    if h is not None and len(h) != out.shape[1]:
        out = out[:, h]
    errs["out"] = assert_close(out, ref["out"], tol, "out")
    if "state_out" in gpu:
        so = gpu["state_out"]
        if h is not None and len(h) != so.shape[1]:
            so = so[:, h]
        errs["state_out"] = assert_close(so, ref["state_out"], tol, "state_out")
    if "conv_state_out" in gpu and "conv_state_out" in ref:
        cs = gpu["conv_state_out"]
        ch = ref.get("channels")
        if ch is not None and len(ch) != cs.shape[1]:
            cs = cs[:, ch]
        # the new conv state is a copy of input columns: bit-exact
        errs["conv_state_out"] = assert_close(cs, ref["conv_state_out"], 0.0, "conv_state_out")
    return errs


def assert_all_finite(gpu: dict):
    """Every element of every returned tensor is finite (checked on the whole
    tensors, before any head selection)."""
    for name, t in gpu.items():
        assert torch.isfinite(t.float()).all(), f"{name}: non-finite values"


def compare_all_heads(gpu: dict, p, tol: float, batch: int = 8, **oracle_kw):
    """Compare every value head of ``gpu`` with the oracle, running the oracle
    over batches of ``batch`` heads to bound host memory.  The error of each
    tensor is its largest deviation over all heads divided by its largest
    oracle magnitude over all heads (the same per-tensor measure as
    ``compare``, taken over the whole tensor); the conv state is compared bit
    for bit on every channel."""
    assert_all_finite(gpu)
    err = {"out": 0.0, "state_out": 0.0}
    scale = {"out": 0.0, "state_out": 0.0}
    seen_channels = set()
    for h0 in range(0, p.Hv, batch):
        heads = list(range(h0, min(p.Hv, h0 + batch)))
        ref = run_oracle(p, heads=heads, **oracle_kw)
        pairs = [("out", gpu["out"][:, heads], ref["out"])]
        if "state_out" in gpu:
            pairs.append(("state_out", gpu["state_out"][:, heads], ref["state_out"]))
        for name, g, r in pairs:
            g, r = _np(g), _np(r)
            assert g.shape == r.shape, (name, g.shape, r.shape)
            if r.size:
                err[name] = max(err[name], float(np.abs(g - r).max()))
                scale[name] = max(scale[name], float(np.abs(r).max()))
        if "conv_state_out" in gpu and "conv_state_out" in ref:
            ch = ref["channels"]
            assert_close(gpu["conv_state_out"][:, ch], ref["conv_state_out"], 0.0, "conv_state_out")
            seen_channels.update(ch)
    if "conv_state_out" in gpu and p.conv is not None:
        assert len(seen_channels) == gpu["conv_state_out"].shape[1], "conv state: channels not all compared"
    out = {}
    for name in err:
        if name == "state_out" and "state_out" not in gpu:
            continue
        e = err[name] / scale[name] if scale[name] > 0 else err[name]
        assert e <= tol, f"{name}: max|gpu - oracle| / max|oracle| = {e:.3e} > {tol:.1e} (all heads)"
        out[name] = e
    return out
