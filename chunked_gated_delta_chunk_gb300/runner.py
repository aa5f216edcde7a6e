"""Device-side plumbing around the C ABI: put a ``Problem`` in device memory,
allocate its outputs and workspace with torch, and call ``gdn_prefill_ex`` /
``gdn_step_ex`` through the ctypes binding.  Marshalling only: no arithmetic
of the method happens here.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import binding as B
from .inputs import Problem

DTYPE_CODE = {torch.bfloat16: B.GDN_BF16, torch.float32: B.GDN_FP32}


class PrefillCall:
    """Device buffers and the descriptor of one ``gdn_prefill_ex`` call.

    ``run()`` may be called repeatedly (benchmarking) and enqueues exactly one
    library call on the given stream.  ``state_in=None`` on the problem means
    a NULL incoming state (zero state)."""

    def __init__(self, p: Problem, device="cuda", chunk: Optional[int] = None,
                 state_in: Optional[torch.Tensor] = None, conv_state_in: Optional[torch.Tensor] = None,
                 write_state: bool = True, write_conv_state: bool = True,
                 alias_state: bool = False, alias_conv_state: bool = False,
                 segment_chunks: int = 0, split_prep: int = 0):
        self.p = p
        dev = torch.device(device)
        self.dev = dev
        T = p.T
        self.cu = p.cu_seqlens.to(dev, torch.int32)
        self.g = p.g.to(dev).contiguous()
        self.beta = p.beta.to(dev).contiguous()
        s_in = state_in if state_in is not None else p.state_in
        self.state_in = None if s_in is None else s_in.to(dev, torch.float32).contiguous()
        self.out = torch.empty(T, p.Hv, p.dv, dtype=p.dtype, device=dev)
        if alias_state:
            assert self.state_in is not None
            self.state_out = self.state_in
        else:
            self.state_out = (torch.empty(p.B, p.Hv, p.dk, p.dv, dtype=torch.float32, device=dev)
                              if write_state else None)
        self.q = self.k = self.v = None
        self.x = self.w = self.cs_in = self.cs_out = self.workspace = None
        fields = dict(dtype=DTYPE_CODE[p.dtype], B=p.B, Hk=p.Hk, Hv=p.Hv, dk=p.dk, dv=p.dv,
                      chunk=int(chunk or p.chunk), T_total=T, g=self.g, beta=self.beta,
                      state_in=self.state_in, state_out=self.state_out, out=self.out,
                      cu_seqlens=self.cu, use_qk_l2norm=int(p.use_l2norm),
                      q_scale=float(p.q_scale), segment_chunks=int(segment_chunks),
                      split_prep=int(split_prep))
        if p.conv is not None:
            self.x = p.conv["x"].to(dev).contiguous()
            self.w = p.conv["w"].to(dev, torch.float32).contiguous()
            cs = conv_state_in if conv_state_in is not None else p.conv.get("state_in")
            self.cs_in = None if cs is None else cs.to(dev, torch.float32).contiguous()
            K = p.conv["w"].shape[1]
            if alias_conv_state:
                assert self.cs_in is not None
                self.cs_out = self.cs_in
            else:
                self.cs_out = (torch.empty(p.B, p.channels, K - 1, dtype=torch.float32, device=dev)
                               if write_conv_state else None)
            fields.update(conv_x=self.x, conv_w=self.w, conv_state_in=self.cs_in,
                          conv_state_out=self.cs_out, conv_kernel=K,
                          conv_act=int(p.conv.get("act", 0)))
        else:
            self.q = p.q.to(dev).contiguous()
            self.k = p.k.to(dev).contiguous()
            self.v = p.v.to(dev).contiguous()
            fields.update(q=self.q, k=self.k, v=self.v)
        self.desc = B.make_desc(**fields)
        nbytes = B.gdn_workspace_bytes(self.desc)
        if nbytes:
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            self.desc.workspace = self.workspace.data_ptr()
            self.desc.workspace_bytes = nbytes
        self.workspace_bytes = nbytes

    def run(self, stream=None):
        B.gdn_prefill_ex(self.desc, stream)

    def results(self):
        r = {"out": self.out}
        if self.state_out is not None:
            r["state_out"] = self.state_out
        if self.cs_out is not None:
            r["conv_state_out"] = self.cs_out
        return r


def prefill(p: Problem, device="cuda", **kw):
    """One synchronous prefill of ``p``; returns CPU tensors."""
    call = PrefillCall(p, device, **kw)
    call.run()
    torch.cuda.synchronize(call.dev)
    return {k: v.cpu() for k, v in call.results().items()}


def step(q, k, v, g, beta, state, Hk, Hv, dk, dv, dtype=torch.bfloat16, conv=None,
         use_l2norm=True, q_scale=1.0, in_place=True, device="cuda"):
    """One decode step through ``gdn_step_ex``; tensors are moved to
    ``device``.  Returns (out, state_out[, conv_state_out]) on the device."""
    dev = torch.device(device)
    Bn = g.shape[0]
    g_d, b_d = g.to(dev).contiguous(), beta.to(dev).contiguous()
    s_in = None if state is None else state.to(dev, torch.float32).contiguous()
    s_out = s_in if (in_place and s_in is not None) else torch.empty(
        Bn, Hv, dk, dv, dtype=torch.float32, device=dev)
    out = torch.empty(Bn, Hv, dv, dtype=dtype, device=dev)
    fields = dict(dtype=DTYPE_CODE[dtype], B=Bn, Hk=Hk, Hv=Hv, dk=dk, dv=dv, g=g_d, beta=b_d,
                  state_in=s_in, state_out=s_out, out=out, use_qk_l2norm=int(use_l2norm),
                  q_scale=float(q_scale))
    keep = [g_d, b_d]
    cs_out = None
    if conv is not None:
        x = conv["x"].to(dev).contiguous()
        w = conv["w"].to(dev, torch.float32).contiguous()
        cs_in = None if conv.get("state_in") is None else conv["state_in"].to(dev, torch.float32).contiguous()
        K = w.shape[1]
        cs_out = cs_in if (in_place and cs_in is not None) else torch.empty(
            Bn, 2 * Hk * dk + Hv * dv, K - 1, dtype=torch.float32, device=dev)
        fields.update(conv_x=x, conv_w=w, conv_state_in=cs_in, conv_state_out=cs_out,
                      conv_kernel=K, conv_act=int(conv.get("act", 0)))
        keep += [x, w, cs_in]
    else:
        qd, kd, vd = (t.to(dev).contiguous() for t in (q, k, v))
        fields.update(q=qd, k=kd, v=vd)
        keep += [qd, kd, vd]
    desc = B.make_desc(**fields)
    B.gdn_step_ex(desc)
    torch.cuda.synchronize(dev)
    del keep
    return (out, s_out) if conv is None else (out, s_out, cs_out)


class ScanCall:
    """Device buffers of one ``gdn_scan_rows`` call over a ``ScanProblem``;
    ``run()`` enqueues the call on the given stream."""

    def __init__(self, p, device="cuda", alias_state: bool = False):
        dev = torch.device(device)
        self.p = p
        self.a = p.a.to(dev).contiguous()
        self.b = p.b.to(dev).contiguous()
        self.cu = p.cu_seqlens.to(dev, torch.int32)
        self.h_in = None if p.h_in is None else p.h_in.to(dev, torch.float32).contiguous()
        if alias_state:
            assert self.h_in is not None
            self.h_out = self.h_in
        else:
            self.h_out = torch.empty(p.B, p.C, dtype=torch.float32, device=dev)
        self.h_rows = torch.empty(p.T, p.C, dtype=torch.float32, device=dev)
        self.ws_bytes = B.gdn_scan_workspace_bytes(p.C, p.T)
        self.workspace = torch.empty(max(self.ws_bytes, 1), dtype=torch.uint8, device=dev)

    def run(self, stream=None):
        B.gdn_scan_rows(self.a, self.b, self.h_in, self.h_out, self.h_rows, self.cu, self.p.B,
                        self.p.C, self.p.T, self.workspace, self.ws_bytes, stream)


def scan_rows(p, device="cuda", **kw):
    """One synchronous selective scan of ``p``; returns CPU (h_rows, h_out)."""
    call = ScanCall(p, device, **kw)
    call.run()
    torch.cuda.synchronize(call.a.device)
    return call.h_rows.cpu(), call.h_out.cpu()


class WkvCall:
    """Device buffers of one ``gdn_wkv_rows`` call over a ``WkvProblem``."""

    def __init__(self, p, device="cuda", alias_state: bool = False):
        dev = torch.device(device)
        self.p = p
        self.k = p.k.to(dev).contiguous()
        self.v = p.v.to(dev).contiguous()
        self.w = p.w.to(dev, torch.float32).contiguous()
        self.u = p.u.to(dev, torch.float32).contiguous()
        self.cu = p.cu_seqlens.to(dev, torch.int32)
        self.state_in = None if p.state_in is None else p.state_in.to(dev, torch.float32).contiguous()
        if alias_state:
            assert self.state_in is not None
            self.state_out = self.state_in
        else:
            self.state_out = torch.empty(p.B, 3, p.C, dtype=torch.float32, device=dev)
        self.wkv = torch.empty(p.T, p.C, dtype=torch.float32, device=dev)
        self.ws_bytes = B.gdn_wkv_workspace_bytes(p.C, p.T)
        self.workspace = torch.empty(max(self.ws_bytes, 1), dtype=torch.uint8, device=dev)

    def run(self, stream=None):
        B.gdn_wkv_rows(self.k, self.v, self.w, self.u, self.state_in, self.state_out, self.wkv,
                       self.cu, self.p.B, self.p.C, self.p.T, self.workspace, self.ws_bytes, stream)


def wkv_rows(p, device="cuda", **kw):
    """One synchronous WKV call over ``p``; returns CPU (wkv, state_out)."""
    call = WkvCall(p, device, **kw)
    call.run()
    torch.cuda.synchronize(call.k.device)
    return call.wkv.cpu(), call.state_out.cpu()


class AttnCall:
    """Device buffers of one ``gdn_attn_rows`` call over an ``AttnProblem``
    (the caches are copied, so ``run()`` may be repeated: it rewrites the
    same appended rows)."""

    def __init__(self, p, device="cuda"):
        dev = torch.device(device)
        self.p = p
        self.q = p.q.to(dev).contiguous()
        self.k = p.k.to(dev).contiguous()
        self.v = p.v.to(dev).contiguous()
        self.k_cache = p.k_cache.to(dev).contiguous()
        self.v_cache = p.v_cache.to(dev).contiguous()
        self.cache_len = p.cache_len.to(dev, torch.int32)
        self.cu = p.cu_seqlens.to(dev, torch.int32)
        self.o = torch.empty_like(self.q)
        self.Hq, self.Hkv, self.D, self.cap = p.q.shape[1], p.k.shape[1], p.q.shape[2], p.k_cache.shape[2]

    def run(self, stream=None):
        B.gdn_attn_rows(self.q, self.k, self.v, self.k_cache, self.v_cache, self.cache_len, self.o,
                        self.cu, self.p.B, self.Hq, self.Hkv, self.D, self.cap, self.p.T, self.p.scale,
                        stream)


def attn_rows(p, device="cuda"):
    """One synchronous attention call; returns CPU (o, k_cache, v_cache)."""
    call = AttnCall(p, device)
    call.run()
    torch.cuda.synchronize(call.q.device)
    return call.o.cpu(), call.k_cache.cpu(), call.v_cache.cpu()
