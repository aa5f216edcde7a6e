"""Seeded synthetic inputs for the chunked Gated DeltaNet prefill.

This module only draws random numbers with the stated distributions; it holds
none of the method's arithmetic (no recurrence, no convolution, no cumulative
sum).  Unit-norm q/k vectors are *sampled* (a Gaussian vector divided by its
norm is a uniform draw on the sphere); the library's own L2 normalisation is
applied again by the GPU path and by the oracle.

Both the CUDA path (through the tests and ``bench.py``) and the float64 oracle
consume the tensors made here, so both sides see bit-identical values: every
floating-point input is drawn in fp32 and, for bf16 workloads, rounded to bf16
once here.

The five named workloads (sizes and distributions):

1. ``tiny``    B=1, Hk=Hv=1, dk=dv=16, T=75 (chunk 64: 64 + 11 rows), fp32.
               q, k ~ N(0,1) made unit-norm; v ~ N(0,1); beta = sigmoid(N(0,1));
               g = -softplus(N(0,1)); S_0 ~ N(0, 0.1).
2. ``prompt4k`` B=1, Hk=Hv=16, dk=dv=128, T=4096, chunk 64, bf16; q, k unit
               norm, v ~ N(0,1); beta = sigmoid(N(0,1)); g = -softplus(N(-2,1));
               S_0 = 0 (a zero state buffer).
3. ``ragged``  8 prompts with lengths uniform in [1, 8192]; Hk=16, Hv=32,
               dk=dv=128, bf16; raw x = [q|k|v] ~ N(0,1) over 8192 channels,
               conv weights ~ U(-0.5, 0.5) with kernel 4, prior conv state
               ~ N(0,1); S_0 ~ N(0, 0.05); beta and g as in ``prompt4k``.
4. ``stress``  2 sequences of 1024 tokens, H=8, dk=dv=128, bf16; per head a
               shared unit direction d; k = unit(d + 0.04 r n) with n a unit
               vector orthogonal to d and r ~ U(0,1) (cosine >= 0.9992);
               q unit norm; beta = sigmoid(6 + U(-0.5, 0.5)); g = -U(0, 20)
               except a quarter of the tokens with g = -U(0, 0.01);
               S_0 ~ N(0, 0.1).
5. ``long``    B=1, Hk=16, Hv=32, dk=dv=128, T=65536, bf16, conv kernel 4;
               as ``ragged`` but g = -softplus(N(-3,1)).  Its incoming state
               and conv state are the result of a prior 4096-token prompt
               drawn with the same distributions (``Problem.prior``); the
               caller runs that prior prompt (the oracle in tests, the GPU
               path in the benchmark) and fills ``state_in`` and
               ``conv["state_in"]``.

Standard deviations are the second parameter of N(., .).
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

CONFIG_NAMES = {1: "tiny", 2: "prompt4k", 3: "ragged", 4: "stress", 5: "long"}
BASE_SEED = 1000


@dataclass
class Problem:
    """One workload: tensors live on the CPU; the caller moves them."""
    name: str
    B: int
    Hk: int
    Hv: int
    dk: int
    dv: int
    chunk: int
    dtype: torch.dtype                 # element type of q, k, v, conv x and out
    cu_seqlens: torch.Tensor           # int32 [B+1]
    g: torch.Tensor                    # fp32 [T, Hv]
    beta: torch.Tensor                 # fp32 [T, Hv]
    q: Optional[torch.Tensor] = None   # [T, Hk, dk] (None when conv is used)
    k: Optional[torch.Tensor] = None
    v: Optional[torch.Tensor] = None   # [T, Hv, dv]
    state_in: Optional[torch.Tensor] = None   # fp32 [B, Hv, dk, dv] or None
    conv: Optional[dict] = None        # x [T, C], w fp32 [C, K], state_in fp32 [B, C, K-1], act
    use_l2norm: bool = True
    q_scale: float = 1.0
    prior: Optional["Problem"] = None  # prompt whose final state feeds this one
    extra: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def channels(self) -> int:
        return 2 * self.Hk * self.dk + self.Hv * self.dv

    def lengths(self):
        return (self.cu_seqlens[1:] - self.cu_seqlens[:-1]).tolist()


def _unit(x: torch.Tensor) -> torch.Tensor:
    """Sample on the unit sphere: a Gaussian draw divided by its norm."""
    return x / x.norm(dim=-1, keepdim=True)


def _cu(lengths) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def _round(x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    return x.to(dtype).contiguous()


def make_problem(seed: int, lengths, Hk: int, Hv: int, dk: int, dv: int, *,
                 dtype=torch.bfloat16, chunk: int = 64, conv_kernel: int = 0,
                 g_mu: float = -2.0, g_sd: float = 1.0, beta_mu: float = 0.0,
                 s0_sd: Optional[float] = 0.05, conv_state_sd: float = 1.0,
                 conv_act: int = 0, unit_qk: bool = True, name: str = "custom") -> Problem:
    """General recipe: q, k unit norm (or, with a conv prologue, raw x ~ N(0,1));
    v ~ N(0,1); beta = sigmoid(N(beta_mu, 1)); g = -softplus(N(g_mu, g_sd));
    S_0 ~ N(0, s0_sd) (None = no incoming state)."""
    gen = torch.Generator().manual_seed(seed)
    cu = _cu(lengths)
    T, B = int(cu[-1]), len(lengths)
    p = Problem(name=name, B=B, Hk=Hk, Hv=Hv, dk=dk, dv=dv, chunk=chunk, dtype=dtype,
                cu_seqlens=cu, g=torch.empty(0), beta=torch.empty(0))
    if conv_kernel:
        C = p.channels
        x = torch.randn(T, C, generator=gen)
        w = torch.rand(C, conv_kernel, generator=gen) - 0.5
        cs = torch.randn(B, C, conv_kernel - 1, generator=gen) * conv_state_sd
        p.conv = {"x": _round(x, dtype), "w": w.contiguous(), "state_in": cs.contiguous(),
                  "act": conv_act, "K": conv_kernel}
    else:
        q = torch.randn(T, Hk, dk, generator=gen)
        k = torch.randn(T, Hk, dk, generator=gen)
        if unit_qk:
            q, k = _unit(q), _unit(k)
        p.q, p.k = _round(q, dtype), _round(k, dtype)
        p.v = _round(torch.randn(T, Hv, dv, generator=gen), dtype)
    p.beta = torch.sigmoid(torch.randn(T, Hv, generator=gen) + beta_mu).contiguous()
    p.g = (-torch.nn.functional.softplus(torch.randn(T, Hv, generator=gen) * g_sd + g_mu)).contiguous()
    if s0_sd is not None:
        p.state_in = (torch.randn(B, Hv, dk, dv, generator=gen) * s0_sd).contiguous()
    return p


def make_stress(seed: int, n_seq: int = 2, L: int = 1024, H: int = 8, d: int = 128,
                dtype=torch.bfloat16, chunk: int = 64, name: str = "stress") -> Problem:
    """Nearly parallel keys with beta near one and decays down to -20 per token."""
    gen = torch.Generator().manual_seed(seed)
    cu = _cu([L] * n_seq)
    T = n_seq * L
    direction = _unit(torch.randn(H, d, generator=gen))                   # [H, d]
    n = torch.randn(T, H, d, generator=gen)
    n = n - (n * direction).sum(-1, keepdim=True) * direction               # orthogonal part
    n = _unit(n)
    r = torch.rand(T, H, 1, generator=gen)
    k = _unit(direction.unsqueeze(0) + 0.04 * r * n)
    q = _unit(torch.randn(T, H, d, generator=gen))
    v = torch.randn(T, H, d, generator=gen)
    beta = torch.sigmoid(6.0 + (torch.rand(T, H, generator=gen) - 0.5))
    g = -20.0 * torch.rand(T, H, generator=gen)
    slow = torch.rand(T, H, generator=gen) < 0.25
    g = torch.where(slow, -0.01 * torch.rand(T, H, generator=gen), g)
    s0 = torch.randn(n_seq, H, d, d, generator=gen) * 0.1
    return Problem(name=name, B=n_seq, Hk=H, Hv=H, dk=d, dv=d, chunk=chunk, dtype=dtype,
                   cu_seqlens=cu, g=g.contiguous(), beta=beta.contiguous(),
                   q=_round(q, dtype), k=_round(k, dtype), v=_round(v, dtype),
                   state_in=s0.contiguous())


def ragged_lengths(seed: int, n: int = 8, lo: int = 1, hi: int = 8192):
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


def make_config(i: int, *, with_prior: bool = True) -> Problem:
    """The five named workloads (see the module docstring)."""
    seed = BASE_SEED + i
    if i == 1:
        p = make_problem(seed, [75], 1, 1, 16, 16, dtype=torch.float32, g_mu=0.0,
                         s0_sd=0.1, name="tiny")
    elif i == 2:
        p = make_problem(seed, [4096], 16, 16, 128, 128, s0_sd=None, name="prompt4k")
        p.state_in = torch.zeros(1, 16, 128, 128)
    elif i == 3:
        p = make_problem(seed, ragged_lengths(seed + 100), 16, 32, 128, 128, conv_kernel=4,
                         s0_sd=0.05, name="ragged")
    elif i == 4:
        p = make_stress(seed)
    elif i == 5:
        p = make_problem(seed, [65536], 16, 32, 128, 128, conv_kernel=4, g_mu=-3.0,
                         s0_sd=None, name="long")
        if with_prior:
            p.prior = make_problem(seed + 500, [4096], 16, 32, 128, 128, conv_kernel=4,
                                   g_mu=-3.0, s0_sd=None, name="long-prior")
    else:
        raise ValueError(f"unknown workload {i}")
    return p


# ---------------------------------------------------------------- selective-scan rows
@dataclass
class ScanProblem:
    """Inputs of the selective-scan rows h_t = a_t h_{t-1} + b_t: a, b
    [T, C] fp32 (token-major), cu_seqlens [B+1] int32, h_in [B, C] fp32 or
    None (zero state)."""
    a: torch.Tensor
    b: torch.Tensor
    cu_seqlens: torch.Tensor
    h_in: Optional[torch.Tensor]
    name: str = ""

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def B(self) -> int:
        return int(self.cu_seqlens.numel() - 1)

    @property
    def C(self) -> int:
        return int(self.a.shape[1])


def make_scan_problem(seed: int, lengths, C: int, *, a_mu: float = -2.0, a_sd: float = 1.0,
                      b_sd: float = 1.0, h_sd: Optional[float] = 0.1, name: str = "") -> ScanProblem:
    """Decays a = exp(-softplus(N(a_mu, a_sd))) in (0, 1] (the page's decay
    factors), inputs b ~ N(0, b_sd), incoming state h ~ N(0, h_sd) (None:
    no state, i.e. zero).  Drawn in fp32 on the CPU."""
    gen = torch.Generator().manual_seed(seed)
    cu = _cu(lengths)
    T = int(cu[-1])
    a = torch.exp(-torch.nn.functional.softplus(a_mu + a_sd * torch.randn(T, C, generator=gen)))
    b = b_sd * torch.randn(T, C, generator=gen)
    h = None if h_sd is None else h_sd * torch.randn(len(lengths), C, generator=gen)
    return ScanProblem(a.contiguous(), b.contiguous(), cu, h, name)


def make_scan_config(i: int) -> ScanProblem:
    """Selective-scan workloads, sized after the Mamba page's model family
    (mamba-130m: 1536 inner channels x 16 state entries = 24576 scan channels):

    1. ``scan-tiny``   B=1, C=16, T=75 (64 + 11 rows).
    2. ``scan-4k``     B=1, C=24576, T=4096 (the benchmark workload).
    3. ``scan-ragged`` 8 prompts with lengths uniform in [1, 2048], C=1536."""
    seed = BASE_SEED + 100 + i
    if i == 1:
        return make_scan_problem(seed, [75], 16, a_mu=0.0, name="scan-tiny")
    if i == 2:
        return make_scan_problem(seed, [4096], 24576, name="scan-4k")
    if i == 3:
        return make_scan_problem(seed, ragged_lengths(seed + 100, hi=2048), 1536, name="scan-ragged")
    raise ValueError(f"unknown scan workload {i}")


# ---------------------------------------------------------------- RWKV-4 WKV rows
@dataclass
class WkvProblem:
    """Inputs of the RWKV-4 WKV rows: k, v [T, C] fp32, per-channel decay
    exponent w [C] (exp(w) in (0, 1)) and bonus u [C], cu_seqlens [B+1],
    state_in [B, 3, C] (num, den, max) or None."""
    k: torch.Tensor
    v: torch.Tensor
    w: torch.Tensor
    u: torch.Tensor
    cu_seqlens: torch.Tensor
    state_in: Optional[torch.Tensor]
    name: str = ""

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def B(self) -> int:
        return int(self.cu_seqlens.numel() - 1)

    @property
    def C(self) -> int:
        return int(self.k.shape[1])


def make_wkv_problem(seed: int, lengths, C: int, *, large_key_frac: float = 0.05,
                     with_state: bool = True, name: str = "") -> WkvProblem:
    """Decays w = -exp(U(-5, 3)) and bonuses u ~ N(0.5, 1) per channel (the
    spread of trained checkpoints the page's test covers); keys k ~ N(0, 1)
    with a fraction replaced by large keys +-U(20, 40); values v ~ N(0, 1);
    state num = den * N(0, 1), den = exp(N(0, 1)), max ~ N(0, 2)."""
    gen = torch.Generator().manual_seed(seed)
    cu = _cu(lengths)
    T = int(cu[-1])
    w = -torch.exp(-5.0 + 8.0 * torch.rand(C, generator=gen))
    u = 0.5 + torch.randn(C, generator=gen)
    k = torch.randn(T, C, generator=gen)
    big = torch.rand(T, C, generator=gen) < large_key_frac
    sign = torch.where(torch.rand(T, C, generator=gen) < 0.5, -1.0, 1.0)
    k = torch.where(big, sign * (20.0 + 20.0 * torch.rand(T, C, generator=gen)), k)
    v = torch.randn(T, C, generator=gen)
    state = None
    if with_state:
        den = torch.exp(torch.randn(len(lengths), C, generator=gen))
        num = den * torch.randn(len(lengths), C, generator=gen)
        mx = 2.0 * torch.randn(len(lengths), C, generator=gen)
        state = torch.stack([num, den, mx], dim=1).contiguous()
    return WkvProblem(k.contiguous(), v.contiguous(), w, u, cu, state, name)


def make_wkv_config(i: int) -> WkvProblem:
    """WKV workloads, sized after the RWKV-4 family the page builds:

    1. ``wkv-tiny``   B=1, C=16, T=75 (64 + 11 rows).
    2. ``wkv-4k``     B=1, C=4096 (the 7B model's width), T=4096: the
                      benchmark workload.
    3. ``wkv-ragged`` 8 prompts with lengths uniform in [1, 2048], C=768
                      (the 169M model the page measures)."""
    seed = BASE_SEED + 200 + i
    if i == 1:
        return make_wkv_problem(seed, [75], 16, name="wkv-tiny")
    if i == 2:
        return make_wkv_problem(seed, [4096], 4096, name="wkv-4k")
    if i == 3:
        return make_wkv_problem(seed, ragged_lengths(seed + 100, hi=2048), 768, name="wkv-ragged")
    raise ValueError(f"unknown WKV workload {i}")


# ---------------------------------------------------------------- attention rows
@dataclass
class AttnProblem:
    """Inputs of the full-attention rows: q [T, Hq, D], k, v [T, Hkv, D]
    (bf16 values), a KV cache k_cache, v_cache [B, Hkv, cap, D] holding
    cache_len[n] rows per sequence, cu_seqlens [B+1]."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    cache_len: torch.Tensor
    cu_seqlens: torch.Tensor
    scale: float
    name: str = ""

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def B(self) -> int:
        return int(self.cu_seqlens.numel() - 1)


def make_attn_problem(seed: int, lengths, cache_lens, Hq: int, Hkv: int, D: int = 128, cap: Optional[int] = None,
                      *, dtype: torch.dtype = torch.bfloat16, name: str = "") -> AttnProblem:
    """q, k, v ~ N(0, 1); the cache's first cache_len[n] rows ~ N(0, 1), the
    rest of its capacity zero; scale 1 / sqrt(D)."""
    gen = torch.Generator().manual_seed(seed)
    cu = _cu(lengths)
    T = int(cu[-1])
    B = len(lengths)
    if cap is None:
        cap = max(int(c) + int(n) for c, n in zip(cache_lens, lengths))
        cap = max(64, -(-cap // 64) * 64)
    q = torch.randn(T, Hq, D, generator=gen)
    k = torch.randn(T, Hkv, D, generator=gen)
    v = torch.randn(T, Hkv, D, generator=gen)
    kc = torch.zeros(B, Hkv, cap, D)
    vc = torch.zeros(B, Hkv, cap, D)
    for n, c in enumerate(cache_lens):
        kc[n, :, :c] = torch.randn(Hkv, int(c), D, generator=gen)
        vc[n, :, :c] = torch.randn(Hkv, int(c), D, generator=gen)
    r = lambda x: _round(x, dtype)
    return AttnProblem(r(q), r(k), r(v), r(kc), r(vc), torch.tensor(cache_lens, dtype=torch.int32), cu,
                       1.0 / D ** 0.5, name)


def make_attn_config(i: int) -> AttnProblem:
    """Attention workloads (GQA 16 query / 2 kv heads, head dim 128, bf16):

    1. ``attn-tiny``  11 rows (the page's 7 + 4 test shape) over a 5-row cache, Hq=4, Hkv=2.
    2. ``attn-4k``    one 4096-row prompt, empty cache: the benchmark workload.
    3. ``attn-ragged`` 4 prompts U[1, 1024] over caches U[0, 2048]."""
    seed = BASE_SEED + 300 + i
    if i == 1:
        return make_attn_problem(seed, [11], [5], 4, 2, name="attn-tiny")
    if i == 2:
        return make_attn_problem(seed, [4096], [0], 16, 2, name="attn-4k")
    if i == 3:
        lens = ragged_lengths(seed + 100, n=4, hi=1024)
        caches = ragged_lengths(seed + 200, n=4, lo=0, hi=2048)
        return make_attn_problem(seed, lens, caches, 16, 2, name="attn-ragged")
    raise ValueError(f"unknown attention workload {i}")
