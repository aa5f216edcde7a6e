"""Benchmark: chunked Gated DeltaNet prefill throughput on one GB300.

One step = one ``gdn_prefill_ex`` call over the whole workload (every stage
of the hot path: the optional short conv, the chunk solve and the chunk-to-
chunk state propagation), inputs resident in HBM.  Default workload: the
4096-token prompt, B=1, Hk=Hv=16, dk=dv=128, chunk 64, bf16 q/k/v/out, fp32
g/beta/state, zero incoming state.

Prints ONE JSON line (rank 0) with tokens/s, the roofline of the dominant
kernel (algorithmic bytes / CUDA-event time vs the measured HBM peak), the
end-to-end number through the C ABI with host buffers, the clocks seen during
the timed region and the float64 CPU oracle timed on the host's cores.

L2: the workload (~70 MB) fits in the 129 MB L2, so the timed steps rotate
through enough independent copies of the inputs and outputs that each step
touches buffers last used more than 2 x L2 bytes earlier.

``--impl reference`` times the float64 oracle (the only reference that
exists for this method) on the host cores instead, on the same workload.
Under torchrun (N > 1) every rank runs its own replica (the path shards over
independent prompts with no exchange); rank 0 prints.
"""

from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FALLBACK_BYTES = 129 * 1024 * 1024   # GB300 L2, used only when the device cannot be queried
L2_NOTE = "rotating independent buffer sets: each timed step touches buffers last used more than 2 x L2 bytes earlier"


def l2_bytes(dev=None):
    """The device's L2 size (cudaDevAttrL2CacheSize through torch)."""
    try:
        import torch
        if torch.cuda.is_available():
            n = int(torch.cuda.get_device_properties(dev if dev is not None else 0).L2_cache_size)
            if n > 0:
                return n
    except (AttributeError, RuntimeError, AssertionError):
        pass
    return L2_FALLBACK_BYTES


def config_dict(workload, p, world):
    """The `config` object of both arms' JSON lines (identical for the same
    workload and launch)."""
    return {"workload": workload, "global_batch": p.B, "seq_len": p.T,
            "parallelism": "replicas" if world > 1 else "single", "l2": L2_NOTE}
WORKLOADS = {
    2: "prompt4k: B=1, Hk=Hv=16, dk=dv=128, T=4096, chunk 64, bf16 q/k/v/out, fp32 g/beta/state",
    4: "stress: B=2 x 1024 tokens, H=8, dk=dv=128, chunk 64, bf16, nearly parallel keys",
    5: "long: B=1, T=65536, Hk=16, Hv=32, dk=dv=128, conv K=4, chunk 64, bf16",
    3: "ragged: 8 prompts U[1,8192], Hk=16, Hv=32, dk=dv=128, conv K=4, chunk 64, bf16",
}
METRIC = "prefill tokens/s (1 GB300) and % of roofline, dk=dv=128, 4096-token prompt"


def algorithmic_bytes(p) -> int:
    """Inputs read once + outputs written once + state in/out (per call)."""
    es = 2 if str(p.dtype).endswith("bfloat16") else 4
    T = p.T
    b = 0
    if p.conv is not None:
        K = p.conv["w"].shape[1]
        b += T * p.channels * es + p.channels * K * 4 + 2 * p.B * p.channels * (K - 1) * 4
    else:
        b += T * (2 * p.Hk * p.dk + p.Hv * p.dv) * es
    b += T * p.Hv * 8                     # g, beta
    b += T * p.Hv * p.dv * es             # out
    b += 2 * p.B * p.Hv * p.dk * p.dv * 4  # state in + out
    b += (p.B + 1) * 4
    return b


def algorithmic_flops(p, C=64) -> int:
    """Full 64-row tiles: per k-head token 4*C*dk (K K^T, Q K^T); per v-head
    token 6*dk*dv + 4*C*dv (K S_0, Q S_0, K~^T U; T rhs, P U)."""
    T = p.T
    return T * (p.Hk * 4 * C * p.dk + p.Hv * (6 * p.dk * p.dv + 4 * C * p.dv))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


def _code_only(text):
    """C/C++ source without its comments and whitespace (so that a comment
    edit leaves a kernel's hash, and its recorded counters, valid)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":                       # string or character literal
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "".join("".join(out).split())


def kernel_source_hash(sources):
    """Hash of the code of the kernel's source files (names under the
    package's csrc/), comments and whitespace left out."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "chunked_gated_delta_chunk_gb300", "csrc")
    for name in sorted(sources):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_name, workload):
    """DRAM bytes (read + write) of the kernel's launches in one step, from
    the committed ncu summary, if it was taken on this workload (its short
    name, before the colon) and on the kernel's current source files (the
    entry lists them); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    entry = d.get(kernel_name)
    if not entry or not entry.get("sources") or entry.get("workload") != workload.split(":")[0]:
        return None
    try:
        if entry.get("source_hash") != kernel_source_hash(entry["sources"]):
            return None
    except OSError:
        return None
    return entry.get("dram_bytes_per_step")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_tokens_per_s(p, budget_s=12.0, nthreads=0):
    """The float64 oracle, as it stands, on the host cores (``nthreads`` = 0:
    all of them): whole-workload passes repeated until ``budget_s`` of wall
    time, or, for a single prompt whose one pass would take longer than the
    budget, a prefix of the prompt sized to it (the oracle's cost is linear in
    tokens).  Returns (tokens/s, threads used, what was timed)."""
    import oracle
    oracle.build_oracle()
    cores = oracle.max_threads() if nthreads <= 0 else nthreads
    run = lambda q: oracle.oracle_prefill(q.q, q.k, q.v, q.g, q.beta, q.cu_seqlens, q.Hk, q.Hv, q.dk, q.dv,
                                          state_in=q.state_in, conv=q.conv, use_l2norm=q.use_l2norm,
                                          q_scale=q.q_scale, nthreads=nthreads)
    sample, S = p, p.T
    if p.B == 1:
        probe = min(256, p.T)
        t0 = time.perf_counter()
        run(_prefix(p, probe))
        per_token = (time.perf_counter() - t0) / probe
        if per_token * p.T > budget_s:
            S = int(max(64, budget_s / 2 / max(per_token, 1e-12)))
            sample = _prefix(p, S)
    done, t0 = 0, time.perf_counter()
    while True:
        run(sample)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    what = (f"{done} full passes of the workload ({p.T} tokens each) in {el:.1f} s" if S == p.T else
            f"{done} passes over the first {S} of {p.T} tokens, all heads, in {el:.1f} s")
    return S * done / el, cores, what


def make_workload(cfg):
    from chunked_gated_delta_chunk_gb300 import inputs
    p = inputs.make_config(cfg)
    if cfg == 5:
        # incoming state: the GPU path's own result for the prior 4096-token prompt
        from chunked_gated_delta_chunk_gb300 import runner
        import torch
        r = runner.prefill(p.prior)
        p.state_in = r["state_out"]
        p.conv["state_in"] = r["conv_state_out"]
        torch.cuda.empty_cache()
    return p


def _prefix(p, S):
    """The first S tokens of a single-sequence workload (inputs only)."""
    import copy
    q = copy.copy(p)
    q.cu_seqlens = p.cu_seqlens.clone()
    q.cu_seqlens[-1] = S
    q.g, q.beta = p.g[:S], p.beta[:S]
    if p.conv is not None:
        q.conv = dict(p.conv, x=p.conv["x"][:S])
    else:
        q.q, q.k, q.v = p.q[:S], p.k[:S], p.v[:S]
    return q


def run_reference(args, rank, world):
    """The float64 oracle as it stands, on the host cores, on the same
    workload; each step is a prefix of the prompt sized so that all steps
    together take about --reference-seconds (two minutes by default; tokens/s
    is then tokens of the prefix over its time: the oracle's cost is linear in
    tokens)."""
    if rank != 0:
        return
    import oracle
    from chunked_gated_delta_chunk_gb300 import inputs
    oracle.build_oracle()
    p = inputs.make_config(args.config, with_prior=False)
    run = lambda q: oracle.oracle_prefill(q.q, q.k, q.v, q.g, q.beta, q.cu_seqlens, q.Hk, q.Hv,
                                          q.dk, q.dv, state_in=q.state_in, conv=q.conv,
                                          use_l2norm=q.use_l2norm, q_scale=q.q_scale)
    if p.B == 1:
        probe = min(256, p.T)
        t0 = time.perf_counter()
        run(_prefix(p, probe))
        per_token = (time.perf_counter() - t0) / probe
        S = int(min(p.T, max(64, args.reference_seconds / max(args.steps, 1) / max(per_token, 1e-9))))
        sample = _prefix(p, S)
        what = f"first {S} of {p.T} tokens, all heads, per step"
    else:
        sample, S = p, p.T
        what = f"the whole workload ({p.T} tokens) per step"
    t_all = time.perf_counter()
    for _ in range(args.steps):
        run(sample)
    total = time.perf_counter() - t_all
    tps = S * args.steps / total
    cores = oracle.max_threads()
    line = {"metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": config_dict(WORKLOADS[args.config], p, world),
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": what},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


SCAN_METRIC = "selective-scan rows: tokens/s (1 GB300) and % of HBM roofline, 24576 channels, 4096-token prompt"
SCAN_WORKLOAD = "scan-4k: B=1, T=4096, C=24576 (1536 x 16), fp32 a, b, h"
WKV_METRIC = "RWKV-4 WKV rows: tokens/s (1 GB300) and % of HBM roofline, 4096 channels, 4096-token prompt"
WKV_WORKLOAD = "wkv-4k: B=1, T=4096, C=4096 (RWKV-4 7B width), fp32 k, v, wkv"
ATTN_METRIC = "full-attention rows: tokens/s (1 GB300) and % of bf16 tensor roofline, 4096-token prompt, Hq=16, Hkv=2, d=128"
ATTN_WORKLOAD = "attn-4k: B=1, T=4096 over an empty cache, Hq=16, Hkv=2, head dim 128, bf16"


class _RowSpec:
    """What the bench needs to know about one row recurrence."""

    def __init__(self, kind):
        from chunked_gated_delta_chunk_gb300 import inputs, runner
        self.kind = kind
        if kind == "scan":
            self.metric, self.workload = SCAN_METRIC, SCAN_WORKLOAD
            self.p = inputs.make_scan_config(2)
            self.make_call = runner.ScanCall
            self.inputs, self.outputs = ("a", "b", "h_in"), ("h_rows", "h_out")
            # a, b read once, h_rows written once, h_in read, h_out written
            self.nbytes = (3 * self.p.T + 2 * self.p.B) * self.p.C * 4
        elif kind == "attn":
            self.metric, self.workload = ATTN_METRIC, ATTN_WORKLOAD
            self.p = inputs.make_attn_config(2)
            self.make_call = runner.AttnCall
            self.inputs, self.outputs = ("q", "k", "v", "k_cache", "v_cache"), ("o", "k_cache", "v_cache")
            p = self.p
            Hq, Hkv, D = p.q.shape[1], p.k.shape[1], p.q.shape[2]
            # q, k, v read once, o written once, the appended k / v rows written once
            self.nbytes = p.T * (2 * Hq + 4 * Hkv) * D * 2
            # Q K^T and P V over the causal prefix: 4 D flops per (query, visible key)
            visible = sum((int(c) + i + 1) for c, L in zip(p.cache_len.tolist(),
                                                             (p.cu_seqlens[1:] - p.cu_seqlens[:-1]).tolist())
                          for i in range(int(L)))
            self.nflops = 4 * D * Hq * visible
        else:
            self.metric, self.workload = WKV_METRIC, WKV_WORKLOAD
            self.p = inputs.make_wkv_config(2)
            self.make_call = runner.WkvCall
            self.inputs, self.outputs = ("k", "v", "w", "u", "state_in"), ("wkv", "state_out")
            # k, v read once, wkv written once, w, u, and the (num, den, max) state in and out
            self.nbytes = (3 * self.p.T + 2 + 6 * self.p.B) * self.p.C * 4

    def oracle_pass(self, cols):
        """One float64 oracle pass over the first ``cols`` channels (query
        heads for the attention rows)."""
        p = self.p
        if self.kind == "attn":
            from oracle import attn_rows as ar
            ar.oracle_attn_rows(self._q, p.k[:self._rows], p.v[:self._rows], p.k_cache, p.v_cache,
                                p.cache_len, [0, self._rows], p.scale)
            return
        if self.kind == "scan":
            from oracle import scan_rows as sr
            sr.oracle_scan_rows(self._a, self._b, p.cu_seqlens, self._h)
        else:
            from oracle import wkv_rows as wr
            wr.oracle_wkv_rows(self._k, self._v, self._w, self._u, p.cu_seqlens, self._s)

    def sample(self, cols):
        p = self.p
        if self.kind == "attn":
            # the first ``cols`` query rows, every head (the oracle is quadratic in rows)
            self._rows = cols
            self._q = p.q[:cols]
            return
        if self.kind == "scan":
            self._a, self._b, self._h = (p.a[:, :cols].numpy(), p.b[:, :cols].numpy(),
                                         p.h_in[:, :cols].numpy())
        else:
            self._k, self._v = p.k[:, :cols].numpy(), p.v[:, :cols].numpy()
            self._w, self._u = p.w[:cols].numpy(), p.u[:cols].numpy()
            self._s = p.state_in[:, :, :cols].numpy()


def timed_steps(calls, steps, stream, barrier, launches_per_call=0, clocks=None):
    """Time `steps` library calls on the stream with CUDA events, barrier and
    device synchronisation on both sides.  launches_per_call > 0 turns the
    library's launch timer on (CUDA events around every one of its launches),
    which adds a little time per launch: the headline number is taken with it
    off, the per-kernel device times in a second region with it on.
    Returns (ms for all steps, launch records, dropped launches)."""
    import torch
    from chunked_gated_delta_chunk_gb300 import binding as B
    if launches_per_call:
        B.gdn_launch_timer_start(steps * launches_per_call)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ctx = clocks if clocks is not None else contextlib.nullcontext()
    with ctx:
        barrier()
        start.record(stream)
        for i in range(steps):
            calls[i % len(calls)].run(stream)
        stop.record(stream)
        barrier()
    records, dropped = [], 0
    if launches_per_call:
        B.gdn_launch_timer_stop()
        records, dropped = B.gdn_launch_timer_read()
    return start.elapsed_time(stop), records, dropped


def timed_blocks(calls, steps, stream, barrier, dev, min_seconds, clocks):
    """The K-step timed region of ``timed_steps``, repeated back to back until
    about ``min_seconds`` have passed (the same repeat count on every rank:
    the first block's time, max over ranks, sizes it), so that the clock
    sampler sees the GPU under load.  Returns the per-block times in ms."""
    first, _, _ = timed_steps(calls, steps, stream, barrier)
    first = max_over_ranks(first, dev)
    reps = max(1, min(200000, int(math.ceil(min_seconds * 1e3 / max(first, 1e-6)))))
    blocks = []
    with clocks:
        for _ in range(reps):
            ms, _, _ = timed_steps(calls, steps, stream, barrier)
            blocks.append(ms)
    return blocks


def max_over_ranks(value, dev):
    """The largest of every rank's value (the job's time is its slowest
    rank's); the value itself outside a process group of more than one."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() < 2:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def e2e_steps_ms(bufs, host_in, host_out, steps, barrier, dev):
    """End to end through host buffers: every step copies its inputs from
    pinned host memory into device set i % len(bufs) (an upload stream), runs
    the library call on that set (a compute stream) and copies its outputs
    back into pinned host memory (a download stream), so the upload of step
    i + 1 and the download of step i - 1 overlap the kernels of step i.
    Events order every reuse of a device set: its inputs are overwritten only
    after the call that read them, its outputs only after their download.
    Returns ms per step from the first timed upload to the last download."""
    import torch
    up, comp, down = (torch.cuda.Stream(dev) for _ in range(3))
    nb = len(bufs)
    comp_done, down_done = [None] * nb, [None] * nb
    e0 = e1 = None
    for it in range(steps + 2):                       # two untimed steps first
        b = it % nb
        if it == 2:
            barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record(up)
        if comp_done[b] is not None:
            up.wait_event(comp_done[b])
        with torch.cuda.stream(up):
            for n, t in host_in.items():
                getattr(bufs[b], n).copy_(t, non_blocking=True)
        landed = torch.cuda.Event()
        landed.record(up)
        comp.wait_event(landed)
        if down_done[b] is not None:
            comp.wait_event(down_done[b])
        bufs[b].run(comp)
        comp_done[b] = torch.cuda.Event()
        comp_done[b].record(comp)
        down.wait_event(comp_done[b])
        with torch.cuda.stream(down):
            for n, t in host_out.items():
                t.copy_(getattr(bufs[b], n), non_blocking=True)
        down_done[b] = torch.cuda.Event()
        down_done[b].record(down)
    e1 = torch.cuda.Event(enable_timing=True)
    e1.record(down)
    barrier()
    return e0.elapsed_time(e1) / steps


def run_row(args, rank, world):
    """A row recurrence of the hot-path table's next rows (the selective-scan
    rows, the RWKV-4 WKV rows): one library call over its workload per step."""
    import torch
    import torch.distributed as dist
    from chunked_gated_delta_chunk_gb300 import binding as B
    from chunked_gated_delta_chunk_gb300 import build as build_mod
    spec = _RowSpec(args.row)
    p = spec.p
    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build_oracle()
        cols = {"scan": 1024, "wkv": 256, "attn": 512}[args.row]   # sampled channels (rows) per step
        spec.sample(cols)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            spec.oracle_pass(cols)
        el = time.perf_counter() - t0
        # whole-row equivalents (attention: rows of the prefix, a lower bound on the full prompt's cost)
        tps = p.T * args.steps / el * cols / p.C if args.row != "attn" else cols * args.steps / el
        line = {"metric": spec.metric, "value": tps, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "impl": "reference",
                "config": config_dict(spec.workload, p, world),
                "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": oracle.max_threads(),
                                 "kind": "oracle",
                                 "sample": (f"the first {cols} of {p.T} rows, all heads, per step"
                                            if args.row == "attn" else
                                            f"{cols} of {p.C} channels, all {p.T} rows, per step")},
                "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    build_mod.build()
    one = spec.make_call(p, dev)
    set_bytes = spec.nbytes
    nsets = max(1, min(8, -(-2 * l2_bytes(dev) // max(set_bytes, 1)) + 1))
    calls = [one] + [spec.make_call(p, dev) for _ in range(nsets - 1)]
    stream = torch.cuda.current_stream(dev)
    for i in range(args.warmup):
        calls[i % nsets].run(stream)
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    clk = ClockSampler(local)
    blocks = timed_blocks(calls, args.steps, stream, barrier, dev, args.min_seconds, clk)
    ms_total = statistics.median(blocks)
    ms_timer, records, dropped = timed_steps(calls, args.steps, stream, barrier, launches_per_call=2)
    per_kernel = {}
    for name, ms in records:
        tot, n = per_kernel.get(name, (0.0, 0))
        per_kernel[name] = (tot + ms, n + 1)
    ms_total = max_over_ranks(ms_total, dev)
    ms_step = ms_total / args.steps
    dominant = max(per_kernel, key=lambda k: per_kernel[k][0])
    kern_ms = per_kernel[dominant][0] / per_kernel[dominant][1]
    hbm, tflops, peak_kind = load_peaks()
    if getattr(spec, "nflops", None) and spec.nflops / (tflops * 1e12) > spec.nbytes / (hbm * 1e9):
        achieved = spec.nflops / (kern_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tflops, "unit": "TFLOP/s",
                "frac": achieved / tflops, "algorithmic_flops": spec.nflops}
    else:
        achieved = spec.nbytes / (kern_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm}
    roof.update({
            "traffic": recorded_traffic(dominant, spec.workload), "peak_source": peak_kind, "kernel": dominant,
            "algorithmic_bytes": spec.nbytes, "kernel_ms_per_launch": kern_ms,
            "kernels": {k: {"launches_per_step": n / args.steps, "ms_per_launch": tot / n,
                            "share": tot / sum(v[0] for v in per_kernel.values())}
                        for k, (tot, n) in sorted(per_kernel.items())},
            "untimed_launches": dropped,
            "kernel_times_from": ("a second timed region of the same steps with the library's launch timer on "
                                  f"({ms_timer / args.steps:.4f} ms per step with it)")})
    # end to end: the inputs from pinned host memory, the outputs back
    host_in = {n: getattr(one, n).cpu().pin_memory() for n in spec.inputs}
    host_out = {n: torch.empty_like(getattr(one, n), device="cpu").pin_memory() for n in spec.outputs}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    e2e_bufs = calls[:2] if len(calls) >= 2 else [one, spec.make_call(p, dev)]
    e2e_ms = e2e_steps_ms(e2e_bufs, host_in, host_out, max(3, min(args.steps, 20)), barrier, dev)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build_oracle()
        cols = {"scan": 2048, "wkv": 512, "attn": 1024}[args.row]
        spec.sample(cols)
        n, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < 10.0:
            spec.oracle_pass(cols)
            n += 1
        el = time.perf_counter() - t0
        if args.row == "attn":
            cpu = {"value": cols * n / el, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
                   "sample": f"{n} passes over the first {cols} of {p.T} rows, all heads"}
        else:
            cpu = {"value": p.T * n / el * cols / p.C, "unit": "tokens/s", "cores": oracle.max_threads(),
                   "kind": "oracle", "sample": f"{n} passes over {cols} of {p.C} channels, all {p.T} rows"}
    if rank == 0:
        line = {"metric": spec.metric, "value": world * p.T / (ms_step * 1e-3), "unit": "tokens/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if args.row == "attn" else "f32",
                "data": "synthetic",
                "config": config_dict(spec.workload, p, world),
                "l2_rotation": f"{nsets} independent buffer sets ({nsets * set_bytes / 2**20:.0f} MiB > 2 x L2)",
                "timed_blocks": {"blocks": len(blocks), "steps_per_block": args.steps,
                                 "seconds": sum(blocks) / 1e3, "statistic": "median block"},
                "roofline": roof,
                "e2e": {"value": world * p.T / (e2e_ms * 1e-3), "unit": "tokens/s",
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
                "gpu_launches": 2 * args.steps * len(blocks), "clocks": clk.summary(), "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=2, choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefix-tokens", type=int, default=0,
                    help="time only the first N tokens of a single-prompt workload (0: all)")
    ap.add_argument("--min-seconds", type=float, default=2.0,
                    help="repeat the K-step timed block back to back for about this long (clocks sampled throughout)")
    ap.add_argument("--reference-seconds", type=float, default=120.0,
                    help="host seconds the reference arm spends over all its steps (it sizes its sample to them)")
    ap.add_argument("--row", default="gdn", choices=["gdn", "scan", "wkv", "attn"],
                    help="gdn: the chunked gated delta rule prefill (the headline); "
                         "scan: the selective-scan rows; wkv: the RWKV-4 WKV rows; "
                         "attn: the full-attention rows over a KV cache")
    args = ap.parse_args()
    assert args.warmup >= 3 or args.impl == "reference", "at least 3 warm-up steps"

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.row != "gdn":
        run_row(args, rank, world)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import torch.distributed as dist
    from chunked_gated_delta_chunk_gb300 import binding as B
    from chunked_gated_delta_chunk_gb300 import build as build_mod
    from chunked_gated_delta_chunk_gb300 import runner

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    build_mod.build()

    p = make_workload(args.config)
    if args.prefix_tokens:
        # the first N tokens of a single-prompt workload (for captures whose
        # device footprint must stay small)
        assert p.B == 1 and 0 < args.prefix_tokens <= p.T, "--prefix-tokens needs one prompt and 0 < N <= T"
        p = _prefix(p, args.prefix_tokens)
    workload = WORKLOADS[args.config] + (f"; its first {args.prefix_tokens} tokens" if args.prefix_tokens else "")
    one = runner.PrefillCall(p, dev)
    set_bytes = sum(t.numel() * t.element_size() for t in
                    (one.q, one.k, one.v, one.x, one.g, one.beta, one.state_in, one.out,
                     one.state_out, one.workspace) if t is not None)
    nsets = max(1, min(16, -(-2 * l2_bytes(dev) // max(set_bytes, 1)) + 1))
    calls = [one] + [runner.PrefillCall(p, dev) for _ in range(nsets - 1)]
    stream = torch.cuda.current_stream(dev)

    for i in range(args.warmup):
        calls[i % nsets].run(stream)
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    launches_per_call = len(B.gdn_prefill_plan(one.desc))
    # value: blocks of K steps with nothing between the library's launches,
    # repeated for about --min-seconds with the clocks sampled throughout (the
    # median block is the figure); then K more steps with the library
    # bracketing each launch with CUDA events on the launch stream: the
    # per-kernel device times
    clk = ClockSampler(local)
    blocks = timed_blocks(calls, args.steps, stream, barrier, dev, args.min_seconds, clk)
    ms_total = statistics.median(blocks)
    ms_timer, records, dropped = timed_steps(calls, args.steps, stream, barrier,
                                             launches_per_call=launches_per_call)
    per_kernel = {}
    for name, ms in records:
        tot, n = per_kernel.get(name, (0.0, 0))
        per_kernel[name] = (tot + ms, n + 1)
    ms_total = max_over_ranks(ms_total, dev)
    ms_step = ms_total / args.steps
    tokens_per_s = world * p.T / (ms_step * 1e-3)

    # End to end through the C ABI with host buffers: pinned H2D of the step's
    # inputs, the call, D2H of out and state_out, every step (pipelined over
    # two device sets, see e2e_steps_ms).
    host_in = {name: getattr(one, name).cpu().pin_memory() for name in
               ("q", "k", "v", "x", "g", "beta", "state_in") if getattr(one, name) is not None}
    host_out = {name: torch.empty(getattr(one, name).shape, dtype=getattr(one, name).dtype).pin_memory()
                for name in ("out", "state_out")}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    e2e_bufs = calls[:2] if len(calls) >= 2 else [one, runner.PrefillCall(p, dev)]
    e2e_ms = e2e_steps_ms(e2e_bufs, host_in, host_out, max(3, min(args.steps, 50)), barrier, dev)
    e2e_ms = max_over_ranks(e2e_ms, dev)

    hbm, tflops, peak_kind = load_peaks()
    bytes_alg = algorithmic_bytes(p)
    flops_alg = algorithmic_flops(p)
    t_bytes = bytes_alg / (hbm * 1e9)
    t_flops = flops_alg / (tflops * 1e12)
    bound = "hbm" if t_bytes >= t_flops else "tensor"
    # dominant kernel: the most device time in the timed region; its unit of
    # work is one step (all of its launches in a step together read the
    # step's inputs once and write its outputs once, algorithmically)
    dominant = max(per_kernel, key=lambda k: per_kernel[k][0])
    kern_ms = per_kernel[dominant][0] / args.steps
    if bound == "hbm":
        achieved = bytes_alg / (kern_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm}
    else:
        achieved = flops_alg / (kern_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tflops, "unit": "TFLOP/s",
                "frac": achieved / tflops}
    # the whole call against the path roofline (the slower of the algorithmic
    # FLOPs at the bf16 peak and the algorithmic bytes at the HBM peak)
    t_roof = max(t_bytes, t_flops)
    roof["path_frac"] = t_roof / (ms_step * 1e-3)
    roof["path_roofline_ms"] = t_roof * 1e3
    roof["path_achieved"] = (bytes_alg / (ms_step * 1e-3) / 1e9 if bound == "hbm"
                             else flops_alg / (ms_step * 1e-3) / 1e12)
    roof["frac_of"] = ("frac: the dominant kernel's device time per step; path_frac: the whole call's "
                       "time per step (ms_per_step)")
    roof["traffic"] = recorded_traffic(dominant, WORKLOADS[args.config]) if not args.prefix_tokens else None
    roof["kernel_ms_per_step"] = kern_ms
    roof["launches_per_step"] = per_kernel[dominant][1] / args.steps
    roof["kernels"] = {k: {"launches_per_step": n / args.steps, "ms_per_launch": tot / n,
                           "share": tot / sum(v[0] for v in per_kernel.values())}
                       for k, (tot, n) in sorted(per_kernel.items())}
    roof["untimed_launches"] = dropped
    roof["kernel_times_from"] = ("a second timed region of the same steps with the library's launch timer on "
                                 f"({ms_timer / args.steps:.4f} ms per step with it)")
    roof["peak_source"] = peak_kind
    roof["kernel"] = dominant
    roof["algorithmic_bytes"] = bytes_alg
    roof["algorithmic_flops"] = flops_alg

    # the plain entry point (gdn_prefill: bf16, no conv, no workspace, so no
    # chunk records or segment maps) on the same inputs, where it applies
    plain = None
    if p.conv is None:
        B.gdn_prefill(one.q, one.k, one.v, one.g, one.beta, one.state_in, one.state_out, one.out, one.cu,
                      p.B, p.Hk, p.Hv, p.dk, p.dv, 64)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(3, min(args.steps, 50))
        barrier()
        e0.record(stream)
        for i in range(reps):
            c = calls[i % nsets]
            B.gdn_prefill(c.q, c.k, c.v, c.g, c.beta, c.state_in, c.state_out, c.out, c.cu,
                          p.B, p.Hk, p.Hv, p.dk, p.dv, 64)
        e1.record(stream)
        barrier()
        plain = {"ms_per_call": e0.elapsed_time(e1) / reps, "calls": reps,
                 "note": "gdn_prefill has no workspace argument, so it runs the plan that needs none"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, cores, sample = cpu_oracle_tokens_per_s(p)
        tps1, _, sample1 = cpu_oracle_tokens_per_s(p, budget_s=10.0, nthreads=1)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
               "one_thread": {"value": tps1, "unit": "tokens/s", "cores": 1, "sample": sample1}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": config_dict(workload, p, world),
            "l2_rotation": f"{nsets} independent buffer sets ({nsets * set_bytes / 2**20:.0f} MiB > 2 x L2)",
            "timed_blocks": {"blocks": len(blocks), "steps_per_block": args.steps,
                             "seconds": sum(blocks) / 1e3, "statistic": "median block"},
            "roofline": roof,
            "e2e": {"value": world * p.T / (e2e_ms * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_call * args.steps * len(blocks),
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "gdn_prefill_entry": plain,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
