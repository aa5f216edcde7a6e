"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Tolerances: per tensor, max|gpu - oracle| <= tol * max|oracle| with tol = 1e-5
for fp32 workloads and 1e-2 for bf16 workloads (bf16 inputs, fp32 accumulation
and state); every output finite; the new conv state bit-exact.

Workloads follow the five named configurations (``inputs.make_config``) at
full size, plus edge cases: ragged and empty sequences, every chunk size,
every supported head size, GQA, NULL and aliased states, the 64 + 11 two-call
resume of the chunked-prefill pages' tests, and the decode step.
"""

import pytest
import torch

from chunked_gated_delta_chunk_gb300 import build as build_mod
from chunked_gated_delta_chunk_gb300 import inputs, runner
from tests.harness import TOL_BF16, TOL_FP32, assert_all_finite, compare, compare_all_heads, run_oracle, tol_for
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()


@pytest.fixture(autouse=True)
def _no_wait_ran_out():
    """Every bounded wait of the tensor-core kernels (mbarriers, the segment
    passes) must have been met: the device counter of waits that ran out
    stays where it was."""
    from chunked_gated_delta_chunk_gb300 import binding as B
    before = B.gdn_wait_timeouts()
    yield
    assert B.gdn_wait_timeouts() == before


def _gpu(p, **kw):
    return runner.prefill(p, **kw)


# ---------------------------------------------------------------- named workloads
def test_tiny_fp32_64_plus_11():
    """Workload 1: 75 tokens, chunk 64 (one call cuts 64 + 11), fp32, 1e-5."""
    p = inputs.make_config(1)
    res = _gpu(p)
    compare(res, run_oracle(p), TOL_FP32)


def test_tiny_fp32_two_chained_calls():
    """The same 75 tokens as two calls, 64 then 11, the state carried through
    state_out -> state_in on the device, equal the oracle's unsplit run."""
    p = inputs.make_config(1)
    ref = run_oracle(p)
    a = inputs.make_problem(1001, [64], 1, 1, 16, 16, dtype=torch.float32)
    b = inputs.make_problem(1001, [11], 1, 1, 16, 16, dtype=torch.float32)
    a.q, a.k, a.v, a.g, a.beta, a.state_in = p.q[:64], p.k[:64], p.v[:64], p.g[:64], p.beta[:64], p.state_in
    first = runner.PrefillCall(a)
    first.run()
    b.q, b.k, b.v, b.g, b.beta = p.q[64:], p.k[64:], p.v[64:], p.g[64:], p.beta[64:]
    second = runner.PrefillCall(b, state_in=first.state_out)
    second.run()
    torch.cuda.synchronize()
    out = torch.cat([first.out.cpu(), second.out.cpu()])
    compare({"out": out, "state_out": second.state_out.cpu()}, ref, TOL_FP32)


@pytest.mark.parametrize("chunk", [1, 8, 16, 32, 63, 64])
def test_tiny_fp32_every_chunk_size(chunk):
    p = inputs.make_config(1)
    compare(_gpu(p, chunk=chunk), run_oracle(p), TOL_FP32)


def test_prompt4k_full():
    """Workload 2: B=1, H=16, dk=dv=128, T=4096, bf16, zero incoming state."""
    p = inputs.make_config(2)
    compare(_gpu(p), run_oracle(p), TOL_BF16)


def test_ragged_conv_gqa_all_heads():
    """Workload 3: 8 ragged prompts (lengths up to 8192), GQA 16/32, conv K=4,
    nonzero state; every value head against the oracle (run in batches of
    heads), every conv-state channel bit for bit."""
    p = inputs.make_config(3)
    res = _gpu(p)
    compare_all_heads(res, p, TOL_BF16)


def test_stress_finite_and_close():
    """Workload 4: nearly parallel keys, beta ~ sigmoid(6), g down to -20."""
    p = inputs.make_config(4)
    res = _gpu(p)
    assert_all_finite(res)
    compare(res, run_oracle(p), TOL_BF16)


def test_long_65536_all_heads():
    """Workload 5: T=65536, GQA 16/32, conv K=4, incoming state and conv state
    from the oracle's run of a prior 4096-token prompt; every value head over
    all 65536 tokens against the oracle (run in batches of heads)."""
    p = inputs.make_config(5)
    prior = run_oracle(p.prior)
    p.state_in = torch.from_numpy(prior["state_out"]).float()
    p.conv["state_in"] = torch.from_numpy(prior["conv_state_out"]).float()
    res = _gpu(p)
    compare_all_heads(res, p, TOL_BF16)


# ---------------------------------------------------------------- edge cases
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 64), (64, 32), (128, 16), (16, 128), (128, 128)])
def test_head_sizes(dtype, dk, dv):
    p = inputs.make_problem(7, [1, 63, 64, 65, 130], 2, 4, dk, dv, dtype=dtype)
    compare(_gpu(p), run_oracle(p), tol_for(p))


@pytest.mark.parametrize("chunk", [1, 7, 16, 33, 64])
def test_ragged_with_empty_sequences(chunk):
    p = inputs.make_problem(8, [0, 5, 0, 128, 129, 0, 1], 1, 2, 64, 64, chunk=chunk)
    res = _gpu(p)
    compare(res, run_oracle(p), TOL_BF16)
    # empty sequences return their incoming state unchanged
    for n in (0, 2, 5):
        assert torch.equal(res["state_out"][n], p.state_in[n])


def test_null_state_in_and_no_state_out():
    p = inputs.make_problem(9, [100, 30], 2, 2, 128, 128, s0_sd=None)
    res = _gpu(p, write_state=False)
    assert "state_out" not in res
    compare(res, run_oracle(p), TOL_BF16)


def test_state_aliasing_in_place():
    p = inputs.make_problem(10, [77, 200], 1, 3, 128, 128)
    ref = run_oracle(p)
    call = runner.PrefillCall(p, alias_state=True)
    call.run()
    torch.cuda.synchronize()
    compare({k: v.cpu() for k, v in call.results().items()}, ref, TOL_BF16)


@pytest.mark.parametrize("act", [0, 1])
def test_conv_prologue_small(act):
    """Short conv in front, ragged lengths shorter than the conv window."""
    p = inputs.make_problem(11, [1, 2, 3, 70, 0, 130], 2, 4, 32, 64, conv_kernel=4, conv_act=act)
    compare(_gpu(p), run_oracle(p), TOL_BF16)


def test_conv_state_aliasing_fp32():
    p = inputs.make_problem(12, [2, 50], 1, 1, 16, 32, conv_kernel=4, dtype=torch.float32)
    ref = run_oracle(p)
    call = runner.PrefillCall(p, alias_conv_state=True)
    call.run()
    torch.cuda.synchronize()
    compare({k: v.cpu() for k, v in call.results().items()}, ref, TOL_FP32)


def test_no_l2norm_and_q_scale():
    p = inputs.make_problem(13, [90], 2, 2, 64, 64, dtype=torch.float32)
    p.use_l2norm = False
    p.q_scale = 0.125
    compare(_gpu(p), run_oracle(p), TOL_FP32)


def test_plain_entry_point_matches_ex():
    """gdn_prefill (bf16, L2 norm on, no conv, no workspace) gives the same
    bits as gdn_prefill_ex with the same description and no workspace, and
    matches the oracle."""
    from chunked_gated_delta_chunk_gb300 import binding as B
    p = inputs.make_problem(14, [300, 64], 4, 8, 128, 128)
    call = runner.PrefillCall(p, segment_chunks=-1, split_prep=-1)
    assert call.workspace is None
    call.run()
    out2 = torch.empty_like(call.out)
    st2 = torch.empty_like(call.state_out)
    B.gdn_prefill(call.q, call.k, call.v, call.g, call.beta, call.state_in, st2, out2, call.cu,
                  p.B, p.Hk, p.Hv, p.dk, p.dv, 64)
    torch.cuda.synchronize()
    assert torch.equal(out2, call.out) and torch.equal(st2, call.state_out)
    compare({"out": out2.cpu(), "state_out": st2.cpu()}, run_oracle(p), TOL_BF16)


def test_two_calls_resume_with_conv():
    """64 + 11 with a short conv: the conv state and the recurrent state
    carried between two calls equal one call (the pages' split-prompt test)."""
    p = inputs.make_problem(15, [75], 2, 2, 64, 64, conv_kernel=4)
    ref = run_oracle(p)
    a = inputs.make_problem(15, [64], 2, 2, 64, 64, conv_kernel=4)
    b = inputs.make_problem(15, [11], 2, 2, 64, 64, conv_kernel=4)
    for part, sl in ((a, slice(0, 64)), (b, slice(64, 75))):
        part.conv["x"] = p.conv["x"][sl]
        part.conv["w"] = p.conv["w"]
        part.g, part.beta = p.g[sl], p.beta[sl]
    a.state_in, a.conv["state_in"] = p.state_in, p.conv["state_in"]
    first = runner.PrefillCall(a)
    first.run()
    second = runner.PrefillCall(b, state_in=first.state_out, conv_state_in=first.cs_out)
    second.run()
    torch.cuda.synchronize()
    res = {"out": torch.cat([first.out.cpu(), second.out.cpu()]),
           "state_out": second.state_out.cpu(), "conv_state_out": second.cs_out.cpu()}
    compare(res, ref, TOL_BF16)


# ---------------------------------------------------------------- decode step
@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 128, 128), (torch.float32, 16, 32),
                                         (torch.bfloat16, 64, 16)])
def test_decode_step_matches_oracle(dtype, dk, dv):
    p = inputs.make_problem(16, [1, 1, 1, 1], 2, 4, dk, dv, dtype=dtype)
    out, st = runner.step(p.q, p.k, p.v, p.g, p.beta, p.state_in, p.Hk, p.Hv, dk, dv, dtype=dtype)
    ref = oracle.oracle_step(p.q, p.k, p.v, p.g, p.beta, p.state_in, p.Hk, p.Hv, dk, dv)
    compare({"out": out.cpu(), "state_out": st.cpu()}, dict(ref, heads=None), tol_for(p))


def test_decode_step_with_conv_in_place():
    p = inputs.make_problem(17, [1, 1, 1], 2, 4, 64, 64, conv_kernel=4)
    conv = dict(p.conv)
    ref = oracle.oracle_step(None, None, None, p.g, p.beta, p.state_in, p.Hk, p.Hv, 64, 64,
                             conv=dict(conv))
    out, st, cs = runner.step(None, None, None, p.g, p.beta, p.state_in, p.Hk, p.Hv, 64, 64,
                              conv=conv)
    compare({"out": out.cpu(), "state_out": st.cpu(), "conv_state_out": cs.cpu()},
            dict(ref, heads=None), TOL_BF16)


def test_prefill_then_decode_equals_token_loop():
    """The pages' test shape: prefill 7 + 4 tokens in two calls, then one
    decode step, against the token-by-token oracle over all 12 tokens."""
    full = inputs.make_problem(18, [12], 1, 2, 128, 128)
    ref = run_oracle(full)
    parts = []
    for sl in (slice(0, 7), slice(7, 11)):
        q = inputs.make_problem(18, [sl.stop - sl.start], 1, 2, 128, 128)
        q.q, q.k, q.v, q.g, q.beta = (t[sl] for t in (full.q, full.k, full.v, full.g, full.beta))
        parts.append(q)
    parts[0].state_in = full.state_in
    c1 = runner.PrefillCall(parts[0])
    c1.run()
    c2 = runner.PrefillCall(parts[1], state_in=c1.state_out)
    c2.run()
    out, st = runner.step(full.q[11:], full.k[11:], full.v[11:], full.g[11:], full.beta[11:],
                          c2.state_out, 1, 2, 128, 128)
    res = {"out": torch.cat([c1.out.cpu(), c2.out.cpu(), out.cpu()]), "state_out": st.cpu()}
    compare(res, ref, TOL_BF16)


# ---------------------------------------------------------------- segment scan
@pytest.mark.parametrize("seg,lengths,chunk", [
    (1, [300], 64), (2, [640], 64), (3, [64 * 7 + 5], 64), (4, [1, 200, 0, 900], 64),
    (2, [333, 64 * 6], 32), (5, [4096], 64), (4, [64 * 7], 64), (1, [64 * 70 + 3], 64)])
def test_segment_scan_matches_oracle(seg, lengths, chunk):
    """The segment-parallel scan (every later segment from a zero state and
    from the identity with V = 0, outputs and maps of both, then the
    segments' incoming states and O = O' + G S_s) equals the token loop;
    segments end on full and partial chunks.  71 segments of one chunk pass
    the 64 segments seg_out_kernel's group table covers (uniform groups)."""
    p = inputs.make_problem(40 + seg, lengths, 2, 4, 128, 128, chunk=chunk)
    call = runner.PrefillCall(p, segment_chunks=seg)
    from chunked_gated_delta_chunk_gb300 import binding as B
    plan = B.gdn_prefill_plan(call.desc)
    assert plan[-2:] == ["chunk_state_kernel", "seg_out_kernel"] and plan.count("chunk_state_kernel") == 1, plan
    call.run()
    torch.cuda.synchronize()
    compare({k: v.cpu() for k, v in call.results().items()}, run_oracle(p), TOL_BF16)


def test_segment_scan_long_groups_and_no_state_out():
    """32 value heads leave seg_out_kernel one chunk group per segment, so a
    CTA walks ten chunks through both tile buffers and refills them; a null
    state_out skips the final-state CTA without touching the outputs."""
    p = inputs.make_problem(53, [64 * 40 + 17, 64 * 9], 16, 32, 128, 128)
    ref = run_oracle(p)
    call = runner.PrefillCall(p, segment_chunks=10)
    call.run()
    torch.cuda.synchronize()
    compare({k: v.cpu() for k, v in call.results().items()}, ref, TOL_BF16)
    p.state_in = None
    ref = run_oracle(p)
    nostate = runner.PrefillCall(p, segment_chunks=10, write_state=False)
    nostate.run()
    torch.cuda.synchronize()
    compare({"out": nostate.out.cpu()}, {"out": ref["out"]}, TOL_BF16)


def test_segment_scan_final_state_after_outputs_of_one_later_segment():
    """96 (sequence, head) units leave no room for final-state CTAs of their
    own, so the single output CTA of each two-segment sequence forms the final
    state after its outputs, from the images it loaded at its start (no state
    step before its outputs)."""
    p = inputs.make_problem(54, [64 * 8, 64 * 7 + 3, 50], 16, 32, 128, 128)
    ref = run_oracle(p)
    call = runner.PrefillCall(p, segment_chunks=4)
    call.run()
    torch.cuda.synchronize()
    compare({k: v.cpu() for k, v in call.results().items()}, ref, TOL_BF16)


def test_segment_scan_with_conv_and_gqa():
    p = inputs.make_problem(50, [700, 90], 2, 4, 128, 128, conv_kernel=4)
    call = runner.PrefillCall(p, segment_chunks=3)
    call.run()
    torch.cuda.synchronize()
    compare({k: v.cpu() for k, v in call.results().items()}, run_oracle(p), TOL_BF16)


def test_segment_scan_off_equals_on_bits_of_segment_zero():
    """Segment 0 runs the same pass with or without the scan, so its output
    rows are bit-identical."""
    p = inputs.make_problem(51, [1000], 1, 2, 128, 128)
    a = runner.PrefillCall(p, segment_chunks=-1)
    b = runner.PrefillCall(p, segment_chunks=4)
    a.run()
    b.run()
    torch.cuda.synchronize()
    assert torch.equal(a.out[:256], b.out[:256])


# ---------------------------------------------------------------- split preparation
@pytest.mark.parametrize("seg,lengths,chunk", [
    (-1, [300], 64), (-1, [1, 64, 0, 129, 7], 64), (3, [64 * 7 + 5], 64),
    (4, [1, 200, 0, 900], 64), (2, [333, 64 * 6], 32), (-1, [250, 3], 17)])
def test_split_preparation_matches_inline_and_oracle(seg, lengths, chunk):
    """Chunk records solved ahead of the state pass (all chunks in parallel,
    then chunk_state_kernel) and the preparation inside the one-kernel pass
    agree with each other and with the token loop.  Ragged ends, empty
    sequences, chunks below 64 rows and the segment scan's map passes all read
    records."""
    from chunked_gated_delta_chunk_gb300 import binding as B
    p = inputs.make_problem(60 + seg + len(lengths), lengths, 2, 4, 128, 128, chunk=chunk)
    inline = runner.PrefillCall(p, segment_chunks=seg, split_prep=-1)
    split = runner.PrefillCall(p, segment_chunks=seg)
    assert "chunk_prep_kernel" not in B.gdn_prefill_plan(inline.desc)
    plan = B.gdn_prefill_plan(split.desc)
    assert plan[0] == "chunk_prep_kernel" and plan[1] == "chunk_state_kernel", plan
    inline.run()
    split.run()
    torch.cuda.synchronize()
    ref = run_oracle(p)
    compare({k: v.cpu() for k, v in split.results().items()}, ref, TOL_BF16)
    compare({k: v.cpu() for k, v in inline.results().items()}, ref, TOL_BF16)
    compare({"out": split.out.cpu(), "state_out": split.state_out.cpu()},
            {"out": inline.out.cpu(), "state_out": inline.state_out.cpu()}, TOL_BF16)


def test_split_preparation_with_conv_gqa_and_aliased_state():
    p = inputs.make_problem(70, [700, 90, 0, 33], 2, 8, 128, 128, conv_kernel=4)
    call = runner.PrefillCall(p, segment_chunks=3, alias_state=True, alias_conv_state=True)
    from chunked_gated_delta_chunk_gb300 import binding as B
    assert "chunk_prep_kernel" in B.gdn_prefill_plan(call.desc)
    ref = run_oracle(p)
    call.run()
    torch.cuda.synchronize()
    compare({k: v.cpu() for k, v in call.results().items()}, ref, TOL_BF16)


# ---------------------------------------------------------------- launch timer
def test_launch_timer_records_every_planned_launch():
    """With the launch timer on, one call records exactly the kernels its
    launch plan lists, in order, each with a positive device time; launches
    past the capacity are counted as dropped."""
    from chunked_gated_delta_chunk_gb300 import binding as B
    p = inputs.make_problem(52, [900, 40], 2, 4, 128, 128, conv_kernel=4)
    call = runner.PrefillCall(p, segment_chunks=4)
    plan = B.gdn_prefill_plan(call.desc)
    B.gdn_launch_timer_start(len(plan) + 1)
    try:
        call.run()
        call.run()
    finally:
        B.gdn_launch_timer_stop()
    records, dropped = B.gdn_launch_timer_read()
    assert [n for n, _ in records] == (plan + plan)[:len(plan) + 1]
    assert dropped == len(plan) - 1
    assert all(ms > 0 for _, ms in records)
    torch.cuda.synchronize()
    compare({k: v.cpu() for k, v in call.results().items()}, run_oracle(p), TOL_BF16)


@pytest.mark.parametrize("conv_kernel,s0_sd,alias", [(4, 0.05, False), (0, None, False), (4, 0.05, True)])
def test_batch_without_tokens_returns_states(conv_kernel, s0_sd, alias):
    """Every sequence empty (T_total == 0) on the tensor-core shape: the token
    tensors have no storage, no kernel runs, and every sequence's states come
    back unchanged (zeros without an incoming state; in place when aliased)."""
    p = inputs.make_problem(61, [0, 0, 0], 2, 4, 128, 128, conv_kernel=conv_kernel, s0_sd=s0_sd)
    call = runner.PrefillCall(p, alias_state=alias, alias_conv_state=alias and conv_kernel > 0)
    from chunked_gated_delta_chunk_gb300 import binding as B
    assert B.gdn_prefill_plan(call.desc) == []
    call.run()
    torch.cuda.synchronize()
    res = {k: v.cpu() for k, v in call.results().items()}
    assert res["out"].numel() == 0
    want = p.state_in if p.state_in is not None else torch.zeros(3, 4, 128, 128)
    assert torch.equal(res["state_out"], want)
    if conv_kernel:
        assert torch.equal(res["conv_state_out"], p.conv["state_in"])


@pytest.mark.parametrize("lengths", [
    [130, 130, 64, 130, 0, 1, 64],                                       # equal lengths: ties by index
    [int(x) for x in torch.randint(0, 100, (80,), generator=torch.Generator().manual_seed(62))],  # > 64 sequences
])
def test_many_sequences_longest_first_and_ties(lengths):
    """The chain kernels take sequences longest first (ties by index, the
    identity past 64 sequences); every sequence's rows and state still match
    the oracle, with the records and without them."""
    p = inputs.make_problem(63, lengths, 2, 4, 128, 128)
    ref = run_oracle(p)
    for split in (0, -1):
        call = runner.PrefillCall(p, split_prep=split, segment_chunks=-1)
        call.run()
        torch.cuda.synchronize()
        compare({k: v.cpu() for k, v in call.results().items()}, ref, TOL_BF16)
