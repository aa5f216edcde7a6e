"""Host side of bench.py's multi-process launch, on CPU: the max-over-ranks
reduction with two gloo ranks, and the reference arm under torchrun with two
ranks (rank 0 alone runs the oracle and prints one JSON line; the other rank
exits without work)."""

import importlib.util
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    return bench


def _rank_max(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _load_bench()
        got = bench.max_over_ranks(1.5 + rank, torch.device("cpu"))
        with open(os.path.join(out_dir, f"rank{rank}"), "w") as f:
            f.write(repr(got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks(tmp_path):
    mp.start_processes(_rank_max, args=(2, _free_port(), str(tmp_path)), nprocs=2, start_method="spawn")
    assert [float((tmp_path / f"rank{r}").read_text()) for r in range(2)] == [2.5, 2.5]


def test_max_over_ranks_without_a_process_group():
    import torch
    assert _load_bench().max_over_ranks(3.25, torch.device("cpu")) == 3.25


def test_reference_arm_under_torchrun_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "2", "--steps", "2", "--warmup", "1",
           "--reference-seconds", "2"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_kernel_hash_ignores_comments_not_code():
    """The recorded DRAM counters stay valid across comment edits of a
    kernel's sources and lapse on any code change."""
    bench = _load_bench()
    base = 'int a = 1; // one\n/* block\n comment */ const char* s = "x // y";\n'
    assert bench._code_only(base) == bench._code_only(base.replace("// one", "// changed"))
    assert bench._code_only(base) == bench._code_only(base.replace("/* block\n comment */", ""))
    assert bench._code_only(base) != bench._code_only(base.replace("a = 1", "a = 2"))
    assert bench._code_only(base) != bench._code_only(base.replace('"x // y"', '"x // z"'))



def test_roofline_numerators_of_prompt4k():
    """The path roofline's numerators for the 4096-token prompt (B=1, 16 heads,
    dk=dv=128, bf16): q, k, v, out in bf16, g and beta in fp32, the fp32 state
    in and out, cu_seqlens; and the FLOPs of full 64-row tiles."""
    bench = _load_bench()
    from chunked_gated_delta_chunk_gb300 import inputs
    p = inputs.make_config(2)
    T, H, d = 4096, 16, 128
    want_bytes = T * 4 * H * d * 2 + T * H * 8 + 2 * H * d * d * 4 + 2 * 4
    assert bench.algorithmic_bytes(p) == want_bytes == 69730312
    want_flops = T * (H * 4 * 64 * d + H * (6 * d * d + 4 * 64 * d))
    assert bench.algorithmic_flops(p) == want_flops == 10737418240
