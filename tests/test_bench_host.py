"""bench.py host logic on the CPU: work accounting, workload parsing, and the
multi-rank path (one replica per rank, max-over-ranks time) with gloo ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_flops_and_bytes_of_the_default_workload():
    w = bench.parse_workload("rmsnorm_gemm_f16_512x4096x4096")
    M = N = K = 4096
    M = 512
    assert bench.flops_per_step(w) == 2.0 * M * N * K + 3 * M * K + M * N
    assert bench.bytes_per_step(w) == 2 * (M * K + N * K + M * N) + 2 * K


def test_flops_of_patterns_and_ffn():
    w = bench.parse_workload("pattern:gemm_bias_gelu:bf16:8:16:32")
    assert bench.flops_per_step(w) == 2.0 * 8 * 16 * 32 + 8 * 16 * (1 + 8)
    assert bench.bytes_per_step(w) == 2 * (8 * 32 + 16 * 32 + 8 * 16) + 2 * 16
    r = bench.parse_workload("pattern:gemm_bias_residual:f16:8:16:32")
    assert bench.bytes_per_step(r) == 2 * (8 * 32 + 16 * 32 + 8 * 16) + 2 * 16 + 2 * 8 * 16
    f = bench.parse_workload("swiglu_ffn_bf16_4096x4096x11008")
    assert bench.flops_per_step(f) >= 6.0 * 4096 * 4096 * 11008
    with pytest.raises(SystemExit):
        bench.parse_workload("nonsense:1")


def test_roofline_bound_follows_arithmetic_intensity():
    peaks = {"bf16_tflops": 1955.0, "hbm_gbs": 6684.0}
    d = bench.parse_workload("norm:rms:f16:1:4096:4096")  # decode: ~1 flop per byte
    r = bench.roofline_of(bench.flops_per_step(d), bench.bytes_per_step(d), 0.010, peaks, "measured", None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - bench.bytes_per_step(d) / 10e-6 / 1e9) < 1e-6 and abs(r["frac"] - r["hbm_frac"]) < 1e-12
    h = bench.parse_workload("rmsnorm_gemm_f16_512x4096x4096")  # ~400 flop per byte
    r = bench.roofline_of(bench.flops_per_step(h), bench.bytes_per_step(h), 0.019, peaks, "measured", 123)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["traffic"] == 123
    assert abs(r["frac"] - r["tensor_frac"]) < 1e-12 and r["hbm_frac"] < r["tensor_frac"]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        m = bench.max_over_ranks(10.0 * (rank + 1), world)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(repr(m))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        assert float((tmp_path / f"r{r}.txt").read_text()) == 20.0


def test_reference_arm_under_torchrun_prints_once():
    """Two ranks of the reference arm: rank 0 times the oracle and prints one line, rank 1 exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "4", "--warmup", "3",
           "--workload", "pattern:gemm_bias:f16:16:64:64"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
