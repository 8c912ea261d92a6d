"""Host-side logic of bench.py on CPU: the cross-rank reduction under a real
2-rank gloo process group, the clock-sample parser, GPU index mapping and the
reference (oracle) arm on a small workload."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, tokens = bench.reduce_across_ranks(10.0 + 5 * rank, 1000 * (rank + 1))
        results[rank] = (ms, tokens, bench.dist_env())
    finally:
        dist.destroy_process_group()


def test_reduce_across_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.start_processes(_rank_main, args=(2, port, results), nprocs=2, join=True, start_method="spawn")
        got = dict(results)
    for rank in (0, 1):
        ms, tokens, env = got[rank]
        assert ms == 15.0 and tokens == 3000  # max of times, sum of tokens
        assert env == (2, rank, rank)


def test_reduce_single_process_is_identity():
    assert not dist.is_initialized()
    assert bench.reduce_across_ranks(3.5, 7) == (3.5, 7)


def test_clock_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler(0)
    c.lines = ["1965, 2070, Not Active, Not Active, Not Active, Active",
               "2070, 2070, Not Active, Not Active, Not Active, Not Active",
               "1500, 2070, Active, Not Active, Not Active, Not Active",
               "garbage line"]
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1965 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert bench.ClockSampler(0).summary()["samples"] == 0


def test_physical_gpu_mapping(monkeypatch):
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3,5")
    assert bench.physical_gpu(1) == 5
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "")
    assert bench.physical_gpu(2) == 2


def test_reference_arm_prints_one_line_on_cpu():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "2",
                          "--steps", "1", "--warmup", "3", "--cpu-seconds", "2"],
                         capture_output=True, text=True, timeout=600, env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["unit"] == bench.UNIT
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"


def test_one_core_oracle_sample():
    """The one-core leg of the CPU baseline: a spawned interpreter pinned to
    one CPU, timing whole oracle steps of the single-stream decode workload."""
    rec = bench.one_core_sample(2, 0.3)
    assert rec is not None and rec["cores"] == 1 and rec["value"] > 0 and rec["steps"] >= 1


def test_prefill_flops_closed_form():
    # causal chunked prefill: chunk c of n queries sees c*n earlier keys plus
    # 1..n of its own; sum over chunks = n^2 * C(C-1)/2 + C * n(n+1)/2 pairs,
    # each 4 * D flops per query head (q.k and p.v)
    n, C, H, D = 2048, 16, 16, 256
    pairs = n * n * C * (C - 1) // 2 + C * n * (n + 1) // 2
    assert bench.prefill_flops(n, C, H, D) == pairs * H * 4 * D
    assert abs(bench.prefill_flops(n, C, H, D) - 8.796e12) < 1e9
    assert bench.prefill_flops(1, 1, 1, 1) == 4.0


@pytest.mark.parametrize("bits,gs,want", [(4, 64, 144), (3, 64, 112), (8, 128, 264), (2, 32, 96), (5, 32, 192)])
def test_row_bytes(bits, gs, want):
    # 256 dims * bits / 8 bytes of codes + a bf16 scale and bias per group
    assert bench.row_bytes(bits, gs) == want
