"""The N > 1 host logic of bench.py on CPU: ranks as gloo processes (world
size 2) agree on the slowest rank's time and the whole-job rate, and the
reference arm runs and prints on rank 0 only.  (The library itself is
single-GPU: N GPUs run N independent replicas, with no collective on the
data path.)"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch as t
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
        got = bench.max_over_ranks(t, local_ms, t.device("cpu"), world)
        rate = bench.whole_job_rate(world, 1000, 4, got)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"max_ms": got, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def test_ranks_agree_on_slowest_time_and_whole_job_rate(tmp_path):
    world = 2
    port = _free_port()
    torch.multiprocessing.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                                          join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["max_ms"] == 15.0
        # 2 ranks x 1,000 elements x 4 steps in 15 ms
        assert r["rate"] == pytest.approx(2 * 1000 * 4 / 15e-3 / 1e9)


def test_one_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(torch, 12.5, torch.device("cpu"), 1) == 12.5
    assert bench.whole_job_rate(1, 2 ** 24, 20, 2.78) == pytest.approx(2 ** 24 * 20 / 2.78e-3 / 1e9)


def _reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus",
                           str(world), "--workload", "sum", "--steps", "1", "--warmup", "3"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_on_rank_zero_only():
    other = _reference(1, 2)
    assert other.returncode == 0, other.stderr
    assert other.stdout.strip() == ""
    zero = _reference(0, 2)
    assert zero.returncode == 0, zero.stderr
    lines = [ln for ln in zero.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
