"""The benchmark's multi-rank host logic on CPU with two gloo ranks: each
rank gets its own batch (weak scaling over rows), timings reduce by max and
work by sum, and the reference leg runs on rank 0 only."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    from pgd_inputs import WORKLOADS, draw_layout
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    cpu = torch.device("cpu")
    wl = WORKLOADS["qwen_serve"]
    seed = bench.rank_seed(wl, rank)
    ctx = draw_layout(wl, seed).contexts
    elapsed = 1.0 + rank                        # rank 1 is the slower one
    t_max = bench.max_over_ranks(elapsed, world, cpu)
    rows = bench.sum_over_ranks(wl.rows, world, cpu)
    bench.barrier(world)
    gathered = [torch.zeros(len(ctx), dtype=torch.int64) for _ in range(world)]
    dist.all_gather(gathered, torch.from_numpy(ctx))
    np.save(os.path.join(out_dir, f"rank{rank}.npy"),
            np.array([t_max, rows, int(not torch.equal(gathered[0], gathered[1]))]))
    dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for rank in range(2):
        t_max, rows, distinct = np.load(tmp_path / f"rank{rank}.npy")
        assert t_max == 2.0          # max over ranks
        assert rows == 2 * 64        # whole-job work = sum over ranks
        assert distinct == 1         # each rank has its own batch


def test_reference_leg_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    from pgd_inputs import WORKLOADS
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, reference_rows = 1, 3, 2
    bench.run_reference(Args, WORKLOADS["qwen_small"])
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_json_line_on_cpu():
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    run = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "qwen_small", "--steps", "2", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert run.returncode == 0, run.stderr[-2000:]
    lines = [x for x in run.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["unit"] == "GB/s"
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
