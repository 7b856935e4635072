"""bench.py's multi-rank host logic on CPU: two gloo ranks (world size 2).

Under torchrun every rank runs its own replica of the workload; the timed
region is bracketed by barriers and the time reported is the maximum over
the ranks.  These tests run bench.py's own helpers (dist_setup, barrier,
max_over_ranks) in two processes with the gloo backend, and check that the
reference arm does its work on rank 0 only.
"""
import argparse
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import torch.distributed as dist

    import bench
    r, world, local = bench.dist_setup(2)
    bench.barrier(world)
    slowest = bench.max_over_ranks(1.0 + 3.0 * r, world)     # rank 1 is the slower one: 4.0
    bench.barrier(world)
    out[r] = (r, world, local, slowest, dist.get_backend())
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    assert res[0] == (0, 2, 0, 4.0, "gloo")
    assert res[1] == (1, 2, 1, 4.0, "gloo")


def test_single_rank_needs_no_process_group(monkeypatch):
    import torch.distributed as dist

    import bench
    for key in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(key, raising=False)
    assert bench.dist_setup(1) == (0, 1, 0)
    assert not dist.is_initialized()
    assert bench.max_over_ranks(2.5, 1) == 2.5
    bench.barrier(1)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import bench
    args = argparse.Namespace(workload=bench.WORKLOAD, steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args, rank=1, world=2) is None
    assert capsys.readouterr().out == ""


@pytest.mark.parametrize("rank", [0, 1])
def test_replicas_draw_different_inputs(rank):
    """Each rank seeds its replica with its rank, so the ranks do not time identical data."""
    import torch

    from chunkwise_gated_delta_gb300.inputs import custom, make_inputs
    w = custom("kda", 1, 64, 1, 64, 64, dtype=torch.float32, h0=False)
    mine, other = make_inputs(w, seed=rank), make_inputs(w, seed=1 - rank)
    assert not torch.equal(mine["q"], other["q"])


def test_gpus_two_entry_launches_two_ranks():
    """`bench.py --gpus 2` with no rank environment starts two ranks itself (gloo on CPU) and
    rank 0 prints one line with n_gpus = 2 (the reference arm, on the small fp32 workload)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--impl", "reference",
                        "--workload", "kda_fp32_b1t256h1d64", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, env=env, timeout=300, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["impl"] == "reference"


def test_gpus_mismatch_with_world_size_fails_loudly():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--impl", "reference",
                        "--workload", "kda_fp32_b1t256h1d64", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=300, cwd=root)
    assert r.returncode != 0 and "WORLD_SIZE" in r.stderr
