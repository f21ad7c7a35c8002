"""The N > 1 host path of bench.py on CPU: two `gloo` ranks.

The path shards by sequence (each rank holds its own batch shard, with its own
checkpoints and buffers) and has no exchange step; the only collective is the
max over ranks of the timed region.  These tests run without a GPU.
"""
import json
import os
import socket
import subprocess
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # the slowest rank's time, on every rank
        got = bench.max_over_ranks(1.5 + rank, world, "cpu")
        # this rank's shard of layer 0: checkpoint and first draft block
        wl = synth.WORKLOADS["b8"]
        init = synth.initial_layer(wl, bench.layer_seed(0, rank))
        blk = synth.draft_block(wl, bench.layer_seed(0, rank), 0)
        np.save(os.path.join(out, f"state{rank}.npy"), init["state"][:1, :1].numpy())
        np.save(os.path.join(out, f"k{rank}.npy"), blk["k"][:1].float().numpy())
        with open(os.path.join(out, f"max{rank}.txt"), "w") as f:
            f.write(repr(got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_and_distinct_shards(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        assert float(open(tmp_path / f"max{r}.txt").read()) == 2.5
    s0, s1 = (np.load(tmp_path / f"state{r}.npy") for r in range(world))
    k0, k1 = (np.load(tmp_path / f"k{r}.npy") for r in range(world))
    assert s0.shape == s1.shape and not np.array_equal(s0, s1)
    assert k0.shape == k1.shape and not np.array_equal(k0, k1)


def test_whole_job_time_per_layer_step():
    import bench
    # two replicas, 10 steps of 24 layers each, in 4.8 ms: 480 layer-steps
    assert bench.per_layer_step_us(4.8, 10, 24, 2) == pytest.approx(10.0)
    assert bench.per_layer_step_us(4.8, 10, 24, 1) == pytest.approx(20.0)
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched as two ranks: rank 0 times the CPU oracle
    and prints the one JSON line, rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "us/layer" and line["value"] > 0
    assert line["n_gpus"] == 2 and line["higher_is_better"] is False
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
