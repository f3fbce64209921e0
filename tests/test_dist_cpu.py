"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

The decode path shards by replica (each rank decodes its own batch; no
data-path collective), so what needs covering off the GPU is the host side:
rendezvous from the torchrun environment, the barrier around the timed
region, the max-over-ranks reduction of step times, and that only rank 0
prints the JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, lr = bench.dist_setup(world)
    assert (w, r, lr) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank reports a different step time; every rank must see the max
    m = bench.max_over_ranks(1.0 + 2.5 * rank, w)
    bench.barrier(w)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"max": m}, f)
    dist.destroy_process_group()


def test_dist_helpers_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        with open(tmp_path / f"r{r}.json") as f:
            assert json.load(f)["max"] == pytest.approx(3.5)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: os.environ.pop(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK") if k in os.environ}
    try:
        assert bench.dist_setup(1) == (1, 0, 0)
        assert bench.max_over_ranks(4.25, 1) == 4.25
        bench.barrier(1)
    finally:
        os.environ.update(env)


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched as two ranks: rank 0 alone runs the
    oracle and prints one JSON line; the other rank exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--config", "1", "--steps", "2", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["n_gpus"] == 2 and rec["steps"] == 2 and rec["warmup"] == 3
    assert rec["value"] > 0 and rec["e2e"]["h2d_bytes_per_step"] == 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
