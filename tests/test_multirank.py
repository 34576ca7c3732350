"""Host-side multi-rank logic of bench.py on CPU with gloo, world size 2: the
barrier, the max-over-ranks timing and the whole-job (weak-scaling) value."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    w, r, local, pg = bench.dist_setup(world)
    assert (w, r) == (world, rank) and pg is not None
    bench.barrier(pg)
    # rank-dependent "elapsed" times: every rank must see the maximum
    m = bench.max_over_ranks(pg, 1.0 + rank)
    out[rank] = m
    pg.destroy_process_group()


def test_two_ranks_gloo_max_over_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    assert dict(out) == {0: 2.0, 1: 2.0}


def test_whole_job_value_is_weak_scaling_sum():
    import bench
    flops_step, steps, elapsed = 7e11, 10, 0.05
    one = bench.whole_job_value(flops_step, steps, 1, elapsed)
    two = bench.whole_job_value(flops_step, steps, 2, elapsed)
    assert abs(two - 2 * one) < 1e-9
    assert abs(one - flops_step * steps / elapsed / 1e12) < 1e-9


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """`bench.py --impl reference` launched as the two-rank job the contract
    describes: rank 0 alone times the oracle and prints one JSON line, the
    other rank exits 0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    res = subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
