"""The N > 1 path of bench.py on CPU: two ranks over gloo (no GPU).

bench.py shards nothing across ranks (every rank runs its own batch), so the
multi-rank logic is the rendezvous, the barrier, the max of the step time
over the ranks, the per-rank seed offset, and the reference arm's
"rank 0 alone prints" rule.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, local, w = bench.dist_setup()
    assert (r, local, w) == (rank, rank, world)
    bench.barrier(w)
    worst = bench.max_over_ranks(1.5 * (rank + 1), w)
    bench.barrier(w)
    q.put((rank, worst))
    torch.distributed.destroy_process_group()


def test_two_ranks_rendezvous_barrier_and_max_over_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got == {0: 3.0, 1: 3.0}  # every rank reports the slowest rank's time


def test_rank_seed_offset_gives_each_rank_its_own_batch():
    sys.path.insert(0, ROOT)
    from exact_blocked_attention_gb300 import workloads
    s = workloads.spec("decode_gqa", small=True)
    a = workloads.generate(workloads.replace(s, seed=s.seed + 1000 * 0))
    b = workloads.generate(workloads.replace(s, seed=s.seed + 1000 * 1))
    assert a["q"].shape == b["q"].shape and not torch.equal(a["q"], b["q"])
    assert not torch.equal(a["seqlens"], b["seqlens"])


def test_reference_arm_under_torchrun_prints_once_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-budget-s", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
