"""Multi-process plumbing of bench.py on CPU (gloo, world size 2): the decode path
shards by sequence with no data-path exchange, so N GPUs run N replicas; the only
collectives are a barrier and the max over ranks of the step time."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    ws, r, local = bench.dist_init(world)
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    m = bench.max_over_ranks(1.5 + rank, ws)
    q.put((rank, m))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_replica_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get() for _ in range(2))
    assert res == {0: 2.5, 1: 2.5}


def test_reference_arm_prints_one_line_on_tiny_workload():
    env = dict(os.environ, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "0", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "queries/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_subset_generation_matches_full_draw():
    from sparse_attention_decode_kpool_gb300 import workloads as W

    g = W.Geometry(index_kpool=4, index_heads=4, index_head_dim=64, index_topk=64, heads=2,
                   hidden=64)
    full = W.make_workload("a", 5, g, [300, 200, 100], invalid_per_seq=5)
    part = W.make_workload("a", 5, g, [300, 200, 100], invalid_per_seq=5, sequences=[1])
    assert torch.equal(full.k_raw[1], part.k_raw[1]) and torch.equal(full.ckv[1], part.ckv[1])
    assert torch.equal(full.valid[1], part.valid[1])
    assert not part.k_raw[0].any()
    again = W.make_workload("a", 5, g, [300, 200, 100], invalid_per_seq=5)
    assert torch.equal(full.ckv, again.ckv) and torch.equal(full.qidx, again.qidx)
