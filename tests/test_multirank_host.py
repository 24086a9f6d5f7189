"""Host logic of the N>1 benchmark path on CPU: two gloo ranks, each with its own
independent batch (weak scaling, no collective on the data path); the timing
reduction takes the maximum over ranks and the throughput sums the ranks'
sequences.  Also the reference arm: rank 0 alone prints, other ranks exit."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, _ = bench._dist()
    assert (ws, r) == (world, rank)
    hist, cont = bench.rs_inputs(rank, B=4, V=1000, n=64, K=3)
    bench._barrier(ws)
    ms = bench._max_over_ranks(1.0 + rank, ws, "cpu")      # slowest rank's step time
    seqs = bench._sum_over_ranks(4.0, ws, "cpu")           # every rank's sequences
    q.put((rank, ms, seqs, hist[0, :16].tolist()))
    dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, ms0, s0, h0), (_, ms1, s1, h1) = out
    assert ms0 == ms1 == 2.0
    assert s0 == s1 == 8.0
    assert h0 != h1  # each rank draws its own batch


def test_reference_arm_rank_layout():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "4",
                        "--warmup", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["steps"] == 4 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert np.isclose(line["e2e"]["value"], line["value"])
