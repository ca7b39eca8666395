"""The benchmark's multi-rank host logic on CPU with the gloo backend, world size 2:
barriers, the max over ranks of the timed region, the whole-job value, and that
only rank 0 runs and prints the CPU reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.dist_init(world, use_cuda=False)
    bench.barrier(dist)
    # rank r "took" 10 + 5r ms: every rank must see the max
    worst = bench.max_over_ranks(dist, 10.0 + 5.0 * rank)
    bench.barrier(dist)
    q.put((rank, worst))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 15.0), (1, 15.0)]


def test_reference_arm_only_rank0_prints():
    """`bench.py --impl reference` under two ranks: rank 1 exits 0 without work,
    rank 0 prints one JSON line (tiny workload, one short step)."""
    outs = []
    for rank in (1, 0):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                            "--workload", "tiny", "--steps", "1", "--warmup", "0"],
                           capture_output=True, text=True, env=env, timeout=300)
        assert r.returncode == 0, r.stderr
        outs.append(r.stdout.strip())
    assert outs[0] == ""
    line = json.loads(outs[1])
    assert line["impl"] == "reference" and line["unit"] == "routed tokens/s"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
