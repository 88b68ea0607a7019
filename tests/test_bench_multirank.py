"""Multi-rank plumbing of bench.py on CPU: two gloo ranks on 127.0.0.1.

The decode path shards by query rows with no exchange (every rank runs its own replica on its
own batch), so the only cross-rank steps are the barriers around the timed region and the
max over ranks of the elapsed time; these run here with the gloo backend. The reference arm
runs on rank 0 alone and the other ranks return without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["BENCH_ROOT"])
import bench

world, rank, local = bench.dist_env()
bench.init_dist(world, "gloo")
bench.barrier(world)
# rank r pretends to have taken 1 + r seconds; the job time is the slowest rank's
t = bench.max_over_ranks(1.0 + rank, world, "cpu")
rate = bench.job_throughput(32, world, t)
bench.barrier(world)


class Args:
    steps = 1
    warmup = 3
    ref_rows = 1


ref = bench.run_reference(Args()) if rank != 0 else "skipped"
print(json.dumps({"rank": rank, "world": world, "local": local, "t": t, "rate": rate,
                  "ref_is_none": ref is None}), flush=True)
import torch.distributed as dist
dist.destroy_process_group()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.timeout(300)
def test_two_gloo_ranks_take_the_slowest_rank_time():
    world = 2
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), BENCH_ROOT=ROOT,
                   CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=240)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    outs.sort(key=lambda d: d["rank"])
    for r, d in enumerate(outs):
        assert d["rank"] == r and d["world"] == world and d["local"] == r
        assert d["t"] == 2.0  # max of 1.0 and 2.0 on every rank
        assert d["rate"] == pytest.approx(32 * world / 2.0)
    assert outs[1]["ref_is_none"] is True


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_throughput(10, 1, 2.0) == 5.0
    bench.barrier(1)


def test_code_hash_ignores_comments_only():
    sys.path.insert(0, ROOT)
    import bench
    a = "int x = 1;  // one\n\n// note\nint y = 2;\n"
    b = "int x = 1;\nint y = 2;  // two\n"
    c = "int x = 1;\nint y = 3;\n"
    d = 'const char* s = "a // b";\n'
    assert bench.code_hash(a) == bench.code_hash(b)
    assert bench.code_hash(a) != bench.code_hash(c)
    assert bench.code_hash(d) != bench.code_hash('const char* s = "a\n')
