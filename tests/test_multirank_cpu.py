"""Multi-rank host logic of bench.py on CPU: world size 2 over gloo (replicas,
no collective on the data path; only the barrier and the max over ranks of
the timed region), and the reference arm's JSON line."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.init_dist(world, rank, "gloo")
    bench.barrier(d)
    got = bench.max_over_ranks(d, 10.0 * (rank + 1), "cpu")
    bench.barrier(d)
    out.put((rank, got, bench.dist_env()))
    dist.destroy_process_group()


def test_two_rank_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, env in res:
        assert got == 20.0
        assert env == (2, rank, rank)


@pytest.mark.parametrize("rank", ["0", "1"])
def test_reference_arm_line(rank):
    env = dict(os.environ, RANK=rank, WORLD_SIZE="2" if rank == "1" else "1", LOCAL_RANK=rank,
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_bf16", "--steps", "1", "--warmup", "0",
                        "--ref-budget", "1"], capture_output=True, text=True, env=env,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    if rank == "1":  # only rank 0 runs and prints the reference arm
        assert r.stdout.strip() == ""
        return
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["workload"] == "tiny_bf16"
