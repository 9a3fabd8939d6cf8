"""The bench's multi-rank plumbing on CPU (gloo, world size 2, 127.0.0.1): rendezvous, the max over
ranks of the step time, the barrier, and the reference arm under torchrun (rank 0 alone prints one
line). No GPU is used: the replicas-only design has no data-path collective."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, _ = bench.dist_setup()
    slowest = bench.max_over_ranks(10.0 + 5.0 * r, w)   # rank r "took" 10 + 5r ms
    bench.barrier(w)
    queue.put((r, w, dist.get_backend(), slowest))
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = [queue.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(r for r, _, _, _ in results) == [0, 1]
    for _, world, backend, slowest in results:
        assert world == 2 and backend == "gloo" and slowest == 15.0


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--steps", "1", "--warmup", "0", "--ref-units", "2"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [line for line in r.stdout.splitlines() if line.startswith("{")]
    assert len(lines) == 1, r.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["steps"] == 1
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["cpu_baseline"]["kind"] == "oracle"
