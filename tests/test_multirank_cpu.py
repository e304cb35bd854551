"""The benchmark's multi-rank path on CPU: two gloo ranks, no GPU.

Under torchrun every rank runs an independent replica; the ranks only meet in
a barrier around the timed region and in a max-reduction of the elapsed times.
These tests run that host logic with world size 2 over gloo, and the reference
arm (rank 0 times the oracle, the other ranks exit without work).
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "BENCH_BACKEND": "gloo"})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    out[rank] = bench.allreduce_max(values[rank], w, "cpu")
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_rank_barrier_and_max_of_times():
    world, port = 2, _free_port()
    values = [3.25, 7.5]
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, values, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        assert dict(out) == {0: 7.5, 1: 7.5}


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    env_keys = ("RANK", "WORLD_SIZE", "LOCAL_RANK")
    saved = {k: os.environ.pop(k) for k in env_keys if k in os.environ}
    try:
        assert bench.dist_setup() == (1, 0, 0)
        assert bench.allreduce_max(2.5, 1, "cpu") == 2.5
    finally:
        os.environ.update(saved)


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    env = dict(os.environ, BENCH_BACKEND="gloo", CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "n64_d32_c32", "--steps", "1", "--warmup", "3", "--cpu-rows", "8", "--cpu-cols", "8"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout  # rank 0 alone prints
    line = lines[0]
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
