"""The N > 1 bench path on CPU: two gloo ranks (no GPU).

* `combine_ranks`, the reduction every multi-GPU bench line goes through: each rank gets the
  longest timed region and the sum of the units, whatever the ranks' own values.
* The reference arm under torchrun with two ranks: rank 0 alone runs the oracle and prints one
  JSON line (n_gpus = 2, impl = reference); rank 1 exits 0 without work or output.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _combine_worker(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, units = bench.combine_ranks(10.0 + 5.0 * rank, 100 * (rank + 1), torch.device("cpu"))
        dist.barrier()
        queue.put((rank, ms, units))
    finally:
        dist.destroy_process_group()


def test_combine_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_combine_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(queue.get(timeout=120) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [g[0] for g in got] == [0, 1]
    for _, ms, units in got:
        assert ms == 15.0 and units == 300.0
    assert all(p.exitcode == 0 for p in procs)


def test_combine_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.combine_ranks(7.5, 42, None) == (7.5, 42.0)


def test_reference_arm_under_torchrun_two_ranks():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["value"] > 0 and d["unit"] == "nodes/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
