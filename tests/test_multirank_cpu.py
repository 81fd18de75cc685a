"""The multi-rank host logic of bench.py on CPU (two gloo ranks).

The verify step shards by sequence with no exchange: each rank runs its own
batch (its own seed), and the only collectives are the barrier and the
max-over-ranks of the timed region. These tests run that logic with the gloo
backend, and the reference arm under torchrun with two ranks (rank 0 prints
one line, rank 1 exits without work).
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads
        cfg = workloads.CONFIGS["tiny"]
        seed = bench.rank_seed(0, rank)
        s = workloads.make_sampling_inputs(cfg, seed=seed)
        local_ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
        total = bench.max_over_ranks(local_ms, torch.device("cpu"), world)
        value = bench.job_steps_per_sec(4, world, total)
        # every rank reports the same job time; inputs differ between ranks
        digest = float(s["target_logits"].double().sum())
        gathered = [None] * world
        dist.all_gather_object(gathered, (total, value, digest))
        if rank == 0:
            out.put(gathered)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time_and_own_distinct_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = q.get(timeout=120)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    (t0, v0, d0), (t1, v1, d1) = res
    assert t0 == t1 == 15.0                        # max over ranks
    assert v0 == v1 == pytest.approx(2 * 4 / 0.015)  # both ranks' steps count
    assert d0 != d1                                # rank r verifies seed + r


def test_single_rank_helpers():
    import bench
    assert bench.max_over_ranks(3.5, None, 1) == 3.5
    assert bench.rank_seed(7, 0) == 7 and bench.rank_seed(7, 3) == 10
    assert bench.job_steps_per_sec(10, 1, 1000.0) == pytest.approx(10.0)


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1                         # rank 0 only
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
