"""Multi-process host logic on CPU (gloo, world size 2). The bench runs one independent replica per GPU
and reports the whole job: the units all ranks processed over the slowest rank's time. Checked here:
the max-over-ranks reduction on a real two-rank process group, the whole-job value, and the reference
arm under a two-rank torchrun launch, where rank 0 alone runs and prints one line."""
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
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r times [1 + r, 10 - r] ms: the job's times are the slowest rank's, element by element
    vals = bench.max_over_ranks([1.0 + rank, 10.0 - rank])
    dist.barrier()
    q.put((rank, vals))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(q.get(timeout=180) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    assert results == [(0, [2.0, 10.0]), (1, [2.0, 10.0])]


def test_max_over_ranks_without_a_process_group_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks([3, 1.5]) == [3.0, 1.5]


def test_whole_job_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_value(549.8e9, 1, 0.5)
    assert one == pytest.approx(1099.6)
    assert bench.job_value(549.8e9, 2, 0.5) == pytest.approx(2 * one)  # weak scaling: two replicas
    assert bench.job_value(549.8e9, 2, 1.0) == pytest.approx(one)      # ... unless the slowest takes longer


def test_reference_arm_under_torchrun_world2():
    import oracle
    oracle.build()
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-rows", "16", "--workload", "b4h8_n1024_d64"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout  # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
