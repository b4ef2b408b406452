"""The N > 1 bench path on CPU: two gloo ranks, each a replica with its own
batch (no collective on the data path); only the step time is reduced (max
over ranks) and the job throughput counts every rank's tokens."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench._PG["on"] = True
    local_ms = [0.25, 0.40][rank]            # a slower second rank
    ms = bench.reduce_max(local_ms)
    value = bench.job_throughput(world, 4096, ms)
    # replicas draw different batches: the seed is the rank
    from memory_bound_moe_gb300.workloads import WORKLOADS, generate
    logits = generate(WORKLOADS["tiny"], seed=rank, parts=("logits",))["logits"]
    q.put((rank, ms, value, float(logits[0, 0])))
    bench.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][1] == res[1][1] == pytest.approx(0.40)
    assert res[0][2] == pytest.approx(2 * 4096 / 0.40e-3)
    assert res[0][3] != res[1][3]


def test_single_rank_reduce_is_identity():
    import bench
    assert bench.reduce_max(1.5) == 1.5
    assert bench.job_throughput(1, 4096, 0.1) == pytest.approx(4096 / 1e-4)


def test_reference_arm_under_torchrun_two_ranks():
    """bench.py --impl reference launched as the driver does for N = 2: rank 0
    times the oracle and prints one JSON line, the other rank exits 0 with no
    work and no output; no GPU is needed."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny"]
    res = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
