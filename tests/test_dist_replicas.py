"""Host logic of the multi-GPU bench (replicas, no data-path collective) on CPU with gloo:
world size 2, each rank reports its own timings; the bench reduces them with MAX (time) and
SUM (work) exactly as it does over NCCL on GPUs."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env()[:2] == (rank, world)
    mx = bench.reduce_over_ranks({"pre_ms": 10.0 + rank, "dec_ms": 5.0 * (rank + 1)}, "max")
    sm = bench.reduce_over_ranks({"tokens": 4096.0}, "sum")
    bench.barrier()
    q.put((rank, mx, sm))
    dist.destroy_process_group()


def test_replica_reduction_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, sm in results:
        assert mx == {"pre_ms": 11.0, "dec_ms": 10.0}
        assert sm == {"tokens": 8192.0}


def test_single_process_is_identity():
    import bench
    assert bench.reduce_over_ranks({"a": 3.0}, "max") == {"a": 3.0}


def test_bench_gpus_flag_starts_the_ranks():
    """`bench.py --gpus 2` outside a launcher starts two ranks itself (torch.distributed.run on
    127.0.0.1; gloo here without GPUs) and they form one group; inside a launcher whose world size
    differs from --gpus it refuses to run."""
    import json
    import subprocess
    import sys
    import bench
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_PORT")}
    res = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--gpus", "2", "--rank-check"],
                         capture_output=True, text=True, timeout=180, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [json.loads(ln) for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert lines == [{"rank_check": True, "world": 2, "ranks_summed": 2.0, "backend": lines[0]["backend"]}]
    env["WORLD_SIZE"] = "3"
    res = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--gpus", "2", "--rank-check"],
                         capture_output=True, text=True, timeout=60, env=env)
    assert res.returncode == 2
