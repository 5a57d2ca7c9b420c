"""The N > 1 benchmark path ("replicas only"): two gloo ranks on CPU check that the
whole-job aggregation is sum of work / max of time and that the barrier completes."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "CUDA_VISIBLE_DEVICES": ""})
    import sys
    from pathlib import Path
    sys.path.insert(0, str(Path(__file__).resolve().parents[1]))
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    t = bench.allreduce(0.5 + r, w, "max")        # per-rank times 0.5 s and 1.5 s
    b = bench.allreduce(100.0 * (r + 1), w, "sum")  # per-rank bytes 100 and 200
    q.put((r, w, t, b, b / t))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, w, t, b, v in res:
        assert w == 2
        assert t == pytest.approx(1.5)
        assert b == pytest.approx(300.0)
        assert v == pytest.approx(200.0)
