"""Host logic of the multi-GPU replica mode, on CPU with gloo (world size 2):
the max-over-ranks step time, the barrier, and the reference arm printing on
rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    ws, r, local = bench.dist_setup(world)
    bench.barrier(ws)
    m = bench.max_over_ranks(float(10 + 5 * rank), ws)
    args = type("A", (), {"config": "tiny", "ref_tokens": 2, "steps": 1, "warmup": 0, "x": "fp8", "shared": 0,
                          "f8_gran": 0})()
    res = bench.run_reference(args, ws, r)
    q.put((rank, ws, m, res is None, None if res is None else res["impl"]))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [2, 2]
    assert [o[2] for o in out] == [15.0, 15.0]            # max over ranks
    assert out[0][3] is False and out[0][4] == "reference" # rank 0 runs the oracle arm
    assert out[1][3] is True                               # rank 1 does no work
