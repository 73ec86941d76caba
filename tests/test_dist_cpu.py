"""The multi-rank path of bench.py on CPU with gloo, world size 2: rendezvous on
127.0.0.1, barrier, max over ranks of the timed region, and only rank 0 printing
the reference arm's line (the other ranks exit without work).  Each rank is an
independent replica of the workload; there is no data-path collective."""
import multiprocessing as mp
import os
import socket


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                      RANK=str(rank), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import torch.distributed as dist
    world, r, _ = bench.dist_setup(2)
    bench.barrier(world)
    mx = bench.max_over_ranks(world, 10.0 * (r + 1))
    # the reference arm: ranks other than 0 return at once, before any work
    import argparse
    args = argparse.Namespace(steps=1, warmup=3, ref_budget=1.0)
    if r != 0:
        bench.reference(args)
    bench.barrier(world)
    assert dist.get_backend() == "gloo"
    dist.destroy_process_group()
    q.put((r, world, mx))


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
    assert all(p.exitcode == 0 for p in ps), [p.exitcode for p in ps]
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r for r, *_ in res] == [0, 1]
    assert all(w == 2 and mx == 20.0 for _, w, mx in res)
