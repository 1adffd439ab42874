"""The multi-process path of bench.py on CPU: two gloo ranks agree on the
barrier and on the max-over-ranks timing, and draw different seeds."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    d = bench.Dist()
    try:
        d.barrier()
        out[rank] = (d.world, d.max(1.5 + rank))
    finally:
        d.close()


def test_two_gloo_ranks_max_and_barrier():
    world, port = 2, _free_port()
    # spawn, not fork: earlier tests may have started threads (the oracle's
    # OpenMP pool) in this process
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        got = dict(out)
    assert got == {0: (2, 2.5), 1: (2, 2.5)}
