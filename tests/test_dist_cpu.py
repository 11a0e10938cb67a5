"""The N-replica plumbing of bench.py (rendezvous, barrier, max over ranks) with two gloo
ranks on CPU."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world)
    bench.barrier(w)
    m = bench.max_over_ranks(10.0 + 3.0 * r, w)
    q.put((r, w, local, m, dist.get_backend()))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 and g[3] == 13.0 and g[4] == "gloo" for g in got)
