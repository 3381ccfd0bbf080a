"""The multi-rank host logic of bench.py on CPU: two gloo ranks agree on the
slowest rank's time and on the whole-job rate (decode batches are
independent problems, so ranks exchange nothing but this timing)."""
import os
import socket
import sys

import torch.multiprocessing as mp

import helpers


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    import torch.distributed as td
    sys.path.insert(0, helpers.ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    td.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 0.5 + rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(my_ms)
        rate = bench.whole_job_rate(4, world, slowest)
        q.put((rank, slowest, rate))
    finally:
        td.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [1.5, 1.5]
    assert all(abs(o[2] - 4 * 2 / 1.5e-3) < 1e-6 for o in out)


def test_single_process_needs_no_group():
    sys.path.insert(0, helpers.ROOT)
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.whole_job_rate(4, 1, 0.05) == 80000.0
