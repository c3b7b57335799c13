"""The replicas-only multi-GPU path of bench.py on CPU: two gloo ranks agree on the slowest rank's
time, which is what the whole-job throughput is computed from."""
import os
import socket
import sys


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, times, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=len(times))
    try:
        got = bench.slowest_rank(dist, times[rank], "cpu")
        dist.barrier()
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    times = [0.125, 0.5]
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 0.5, 1: 0.5}


def test_one_rank_is_its_own_slowest():
    import bench
    assert bench.slowest_rank(None, 0.25) == 0.25
