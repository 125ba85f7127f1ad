"""The multi-GPU form is replicas only (one independent context per GPU, no
collective on the data path): bench.py combines the ranks' timings by their
maximum and counts every replica's tokens. Checked here with two gloo ranks
on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import importlib.util
    here = os.path.dirname(os.path.abspath(__file__))
    spec = importlib.util.spec_from_file_location("bench", os.path.join(here, "..", "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    # rank r pretends its timed steps took (100 + 50 r) ms on the device and (120 + 10 r) ms of wall time
    dev_ms, wall_ms = bench.max_over_ranks([100.0 + 50 * rank, 120.0 + 10 * rank], dist, "cpu")
    value = bench.replica_throughput(world, 8192, 5, dev_ms / 1e3)
    out[rank] = (dev_ms, wall_ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        dev_ms, wall_ms, value = res[r]
        assert dev_ms == 150.0 and wall_ms == 130.0  # every rank sees the slowest rank's times
        assert value == pytest.approx(2 * 8192 * 5 / 0.150)


def test_single_process_is_identity():
    import importlib.util
    here = os.path.dirname(os.path.abspath(__file__))
    spec = importlib.util.spec_from_file_location("bench", os.path.join(here, "..", "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    assert bench.max_over_ranks([1.5, 2.5], None, "cpu") == [1.5, 2.5]
    assert bench.replica_throughput(1, 100, 2, 0.5) == 400.0
