"""Replica aggregation of bench.py on two gloo ranks (CPU): the time is the maximum over ranks and
the work is the sum, as the multi-GPU benchmark reports it."""
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


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://")
    import bench
    assert bench.dist_info() == (rank, world, rank)
    bench.barrier()
    t, u = bench.aggregate(1.5 + rank, 100.0 * (rank + 1))
    out[rank] = (t, u)
    dist.destroy_process_group()


def test_aggregate_max_time_sum_units():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: (2.5, 300.0), 1: (2.5, 300.0)}


def test_single_process_aggregate_is_identity():
    import bench
    assert bench.aggregate(3.0, 7.0) == (3.0, 7.0)


@pytest.mark.parametrize("name", ["llama2-7b-ffn-b1", "llama2-7b-ffn-b16", "llama-70b-ffn-b64-p16"])
def test_workload_counts_and_bytes(name):
    # the benchmark's touched-byte accounting uses the counting rule the oracle defines
    import bench
    import oracle
    wl = bench.WORKLOADS[name]
    c = oracle.region_counts(wl["N"], wl["r"], wl["gamma"])
    gu, dn = bench.touched_bytes(c, wl["D"])
    assert gu == 2 * (c.n_R + c.n_C) * wl["D"] * 2 and dn == c.keep * wl["D"] * 2
    if name == "llama2-7b-ffn-b1":
        assert abs((gu + dn) / 1e6 - 207.68) < 0.01   # 7B, B=1: 207.68 MB touched per decode step
