"""World-size-2 checks (gloo, CPU) of the host logic bench.py uses when run
under torchrun: independent (batch, head) units are split across ranks with
no data-path collective, and the step time is the max over ranks."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        units = bench.shard_units(37, rank, world)
        times = [3.0, 5.0]
        mx = bench.reduce_max(times[rank], dist)
        out[rank] = (units.start, units.stop, mx)
    finally:
        dist.destroy_process_group()


def test_two_ranks_shard_and_max():
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, free_port(), out), nprocs=2, start_method="spawn")
    a, b = out[0], out[1]
    assert (a[0], a[1]) == (0, 19) and (b[0], b[1]) == (19, 37)   # disjoint, complete
    assert a[2] == b[2] == 5.0                                     # max over ranks


@pytest.mark.parametrize("n,world", [(1, 1), (5, 8), (32, 4), (33, 4)])
def test_shard_units_partition(n, world):
    seen = []
    for r in range(world):
        seen.extend(bench.shard_units(n, r, world))
    assert seen == list(range(n))


def test_reduce_max_single_process_is_identity():
    assert bench.reduce_max(1.5, None) == 1.5


def test_flop_formula():
    from exact_second_order_two_gb300.synthetic import WORKLOADS
    w = WORKLOADS["bf16_causal_b2h16_n16384_d128"]
    assert bench.flops_bob(w) == pytest.approx(30 * 2 * 16 * 16384**2 * 128 / 2)
    assert bench.flops_bob(w, 10) == pytest.approx(bench.flops_bob(w) * 10 / 15)
