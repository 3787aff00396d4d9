"""Host-side logic of bench.py at N > 1 (the barrier and the max over
ranks), run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench._barrier(world)
    got = bench._max_over_ranks(10.0 + rank * 5.0, world, torch.device("cpu"))
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_flop_and_byte_conventions():
    import bench
    # 4 * B * Hq * d * S(S+1)/2 at the long-context prefill
    assert bench.causal_flops(1, 32, 131072, 128) == pytest.approx(1.4074e14, rel=1e-4)
    assert bench.causal_flops(1, 1, 1, 1) == 4.0
