"""The multi-process (replica) path of the benchmark on CPU: two gloo ranks, no GPU.

Every (batch, channel) and (batch, head) recurrence is independent, so N GPUs run N replicas
with no data-path collective; the only cross-rank steps are the barrier around the timed
region and the max over ranks of the step time. Each rank draws its own inputs (seed offset
by the rank)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from selective_state_space_127_b300.synth import scan_workload_inputs

    ms = bench._max_over_ranks(1.0 + 2.0 * rank, torch.device("cpu"), world)
    inp = scan_workload_inputs(0, rank=rank)
    dist.barrier()
    out[rank] = (ms, float(inp["x"].sum()))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_draw_different_inputs():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 3.0
    assert res[0][1] != res[1][1]
