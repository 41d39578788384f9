"""The bench's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

Each rank draws its own batch (weak scaling, no collective on the data path);
timing is bracketed by barriers and the slowest rank's time sets the whole-job
throughput."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from gated_delta_rule_166_b300.inputs import make_prefill_inputs

    w, r, _ = bench.dist_setup(None)
    assert (w, r) == (world, rank)
    x = make_prefill_inputs(1, 8, 2, 32, 32, dtype=torch.float32, seed=bench.rank_seed(7, rank))
    bench.barrier(world)
    local_ms = 10.0 + 5.0 * rank
    ms_max = bench.max_over_ranks(local_ms, world)
    out[rank] = (ms_max, float(x.q.sum()), bench.aggregate_tokens_per_s(8, ms_max, world))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_independent_batches():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:   # no fork of a multi-threaded process
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0                      # slowest rank's time on every rank
    assert res[0][1] != res[1][1]                              # ranks draw different batches
    assert res[0][2] == pytest.approx(2 * 8 / 15e-3)           # all ranks' tokens / max time
