"""The multi-rank bench logic on CPU with gloo, world size 2: every rank runs
its own replica (seeded by rank, so the batches differ), the step time is the
maximum over ranks, and the value counts the work of all ranks."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from llama_decoder_layer_gb300 import inputs as I
    bl = I.make_batch(I.SPECS["decode_70b"], seed=rank, device="cpu")
    my_ms = 10.0 + 5.0 * rank
    ms = bench.max_over_ranks(my_ms, world)
    rate = bench.whole_job_rate(bl.num_tokens, ms, world)
    bench.barrier(world)
    out[rank] = (ms, rate, sum(bl.ctx_lens))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_max_time_and_whole_job_value():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0          # slowest rank's time on every rank
    assert res[0][1] == res[1][1] == pytest.approx(128 * 2 / 0.015)
    assert res[0][2] != res[1][2]                   # independent replicas: different batches
