"""The N > 1 path of the benchmark on CPU: two gloo ranks on 127.0.0.1.

Every (batch, head) sequence of the scan is independent, so N ranks each run
their own batch with no collective on the data path; the only exchange is
the max over ranks of the timed region.  This checks that reduction and that
ranks draw distinct shards."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import synth
    t = bench.max_over_ranks(10.0 + rank * 5.0, world)
    sh = synth.SDM_TINY.with_(T=4)
    s1 = synth.sdm_inputs(sh, seed=bench.shard_seed(rank))["s1w"]
    gathered = [torch.zeros(s1.size) for _ in range(world)]
    dist.all_gather(gathered, torch.from_numpy(s1.ravel().copy()))
    out[rank] = (t, [bool(torch.equal(gathered[0], g)) for g in gathered])
    dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_distinct_shards():
    ctx = tmp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 15.0          # the slowest rank's time
    assert out[0][1] == [True, False]              # rank 1 drew a different batch


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
