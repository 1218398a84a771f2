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


def test_reference_arm_prints_one_contract_line():
    """bench.py --impl reference (the fp64 oracle on this host's cores) prints
    one JSON line with the keys of the benchmark contract, on CPU, for the tiny
    workload; the 1.4B-layer metric name is kept for the default workload only."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload",
                        "sdm_tiny", "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=600,
                       cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["config"]["workload"] == "sdm_tiny" and "sdm_tiny" in d["metric"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
