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


def _split_worker(rank, world, port, out):
    """Rank r runs the oracle on its own shard of the global tiny SDM workload
    (its batch elements, drawn with its seed) and the shards are gathered."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np
    import bench
    import oracle
    import synth
    sh = synth.SDM_TINY.with_(B=2, H=2, T=48)
    inp = synth.sdm_inputs(sh, seed=bench.shard_seed(rank))
    ref = oracle.sdm_forward(inp, sh.k, sh.W, sh.R)
    ys = [torch.zeros(ref["y"].size, dtype=torch.float64) for _ in range(world)]
    ms = [torch.zeros(ref["state"].size, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(ys, torch.from_numpy(np.ascontiguousarray(ref["y"]).ravel()))
    dist.all_gather(ms, torch.from_numpy(np.ascontiguousarray(ref["state"]).ravel()))
    if rank == 0:
        out["y"] = np.concatenate([g.numpy().reshape(ref["y"].shape) for g in ys], axis=0)
        out["state"] = np.concatenate([g.numpy().reshape(ref["state"].shape) for g in ms], axis=0)
    dist.destroy_process_group()


def test_bh_split_over_two_ranks_reassembles_the_single_process_result():
    """The multi-GPU split: one global workload of 2 x 2 batch elements, rank r
    taking rank_shard(r) (drawn with shard_seed(r)); the shards' oracle
    outputs, concatenated in rank order, equal the single-process oracle on the
    global input bit for bit (the sequences are independent: no exchange)."""
    import numpy as np
    import bench
    import oracle
    import synth
    ctx = tmp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    world = 2
    procs = [ctx.Process(target=_split_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    sh = synth.SDM_TINY.with_(B=2, H=2, T=48)
    parts = [synth.sdm_inputs(sh, seed=bench.shard_seed(r)) for r in range(world)]
    glob = {k: (np.concatenate([p[k] for p in parts], axis=0) if isinstance(parts[0][k], np.ndarray) else parts[0][k])
            for k in parts[0]}
    assert glob["s1w"].shape[0] == bench.global_batch(sh.B, world)
    for r in range(world):
        sl = bench.rank_shard(sh.B, world, r)
        assert np.array_equal(glob["v"][sl], parts[r]["v"])
    ref = oracle.sdm_forward(glob, sh.k, sh.W, sh.R)
    assert np.array_equal(out["y"], ref["y"])
    assert np.array_equal(out["state"], ref["state"])


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
