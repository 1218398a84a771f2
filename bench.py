#!/usr/bin/env python3
"""Benchmark of the sparse-routed gated delta-rule memory scan on GB300.

Default workload: the SDM 1.4B-layer shape (d=1920, H=2 -> N=57600 slots per
head, d_v=960, per-half top-k=16, W=R=16, B=8, T=4096, bf16 values, fp32
table).  One step = write addressing + read addressing + the scan over the
whole batch, continuing the table from the previous step (the scan is a
recurrence; a step is the next B*T tokens of the same sequences, so every
step does identical work).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload sdm_14b_layer|sdm_sweep_H2|H4|H8|gdn|kda|gdn2|sse|sse_delta|sdm_tiny|sdm_decode|sse_decode|
                               sdm_train|sdm_chunked]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own batch
(independent sequences, no collective in the data path) and the time is the
max over ranks.  `--impl reference` times the fp64 CPU oracle on this host's
cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SDM scan tokens/s (d=1920,H=2,N=57600,W=R=16); achieved HBM GB/s vs peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the dominant
# call of a workload, recorded from an ncu capture.  It is a record, not a
# measurement of this run, and is reported only while the kernel source still
# hashes to the digest it was taken at; otherwise the line carries null.
NCU_TRAFFIC = {
    # one full-size sparse scan launch: 7.98 GB read + 4.17 GB written
    ("sdm_14b_layer", "sdm"): {"bytes": 12.15e9, "digest": "9010d40ae7b9"},
    # both kernels of one full-size gdn_scan call: 746.1 MB read + 591.0 MB written
    ("gdn", "gdn"): {"bytes": 1.337e9, "digest": "c77c8abaf750"},
    # both kernels of one full-size KDA gdn_scan call: 947.1 MB read + 663.2 MB written
    ("kda", "kda"): {"bytes": 1.610e9, "digest": "c77c8abaf750"},
    # both kernels of one full-size gdn2_scan call: 1214.6 MB read + 673.5 MB written
    ("gdn2", "gdn2"): {"bytes": 1.888e9, "digest": "c77c8abaf750"},
    # the five kernels of one full-size sse_scan call on the chunked path: 1.063 GB read + 0.807 GB written
    ("sse", "sse"): {"bytes": 1.869e9, "digest": "106dd028442b"},
    # the five kernels of one full-size delta-write sse_scan call: 1.387 GB read + 1.110 GB written
    ("sse_delta", "sse"): {"bytes": 2.497e9, "digest": "c77c8abaf750"},
}


def _src_digest(name: str) -> str:
    p = os.path.join(ROOT, "delta_rule_memory_gb300", "csrc", name)
    return hashlib.sha1(open(p, "rb").read()).hexdigest()[:12]


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest x over all ranks (the slowest rank's time); x itself at N=1.
    Works on the nccl (CUDA tensor) and gloo (CPU tensor) backends."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard_seed(rank: int) -> int:
    """Each rank draws its own batch: independent sequences, no exchange."""
    return rank


def global_batch(B: int, world: int) -> int:
    """Under N ranks the job is one global workload of B * N sequences per
    head: rank r owns the batch elements rank_shard(r) and draws them with
    seed shard_seed(r), so the global input is the per-rank draws
    concatenated along the batch axis."""
    return B * world


def rank_shard(B: int, world: int, rank: int) -> slice:
    """The batch elements of the global workload (global_batch(B, world)
    sequences per head) that rank `rank` runs: a contiguous block of B.
    Every (batch, head) sequence of the scan is independent, so the ranks
    exchange nothing and their outputs, concatenated in rank order along the
    batch axis, are the global workload's outputs."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    return slice(rank * B, (rank + 1) * B)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 - 1 <= r[0] <= (self.t1 or r[0]) + 1]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use)}


# ------------------------------------------------------- CPU oracle (spawn)
def _oracle_sdm_seq(args):
    """One (b, h) sequence through the oracle: both addressings and the scan."""
    import numpy as np
    import oracle
    s1w, s2w, s1r, s2r, v, alpha, beta, k, W, R, mode = args
    t0 = time.perf_counter()
    iw, ww = oracle.address(s1w, s2w, k, W)
    ir, wr = oracle.address(s1r, s2r, k, R)
    n = s1w.shape[-1] ** 2
    M0 = np.zeros((1, 1, n, v.shape[-1]))
    oracle.sdm_scan(M0, v, alpha, beta, iw, ww, ir, wr, mode)
    return time.perf_counter() - t0


def _oracle_gdn_seq(args):
    import numpy as np
    import oracle
    q, k, v, a, beta, per_channel = args
    t0 = time.perf_counter()
    oracle.gdn_scan(np.zeros((1, 1, q.shape[-1], v.shape[-1])), q, k, v, a, beta, per_channel)
    return time.perf_counter() - t0


def _oracle_gdn2_seq(args):
    import numpy as np
    import oracle
    q, k, v, a, b_erase, w_write = args
    t0 = time.perf_counter()
    oracle.gdn2_scan(np.zeros((1, 1, q.shape[-1], v.shape[-1])), q, k, v, a, b_erase, w_write)
    return time.perf_counter() - t0


def _oracle_sse_seq(args):
    import numpy as np
    import oracle
    route, topk, klog, q, v, alpha, mode = args
    t0 = time.perf_counter()
    N, c, d = route.shape[-1], klog.shape[-1], v.shape[-1]
    oracle.sse_scan(np.zeros((1, 1, N + 1, c, d)), route, topk, klog, q, v, alpha, mode)
    return time.perf_counter() - t0


def cpu_model() -> str:
    """The host CPU's model name (x86: /proc/cpuinfo; Arm: lscpu)."""
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


class OracleSampler:
    """Runs the oracle over whole (b, h) sequences (first t_sample tokens) in a
    spawn process pool created before any GPU work.

    The GPU's `value` counts tokens (B*T, each with all H heads), so a sample
    of `nseq` (b, h) sequences of t_sample tokens is nseq*t_sample/H tokens."""

    def __init__(self, cores: int):
        self.cores = max(1, cores)
        self.pool = mp.get_context("spawn").Pool(self.cores)

    def close(self):
        self.pool.close()
        self.pool.join()

    def run(self, wl: "Workload", inp: dict, t_sample: int, nseq: int):
        """All-core run: (tokens, wall seconds), one process per sequence."""
        jobs = wl.oracle_jobs(inp, t_sample, nseq)
        fn = {"sdm": _oracle_sdm_seq, "gdn": _oracle_gdn_seq, "kda": _oracle_gdn_seq, "gdn2": _oracle_gdn2_seq,
              "sse": _oracle_sse_seq}[wl.kind]
        t0 = time.perf_counter()
        self.pool.map(fn, jobs, chunksize=1)
        wall = time.perf_counter() - t0
        return len(jobs) * t_sample / wl.shape.H, wall

    def run_single(self, wl: "Workload", inp: dict, t_sample: int):
        """One sequence on one core: (tokens, seconds) of the oracle alone."""
        job = wl.oracle_jobs(inp, t_sample, 1)
        fn = {"sdm": _oracle_sdm_seq, "gdn": _oracle_gdn_seq, "kda": _oracle_gdn_seq, "gdn2": _oracle_gdn2_seq,
              "sse": _oracle_sse_seq}[wl.kind]
        secs = self.pool.map(fn, job, chunksize=1)[0]
        return t_sample / wl.shape.H, secs


def metric_name(wl) -> str:
    if wl.decode:
        return f"{wl.kind} decode tokens/s (one token per sequence per step; ms_per_step is the step latency)"
    if wl.train:
        return "SDM training step tokens/s (addressing, forward with undo log, scan and address backward)"
    import synth
    sh = wl.shape
    if wl.kind == "sdm":
        if wl.chunked:
            return "SDM scan tokens/s in chunked form (sdm_scan_chunked, 1.4B layer); achieved HBM GB/s vs peak"
        if wl.name != "sdm_14b_layer":
            return f"SDM scan tokens/s ({wl.name}); achieved HBM GB/s vs peak"
        ref = synth.SDM_14B_LAYER
        changed = [f"{k}={getattr(sh, k)}" for k in ("B", "T") if getattr(sh, k) != getattr(ref, k)]
        if wl.mode != 0:
            changed.append("perslot")
        if changed:
            # a modified run never reports under the 1.4B layer's metric name
            return f"SDM scan tokens/s (1.4B layer, {', '.join(changed)}); achieved HBM GB/s vs peak"
        return METRIC
    if sh.B != {"gdn": synth.GDN_DENSE, "kda": synth.GDN_DENSE, "gdn2": synth.GDN_DENSE,
                "sse": synth.SSE_PART}[wl.kind].B:
        return f"{wl.kind} scan tokens/s (B={sh.B})"
    return f"{wl.kind} scan tokens/s"


# ---------------------------------------------------------------- workloads
class Workload:
    def __init__(self, name: str, mode: str, batch: int = 0):
        import synth
        self.name = name
        self.mode = {"shared": 0, "perslot": 1}[mode]
        # decode: one token per sequence per step (T = 1), the state carried across steps
        self.decode = name.endswith("_decode")
        if self.decode:
            name = {"sdm_decode": "sdm_14b_layer", "sse_decode": "sse"}[name]
        # train: forward with the undo log, the scan backward and the address backward
        self.train = name == "sdm_train"
        # chunked: the same scan in chunked form (sdm_scan_chunked)
        self.chunked = name == "sdm_chunked"
        if self.train or self.chunked:
            name = "sdm_14b_layer"
        if name == "sdm_14b_layer":
            self.kind, self.shape = "sdm", synth.SDM_14B_LAYER
        elif name.startswith("sdm_sweep_H"):
            self.kind, self.shape = "sdm", synth.sdm_sweep_shape(int(name[len("sdm_sweep_H"):]))
        elif name == "sdm_tiny":
            self.kind, self.shape = "sdm", synth.SDM_TINY
        elif name in ("gdn", "kda", "gdn2"):
            self.kind, self.shape = name, synth.GDN_DENSE
        elif name in ("sse", "sse_delta"):
            self.kind, self.shape = "sse", synth.SSE_PART
        else:
            raise SystemExit(f"unknown workload {name}")
        self.sse_mode = 1 if name == "sse_delta" else 0  # sse_scan write mode: additive / delta
        self.sse_chunked = False  # set once the workspace query tells which path sse_scan takes
        if batch:
            self.shape = self.shape.with_(B=batch)
        if self.decode:
            self.shape = self.shape.with_(T=1, name=self.shape.name + "_decode")
        if self.train:
            self.shape = self.shape.with_(name=self.shape.name + "_train")
        if self.chunked:
            self.shape = self.shape.with_(name=self.shape.name + "_chunked")
        sh = self.shape
        self.tokens = sh.B * sh.T

    def inputs(self, seed: int) -> dict:
        import synth
        if self.kind == "sdm":
            return synth.sdm_inputs(self.shape, seed)
        if self.kind in ("gdn", "kda", "gdn2"):
            return synth.gdn_inputs(self.shape, seed)
        return synth.sse_inputs(self.shape, seed)

    def config(self) -> dict:
        sh = self.shape
        if self.kind == "sdm":
            state_gb = sh.B * sh.H * sh.N * sh.d_v * 4 / 1e9
            return {"workload": sh.name, "B": sh.B, "T": sh.T, "H": sh.H, "N": sh.N, "sqrtN": sh.sqrtN, "d_v": sh.d_v,
                    "k": sh.k, "W": sh.W, "R": sh.R, "v_dtype": "bf16" if sh.v_bf16 else "fp32",
                    "resid": ["shared", "per_slot"][self.mode], "state": f"fp32 {state_gb:.2f} GB, continued across steps",
                    "l2": f"inputs larger than L2 (table {state_gb:.2f} GB); no flush"}
        if self.kind in ("gdn", "kda", "gdn2"):
            return {"workload": f"{self.kind}_dense", "B": sh.B, "T": sh.T, "H": sh.H,
                    "dk": sh.dk, "dv": sh.dv, "qkv_dtype": "bf16", "state": "fp32, continued across steps",
                    "l2": "inputs (q,k,v,alpha,y ~340-470 MB) larger than L2; no flush"}
        return {"workload": sh.name, "B": sh.B, "T": sh.T, "H": sh.H, "N": sh.N, "topk": sh.topk, "c": sh.c, "d": sh.d,
                "write": ["additive", "delta"][self.sse_mode], "qv_dtype": "bf16",
                "state": "fp32, continued across steps",
                "l2": "inputs (~1.1 GB) larger than L2; no flush"}

    def oracle_jobs(self, inp: dict, t_sample: int, nseq: int):
        sh = self.shape
        pairs = [(b, h) for b in range(sh.B) for h in range(sh.H)][:nseq]
        jobs = []
        for b, h in pairs:
            sl = (slice(b, b + 1), slice(0, t_sample), slice(h, h + 1))
            if self.kind == "sdm":
                jobs.append((inp["s1w"][sl].copy(), inp["s2w"][sl].copy(), inp["s1r"][sl].copy(),
                             inp["s2r"][sl].copy(), inp["v"][sl].copy(), inp["alpha"][sl].copy(),
                             inp["beta"][sl].copy(), sh.k, sh.W, sh.R, self.mode))
            elif self.kind == "gdn2":
                jobs.append((inp["q"][sl].copy(), inp["k"][sl].copy(), inp["v"][sl].copy(), inp["alpha_kda"][sl].copy(),
                             inp["b_erase"][sl].copy(), inp["w_write"][sl].copy()))
            elif self.kind in ("gdn", "kda"):
                a = inp["alpha_kda" if self.kind == "kda" else "alpha_gdn"]
                jobs.append((inp["q"][sl].copy(), inp["k"][sl].copy(), inp["v"][sl].copy(), a[sl].copy(),
                             inp["beta"][sl].copy(), self.kind == "kda"))
            else:
                jobs.append((inp["route"][sl].copy(), sh.topk, inp["klog"][sl].copy(), inp["q"][sl].copy(),
                             inp["v"][sl].copy(), inp["alpha"][sl].copy(), self.sse_mode))
        return jobs


# ------------------------------------------------------------ GPU runners
def _t(x, bf16=False):
    import numpy as np
    import torch
    x = np.ascontiguousarray(x)
    if bf16 or x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16)
    return torch.from_numpy(x.copy())


class GpuRun:
    """Device buffers plus one step of the workload through the binding."""

    def __init__(self, wl: Workload, inp: dict, device):
        import torch
        import delta_rule_memory_gb300 as sdm
        self.sdm, self.wl, self.dev = sdm, wl, device
        self.overlap = False
        sh = wl.shape
        self.host = {}
        self.d = {}
        if wl.kind == "sdm":
            names = ("s1w", "s2w", "s1r", "s2r", "v", "alpha", "beta")
        elif wl.kind == "gdn2":
            names = ("q", "k", "v", "alpha_kda", "b_erase", "w_write")
        elif wl.kind in ("gdn", "kda"):
            names = ("q", "k", "v", "alpha_kda" if wl.kind == "kda" else "alpha_gdn", "beta")
        else:
            names = ("route", "klog", "q", "v", "alpha")
        for n in names:
            h = _t(inp[n]).pin_memory()
            self.host[n] = h
            self.d[n] = h.to(device)
        if wl.kind == "sdm":
            B, T, H = sh.B, sh.T, sh.H
            self.state = torch.zeros((B, H, sh.N, sh.d_v), dtype=torch.float32, device=device)
            # two sets of addressing outputs: with the pipelined schedule the next
            # step's addresses are written into one while this step's scan reads the other
            self.addr_sets = [tuple(torch.empty((B, T, H, n), dtype=dt, device=device)
                                    for n, dt in ((sh.W, torch.int32), (sh.W, torch.float32),
                                                  (sh.R, torch.int32), (sh.R, torch.float32)))
                              for _ in range(2)]
            self.use_set(0)
            self.y = torch.empty((B, T, H, sh.d_v), dtype=torch.float32, device=device)
            self.ws = torch.empty(sdm.sdm_scan_workspace_size(B, T, H, sh.W, sh.R), dtype=torch.uint8, device=device)
            self.launches_per_step = 4
            if wl.chunked:
                self.ws_c = torch.empty(sdm.sdm_scan_chunked_workspace_size(B, T, H, sh.W, sh.R), dtype=torch.uint8,
                                        device=device)
            if wl.train:
                g = torch.Generator(device=device)
                g.manual_seed(12345)
                self.undo = torch.empty((B, T, H, sh.W, sh.d_v), dtype=torch.float32, device=device)
                # dL/dM_T carries over from step to step (accumulated), so no table-sized memset per step
                self.dstate = torch.zeros_like(self.state)
                self.dy = torch.randn((B, T, H, sh.d_v), generator=g, device=device)
                self.ws_b = torch.empty(sdm.sdm_scan_backward_workspace_size(B, T, H, sh.W, sh.R, sh.d_v),
                                        dtype=torch.uint8, device=device)
                self.launches_per_step = 8  # 2 address, record + scan, backward + reduce, 2 address backward
        elif wl.kind == "gdn2":
            self.state = torch.zeros((sh.B, sh.H, sh.dk, sh.dv), dtype=torch.float32, device=device)
            self.y = torch.empty((sh.B, sh.T, sh.H, sh.dv), dtype=torch.float32, device=device)
            nws = sdm.gdn2_scan_workspace_size(sh.B, sh.T, sh.H, sh.dk, sh.dv)
            self.ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=device)
            # chunked: preparation kernel + chain kernel; token-recurrent: one kernel
            self.launches_per_step = 2 if nws > 0 else 1
        elif wl.kind in ("gdn", "kda"):
            self.state = torch.zeros((sh.B, sh.H, sh.dk, sh.dv), dtype=torch.float32, device=device)
            self.y = torch.empty((sh.B, sh.T, sh.H, sh.dv), dtype=torch.float32, device=device)
            nws = sdm.gdn_scan_workspace_size(sh.B, sh.T, sh.H, sh.dk, sh.dv, wl.kind == "kda")
            self.ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=device)
            # chunked GDN / KDA: preparation kernel + chain kernel; token-recurrent: one kernel
            self.launches_per_step = 2 if nws > 0 else 1
        else:
            self.state = torch.zeros((sh.B, sh.H, sh.N + 1, sh.c, sh.d), dtype=torch.float32, device=device)
            self.y = torch.empty((sh.B, sh.T, sh.H, sh.d), dtype=torch.float32, device=device)
            nws = sdm.sse_scan_workspace_size(sh.B, sh.T, sh.H, sh.N, sh.topk, sh.c, sh.d, wl.sse_mode)
            self.ws = torch.empty(nws, dtype=torch.uint8, device=device)
            # chunked prefill: route, group, chunk preparation, chain, combine; else route + scan kernel
            rec = (sh.B * sh.T * sh.H * ((2 * sh.topk + 5) & ~3) * 4 + 255) // 256 * 256
            wl.sse_chunked = nws > rec
            self.launches_per_step = 5 if wl.sse_chunked else 2
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.y_host = torch.empty(self.y.shape, dtype=torch.float32).pin_memory()

    def use_set(self, k: int):
        self.iw, self.ww, self.ir, self.wr = self.addr_sets[k]

    def pipelined(self) -> bool:
        """With --overlap-addressing, the sparse inference step: the two
        addressing calls of step s+1 do not depend on the scan of step s,
        whose 960 warps leave SMs free, so they run on a second stream while
        that scan runs.  Every step still does its full addressing and scan
        exactly once."""
        wl = self.wl
        return self.overlap and wl.kind == "sdm" and not (wl.train or wl.chunked or wl.decode)

    def run_steps(self, K: int, ev, stream):
        """K timed steps; ev[i] brackets step i's scan call on the main stream."""
        import torch
        if not self.pipelined():
            for i in range(K):
                self.pre()
                ev[i][0].record(stream)
                self.main()
                ev[i][1].record(stream)
            return
        side = getattr(self, "side", None) or torch.cuda.Stream()
        self.side = side
        addr_done = [torch.cuda.Event(), torch.cuda.Event()]
        scan_done = [torch.cuda.Event(), torch.cuda.Event()]
        self.use_set(0)
        self._run_pre()  # step 0's addresses, on the main stream
        for i in range(K):
            s = i & 1
            if i > 0:
                stream.wait_event(addr_done[s])
            if i + 1 < K:
                side.wait_stream(stream) if i == 0 else side.wait_event(scan_done[s ^ 1])
                with torch.cuda.stream(side):
                    self.use_set(s ^ 1)
                    self._run_pre()
                    addr_done[s ^ 1].record(side)
            self.use_set(s)
            ev[i][0].record(stream)
            self._run_main()
            ev[i][1].record(stream)
            scan_done[s].record(stream)
        stream.wait_stream(side)
        self.use_set(0)

    def enable_graphs(self):
        """Replay the step's launches as CUDA graphs (decode: a handful of short
        kernels per token, so host launch latency would otherwise dominate).
        Every buffer, the state included, stays where it is, so a replay is the
        same step; the library's calls allocate nothing and never synchronise,
        which makes them capturable."""
        import torch
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self._run_pre()
            self._run_main()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        if self.wl.kind == "sdm":
            # the two addressing calls are independent: parallel branches of the graph
            fork = torch.cuda.Stream()
            self.g_pre = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.g_pre):
                self._run_pre(fork)
        self.g_main = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_main):
            self._run_main()
        torch.cuda.synchronize()

    def pre(self):
        if getattr(self, "g_pre", None) is not None:
            self.g_pre.replay()
        elif getattr(self, "g_main", None) is None:
            self._run_pre()

    def main(self):
        if getattr(self, "g_main", None) is not None:
            self.g_main.replay()
        else:
            self._run_main()

    def _run_pre(self, fork=None):
        """Work before the dominant kernel (addressing).  With `fork`, the read
        addressing runs on that stream beside the write addressing."""
        import torch
        sh, d = self.wl.shape, self.d
        if self.wl.kind == "sdm":
            if fork is None:
                self.sdm.sdm_address(d["s1w"], d["s2w"], sh.k, sh.W, self.iw, self.ww, self.err)
                self.sdm.sdm_address(d["s1r"], d["s2r"], sh.k, sh.R, self.ir, self.wr, self.err)
                return
            cur = torch.cuda.current_stream()
            fork.wait_stream(cur)
            with torch.cuda.stream(fork):
                self.sdm.sdm_address(d["s1r"], d["s2r"], sh.k, sh.R, self.ir, self.wr, self.err)
            self.sdm.sdm_address(d["s1w"], d["s2w"], sh.k, sh.W, self.iw, self.ww, self.err)
            cur.wait_stream(fork)

    def _run_main(self):
        """The dominant kernel's call."""
        sh, d = self.wl.shape, self.d
        if self.wl.kind == "sdm" and self.wl.train:
            self.sdm.sdm_scan_train(self.state, d["v"], d["alpha"], d["beta"], self.iw, self.ww, self.ir, self.wr,
                                    self.wl.mode, self.y, self.undo, self.ws, self.err)
            _, _, _, dww, dwr = self.sdm.sdm_scan_backward(self.state, self.dstate, d["v"], d["alpha"], d["beta"],
                                                           self.iw, self.ww, self.ir, self.wr, self.undo, self.dy,
                                                           self.wl.mode, self.ws_b, self.err)
            self.sdm.sdm_address_backward(self.iw, self.ww, dww, sh.sqrtN, self.err)
            self.sdm.sdm_address_backward(self.ir, self.wr, dwr, sh.sqrtN, self.err)
        elif self.wl.kind == "sdm" and self.wl.chunked:
            self.sdm.sdm_scan_chunked(self.state, d["v"], d["alpha"], d["beta"], self.iw, self.ww, self.ir, self.wr,
                                      self.wl.mode, self.y, self.ws_c, self.err)
        elif self.wl.kind == "sdm":
            self.sdm.sdm_scan(self.state, d["v"], d["alpha"], d["beta"], self.iw, self.ww, self.ir, self.wr,
                              self.wl.mode, self.y, self.ws, self.err)
        elif self.wl.kind == "gdn2":
            self.sdm.gdn2_scan(self.state, d["q"], d["k"], d["v"], d["alpha_kda"], d["b_erase"], d["w_write"], self.y,
                               workspace=self.ws, dev_err=self.err)
        elif self.wl.kind in ("gdn", "kda"):
            a = d["alpha_kda" if self.wl.kind == "kda" else "alpha_gdn"]
            self.sdm.gdn_scan(self.state, d["q"], d["k"], d["v"], a, d["beta"], self.wl.kind == "kda", self.y,
                              workspace=self.ws, dev_err=self.err)
        else:
            self.sdm.sse_scan(self.state, d["route"], sh.topk, d["klog"], d["q"], d["v"], d["alpha"], self.y,
                              None, self.ws, self.err, write_mode=self.wl.sse_mode)

    def step(self):
        self.pre()
        self.main()

    def e2e_step(self, chunk_T: int = 384):
        """One step through the public API from host buffers: for the sparse
        workloads the native pipelined entry point sdm_forward_host (inputs
        copied in and y copied out per chunk, overlapped with compute); for the
        dense and SSE scans and the training step, copies of the step's inputs
        and y around the call."""
        if self.wl.kind == "sdm" and not self.wl.train and not self.wl.chunked:
            import torch
            sh, hst = self.wl.shape, self.host
            if not hasattr(self, "fh_ws"):
                need = self.sdm.sdm_forward_host_workspace_size(sh.B, sh.T, sh.H, sh.sqrtN, sh.d_v, sh.W, sh.R,
                                                                sh.v_bf16, chunk_T)
                self.fh_ws = torch.empty(need, dtype=torch.uint8, device=self.dev)
            self.sdm.sdm_forward_host(hst["s1w"], hst["s2w"], hst["s1r"], hst["s2r"], hst["v"], hst["alpha"],
                                      hst["beta"], sh.k, sh.W, sh.R, self.state, self.y_host, self.wl.mode, chunk_T,
                                      self.fh_ws, self.err)
        else:
            self.h2d()
            self.step()
            self.d2h()

    def h2d(self):
        for n, h in self.host.items():
            self.d[n].copy_(h, non_blocking=True)

    def d2h(self):
        self.y_host.copy_(self.y, non_blocking=True)

    def io_bytes(self):
        return sum(h.numel() * h.element_size() for h in self.host.values()), self.y.numel() * 4

    def algorithmic(self):
        """(bytes or flops, unit, bound) of one launch of the dominant call."""
        import torch
        sh = self.wl.shape
        if self.wl.kind == "sdm":
            W, R = sh.W, sh.R
            both = torch.cat([self.iw, self.ir], dim=-1).reshape(-1, W + R)
            srt, _ = torch.sort(both, dim=-1)
            union = (srt[:, 1:] != srt[:, :-1]).sum(dim=-1) + 1
            rows = float((union + W).sum().item())       # rows loaded once + written rows stored once
            tokh = sh.B * sh.T * sh.H
            vbytes = 2 if sh.v_bf16 else 4
            per_tok = sh.d_v * vbytes + sh.d_v * 4 + 8 + (W + R) * 8
            total = rows * sh.d_v * 4 + tokh * per_tok
            if self.wl.train:
                # + the undo log written; backward: M rows read for the read slots, gradient rows read and
                # written for read and write slots, the log read and the table rows restored; v, dy read,
                # dv written; per-tile column sums written and read; both address backwards' score rows
                tiles = (sh.d_v + 31) // 32
                total += tokh * (W * sh.d_v * 4 + (3 * R + 4 * W) * sh.d_v * 4 + sh.d_v * (vbytes + 8) + 8
                                 + 2 * tiles * (W + R + 2) * 4 + 2 * 2 * sh.sqrtN * 4 + (W + R) * 16)
            return total, "GB/s", "hbm", {
                "mean_union_rows": float(union.float().mean().item()),
                "bytes_per_token_head": total / tokh}
        if self.wl.kind == "gdn2":
            tokh = sh.B * sh.T * sh.H
            per = 2 * (sh.dk + sh.dk + sh.dv) + 4 * sh.dk * 2 + 4 * sh.dv + 4 * sh.dv  # q k v, alpha b, w, y
            state = 2 * sh.B * sh.H * sh.dk * sh.dv * 4
            return tokh * per + state, "GB/s", "hbm", {"bytes_per_token_head": per}
        if self.wl.kind in ("gdn", "kda"):
            tokh = sh.B * sh.T * sh.H
            per = 2 * (sh.dk + sh.dk + sh.dv) + 4 * (sh.dk if self.wl.kind == "kda" else 1) + 4 + 4 * sh.dv
            state = 2 * sh.B * sh.H * sh.dk * sh.dv * 4
            return tokh * per + state, "GB/s", "hbm", {"bytes_per_token_head": per}
        tokh = sh.B * sh.T * sh.H
        # Both SSE paths are measured against the FP32-pipe roofline of the recurrence's own arithmetic:
        # per visited partition and state element a decay mul, a write fma and a read fma (1 + 2 + 2
        # flop; the delta write adds the prediction fma, 2).  The chunked prefill does that work in
        # another order (partly on the tensor cores), so for it this is an effective rate; its HBM
        # I/O (router and key logits, q, v, alpha in; y out; every partition's state read and written
        # once) is reported beside it.
        flops = tokh * (sh.topk + 1) * sh.c * sh.d * (7.0 if self.wl.sse_mode else 5.0)
        info = {"flops_per_token_head": flops / tokh}
        if self.wl.sse_chunked:
            per = 4 * sh.N + 4 * sh.c + 2 * sh.c + 2 * sh.d + 4 * sh.c + 4 * sh.d
            state = 2 * sh.B * sh.H * (sh.N + 1) * sh.c * sh.d * 4
            info.update({"io_bytes_per_token_head": per, "io_bytes": tokh * per + state})
        return flops, "TFLOP/s", "alu", info


def run_ours(args, rank, world, local_rank, sampler):
    import numpy as np
    import torch
    import torch.distributed as dist

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = Workload(args.workload, args.mode, args.batch)
    inp = wl.inputs(seed=shard_seed(rank))
    cpu = None
    if sampler is not None:
        nseq = min(sampler.cores, wl.shape.B * wl.shape.H)
        t_sample = args.cpu_tokens or wl.shape.T
        tok, wall = sampler.run(wl, inp, t_sample, nseq)
        tok1, secs1 = sampler.run_single(wl, inp, t_sample)
        cpu = {"value": tok / wall, "unit": "tokens/s", "cores": nseq, "kind": "oracle",
               "single_thread": {"value": tok1 / secs1, "unit": "tokens/s", "seconds": secs1},
               "cpu_model": cpu_model(), "host_cores": os.cpu_count(),
               "sample": f"{nseq} whole (b,h) sequences x first {t_sample} tokens of the same workload, fp64 "
                         f"oracle, one process per sequence ({wall:.1f} s wall); tokens = (b,h) token-steps / "
                         f"H={wl.shape.H}, the unit of the GPU value; single_thread = one sequence on one core"}
    run = GpuRun(wl, inp, device)
    run.overlap = args.overlap_addressing
    del inp
    stream = torch.cuda.current_stream()

    for _ in range(max(args.warmup, 3)):
        run.step()
    torch.cuda.synchronize()
    if int(run.err.item()) != 0:
        raise SystemExit(f"device error flag {int(run.err.item())} during warm-up")
    if wl.decode:
        run.enable_graphs()
    algo, algo_unit, bound, algo_info = run.algorithmic()

    clocks = ClockSampler(local_rank)
    clocks.start()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark(True)
    start.record(stream)
    run.run_steps(K, ev, stream)
    end.record(stream)
    torch.cuda.synchronize()
    clocks.mark(False)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = start.elapsed_time(end)
    main_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    total_ms = max_over_ranks(total_ms, world, device)
    ms_per_step = total_ms / K

    # end to end through the public API: pinned host inputs -> device -> the
    # same step -> y back to pinned host memory, every step
    KE = max(3, K // 2)
    for _ in range(2):
        run.e2e_step(args.e2e_chunk)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(KE):
        run.e2e_step(args.e2e_chunk)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / KE
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    h2d, d2h = run.io_bytes()

    pk, src = peaks()
    if bound == "hbm":
        peak = float(pk["hbm_gbs"])
        achieved = algo / (main_ms * 1e-3) / 1e9
    else:
        # FP32 FMA pipe: 152 SMs x 128 lanes x 2 flop x max SM clock
        peak = 152 * 128 * 2 * float(pk.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12
        achieved = algo / (main_ms * 1e-3) / 1e12
    kernel_file = {"sdm": "sparse_scan.cu", "gdn": "gdn_chunk.cu", "kda": "gdn_chunk.cu", "gdn2": "gdn_chunk.cu",
                   "sse": ("gdn_chunk.cu" if wl.sse_mode else "sse_chunk.cu") if wl.sse_chunked else "sse_scan.cu"}[wl.kind]
    tr = NCU_TRAFFIC.get((wl.name, wl.kind)) if not args.batch else None  # recorded at the configured sizes only
    traffic = tr["bytes"] if tr and tr["digest"] == _src_digest(kernel_file) else None
    tokens = wl.tokens * world
    cfg = wl.config()
    if world > 1:
        sl = rank_shard(wl.shape.B, world, rank)
        cfg["parallelism"] = (f"dp{world}: one global batch of {global_batch(wl.shape.B, world)} sequences per head, "
                              f"rank r runs batch elements [r*{wl.shape.B}, (r+1)*{wl.shape.B}) drawn with seed r "
                              f"(rank 0: {sl.start}..{sl.stop - 1}); no exchange on the data path")
    out = {
        "metric": metric_name(wl),
        "value": tokens / (ms_per_step * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": max(args.warmup, 3),
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded generators; no dataset or weights)",
        "config": cfg,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": algo_unit,
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "sdm_scan_train + sdm_scan_backward + 2 sdm_address_backward" if wl.train else
                     "sdm_scan_chunked (chunk preparation + chain kernels)" if wl.chunked else
                     {"sdm": "sdm_scan (hazard prepass + sparse_scan_kernel)",
                      "gdn": "gdn_scan (chunk preparation + chain kernels)",
                      "kda": "gdn_scan, per-channel decay (KDA chunk preparation + chain kernels)",
                      "gdn2": "gdn2_scan (GDN2 chunk preparation + chain kernels)",
                      "sse": ("sse_scan, delta write (route, group, KDA-form chunk preparation, chain, combine "
                              "kernels)" if wl.sse_mode else
                              "sse_scan (route, group, chunk preparation, chain, combine kernels)")
                      if wl.sse_chunked else "sse_scan (route prepass + sse_scan_kernel)"}[wl.kind],
                     "launch_ms": main_ms, "peak_source": f"{src} ({'hbm_gbs' if bound == 'hbm' else 'FP32 lanes x clock'})",
                     **algo_info},
        "cpu_baseline": cpu,
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "path": f"sdm_forward_host (copy/compute pipeline, {args.e2e_chunk}-token chunks)"
                if wl.kind == "sdm" and not wl.train and not wl.chunked
                else "pinned H2D copies + scan call + D2H of y"},
        "gpu_launches": K * run.launches_per_step,
        "step_launch": "CUDA graph replay of the step's kernels" if wl.decode else "stream launches",
        "clocks": clk,
    }
    if wl.kind == "sdm":
        out["step_breakdown_ms"] = {"addressing_x2": ms_per_step - main_ms, "scan": main_ms}
    if run.pipelined():
        out["schedule"] = ("the two addressing calls of step s+1 run on a second stream during the scan of "
                           "step s (every step does its full addressing and scan once)")
        out["step_breakdown_ms"] = {"scan": main_ms, "addressing_x2": "overlapped with the previous step's scan"}
    return out


def run_reference(args, rank, world):
    """The fp64 CPU oracle on this host's cores, on a bounded sample."""
    wl = Workload(args.workload, args.mode, args.batch)
    inp = wl.inputs(seed=0)
    cores = args.cpu_cores or min(os.cpu_count() or 1, 16)
    nseq = min(cores, wl.shape.B * wl.shape.H)
    t_sample = args.cpu_tokens or min(wl.shape.T, 1024 if wl.kind == "sdm" else 256)
    sampler = OracleSampler(nseq)
    for _ in range(max(args.warmup, 0)):
        sampler.run(wl, inp, t_sample, nseq)
    walls = []
    tok = 0
    for _ in range(args.steps):
        tok, wall = sampler.run(wl, inp, t_sample, nseq)
        walls.append(wall)
    tok1, secs1 = sampler.run_single(wl, inp, t_sample)
    sampler.close()
    ms = 1e3 * statistics.mean(walls)
    value = tok / (ms * 1e-3)
    sample = (f"{nseq} whole (b,h) sequences x first {t_sample} tokens per step, fp64 oracle, one process per "
              f"sequence; tokens = (b,h) token-steps / H={wl.shape.H}")
    return {"impl": "reference", "metric": metric_name(wl),
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generators; no dataset or weights)", "config": wl.config(),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nseq, "kind": "oracle", "sample": sample,
                             "single_thread": {"value": tok1 / secs1, "unit": "tokens/s", "seconds": secs1},
                             "cpu_model": cpu_model(), "host_cores": os.cpu_count()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sdm_14b_layer")
    ap.add_argument("--mode", choices=["shared", "perslot"], default="shared")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=0, help="tokens per sampled sequence for the oracle")
    ap.add_argument("--cpu-cores", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0, help="override B (small cases for profiling only)")
    ap.add_argument("--e2e-chunk", type=int, default=384,
                    help="tokens per pipelined chunk of the end-to-end sparse step (sdm_forward_host chunk_T)")
    ap.add_argument("--overlap-addressing", action="store_true",
                    help="sparse inference step: run step s+1's addressing on a second stream during step s's "
                         "scan (the scan's own time then includes the interference; on the 1.4B layer the "
                         "step is no faster than the serial one)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    # the oracle's process pool starts before any GPU work
    sampler = None
    if rank == 0 and not args.no_cpu_baseline:
        sampler = OracleSampler(args.cpu_cores or min(os.cpu_count() or 1, 16))
    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo", device_id=torch.device("cuda", local_rank)
                                if torch.cuda.is_available() else None)
    try:
        out = run_ours(args, rank, world, local_rank, sampler)
    finally:
        if sampler is not None:
            sampler.close()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
