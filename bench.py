"""Benchmark: attention TFLOP/s, forward and forward+backward, bf16 causal.

Workload: causal GQA, q [1, 8192, 32, 128], k/v [1, 8192, 8, 128] (group 4),
rotary embedding applied on the host, softmax_scale 1/sqrt(128) — the causal
bf16 L=8192 d=128 configuration the throughput target is quoted on. One step
is the whole hot path on one batch: the forward (O and the log-sum-exp) and
the backward recomputed from it (D/lse preprocess, the tcgen05 main kernel,
dQ convert). Algorithmic FLOPs: 4*n*h*l^2*d/2 forward, 2.5x that backward.

Besides the headline line it reports, in the same JSON line: the ring_merge
kernel standalone on [1, 16384, 16, 128] (fp32 accumulator, bf16 block; GB/s
of algorithmic bytes, L2 flushed), the ring replay of the 16k causal workload
(8 chunks), the end-to-end number through the public API with host buffers,
and the fp64 CPU oracle on a bounded sample of the same workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 it runs under torchrun, one independent replica per GPU (the path
does not shard): value = all replicas' FLOPs / max-over-ranks time.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s fwd & fwd+bwd (bf16, causal) and % of GB300 BF16 tensor peak"
WORKLOAD = "causal_gqa_8k_rope"
L2_FLUSH_BYTES = 256 << 20

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# each kernel on the workloads below, from one ncu capture of
# `bench.py --only {fwd,bwd,merge}` (profiles/), each with the hash of the
# kernel sources it was taken on. When the current sources hash differently the
# figure no longer describes the kernel, and the JSON line reports null.
NCU_TRAFFIC = {
    # kernel: (bytes per launch, source hash at capture)
    "bwd_bf16_kernel<128>": (354.9e6 + 144.5e6, "1f52ed6e8886"),   # causal GQA 8k, one launch
    "fwd_bf16_kernel<128>": (101.0e6 + 36.4e6, "eda1cfd6e9a0"),    # causal GQA 8k, one launch
    "ring_merge_kernel": (204.1e6 + 76.2e6, "531d70872b16"),       # [1,16384,16,128], L2 flushed before
    # the fused ring step of the 16k ring, step 1 (7 chunk pairs, 896 CTAs); same sources as the forward
    "fwd_bf16_kernel<128, merge>": (294.7e6 + 90.3e6, "eda1cfd6e9a0"),
}
# Algorithmic bytes of that fused step: q, k, v (bf16) of 7 chunks of [2048, 16, 128], the fp32
# accumulator read and written, the log-sum-exp read and written.
RING_STEP1_BYTES = 7 * 2048 * 16 * (3 * 128 * 2 + 2 * 128 * 4 + 2 * 4)
KERNEL_SOURCES = {
    "bwd_bf16_kernel<128>": ("bwd_sm103.cu", "ptx.cuh", "common.cuh"),
    "fwd_bf16_kernel<128>": ("fwd_sm103.cu", "ptx.cuh", "common.cuh"),
    "ring_merge_kernel": ("merge.cu", "common.cuh"),
    "fwd_bf16_kernel<128, merge>": ("fwd_sm103.cu", "ptx.cuh", "common.cuh"),
}


def kernel_source_hash(kernel: str) -> str:
    """sha256 (first 12 hex digits) of the source files a kernel is built from."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "blockwise_exact_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def ncu_traffic(kernel: str):
    """The captured DRAM bytes per launch, or None when the sources changed since."""
    nbytes, at = NCU_TRAFFIC[kernel]
    return nbytes if at is not None and at == kernel_source_hash(kernel) else None


def bench_config(world: int) -> dict:
    return {"workload": "causal GQA bf16 q[1,8192,32,128] k/v[1,8192,8,128], RoPE on host, scale 1/sqrt(128)",
            "global_batch": world, "seq_len": 8192, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (~300 MB per step) and a 256 MB read-based L2 flush before every timed step"}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), float(d["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 10 ms; the summary keeps the
    samples taken between mark_start() and mark_end() (the timed region)."""

    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"bea_clocks_{os.getpid()}.csv")
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "10"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        import datetime
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]),
                             {nm for nm, val in zip(names, parts[5:9]) if val.lower().startswith("active")}))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t1 is not None
                  and self.t0 - 0.02 <= r[0] <= self.t1 + 0.02]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0, "reasons": ["no samples"]}
        reasons = set().union(*(r[3] for r in use))
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": use[-1][2],
                "samples": len(use), "samples_in_timed_region": len(inside), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# FLOP counting (the throughput metric's definition; no attention arithmetic)
# ---------------------------------------------------------------------------

def visible_pairs(lq: int, lk: int, is_causal: bool, window=(-1, -1)) -> float:
    """Number of (query i, key j) pairs with key j visible to query i: j in
    [i - left, i + right] (an unbounded side is -1; causal forces right = 0),
    clipped to [0, lk)."""
    import numpy as np
    left, right = window
    if is_causal:
        right = 0
    i = np.arange(lq, dtype=np.int64)
    lo = np.zeros(lq, dtype=np.int64) if left < 0 else np.maximum(i - left, 0)
    hi = np.full(lq, lk - 1, dtype=np.int64) if right < 0 else np.minimum(i + right, lk - 1)
    return float(np.maximum(hi - lo + 1, 0).sum())


def attention_flops(n, h, lq, lk, d, is_causal, window=(-1, -1)):
    """(fwd, bwd) algorithmic FLOPs: 4 n h l^2 d forward, halved for causal
    (l^2 / 2 pairs), 2.5x that backward; a window counts its visible pairs."""
    left, right = window
    if left < 0 and (right < 0 and not is_causal):
        pairs = float(lq) * lk
    elif is_causal and left < 0:
        pairs = float(lq) * lk / 2.0
    else:
        pairs = visible_pairs(lq, lk, is_causal, window)
    f = 4.0 * n * h * d * pairs
    return f, 2.5 * f


# ---------------------------------------------------------------------------
# replicas: the slowest rank sets the pace
# ---------------------------------------------------------------------------

def max_over_ranks(values, dist=None, device=None):
    """Element-wise maximum over ranks of per-rank timings (identity with one
    rank or without an initialised process group)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return [float(x) for x in values]
    import torch
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_tflops(world: int, flops_per_rank: float, ms: float) -> float:
    """Whole-job throughput: the work of every replica over the slowest rank's time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------------------
# CPU oracle legs (the reference arm and the cpu_baseline field)
# ---------------------------------------------------------------------------

def oracle_sample_step(x, w, heads_kv):
    """fwd + bwd of the fp64 oracle on the query heads of `heads_kv`; returns FLOPs done."""
    import numpy as np
    import oracle
    g = w.h // w.h_kv
    hqs = [kv * g + t for kv in heads_kv for t in range(g)]
    q, k, v, do = x["q"][:, :, hqs], x["k"][:, :, heads_kv], x["v"][:, :, heads_kv], x["dout"][:, :, hqs]
    out, lse = oracle.attention_fwd(q, k, v, w.softmax_scale, w.is_causal, w.window)
    oracle.attention_bwd(do, q, k, v, out.astype(np.float32), lse, w.softmax_scale, w.is_causal, w.window)
    f, b = attention_flops(w.n, len(hqs), w.l, w.l, w.d, w.is_causal, w.window)
    return f + b


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from blockwise_exact_attention_gb300 import workloads
    w = workloads.WORKLOADS[WORKLOAD]
    x = workloads.make_inputs(w)
    for _ in range(max(0, args.warmup)):
        oracle_sample_step(x, w, [0])
    times, flops = [], 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        flops = oracle_sample_step(x, w, [0])
        times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    val = flops / sec / 1e12
    sample = (f"K/V head 0 of {w.h_kv} (query heads 0..{w.h // w.h_kv - 1}), all 8192 rows, fwd+bwd in fp64 numpy; "
              f"{flops:.3e} algorithmic FLOPs per step")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(args.gpus),
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_only(which, fwd, bwd, dev, workloads, bea):
    """A handful of launches of one kernel, nothing else timed (profiler runs)."""
    import torch
    if which == "fwd":
        for _ in range(4):
            fwd()
    elif which == "bwd":
        fwd()
        for _ in range(4):
            bwd()
    elif which == "bwd_d64":
        # the d=64 full-attention workload [1,32768,32,64] of the measurement plan
        wo = workloads.WORKLOADS["full_32k_d64"]
        qo = torch.randn((wo.n, wo.l, wo.h, wo.d), device=dev).to(torch.bfloat16)
        ko = torch.randn((wo.n, wo.l, wo.h_kv, wo.d), device=dev).to(torch.bfloat16)
        vo, doo = torch.randn_like(ko), torch.randn_like(qo)
        oo, lo_ = bea.flash_mha_fwd(qo, ko, vo, wo.softmax_scale, wo.is_causal, wo.window)
        for _ in range(4):
            bea.flash_mha_bwd(doo, qo, ko, vo, oo, lo_, wo.softmax_scale, wo.is_causal, wo.window)
    elif which in ("swa_fwd", "swa_bwd"):
        # the sliding-window workload (1024, 0) [1,32768,32,128] of the measurement plan
        wo = workloads.WORKLOADS["swa_32k_d128"]
        qo = torch.randn((wo.n, wo.l, wo.h, wo.d), device=dev).to(torch.bfloat16)
        ko = torch.randn((wo.n, wo.l, wo.h_kv, wo.d), device=dev).to(torch.bfloat16)
        vo, doo = torch.randn_like(ko), torch.randn_like(qo)
        oo, lo_ = bea.flash_mha_fwd(qo, ko, vo, wo.softmax_scale, wo.is_causal, wo.window)
        for _ in range(4):
            if which == "swa_fwd":
                bea.flash_mha_fwd(qo, ko, vo, wo.softmax_scale, wo.is_causal, wo.window)
            else:
                bea.flash_mha_bwd(doo, qo, ko, vo, oo, lo_, wo.softmax_scale, wo.is_causal, wo.window)
    elif which in ("ring", "ring_unfused", "ring_bwd"):
        # the 16k causal ring replay (8 chunks): two forward replays, or two backward replays
        wr = workloads.WORKLOADS["ring_causal_16k"]
        qr = torch.randn((1, wr.l, wr.h, wr.d), device=dev).to(torch.bfloat16)
        kr, vr, dor = torch.randn_like(qr), torch.randn_like(qr), torch.randn_like(qr)
        if which == "ring_bwd":
            o_r, l_r = bea.flash_mha_fwd(qr, kr, vr, wr.softmax_scale, True)
            for _ in range(2):
                bea.ring_attention_bwd(dor, qr, kr, vr, o_r, l_r, wr.ring_chunks, wr.softmax_scale, True)
        else:
            kw = {} if which == "ring" else {"block_dtype": torch.bfloat16, "fused": False}
            for _ in range(2):
                bea.ring_attention_fwd(qr, kr, vr, wr.ring_chunks, wr.softmax_scale, True, **kw)
    else:
        wr = workloads.WORKLOADS["ring_causal_16k"]
        acc = torch.randn((1, wr.l, wr.h, wr.d), device=dev)
        lacc = torch.randn((1, wr.h, wr.l), device=dev)
        blk = torch.randn((1, wr.l, wr.h, wr.d), device=dev).to(torch.bfloat16)
        lblk = torch.randn((1, wr.h, wr.l), device=dev)
        flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        for _ in range(4):
            flush.sum()   # as in the timed runs: every launch starts with L2 flushed
            bea.ring_merge(acc, lacc, blk, lblk)
    torch.cuda.synchronize()
    print(json.dumps({"only": which, "status": bea.device_status()}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["fwd", "bwd", "merge", "bwd_d64", "swa_fwd", "swa_bwd", "ring", "ring_unfused",
                                       "ring_bwd"],
                    help="run just this kernel a few times on the bench workload, bwd_d64 on the d=64 "
                         "full-attention workload, swa_* on the sliding-window workload, or two ring replays "
                         "of the 16k causal workload (for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    import __graft_entry__ as ge
    ge.build()
    import blockwise_exact_attention_gb300 as bea
    from blockwise_exact_attention_gb300 import workloads

    pk_burst, pk_sust, pk_hbm, pk_kind = peaks()
    w = workloads.WORKLOADS[WORKLOAD]
    x = workloads.make_inputs(w)
    dev = torch.device("cuda", local)
    q, k, v, do = (torch.from_numpy(x[s]).to(dev).to(torch.bfloat16) for s in ("q", "k", "v", "dout"))
    s = w.softmax_scale
    out = torch.empty_like(q)
    lse = torch.empty((w.n, w.h, w.l), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(bea.bwd_workspace_bytes(q), dtype=torch.uint8, device=dev)
    # L2 flush by READING a buffer twice the size of L2: it evicts every line
    # the step touched without leaving dirty lines behind whose write-back
    # would land inside the next timed region (a write-based flush does).
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        flush.sum()
    f_fwd, f_bwd = attention_flops(w.n, w.h, w.l, w.l, w.d, w.is_causal, w.window)
    stream = torch.cuda.current_stream()

    def fwd():
        bea.flash_mha_fwd(q, k, v, s, True, out=out, lse=lse)

    def bwd():
        bea.flash_mha_bwd(do, q, k, v, out, lse, s, True, dq=dq, dk=dk, dv=dv, workspace=ws)

    # The same backward as its three stages (exactly the kernels flash_mha_bwd
    # launches), with events between them so that the dominant kernel, the
    # backward main kernel, is timed on its own.
    def bwd_staged(ev):
        bea.flash_mha_bwd_prepare(do, out, lse, ws)
        ev[0].record(stream)
        bea.flash_mha_bwd_kv_block(do, q, k, v, dk, dv, s, True, workspace=ws)
        ev[1].record(stream)
        bea.flash_mha_bwd_finish(dq, s, workspace=ws)

    def timed(fn, reps, warm):
        for _ in range(warm):
            fn()
        ts = []
        for _ in range(reps):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return ts

    if args.only:
        return run_only(args.only, fwd, bwd, dev, workloads, bea)

    # ---- headline: K steps of fwd + bwd, each step timed between L2 flushes ----
    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    bea.launches_since_reset(reset=True)
    t_fwd, t_bwd, t_main = [], [], []
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        clk.mark_start()
        for _ in range(args.steps):
            flush_l2()
            e0, e1, e2, m0, m1 = (torch.cuda.Event(enable_timing=True) for _ in range(5))
            e0.record(stream)
            fwd()
            e1.record(stream)
            bwd_staged((m0, m1))
            e2.record(stream)
            e2.synchronize()
            t_fwd.append(e0.elapsed_time(e1))
            t_bwd.append(e1.elapsed_time(e2))
            t_main.append(m0.elapsed_time(m1))
        torch.cuda.synchronize()
        clk.mark_end()
    launches = bea.launches_since_reset(reset=True)
    status = bea.device_status()
    ms_fwd = sum(t_fwd) / len(t_fwd)
    ms_bwd = sum(t_bwd) / len(t_bwd)
    ms_main = sum(t_main) / len(t_main)
    ms_step = ms_fwd + ms_bwd
    ms_step, ms_fwd, ms_bwd, ms_main = max_over_ranks([ms_step, ms_fwd, ms_bwd, ms_main], dist, dev)
    value = job_tflops(world, f_fwd + f_bwd, ms_step)
    fwd_tf = f_fwd / (ms_fwd * 1e-3) / 1e12
    bwd_tf = f_bwd / (ms_bwd * 1e-3) / 1e12
    main_tf = f_bwd / (ms_main * 1e-3) / 1e12

    # ---- end to end through the public API with host buffers ----
    # Every step uploads its q, k, v, dout from pinned host memory and reads out, lse,
    # dq, dk, dv back, inside the timed region. Device buffers are double-buffered, so
    # step s+1's uploads (copy-in stream) run while step s computes and step s-1's
    # results come down (copy-out stream): the copies overlap compute instead of
    # adding to it. ms_per_step = the time of K back-to-back steps / K.
    hq_, hk_, hv_, hdo_ = (t.cpu().pin_memory() for t in (q, k, v, do))
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h_dq, h_dk, h_dv = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv))
    h2d = sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_, hdo_))
    d2h = sum(t.numel() * t.element_size() for t in (h_out, h_lse, h_dq, h_dk, h_dv))
    bufs = [dict(q=q, k=k, v=v, do=do, out=out, lse=lse, dq=dq, dk=dk, dv=dv, ws=ws)]
    bufs.append({key: torch.empty_like(t) for key, t in bufs[0].items()})
    up_stream = torch.cuda.Stream(device=dev)
    down_stream = torch.cuda.Stream(device=dev)

    def e2e_run(nsteps):
        """nsteps end-to-end steps, pipelined over the two buffer sets; returns ms per step."""
        free = [stream.record_event(), stream.record_event()]   # compute done with buffer set b
        drained = [stream.record_event(), stream.record_event()]  # results of buffer set b read back
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        up_stream.wait_stream(stream)
        down_stream.wait_stream(stream)
        for st in range(nsteps):
            bset = bufs[st % 2]
            with torch.cuda.stream(up_stream):
                up_stream.wait_event(free[st % 2])
                bset["q"].copy_(hq_, non_blocking=True)
                bset["k"].copy_(hk_, non_blocking=True)
                bset["v"].copy_(hv_, non_blocking=True)
                bset["do"].copy_(hdo_, non_blocking=True)
                uploaded = up_stream.record_event()
            stream.wait_event(uploaded)
            stream.wait_event(drained[st % 2])   # the previous results in this set have come down
            bea.flash_mha_fwd(bset["q"], bset["k"], bset["v"], s, True, out=bset["out"], lse=bset["lse"])
            fwd_done = stream.record_event()
            with torch.cuda.stream(down_stream):
                down_stream.wait_event(fwd_done)
                h_out.copy_(bset["out"], non_blocking=True)
                h_lse.copy_(bset["lse"], non_blocking=True)
            bea.flash_mha_bwd(bset["do"], bset["q"], bset["k"], bset["v"], bset["out"], bset["lse"], s, True,
                              dq=bset["dq"], dk=bset["dk"], dv=bset["dv"], workspace=bset["ws"])
            free[st % 2] = stream.record_event()
            with torch.cuda.stream(down_stream):
                down_stream.wait_event(free[st % 2])
                h_dq.copy_(bset["dq"], non_blocking=True)
                h_dk.copy_(bset["dk"], non_blocking=True)
                h_dv.copy_(bset["dv"], non_blocking=True)
                drained[st % 2] = down_stream.record_event()
        stream.wait_stream(up_stream)
        stream.wait_stream(down_stream)
        t1.record(stream)
        t1.synchronize()
        return t0.elapsed_time(t1) / nsteps

    e2e_run(3)
    e2e_ms = e2e_run(max(6, args.steps))
    e2e_ms, = max_over_ranks([e2e_ms], dist, dev)
    e2e_val = job_tflops(world, f_fwd + f_bwd, e2e_ms)
    del bufs[1]

    # ---- ring_merge standalone, [1, 16384, 16, 128], L2 flushed ----
    wr = workloads.WORKLOADS["ring_causal_16k"]
    acc = torch.randn((1, wr.l, wr.h, wr.d), device=dev)
    lacc = torch.randn((1, wr.h, wr.l), device=dev)
    blk = torch.randn((1, wr.l, wr.h, wr.d), device=dev).to(torch.bfloat16)
    lblk = torch.randn((1, wr.h, wr.l), device=dev)
    merge_ms = statistics.median(timed(lambda: bea.ring_merge(acc, lacc, blk, lblk), 20, 3))
    rows = wr.n * wr.l * wr.h
    merge_bytes = rows * (wr.d * (4 + 4 + 2) + 12)
    merge_gbs = merge_bytes / (merge_ms * 1e-3) / 1e9

    # ---- ring replay of the 16k causal workload, 8 chunks ----
    qr = torch.randn((1, wr.l, wr.h, wr.d), device=dev).to(torch.bfloat16)
    kr = torch.randn_like(qr)
    vr = torch.randn_like(qr)
    # the ring replay, its unfused form (each block written out in bf16, then ring_merge) and the
    # single call on the same problem, timed in turn within each repetition so that all three
    # see the same clocks
    ring_fns = (lambda: bea.ring_attention_fwd(qr, kr, vr, wr.ring_chunks, wr.softmax_scale, True),
                lambda: bea.ring_attention_fwd(qr, kr, vr, wr.ring_chunks, wr.softmax_scale, True,
                                               block_dtype=torch.bfloat16, fused=False),
                lambda: bea.flash_mha_fwd(qr, kr, vr, wr.softmax_scale, True))
    for fn in ring_fns:
        timed(fn, 0, 2)
    ring_ts = [[], [], []]
    for _ in range(9):
        for i, fn in enumerate(ring_fns):
            ring_ts[i] += timed(fn, 1, 0)
    ring_ms, ring_unfused_ms, single_ms = (statistics.median(t) for t in ring_ts)
    rf, rb = attention_flops(1, wr.h, wr.l, wr.l, wr.d, True)

    # host time to issue one ring replay (the calls return before the GPU is done): the library
    # call issuing all 8 steps, against the same replay composed from Python (forward + merge calls)
    def host_us(fn, n=20):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        t1 = time.perf_counter()
        torch.cuda.synchronize()
        return (t1 - t0) / n * 1e6
    ring_host_us = host_us(lambda: bea.ring_attention_fwd(qr, kr, vr, wr.ring_chunks, wr.softmax_scale, True))
    unfused_host_us = host_us(lambda: bea.ring_attention_fwd(qr, kr, vr, wr.ring_chunks, wr.softmax_scale, True,
                                                             block_dtype=torch.bfloat16, fused=False))
    # the ring backward: every live chunk pair once, from the single call's out/lse
    dor = torch.randn_like(qr)
    o_r, l_r = bea.flash_mha_fwd(qr, kr, vr, wr.softmax_scale, True)
    bea.launches_since_reset(reset=True)
    bea.ring_attention_bwd(dor, qr, kr, vr, o_r, l_r, wr.ring_chunks, wr.softmax_scale, True)
    ring_bwd_launches = bea.launches_since_reset(reset=True)
    wsr = torch.empty(bea.bwd_workspace_bytes(qr), dtype=torch.uint8, device=dev)
    gr = [torch.empty(t.shape, dtype=torch.float32, device=dev) for t in (qr, kr, vr)]
    bwd_fns = (lambda: bea.ring_attention_bwd(dor, qr, kr, vr, o_r, l_r, wr.ring_chunks, wr.softmax_scale, True),
               lambda: bea.flash_mha_bwd(dor, qr, kr, vr, o_r, l_r, wr.softmax_scale, True, dq=gr[0], dk=gr[1],
                                         dv=gr[2], workspace=wsr))
    for fn in bwd_fns:
        timed(fn, 0, 2)
    bwd_ts = [[], []]
    for _ in range(5):  # in turn, as for the forward
        for i, fn in enumerate(bwd_fns):
            bwd_ts[i] += timed(fn, 1, 0)
    ring_bwd_ms, single_bwd_ms = (statistics.median(t) for t in bwd_ts)
    del qr, kr, vr, acc, lacc, blk, lblk, dor, o_r, l_r, wsr, gr

    # ---- the other workloads of the measurement plan: forward and backward alone ----
    others = {}
    for name in ("causal_mha_4k", "swa_32k_d128", "full_32k_d64"):
        wo = workloads.WORKLOADS[name]
        qo = torch.randn((wo.n, wo.l, wo.h, wo.d), device=dev)
        if wo.head_scale:  # one factor U(0.5, 2) per query head, as the workload draws it
            qo *= (0.5 + 1.5 * torch.rand((1, 1, wo.h, 1), device=dev))
        qo = qo.to(torch.bfloat16)
        ko = torch.randn((wo.n, wo.l, wo.h_kv, wo.d), device=dev).to(torch.bfloat16)
        vo = torch.randn_like(ko)
        doo = torch.randn_like(qo)
        oo = torch.empty_like(qo)
        lo_ = torch.empty((wo.n, wo.h, wo.l), dtype=torch.float32, device=dev)
        dqo, dko, dvo = torch.empty_like(qo), torch.empty_like(ko), torch.empty_like(vo)
        wso = torch.empty(bea.bwd_workspace_bytes(qo), dtype=torch.uint8, device=dev)
        so = wo.softmax_scale
        fo, bo = attention_flops(wo.n, wo.h, wo.l, wo.l, wo.d, wo.is_causal, wo.window)
        tf = statistics.median(timed(lambda: bea.flash_mha_fwd(qo, ko, vo, so, wo.is_causal, wo.window, out=oo,
                                                                lse=lo_), 3, 1))
        tb = statistics.median(timed(lambda: bea.flash_mha_bwd(doo, qo, ko, vo, oo, lo_, so, wo.is_causal, wo.window,
                                                                dq=dqo, dk=dko, dv=dvo, workspace=wso), 3, 1))
        others[name] = {"workload": wo.description, "ms_fwd": tf, "ms_bwd": tb,
                        "fwd_tflops": fo / (tf * 1e-3) / 1e12, "bwd_tflops": bo / (tb * 1e-3) / 1e12,
                        "pct_peak_fwd": fo / (tf * 1e-3) / 1e12 / pk_burst,
                        "pct_peak_bwd": bo / (tb * 1e-3) / 1e12 / pk_burst}
        del qo, ko, vo, doo, oo, lo_, dqo, dko, dvo, wso

    # ---- CPU oracle on a bounded sample (rank 0, N = 1 only) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # three of the eight K/V heads: about 10 s of fp64 work on the host cores
        heads_kv = [0, 1, 2]
        t0 = time.perf_counter()
        fl = oracle_sample_step(x, w, heads_kv)
        sec = time.perf_counter() - t0
        g = w.h // w.h_kv
        cpu = {"value": fl / sec / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"fwd+bwd of K/V heads 0..{len(heads_kv) - 1} (query heads 0..{len(heads_kv) * g - 1}) "
                         f"of the same workload, all rows, fp64 numpy, {fl:.3e} FLOPs in {sec:.1f} s"}

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": bench_config(world),
        "fwd_tflops": fwd_tf,
        "bwd_tflops": bwd_tf,
        "ms_fwd": ms_fwd,
        "ms_bwd": ms_bwd,
        "pct_peak": {"fwd": fwd_tf / pk_burst, "bwd": bwd_tf / pk_burst, "fwd_bwd": value / world / pk_burst,
                     "peak_tflops": pk_burst, "peak_kind": f"{pk_kind} bf16 burst"},
        # dominant kernel: the backward main kernel (~71% of a step), timed alone with
        # events around its launch; algorithmic work = the backward's 2.5 x forward FLOPs
        "roofline": {"bound": "tensor", "kernel": "bwd_bf16_kernel<128>", "ms": ms_main,
                     "achieved": main_tf, "peak": pk_burst, "unit": "TFLOP/s", "frac": main_tf / pk_burst,
                     "traffic": ncu_traffic("bwd_bf16_kernel<128>"),
                     "source_hash": kernel_source_hash("bwd_bf16_kernel<128>"),
                     "peak_kind": f"{pk_kind} bf16 burst (a ~2 ms step, L2 flushed before it)"},
        "roofline_fwd": {"bound": "tensor", "kernel": "fwd_bf16_kernel<128>", "ms": ms_fwd, "achieved": fwd_tf,
                         "peak": pk_burst, "unit": "TFLOP/s", "frac": fwd_tf / pk_burst,
                         "traffic": ncu_traffic("fwd_bf16_kernel<128>"),
                         "source_hash": kernel_source_hash("fwd_bf16_kernel<128>")},
        "merge": {"kernel": "ring_merge [1,16384,16,128] f32 acc + bf16 blk", "ms": merge_ms,
                  "bytes": merge_bytes, "gbs": merge_gbs, "peak_gbs": pk_hbm, "frac": merge_gbs / pk_hbm,
                  "bound": "hbm", "traffic": ncu_traffic("ring_merge_kernel"),
                  "source_hash": kernel_source_hash("ring_merge_kernel")},
        "ring": {"workload": "causal bf16 [1,16384,16,128] as 8 chunks: the 36 chunk pairs in ring order, one "
                             "launch per ring step issued by one library call, 28 pairs as fused ring steps "
                             "(merge in the forward epilogue), steps chained by programmatic dependent launch; "
                             "8 launches", "ms": ring_ms,
                 "tflops": rf / (ring_ms * 1e-3) / 1e12, "single_call_ms": single_ms,
                 "unfused_ms": ring_unfused_ms, "unfused": "forward + ring_merge per ring step (bf16 blocks): 15 launches",
                 "host_us_per_call": ring_host_us, "unfused_host_us_per_call": unfused_host_us,
                 "step1_traffic": ncu_traffic("fwd_bf16_kernel<128, merge>"), "step1_algorithmic_bytes": RING_STEP1_BYTES,
                 "step1": "ncu DRAM bytes of ring step 1 (7 fused chunk pairs) against its algorithmic bytes"},
        "ring_bwd": {"workload": "causal bf16 [1,16384,16,128] as 8 chunks: the backward of every live chunk pair "
                                 "(36) once, fp32 dq/dk/dv accumulated over the pairs, from the final out/lse",
                     "ms": ring_bwd_ms, "tflops": rb / (ring_bwd_ms * 1e-3) / 1e12, "launches": ring_bwd_launches,
                     "single_call_ms": single_bwd_ms, "single_call_tflops": rb / (single_bwd_ms * 1e-3) / 1e12},
        "other_workloads": others,
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms,
                "how": "public API (flash_mha_fwd, flash_mha_bwd) on inputs uploaded from pinned host memory "
                       "every step, results read back every step; two device buffer sets, uploads and "
                       "read-backs on their own streams overlapping the neighbouring steps' compute; "
                       "time of back-to-back steps / steps"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "device_status": status,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
