#!/usr/bin/env python
"""Benchmark of the ZeRO-DP partitioned mixed-precision AdamW step on GB300.

Metric: ZeRO step params/s (and achieved HBM GB/s, % of 8 TB/s) for the GPT-2
1.5B layout (48 blocks, d = 1600, ffn 6400, vocab 50257, tied head; Psi =
1,557,611,200) with N_d = 8 simulated ranks, ZeRO-2, fp16 gradients under a
dynamic loss scale of 2^16 and global-norm clipping at 1.0.  One step = the
whole hot path over one batch of synthetic gradients resident in HBM:
4 bucketed reduce-scatters (bucket 5e8, last first) -> two-pass global norm and
step decision -> sharded AdamW with the all-gather fused in.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload gpt2_xl|gpt2_small|llama7b|gpt2_medium|tiny|gpt2_xl_block|llama7b_block]
                  [--graph] [--whole-buffer] [--micro M] [--sweep] [--prefetch] [--checkpoint DIR]

The e2e value repeats the step through the library's host-buffer entry point
(zero_step_from_host, one C-ABI call per step): the gradient replicas are
copied every step from pinned host memory, per bucket, overlapped with the
reduce-scatter, and the step state is copied back to host memory, after
untimed warm-up steps; it reports the host link's rate and the copies' time
beside it.

Under torchrun (N > 1) every rank runs its own independent replica of the
step on its own GPU (the simulated ranks live inside one GPU; there is no
data-path collective); a gloo barrier brackets the timed region and rank 0
prints the max-over-ranks time.  ``--impl reference`` times the CPU oracle on
the host cores instead (rank 0 only): exactly W untimed and K timed steps over
the whole workload, each step's wall time measured.  One JSON line is printed
by rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ZeRO step params/s and achieved HBM GB/s (% of 8 TB/s) at Ψ=1.5B, N_d=8"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["zero_rs.cu", "zero_adamw.cu", "zero_norm.cu", "zero_gather.cu", "zero_device.cuh",
                  "zero_accum.cu"]


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=60)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="gpt2_xl")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--cpu-blocks", type=int, default=0,
                   help="oracle timing on the workload's first N transformer blocks (0: the cpu_baseline "
                        "takes about 10-30 s of blocks; the reference arm takes the whole layout if it fits)")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--graph", action="store_true", help="replay each step from a CUDA graph")
    p.add_argument("--whole-buffer", action="store_true",
                   help="fused path: one launch over the whole buffer instead of one per bucket")
    p.add_argument("--timeline", default="",
                   help="write every traced call of the timed steps as a Chrome trace (JSON) to this path, "
                        "and add launch-gap and overlap figures to the line (eager steps only: calls replayed "
                        "from a CUDA graph are not traced)")
    p.add_argument("--sweep", action="store_true",
                   help="350M+1 layout: GB/s vs bucket size and N_d for stages 1/2/3 (one JSON line per point)")
    p.add_argument("--sweep-nd", default="2,4,8,16,64")
    p.add_argument("--live-units", type=int, default=2,
                   help="ZeRO-3: transient buffers per rank (2, the default: the executor gathers the next unit "
                        "while the previous one is reduced and updated; 1: one buffer, one stream)")
    p.add_argument("--micro", type=int, default=1,
                   help="micro-batches per optimizer step (gradient accumulation, split step)")
    p.add_argument("--prefetch", action="store_true",
                   help="ZeRO-3: gathers on a second stream under a stand-in per-unit GEMM (one JSON line)")
    p.add_argument("--comm-ctas", type=int, default=0, help="prefetch: CTA cap of the library's launches")
    p.add_argument("--compute-tokens", type=int, default=8192,
                   help="rows of the stand-in GEMM [tokens x d] x [d x d] per unit and pass")
    p.add_argument("--checkpoint", default="",
                   help="directory: time a sharded checkpoint save and a load resharded to N_d/2 (one JSON line)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# workload arithmetic
# ---------------------------------------------------------------------------

def bytes_per_param(w, fused: bool, n_micro: int = 1) -> float:
    """Algorithmic HBM bytes per parameter per optimizer step (16-bit = 2
    bytes).  With n_micro > 1 micro-batches (split step): ZeRO-1 accumulates
    each rank's full gradient in fp32 (first 6 N_d, then 10 N_d per micro-batch)
    and reduce-scatters the accumulators once (4 N_d + 4); ZeRO-2/3 reduce every
    micro-batch into the fp32 shard (2 N_d + 4 first, 2 N_d + 8 after); ZeRO-3
    gathers forward and backward every micro-batch."""
    nd = w.n_d
    M = n_micro
    if M > 1:
        adamw = 28 + (2 if w.stage == 3 else 2 * nd)
        if w.stage == 1:
            return 6 * nd + 10 * nd * (M - 1) + 4 * nd + 4 + adamw
        rs = 2 * nd * M + 4 + 8 * (M - 1)
        gathers = 2 * (2 + 2 * nd) * M if w.stage == 3 else 0
        return rs + gathers + adamw
    if w.stage == 3:
        if fused:
            return 2 * (2 + 2 * nd) + 2 * nd + 24 + 2        # 2 gathers + RS + AdamW + shard write
        return 2 * (2 + 2 * nd) + 2 * nd + 4 + 4 + 24 + 2
    if fused:
        return 4 * nd + 24
    return 4 * nd + 24 + min(2 * nd, 8)


def kernel_bytes(name: str, w, elems: float, n_micro: int = 1) -> float:
    """Algorithmic bytes of one launch of ``name`` over ``elems`` elements
    (16-bit = 2 bytes).  Under micro-batching the reduce-scatter and the
    ZeRO-1 accumulation average their first and later modes."""
    nd, M = w.n_d, n_micro
    rs = 2 * nd + 4
    acc = 10 * nd
    if M > 1:
        rs = 4 * nd + 4 if w.stage == 1 else 2 * nd + 4 + 4 * (M - 1) / M   # later ones also read the fp32 shard
        acc = (6 * nd + 10 * nd * (M - 1)) / M
    per = {"reduce_scatter": rs, "accumulate": acc,
           "adamw": 4 + 24 + (2 * nd if w.stage != 3 else 2),
           "fused_step": 2 * nd + 24 + (2 * nd if w.stage != 3 else 2), "stage3_gather": 2 + 2 * nd,
           "allgather": 2 + 2 * nd, "grad_norm": 4 / 32}[name]
    return per * elems


def elems_per_launch(name: str, w, psi_pad: int, launches_per_step: float, n_micro: int = 1) -> float:
    """Elements one launch of ``name`` processes, on average over a step."""
    M = n_micro
    if name == "reduce_scatter":        # every micro-batch reduces the whole buffer (ZeRO-2/3)
        return psi_pad * (M if w.stage != 1 else 1) / max(1.0, launches_per_step)
    if name == "fused_step":
        return psi_pad / max(1.0, launches_per_step)
    if name == "stage3_gather":         # real elements, forward and backward, every micro-batch
        return 2 * w.psi * M / max(1.0, launches_per_step)
    return psi_pad                      # adamw, accumulate, allgather, grad_norm: the whole buffer


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for n in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "zero_partitioned_mixed_replica_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of ``kernel`` from the committed ncu summary, if
    it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        e = rec[workload][kernel]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


def host_mem_available():
    """MemAvailable of this host in bytes (Linux /proc/meminfo), or None."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def e2e_fits(need_bytes: int, local_world: int, avail) -> bool:
    """Whether every local rank can pin its own copy of the step's gradients
    while keeping at least half of the host's available memory free."""
    return avail is None or need_bytes * local_world <= avail // 2


def host_link_gbs(host: torch.Tensor, dev_buf: torch.Tensor, stream) -> float:
    """Host-to-device rate of this box's link, measured just before the e2e
    leg: the better of two pinned copies of the whole gradient buffer into
    its device twin (whose contents the e2e steps overwrite anyway).  The
    link is shared with other tenants of the host, so it is taken at the
    size and moment of the e2e leg."""
    import torch
    src, dst = host.view(-1), dev_buf.view(-1)
    best = float("inf")
    with torch.cuda.stream(stream):
        for _ in range(2):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dst.copy_(src, non_blocking=True)
            b.record(stream)
            b.synchronize()
            best = min(best, a.elapsed_time(b))
    return src.numel() * host.element_size() / (best / 1e3) / 1e9


def max_over_ranks(value: float, world: int) -> float:
    """The slowest rank's time (gloo all-reduce MAX on the host); the value
    itself on a single rank."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        cmd = ["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits", "-lms", "200"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.p = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except Exception:
            self.p.kill()
            out = ""
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(w, blocks):
    """The tensors of the workload that the oracle is timed on: all of them
    (``blocks`` None), or those of its first ``blocks`` transformer blocks
    (ZeRO-3 units 1..blocks), each with its own per-tensor scale.  Returns
    (numels, unit ids, scales, description)."""
    from zero_partitioned_mixed_replica_gb300 import synth
    scales_all = synth.tensor_scales(len(w.numels)) if w.per_tensor_scale else None
    n_blocks = max(w.unit_of_tensor)
    if blocks is None or blocks >= n_blocks:
        return (list(w.numels), list(w.unit_of_tensor), scales_all,
                "the whole layout: %d tensors, Psi = %d" % (len(w.numels), w.psi))
    keep = [t for t, u in enumerate(w.unit_of_tensor) if 1 <= u <= blocks]
    numels = [w.numels[t] for t in keep]
    units = [w.unit_of_tensor[t] - 1 for t in keep]
    scales = [scales_all[t] for t in keep] if scales_all is not None else None
    return (numels, units, scales,
            "the first %d of %d transformer blocks (%d tensors, %d parameters, %.2f%% of Psi)"
            % (blocks, n_blocks, len(numels), sum(numels), 100.0 * sum(numels) / w.psi))


def oracle_bytes(w, psi: int) -> int:
    """Host bytes the oracle's ZeRO simulation holds for ``psi`` parameters:
    the N_d 16-bit gradient replicas, fp32 master/m/v/reduced shards, the
    16-bit parameters (full replicas for ZeRO-1/2) and the initial master."""
    p16 = 2 * w.n_d if w.stage != 3 else 2
    return int(psi * (2 * w.n_d + 16 + p16 + 4) * 1.1)


def oracle_blocks_that_fit(w, avail) -> object:
    """None (the whole layout) if its oracle state takes at most 60% of the
    host's available memory, else the most leading blocks that do."""
    if avail is None or oracle_bytes(w, w.psi) <= 0.6 * avail:
        return None
    per_block = max(1, sum(n for n, u in zip(w.numels, w.unit_of_tensor) if u == 1))
    return max(1, int(0.6 * avail // oracle_bytes(w, per_block)))


def oracle_timing(w, blocks, min_seconds: float, min_steps: int = 3, max_steps: int = 10 ** 6, warmup: int = 1):
    """The oracle (its literal ZeRO simulation, as it stands) on the
    workload's tensors (see :func:`oracle_sample`) with the workload's
    settings: N_d, stage, bucket size, 16-bit format, per-tensor scales, loss
    scale, clipping.  ``warmup`` untimed steps, then at least ``min_steps``
    timed steps and at least ``min_seconds`` of them (at most ``max_steps``).
    Each step's wall time is measured; nothing is extrapolated."""
    from oracle.layout import make_layout
    from oracle.step import AdamWHP, ZeroSimulation, num_threads
    from zero_partitioned_mixed_replica_gb300 import synth

    numels, units, scales, desc = oracle_sample(w, blocks)
    L = make_layout(numels, w.n_d, w.stage, bucket_elems=w.bucket_elems if w.stage != 3 else 0,
                    unit_of_tensor=units if w.stage == 3 else None)
    m0 = synth.master_init(numels, L.tensor_offsets, L.psi_pad, w.master_std).numpy()
    reps = [synth.as_u16(synth.grad_replica(numels, L.tensor_offsets, L.psi_pad, w.dtype, r, 1, w.grad_std,
                                            scales, w.loss_scale)) for r in range(w.n_d)]
    zs = ZeroSimulation(L, m0, w.dtype, AdamWHP(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay),
                        max_norm=w.max_norm, loss_scale=w.loss_scale, dynamic=w.dynamic_scale,
                        growth_interval=w.growth_interval)
    del m0
    for _ in range(warmup):                         # untimed warm-up steps
        zs.step(reps)
    times = []
    t0 = time.perf_counter()
    while len(times) < max_steps and (len(times) < min_steps or time.perf_counter() - t0 < min_seconds):
        a = time.perf_counter()
        zs.step(reps)
        times.append(time.perf_counter() - a)
    dt = sum(times) / len(times)
    psi = sum(numels)
    return {"value": psi / dt, "unit": "params/s", "cores": num_threads(), "kind": "oracle",
            "sample": "%s; N_d=%d, stage %d, %s grads, %d untimed + %d timed steps of %.3f s (measured, mean)"
                      % (desc, w.n_d, w.stage, "fp16" if w.dtype == 1 else "bf16", warmup, len(times), dt),
            "s_per_step": dt, "steps": len(times), "psi": psi}


def default_cpu_blocks(w) -> int:
    """Leading blocks for the repo arm's cpu_baseline: about 10-30 s of CPU
    work on the machine's cores (a GPT-2 1.5B block is 30.7M parameters)."""
    per_block = sum(n for n, u in zip(w.numels, w.unit_of_tensor) if u == 1)
    return max(1, min(max(w.unit_of_tensor), int(120_000_000 // max(1, per_block))))


# ---------------------------------------------------------------------------
# GPU run
# ---------------------------------------------------------------------------

def timeline_summary(records) -> dict:
    """Launch gaps and overlap of a traced timeline (one device): the span
    from the first start to the last end, the time with at least one call in
    flight (busy), the idle gaps between calls, and how many calls started
    before the previous one (in start order) had ended."""
    recs = sorted(records, key=lambda r: r["start_ms"])
    if not recs:
        return {"records": 0}
    span = recs[-1]["end_ms"] - recs[0]["start_ms"]
    busy, lo, hi, gaps, overlapped = 0.0, recs[0]["start_ms"], recs[0]["end_ms"], [], 0
    for r in recs[1:]:
        if r["start_ms"] < hi:
            overlapped += 1
        if r["start_ms"] > hi:
            busy += hi - lo
            gaps.append(r["start_ms"] - hi)
            lo, hi = r["start_ms"], r["end_ms"]
        else:
            hi = max(hi, r["end_ms"])
    busy += hi - lo
    return {"records": len(recs), "streams": len({r["stream"] for r in recs}), "span_ms": span, "busy_ms": busy,
            "idle_frac": 1.0 - busy / span if span > 0 else 0.0, "gaps": len(gaps),
            "mean_gap_us": 1e3 * sum(gaps) / len(gaps) if gaps else 0.0,
            "max_gap_us": 1e3 * max(gaps) if gaps else 0.0, "overlapped_starts": overlapped}


def write_timeline(records, path: str) -> dict:
    """Chrome trace (chrome://tracing, Perfetto) of the traced calls: one
    row per stream; returns the summary with the file's path."""
    streams = {}
    events = []
    for r in records:
        tid = streams.setdefault((r["device"], r["stream"]), len(streams))
        events.append({"name": r["kind"], "ph": "X", "pid": r["device"], "tid": tid,
                       "ts": 1e3 * r["start_ms"], "dur": 1e3 * (r["end_ms"] - r["start_ms"])})
    with open(path, "w") as f:
        json.dump({"traceEvents": events, "displayTimeUnit": "ms"}, f)
    return dict(timeline_summary(records), file=path)


def gpu_run(args, w, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from zero_partitioned_mixed_replica_gb300 import binding as B
    from zero_partitioned_mixed_replica_gb300 import build as zbuild
    from zero_partitioned_mixed_replica_gb300 import synth
    from zero_partitioned_mixed_replica_gb300.engine import AdamW, ZeroStep

    zbuild.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    units = w.unit_of_tensor if w.stage == 3 else None
    eng = ZeroStep(w.numels, w.n_d, w.stage, w.dtype, w.bucket_elems if w.stage != 3 else 0, units,
                   AdamW(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay), w.max_norm, w.loss_scale,
                   w.dynamic_scale, w.growth_interval, per_bucket=not args.whole_buffer, n_micro=args.micro,
                   device=str(dev), live_units=args.live_units)
    info = eng.info
    m0 = synth.master_init(w.numels, eng.tensor_offsets, info.psi_pad, w.master_std, device=dev)
    eng.load_master(m0)
    del m0
    scales = synth.tensor_scales(len(w.numels)) if w.per_tensor_scale else None
    for r in range(w.n_d):
        synth.grad_replica(w.numels, eng.tensor_offsets, info.psi_pad, w.dtype, r, 1, w.grad_std, scales,
                           w.loss_scale, device=dev, out=eng.grads[r])
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    graph = eng.capture() if args.graph else None
    if args.micro > 1:
        def run():
            for mb in range(args.micro):
                eng.micro_step(mb)
    else:
        run = (lambda: graph.replay()) if graph is not None else eng.step
    # the warm-up steps run traced too, so that the timed steps reuse the trace's events
    # instead of creating them inside the timed region
    trace = graph is None
    B.zero_trace_enable(trace)
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize(dev)
    B.zero_trace_enable(False)
    B.zero_trace_read(reset=True)
    # --- timed region -----------------------------------------------------------
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    time.sleep(0.3)
    # per-call durations from CUDA events on each call's launching stream: the library's
    # launch tracing of the step executor (zero_step, zero_micro_step)
    if trace:
        B.zero_trace_enable(True)
    B.zero_launch_count(reset=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    launches = B.zero_launch_count()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    traced = None
    timeline = None
    if trace:
        B.zero_trace_enable(False)
        if args.timeline and rank == 0:
            timeline = write_timeline(B.zero_trace_timeline(), args.timeline)
        traced = B.zero_trace_read(reset=True)
    ms = max_over_ranks(ms, world)
    if graph is not None:
        # launches inside a replayed graph are the captured ones
        B.zero_launch_count(reset=True)
        eng.step()
        torch.cuda.synchronize(dev)
        launches = B.zero_launch_count() * args.steps
    st = eng.read_state()

    # --- per-kernel averages from events on the launching stream ------------------
    kern = traced or {}
    # --- e2e: host buffers, H2D of the step's gradients + D2H of the step result ----
    e2e = None
    need = int(eng.grads.numel() * eng.grads.element_size())
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    avail = host_mem_available()
    if args.e2e_steps > 0 and not e2e_fits(need, local_world, avail):
        # every local rank pins its own copy of the step's gradients; more than half of the
        # host's available memory in pinned pages would put the host at risk
        e2e = {"value": None, "unit": "params/s",
               "skipped": "host memory: %d ranks x %.1f GB pinned > half of %.1f GB available"
                          % (local_world, need / 1e9, avail / 1e9)}
    elif args.e2e_steps > 0:
        try:
            host_grads = torch.empty(tuple(eng.grads.shape), dtype=eng.grads.dtype, pin_memory=True)
            host_grads.copy_(eng.grads)
            host_state = torch.empty(96, dtype=torch.uint8).pin_memory()
            link_gbs = host_link_gbs(host_grads, eng.grads, stream)

            def e2e_step():
                if args.micro == 1:
                    # one C-ABI call (zero_step_from_host): the per-bucket host-to-device copies
                    # overlap the reduce-scatter and, from the second step on, the previous step's
                    # norm and update; the step state is copied back to host_state
                    eng.step_from_host(host_grads, state_out=host_state, overlap_previous=True)
                else:
                    for mb in range(args.micro):
                        eng.upload_grads(host_grads)
                        eng.micro_step(mb)
                    host_state.copy_(eng.state, non_blocking=True)

            # the copies alone (same chunks on the same two streams), to read the e2e value against
            copy_ms = []
            for _ in range(2):
                c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                c0.record(stream)
                eng.upload_grads(host_grads)
                c1.record(stream)
                c1.synchronize()
                copy_ms.append(c0.elapsed_time(c1))
            # Untimed warm-up, as for the device-resident steps: the first
            # whole-buffer passes over a freshly pinned buffer cross the host
            # link at 90-140 GB/s before settling at the link rate.  After it,
            # every step's copies overlap the previous step's update.
            for _ in range(max(3, args.warmup)):
                e2e_step()
            torch.cuda.synchronize(dev)
            if world > 1:
                dist.barrier()
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.e2e_steps + 1)]
            evs[0].record(stream)
            for i in range(args.e2e_steps):
                e2e_step()
                evs[i + 1].record(stream)
            torch.cuda.synchronize(dev)
            a, b = evs[0], evs[-1]
            ems = max_over_ranks(a.elapsed_time(b), world)
            e2e = {"value": world * w.psi * args.e2e_steps / (ems / 1e3), "unit": "params/s",
                   "h2d_bytes_per_step": int(eng.grads.numel() * eng.grads.element_size()) * args.micro,
                   "d2h_bytes_per_step": 96, "ms_per_step": ems / args.e2e_steps,
                   "warmup_steps": max(3, args.warmup), "host_link_gbs": link_gbs,
                   "overlap_previous": args.micro == 1,
                   "h2d_floor_ms": int(eng.grads.numel() * eng.grads.element_size()) * args.micro / link_gbs / 1e6,
                   "copy_only_ms": min(copy_ms),
                   "ms_each": [round(evs[i].elapsed_time(evs[i + 1]), 2) for i in range(args.e2e_steps)]}
            del host_grads
        except RuntimeError as ex:
            e2e = {"value": None, "unit": "params/s", "error": str(ex)[:200]}
    return eng, info, ms, kern, launches, clk, st, e2e, timeline


def sweep(args):
    """GB/s vs bucket size and N_d on the GPT-2 medium 350M + 1 layout (odd
    Psi), fused step (no clipping, no scaler), stages 1/2 per bucket and
    stage 3 per unit.  Rank 0's gradients are drawn by the input generator and
    copied to the other ranks (values do not change the traffic)."""
    import torch
    from zero_partitioned_mixed_replica_gb300 import binding as B
    from zero_partitioned_mixed_replica_gb300 import build as zbuild
    from zero_partitioned_mixed_replica_gb300 import synth, workloads
    from zero_partitioned_mixed_replica_gb300.engine import ZeroStep
    zbuild.build()
    dev = torch.device("cuda", 0)
    buckets = [100_000, 500_000, 1_000_000, 5_000_000, 10_000_000, 50_000_000]
    for nd in [int(x) for x in args.sweep_nd.split(",")]:
        for stage in (1, 2, 3):
            w = workloads.gpt2_medium_odd(n_d=nd, stage=stage, bucket_elems=buckets[0])
            eng = ZeroStep(w.numels, nd, stage, w.dtype, buckets[0] if stage != 3 else 0,
                           w.unit_of_tensor if stage == 3 else None, device=str(dev), live_units=args.live_units)
            eng.load_master(synth.master_init(w.numels, eng.tensor_offsets, eng.info.psi_pad, device=dev))
            synth.grad_replica(w.numels, eng.tensor_offsets, eng.info.psi_pad, w.dtype, 0, 1, w.grad_std,
                               synth.tensor_scales(len(w.numels)), device=dev, out=eng.grads[0])
            for r in range(1, nd):
                eng.grads[r].copy_(eng.grads[0])
            bpp = bytes_per_param(w, True)
            for b in (buckets if stage != 3 else [0]):
                if stage != 3:
                    eng.set_bucket_elems(b)
                for _ in range(2):
                    eng.step()
                torch.cuda.synchronize(dev)
                B.zero_launch_count(reset=True)
                for _ in range(args.steps):   # launch count of eager steps
                    eng.step()
                torch.cuda.synchronize(dev)
                launches = B.zero_launch_count() // args.steps
                graph = eng.capture() if args.graph else None
                run = graph.replay if graph is not None else eng.step
                run()
                torch.cuda.synchronize(dev)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(args.steps):
                    run()
                e1.record()
                torch.cuda.synchronize(dev)
                ms = e0.elapsed_time(e1) / args.steps
                del graph
                print(json.dumps({"sweep": "gpt2_medium_350M+1", "n_d": nd, "stage": stage,
                                  "bucket_elems": b if stage != 3 else "per unit",
                                  "n_buckets": eng.n_buckets if stage != 3 else len(eng.units),
                                  "ms_per_step": ms, "params_per_s": w.psi / (ms / 1e3),
                                  "hbm_gbs": bpp * eng.info.psi_pad / (ms / 1e3) / 1e9,
                                  "bytes_per_param": bpp, "graph": bool(args.graph),
                                  "live_units": args.live_units if stage == 3 else None,
                                  "launches_per_step": launches}), flush=True)
            del eng
            torch.cuda.empty_cache()


def checkpoint_bench(args):
    """Sharded checkpoint of the chosen workload: every simulated rank writes
    its shard in parallel; then a layout with half the ranks (ZeRO-2) loads it
    through the reshard plan."""
    import shutil
    import torch
    from zero_partitioned_mixed_replica_gb300 import build as zbuild
    from zero_partitioned_mixed_replica_gb300 import synth, workloads
    from zero_partitioned_mixed_replica_gb300.engine import ZeroStep
    zbuild.build()
    w = workloads.ALL[args.workload]()
    units = w.unit_of_tensor if w.stage == 3 else None
    a = ZeroStep(w.numels, w.n_d, w.stage, w.dtype, w.bucket_elems if w.stage != 3 else 0, units)
    a.load_master(synth.master_init(w.numels, a.tensor_offsets, a.info.psi_pad, device=a.device))
    path = os.path.join(args.checkpoint, "ckpt")
    shutil.rmtree(path, ignore_errors=True)
    t0 = time.perf_counter()
    out = a.save_checkpoint(path)
    t_save = time.perf_counter() - t0
    nd2 = max(1, w.n_d // 2)
    del a
    torch.cuda.empty_cache()
    b = ZeroStep(w.numels, nd2, 2, w.dtype, w.bucket_elems if w.bucket_elems > 0 else 0, None)
    t0 = time.perf_counter()
    info = b.load_checkpoint(path)
    t_load = time.perf_counter() - t0
    shutil.rmtree(path, ignore_errors=True)
    print(json.dumps({"checkpoint": w.name, "bytes": out["bytes"], "save_s": t_save, "load_s": t_load,
                      "save_gbs": out["bytes"] / t_save / 1e9, "load_gbs": info["bytes"] / t_load / 1e9,
                      "reshard": "N_d %d stage %d -> N_d %d stage 2" % (w.n_d, w.stage, nd2),
                      "segments": info["segments"]}), flush=True)


def prefetch_bench(args):
    """ZeRO-3 forward/backward prefetch: each unit's forward and backward is
    stood in for by one bf16 GEMM [tokens x d] x [d x d] on the compute stream
    (d = the model width, the weight being the first d x d block of the
    gathered unit); the unit gathers (and, in backward, the unit's
    reduce-scatter + update) run on a second stream.  Reports the step time
    with 1 live unit (no prefetch) and 2 (prefetch), the compute-only and
    communication-only times, and the fraction of the smaller one hidden."""
    import torch
    from zero_partitioned_mixed_replica_gb300 import build as zbuild
    from zero_partitioned_mixed_replica_gb300 import synth, workloads
    from zero_partitioned_mixed_replica_gb300.engine import ZeroStep
    zbuild.build()
    w = workloads.ALL[args.workload]()
    assert w.stage == 3, "prefetch needs a ZeRO-3 workload"
    dev = torch.device("cuda", 0)
    eng = ZeroStep(w.numels, w.n_d, 3, w.dtype, 0, w.unit_of_tensor, device=str(dev))
    eng.load_master(synth.master_init(w.numels, eng.tensor_offsets, eng.info.psi_pad, device=dev))
    synth.grad_replica(w.numels, eng.tensor_offsets, eng.info.psi_pad, w.dtype, 0, 1, w.grad_std,
                       device=dev, out=eng.grads[0])
    for r in range(1, w.n_d):
        eng.grads[r].copy_(eng.grads[0])
    d = 4096 if w.numels[0] % 4096 == 0 else 1600   # model width of the Llama / GPT-2 1.5B layouts
    x = torch.randn(args.compute_tokens, d, device=dev, dtype=torch.bfloat16)
    y = torch.empty(args.compute_tokens, d, device=dev, dtype=torch.bfloat16)

    def compute(kind, u, rows):
        wgt = rows[0][:d * d].view(d, d)
        torch.matmul(x, wgt, out=y)

    def timed(fn, reps):
        for _ in range(2):
            fn()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / reps

    U = len(eng.units)
    reps = max(1, args.steps)
    t_seq = timed(lambda: eng.step_overlapped(compute, 1), reps)
    t_ovl = timed(lambda: eng.step_overlapped(compute, 2, args.comm_ctas), reps)
    t_comp = timed(lambda: [compute("fwd", u, [eng.transient[r] for r in range(w.n_d)]) for u in range(2 * U)],
                   reps)
    t_comm = timed(eng.step, reps)
    hidden = (t_seq - t_ovl) / min(t_comp, t_comm)
    print(json.dumps({"prefetch": w.name, "units": U, "compute_tokens": args.compute_tokens, "gemm_d": d,
                      "comm_ctas": args.comm_ctas,
                      "ms_no_prefetch": t_seq, "ms_prefetch": t_ovl, "ms_compute_only": t_comp,
                      "ms_comm_only": t_comm, "hidden_fraction": hidden,
                      "t_compute_ge_t_comm": t_comp >= t_comm}), flush=True)


def main():
    args = parse()
    if args.prefetch:
        prefetch_bench(args)
        return
    if args.sweep:
        sweep(args)
        return
    if args.checkpoint:
        checkpoint_bench(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    from zero_partitioned_mixed_replica_gb300 import workloads
    w = workloads.ALL[args.workload]()
    fused = w.fused() and args.micro == 1
    bpp = bytes_per_param(w, fused, args.micro)
    workload_desc = {"workload": w.name, "psi": w.psi, "n_d": w.n_d, "stage": w.stage,
                     "grad_dtype": "fp16" if w.dtype == 1 else "bf16", "state_dtype": "fp32",
                     "bucket_elems": w.bucket_elems, "max_norm": w.max_norm, "loss_scale": w.loss_scale,
                     "algorithmic_bytes_per_param": bpp, "micro_batches": args.micro,
                     "live_units": args.live_units if w.stage == 3 else None,
                     "l2": "no flush: the step streams > 60 GB per pass, far above the 129 MB L2"}

    if args.impl == "reference":
        if rank != 0:
            return
        # the oracle on the host cores, exactly W untimed and K timed steps over the whole
        # workload (or, where its state would not fit the host's memory, named leading blocks)
        blocks = args.cpu_blocks if args.cpu_blocks > 0 else oracle_blocks_that_fit(w, host_mem_available())
        cb = oracle_timing(w, blocks, min_seconds=0.0, min_steps=max(1, args.steps), max_steps=max(1, args.steps),
                           warmup=max(0, args.warmup))
        line = {"metric": METRIC, "value": cb["value"], "unit": "params/s", "impl": "reference",
                "n_gpus": args.gpus, "steps": cb["steps"], "warmup": max(0, args.warmup),
                "ms_per_step": cb["s_per_step"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic", "config": workload_desc,
                "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
                "e2e": {"value": cb["value"], "unit": "params/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        if cb["psi"] != w.psi:
            line["config"] = dict(workload_desc, sample=cb["sample"].split(";")[0], sample_psi=cb["psi"])
        print(json.dumps(line), flush=True)
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo", rank=rank, world_size=world)
    eng, info, ms, kern, launches, clk, st, e2e, timeline = gpu_run(args, w, rank, world, local_rank)
    step_s = ms / 1e3 / args.steps
    value = world * w.psi / step_s
    step_gbs = bpp * info.psi_pad / step_s / 1e9
    peak, peak_kind = measured_peak()
    roof = None
    if kern:
        for name, k in kern.items():       # achieved GB/s of every kernel, algorithmic bytes
            e = elems_per_launch(name, w, info.psi_pad, k["launches"] / args.steps, args.micro)
            k["gbs"] = kernel_bytes(name, w, e, args.micro) / (k["avg_ms"] / 1e3) / 1e9
        dom = max(kern, key=lambda k: kern[k]["total_ms"])
        elems = elems_per_launch(dom, w, info.psi_pad, kern[dom]["launches"] / args.steps, args.micro)
        ach = kernel_bytes(dom, w, elems, args.micro) / (kern[dom]["avg_ms"] / 1e3) / 1e9
        overlap = any(k["total_ms"] > k["busy_ms"] * 1.001 for k in kern.values() if "busy_ms" in k) or \
            (w.stage == 3 and args.live_units >= 2)
        roof = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": peak, "unit": "GB/s",
                "frac": ach / peak, "peak_kind": peak_kind + " (copy bandwidth)",
                "traffic": ncu_traffic(dom, args.workload),
                "algorithmic_bytes_per_launch": kernel_bytes(dom, w, elems, args.micro),
                "avg_launch_ms": kern[dom]["avg_ms"]}
        if overlap:
            roof["note"] = ("launches of the step overlap (alternating streams): a launch's duration includes "
                            "time it shares with others, so per-kernel rates understate the kernels; the step's "
                            "own rate is hbm_gbs")
        if roof["traffic"] is not None:        # the same launch time over the ncu DRAM bytes
            roof["achieved_by_ncu_bytes"] = roof["traffic"] / (kern[dom]["avg_ms"] / 1e3) / 1e9
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:   # the oracle baseline: rank 0 at N = 1 only
        blocks = args.cpu_blocks if args.cpu_blocks > 0 else default_cpu_blocks(w)
        cb = oracle_timing(w, blocks, min_seconds=args.cpu_seconds)
        cpu = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
        cpu["gbs"] = cb["value"] * bpp / 1e9     # the host's rate in the step's algorithmic bytes
    if rank != 0:
        return
    line = {"metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_desc,
            "hbm_gbs": step_gbs, "hbm_pct_of_8tbs": 100.0 * step_gbs / NOMINAL_HBM_GBS,
            "hbm_frac_of_measured_copy": step_gbs / peak,
            "gpu_launches": launches, "clocks": clk, "e2e": e2e, "roofline": roof,
            # the whole step against the same peak: the step's algorithmic bytes over its time
            "step_roofline": {"bound": "hbm", "achieved": step_gbs, "peak": peak, "unit": "GB/s",
                              "frac": step_gbs / peak, "bytes_per_step": bpp * info.psi_pad},
            "cpu_baseline": cpu,
            "kernels": kern, "graph": bool(args.graph),
            "last_step_state": {k: st[k] for k in ("t", "skipped", "overflow", "grad_norm", "clip_coef",
                                                   "loss_scale")}}
    if timeline is not None:
        line["timeline"] = timeline
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
