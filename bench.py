#!/usr/bin/env python
"""Throughput of the MSDeformAttn core on B300: sampled points/s of one
forward + backward step, achieved HBM bandwidth against the measured peak,
the same step end to end from host memory, and the fp64 CPU oracle beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is msda_forward followed by msda_backward (atomic mode) on the
Deformable DETR encoder workload (N=2, M=8, D=32, four levels 100x167, 50x84,
25x42, 13x21, Len_q = Len_in = 22223, K=4, fp32), seeded synthetic inputs.
L2 is flushed (a 256 MB write) before every step; per-step CUDA events on the
launching stream exclude the flush and a ~1 ms GPU spin after it that lets the
host enqueue the whole step before its start event runs.  For N > 1 (torchrun) every rank runs its
own batch (weak scaling, no collective on the data path); the time is the
maximum over ranks and the value counts the points of all ranks.

Prints one JSON line on rank 0.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "MSDeformAttn sampled-points/s fwd & fwd+bwd; achieved HBM GB/s vs B300 peak"
UNIT = "sampled-points/s"
WORKLOAD = "encoder_train"
FLUSH_BYTES = 256 << 20
# Before a timed call's start event the GPU spins this many cycles (about
# 1 ms), so that Python has enqueued the whole call by the time the event
# runs: the interval then holds the call's device time, not the GPU waiting
# for the host's marshalling (which exposed up to ~150 us per call on a busy
# host, on calls of ~25 us)
HOLD_CYCLES = 2_000_000
NOMINAL_HBM_GBS = 8000.0      # the roofline denominator the targets are stated against (8 TB/s)
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "dram_traffic.json")
CSRC = os.path.join(ROOT, "scale_deformable_attention_06_b300", "csrc")


# ----------------------------------------------------------------------------- host logic
def dist_env():
    """(rank, local_rank, world_size) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def rank_seed(base_seed, rank):
    """Each rank draws its own batch (weak scaling: independent problems)."""
    return base_seed + 7919 * rank


def max_over_ranks(x, dist=None):
    """Maximum of a float over all ranks (the slowest rank sets the time)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(points_per_rank, world, seconds_max):
    """Whole-job throughput: points of all ranks over the slowest rank's time."""
    return points_per_rank * world / seconds_max if seconds_max > 0 else 0.0


def algorithmic_bytes(w, groups=None):
    """Compulsory HBM bytes of each call on workload w: every tensor the call
    reads or writes, counted once (value re-reads and the grad_value memset
    are not counted).  groups: sets of locations and weights, if the heads
    share them in groups."""
    vb = 2 if w.dtype == "bf16" else 4
    n_val = w.N * w.Len_in * w.M * w.D
    n_out = w.N * w.Lq * w.M * w.D
    n_smp = w.N * w.Lq * (groups or w.M) * w.L * w.K
    fwd = n_val * vb + n_smp * 2 * 4 + n_smp * 4 + n_out * vb
    bwd = n_val * vb + n_smp * 2 * 4 + n_smp * 4 + n_out * vb + n_val * 4 + n_smp * 2 * 4 + n_smp * 4
    n_ref = w.N * w.Lq * w.L * 2
    fused = n_val * vb + n_ref * 4 + n_smp * 2 * 4 + n_smp * 4 + n_out * vb
    # fused backward: value, ref, offsets, logits, grad_output in; grad_value,
    # grad_ref, grad_offsets, grad_logits out
    fused_bwd = (n_val * vb + n_ref * 4 + n_smp * 3 * 4 + n_out * vb
                 + n_val * 4 + n_ref * 4 + n_smp * 3 * 4)
    return {"fwd": fwd, "bwd": bwd, "fused_fwd": fused, "fused_bwd": fused_bwd}


def workload_config(args, w, world):
    """The config keys both arms report: the workload, the step, the batch."""
    return {"workload": "Deformable DETR encoder fwd+bwd: N=2, M=8, D=32, L=4 levels 100x167, 50x84, "
                        "25x42, 13x21 (Len_in=22223), Len_q=Len_in, K=4, fp32"
                        if args.workload == WORKLOAD else args.workload,
            "step": "forward + backward (fused calls)" if args.step == "fused" else "forward + backward",
            "per_rank_batch": w.N, "sampled_points_per_step_per_rank": w.samples,
            "parallelism": f"dp{world} (independent batches per rank)"}


def location_inputs(raw, sh):
    """(sampling_locations float32, reference_points, sampling_offsets) of a
    draw, as torch CPU tensors (input preparation, outside every timed region).
    Drawn references and offsets give the locations ref + off / (W, H) in
    float64; locations drawn directly (the tiny workload) give a reference at
    each row's first sample and pixel offsets to the others."""
    import torch
    if "sampling_locations" in raw:
        loc_h = torch.from_numpy(raw["sampling_locations"]).contiguous()
        ref_h = loc_h[:, :, 0, :, 0, :].clone().contiguous()
        whf = sh[:, [1, 0]].float()
        off_h = ((loc_h - ref_h[:, :, None, :, None, :]) * whf[None, None, None, :, None, :]).contiguous()
        return loc_h, ref_h, off_h
    ref_h = torch.from_numpy(raw["reference_points"])
    off_h = torch.from_numpy(raw["sampling_offsets"])
    wh = sh[:, [1, 0]].to(torch.float64)
    loc_h = (ref_h.double()[:, :, None, :, None, :] + off_h.double() / wh[None, None, None, :, None, :]).float()
    return loc_h.contiguous(), ref_h, off_h


def touched_value_bytes(w, loc):
    """Byte accounting for workloads whose queries are sparse: the bytes of
    the distinct 32-byte sectors of value that the in-map corners of all
    samples touch (the compulsory value traffic, where the whole tensor is
    an upper bound).  loc: sampling locations [N, Len_q, M, L, K, 2]."""
    sh, st = w.spatial_shapes(), w.level_start_index()
    N, Lq, M, L, K, _ = loc.shape
    row_bytes = w.D * (2 if w.dtype == "bf16" else 4)
    n = np.arange(N)[:, None, None, None]
    m = np.arange(M)[None, None, :, None]
    rows = []
    for l in range(L):
        H, W = int(sh[l][0]), int(sh[l][1])
        x0 = np.floor(loc[:, :, :, l, :, 0].astype(np.float64) * W - 0.5).astype(np.int64)
        y0 = np.floor(loc[:, :, :, l, :, 1].astype(np.float64) * H - 0.5).astype(np.int64)
        for dy in (0, 1):
            for dx in (0, 1):
                xc, yc = x0 + dx, y0 + dy
                inside = (xc >= 0) & (xc < W) & (yc >= 0) & (yc < H)
                rows.append((((n * w.Len_in + st[l] + yc * W + xc) * M + m))[inside])
    rows = np.unique(np.concatenate(rows))
    if row_bytes >= 32:
        return int(rows.size) * row_bytes
    return int(np.unique(rows * row_bytes // 32).size) * 32


# The source files each profiled kernel is built from (its translation unit
# and the headers it includes).
KERNEL_SOURCES = {
    "msda_forward_kernel": ("msda_forward.cu", "msda_device.cuh", "msda_launch.h"),
    "msda_forward_kernel_fused": ("msda_forward.cu", "msda_device.cuh", "msda_launch.h"),
    "msda_backward_kernel": ("msda_backward.cu", "msda_device.cuh", "msda_launch.h"),
    "msda_backward_kernel_fused": ("msda_backward.cu", "msda_device.cuh", "msda_launch.h"),
    "ref_grad_kernel": ("msda_backward.cu", "msda_device.cuh", "msda_launch.h"),
    "msda3d_forward_kernel": ("msda3d.cu", "msda_device.cuh", "msda_launch.h"),
    "msda3d_backward_kernel": ("msda3d.cu", "msda_device.cuh", "msda_launch.h"),
}


def _code_only(text):
    """Source text without comments and whitespace runs: edits to comments
    leave the hash (and the profiled counters it keys) valid."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel=None):
    """Hash of the code of `kernel`'s sources (of every kernel source when None)."""
    files = KERNEL_SOURCES[kernel] if kernel else sorted(f for f in os.listdir(CSRC)
                                                          if os.path.isfile(os.path.join(CSRC, f)))
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when the kernel's sources changed since it was captured."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    k = rec.get("kernels", {}).get(kernel, {})
    if not k or k.get("source_hash") != kernel_source_hash(kernel):
        return None
    return k.get("dram_bytes_per_launch")


def step_kernels(step, ms):
    """(kernel, ms a launch, key of its algorithmic bytes) of the step's two
    calls: the fused calls' kernels under the fused step.  `ms` maps the keys
    fwd, bwd, fused_fwd and fused_bwd to CUDA-event times."""
    if step == "fused":
        return {"fwd": ("msda_forward_kernel_fused", ms["fused_fwd"], "fused_fwd"),
                "bwd": ("msda_backward_kernel_fused", ms["fused_bwd"], "fused_bwd")}
    return {"fwd": ("msda_forward_kernel", ms["fwd"], "fwd"), "bwd": ("msda_backward_kernel", ms["bwd"], "bwd")}


def roofline_traffic(kernel, workload):
    """DRAM bytes a launch for the roofline: the committed counts are of the
    encoder training workload's launches, so None for any other workload."""
    return profiled_traffic(kernel) if workload == WORKLOAD else None


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    except (OSError, ValueError, KeyError):
        return 6400.0, "fallback 6.4 TB/s"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons around a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_ms=100):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", str(self.period)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(1.0)
        except OSError:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import torch.distributed as dist
    import scale_deformable_attention_06_b300 as msda

    rank, local_rank, world = dist_env()
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = workloads.WORKLOADS[args.workload]
    raw = workloads.draw(w, seed=rank_seed(w.seed, rank))

    # input preparation (outside every timed region): the unfused inputs are
    # the location step and the softmax of the raw draws, in float64 on the host
    sh = torch.from_numpy(raw["spatial_shapes"])
    loc_h, ref_h, off_h = location_inputs(raw, sh)
    attn_h = torch.softmax(torch.from_numpy(raw["attention_logits"]).double(), -1).float() \
        .reshape(loc_h.shape[:-1]).contiguous()
    vdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    value_h = torch.from_numpy(raw["value"]).to(vdt).contiguous()
    gout_h = torch.from_numpy(raw["grad_output"]).to(vdt).contiguous()
    starts = raw["level_start_index"]

    value, loc, attn, gout = (t.to(dev) for t in (value_h, loc_h, attn_h, gout_h))
    ref_d, off_d = ref_h.contiguous().to(dev), off_h.contiguous().to(dev)
    logit_d = torch.from_numpy(raw["attention_logits"]).to(dev)
    out = torch.empty((w.N, w.Lq, w.M * w.D), dtype=vdt, device=dev)
    gv = torch.empty(value.shape, dtype=torch.float32, device=dev)
    gl = torch.empty_like(loc)
    ga = torch.empty_like(attn)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        msda.msda_forward(value, sh, starts, loc, attn, output=out)

    def bwd(flags=0):
        msda.msda_backward(value, sh, starts, loc, attn, gout, grad_value=gv, grad_sampling_locations=gl,
                           grad_attention_weights=ga, flags=flags)

    def fused():
        msda.msda_forward_fused(value, sh, starts, ref_d, off_d, logit_d, output=out)

    gref = torch.empty_like(ref_d)
    goff = torch.empty_like(off_d)
    glog = torch.empty_like(logit_d)

    def fused_bwd(flags=0):
        msda.msda_backward_fused(value, sh, starts, ref_d, off_d, logit_d, gout, grad_value=gv,
                                 grad_reference_points=gref, grad_sampling_offsets=goff, grad_attention_logits=glog,
                                 flags=flags)

    def step():
        if args.step == "fused":
            fused()
            fused_bwd()
        else:
            fwd()
            bwd()

    def timed(fn, iters, pre=None, warm=False):
        """Per-call device times (ms) with an L2 flush before each call, unless
        warm (then the call's inputs are left in L2 by the call before)."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for e0, e1 in evs:
            if not warm:
                flush.fill_(1.0)
            if pre is not None:
                pre()
            torch.cuda._sleep(HOLD_CYCLES)
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return [e0.elapsed_time(e1) for e0, e1 in evs]

    for _ in range(max(args.warmup, 3)):
        step()
        fused()
    torch.cuda.synchronize(dev)

    # ---- the timed step: K steps between a barrier + synchronize on each side
    clocks = ClockSampler(local_rank)
    if rank == 0:
        clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    step_ms = timed(step, args.steps)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if rank == 0 else None
    total_s = max_over_ranks(sum(step_ms) / 1e3, dist if world > 1 else None)

    pts = w.samples
    value_pts = aggregate(pts, world, total_s / args.steps)
    ab = algorithmic_bytes(w)
    if args.only_step:          # profiling runs: the timed step alone
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value_pts, "unit": UNIT, "n_gpus": world,
                              "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_s * 1e3 / args.steps,
                              "only_step": True}))
        if world > 1:
            dist.destroy_process_group()
        return

    # ---- per-kernel times (same protocol) for the roofline and the parts
    reps = max(10, min(args.steps, 200))
    fwd_ms = statistics.mean(timed(fwd, reps))
    fused_ms = statistics.mean(timed(fused, reps))
    bwd_ms = statistics.mean(timed(lambda: bwd(msda.MSDA_ACCUMULATE_GRAD_VALUE), reps, pre=lambda: gv.zero_()))
    fwd_warm_ms = statistics.mean(timed(fwd, reps, warm=True))
    bwd_warm_ms = statistics.mean(timed(lambda: bwd(msda.MSDA_ACCUMULATE_GRAD_VALUE), reps, pre=lambda: gv.zero_(),
                                        warm=True))
    det_ms = statistics.mean(timed(lambda: bwd(msda.MSDA_DETERMINISTIC), max(5, reps // 4)))
    fused_bwd_ms = statistics.mean(timed(lambda: fused_bwd(msda.MSDA_ACCUMULATE_GRAD_VALUE), reps,
                                         pre=lambda: gv.zero_()))
    peak, peak_src = measured_peak()
    kern = step_kernels(args.step, {"fwd": fwd_ms, "bwd": bwd_ms, "fused_fwd": fused_ms, "fused_bwd": fused_bwd_ms})
    dom = max(kern, key=lambda k: kern[k][1])
    name, ms, ab_key = kern[dom]
    achieved = ab[ab_key] / (ms / 1e3) / 1e9
    traffic = roofline_traffic(name, args.workload)

    # ---- the SM line-rate ceilings (probes over a value-sized buffer): the
    # forward's floor is its corner gathers at the gather rate, the backward's
    # those plus its grad_value reductions at the reduction rate
    line = None
    if w.D == 32 and w.dtype == "f32":
        gathers = w.samples * 4
        rates = line_rates(dev, w.N * w.Len_in * w.M * w.D * 4, gathers, reps=5)
        reds = backward_reduction_lines(w, loc_h.numpy())
        g_rate, r_rate = rates["gather"]["lines_per_s"], rates["reduce"]["lines_per_s"]
        ceil_us = {"fwd": gathers / g_rate * 1e6, "bwd": gathers / g_rate * 1e6 + reds / r_rate * 1e6}
        line = {"gather_lines_per_s": g_rate, "reduce_lines_per_s": r_rate,
                "gathers_per_launch": gathers, "backward_reductions_per_launch": reds,
                "fwd_ceiling_us": ceil_us["fwd"], "bwd_ceiling_us": ceil_us["bwd"],
                "frac_fwd": ceil_us["fwd"] / (kern["fwd"][1] * 1e3), "frac_bwd": ceil_us["bwd"] / (kern["bwd"][1] * 1e3),
                "probes": rates,
                "note": "ceiling = the launch's 128-byte line gathers at the probed gather rate (+ its grad_value "
                        "reductions at the probed reduction rate, taken one after the other); frac = ceiling / "
                        "the launch's CUDA-event time"}

    # ---- end to end from pinned host memory through the same calls
    if args.step == "fused":
        d_in = (value, ref_d, off_d, logit_d, gout)
        d_out = (out, gv, gref, goff, glog)
    else:
        d_in = (value, loc, attn, gout)
        d_out = (out, gv, gl, ga)
    h_in = [t.cpu().pin_memory() for t in d_in]
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in d_out]

    def e2e_step():
        for h, d in zip(h_in, d_in):
            d.copy_(h, non_blocking=True)
        step()
        for h, d in zip(h_out, d_out):
            h.copy_(d, non_blocking=True)

    for _ in range(2):
        e2e_step()
    e2e_iters = max(3, min(args.steps, 20))
    e2e_serial_ms = sum(timed(e2e_step, e2e_iters)) / e2e_iters

    # Pipelined end to end: two buffer sets; the upload of step i+1 and the
    # download of step i-1 run on their own streams (the copy engines) while
    # step i computes.  Every step still copies its own inputs from pinned host
    # memory and its own results back inside the timed region.
    def run_step(io, stream):
        i, o = io
        if args.step == "fused":
            msda.msda_forward_fused(i[0], sh, starts, i[1], i[2], i[3], output=o[0], stream=stream)
            msda.msda_backward_fused(i[0], sh, starts, i[1], i[2], i[3], i[4], grad_value=o[1],
                                     grad_reference_points=o[2], grad_sampling_offsets=o[3],
                                     grad_attention_logits=o[4], stream=stream)
        else:
            msda.msda_forward(i[0], sh, starts, i[1], i[2], output=o[0], stream=stream)
            msda.msda_backward(i[0], sh, starts, i[1], i[2], i[3], grad_value=o[1], grad_sampling_locations=o[2],
                               grad_attention_weights=o[3], stream=stream)

    sets = [(d_in, d_out), (tuple(torch.empty_like(t) for t in d_in), tuple(torch.empty_like(t) for t in d_out))]
    h_outs = [h_out, [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in d_out]]
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))

    def pipelined(iters):
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_cmp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        torch.cuda.synchronize(dev)
        for b in range(2):
            ev_cmp[b].record(s_cmp)
            ev_out[b].record(s_out)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(iters):
            b = i % 2
            s_in.wait_event(ev_cmp[b])            # step i-2 no longer reads these inputs
            with torch.cuda.stream(s_in):
                for h, d in zip(h_in, sets[b][0]):
                    d.copy_(h, non_blocking=True)
            ev_in[b].record(s_in)
            s_cmp.wait_event(ev_in[b])
            s_cmp.wait_event(ev_out[b])           # step i-2's results are back on the host
            run_step(sets[b], s_cmp)
            ev_cmp[b].record(s_cmp)
            s_out.wait_event(ev_cmp[b])
            with torch.cuda.stream(s_out):
                for h, d in zip(h_outs[b], sets[b][1]):
                    h.copy_(d, non_blocking=True)
            ev_out[b].record(s_out)
        t1.record(s_out)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1)

    def copies_only(iters):
        """The same uploads and downloads, concurrent on their two streams,
        with no compute: the host link's floor for the pipelined step."""
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        s_out.wait_event(t0)
        for i in range(iters):
            b = i % 2
            with torch.cuda.stream(s_in):
                for h, d in zip(h_in, sets[b][0]):
                    d.copy_(h, non_blocking=True)
            with torch.cuda.stream(s_out):
                for h, d in zip(h_outs[b], sets[1 - b][1]):
                    h.copy_(d, non_blocking=True)
        s_in.wait_stream(s_out)
        t1.record(s_in)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1)

    pipelined(4)
    e2e_s = max_over_ranks(pipelined(e2e_iters) / 1e3 / e2e_iters, dist if world > 1 else None)
    copies_only(2)
    link_floor_ms = copies_only(e2e_iters) / e2e_iters
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, raw, loc_h.numpy(), attn_h.numpy(), value_h.float().numpy(), gout_h.float().numpy())

    if world > 1:
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": value_pts, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_s * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32" if w.dtype == "f32" else "bf16-storage/f32",
        "data": "synthetic (seeded PCG64 draws with the encoder workload's shapes and distributions)",
        "config": dict(workload_config(args, w, world),
                       calls=("msda_forward_fused + msda_backward_fused" if args.step == "fused" else
                              "msda_forward + msda_backward") + " (atomic grad_value)",
                       l2="flushed before every step (256 MB write); per-step events exclude the flush and a ~1 ms GPU "
                          "spin after it (the host enqueues the step meanwhile)"),
        "fwd": {"ms": fwd_ms, "points_per_s": pts / (fwd_ms / 1e3), "gbs": ab["fwd"] / (fwd_ms / 1e3) / 1e9,
                "frac_of_peak": ab["fwd"] / (fwd_ms / 1e3) / 1e9 / peak,
                "frac_of_nominal_8tbs": ab["fwd"] / (fwd_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                "algorithmic_bytes": ab["fwd"], "warm_l2_ms": fwd_warm_ms},
        "bwd": {"ms": bwd_ms, "points_per_s": pts / (bwd_ms / 1e3), "gbs": ab["bwd"] / (bwd_ms / 1e3) / 1e9,
                "frac_of_peak": ab["bwd"] / (bwd_ms / 1e3) / 1e9 / peak,
                "frac_of_nominal_8tbs": ab["bwd"] / (bwd_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                "algorithmic_bytes": ab["bwd"],
                "deterministic_ms": det_ms, "warm_l2_ms": bwd_warm_ms},
        "fused_fwd": {"ms": fused_ms, "points_per_s": pts / (fused_ms / 1e3),
                      "gbs": ab["fused_fwd"] / (fused_ms / 1e3) / 1e9},
        "fused_bwd": {"ms": fused_bwd_ms, "points_per_s": pts / (fused_bwd_ms / 1e3),
                      "gbs": ab["fused_bwd"] / (fused_bwd_ms / 1e3) / 1e9},
        "fwd_bwd_gbs": (ab[kern["fwd"][2]] + ab[kern["bwd"][2]]) / (total_s / args.steps) / 1e9,
        "fwd_bwd_frac_of_nominal_8tbs": (ab[kern["fwd"][2]] + ab[kern["bwd"][2]]) / (total_s / args.steps) / 1e9
                                        / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": peak, "peak_source": peak_src,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": ab[ab_key], "launch_ms": ms,
                     "frac_of_line_ceiling": line[f"frac_{dom}"] if line else None},
        "line_ceiling": line,
        "e2e": {"value": aggregate(pts, world, e2e_s), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                "pipeline": "double-buffered: upload of step i+1 and download of step i-1 on their own streams "
                            "while step i computes",
                "serial_ms_per_step": e2e_serial_ms,
                "copies_only_ms_per_step": link_floor_ms,
                "copies_only": "the same uploads and downloads run concurrently with no compute: the host link's "
                               "floor for the pipelined step"},
        # per step: forward 1; backward: grad_value zeroing + backward kernel
        # (+ reference-point reduction in the fused step)
        "gpu_launches": (4 if args.step == "fused" else 3) * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
        "library": msda.LIBRARY,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- line-rate ceilings
PROBES = os.path.join(ROOT, "scale_deformable_attention_06_b300", "libmsda_probes.so")


def _probes():
    import ctypes
    lib = ctypes.CDLL(PROBES)
    i64, vp, u32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint32
    lib.msda_probe_sink_bytes.restype = ctypes.c_size_t
    lib.msda_probe_gather.argtypes = [vp, i64, i64, i64, vp, u32, vp]
    lib.msda_probe_reduce.argtypes = [vp, i64, i64, i64, u32, vp]
    lib.msda_probe_mixed.argtypes = [vp, i64, i64, ctypes.c_int, vp, u32, vp]
    lib.msda_probe_bulk_reduce.argtypes = [vp, i64, i64, u32, vp]
    lib.msda_probe_accesses.argtypes = [i64]
    lib.msda_probe_accesses.restype = i64
    return lib


def line_rates(dev, buf_bytes, lines, reps=10):
    """Random 128-byte line operations per second on this GPU, measured with
    the probes of libmsda_probes.so over a buffer of buf_bytes (the value
    tensor's size: L2-resident for the encoder), `lines` operations per
    launch, CUDA events, median of `reps` launches:
      gather            four lines per warp instruction (LDG.128), uniform
      gather_hot        the same over the first 128 KB (L1-resident)
      reduce            red.global.add.v4.f32 into uniform lines
      reduce_hot        the same over 128 KB (contended)
      bulk_reduce       the same reductions through the TMA unit (a 128-byte
                        cp.reduce.async.bulk per line, staged in shared memory)
      mixed_r           eight gathers and r reductions per quarter-warp round
    """
    import ctypes
    import torch
    lib = _probes()
    n_lines = buf_bytes // 128
    buf = torch.zeros(n_lines * 32, dtype=torch.float32, device=dev)
    sink = torch.empty(lib.msda_probe_sink_bytes() // 4, dtype=torch.float32, device=dev)
    sp = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    bp, kp = ctypes.c_void_p(buf.data_ptr()), ctypes.c_void_p(sink.data_ptr())

    def timed_ms(fn):
        for _ in range(2):
            if fn() != 0:
                raise RuntimeError("probe launch failed")
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for i, (e0, e1) in enumerate(evs):
            e0.record()
            fn(i)
            e1.record()
        torch.cuda.synchronize(dev)
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)

    hot = (128 << 10) // 128
    done = int(lib.msda_probe_accesses(lines))          # whole rounds: at least `lines`
    out = {"buffer_bytes": n_lines * 128, "lines_per_launch": done, "reps": reps}
    ms = {
        "gather": timed_ms(lambda i=0: lib.msda_probe_gather(bp, n_lines, 0, lines, kp, 17 + i, sp)),
        "gather_hot": timed_ms(lambda i=0: lib.msda_probe_gather(bp, n_lines, hot, lines, kp, 17 + i, sp)),
        "reduce": timed_ms(lambda i=0: lib.msda_probe_reduce(bp, n_lines, 0, lines, 17 + i, sp)),
        "reduce_hot": timed_ms(lambda i=0: lib.msda_probe_reduce(bp, n_lines, hot, lines, 17 + i, sp)),
        "bulk_reduce": timed_ms(lambda i=0: lib.msda_probe_bulk_reduce(bp, n_lines, lines, 17 + i, sp)),
    }
    for r in (2, 4, 6, 8):
        ms[f"mixed_{r}"] = timed_ms(lambda i=0, r=r: lib.msda_probe_mixed(bp, n_lines, lines, r, kp, 17 + i, sp))
    for k, v in ms.items():
        if k.startswith("mixed"):
            r = int(k.split("_")[1])
            out[k] = {"us": v * 1e3, "gathers": done, "reductions": done * r // 8}
        else:
            out[k] = {"us": v * 1e3, "lines_per_s": done / (v / 1e3)}
    return out


def backward_reduction_lines(w, loc):
    """red.global.add.v4 line operations of msda_backward on workload w (head_dim
    32, fp32: one line per corner row), as its kernel issues them: one per
    in-map corner, except on levels with at least 32 samples per pixel
    (Len_q * K >= 32 * H * W), where the warp's four consecutive queries of one
    head first merge coinciding corners (one reduction per distinct pixel of
    the group and level).  loc: sampling locations [N, Len_q, M, L, K, 2]."""
    sh = w.spatial_shapes()
    N, Lq, M, L, K, _ = loc.shape
    total = 0
    for l in range(L):
        H, W = int(sh[l][0]), int(sh[l][1])
        x0 = np.floor(loc[:, :, :, l, :, 0].astype(np.float64) * W - 0.5).astype(np.int64)
        y0 = np.floor(loc[:, :, :, l, :, 1].astype(np.float64) * H - 0.5).astype(np.int64)
        keys = []
        for dy in (0, 1):
            for dx in (0, 1):
                xc, yc = x0 + dx, y0 + dy
                keys.append(np.where((xc >= 0) & (xc < W) & (yc >= 0) & (yc < H), yc * W + xc, -1))
        keys = np.stack(keys, -1)                                           # [N, Lq, M, K, 4]
        if Lq * K < 32 * H * W:
            total += int((keys >= 0).sum())
            continue
        G = 4
        pad = (-Lq) % G
        kk = np.concatenate([keys, np.full((N, pad) + keys.shape[2:], -1, np.int64)], axis=1)
        kk = kk.reshape(N, -1, G, M, K * 4).transpose(0, 1, 3, 2, 4).reshape(N, -1, M, G * K * 4)
        kk = np.sort(kk, axis=-1)
        total += int(((kk[..., 1:] != kk[..., :-1]) & (kk[..., 1:] >= 0)).sum() + (kk[..., 0] >= 0).sum())
    return total


def run_line_rates(args):
    """One JSON line: the probes' rates over the encoder's value-sized buffer,
    and the encoder calls' line ceilings that follow from them."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = workloads.WORKLOADS[WORKLOAD]
    lines = w.samples * 4
    rates = line_rates(dev, w.N * w.Len_in * w.M * w.D * 4, lines)
    print(json.dumps({"line_rates": True, "workload_buffer": "encoder value tensor (N=2, Len_in=22223, M=8, D=32, "
                      "fp32)", **rates}))


# ----------------------------------------------------------------------------- every workload
def run_sweep(args):
    """Per-call device times on every workload (one JSON line each): forward,
    fused forward, backward (fp32 atomics and deterministic), fused backward,
    with the algorithmic bytes of each call; the oracle's single-core time on a
    bounded query sample beside them."""
    import torch
    import scale_deformable_attention_06_b300 as msda
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    peak, _ = measured_peak()

    def timed(fn, iters, pre=None, warm=False):
        """Median device time (ms); L2 flushed before each call unless warm
        (then the call's inputs are left in L2 by the call before)."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for _ in range(3):
            fn()
        for e0, e1 in evs:
            if not warm:
                flush.fill_(1.0)
            if pre is not None:
                pre()
            torch.cuda._sleep(HOLD_CYCLES)
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)

    chosen = args.sweep_only.split(",") if args.sweep_only else None
    for name in ("tiny", "encoder", "decoder", "encoder_train", "large", "encoder_g1", "encoder_g2", "encoder_g4"):
        if chosen is not None and name not in chosen:
            continue
        # encoder_gG: the encoder workload with G sets of locations and weights,
        # each shared by 8 / G heads (head groups: 256, 128 or 64 channels a set)
        groups = int(name[len("encoder_g"):]) if name.startswith("encoder_g") else None
        w = workloads.WORKLOADS["encoder" if groups else name]
        raw = workloads.draw(w)
        if groups:
            for k in ("sampling_offsets", "attention_logits"):
                raw[k] = np.ascontiguousarray(raw[k][:, :, :groups])
        sh, starts = torch.from_numpy(raw["spatial_shapes"]), raw["level_start_index"]
        vdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        loc_h, ref_h, off_h = location_inputs(raw, sh)
        lg_h = torch.from_numpy(raw["attention_logits"])
        attn_h = torch.softmax(lg_h.double(), -1).float().reshape(loc_h.shape[:-1]).contiguous()
        value = torch.from_numpy(raw["value"]).to(vdt).to(dev)
        gout = torch.from_numpy(raw["grad_output"]).to(vdt).to(dev)
        loc, attn, ref, off, lg = (t.contiguous().to(dev) for t in (loc_h, attn_h, ref_h, off_h, lg_h))
        out = torch.empty((w.N, w.Lq, w.M * w.D), dtype=vdt, device=dev)
        gv = torch.empty(value.shape, dtype=torch.float32, device=dev)
        gl, ga = torch.empty_like(loc), torch.empty_like(attn)
        gr, go, glg = torch.empty_like(ref), torch.empty_like(off), torch.empty_like(lg)
        acc = msda.MSDA_ACCUMULATE_GRAD_VALUE
        reps = 20
        t = {
            "fwd": timed(lambda: msda.msda_forward(value, sh, starts, loc, attn, output=out), reps),
            "fused_fwd": timed(lambda: msda.msda_forward_fused(value, sh, starts, ref, off, lg, output=out), reps),
            "bwd": timed(lambda: msda.msda_backward(value, sh, starts, loc, attn, gout, grad_value=gv,
                                                    grad_sampling_locations=gl, grad_attention_weights=ga,
                                                    flags=acc), reps, pre=lambda: gv.zero_()),
            "bwd_deterministic": timed(lambda: msda.msda_backward(value, sh, starts, loc, attn, gout, grad_value=gv,
                                                                  grad_sampling_locations=gl,
                                                                  grad_attention_weights=ga,
                                                                  flags=msda.MSDA_DETERMINISTIC), 5),
            "fused_bwd": timed(lambda: msda.msda_backward_fused(value, sh, starts, ref, off, lg, gout,
                                                                grad_value=gv, grad_reference_points=gr,
                                                                grad_sampling_offsets=go,
                                                                grad_attention_logits=glg, flags=acc), reps,
                               pre=lambda: gv.zero_()),
        }
        # the same calls with L2 warm (no flush between them): reported beside
        # the flushed times, which are the ones the rates use
        warm = {"fwd": timed(lambda: msda.msda_forward(value, sh, starts, loc, attn, output=out), reps, warm=True),
                "bwd": timed(lambda: msda.msda_backward(value, sh, starts, loc, attn, gout, grad_value=gv,
                                                        grad_sampling_locations=gl, grad_attention_weights=ga,
                                                        flags=acc), reps, pre=lambda: gv.zero_(), warm=True)}
        ab = algorithmic_bytes(w, groups)
        ab["bwd_deterministic"] = ab["bwd"]
        # sparse queries: value traffic counted as the sectors the samples touch
        vbytes = w.N * w.Len_in * w.M * w.D * (2 if w.dtype == "bf16" else 4)
        touched = touched_value_bytes(w, loc_h.numpy()) if w.Lq * 4 <= w.Len_in else None
        calls = {}
        for k, ms in t.items():
            gbs = ab[k] / (ms / 1e3) / 1e9
            calls[k] = {"us": ms * 1e3, "points_per_s": w.samples / (ms / 1e3), "gbs": gbs,
                        "frac_of_measured_hbm_peak": gbs / peak, "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
                        "algorithmic_bytes": ab[k]}
            if k in warm:
                calls[k]["warm_l2_us"] = warm[k] * 1e3
            if touched is not None:
                tb = ab[k] - vbytes + touched
                calls[k].update({"algorithmic_bytes_touched_value": tb,
                                 "frac_touched_of_measured_hbm_peak": tb / (ms / 1e3) / 1e9 / peak})
        # oracle, single core, forward + backward on a bounded query sample of this workload
        q = max(1, min(w.Lq, int(2.0e5 // (w.M * w.L * w.K * max(w.N, 1)))))
        smp = _oracle_sample(w, raw, loc_h.numpy(), attn_h.numpy(), value.float().cpu().numpy(),
                             gout.float().cpu().numpy(), 0, q)
        t0 = time.perf_counter()
        ref_out, ref_gv, _, ref_ga = _oracle_step(smp)
        el = time.perf_counter() - t0
        pts = w.N * q * w.M * w.L * w.K
        # the library on the same sample and the same (storage-rounded) inputs:
        # a forward and a backward call on the sample's queries alone
        lq, aq, gq = (t[:, :q].contiguous() for t in (loc, attn, gout))
        got_out = msda.msda_forward(value, sh, starts, lq, aq).float().cpu().numpy()
        got_gv, _, got_ga = msda.msda_backward(value, sh, starts, lq, aq, gq)

        def rel(a, b):
            return float(np.abs(a - b).max() / max(float(np.abs(b).max()), 1e-30))
        line = {"sweep": True, "workload": name, "dtype": w.dtype, "samples": w.samples,
                "head_groups": groups or w.M, "value_bytes": vbytes, "value_bytes_touched": touched, "calls": calls,
                "oracle_fwd_bwd_points_per_s_1core": pts / el,
                "oracle_sample": f"{q} of {w.Lq} queries x {w.N} batches",
                "rel_error_vs_oracle": {
                    "output": rel(got_out, ref_out), "grad_value": rel(got_gv.cpu().numpy(), ref_gv),
                    "grad_attention_weights": rel(got_ga.cpu().numpy(), ref_ga),
                    "norm": "max |lib - oracle| / max |oracle| on the oracle's query sample, same inputs "
                            "(grad_sampling_locations is compared in the tests, which handle its one-sided "
                            "derivative at cell edges)"}}
        if w.dtype == "bf16":
            # the storage error itself: the forward against the oracle on the
            # unrounded fp32 draws, on the same query sample (normwise rel)
            import oracle
            got = msda.msda_forward(value, sh, starts, loc, attn, output=out)[:, :q].float().cpu().numpy()
            ref_u = oracle.forward(raw["value"], raw["spatial_shapes"], raw["level_start_index"],
                                   loc_h.numpy()[:, :q], attn_h.numpy()[:, :q])
            line["bf16_storage_rel_error_vs_unrounded_fp32"] = float(np.abs(got - ref_u).max() / np.abs(ref_u).max())
        print(json.dumps(line))
    if chosen is None or "video" in chosen:
        run_sweep_volumes(timed, peak)


def run_sweep_volumes(timed, peak):
    """The 3-D variant on a video-like workload: three levels of (frames, rows,
    columns) = (8, 50, 84), (4, 25, 42), (2, 13, 21), one query per voxel,
    uniformly drawn locations, fp32."""
    import torch
    import scale_deformable_attention_06_b300 as msda
    import oracle
    dev = torch.device("cuda", 0)
    levels = workloads.VIDEO_LEVELS
    S = sum(d * h * w for d, h, w in levels)
    N, M, D, K, Lq = 1, 8, 32, 4, S
    raw = workloads.draw_volumes(N, M, D, levels, K, Lq, seed=1240)
    L = len(levels)
    sh, st = raw["spatial_shapes"], raw["level_start_index"]
    attn_h = torch.softmax(torch.from_numpy(raw["attention_logits"]).double(), -1).float().reshape(N, Lq, M, L, K)
    value = torch.from_numpy(raw["value"]).to(dev)
    gout = torch.from_numpy(raw["grad_output"]).to(dev)
    loc = torch.from_numpy(raw["sampling_locations"]).to(dev)
    attn = attn_h.contiguous().to(dev)
    out = torch.empty((N, Lq, M * D), device=dev)
    gv = torch.empty(value.shape, device=dev)
    gl, ga = torch.empty_like(loc), torch.empty_like(attn)
    samples = N * Lq * M * L * K
    t = {"fwd": timed(lambda: msda.msda3d_forward(value, sh, st, loc, attn, output=out), 20),
         "bwd": timed(lambda: msda.msda3d_backward(value, sh, st, loc, attn, gout, grad_value=gv,
                                                   grad_sampling_locations=gl, grad_attention_weights=ga,
                                                   flags=msda.MSDA_ACCUMULATE_GRAD_VALUE), 20,
                      pre=lambda: gv.zero_())}
    nval, nout = N * S * M * D, N * Lq * M * D
    ab = {"fwd": 4 * (nval + samples * 4 + nout), "bwd": 4 * (nval + samples * 4 + nout + nval + samples * 4)}
    calls = {k: {"us": ms * 1e3, "points_per_s": samples / (ms / 1e3), "gbs": ab[k] / (ms / 1e3) / 1e9,
                 "frac_of_measured_hbm_peak": ab[k] / (ms / 1e3) / 1e9 / peak,
                 "frac_of_nominal_8tbs": ab[k] / (ms / 1e3) / 1e9 / NOMINAL_HBM_GBS, "algorithmic_bytes": ab[k]}
             for k, ms in t.items()}
    q = 64
    lv = raw["sampling_locations"][:, :q].astype(np.float64)
    t0 = time.perf_counter()
    ref_out = oracle.forward3d(raw["value"].astype(np.float64), sh, st, lv, attn_h.numpy()[:, :q].astype(np.float64))
    ref_gv, _, ref_ga = oracle.backward3d(raw["value"].astype(np.float64), sh, st, lv,
                                          attn_h.numpy()[:, :q].astype(np.float64),
                                          raw["grad_output"][:, :q].astype(np.float64))
    el = time.perf_counter() - t0
    # the library on the same sample (same inputs)
    lq, aq, gq = (t[:, :q].contiguous() for t in (loc, attn, gout))
    got_out = msda.msda3d_forward(value, sh, st, lq, aq).cpu().numpy()
    got_gv, _, got_ga = msda.msda3d_backward(value, sh, st, lq, aq, gq)

    def rel(a, b):
        return float(np.abs(a - b).max() / max(float(np.abs(b).max()), 1e-30))
    print(json.dumps({"sweep": True, "workload": "video (3-D, trilinear)", "dtype": "f32", "samples": samples,
                      "calls": calls, "oracle_fwd_bwd_points_per_s_1core": N * q * M * L * K / el,
                      "oracle_sample": f"{q} of {Lq} queries",
                      "rel_error_vs_oracle": {"output": rel(got_out, ref_out),
                                              "grad_value": rel(got_gv.cpu().numpy(), ref_gv),
                                              "grad_attention_weights": rel(got_ga.cpu().numpy(), ref_ga)}}))


# ----------------------------------------------------------------------------- oracle timings
def _oracle_sample(w, raw, loc, attn, value, gout, q0, q1):
    """float64 inputs of queries [q0, q1) (all batches); the oracle's own input format."""
    return dict(value=np.ascontiguousarray(value, dtype=np.float64), sh=raw["spatial_shapes"],
                st=raw["level_start_index"], loc=np.ascontiguousarray(loc[:, q0:q1], dtype=np.float64),
                attn=np.ascontiguousarray(attn[:, q0:q1], dtype=np.float64),
                g=np.ascontiguousarray(gout[:, q0:q1], dtype=np.float64))


def _oracle_step(s):
    """Forward and backward of the oracle on a sample: (out, grad_value, grad_loc, grad_attn)."""
    import oracle
    out = oracle.forward(s["value"], s["sh"], s["st"], s["loc"], s["attn"])
    return (out,) + tuple(oracle.backward(s["value"], s["sh"], s["st"], s["loc"], s["attn"], s["g"]))


def cpu_model():
    """The host CPU's model name (from /proc/cpuinfo), or None."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


_WORKER_INPUTS = {}


def _oracle_inputs(name):
    """The oracle's float64 inputs of a whole workload (storage-rounded value
    and grad_output, as the GPU sees them), drawn from the workload's seed."""
    import torch
    w = workloads.WORKLOADS[name]
    raw = workloads.draw(w)
    sh = torch.from_numpy(raw["spatial_shapes"])
    loc_h, _, _ = location_inputs(raw, sh)
    attn_h = torch.softmax(torch.from_numpy(raw["attention_logits"]).double(), -1).float().reshape(loc_h.shape[:-1])
    vdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    value = torch.from_numpy(raw["value"]).to(vdt).float().numpy()
    gout = torch.from_numpy(raw["grad_output"]).to(vdt).float().numpy()
    return w, raw, loc_h.numpy(), attn_h.numpy(), value, gout


def _worker_prepare(name):
    """Pool worker: draw and keep the workload's oracle inputs (untimed)."""
    if name not in _WORKER_INPUTS:
        _WORKER_INPUTS[name] = _oracle_inputs(name)
    w, raw, loc, attn, value, gout = _WORKER_INPUTS[name]
    _oracle_step(_oracle_sample(w, raw, loc, attn, value, gout, 0, 1))     # loads the oracle library
    return os.getpid()


def _worker_range(task):
    """Pool worker: the oracle's forward + backward on queries [q0, q1) of all batches."""
    name, q0, q1 = task
    w, raw, loc, attn, value, gout = _WORKER_INPUTS[name]
    _oracle_step(_oracle_sample(w, raw, loc, attn, value, gout, q0, q1))
    return q1 - q0


def run_cpu_all_cores(args):
    """The fp64 oracle, as it stands, on every host core: the workload's queries
    split over one process per core (a spawn-started pool that never touches
    the GPU), forward + backward of the whole workload timed by wall clock.
    Prints one JSON line."""
    import multiprocessing as mp
    w = workloads.WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        pids = set(pool.map(_worker_prepare, [args.workload] * (4 * cores)))
        if len(pids) < cores:          # every worker prepared before the clock starts
            pool.map(_worker_prepare, [args.workload] * (16 * cores))
        chunk = max(1, -(-w.Lq // (4 * cores)))
        tasks = [(args.workload, q0, min(w.Lq, q0 + chunk)) for q0 in range(0, w.Lq, chunk)]
        times = []
        for _ in range(3):             # the median of three passes over the whole workload
            t0 = time.perf_counter()
            done = sum(pool.map(_worker_range, tasks, chunksize=1))
            times.append(time.perf_counter() - t0)
            assert done == w.Lq
    el = statistics.median(times)
    print(json.dumps({"cpu_baseline_all_cores": {
        "value": w.samples / el, "unit": UNIT, "cores": cores, "kind": "oracle", "seconds": el,
        "sample": f"whole {args.workload} workload, forward + backward, its {w.Lq} queries (x{w.N} batches) in "
                  f"{len(tasks)} ranges over {cores} processes; median of 3 passes", "cpu_model": cpu_model()}}))


def cpu_baseline(w, raw, loc, attn, value, gout, budget_s=12.0):
    """The fp64 oracle, as it stands, single-threaded on this host: forward +
    backward on the whole workload, repeated until about `budget_s` seconds."""
    s = _oracle_sample(w, raw, loc, attn, value, gout, 0, w.Lq)
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(s)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 10:
            break
    return {"value": w.samples * reps / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"whole {w.name} workload (all {w.N * w.Lq} queries), forward + backward, {reps} repetitions, "
                      f"{el:.1f} s", "host_cores_available": os.cpu_count(), "cpu_model": cpu_model()}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    import oracle
    w = workloads.WORKLOADS[args.workload]
    raw = workloads.draw(w)
    if "sampling_locations" in raw:        # locations drawn directly (the tiny workload)
        loc = raw["sampling_locations"].astype(np.float32)
    else:
        loc = oracle.locations(raw["spatial_shapes"], raw["reference_points"],
                               raw["sampling_offsets"]).astype(np.float32)
    attn = oracle.softmax(raw["attention_logits"]).astype(np.float32).reshape(loc.shape[:-1])
    # one step = forward + backward of a bounded query sample (all batches)
    q_per_step = max(1, w.Lq // 16)
    starts = [(i * q_per_step) % max(1, w.Lq - q_per_step) for i in range(args.warmup + args.steps)]
    samples = [_oracle_sample(w, raw, loc, attn, raw["value"], raw["grad_output"], q, q + q_per_step) for q in starts]
    for s in samples[:args.warmup]:
        _oracle_step(s)
    t0 = time.perf_counter()
    for s in samples[args.warmup:]:
        _oracle_step(s)
    el = time.perf_counter() - t0
    pts = w.N * q_per_step * w.M * w.L * w.K * args.steps
    v = pts / el
    sample = f"{q_per_step} of {w.Lq} queries (x{w.N} batches) per step, forward + backward"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(args, w, world),
                           calls="oracle forward + backward (fp64, one host core) on a bounded query sample per step"),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-step", action="store_true", help="time the step only (for profiler runs)")
    ap.add_argument("--sweep", action="store_true", help="per-call times on every workload (one JSON line each)")
    ap.add_argument("--line-rates", action="store_true",
                    help="random 128-byte line gather / reduction rates of this GPU (libmsda_probes.so)")
    ap.add_argument("--sweep-only", default="",
                    help="comma list of sweep workloads (tiny, encoder, decoder, encoder_train, large, encoder_g1, encoder_g2, "
                         "encoder_g4, "
                         "video)")
    ap.add_argument("--cpu-all-cores", action="store_true",
                    help="the oracle on every host core (one process each), the whole workload once; no GPU")
    ap.add_argument("--step", choices=["unfused", "fused"], default="unfused",
                    help="unfused: msda_forward + msda_backward on locations and weights; fused: msda_forward_fused + "
                         "msda_backward_fused on reference points, offsets and logits")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.cpu_all_cores:
        run_cpu_all_cores(args)
    elif args.line_rates:
        run_line_rates(args)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
