#!/usr/bin/env python3
"""Benchmark of the HCCL-style collective data plane on one GB300.

Default workload (one "step" = one AllReduce call over the whole batch):
  Ring AllReduce, sum, P = 8 virtual ranks, fp32, 16,777,216 elements per rank
  (64 MiB per rank), values N(0,1) * 1e-3 (synthetic gradients, seed 0),
  fused mode (one kernel per call), out of place.
Metric: effective algbw = n * b / t (bytes of one rank's vector per second of
one call), GB/s.  The inputs (512 MiB) and outputs (512 MiB) are larger than
the 129 MB L2, so no flush is needed between calls.

Prints one JSON line (rank 0).  Other workloads (--workload) print the same
line for the other configurations.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
"""
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

import numpy as np  # noqa: E402

import hc_inputs  # noqa: E402

METRIC = "AllReduce effective algbw GB/s and % of HBM roofline vs P, size, algo (1xGB300)"

WORKLOADS = {
    "ring_fp32_p8": dict(desc="Ring AllReduce sum, P=8 virtual ranks, fp32, 16,777,216 elements "
                              "per rank (64 MiB), N(0,1)*1e-3, fused mode, out of place",
                         algo="ring", coll="allreduce", P=8, n=16777216, dtype="float32", op="sum",
                         mode="fused", p_intra=1, loop_bytes=0, scale=1e-3),
    "ring_fp32_p8_step": dict(desc="Ring AllReduce sum, P=8, fp32, 16,777,216 elements per rank, "
                                   "step-faithful mode (14 launches)",
                              algo="ring", coll="allreduce", P=8, n=16777216, dtype="float32",
                              op="sum", mode="step", p_intra=1, loop_bytes=0, scale=1e-3),
    "ring_fp32_p8_rs": dict(desc="Ring ReduceScatter sum, P=8, fp32, 16,777,216 elements per rank, fused",
                            algo="ring", coll="reducescatter", P=8, n=16777216, dtype="float32",
                            op="sum", mode="fused", p_intra=1, loop_bytes=0, scale=1e-3),
    "ring_fp32_p8_ag": dict(desc="Ring AllGather, P=8, fp32, 16,777,216 elements per rank, fused, "
                                 "out of place",
                            algo="ring", coll="allgather", P=8, n=16777216, dtype="float32",
                            op="sum", mode="fused", p_intra=1, loop_bytes=0, scale=1e-3),
    "ring_bf16_p8": dict(desc="Ring AllReduce sum, P=8, bf16 (per-step rounding), 67,108,864 "
                              "elements per rank (128 MiB), N(0,1)*1e-2, fused",
                         algo="ring", coll="allreduce", P=8, n=67108864, dtype="bfloat16", op="sum",
                         mode="fused", p_intra=1, loop_bytes=0, scale=1e-2),
    "rhd_bf16_p8": dict(desc="RHD AllReduce sum, P=8, bf16, 67,108,864 elements per rank, fused",
                        algo="rhd", coll="allreduce", P=8, n=67108864, dtype="bfloat16", op="sum",
                        mode="fused", p_intra=1, loop_bytes=0, scale=1e-2),
    "rhd_bf16_p8_max": dict(desc="RHD AllReduce max, P=8, bf16, 67,108,864 elements per rank, fused",
                            algo="rhd", coll="allreduce", P=8, n=67108864, dtype="bfloat16",
                            op="max", mode="fused", p_intra=1, loop_bytes=0, scale=1e-2),
    "pipe_fp32_4x8": dict(desc="Pipeline AllReduce sum, 4 servers x 8 ranks (P=32), fp32, "
                               "8,388,608 elements per rank (32 MiB), N(0,1)*1e-3, fused",
                          algo="pipeline", coll="allreduce", P=32, n=8388608, dtype="float32",
                          op="sum", mode="fused", p_intra=8, loop_bytes=0, scale=1e-3),
    "pipe_fp32_4x8_step": dict(desc="Pipeline AllReduce sum, 4x8, fp32, 8,388,608 elements per "
                                    "rank, step mode, 64 MiB loop limit (4 loops, tail 37,504)",
                               algo="pipeline", coll="allreduce", P=32, n=8388608,
                               dtype="float32", op="sum", mode="step", p_intra=8,
                               loop_bytes=64 << 20, scale=1e-3),
    "hier_fp32_4x8": dict(desc="Plain hierarchical AllReduce sum (mesh RS, inter-server RHD AR, "
                               "mesh AG), 4 servers x 8 ranks (P=32), fp32, 8,388,608 elements per "
                               "rank, fused",
                          algo="hier", coll="allreduce", P=32, n=8388608, dtype="float32",
                          op="sum", mode="fused", p_intra=8, loop_bytes=0, scale=1e-3),
    "hier_fp32_4x8_step": dict(desc="Plain hierarchical AllReduce sum, 4x8, fp32, 8,388,608 "
                                    "elements per rank, step mode (6 launches)",
                               algo="hier", coll="allreduce", P=32, n=8388608, dtype="float32",
                               op="sum", mode="step", p_intra=8, loop_bytes=0, scale=1e-3),
    "rhd_fp32_p8_small": dict(desc="RHD AllReduce sum, P=8, fp32, 4096 elements per rank "
                                   "(latency regime, L2-resident), fused",
                              algo="rhd", coll="allreduce", P=8, n=4096, dtype="float32",
                              op="sum", mode="fused", p_intra=1, loop_bytes=0, scale=1.0),
    "rhd_fp32_p8_small_step": dict(desc="RHD AllReduce sum, P=8, fp32, 4096 elements per rank, "
                                        "step mode (6 launches)",
                                   algo="rhd", coll="allreduce", P=8, n=4096, dtype="float32",
                                   op="sum", mode="step", p_intra=1, loop_bytes=0, scale=1.0),
}


def _add(name, desc, algo, coll, P, n, dtype, op, mode, p_intra=1, loop_bytes=0, scale=1e-3):
    WORKLOADS[name] = dict(desc=desc, algo=algo, coll=coll, P=P, n=n, dtype=dtype, op=op, mode=mode,
                           p_intra=p_intra, loop_bytes=loop_bytes, scale=scale)


# the rest of the benchmark's configurations, each a workload of its own
_add("ring_fp32_p8_rs_step", "Ring ReduceScatter sum, P=8, fp32, 16,777,216 elements per rank, "
     "step mode, out of place (caller scratch)", "ring", "reducescatter", 8, 16777216, "float32",
     "sum", "step")
_add("ring_fp32_p8_ag_step", "Ring AllGather, P=8, fp32, 16,777,216 elements per rank, step mode, "
     "out of place", "ring", "allgather", 8, 16777216, "float32", "sum", "step")
for _a in ("ring", "rhd"):
    for _o in ("sum", "max"):
        for _m in ("fused", "step"):
            _k = "%s_bf16_p8%s%s" % (_a, "" if _o == "sum" else "_max", "" if _m == "fused" else "_step")
            if _k not in WORKLOADS:
                _add(_k, "%s AllReduce %s, P=8, bf16 (per-step rounding), 67,108,864 elements per "
                     "rank (128 MiB), N(0,1)*1e-2, %s mode" % (_a.upper() if _a == "rhd" else "Ring",
                                                               _o, _m),
                     _a, "allreduce", 8, 67108864, "bfloat16", _o, _m, scale=1e-2)
for _c, _t in (("reducescatter", "rs"), ("allgather", "ag")):
    _add("pipe_fp32_4x8_%s" % _t, "Pipeline %s, 4 servers x 8 ranks (P=32), fp32, 8,388,608 "
         "elements per rank, fused" % ("ReduceScatter" if _t == "rs" else "AllGather"),
         "pipeline", _c, 32, 8388608, "float32", "sum", "fused", p_intra=8)
    _add("pipe_fp32_4x8_%s_step" % _t, "Pipeline %s, 4x8, fp32, 8,388,608 elements per rank, step "
         "mode, 64 MiB loop limit (4 loops, tail 37,504)" % ("ReduceScatter" if _t == "rs" else
                                                             "AllGather"),
         "pipeline", _c, 32, 8388608, "float32", "sum", "step", p_intra=8, loop_bytes=64 << 20)

# The configurations timed in one default run (N = 1), grouped by their
# input buffers (each group's rank vectors are drawn once).
SWEEP = [
    ["ring_fp32_p8_step", "ring_fp32_p8_rs", "ring_fp32_p8_rs_step", "ring_fp32_p8_ag",
     "ring_fp32_p8_ag_step"],
    ["ring_bf16_p8", "ring_bf16_p8_max", "rhd_bf16_p8", "rhd_bf16_p8_max", "ring_bf16_p8_step",
     "ring_bf16_p8_max_step", "rhd_bf16_p8_step", "rhd_bf16_p8_max_step"],
    ["pipe_fp32_4x8", "pipe_fp32_4x8_rs", "pipe_fp32_4x8_ag", "pipe_fp32_4x8_step",
     "pipe_fp32_4x8_rs_step", "pipe_fp32_4x8_ag_step", "hier_fp32_4x8", "hier_fp32_4x8_step"],
]
DTYPE_TAG = {"float32": "f32", "bfloat16": "bf16", "int32": "int32"}
ESIZE = {"float32": 4, "bfloat16": 2, "int32": 4}
KERNEL_DIR = os.path.join(ROOT, "collective_communication_algorithms_gb300", "csrc")
KERNEL_FILES = ("hc_device.cuh", "hc_kernels.cu", "hc_fused_ring.cu", "hc_fused_rhd.cu",
                "hc_fused_pipe.cu", "hc_fused_hier.cu")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="ring_fp32_p8", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configurations (the `configs` array of the line)")
    ap.add_argument("--sweep", choices=["small", "select", "hostlink", "hbm"], default=None,
                    help="small: RHD AllReduce latency sweep (P x n), eager vs graph mode; "
                         "select: cost-model selector against measured times; "
                         "hostlink: the default workload with pinned host buffers, zero-copy "
                         "against staged copies; hbm: write-only and copy bandwidth of the "
                         "device (torch kernels) beside the AllGather")
    return ap.parse_args()


def algorithmic_bytes(w):
    """Minimum bytes one fused call moves (reads + writes)."""
    P, n, b = w["P"], w["n"], ESIZE[w["dtype"]]
    if w["coll"] == "allreduce":
        return 2 * P * n * b
    if w["coll"] == "reducescatter":
        return (P + 1) * n * b
    return (P + 1) * n * b  # allgather out of place


def inputs_for(w, n=None, seed=0):
    n = w["n"] if n is None else n
    if w["dtype"] == "float32":
        return hc_inputs.gradients_f32(w["P"], n, seed=seed, scale=w["scale"])
    if w["dtype"] == "bfloat16":
        return hc_inputs.gradients_bf16(w["P"], n, seed=seed, scale=w["scale"])
    return hc_inputs.uniform_int32(w["P"], n, seed=seed)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash():
    """sha256 prefix over every device source file, in a fixed order."""
    h = hashlib.sha256()
    for name in KERNEL_FILES:
        with open(os.path.join(KERNEL_DIR, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def l2_note(coll, P, rank_bytes):
    """How the timed steps avoid reusing the 129 MB L2: the inputs (P n b for
    AllReduce and ReduceScatter, n b for AllGather) are larger than it, or
    every step writes more than it (AllGather: P n b), which evicts the
    inputs between steps."""
    l2 = 129 << 20
    inputs = rank_bytes if coll == "allgather" else P * rank_bytes
    if inputs > l2:
        return "inputs (%d MiB) larger than the 129 MB L2; no flush" % (inputs >> 20)
    if coll == "allgather" and P * rank_bytes > l2:
        return ("inputs %d MiB; every step writes %d MiB (more than the 129 MB L2), which evicts "
                "them between steps; no other flush" % (inputs >> 20, (P * rank_bytes) >> 20))
    return "L2-resident (hot-cache latency regime)"


def hold_device(steps):
    """Queue a spin kernel on the current stream ahead of a timed region, so
    that the host enqueues all `steps` calls before the device starts them
    and the events time the device work, not the host's launch rate (one
    call from Python takes tens of microseconds, about as long as a 0.1 ms
    collective).  About 0.2 ms per step at 2 GHz."""
    import torch
    torch.cuda._sleep(int(4e5 * max(steps, 10)))


def traffic_from_profiles(workload):
    """DRAM read + write bytes of one call (fused mode: its one launch; step
    mode: all its launches) from a committed ncu summary, if it was taken on
    the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t.get(workload)
        if e and e.get("kernel_source_sha256_16") == kernel_source_hash():
            return float(e.get("dram_bytes_per_call", e["dram_bytes_per_launch"]))
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------
# clocks sampled with nvidia-smi while the GPU runs the step
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_uuid):
        self.proc = None
        self.out = os.path.join("/tmp", "hc_bench_clocks_%d.csv" % os.getpid())
        cmd = ["nvidia-smi", "--query-gpu=" + CLOCK_FIELDS, "--format=csv,noheader,nounits",
               "-lms", "100"]
        if device_uuid:
            cmd += ["-i", device_uuid]
        try:
            self.f = open(self.out, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"error": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.out) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for name, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(name)
        os.remove(self.out)
        if not sm:
            return {"error": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# replicas: one process per GPU, each running the whole collective on its own
# buffers (no data-path exchange); the job's time is the slowest rank's
# ---------------------------------------------------------------------------
def max_over_ranks(values, world, device):
    """Element-wise maximum of a list of floats over all ranks of the
    default process group (the values themselves when world == 1)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def replica_algbw(world, bytes_per_rank, ms):
    """Whole-job algbw in GB/s: every replica moves bytes_per_rank of
    per-rank data in ms (the slowest rank's time)."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
class Collective:
    """One workload's device buffers and its call through the C ABI.
    send: the (P, n) rank vectors on the device (bf16 as int16 bits); the
    outputs are new (P, n) rows (AllReduce, AllGather) or one buffer per
    segment (ReduceScatter), all out of place; a step-mode ReduceScatter gets
    the scratch hc_scratch_bytes asks for."""

    def __init__(self, B, w, send, stream):
        import torch
        P, n, dt = w["P"], w["n"], w["dtype"]
        self.B, self.w, self.stream = B, w, stream
        self.send = send
        self.recv = torch.empty_like(send)
        send_p = [send[r].data_ptr() for r in range(P)]
        recv_p = [self.recv[r].data_ptr() for r in range(P)]
        self.segs = self.rs_out = self.ag_in = self.scratch = None
        if w["coll"] in ("reducescatter", "allgather"):
            self.segs = [B.hc_segment_range(w["algo"], w["coll"], P, n, dt, k) for k in range(P)]
        if w["coll"] == "reducescatter":
            self.rs_out = [torch.empty(max(ln, 8), dtype=send.dtype, device=send.device)
                           for _, ln in self.segs]
            recv_p = [t.data_ptr() for t in self.rs_out]
        if w["coll"] == "allgather":
            self.ag_in = [send[k, off:off + ln].clone() for k, (off, ln) in enumerate(self.segs)]
            send_p = [t.data_ptr() for t in self.ag_in]
        sb = 0
        if w["coll"] == "reducescatter" and w["mode"] == "step":
            sb = B.hc_scratch_bytes(w["algo"], P, n, dt)
            self.scratch = torch.empty(sb, dtype=torch.uint8, device=send.device)
        self.opts = B.make_opts(w["mode"], ranks_per_server=w["p_intra"],
                                max_loop_bytes=w["loop_bytes"],
                                scratch=self.scratch.data_ptr() if sb else 0, scratch_bytes=sb)
        self.sp, self.rp = B.ptr_array(send_p), B.ptr_array(recv_p)

    def __call__(self):
        B, w = self.B, self.w
        P, n, dt = w["P"], w["n"], w["dtype"]
        if w["coll"] == "allreduce":
            B.hc_allreduce(self.sp, self.rp, P, n, dt, w["op"], w["algo"], self.opts, self.stream)
        elif w["coll"] == "reducescatter":
            B.hc_reduce_scatter(self.sp, self.rp, P, n, dt, w["op"], w["algo"], self.opts,
                                self.stream)
        else:
            B.hc_allgather(self.sp, self.rp, P, n, dt, w["algo"], self.opts, self.stream)


def step_call_stats(B, w):
    """(kernel launches, bytes the step kernels read + write) of one
    out-of-place step-mode call of workload w, from its exported plan: every
    record moves (hi - lo) elements of each input, the accumulator and each
    output."""
    recs, launches = B.hc_step_plan(w["algo"], w["coll"], w["P"], w["n"], w["dtype"], w["p_intra"],
                                    w["loop_bytes"], in_place=False)
    b = ESIZE[w["dtype"]]
    moved = sum((r["hi"] - r["lo"]) * b * (len(r["in_ranks"]) + (r["acc_rank"] >= 0) +
                                          len(r["out_ranks"])) for r in recs)
    return launches, moved


def time_device(call, steps, warmup, stream):
    """W untimed calls, then K calls queued behind a spin kernel and timed
    with CUDA events on the launch stream: (ms per call over the whole
    region, mean ms between the events around each call)."""
    import torch
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ka = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    hold_device(steps)
    ev0.record(stream)
    for i in range(steps):
        ka[i].record(stream)
        call()
        kb[i].record(stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    return (ev0.elapsed_time(ev1) / steps,
            statistics.mean(a.elapsed_time(bb) for a, bb in zip(ka, kb)))


def time_queued(call, reps, stream):
    """Device microseconds per call of `reps` calls queued behind a spin
    kernel, with CUDA events only around the whole batch (events between
    calls would break the launches' programmatic overlap and, for calls of a
    few microseconds, dominate them)."""
    import torch
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    hold_device(reps)
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps * 1e3


def config_sweep(args, dev):
    """Every configuration of the benchmark besides the headline, timed like
    it: the large ones (SWEEP) as algbw and fraction of the copy peak, the
    latency regime (int32 P = 4 Ring and P = 5 RHD at 4096 elements; RHD fp32
    P in {5, 8, 12, 16} x 256 .. 16384 elements) as microseconds per call."""
    import torch
    from collective_communication_algorithms_gb300 import _binding as B
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    peak, _ = measured_peak()
    out = []
    for group in SWEEP:
        w0 = WORKLOADS[group[0]]
        X = inputs_for(w0)
        Xd = torch.from_numpy(X.view(np.int16) if w0["dtype"] == "bfloat16" else X).to(dev)
        del X
        for name in group:
            w = WORKLOADS[name]
            P, n, dt = w["P"], w["n"], w["dtype"]
            c = Collective(B, w, Xd, sh)
            if w["mode"] == "fused":
                launches, alg = 1, algorithmic_bytes(w)
            else:
                launches, alg = step_call_stats(B, w)
            ms, kern = time_device(c, args.steps, args.warmup, stream)
            out.append({"name": name, "workload": w["desc"],
                        "value": round(n * ESIZE[dt] / (ms * 1e-3) / 1e9, 3), "unit": "GB/s",
                        "ms_per_call": round(ms, 5), "kernel_ms": round(kern, 5),
                        "bytes_per_call": alg, "bytes": "fused minimum" if w["mode"] == "fused"
                        else "step mode's own (inputs + accumulator + outputs of every step)",
                        "achieved_GBps": round(alg / (kern * 1e-3) / 1e9, 1),
                        "frac": round(alg / (kern * 1e-3) / 1e9 / peak, 4),
                        "traffic": traffic_from_profiles(name), "launches_per_call": launches,
                        "l2": l2_note(w["coll"], P, n * ESIZE[dt])})
            del c
        del Xd
        torch.cuda.empty_cache()
    out += latency_sweep(B, dev)
    return out


def latency_sweep(B, dev, reps=100):
    """Per-call microseconds of small in-place AllReduces (hot L2): `eager`
    is back-to-back calls from Python (host and device overlap, so the
    slower of the two decides), `eager_bound` the same with the arguments
    converted once (_binding.bind_allreduce), `queued` the same calls
    enqueued behind a spin kernel (the device's own time per call), `graph`
    one CUDA graph of `reps` calls (graph mode) launched once."""
    import math
    import torch
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    points = [("int32_ring_p4", "ring", "int32", 4, 4096), ("int32_rhd_p5", "rhd", "int32", 5, 4096)]
    points += [("rhd_fp32_small", "rhd", "float32", P, n)
               for P in (5, 8, 12, 16) for n in (256, 512, 1024, 2048, 4096, 8192, 16384)]
    out = []
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for name, algo, dt, P, n in points:
        X = hc_inputs.uniform_int32(P, n, seed=0) if dt == "int32" else \
            hc_inputs.gradients_f32(P, n, seed=0, scale=1.0)
        xd = torch.from_numpy(X).to(dev)
        ptrs = B.ptr_array([xd[r].data_ptr() for r in range(P)])
        st, _ = B.hc_schedule_stats(algo, "allreduce", P, n, dt)
        line = {"name": name, "algo": algo, "dtype": dt, "P": P, "elements_per_rank": n,
                "steps": st["steps_per_loop"], "two_ceil_log2_P": 2 * math.ceil(math.log2(P)),
                "launches_step": st["launches_step"], "unit": "us per call"}
        for mode in ("fused", "step"):
            opts = B.make_opts(mode)

            def call():
                B.hc_allreduce(ptrs, ptrs, P, n, dt, "sum", algo, opts, sh)
            for _ in range(5):
                call()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(reps):
                call()
            e1.record(stream)
            torch.cuda.synchronize()
            line[mode + "_eager_us"] = round(e0.elapsed_time(e1) / reps * 1e3, 2)
            # the same from Python with the arguments converted once
            bound = B.bind_allreduce(ptrs, ptrs, P, n, dt, "sum", algo, opts, sh)
            bound()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(reps):
                bound()
            e1.record(stream)
            torch.cuda.synchronize()
            line[mode + "_eager_bound_us"] = round(e0.elapsed_time(e1) / reps * 1e3, 2)
            hold_device(reps)
            e0.record(stream)
            for _ in range(reps):
                call()
            e1.record(stream)
            torch.cuda.synchronize()
            line[mode + "_queued_us"] = round(e0.elapsed_time(e1) / reps * 1e3, 2)
            g = B.Graph()
            for _ in range(reps):
                g.add_allreduce(ptrs, ptrs, P, n, dt, "sum", algo, opts)
            g.build()
            g.launch(sh)
            torch.cuda.synchronize()
            e0.record(stream)
            g.launch(sh)
            e1.record(stream)
            torch.cuda.synchronize()
            line[mode + "_graph_us"] = round(e0.elapsed_time(e1) / reps * 1e3, 2)
            g.close()
        out.append(line)
    return out


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from collective_communication_algorithms_gb300 import _binding as B
    B.lib()  # loud failure if the library is missing

    P, n, dt = w["P"], w["n"], w["dtype"]
    b = ESIZE[dt]
    X = inputs_for(w)
    Xt = torch.from_numpy(X.view(np.int16) if dt == "bfloat16" else X)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    coll = Collective(B, w, Xt.to(dev), sh)
    send, recv, rs_out, ag_in, segs, call = coll.send, coll.recv, coll.rs_out, coll.ag_in, coll.segs, coll
    if w["mode"] == "fused":
        launches, step_bytes = 1, None
    else:
        launches, step_bytes = step_call_stats(B, w)

    # warm-up, then a sustained run of the same step while clocks are sampled
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    t_end = time.time() + 1.5
    while time.time() < t_end:
        for _ in range(20):
            call()
        torch.cuda.synchronize()

    # timed region: exactly K steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ka = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    hold_device(args.steps)
    ev0.record(stream)
    for i in range(args.steps):
        ka[i].record(stream)
        call()
        kb[i].record(stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = ev0.elapsed_time(ev1)
    kern_ms = [a.elapsed_time(bb) for a, bb in zip(ka, kb)]
    total_ms, kern_avg = max_over_ranks([total_ms, statistics.mean(kern_ms)], world, dev)
    ms_per_step = total_ms / args.steps
    value = replica_algbw(world, n * b, ms_per_step)

    # end to end through the C ABI with host buffers (pinned), copies timed
    e2e = None
    if not args.no_e2e:
        Xh = Xt.pin_memory()
        Yh = torch.empty((P, n), dtype=Xt.dtype).pin_memory()
        if w["mode"] == "fused":
            # one call on the pinned host buffers (hc_opts_t.host_buffers):
            # the kernel pulls every input over the host link and pushes
            # every output back, no staging copies
            hopts = B.make_opts("fused", ranks_per_server=w["p_intra"], host_buffers=True)
            hs = [Xh[r].data_ptr() for r in range(P)]
            hr = [Yh[r].data_ptr() for r in range(P)]
            if w["coll"] == "allreduce":
                h2d, d2h = P * n * b, P * n * b

                def e2e_step():
                    B.hc_allreduce(hs, hr, P, n, dt, w["op"], w["algo"], hopts, sh)
            elif w["coll"] == "reducescatter":
                h2d, d2h = P * n * b, n * b
                hr = [Yh[r].data_ptr() + segs[r][0] * b for r in range(P)]

                def e2e_step():
                    B.hc_reduce_scatter(hs, hr, P, n, dt, w["op"], w["algo"], hopts, sh)
            else:
                h2d, d2h = n * b, P * n * b
                hs = [Xh[k].data_ptr() + segs[k][0] * b for k in range(P)]

                def e2e_step():
                    B.hc_allgather(hs, hr, P, n, dt, w["algo"], hopts, sh)
            e2e_path = "one fused call on pinned host buffers (host_buffers=1)"
        elif w["coll"] == "allreduce":
            h2d, d2h = P * n * b, P * n * b

            def e2e_step():
                send.copy_(Xh, non_blocking=True)
                call()
                Yh.copy_(recv, non_blocking=True)
        elif w["coll"] == "reducescatter":
            h2d, d2h = P * n * b, n * b

            def e2e_step():
                send.copy_(Xh, non_blocking=True)
                call()
                for r in range(P):
                    ln = segs[r][1]
                    Yh[r, :ln].copy_(rs_out[r][:ln], non_blocking=True)
        else:
            h2d, d2h = n * b, P * n * b

            def e2e_step():
                for k, (off, ln) in enumerate(segs):
                    ag_in[k].copy_(Xh[k, off:off + ln], non_blocking=True)
                call()
                Yh.copy_(recv, non_blocking=True)
        if w["mode"] != "fused":
            e2e_path = "pinned host -> device copy, step-mode call, device -> pinned host copy"
        for _ in range(max(2, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1) / args.steps
        # the host-side results must equal the device-side ones bit for bit
        if w["coll"] == "reducescatter":
            same = all(torch.equal(Yh[r, segs[r][0]:segs[r][0] + segs[r][1]],
                                   rs_out[r][:segs[r][1]].cpu()) for r in range(P))
        else:
            same = torch.equal(Yh, recv.cpu())
        if not same:
            raise SystemExit("e2e outputs differ from the device-buffer outputs")
        e_ms = max_over_ranks([e_ms], world, dev)[0]
        e2e = {"value": round(replica_algbw(world, n * b, e_ms), 3), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e_ms, 4), "path": e2e_path}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, budget_s=10.0)

    # every other configuration of the benchmark, with clocks sampled over
    # the whole sweep (one GPU only: replicas would repeat it)
    configs = configs_clocks = None
    if world == 1 and not args.no_configs:
        del coll, send, recv, rs_out, ag_in, call
        torch.cuda.empty_cache()
        sweep_sampler = ClockSampler(uuid)
        configs = config_sweep(args, dev)
        configs_clocks = sweep_sampler.stop()

    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return
    peak, peak_kind = measured_peak()
    alg = algorithmic_bytes(w) if w["mode"] == "fused" else step_bytes
    achieved = alg / (kern_avg * 1e-3) / 1e9
    traffic = traffic_from_profiles(args.workload)
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": DTYPE_TAG[dt],
        "data": "synthetic (seeded N(0,1) gradients, numpy PCG64 seed 0)",
        "config": {"workload": w["desc"], "algo": w["algo"], "collective": w["coll"], "P": P,
                   "elements_per_rank": n, "mode": w["mode"], "op": w["op"],
                   "ranks_per_server": w["p_intra"], "max_loop_bytes": w["loop_bytes"],
                   "l2": l2_note(w["coll"], P, n * b),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "clock_window": "1.5 s sustained run of the same step + the timed steps"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "peak_kind": peak_kind + " (hbm_gbs, copy burst)",
                     "algorithmic_bytes_per_launch": alg // max(1, launches) if w["mode"] == "step" else alg,
                     "kernel_ms": round(kern_avg, 5),
                     "frac_of_8TBps_nominal": round(achieved / 8000.0, 4)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * launches,
        "clocks": clocks,
        "configs": configs,
        "configs_clocks": configs_clocks,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample_n(w, n_target):
    A = 16 // ESIZE[w["dtype"]]
    S = w["P"]
    return max(S * A, (n_target // (S * A)) * S * A)


def time_oracle_once(w, X):
    import oracle as O
    t0 = time.perf_counter()
    O.replay(w["algo"], w["coll"], X, w["op"], w["dtype"], p_intra=w["p_intra"])
    return time.perf_counter() - t0


# ---------------------------------------------------------------------------
# the oracle on every host core: one spawned process per core, each replaying
# the same schedule on its own seeded sample of the workload; two barriers
# bracket every round, so a round's wall time covers all processes' replays
# ---------------------------------------------------------------------------
BARRIER_S = 600


def _oracle_worker(w, ns, seed, rounds, start, end):
    try:
        X = inputs_for(w, ns, seed=seed)
        time_oracle_once(w, X)  # load the library and page the inputs in
        for _ in range(rounds):
            start.wait(timeout=BARRIER_S)
            time_oracle_once(w, X)
            end.wait(timeout=BARRIER_S)
    except Exception:
        start.abort()
        end.abort()
        raise


class ParallelOracle:
    """`procs` spawned processes (spawn: safe after CUDA initialisation)."""

    def __init__(self, w, ns, procs, rounds):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.start = ctx.Barrier(procs + 1)
        self.end = ctx.Barrier(procs + 1)
        self.procs = [ctx.Process(target=_oracle_worker, daemon=True,
                                  args=(w, ns, 1000 + k, rounds, self.start, self.end))
                      for k in range(procs)]
        for p in self.procs:
            p.start()

    def round(self):
        self.start.wait(timeout=BARRIER_S)
        t0 = time.perf_counter()
        self.end.wait(timeout=BARRIER_S)
        return time.perf_counter() - t0

    def close(self):
        for p in self.procs:
            p.join(timeout=60)


def host_procs():
    return max(1, os.cpu_count() or 1)


def cpu_baseline(w, budget_s=5.0, parallel_s=8.0):
    ns = oracle_sample_n(w, 1 << 21)
    X = inputs_for(w, ns)
    b = ESIZE[w["dtype"]]
    times = []
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < budget_s or len(times) < 2:
        times.append(time_oracle_once(w, X))
        if len(times) >= 50:
            break
    t1 = statistics.median(times)
    procs = host_procs()
    rounds = max(3, min(50, int(round(parallel_s / t1))))
    po = ParallelOracle(w, ns, procs, rounds)
    rt = [po.round() for _ in range(rounds)]
    po.close()
    tp = statistics.median(rt)
    return {"value": round(procs * ns * b / tp / 1e9, 5), "unit": "GB/s", "cores": procs,
            "kind": "oracle",
            "sample": "step-by-step replay of the same schedule, one process per host core, each "
                      "on its own seeded sample of %d elements of each of the %d rank vectors; "
                      "median of %d rounds (%.1f s)" % (ns, w["P"], rounds, sum(rt)),
            "single_thread": {"value": round(ns * b / t1 / 1e9, 5), "cores": 1,
                              "sample": "the first %d elements of each rank vector, median of "
                                        "%d runs (%.1f s)" % (ns, len(times), sum(times))},
            "cpu": cpu_model()}


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip() + ", %d cores" % os.cpu_count()
    except Exception:
        pass
    return "%d cores" % os.cpu_count()


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    ns = oracle_sample_n(w, 1 << 20)
    procs = host_procs()
    po = ParallelOracle(w, ns, procs, args.warmup + args.steps)
    for _ in range(args.warmup):
        po.round()
    total = sum(po.round() for _ in range(args.steps))
    po.close()
    ms = total / args.steps * 1e3
    value = procs * ns * ESIZE[w["dtype"]] / (ms * 1e-3) / 1e9
    sample = ("oracle step-by-step replay (plain C) of the same schedule, one process per host "
              "core (%d), each on its own seeded sample of %d elements of each of the %d rank "
              "vectors per step" % (procs, ns, w["P"]))
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 5),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": DTYPE_TAG[w["dtype"]],
        "data": "synthetic (seeded N(0,1) gradients, numpy PCG64 seed 0)",
        "config": {"workload": w["desc"], "algo": w["algo"], "collective": w["coll"],
                   "P": w["P"], "elements_per_rank": w["n"], "mode": "oracle",
                   "sample_elements_per_rank": ns},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": procs,
                         "kind": "oracle", "sample": sample, "cpu": cpu_model()},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def sweep_small(args):
    """RHD AllReduce sum fp32, P in {5, 8, 12, 16}, n = 256 .. 16384: per-call
    time eager (one host call per collective) and in graph mode (a graph of
    `reps` dependent in-place AllReduces launched once), fused and step mode;
    steps per call against ceil(log2 P).  Hot L2 (the data is tiny)."""
    import math
    import torch
    from collective_communication_algorithms_gb300 import _binding as B
    torch.cuda.set_device(0)
    B.lib()
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    reps = 200
    for P in (5, 8, 12, 16):
        for n in (256, 512, 1024, 2048, 4096, 8192, 16384):
            X = hc_inputs.gradients_f32(P, n, seed=0, scale=1.0)
            dev = torch.from_numpy(X).cuda()
            ptrs = [dev[r].data_ptr() for r in range(P)]
            st, _ = B.hc_schedule_stats("rhd", "allreduce", P, n, "float32")
            line = {"sweep": "small", "algo": "rhd", "P": P, "elements_per_rank": n,
                    "steps": st["steps_per_loop"], "ceil_log2_P": math.ceil(math.log2(P)),
                    "launches_step": st["launches_step"]}
            for mode in ("fused", "step"):
                opts = B.make_opts(mode)
                for _ in range(5):
                    B.hc_allreduce(ptrs, ptrs, P, n, "float32", "sum", "rhd", opts, sh)
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    B.hc_allreduce(ptrs, ptrs, P, n, "float32", "sum", "rhd", opts, sh)
                e1.record(stream)
                torch.cuda.synchronize()
                line["eager_%s_us" % mode] = round(e0.elapsed_time(e1) / reps * 1e3, 2)
                g = B.Graph()
                for _ in range(reps):
                    g.add_allreduce(ptrs, ptrs, P, n, "float32", "sum", "rhd", opts)
                g.build()
                g.launch(sh)
                torch.cuda.synchronize()
                e0.record(stream)
                g.launch(sh)
                e1.record(stream)
                torch.cuda.synchronize()
                line["graph_%s_us" % mode] = round(e0.elapsed_time(e1) / reps * 1e3, 2)
                g.close()
            print(json.dumps(line), flush=True)


def sweep_select(args):
    """For each (collective, P, ranks per server, n, mode) time every
    candidate schedule and compare the cost model's choice and prediction
    with the measured best.  Each candidate's time is the device time per
    call of calls queued behind a spin kernel (the cost model predicts for a
    caller whose launches keep the device busy), the best of three rounds
    that visit the candidates in turn."""
    import torch
    from collective_communication_algorithms_gb300 import _binding as B
    torch.cuda.set_device(0)
    B.lib()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    cases = []
    for coll in ("allreduce", "reducescatter", "allgather"):
        for P, rps in ((8, 1), (32, 8)):
            for n in (4096, 262144, 4194304):
                for mode in ("step", "fused"):
                    cases.append((coll, P, rps, n, mode))
    for coll, P, rps, n, mode in cases:
        X = torch.from_numpy(hc_inputs.gradients_f32(P, n, seed=0, scale=1e-3)).to(dev)
        cands = ["ring", "rhd"] + (["pipeline"] if rps > 1 else []) + \
            (["hier"] if rps > 1 and coll == "allreduce" else [])
        pick, pred = B.hc_select_algo(coll, P, n, "float32", mode, rps)
        calls = {}
        for algo in cands:
            w = dict(algo=algo, coll=coll, P=P, n=n, dtype="float32", op="sum", mode=mode,
                     p_intra=rps if algo in ("pipeline", "hier") else 1, loop_bytes=0)
            calls[algo] = Collective(B, w, X, sh)
        reps = 100 if n <= 262144 else 20
        meas = {a: float("inf") for a in cands}
        for _ in range(3):
            for algo in cands:
                meas[algo] = min(meas[algo], time_queued(calls[algo], reps, stream))
        best = min(meas, key=meas.get)
        line = {"sweep": "select", "collective": coll, "P": P, "ranks_per_server": rps,
                "elements_per_rank": n, "mode": mode, "selected": pick,
                "predicted_us": round(pred, 2), "measured_us": {a: round(t, 2) for a, t in meas.items()},
                "measured_best": best,
                "selected_over_best": round(meas[pick] / meas[best], 3)}
        print(json.dumps(line), flush=True)
        del calls, X
        torch.cuda.empty_cache()


def sweep_hostlink(args):
    """The default workload (Ring AllReduce fp32 sum, P=8, 16,777,216
    elements per rank) with its inputs and outputs in pinned host memory:
    the copy engines alone and overlapped, the staged call (copy in, fused
    kernel, copy out) and the fused kernel on the host buffers
    (host_buffers=1), each checked bit for bit against the device path."""
    import torch
    from collective_communication_algorithms_gb300 import _binding as B
    w = WORKLOADS["ring_fp32_p8"]
    P, n, b = w["P"], w["n"], 4
    torch.cuda.set_device(0)
    B.lib()
    s0 = torch.cuda.current_stream()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    Xh = torch.from_numpy(inputs_for(w)).pin_memory()
    Yh = torch.empty_like(Xh).pin_memory()
    Xd = Xh.to("cuda")
    Yd = torch.empty_like(Xd)
    Zd = torch.empty_like(Xd)
    dev_opts = B.make_opts("fused")
    host_opts = B.make_opts("fused", host_buffers=True)

    def ar(x, y, opts):
        B.hc_allreduce([x[r].data_ptr() for r in range(P)], [y[r].data_ptr() for r in range(P)],
                       P, n, "float32", "sum", "ring", opts, s0.cuda_stream)

    def both_directions():
        ev = torch.cuda.Event()
        ev.record(s0)
        s1.wait_event(ev)
        s2.wait_event(ev)
        with torch.cuda.stream(s1):
            Zd.copy_(Xh, non_blocking=True)
        with torch.cuda.stream(s2):
            Yh.copy_(Yd, non_blocking=True)
        for s in (s1, s2):
            e = torch.cuda.Event()
            e.record(s)
            s0.wait_event(e)

    def staged():
        Xd.copy_(Xh, non_blocking=True)
        ar(Xd, Yd, dev_opts)
        Yh.copy_(Yd, non_blocking=True)

    ar(Xd, Yd, dev_opts)
    torch.cuda.synchronize()
    ref = Yd.cpu()
    cases = [("h2d copy, 512 MiB", lambda: Xd.copy_(Xh, non_blocking=True), None),
             ("d2h copy, 512 MiB", lambda: Yh.copy_(Yd, non_blocking=True), None),
             ("h2d and d2h copies on two streams", both_directions, None),
             ("staged: h2d copy, fused kernel, d2h copy", staged, lambda: Yh),
             ("fused kernel, device buffers", lambda: ar(Xd, Yd, dev_opts), lambda: Yd.cpu()),
             ("fused kernel, host inputs, device outputs", lambda: ar(Xh, Yd, host_opts),
              lambda: Yd.cpu()),
             ("fused kernel, device inputs, host outputs", lambda: ar(Xd, Yh, host_opts),
              lambda: Yh),
             ("fused kernel, host inputs and outputs", lambda: ar(Xh, Yh, host_opts),
              lambda: Yh)]
    for name, fn, out in cases:
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s0)
        for _ in range(args.steps):
            fn()
        e1.record(s0)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        line = {"sweep": "hostlink", "case": name, "ms": round(ms, 4),
                "algbw_GBps": round(n * b / ms / 1e6, 2)}
        if out is not None:
            line["bit_exact"] = bool(torch.equal(out(), ref))
            Yh.zero_()
            Yd.zero_()
        print(json.dumps(line), flush=True)


def sweep_hbm(args):
    """Device-memory ceilings for write-heavy collectives: torch's fill
    (write only), copy (read = write) and broadcast copy (one read, P = 8
    writes, the AllGather's mix) over 1 GiB; fill and sum (read only) over
    exactly the AllGather's write and read volumes; and the fused Ring
    AllGather fp32 P=8 (writes P bytes per byte read), in GB/s of bytes
    moved."""
    import torch
    from collective_communication_algorithms_gb300 import _binding as B
    torch.cuda.set_device(0)
    B.lib()
    s0 = torch.cuda.current_stream()
    nb = 1 << 30
    a = torch.empty(nb // 4, dtype=torch.float32, device="cuda")
    c = torch.empty_like(a)
    a.normal_()
    w = WORKLOADS["ring_fp32_p8_ag"]
    P, n = w["P"], w["n"]
    segs = [B.hc_segment_range("ring", "allgather", P, n, "float32", k) for k in range(P)]
    X = torch.from_numpy(inputs_for(w)).cuda()
    ag_in = [X[k, off:off + ln].clone() for k, (off, ln) in enumerate(segs)]
    Y = torch.empty_like(X)
    opts = B.make_opts("fused")
    src = a[:nb // 4 // P]
    dst = c.view(P, nb // 4 // P)
    cases = [("fill (write only), 1 GiB", lambda: c.fill_(1.0), nb),
             ("fill (write only), 512 MiB: the AllGather's writes P n b",
              lambda: c[:P * n].fill_(1.0), P * n * 4),
             ("sum (read only), 64 MiB: the AllGather's reads n b", lambda: a[:n].sum(), n * 4),
             ("copy (read 1 GiB, write 1 GiB)", lambda: c.copy_(a), 2 * nb),
             ("broadcast copy (read 128 MiB, write 8 x 128 MiB)",
              lambda: dst.copy_(src.expand(P, -1)), nb + nb // P),
             ("fused Ring AllGather fp32 P=8 (read n b, write P n b)",
              lambda: B.hc_allgather([t.data_ptr() for t in ag_in], [Y[r].data_ptr() for r in range(P)],
                                     P, n, "float32", "ring", opts, s0.cuda_stream),
              (P + 1) * n * 4)]
    for name, fn, moved in cases:
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        hold_device(args.steps)
        e0.record(s0)
        for _ in range(args.steps):
            fn()
        e1.record(s0)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        print(json.dumps({"sweep": "hbm", "case": name, "ms": round(ms, 4),
                          "GBps_moved": round(moved / ms / 1e6, 1)}), flush=True)


def main():
    args = parse_args()
    if args.sweep == "small":
        sweep_small(args)
        return
    if args.sweep == "select":
        sweep_select(args)
        return
    if args.sweep == "hostlink":
        sweep_hostlink(args)
        return
    if args.sweep == "hbm":
        sweep_hbm(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
