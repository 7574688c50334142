"""Benchmark of the normalization hot path on GB300 (one JSON line on rank 0).

One step = one pass of every hot-path operation over its workload:

  bn_f32_fwd   BatchNorm2d training forward  fp32 [256,32,32,32], |mean| <= 1000
  bn_f32_bwd   BatchNorm2d training backward fp32 [256,32,32,32]
  rms_bf16_bwd RMSNorm backward bf16 [2048, 8192]
  rms_f32_bwd  RMSNorm backward fp32 [2048, 8192]
  ln_bf16_bwd  bias+dropout+add+LayerNorm backward bf16 [16*512, 1600]
  bn_bf16_fwd  BatchNorm2d training forward  bf16 [128,256,56,56]
  bn_bf16_bwd  BatchNorm2d training backward bf16 [128,256,56,56]

Also available through --ops (not part of the default step, whose
operations are the configured workloads): rms_bf16_fwd, rms_f32_fwd
(RMSNorm training forward [2048, 8192]), ln_bf16_fwd (bias+dropout+add
LayerNorm training forward [16*512, 1600]), and the BatchNorm variants
bn_relu_{f32,bf16}_{fwd,bwd} (fused ReLU), bn_nhwc_{f32,bf16}_{fwd,bwd}
(channels-last, the same data permuted to [N,H,W,C]) and
bn_relu_nhwc_{f32,bf16}_{fwd,bwd}.

Every call goes through the C ABI (ctypes binding).  Each operation is timed
with CUDA events on the stream it runs on, after an L2 flush (a 256 MB write
then a 256 MB read of another buffer, outside the events).  BatchNorm runs
through the composite calls (bn_forward_train, bn_backward): one launch of the
persistent kernel for inputs of 128 MiB and more, two launches below.
value = unique bytes of every input and
output tensor of the step / summed device time (the effective-bandwidth
convention), in GB/s, over all ranks.  Each op also gets a warm-L2 time
(the same calls back to back, no flush; labelled, not used in value), and
the oracle baseline is reported on one thread and on every host core.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--ops a,b,...] [--no-e2e] [--no-cpu-baseline]

Under torchrun each rank runs the same workload on its own GPU (replicas; the
path needs no cross-GPU exchange); value sums the ranks' bytes over the
slowest rank's time.  ``--impl reference`` times the float64 CPU oracle on a
bounded sample of the same workload on the host cores (rank 0 only).
"""

import argparse
import gc
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "norm fwd+bwd effective HBM GB/s and % of GB300 peak; µs per call"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20

# Latency-bound BatchNorm shapes (the tiny [8,4,8,8] and the ragged
# [3,37,41,40] workloads): microseconds per call, eager and from a CUDA-graph
# replay, reported in `latency_ops` and kept out of `value`.
LATENCY_OPS = ["bn_tiny_f32_fwd", "bn_tiny_f32_bwd", "bn_ragged_f32_fwd", "bn_ragged_f32_bwd"]

OPS_ALL = ["bn_f32_fwd", "bn_f32_bwd", "rms_bf16_bwd", "rms_f32_bwd", "ln_bf16_bwd",
           "bn_bf16_fwd", "bn_bf16_bwd"]


# ----------------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def aggregate(local_seconds, local_bytes, world):
    """Whole-job numbers: max time over ranks, sum of bytes over ranks."""
    if world == 1:
        return local_seconds, local_bytes
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_seconds], dtype=torch.float64)
    b = torch.tensor([local_bytes], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t, b = t.cuda(), b.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        # under load = samples above half the max clock (idle samples are low)
        loaded = [v for v in sm if mx is None or v > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- workloads

class Op:
    """One hot-path operation on its workload.

    phases: list of (kernel-name, fn) run in order; each fn launches one
    kernel-pair call of the C ABI on the current stream.
    unique_bytes: bytes of every input and output tensor (algorithmic).
    phase_bytes: algorithmic bytes per phase launch (for the roofline).
    """

    def __init__(self, name, desc, phases, unique_bytes, phase_bytes, launches,
                 h2d, d2h, host_call):
        self.name = name
        self.desc = desc
        self.phases = phases
        self.unique_bytes = unique_bytes
        self.phase_bytes = phase_bytes
        self.launches = launches
        self.h2d = h2d          # list of (pinned host tensor, device tensor)
        self.d2h = d2h          # list of (device tensor, pinned host tensor)
        self.host_call = host_call


def _nbytes(*ts):
    return sum(t.numel() * t.element_size() for t in ts if t is not None)


def _pin(t):
    return t.contiguous().pin_memory()


def build_ops(names, dev):
    import torch
    from bwd_bn_pass_gb300 import gbnorm as G, synth

    ops = []
    for name in names:
        if name.startswith("bn_"):
            # bn[_relu][_nhwc]_{f32,bf16}_{fwd,bwd}; bn_{tiny,ragged}_f32_{fwd,bwd}
            if name.startswith("bn_tiny_"):
                case = synth.CASES["bn_tiny_f32"]
            elif name.startswith("bn_ragged_"):
                case = synth.CASES["bn_ragged_f32"]
            else:
                case = synth.CASES["bn_offset_f32" if "f32" in name else "bn_offset_bf16"]
            act = "relu" if "_relu_" in name else None
            nhwc = "_nhwc_" in name
            inp = synth.bn_inputs(case)
            if nhwc:  # the same data, channels last
                inp["x"] = inp["x"].permute(0, 2, 3, 1).contiguous()
                inp["dy"] = inp["dy"].permute(0, 2, 3, 1).contiguous()
            hx, hdy = _pin(inp["x"]), _pin(inp["dy"])
            x, dy = hx.to(dev), hdy.to(dev)
            C = x.shape[-1] if nhwc else x.shape[1]
            # per-channel vectors in one buffer [gamma | beta | running_mean |
            # running_var | stats (8 C)], so that the end-to-end leg moves
            # them with one copy each way
            par = torch.empty(12 * C, dtype=torch.float32, device=dev)
            g, b, rm, rv = (par[k * C:(k + 1) * C] for k in range(4))
            stats = par[4 * C:]
            for t, src in ((g, "gamma"), (b, "beta"), (rm, "running_mean"),
                           (rv, "running_var")):
                t.copy_(inp[src])
            y = torch.empty_like(x)
            fwd_fn = G.bn_nhwc_forward_train if nhwc else G.bn_forward_train
            bwd_fn = G.bn_nhwc_backward if nhwc else G.bn_backward
            ws = G.bn_nhwc_workspace(x) if nhwc else G.bn_workspace(x)
            # a forward once so the backward has valid stats
            fwd_fn(x, g, b, rm, rv, case.momentum, case.eps, y=y, stats=stats, ws=ws, act=act)
            T = _nbytes(x)
            small = _nbytes(g, b, rm, rv) + 4 * C * 4
            shape = "x".join(map(str, x.shape))
            kind = ("BatchNorm2d" + ("+ReLU" if act else "")
                    + (" channels-last" if nhwc else ""))
            key = "bn_forward_train" if name.endswith("fwd") else "bn_backward"
            # NCHW: one launch of the persistent kernel from the library's size
            # threshold on, or of the small-channel kernels where the library
            # takes them (a block or a cluster of up to 8 blocks per channel,
            # one resident wave), else stats + apply (grad sums + dx); NHWC:
            # three.
            in_bytes = T * (1 if name.endswith("fwd") else 2)
            M = x.numel() // C
            if nhwc:
                launches = 3
            elif in_bytes >= G.bn_persistent_min_bytes() or G.bn_small_blocks_per_channel(x.shape):
                launches = 1  # the persistent kernel, or a small-channel kernel
            else:
                launches = 2
            pin = lambda t: torch.empty_like(t, device="cpu").pin_memory()  # noqa: E731
            if name.endswith("fwd"):
                # the composite call a user makes: statistics, finalize and apply
                phases = [
                    (key,
                     lambda x=x, g=g, b=b, rm=rm, rv=rv, y=y, stats=stats, ws=ws, c=case,
                     f=fwd_fn, a=act:
                     f(x, g, b, rm, rv, c.momentum, c.eps, y=y, stats=stats, ws=ws, act=a)),
                ]
                # end to end: every input up (x; gamma, beta and the running
                # stats in one copy), every output down (y; the updated
                # running stats and stats in one copy)
                h2d = [(hx, x), (_pin(par[:4 * C].cpu()), par[:4 * C])]
                d2h = [(y, pin(y)), (par[2 * C:], pin(par[2 * C:]))]
                ops.append(Op(name, f"{kind} fwd {case.dtype} [{shape}]", phases,
                              2 * T + small, {key: 2 * T + small}, launches, h2d, d2h, None))
            else:
                dx = torch.empty_like(x)
                grads = torch.empty(4 * C, dtype=torch.float32, device=dev)
                phases = [
                    (key, lambda x=x, dy=dy, s=stats, dx=dx, gr=grads, ws=ws, b=b, f=bwd_fn,
                     a=act: f(x, dy, s, dx=dx, grads=gr, ws=ws, beta=b if a else None, act=a)),
                ]
                ub = 3 * T + 8 * C * 4 + 4 * C * 4
                # end to end: x, dy and the saved stats up (beta too with an
                # activation); dx and grads down
                h2d = [(hx, x), (hdy, dy), (_pin(stats.cpu()), stats)]
                if act:
                    h2d.append((_pin(b.cpu()), b))
                d2h = [(dx, pin(dx)), (grads, pin(grads))]
                ops.append(Op(name, f"{kind} bwd {case.dtype} [{shape}]", phases,
                              ub, {key: ub}, launches, h2d, d2h, None))
        elif name in ("rms_bf16_fwd", "rms_f32_fwd"):
            case = synth.CASES["rms_bf16" if "bf16" in name else "rms_f32"]
            inp = synth.rms_inputs(case)
            hx, hw = _pin(inp["x"]), _pin(inp["w"])
            x, w = hx.to(dev), hw.to(dev)
            y = torch.empty_like(x)
            rstd = torch.empty(case.rows, dtype=torch.float32, device=dev)
            phases = [("rms_fwd", lambda x=x, w=w, y=y, rstd=rstd, e=case.eps:
                        G.rmsnorm_forward(x, w, e, y=y, rstd=rstd))]
            ub = _nbytes(x, w, y, rstd)
            hy, hr = torch.empty_like(hx).pin_memory(), torch.empty_like(rstd, device="cpu").pin_memory()
            ops.append(Op(name, f"RMSNorm fwd {case.dtype} [{case.rows}x{case.hidden}]",
                          phases, ub, {"rms_fwd": ub}, 1, [(hx, x), (hw, w)],
                          [(y, hy), (rstd, hr)], None))
        elif name == "ln_bf16_fwd":
            case = synth.CASES["ln_fused_bf16"]
            inp = synth.ln_inputs(case)
            host = {k: _pin(v) for k, v in inp.items() if torch.is_tensor(v)}
            d = {k: v.to(dev) for k, v in host.items()}
            s = inp["dropout_scale"]
            y, z = torch.empty_like(d["inp"]), torch.empty_like(d["inp"])
            mean = torch.empty(case.rows, dtype=torch.float32, device=dev)
            rstd = torch.empty_like(mean)
            phases = [("ln_fwd", lambda d=d, s=s, y=y, z=z, mean=mean, rstd=rstd, e=case.eps:
                       G.layernorm_forward(d["inp"], d["gamma"], d["beta"], e,
                                           residual=d["residual"], bias=d["bias"],
                                           mask=d["mask"], dropout_scale=s, y=y, z=z,
                                           mean=mean, rstd=rstd))]
            ub = _nbytes(d["inp"], d["residual"], d["mask"], d["bias"], d["gamma"], d["beta"],
                         y, z, mean, rstd)
            order = ["inp", "residual", "mask", "bias", "gamma", "beta"]
            outs = [(t, torch.empty_like(t, device="cpu").pin_memory())
                    for t in (y, z, mean, rstd)]
            ops.append(Op(name, f"bias+dropout+add+LayerNorm fwd bf16 "
                          f"[{case.rows}x{case.hidden}]", phases, ub, {"ln_fwd": ub}, 1,
                          [(host[k], d[k]) for k in order], outs, None))
        elif name.startswith("rms_"):
            case = synth.CASES["rms_bf16" if "bf16" in name else "rms_f32"]
            inp = synth.rms_inputs(case)
            hx, hdy, hw = _pin(inp["x"]), _pin(inp["dy"]), _pin(inp["w"])
            x, dy, w = hx.to(dev), hdy.to(dev), hw.to(dev)
            rstd = torch.rsqrt(x.double().pow(2).mean(dim=1) + case.eps).float()
            hr = _pin(rstd.cpu())
            dx = torch.empty_like(x)
            dw = torch.empty_like(w)
            ws = G.rowwise_workspace(case.rows, case.hidden, G.GBN_ROW_RMS, x.dtype, dev)
            phases = [("rms_bwd", lambda dy=dy, x=x, w=w, rstd=rstd, dx=dx, dw=dw, ws=ws:
                        G.rmsnorm_backward(dy, x, w, rstd, dx=dx, dw=dw, ws=ws))]
            ub = _nbytes(x, dy, dx, w, dw, rstd)
            hdx, hdw = torch.empty_like(hx).pin_memory(), torch.empty_like(hw).pin_memory()
            # one launch: the ring kernel finishes dweight in the same launch
            ops.append(Op(name, f"RMSNorm bwd {case.dtype} [{case.rows}x{case.hidden}]",
                          phases, ub, {"rms_bwd": ub}, 1, [(hx, x), (hdy, dy), (hw, w), (hr, rstd)],
                          [(dx, hdx), (dw, hdw)], None))
        elif name.startswith("ln_"):
            case = synth.CASES["ln_fused_bf16"]
            inp = synth.ln_inputs(case)
            host = {k: _pin(v) for k, v in inp.items() if torch.is_tensor(v)}
            d = {k: v.to(dev) for k, v in host.items()}
            s = inp["dropout_scale"]
            z = (d["residual"].float() + d["mask"].float() * s
                 * (d["inp"].float() + d["bias"].float()))
            mean = z.mean(dim=1)
            rstd = torch.rsqrt(z.var(dim=1, unbiased=False) + case.eps)
            del z
            host["mean"], host["rstd"] = _pin(mean.cpu()), _pin(rstd.cpu())
            d["mean"], d["rstd"] = mean, rstd
            dx, dres = torch.empty_like(d["inp"]), torch.empty_like(d["inp"])
            dg, db, dbias = (torch.empty_like(d["gamma"]) for _ in range(3))
            ws = G.rowwise_workspace(case.rows, case.hidden, G.GBN_ROW_LN_FUSED,
                                     d["inp"].dtype, dev)
            phases = [("ln_bwd", lambda d=d, s=s, dx=dx, dres=dres, dg=dg, db=db, dbias=dbias,
                        ws=ws: G.layernorm_backward(
                            d["dy"], d["inp"], d["mean"], d["rstd"], d["gamma"],
                            residual=d["residual"], bias=d["bias"], mask=d["mask"],
                            dropout_scale=s, dx=dx, dresidual=dres, dgamma=dg, dbeta=db,
                            dbias=dbias, ws=ws))]
            ub = _nbytes(d["dy"], d["inp"], d["residual"], d["mask"], d["mean"], d["rstd"],
                         d["gamma"], d["bias"], dx, dres, dg, db, dbias)
            order = ["dy", "inp", "residual", "mask", "mean", "rstd", "gamma", "bias"]
            outs = [(t, torch.empty_like(t, device="cpu").pin_memory())
                    for t in (dx, dres, dg, db, dbias)]
            # one launch: the ring kernel finishes the column sums in the same launch
            ops.append(Op(name, f"bias+dropout+add+LayerNorm bwd bf16 "
                          f"[{case.rows}x{case.hidden}]", phases, ub, {"ln_bwd": ub}, 1,
                          [(host[k], d[k]) for k in order], outs, None))
        else:
            raise ValueError(f"unknown op {name}")
    return ops


# ------------------------------------------------------------- our arm

# The sources the dominant kernel (the persistent BatchNorm kernel) is built
# from; a recorded ncu traffic figure is used only while they are unchanged.
ROOFLINE_KERNEL_SOURCES = ("bn_fused.cu", "bn_finalize.cuh", "gbn_common.cuh")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bwd_bn_pass_gb300", "csrc")
    for fn in ROOFLINE_KERNEL_SOURCES:
        with open(os.path.join(csrc, fn), "rb") as fh:
            h.update(fn.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it
    was captured from the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    v = d.get("per_launch_dram_bytes", {}).get(kernel)
    return None if v is None else float(v)


def run_ours(args, rank, world, local_rank):
    import torch
    from bwd_bn_pass_gb300 import build, gbnorm

    if not os.path.exists(gbnorm.library_path()):
        build.build_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    gbnorm.init(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    names = args.ops.split(",") if args.ops else OPS_ALL
    ops = build_ops(names, dev)
    # L2 flush: write one 256 MB buffer, then read another, so L2 is left
    # holding clean lines of the second buffer -- no dirty write-back of the
    # flush lands in the next timed operation.
    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_out)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def one_step(record):
        for op in ops:
            flush_l2()
            evs = [torch.cuda.Event(enable_timing=True)]
            evs[0].record(stream)
            for _, fn in op.phases:
                fn()
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                evs.append(e)
            record.append((op, evs))

    # The events bracket device work only, but a call's host-side cost
    # (~25 us for a BatchNorm call) overlaps the L2 flush only as long as the
    # host does not stall; a garbage-collector pause longer than the flush
    # would land inside an operation's events.  As timeit does, the
    # collector stays off while the GPU legs are timed.
    gc.collect()
    gc.disable()
    rec = []
    with ClockSampler(local_rank) as clk:
        # the warm-up runs after the sampler has started (it waits 0.3 s for
        # nvidia-smi): a GPU left idle that long takes its first call of the
        # timed region several times slower (measured: 100 us for a 23 us
        # call), so the idle gap belongs before the warm-up, not after it
        for _ in range(args.warmup):
            one_step([])
        barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            one_step(rec)
        barrier()
        wall = time.perf_counter() - t0
    clocks = clk.summary()

    per_op = {op.name: [] for op in ops}
    per_phase = {}
    for op, evs in rec:
        per_op[op.name].append(evs[0].elapsed_time(evs[-1]) * 1e-3)
        for i, (pname, _) in enumerate(op.phases):
            per_phase.setdefault((op.name, pname), []).append(
                evs[i].elapsed_time(evs[i + 1]) * 1e-3)
    step_s = sum(statistics.mean(v) for v in per_op.values())
    step_bytes = sum(op.unique_bytes for op in ops)
    job_s, job_bytes = aggregate(step_s, step_bytes, world)
    value = job_bytes / job_s / 1e9
    peak, peak_kind = measured_peaks()

    # dominant kernel: the phase with the largest share of the step
    (dop, dphase), dtimes = max(per_phase.items(), key=lambda kv: statistics.mean(kv[1]))
    dmean = statistics.mean(dtimes)
    dbytes = next(op.phase_bytes[dphase] for op in ops if op.name == dop)
    achieved = dbytes / dmean / 1e9
    roofline = {"bound": "hbm", "kernel": f"{dphase} ({dop})", "achieved": round(achieved, 1),
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": dbytes,
                "traffic": recorded_traffic(f"{dop}:{dphase}")}
    if roofline["traffic"]:
        # what DRAM actually moved (the recorded ncu bytes) over the live time
        dram = roofline["traffic"] / dmean / 1e9
        roofline["dram_achieved"] = round(dram, 1)
        roofline["dram_frac"] = round(dram / peak, 4)

    # Warm-L2 figures, labelled as such and not part of `value`: each op
    # called back to back without the flush, so whatever fits in L2 stays.
    warm = {}
    for op in ops:
        for _ in range(2):
            for _, fn in op.phases:
                fn()
        evs = []
        for _ in range(max(args.steps, 5)):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _, fn in op.phases:
                fn()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        warm[op.name] = statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e-3

    ops_out = {}
    for op in ops:
        t = statistics.mean(per_op[op.name])
        ops_out[op.name] = {
            "desc": op.desc, "us": round(t * 1e6, 2),
            "us_median": round(statistics.median(per_op[op.name]) * 1e6, 2),
            "us_min": round(min(per_op[op.name]) * 1e6, 2),
            "unique_bytes": op.unique_bytes,
            "eff_gbs": round(op.unique_bytes / t / 1e9, 1),
            "frac_of_measured_peak": round(op.unique_bytes / t / 1e9 / peak, 4),
            "phases_us": {p: round(statistics.mean(per_phase[(op.name, p)]) * 1e6, 2)
                          for p, _ in op.phases},
            "us_warm_l2": round(warm[op.name] * 1e6, 2),
            "eff_gbs_warm_l2": round(op.unique_bytes / warm[op.name] / 1e9, 1),
        }

    graph = run_graph(ops, stream, dev, args.steps, world, flush_l2)
    latency = None if args.ops else run_latency(build_ops(LATENCY_OPS, dev), stream, dev,
                                                max(args.steps, 200), flush_l2)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(ops, stream, dev, args.steps, world)
    gc.enable()

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(job_s * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, the pages' value laws)",
        "config": {
            "workload": "; ".join(op.desc for op in ops),
            "ops": names,
            "l2": "before every operation: 256 MB write + 256 MB read of another buffer "
                  "(outside the timed events; L2 left clean)",
            "timing": "CUDA events per operation on the launching stream; sum over ops; "
                      "Python's garbage collector off while the GPU legs are timed",
            "warm_l2": "ops.*.us_warm_l2: the same calls back to back without the flush "
                       "(labelled, not used in value)",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
        },
        "pct_of_measured_peak": round(100 * value / world / peak, 2),
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "ops": ops_out,
        "roofline": roofline,
        "gpu_launches": sum(op.launches for op in ops) * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
        "e2e": e2e,
        "graph_step": graph,
        "latency_ops": latency,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return line


def run_latency(ops, stream, dev, steps, flush_l2):
    """Microseconds per call of latency-bound ops: each call timed alone with
    CUDA events after an L2 flush, eagerly and as a replay of a CUDA graph
    that holds just that call (the launch overhead a graph removes).  The
    event timer advances in steps of about 2 us on this device, so a single
    sample, and hence the median and the minimum, snap to a step; the mean
    over many calls resolves finer differences."""
    import torch
    out = {}
    for op in ops:
        def call(op=op):
            for _, fn in op.phases:
                fn()

        eager = []
        for it in range(steps + 3):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            e1.synchronize()
            if it >= 3:
                eager.append(e0.elapsed_time(e1) * 1e3)
        graph = []
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call()
            for it in range(steps + 3):
                flush_l2()
                e0, e1 = (torch.cuda.Event(enable_timing=True),
                          torch.cuda.Event(enable_timing=True))
                e0.record(stream)
                g.replay()
                e1.record(stream)
                e1.synchronize()
                if it >= 3:
                    graph.append(e0.elapsed_time(e1) * 1e3)
        except RuntimeError:
            graph = []
        out[op.name] = {
            "desc": op.desc, "launches": op.launches,
            "us_median": round(statistics.median(eager), 2), "us_min": round(min(eager), 2),
            "us_mean": round(statistics.mean(eager), 2), "samples": len(eager),
            "us_graph_median": round(statistics.median(graph), 2) if graph else None,
            "us_graph_min": round(min(graph), 2) if graph else None,
            "us_graph_mean": round(statistics.mean(graph), 2) if graph else None,
        }
    return out


def run_graph(ops, stream, dev, steps, world, flush_l2):
    """The whole step (every op's calls, back to back) captured once in a CUDA
    graph and replayed: the same work without the per-call launch latency
    that the per-operation events include.  L2 is flushed before every
    replay, outside the events.  Reported beside `value`, not instead of it."""
    import torch
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for op in ops:
                for _, fn in op.phases:
                    fn()
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for op in ops:
                for _, fn in op.phases:
                    fn()
        times = []
        for it in range(steps + 1):
            flush_l2()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            if it > 0:
                times.append(a.elapsed_time(b) * 1e-3)
    except Exception as exc:  # reported, never fatal: `value` stands alone
        failure = f"{type(exc).__name__}: {exc}"[:200]
        times = [math.inf]
    else:
        failure = None
    # every rank takes part in the aggregation, a failed one with an
    # infinite time, so that no rank waits on a collective the others skip
    t = statistics.mean(times)
    job_s, job_bytes = aggregate(t, sum(op.unique_bytes for op in ops), world)
    if failure is not None or not math.isfinite(job_s):
        return {"unavailable": failure or "graph replay failed on another rank"}
    return {"value": round(job_bytes / job_s / 1e9, 1), "unit": UNIT,
            "ms_per_step": round(job_s * 1e3, 4),
            "note": "whole step in one CUDA graph replay; L2 flushed before each replay"}


def johnson_order(ops):
    """Johnson's rule (S. M. Johnson, 1954, two-machine flow shop) on each
    op's upload and download bytes: ops that upload less than they download
    first, by increasing upload; then the rest by decreasing download."""
    up = {id(op): sum(_nbytes(h) for h, _ in op.h2d) for op in ops}
    down = {id(op): sum(_nbytes(h) for _, h in op.d2h) for op in ops}
    first = sorted((op for op in ops if up[id(op)] < down[id(op)]), key=lambda op: up[id(op)])
    last = sorted((op for op in ops if up[id(op)] >= down[id(op)]),
                  key=lambda op: -down[id(op)])
    return first + last


def run_e2e(ops, stream, dev, steps, world):
    """Same metric through the C ABI with host buffers: per step every op
    copies its inputs from pinned host memory, runs, and copies its outputs
    back, all inside the timed region.  The copies run on their own streams
    (host-to-device and device-to-host engines work concurrently), so op
    i+1's upload and op i-1's download overlap op i's kernels; each op's
    kernels wait for its own upload, its download waits for its kernels.
    (Splitting large copies over several streams per direction was slower.)
    The ops run in the order of Johnson's rule for a two-stage flow shop
    (upload, then download; the kernels are short beside the copies), which
    minimises the time the two copy engines leave each other idle."""
    import torch
    h2d = sum(_nbytes(h) for op in ops for h, _ in op.h2d)
    d2h = sum(_nbytes(h) for op in ops for _, h in op.d2h)
    ops = johnson_order(ops)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    times = []
    for it in range(steps + 1):
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(up)
        for op in ops:
            loaded, done = torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(up):
                for h, d in op.h2d:
                    d.copy_(h, non_blocking=True)
                loaded.record(up)
            stream.wait_event(loaded)
            with torch.cuda.stream(stream):
                for _, fn in op.phases:
                    fn()
                done.record(stream)
            down.wait_event(done)
            with torch.cuda.stream(down):
                for d, h in op.d2h:
                    h.copy_(d, non_blocking=True)
        b.record(down)
        b.synchronize()
        if it > 0:
            times.append(a.elapsed_time(b) * 1e-3)
    t = statistics.mean(times)
    step_bytes = sum(op.unique_bytes for op in ops)
    job_s, job_bytes = aggregate(t, step_bytes, world)
    return {"value": round(job_bytes / job_s / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(job_s * 1e3, 3),
            "order": [op.name for op in ops]}


# ------------------------------------------------------------ CPU oracle

class OracleSample:
    """A bounded sample of every op's workload, prepared once as float64
    arrays for the oracle: BatchNorm on the first `bn_channels` channels (all
    batches and pixels), RMSNorm / LayerNorm on the first rows.  Each op is
    split into independent units (BatchNorm channels, rows), so the sample
    can also be cut into shards for several host threads.  `time_pass` runs
    the oracle once over all ops on one thread and returns (unique storage
    bytes of the sample, seconds of oracle time)."""

    def __init__(self, bn_f32_channels, bn_bf16_channels, rms_rows, ln_rows):
        import numpy as np
        import oracle
        from bwd_bn_pass_gb300 import synth

        self.items = []  # (name, units, storage bytes per unit, make(lo, hi) -> callable)
        self.desc = {}
        for name in OPS_ALL:
            if name.startswith("bn_"):
                case = synth.CASES["bn_offset_f32" if "f32" in name else "bn_offset_bf16"]
                k = bn_f32_channels if "f32" in name else bn_bf16_channels
                inp = synth.bn_inputs(case)
                x = np.ascontiguousarray(inp["x"][:, :k].double().numpy())
                dy = np.ascontiguousarray(inp["dy"][:, :k].double().numpy())
                g = inp["gamma"][:k].double().numpy()
                b = inp["beta"][:k].double().numpy()
                plane = x.shape[0] * x.shape[2] * x.shape[3] * inp["x"].element_size()
                if name.endswith("fwd"):
                    def make(lo, hi, x=x, g=g, b=b, c=case):
                        xs = np.ascontiguousarray(x[:, lo:hi])
                        return lambda: oracle.batch_norm_forward_train(
                            xs, g[lo:hi], b[lo:hi], np.zeros(hi - lo), np.ones(hi - lo),
                            c.momentum, c.eps)
                    per = 2 * plane
                else:
                    def make(lo, hi, x=x, dy=dy, g=g, c=case):
                        xs = np.ascontiguousarray(x[:, lo:hi])
                        ds = np.ascontiguousarray(dy[:, lo:hi])
                        return lambda: oracle.batch_norm_backward(xs, ds, g[lo:hi], c.eps)
                    per = 3 * plane
                self.items.append((name, k, per, make))
                self.desc[name] = f"{k}/{case.shape[1]} channels"
            elif name.startswith("rms_"):
                case = synth.CASES["rms_bf16" if "bf16" in name else "rms_f32"]
                inp = synth.rms_inputs(case)
                x = inp["x"][:rms_rows].double().numpy()
                dy = inp["dy"][:rms_rows].double().numpy()
                w = inp["w"].double().numpy()
                rstd = oracle.rms_norm_rstd(x, case.eps)

                def make(lo, hi, x=x, dy=dy, w=w, r=rstd):
                    xs, ds, rs = x[lo:hi], dy[lo:hi], r[lo:hi]
                    return lambda: oracle.rms_norm_backward(xs, ds, w, rs)
                self.items.append((name, rms_rows, 3 * case.hidden * inp["x"].element_size(),
                                   make))
                self.desc[name] = f"{rms_rows}/{case.rows} rows"
            else:
                case = synth.CASES["ln_fused_bf16"]
                inp = synth.ln_inputs(case)
                f = {n: inp[n][:ln_rows].double().numpy()
                     for n in ("inp", "residual", "dy", "mask")}
                bias = inp["bias"].double().numpy()
                gamma = inp["gamma"].double().numpy()
                sc = inp["dropout_scale"]
                z = oracle.dropout_add(f["inp"], f["residual"], bias, f["mask"], sc)
                mu, rs = oracle.layer_norm_saved_stats(z, case.eps)

                def make(lo, hi, f=f, bias=bias, gamma=gamma, sc=sc, mu=mu, rs=rs):
                    p = {n: v[lo:hi] for n, v in f.items()}
                    m, r = mu[lo:hi], rs[lo:hi]
                    return lambda: oracle.fused_bias_dropout_add_layer_norm_backward(
                        p["dy"], p["inp"], p["residual"], bias, p["mask"], sc, m, r, gamma)
                self.items.append((name, ln_rows, case.hidden * (5 * 2 + 1), make))
                self.desc[name] = f"{ln_rows}/{case.rows} rows"
        self.whole = [make(0, units) for _, units, _, make in self.items]
        self.nbytes = sum(units * per for _, units, per, _ in self.items)

    def time_pass(self):
        secs = 0.0
        for fn in self.whole:
            t0 = time.perf_counter()
            fn()
            secs += time.perf_counter() - t0
        return self.nbytes, secs

    def shards(self, n):
        """n lists of calls that together cover the sample once (each op's
        units split into n contiguous ranges)."""
        out = [[] for _ in range(n)]
        for _, units, _, make in self.items:
            for s in range(n):
                lo, hi = units * s // n, units * (s + 1) // n
                if hi > lo:
                    out[s].append(make(lo, hi))
        return out

    def describe(self):
        return ", ".join(f"{k} {v}" for k, v in self.desc.items())


def cpu_model():
    """One line naming the host CPU (lscpu's model name, else /proc/cpuinfo),
    else the machine type."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() == "Model name":
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        lines = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        lines = []
    kv = {}
    for ln in lines:
        if ":" in ln:
            k, v = ln.split(":", 1)
            kv.setdefault(k.strip(), v.strip())
    if "model name" in kv:
        return kv["model name"]
    if "CPU implementer" in kv:
        return (f"{platform.machine()}, CPU implementer {kv['CPU implementer']} "
                f"part {kv.get('CPU part', '?')}")
    return platform.machine()


def cpu_parallel(sample, budget_s):
    """The same oracle sample cut into one shard per host core and run on
    that many threads (numpy releases the interpreter lock inside its array
    loops); wall-clock time per pass."""
    from concurrent.futures import ThreadPoolExecutor
    n = os.cpu_count() or 1
    lists = sample.shards(n)
    run = lambda fns: [fn() for fn in fns]
    nb, secs, passes = 0, 0.0, 0
    with ThreadPoolExecutor(max_workers=n) as pool:
        list(pool.map(run, lists))  # warm-up pass
        while secs < budget_s and passes < 8:
            t0 = time.perf_counter()
            list(pool.map(run, lists))
            secs += time.perf_counter() - t0
            nb += sample.nbytes
            passes += 1
    return {"value": round(nb / secs / 1e9, 4), "unit": UNIT, "cores": n,
            "sample": f"the same sample in {n} shards (BatchNorm channels, rows) on {n} "
                      f"threads; {passes} pass(es)",
            "seconds": round(secs, 2)}


def cpu_baseline(budget_s):
    """The oracle as it stands, single-threaded, on a bounded sample of the
    step (about `budget_s` seconds of oracle time); beside it the same
    sample spread over every host core."""
    sample = OracleSample(bn_f32_channels=32, bn_bf16_channels=32, rms_rows=2048,
                          ln_rows=8192)
    nb, secs, passes = 0, 0.0, 0
    while secs < budget_s and passes < 8:
        b, s = sample.time_pass()
        nb += b
        secs += s
        passes += 1
    return {"value": round(nb / secs / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "float64 numpy oracle, one thread; per op: " + sample.describe()
            + f"; {passes} pass(es)", "seconds": round(secs, 2),
            "nproc": os.cpu_count(), "cpu_model": cpu_model(),
            "all_cores": cpu_parallel(sample, budget_s / 4)}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is one bounded sample."""
    if rank != 0:
        return None
    sample = OracleSample(bn_f32_channels=8, bn_bf16_channels=8, rms_rows=256, ln_rows=1024)
    for _ in range(args.warmup):
        sample.time_pass()
    nb, secs = 0, 0.0
    for _ in range(args.steps):
        b, s = sample.time_pass()
        nb += b
        secs += s
    value = nb / secs / 1e9
    desc = "float64 numpy oracle, one thread; per step: " + sample.describe()
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, the pages' value laws)",
        "config": {"workload": "bounded sample of: " + "; ".join(OPS_ALL), "ops": OPS_ALL},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ops", default="")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local_rank)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
