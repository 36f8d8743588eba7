"""Benchmark of the fused grouped-MLP forward (MXFP8 / NVFP4 block quantisation) on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gmlp|reference] [--workload NAME]

One step = one gmlp_forward over the workload's synthetic batch: x quantise,
fc1 grouped GEMM with the fused activation x prob and fc2_x requantisation,
fc2 grouped GEMM (NVFP4 adds the x amax pass and the fc2_x cast).  Weights are
quantised once before timing.  The default workload is the largest
configuration: the MXFP8 SwiGLU MoE layer with 64 Zipf-routed experts,
K=7168, N=2048 and 65536 tokens.

Prints one JSON line (rank 0).  value = TFLOP/s of the GEMMs (2*M*K*N1 +
2*M*N*K) over the device-timed steps, inputs resident in HBM, L2 flushed
between steps.  e2e = the same metric through the C ABI with the step's x,
probs and split sizes copied from pinned host memory and y copied back inside
the timed region, double-buffered across steps (the sequential figure is
reported beside it).  The same line carries, under "workloads", the NVFP4 SReLU
forward and the MXFP8 SwiGLU forward + backward legs, and under
"group_quantize" the standalone NVFP4 quantiser (--no-extra / --no-quant skip
them).  --impl reference times the oracle (the CPU restatement) on the host
cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mxfp8_nvfp4_block_gb300.inputs import WORKLOADS, bits, make_inputs  # noqa: E402

METRIC = "fused grouped-MLP fwd TFLOPS (% FP8/FP4 peak); group-quantize GB/s (% HBM)"
WORKLOAD_TEXT = {
    "mx_swiglu": "MXFP8 SwiGLU grouped MLP: 8 experts, K=2048, N=1024 (W1_g [2N,K], W2_g [K,N]), 16384 tokens, "
                 "Dirichlet(1) splits with one empty expert, seed 1",
    "nv_srelu": "NVFP4+RHT SReLU grouped MLP: 8 experts, K=4096, N=2048, 32768 tokens uniform, 0.1% x outliers x50, "
                "seed 2",
    "mx_skew": "MXFP8 SwiGLU grouped MLP, Zipf(1.1) routing: 64 experts, K=7168, N=2048, 65536 tokens, seed 3",
    "nv_tanh_srelu": "NVFP4+RHT tanh-SReLU (soft-clamp scale 8) grouped MLP on the nv_srelu inputs: 8 experts, "
                     "K=4096, N=2048, 32768 tokens, seed 2",
    "tiny": "MXFP8 SwiGLU grouped MLP: 4 experts, K=256, N=256, 512 tokens, seed 0",
}
NOMINAL_RATIO = {0: 2.0, 1: 6.0}   # dense FP8 / bf16 and FP4 / bf16 (4.5 and 13.5 vs 2.25 PFLOP/s)
# DRAM bytes (read + write) per fc1 launch from one ncu capture of the gemm.cu
# whose sha1 is in the key, valid only for that source.
FC1_TRAFFIC = {("mx_skew", "d5781b20ab7b176d6112da523493e7263b030ea0"): 2398632960 + 140919808,
               ("nv_srelu", "d5781b20ab7b176d6112da523493e7263b030ea0"): 113472256 + 92643584}


def fc1_traffic(workload: str):
    import hashlib
    src = os.path.join(ROOT, "mxfp8_nvfp4_block_gb300", "csrc", "gemm.cu")
    digest = hashlib.sha1(open(src, "rb").read()).hexdigest()
    return FC1_TRAFFIC.get((workload, digest))


def oracle_threads() -> int:
    """Threads the oracle runs on: the host cores this process may use, capped
    by OMP_NUM_THREADS when it is set (torchrun sets it to 1 per rank), which
    both numpy's BLAS and the oracle's OpenMP loops follow."""
    n = len(os.sched_getaffinity(0))
    v = os.environ.get("OMP_NUM_THREADS", "")
    return min(n, int(v)) if v.isdigit() and int(v) > 0 else n


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples taken while the timed region runs."""

    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines: list[tuple[float, str]] = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        self.t0 = time.time()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        t1 = getattr(self, "t1", time.time())
        rows = [ln for ts, ln in self.lines if self.t0 - 0.05 <= ts <= t1 + 0.05]
        if not rows:
            rows = [ln for _, ln in self.lines[-3:]]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [c.strip() for c in r.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ multi-rank timing

def max_over_ranks(total_ms: float, world: int, device) -> float:
    """Slowest rank's timed total (every rank processes its own batch)."""
    if world <= 1:
        return total_ms
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: the FLOPs all ranks processed over the slowest rank's time."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


# ------------------------------------------------------------------ GPU arm

L2_TEXT = {"write": "flushed between timed steps (256 MiB write, outside the step events)",
           "clean": "flushed between timed steps (256 MiB write, then a 256 MiB read of a second buffer so the "
                    "step starts on a cold L2 without the write's dirty lines; outside the step events)"}


def made_events(n: int) -> list:
    """n timing events, each recorded once now (before the L2 flush) so that it
    has its device handle: the binding would otherwise record a new event once
    before the call's first kernel, inside the timed region."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record()
    return evs


class L2Flush:
    """Flush L2 between timed steps: write 256 MiB; in "clean" mode then read
    another 256 MiB, so the write's dirty lines are written back here and the
    step starts on a cold, clean L2 (it does not pay for the flush's write-back).
    Then a GPU-side wait (about 0.25 ms of clock cycles) keeps the stream busy
    while the host enqueues the step's start event and its kernels, so a step
    never starts with the GPU idle on the host's launch path (the binding's
    argument checks take tens of microseconds): the timed region holds the
    step's kernels only."""

    def __init__(self, mode: str, dev):
        self.buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)   # > 129 MB of L2
        self.sweep = torch.zeros(64 * 1024 * 1024, dtype=torch.int32, device=dev) if mode == "clean" else None

    def __call__(self):
        self.buf.zero_()
        if self.sweep is not None:
            torch.amax(self.sweep)
        torch.cuda._sleep(500_000)


def forward_leg(gmlp, name: str, args, dev, world: int, steps: int, warmup: int, *, e2e: bool, rank: int = 0,
                keep_weights: bool = False) -> dict:
    """The forward of one workload: per-step time (value), per-kernel times,
    the fc1 roofline, and (e2e) the host-to-host figure through the C ABI."""
    d = make_inputs(name)
    w = d["workload"]
    fmt, act = w.fmt, w.act
    rec = gmlp.recipe(fmt, use_rht=True, mask=d["mask"])
    stream = torch.cuda.current_stream()
    x = d["x"].to(dev)
    splits = d["splits"].to(dev)
    probs = d["probs"].to(dev)
    x4 = {"auto": fmt == gmlp.NVFP4 and args.gemm_mode == 2, "x4": True, "tiled": False}[args.weight_scales]
    W1 = gmlp.prepare_weights(d["W1"].to(dev), fmt, swiglu_interleave=(act == gmlp.SWIGLU), x4=x4)
    W2 = gmlp.prepare_weights(d["W2"].to(dev), fmt, x4=x4)
    if not keep_weights:
        del d["W1"], d["W2"]
    y = torch.empty((w.M, w.K), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(gmlp.forward_workspace_size(w.M, w.K, w.N, w.G, act, rec), dtype=torch.uint8, device=dev)
    fwd_aux = None
    if fmt == gmlp.NVFP4:
        # the step's own outputs for the backward: fc2_x's amaxes (pre- and
        # post-RHT; the wgrad operand's global scale comes from the latter)
        fwd_aux = {"fc2x_amax_pre": torch.empty(w.G, dtype=torch.float32, device=dev),
                   "fc2x_amax_post": torch.empty(w.G, dtype=torch.float32, device=dev)}
    if args.fc2x_colwise and fmt == gmlp.NVFP4:
        # the no-recompute training variant: fc2_x also cast columnwise (RHT) in the same pass
        ncol = w.N * (w.M + 16 * w.G)
        fwd_aux.update({"fc2x_col_codes": torch.empty(ncol // 2, dtype=torch.uint8, device=dev),
                        "fc2x_col_scales": torch.empty(ncol // 16, dtype=torch.uint8, device=dev)})
    flush_l2 = L2Flush(args.l2_flush, dev)
    n_stage = 3 if fmt == gmlp.MXFP8 else 5

    def fwd(**kw):
        gmlp.forward(x, splits, W1, W2, probs, act, rec, y=y, workspace=ws, gemm_mode=args.gemm_mode, aux=fwd_aux,
                     tanh_clamp_scale=w.tanh_clamp_scale, **kw)

    def ev():
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        return e

    starts = [ev() for _ in range(steps)]
    ends = [ev() for _ in range(steps)]
    starts2 = [ev() for _ in range(steps)]
    stages = [[ev() for _ in range(n_stage)] for _ in range(steps)]
    torch.cuda.synchronize()

    for _ in range(warmup):
        flush_l2()
        fwd()
    gmlp.check_device_status()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        # pass 1 (the reported steps): one event before and after each step, so the
        # kernels of a step overlap their neighbours' prologues as in normal use
        for i in range(steps):
            flush_l2()
            starts[i].record(stream)
            fwd()
            ends[i].record(stream)
        torch.cuda.synchronize()
        # pass 2: events after every kernel of the step, for per-kernel times
        # (an event between kernels stops that overlap, so these steps run slightly longer)
        for i in range(steps):
            flush_l2()
            starts2[i].record(stream)
            fwd(events=stages[i])
        torch.cuda.synchronize()
        clk.mark_end()
    if world > 1:
        torch.distributed.barrier()
    gmlp.check_device_status()
    step_ms = [starts[i].elapsed_time(ends[i]) for i in range(steps)]
    bounds = [[starts2[i]] + stages[i] for i in range(steps)]
    stage_ms = [statistics.mean(b[j].elapsed_time(b[j + 1]) for b in bounds) for j in range(n_stage)]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / steps
    value = job_tflops(w.flops, world, ms_per_step)

    hbm, bf16_burst, _, src = peaks()
    fc1_idx = 1 if fmt == gmlp.MXFP8 else 2
    fc1_flops = 2.0 * w.M * w.K * w.n1
    fc1_ms = stage_ms[fc1_idx]
    peak = bf16_burst * NOMINAL_RATIO[fmt]
    quant_idx = 0 if fmt == gmlp.MXFP8 else 1
    cdiv, blk = (1, 32) if fmt == gmlp.MXFP8 else (2, 16)
    q_bytes = w.M * w.K * 2 + w.M * w.K // cdiv + w.M * w.K // blk
    achieved = fc1_flops / (fc1_ms * 1e-3) / 1e12
    # the GEMM path alone: from the quantised x to y (fc1, NVFP4's fc2_x cast, fc2)
    gemm_ms = sum(stage_ms[quant_idx + 1:])
    out = {
        "value": round(value, 3),
        "ms_per_step": round(ms_per_step, 5),
        "dtype": "mxfp8" if fmt == gmlp.MXFP8 else "nvfp4",
        "config": {"workload": f"{name}: {WORKLOAD_TEXT.get(name, name)}",
                   "l2": L2_TEXT[args.l2_flush],
                   "timing": "value: per-step start/end events (the stream held busy by a GPU-side wait after "
                             "the L2 flush, so host launch latency is not timed); stages_ms and roofline: a second "
                             "timed pass with "
                             "an event after every kernel",
                   "weights": "quantised once before timing; scales read in the " + (
                       "replicated GEMM_TILED_X4 layout" if W1.scales_x4 is not None else "GEMM_TILED layout"),
                   "flops_per_step": w.flops,
                   "gemm_mode": args.gemm_mode,
                   "fc2x_columnwise": bool(fwd_aux and "fc2x_col_codes" in fwd_aux)},
        "gpu_launches": steps * n_stage,
        "stages_ms": [round(t, 5) for t in stage_ms],
        "gemm_path": {"ms": round(gemm_ms, 5), "TFLOP_s": round(w.flops / (gemm_ms * 1e-3) / 1e12, 1),
                      "frac": round(w.flops / (gemm_ms * 1e-3) / 1e12 / peak, 4),
                      "what": "the step's kernels after the x cast (quantised x to bf16 y), per-kernel events"},
        "roofline": {"kernel": "fc1 grouped GEMM (gemm_kernel, fused activation + requant epilogue)",
                     "bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "peak_source": f"{src} bf16 burst {bf16_burst} x nominal {'FP8' if fmt == 0 else 'FP4'}/bf16 "
                                    f"ratio {NOMINAL_RATIO[fmt]}",
                     "traffic": fc1_traffic(name), "traffic_unit": "bytes per launch (ncu, null if the kernel "
                                                                   "changed since the capture)"},
        "x_quantize": {"ms": round(stage_ms[quant_idx], 5), "bytes": q_bytes,
                       "GB_s": round(q_bytes / (stage_ms[quant_idx] * 1e-3) / 1e9, 1),
                       "frac_hbm": round(q_bytes / (stage_ms[quant_idx] * 1e-3) / 1e9 / hbm, 4)},
        "clocks": clk.summary(),
    }
    has_col = bool(fwd_aux and "fc2x_col_codes" in fwd_aux)
    f_bytes = w.M * w.N * 2 + (w.M * w.N // 2 + w.M * w.N // 16) * (2 if has_col else 1)
    if fmt == gmlp.NVFP4:
        # fc2_x cast: bf16 in, rowwise NVFP4 out and the post-RHT amax (+ the
        # columnwise copy with --fc2x-colwise)
        out["fc2x_cast"] = {"ms": round(stage_ms[3], 5), "bytes": f_bytes, "columnwise": has_col,
                            "GB_s": round(f_bytes / (stage_ms[3] * 1e-3) / 1e9, 1),
                            "frac_hbm": round(f_bytes / (stage_ms[3] * 1e-3) / 1e9 / hbm, 4)}

    # every kernel of the step against its own roofline (algorithmic bytes or FLOPs / event time)
    def k_mem(nbytes, ms):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "ms": round(ms, 5), "GB_s": round(gbs, 1), "frac": round(gbs / hbm, 4)}

    def k_tensor(flops, ms):
        tf = flops / (ms * 1e-3) / 1e12
        return {"bound": "tensor", "ms": round(ms, 5), "TFLOP_s": round(tf, 1), "frac": round(tf / peak, 4)}

    kern = {}
    if fmt == gmlp.NVFP4:
        kern["x amax"] = k_mem(w.M * w.K * 2, stage_ms[0])
    kern["x quantise"] = k_mem(q_bytes, stage_ms[quant_idx])
    kern["fc1 GEMM"] = k_tensor(fc1_flops, fc1_ms)
    if fmt == gmlp.NVFP4:
        kern["fc2_x cast"] = k_mem(f_bytes, stage_ms[3])
    kern["fc2 GEMM"] = k_tensor(2.0 * w.M * w.N * w.K, stage_ms[-1])
    out["kernels"] = kern
    ceiling = mma_ceiling(gmlp, fmt)
    out["roofline"]["mma_loop_tflops"] = ceiling
    # the loop with the scale-factor path the forward's fc1 GEMM takes: NVFP4 with
    # replicated weight scales copies them (X4); with GEMM_TILED ones, single-CTA
    # tiles have them written by warps
    if fmt == gmlp.MXFP8:
        loop = ceiling["with_scale_copies"]
    elif W1.scales_x4 is not None:
        loop = ceiling["with_x4_scale_copies"]
    else:
        loop = ceiling["scales_written_by_warps" if args.gemm_mode == 0 else "with_scale_copies"]
    out["roofline"]["frac_of_mma_loop"] = round(achieved / loop, 4)

    if e2e:
        # ---- end to end through the C ABI with host buffers
        x_h = d["x"].pin_memory()
        p_h = d["probs"].pin_memory()
        s_h = d["splits"].pin_memory()
        y_h = torch.empty((w.M, w.K), dtype=torch.bfloat16).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for it in range(warmup + steps):
            if it == warmup:
                torch.cuda.synchronize()
                e0.record()
            x.copy_(x_h, non_blocking=True)
            probs.copy_(p_h, non_blocking=True)
            splits.copy_(s_h, non_blocking=True)
            fwd()
            y_h.copy_(y, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        gmlp.check_device_status()
        e2e_seq_ms = e0.elapsed_time(e1) / steps
        e2e_ms = e2e_pipelined(gmlp, args, w, x, probs, splits, y, x_h, p_h, s_h, W1, W2, act, rec, ws, fwd_aux,
                               steps, warmup)
        h2d = x_h.numel() * 2 + p_h.numel() * 4 + s_h.numel() * 8
        d2h = y_h.numel() * 2
        out["e2e"] = {"value": round(world * w.flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                      "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "how": "double-buffered across steps: step i's inputs copy in while step i-1 computes and "
                             "step i-2's y copies out, on separate streams",
                      "copy_streams_per_direction": args.e2e_streams,
                      "copy_GB_s_per_direction": round(h2d / (e2e_ms * 1e-3) / 1e9, 1),
                      "sequential": {"value": round(world * w.flops / (e2e_seq_ms * 1e-3) / 1e12, 3),
                                     "ms_per_step": round(e2e_seq_ms, 5)}}
    if keep_weights:
        out["_inputs"] = (d, x, splits, probs)
    return out


def run_gpu(args, rank: int, world: int) -> dict:
    from mxfp8_nvfp4_block_gb300 import gmlp
    gmlp.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    name = args.workload
    main_bwd = args.backward and name == "mx_swiglu"
    main = forward_leg(gmlp, name, args, dev, world, args.steps, args.warmup, e2e=True, rank=rank,
                       keep_weights=main_bwd)
    if main_bwd:
        d, x, splits, probs = main.pop("_inputs")
        main["backward_dgrad"] = bench_backward(gmlp, d, d["workload"], d["W1"].to(dev), d["W2"].to(dev), x, splits,
                                                probs, args.steps, args.warmup, dev, args.l2_flush)
        del d, x, splits, probs
    out = {"metric": METRIC, "value": main.pop("value"), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": main.pop("ms_per_step"), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": main.pop("dtype"), "data": "synthetic",
           "config": main.pop("config"), "e2e": main.pop("e2e"), "gpu_launches": main.pop("gpu_launches")}
    out.update(main)
    torch.cuda.empty_cache()
    if args.extra:
        # the other configurations of the path, each its own forward leg on this GPU
        # (fewer steps; no host copies); the MXFP8 SwiGLU leg also times the backward
        steps = max(3, min(args.steps, args.extra_steps))
        legs = {}
        for leg in ("nv_srelu", "mx_swiglu"):
            if leg == name:
                continue
            want_bwd = args.backward and leg == "mx_swiglu"
            r = forward_leg(gmlp, leg, args, dev, world, steps, args.warmup, e2e=False, rank=rank,
                            keep_weights=want_bwd)
            if want_bwd:
                d, x, splits, probs = r.pop("_inputs")
                w = d["workload"]
                r["backward_dgrad"] = bench_backward(gmlp, d, w, d["W1"].to(dev), d["W2"].to(dev), x, splits, probs,
                                                     steps, args.warmup, dev, args.l2_flush)
                del d, x, splits, probs
            legs[leg] = r
            torch.cuda.empty_cache()
        out["workloads"] = legs
    if args.quant and rank == 0:
        out["group_quantize"] = bench_quantizer(gmlp, dev, peaks()[0], args.quant_rows)
    return out


def e2e_pipelined(gmlp, args, w, x, probs, splits, y, x_h, p_h, s_h, W1, W2, act, rec, ws, fwd_aux,
                  K_steps: int, W_steps: int) -> float:
    """ms per step of the host-to-host forward with two slots of device and
    pinned host buffers: every step copies its x, probs and split sizes in
    and its y out inside the timed region, on copy streams ordered by events
    around one compute stream, so the copies of neighbouring steps overlap.
    With args.e2e_streams = S > 1, x and y move as S row slices on S streams
    per direction (concurrent copies)."""
    S = max(1, int(args.e2e_streams))
    M = x.shape[0]
    cuts = [M * k // S for k in range(S + 1)]
    xs, ps, ss, ys = [x, x.clone()], [probs, probs.clone()], [splits, splits.clone()], [y, torch.empty_like(y)]
    yh = [torch.empty(y.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    s_in = [torch.cuda.Stream() for _ in range(S)]
    s_out = [torch.cuda.Stream() for _ in range(S)]
    s_cmp = torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in range(S)] for _ in range(2)]
    ev_out = [[torch.cuda.Event() for _ in range(S)] for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    started = [False, False]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    for it in range(W_steps + K_steps):
        b = it & 1
        if it == W_steps:
            torch.cuda.synchronize()
            e0.record(s_in[0])
            for st in s_in[1:] + s_out:
                st.wait_event(e0)
        for k, st in enumerate(s_in):
            with torch.cuda.stream(st):
                if started[b]:
                    st.wait_event(ev_cmp[b])      # the slot's previous forward has read its inputs
                xs[b][cuts[k]:cuts[k + 1]].copy_(x_h[cuts[k]:cuts[k + 1]], non_blocking=True)
                if k == 0:
                    ps[b].copy_(p_h, non_blocking=True)
                    ss[b].copy_(s_h, non_blocking=True)
                ev_in[b][k].record(st)
        for k in range(S):
            s_cmp.wait_event(ev_in[b][k])
            if started[b]:
                s_cmp.wait_event(ev_out[b][k])    # the slot's previous y has been read out
        gmlp.forward(xs[b], ss[b], W1, W2, ps[b], act, rec, y=ys[b], workspace=ws, gemm_mode=args.gemm_mode,
                     aux=fwd_aux, tanh_clamp_scale=w.tanh_clamp_scale, stream=s_cmp)
        ev_cmp[b].record(s_cmp)
        for k, st in enumerate(s_out):
            with torch.cuda.stream(st):
                st.wait_event(ev_cmp[b])
                yh[b][cuts[k]:cuts[k + 1]].copy_(ys[b][cuts[k]:cuts[k + 1]], non_blocking=True)
                ev_out[b][k].record(st)
        started[b] = True
    b = (W_steps + K_steps - 1) & 1
    for k in range(1, S):
        s_out[0].wait_event(ev_out[b][k])
    e1.record(s_out[0])
    torch.cuda.synchronize()
    gmlp.check_device_status(stream=s_cmp)
    return e0.elapsed_time(e1) / K_steps


def mma_ceiling(gmlp, fmt: int, iters: int = 32768, reps: int = 5) -> dict:
    """Tensor-core ceiling of the GEMM mainloop's MMA shape: gmlp_mma_peak on
    every SM (no global memory), with the per-stage scale copies of GEMM_TILED
    weight scales, of GEMM_TILED_X4 ones (NVFP4), with the scales written into
    tensor memory by the warps (tcgen05.st), and with none."""
    names = {1: "with_scale_copies", 2: "with_x4_scale_copies", 3: "scales_written_by_warps", 0: "scales_resident"}
    out = {}
    for copy in ((1, 2, 3, 0) if fmt == gmlp.NVFP4 else (1, 3, 0)):
        for _ in range(3):
            gmlp.mma_peak(fmt, copy, iters)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            gmlp.mma_peak(fmt, copy, iters)
        e1.record()
        torch.cuda.synchronize()
        gmlp.check_device_status()
        ms = e0.elapsed_time(e1) / reps
        n_sm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        tf = gmlp.mma_peak_flops(fmt, iters, n_sm) / (ms * 1e-3) / 1e12
        out[names[copy]] = round(tf, 1)
    return out


def bench_backward(gmlp, d, w, W1b, W2b, x, splits, probs, K_steps: int, W_steps: int, dev, l2_mode: str) -> dict:
    """Data-gradient backward (MXFP8): dy quantise -> fc2 dGLU GEMM (dSwiGLU /
    dSReLU x prob, dprob, MXFP8 fc1_dy) -> fc1 dgrad GEMM, on the forward's own
    saved activation input; L2 flushed between steps, per-step events."""
    rec = gmlp.recipe(w.fmt)
    w1 = gmlp.prepare_weights(W1b, w.fmt, swiglu_interleave=(w.act == gmlp.SWIGLU))
    w2 = gmlp.prepare_weights(W2b, w.fmt)
    h = torch.empty((w.M, w.n1), dtype=torch.bfloat16, device=dev)
    gmlp.forward(x, splits, w1, w2, probs, w.act, rec, aux={"fc1_pre_act": h})
    w2t = gmlp.prepare_transposed_weights(W2b)
    w1t = gmlp.prepare_transposed_weights(W1b)
    gen = torch.Generator().manual_seed(w.seed + 77)
    dy = torch.randn((w.M, w.K), generator=gen, dtype=torch.float32).to(torch.bfloat16).to(dev)
    dx = torch.empty_like(dy)
    ws = torch.empty(gmlp.load().gmlp_backward_workspace_size(w.M, w.K, w.N, w.G, w.act), dtype=torch.uint8,
                     device=dev)
    flush = L2Flush(l2_mode, dev)
    for _ in range(W_steps):
        flush()
        gmlp.backward_dgrad(dy, splits, w2t, w1t, h, probs, w.act, rec, dx=dx, workspace=ws)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_steps)]
    for e0, e1 in ev:
        flush()
        e0.record()
        gmlp.backward_dgrad(dy, splits, w2t, w1t, h, probs, w.act, rec, dx=dx, workspace=ws)
        e1.record()
    torch.cuda.synchronize()
    gmlp.check_device_status()
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
    # second pass: an event after every kernel (dy quantise, dGLU GEMM, dgrad GEMM)
    st = [0.0, 0.0, 0.0]
    for _ in range(K_steps):
        se = made_events(4)
        flush()
        se[0].record()
        gmlp.backward_dgrad(dy, splits, w2t, w1t, h, probs, w.act, rec, dx=dx, workspace=ws, events=se[1:])
        torch.cuda.synchronize()
        for i in range(3):
            st[i] += se[i].elapsed_time(se[i + 1]) / K_steps
    gmlp.check_device_status()
    flops = 2.0 * w.M * w.K * w.N + 2.0 * w.M * w.n1 * w.K
    # weight gradients on the dgrad's own bf16 fc1_dy: columnwise MXFP8 of dy,
    # fc2_x (rebuilt from h), fc1_dy and x, the two grouped wgrad GEMMs (FP32
    # dW) and the bias gradients
    f1 = torch.empty((w.M, w.n1), dtype=torch.bfloat16, device=dev)
    gmlp.backward_dgrad(dy, splits, w2t, w1t, h, probs, w.act, rec, dx=dx, workspace=ws, fc1_dy_bf16=f1)
    xin = x
    wws = torch.empty(gmlp.load().gmlp_backward_wgrad_workspace_size(w.M, w.K, w.N, w.G, w.act), dtype=torch.uint8,
                      device=dev)
    grads = gmlp.backward_wgrad(xin, dy, h, probs, f1, splits, w.act, workspace=wws)
    kern = {}
    for _ in range(W_steps):
        flush()
        gmlp.backward_wgrad(xin, dy, h, probs, f1, splits, w.act, workspace=wws, **grads)
    torch.cuda.synchronize()
    ew = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_steps)]
    for e0, e1 in ew:
        flush()
        e0.record()
        gmlp.backward_wgrad(xin, dy, h, probs, f1, splits, w.act, workspace=wws, **grads)
        e1.record()
    torch.cuda.synchronize()
    gmlp.check_device_status()
    wms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ew)
    # second pass: an event after every kernel (dy cast, fc2_x cast, dW2 GEMM,
    # fc1_dy cast, x cast, dW1 GEMM)
    wst = [0.0] * 6
    for _ in range(K_steps):
        se = made_events(7)
        flush()
        se[0].record()
        gmlp.backward_wgrad(xin, dy, h, probs, f1, splits, w.act, workspace=wws, events=se[1:], **grads)
        torch.cuda.synchronize()
        for i in range(6):
            wst[i] += se[i].elapsed_time(se[i + 1]) / K_steps
    gmlp.check_device_status()
    del grads, wws, f1
    hbm, bf16_burst, _, _ = peaks()
    fp8 = bf16_burst * NOMINAL_RATIO[gmlp.MXFP8]
    M, K, N, N1 = w.M, w.K, w.N, w.n1

    def tensor(name, flops, ms):
        tf = flops / (ms * 1e-3) / 1e12
        kern[name] = {"bound": "tensor", "ms": round(ms, 5), "TFLOP_s": round(tf, 1), "frac": round(tf / fp8, 4)}

    def mem(name, nbytes, ms):
        gbs = nbytes / (ms * 1e-3) / 1e9
        kern[name] = {"bound": "hbm", "ms": round(ms, 5), "GB_s": round(gbs, 1), "frac": round(gbs / hbm, 4)}

    colq = M * (1 + 1 / 32)  # codes + scales written per column (padding excluded)
    mem("dy columnwise cast", M * K * 2 + K * colq, wst[0])
    mem("fc2_x rebuild + columnwise cast", M * N1 * 2 + M * 4 + N * colq, wst[1])
    tensor("dW2 GEMM", 2.0 * M * K * N, wst[2])
    mem("fc1_dy columnwise cast", M * N1 * 2 + N1 * colq, wst[3])
    mem("x columnwise cast", M * K * 2 + K * colq, wst[4])
    tensor("dW1 GEMM", 2.0 * M * N1 * K, wst[5])
    wgrad = {"what": "dW1, dW2 (FP32) and dbias1, dbias2: columnwise MXFP8 of dy, fc2_x (rebuilt from the saved "
                     "activation input), fc1_dy and x, two grouped wgrad GEMMs over each expert's tokens",
             "ms_per_step": round(wms, 5), "flops_per_step": flops, "TFLOP_s": round(flops / (wms * 1e-3) / 1e12, 2),
             "kernels": kern,
             "roofline_note": "per kernel, from a second pass with an event after every kernel; tensor kernels "
                              f"against the measured bf16 burst x {NOMINAL_RATIO[gmlp.MXFP8]} (FP8), casts "
                              "against the measured HBM copy bandwidth; algorithmic bytes"}
    return {"what": "dx and dprob: dy MXFP8 cast, fc2 dGLU GEMM (fused dact x prob, dprob, MXFP8 fc1_dy), "
                    "fc1 dgrad GEMM",
            "wgrad": wgrad,
            "ms_per_step": round(ms, 5), "flops_per_step": flops, "TFLOP_s": round(flops / (ms * 1e-3) / 1e12, 2),
            "stages_ms": [round(t, 5) for t in st],
            "stage_tflops": {"dglu": round(2.0 * w.M * w.K * w.N / (st[1] * 1e-3) / 1e12, 1),
                             "dgrad": round(2.0 * w.M * w.n1 * w.K / (st[2] * 1e-3) / 1e12, 1)},
            "kernels": {
                "dy cast (+ dprob memset)": {"bound": "hbm", "ms": round(st[0], 5),
                                             "GB_s": round((M * K * (3 + 1 / 32)) / (st[0] * 1e-3) / 1e9, 1),
                                             "frac": round((M * K * (3 + 1 / 32)) / (st[0] * 1e-3) / 1e9 / hbm, 4)},
                "dGLU GEMM": {"bound": "tensor", "ms": round(st[1], 5),
                              "frac": round(2.0 * M * K * N / (st[1] * 1e-3) / 1e12 / fp8, 4)},
                "dgrad GEMM": {"bound": "tensor", "ms": round(st[2], 5),
                               "frac": round(2.0 * M * N1 * K / (st[2] * 1e-3) / 1e12 / fp8, 4)}}}


def bench_quantizer(gmlp, dev, hbm, rows: int = 0) -> dict:
    """Standalone NVFP4 group Hadamard-amax + quantize-with-amax (row + column,
    RHT) on bf16 [131072, 4096], 8 groups (inputs 1 GiB, larger than L2).
    rows > 0 takes only the first `rows` tokens (the groups cut to fit; a
    smaller case for profiling)."""
    d = make_inputs("nv_quant")
    w = d["workload"]
    x, sp = d["x"], d["splits"]
    if 0 < rows < w.M:
        cut = np.minimum(np.cumsum(sp.numpy()), rows)
        sp = torch.from_numpy(np.diff(np.concatenate([[0], cut])))
        x = x[:rows].contiguous()
    M, K = x.shape
    x = x.to(dev)
    splits = sp.to(dev)
    sh = sp.tolist()
    rec = gmlp.recipe(gmlp.NVFP4, use_rht=True, mask=d["mask"])
    reps = 10
    for _ in range(2):
        pre, post = gmlp.group_hadamard_amax(x, splits, d["mask"])
    torch.cuda.synchronize()
    e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    e[0].record()
    for _ in range(reps):
        gmlp.group_hadamard_amax(x, splits, d["mask"])
    e[1].record()
    torch.cuda.synchronize()
    t_amax = e[0].elapsed_time(e[1]) / reps
    for _ in range(2):
        out = gmlp.group_quantize_with_amax(x, splits, rec, pre, post, rowwise=True, columnwise=True, splits_host=sh)
    torch.cuda.synchronize()
    e[0].record()
    for _ in range(reps):
        out = gmlp.group_quantize_with_amax(x, splits, rec, pre, post, rowwise=True, columnwise=True, splits_host=sh)
    e[1].record()
    torch.cuda.synchronize()
    gmlp.check_device_status()
    t_cast = e[0].elapsed_time(e[1]) / reps
    mpad = sum((m + 15) // 16 * 16 for m in sh)
    rd = M * K * 2
    wr = M * K // 2 + M * K // 16 + K * mpad // 2 + K * mpad // 16
    del out, x
    return {"workload": f"nv_quant: NVFP4 group quantise, bf16 [{M}, {K}], 8 groups Dirichlet(0.5), "
                        "row + column (RHT)",
            "timing": "mean of 10 back-to-back launches (inputs of 1 GiB, larger than L2)",
            "hadamard_amax": {"ms": round(t_amax, 4), "bytes": rd, "GB_s": round(rd / t_amax / 1e6, 1),
                              "frac_hbm": round(rd / t_amax / 1e6 / hbm, 4)},
            "quantize_with_amax": {"ms": round(t_cast, 4), "bytes": rd + wr,
                                   "GB_s": round((rd + wr) / t_cast / 1e6, 1),
                                   "frac_hbm": round((rd + wr) / t_cast / 1e6 / hbm, 4)}}


# ------------------------------------------------------------------ CPU oracle

class OracleSteps:
    """Bounded samples of a workload for the oracle on the host cores.  Step i
    runs the oracle's forward on one expert, rotating over the non-empty
    experts: all of its tokens for NVFP4 (its amaxes need the whole group),
    at most `rows` random tokens of it for MXFP8 (MXFP8 rows are independent,
    so a row's result does not depend on the others).  An expert's weights are
    quantised by the oracle the first time the expert is used, before its step
    is timed (the GPU arm also quantises weights before timing)."""

    def __init__(self, name: str, rows: int = 128):
        import oracle
        self.oracle = oracle
        self.d = make_inputs(name)
        self.w = self.d["workload"]
        self.xb, self.W1, self.W2 = bits(self.d["x"]), bits(self.d["W1"]), bits(self.d["W2"])
        self.probs = self.d["probs"].numpy()
        sp = self.d["splits"].numpy()
        self.offs = np.concatenate([[0], np.cumsum(sp)])
        self.experts = [g for g in range(self.w.G) if sp[g] > 0]
        self.rows = rows
        self.qw = {}
        self.rng = np.random.default_rng(0)

    def prepare(self, i: int):
        """(expert, token indices) of step i, with the expert's weights quantised."""
        w, o = self.w, self.oracle
        e = self.experts[i % len(self.experts)]
        if e not in self.qw:
            self.qw[e] = (o.quantize_weights(self.W1[e:e + 1], w.fmt), o.quantize_weights(self.W2[e:e + 1], w.fmt))
        lo, hi = int(self.offs[e]), int(self.offs[e + 1])
        idx = np.arange(lo, hi)
        if w.fmt == 0 and hi - lo > self.rows:
            idx = np.sort(self.rng.choice(idx, self.rows, replace=False))
        return e, idx

    def run(self, e: int, idx) -> float:
        """One oracle forward of expert e on tokens idx; returns its GEMM FLOPs."""
        w = self.w
        q1, q2 = self.qw[e]
        self.oracle.forward(np.ascontiguousarray(self.xb[idx]), [len(idx)], self.W1[e:e + 1], self.W2[e:e + 1],
                            self.probs[idx], w.act, w.fmt, qw1=q1, qw2=q2, rht_mask=self.d["mask"],
                            tanh_clamp_scale=w.tanh_clamp_scale)
        return 2.0 * len(idx) * w.K * w.n1 + 2.0 * len(idx) * w.N * w.K

    def describe(self) -> str:
        what = "all tokens of one expert" if self.w.fmt == 1 else f"at most {self.rows} random tokens of one expert"
        return (f"per step {what}, experts in turn ({len(self.experts)} non-empty of {self.w.G}); numpy float64 "
                "GEMMs + C format arithmetic; weights quantised before timing")


def oracle_sample(name: str, target_s: float = 15.0) -> dict:
    """The oracle as it stands on the host cores, on bounded samples of the
    workload (OracleSteps), repeated until about target_s of CPU work."""
    st = OracleSteps(name)
    flops = el = 0.0
    i = 0
    while el < target_s and i < 4 * len(st.experts):
        e, idx = st.prepare(i)
        t0 = time.time()
        flops += st.run(e, idx)
        el += time.time() - t0
        i += 1
    return {"value": round(flops / el / 1e12, 6), "unit": "TFLOP/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{i} oracle forward steps of {name} ({flops / 1e9:.1f} GFLOP, {el:.1f} s): {st.describe()}"}


def oracle_backward_sample(name: str, max_tokens: int = 16384, max_experts: int = 8, target_s: float = 10.0,
                           max_reps: int = 3) -> dict:
    """The oracle's backward (data, weight and bias gradients) on the host
    cores, on whole experts of the workload, smallest first, up to max_tokens
    tokens and max_experts experts (the weight gradients contract over each
    expert's tokens, so experts are not cut), repeated until about target_s of
    CPU work."""
    import oracle
    d = make_inputs(name)
    w = d["workload"]
    sp = d["splits"].numpy()
    offs = np.concatenate([[0], np.cumsum(sp)])
    picked, tok = [], 0
    for g in np.argsort(sp):                      # smallest non-empty experts first
        if sp[g] > 0 and tok + sp[g] <= max_tokens and len(picked) < max_experts:
            picked.append(int(g))
            tok += int(sp[g])
    picked.sort()
    rows = np.concatenate([np.arange(offs[g], offs[g + 1]) for g in picked])
    ssp = np.array([sp[g] for g in picked])
    gen = torch.Generator().manual_seed(w.seed + 77)
    dy = torch.randn((len(rows), w.K), generator=gen).to(torch.bfloat16)
    h = (1.5 * torch.randn((len(rows), w.n1), generator=gen)).to(torch.bfloat16)
    xs, W1, W2 = bits(d["x"])[rows], bits(d["W1"])[picked], bits(d["W2"])[picked]
    probs = d["probs"].numpy()[rows]
    t0 = time.time()
    reps = 0
    while True:
        rb = oracle.backward_dgrad(bits(dy), ssp, W1, W2, bits(h), probs, w.act)
        oracle.backward_wgrad(xs, bits(dy), bits(h), probs, rb["fc1_dy"], ssp, w.act)
        reps += 1
        el = time.time() - t0
        if el >= target_s or reps >= max_reps:
            break
    m = len(rows)
    flops = reps * 2 * (2.0 * m * w.K * w.N + 2.0 * m * w.n1 * w.K)
    cores = oracle_threads()
    return {"value": round(flops / el / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} backward(s) of experts {picked} of {name} ({m} tokens): backward_dgrad + "
                      f"backward_wgrad (weights quantised inside), {el:.1f} s, numpy float64 GEMMs + C format "
                      "arithmetic"}


def run_reference(args) -> dict:
    """The reference arm: the oracle on the host, each step a bounded sample of
    the same workload (OracleSteps: one expert per step)."""
    st = OracleSteps(args.workload)
    w = st.w
    n = args.warmup + args.steps
    plan = [st.prepare(i) for i in range(n)]
    for e, idx in plan[:args.warmup]:
        st.run(e, idx)
    flops = 0.0
    t0 = time.time()
    for e, idx in plan[args.warmup:]:
        flops += st.run(e, idx)
    el = time.time() - t0
    v = flops / el / 1e12
    cores = oracle_threads()
    return {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT.get(args.workload)}",
                                            "flops_per_step": w.flops},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": st.describe()},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gmlp", choices=["gmlp", "reference"])
    ap.add_argument("--workload", default="mx_skew", choices=[k for k in WORKLOADS if k != "nv_quant"])
    ap.add_argument("--gemm-mode", type=int, default=0, choices=[0, 2],
                    help="0: one CTA per 128x256 tile; 2: CTA pairs on 256x256 tiles")
    ap.add_argument("--backward", dest="backward", action="store_true", default=True,
                    help="time the backward (data and weight gradients) on the MXFP8 SwiGLU leg (the default)")
    ap.add_argument("--no-backward", dest="backward", action="store_false", help="skip the backward leg")
    ap.add_argument("--no-extra", dest="extra", action="store_false",
                    help="skip the other workloads' forward legs (nv_srelu, mx_swiglu)")
    ap.add_argument("--extra-steps", type=int, default=50, help="timed steps of each extra leg (at most --steps)")
    ap.add_argument("--weight-scales", default="auto", choices=["auto", "x4", "tiled"],
                    help="weight scale layout the forward GEMMs read: auto = GEMM_TILED, except the replicated "
                         "GEMM_TILED_X4 copy for NVFP4 in CTA-pair mode; x4 (NVFP4 only); tiled")
    ap.add_argument("--fc2x-colwise", action="store_true",
                    help="NVFP4: also write the columnwise (RHT) NVFP4 fc2_x each step (no-recompute training path)")
    ap.add_argument("--l2-flush", default="clean", choices=["write", "clean"],
                    help="between timed steps: write 256 MiB, or write 256 MiB then read another 256 MiB")
    ap.add_argument("--e2e-streams", type=int, default=1,
                    help="e2e leg: copy x and y as this many row slices on as many streams per direction")
    ap.add_argument("--no-quant", dest="quant", action="store_false", help="skip the standalone quantiser leg")
    ap.add_argument("--quant-only", action="store_true",
                    help="run only the standalone NVFP4 quantiser leg and print its JSON")
    ap.add_argument("--quant-rows", type=int, default=0,
                    help="standalone quantiser leg on the first N tokens only (a smaller case for profiling)")
    ap.add_argument("--no-cpu", dest="cpu", action="store_false", help="skip the oracle CPU-baseline leg")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a GPU for the gmlp arm")
    if args.quant_only:
        from mxfp8_nvfp4_block_gb300 import gmlp
        gmlp.load()
        if rank == 0:
            print(json.dumps(bench_quantizer(gmlp, torch.device("cuda", torch.cuda.current_device()), peaks()[0],
                                             args.quant_rows)))
        return
    out = run_gpu(args, rank, world)
    if rank == 0:
        if args.cpu:
            out["cpu_baseline"] = oracle_sample(args.workload)
            bwd = out.get("backward_dgrad") or out.get("workloads", {}).get("mx_swiglu", {}).get("backward_dgrad")
            if bwd is not None:
                bwd["cpu_baseline"] = oracle_backward_sample("mx_swiglu")
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
