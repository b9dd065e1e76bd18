#!/usr/bin/env python3
"""Benchmark of the low-precision MoE expert path on GB300.

One step = one pass of the whole hot path over one batch of the skewed
long-batch MoE workload (32 experts, hidden 7168, intermediate 2048, 262144
routed rows, Zipf(1.2) loads with 3 empty experts):

  forward (NVFP4):  quantize X and W_gate/up -> grouped GEMM gate/up,
                    quantize H and W_down    -> grouped GEMM down
  backward (MXFP8): quantize dY row-wise and column-wise in one pass,
                    W_down column-wise -> dgrad; H column-wise -> wgrad

11 launches of libfme.so per step, inputs resident in HBM (every input is
larger than the 129 MB L2).  The headline value is grouped-GEMM TFLOP/s over
the whole step (GEMM FLOPs / step time, quantizers included); each call's time,
GB/s or TFLOP/s and roofline fraction are reported in "breakdown".

--impl reference times the CPU oracle (oracle/) on a bounded sample of the
same workload, the only other place this file runs the oracle.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "grouped expert GEMM TFLOP/s & quantize GB/s on 1 GB300, % of FP4/FP8/HBM roofline"
WORKLOADS = {
    # the skewed long-batch stress case: the largest single-GPU workload, every step of the path
    "moe-fwd-bwd-zipf-262144": dict(rows=262144, experts=32, loads="zipf", seed=4),
    # the forward/backward pair at 65536 routed rows with Dirichlet(1) loads
    "moe-fwd-bwd-dirichlet-65536": dict(rows=65536, experts=32, loads="dirichlet", seed=2),
    # a small case (8 experts, about 2 GB on the device) for ncu captures
    "profile-8x16384": dict(rows=16384, experts=8, loads="dirichlet", seed=2),
}
DEFAULT_WORKLOAD = "moe-fwd-bwd-zipf-262144"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# dense tensor-core throughput relative to bf16 (nominal GB300 figures: bf16 2.25, fp8 4.5, fp4 13.5 PF)
DTYPE_RATIO = {"fp8": 4.5 / 2.25, "fp4": 13.5 / 2.25}
# What the tensor pipe itself delivers on this GB300 for the MMA shape the
# kernels issue (cta_group::2, M = 256, N = 256; K = 64 FP4 or 32 FP8), measured
# with back-to-back MMAs on every SM at 2.07 GHz: 65 ns per instruction for both.
PIPE_RATE_TFLOPS = {"fp4": 9749.0, "fp8": 4866.0}


# --------------------------------------------------------------------- helpers --
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The slowest rank's time: an all-reduce MAX over the process group (any backend)."""
    if world <= 1:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, flops_per_rank: float, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: every rank's work over the slowest rank's step time."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def counts_for(wl):
    from fp8_moe_expert_gb300 import synth

    if wl["loads"] == "zipf":
        return synth.zipf_counts(rows=wl["rows"], experts=wl["experts"], seed=wl["seed"])
    return synth.dirichlet_counts(rows=wl["rows"], experts=wl["experts"], seed=wl["seed"])


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.reader.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
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
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ the step --
class MoEStep:
    """Device buffers of one MoE-layer forward+backward and the 11 calls over them."""

    CALLS = ["quant_x_nvfp4", "quant_wgu_nvfp4", "gemm_fwd_gate_up", "quant_h_nvfp4", "quant_wd_nvfp4",
             "gemm_fwd_down", "quant_dy_rowcol_mxfp8", "quant_wd_cols_mxfp8", "gemm_dgrad",
             "quant_h_cols_mxfp8", "gemm_wgrad"]

    def __init__(self, counts, seed, device, inputs_only=False):
        import torch

        import fp8_moe_expert_gb300 as fme
        from fp8_moe_expert_gb300 import synth

        self.fme = fme
        self.counts = counts
        E, H, I = len(counts), synth.HIDDEN, synth.INTERMEDIATE
        R = int(sum(counts))
        self.E, self.H, self.I, self.R = E, H, I, R
        dev = device
        self.dev = dev
        self.offsets = torch.from_numpy(synth.offsets_from_counts(counts)).to(dev)
        # inputs (bf16, seeded, made on the device)
        self.x = synth.torch_normal((R, H), 1.0, seed * 10 + 1, dev)
        self.w_gu = synth.torch_normal((E * 2 * I, H), 0.02, seed * 10 + 2, dev)
        self.h = synth.torch_normal((R, I), 1.0, seed * 10 + 3, dev)
        self.w_d = synth.torch_normal((E * H, I), 0.02, seed * 10 + 4, dev)
        self.dy = synth.torch_normal((R, H), 1e-2, seed * 10 + 5, dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        if inputs_only:
            return
        u8, f32, bf16, i32 = torch.uint8, torch.float32, torch.bfloat16, torch.int32
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)  # noqa: E731
        # quantized operands and outputs, allocated once
        self.xq = (e((R, H // 2), u8), e((fme.sf_bytes(R, H, 16, E),), u8), e((R,), f32))
        self.wguq = (e((E * 2 * I, H // 2), u8), e((fme.sf_bytes(E * 2 * I, H, 16, 1),), u8), e((E * 2 * I,), f32))
        self.hq = (e((R, I // 2), u8), e((fme.sf_bytes(R, I, 16, E),), u8), e((R,), f32))
        self.wdq = (e((E * H, I // 2), u8), e((fme.sf_bytes(E * H, I, 16, 1),), u8), e((E * H,), f32))
        self.y_gu = e((R, 2 * I), bf16)
        self.y_d = e((R, H), bf16)
        self.dyr = (e((R, H), u8), e((fme.sf_bytes(R, H, 32, E),), u8))
        self.ld_w = fme.colwise_ld(E * H, 1)
        self.wdc = (e((I, self.ld_w), u8), e((fme.sf_bytes(I, self.ld_w, 32, 1),), u8), e((2,), i32))
        self.dh = e((R, I), bf16)
        self.ld_r = fme.colwise_ld(R, E)
        self.dyc = (e((H, self.ld_r), u8), e((fme.sf_bytes(H, self.ld_r, 32, 1),), u8), e((E + 1,), i32))
        self.hc = (e((I, self.ld_r), u8), e((fme.sf_bytes(I, self.ld_r, 32, 1),), u8), e((E + 1,), i32))
        self.dw = e((E, H, I), bf16)

    # algorithmic work per call: ("bytes"|"flops", amount)
    def work(self):
        R, H, I, E = self.R, self.H, self.I, self.E
        # per row: bf16 in, E2M1 codes, E4M3 block scales, fp32 row scale
        nv = lambda rows, k: rows * (2 * k + k // 2 + k // 16 + 4)  # noqa: E731
        mx = lambda rows, c: rows * (2 * c + c + c // 32)  # noqa: E731
        return {
            "quant_x_nvfp4": ("bytes", nv(R, H)),
            "quant_wgu_nvfp4": ("bytes", nv(E * 2 * I, H)),
            "gemm_fwd_gate_up": ("flops", 2 * R * 2 * I * H),
            "quant_h_nvfp4": ("bytes", nv(R, I)),
            "quant_wd_nvfp4": ("bytes", nv(E * H, I)),
            "gemm_fwd_down": ("flops", 2 * R * H * I),
            # one read of dY, row-wise and column-wise outputs
            "quant_dy_rowcol_mxfp8": ("bytes", R * (2 * H + 2 * (H + H // 32))),
            "quant_wd_cols_mxfp8": ("bytes", mx(E * H, I)),
            "gemm_dgrad": ("flops", 2 * R * I * H),
            "quant_h_cols_mxfp8": ("bytes", mx(R, I)),
            "gemm_wgrad": ("flops", 2 * R * H * I),
        }

    def gemm_dtype(self, call):
        return "fp4" if call.startswith("gemm_fwd") else "fp8"

    def calls(self):
        f, off, st, E, H, I = self.fme, self.offsets, self.status, self.E, self.H, self.I
        return [
            lambda: f.quantize_nvfp4_pertoken(self.x, off, codes=self.xq[0], sf=self.xq[1], row_scale=self.xq[2],
                                              status=st),
            lambda: f.quantize_nvfp4_pertoken(self.w_gu, codes=self.wguq[0], sf=self.wguq[1], row_scale=self.wguq[2],
                                              status=st),
            lambda: f.grouped_gemm_fwd_nvfp4(*self.xq, *self.wguq, off, 2 * I, H, y=self.y_gu, status=st),
            lambda: f.quantize_nvfp4_pertoken(self.h, off, codes=self.hq[0], sf=self.hq[1], row_scale=self.hq[2],
                                              status=st),
            lambda: f.quantize_nvfp4_pertoken(self.w_d, codes=self.wdq[0], sf=self.wdq[1], row_scale=self.wdq[2],
                                              status=st),
            lambda: f.grouped_gemm_fwd_nvfp4(*self.hq, *self.wdq, off, H, I, y=self.y_d, status=st),
            lambda: f.quantize_mxfp8_rowcol(self.dy, off, row_codes=self.dyr[0], row_sf=self.dyr[1],
                                            col_codes=self.dyc[0], col_sf=self.dyc[1], padded_offsets=self.dyc[2],
                                            status=st),
            lambda: f.quantize_mxfp8(self.w_d, f.COLWISE, codes=self.wdc[0], sf=self.wdc[1], padded_offsets=self.wdc[2],
                                     status=st),
            lambda: f.grouped_gemm_dgrad_mxfp8(*self.dyr, self.wdc[0], self.wdc[1], self.ld_w, off, I, H, y=self.dh,
                                               status=st),
            lambda: f.quantize_mxfp8(self.h, f.COLWISE, off, codes=self.hc[0], sf=self.hc[1], padded_offsets=self.hc[2],
                                     status=st),
            lambda: f.grouped_gemm_wgrad_mxfp8(self.dyc[0], self.dyc[1], self.ld_r, self.hc[0], self.hc[1], self.ld_r,
                                               self.dyc[2], H, I, y=self.dw, status=st),
        ]

    def gemm_flops(self):
        return sum(v for k, (kind, v) in self.work().items() if kind == "flops")

    def inputs(self):
        return [self.x, self.w_gu, self.h, self.w_d, self.dy]

    def outputs(self):
        return [self.y_gu, self.y_d, self.dh, self.dw]


def run_ours(args, rank, world, local_rank):
    import torch

    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    import fp8_moe_expert_gb300 as fme

    fme.lib()  # fails loudly without the CUDA library
    wl = WORKLOADS[args.workload]
    counts = counts_for(wl)
    step = MoEStep(counts, wl["seed"], dev)
    calls = step.calls()
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        for c in calls:
            c()
    torch.cuda.synchronize()
    code, raw = fme.read_device_status(step.status)
    if code != 0:
        raise RuntimeError(f"device status {raw:#x} after warm-up")

    # ------------------------------------------------------------ timed region
    n_calls = len(calls)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_calls + 1)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        start.record(stream)
        for s in range(args.steps):
            for i, c in enumerate(calls):
                ev[s][i].record(stream)
                c()
            ev[s][n_calls].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(end), world, dev)
    code, raw = fme.read_device_status(step.status)
    if code != 0:
        raise RuntimeError(f"device status {raw:#x} in the timed region")

    per_call = {name: statistics.mean(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(args.steps))
                for i, name in enumerate(MoEStep.CALLS)}
    ms_per_step = elapsed_ms / args.steps
    flops = step.gemm_flops()
    value = job_value(world, flops, ms_per_step)

    peaks, peak_kind = load_peaks()
    # Each call is timed on its own (a few ms): the burst bf16 figure is the
    # denominator; the sustained one (a seconds-long loop under the power cap) is
    # reported beside it.
    bf16_burst = float(peaks["bf16_tflops"])
    bf16_sus = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    hbm = float(peaks["hbm_gbs"])
    breakdown = {}
    for name, (kind, amount) in step.work().items():
        ms = per_call[name]
        if kind == "bytes":
            ach = amount / (ms * 1e-3) / 1e9
            breakdown[name] = {"ms": round(ms, 4), "GB/s": round(ach, 1), "frac_hbm": round(ach / hbm, 3)}
        else:
            ach = amount / (ms * 1e-3) / 1e12
            dt = step.gemm_dtype(name)
            breakdown[name] = {"ms": round(ms, 4), "TFLOP/s": round(ach, 1),
                               f"frac_{dt}": round(ach / (bf16_burst * DTYPE_RATIO[dt]), 3),
                               f"frac_{dt}_sustained": round(ach / (bf16_sus * DTYPE_RATIO[dt]), 3)}
    top = max(per_call, key=per_call.get)
    kind, amount = step.work()[top]
    if kind == "flops":
        dt = step.gemm_dtype(top)
        pk = bf16_burst * DTYPE_RATIO[dt]
        ach = amount / (per_call[top] * 1e-3) / 1e12
        roof = {"kernel": top, "bound": "tensor", "achieved": round(ach, 1), "peak": round(pk, 1),
                "unit": "TFLOP/s", "frac": round(ach / pk, 3),
                "frac_sustained": round(ach / (bf16_sus * DTYPE_RATIO[dt]), 3),
                "peak_source": f"{peak_kind} bf16_tflops (burst) x {DTYPE_RATIO[dt]:g} ({dt} / bf16 nominal ratio)",
                "pipe_rate": PIPE_RATE_TFLOPS.get(dt)}
    else:
        ach = amount / (per_call[top] * 1e-3) / 1e9
        roof = {"kernel": top, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 3), "peak_source": f"{peak_kind} hbm_gbs"}
    roof["traffic"] = lookup_traffic(top, args.workload)

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 fwd / mxfp8 bwd, fp32 accumulate",
        "data": "synthetic (seeded torch normal on device; Zipf/Dirichlet expert loads from numpy)",
        "config": {"workload": args.workload, "experts": step.E, "hidden": step.H, "intermediate": step.I,
                   "routed_rows": step.R, "expert_rows_max": int(max(counts)),
                   "empty_experts": int(sum(1 for c in counts if c == 0)),
                   "l2": "inputs larger than L2 (129 MB) every call", "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "breakdown": breakdown,
        "gpu_launches": n_calls * args.steps,
        "clocks": clocks.summary(),
    }
    if not args.no_extras:
        # the extras follow the step back to back; their clocks are recorded apart,
        # since the instruction-bound ones follow the SM clock where copies do not
        with ClockSampler(local_rank) as extras_clocks:
            line["extras"] = run_extras(step, args, bf16_burst)
        line["extras_clocks"] = extras_clocks.summary()
    if not args.no_e2e:
        line["e2e"] = run_e2e(step, calls, args, world)
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(step, counts)
    elif rank == 0 and world > 1:
        line["cpu_baseline"] = None
    return line


def run_extras(step, args, bf16_peak):
    """Calls beyond the step's path, timed on the same workload after it (not part
    of `value`): the MXFP8 forward grouped GEMMs (gate/up and down) on row-wise
    MXFP8 operands, and the fused SwiGLU + NVFP4 quantization of the gate/up
    output (writing h for the backward).  CUDA events on the launching stream, 3
    warm-up and `args.steps` timed launches each."""
    import torch

    f, off, st = step.fme, step.offsets, step.status
    R, H, I, E = step.R, step.H, step.I, step.E
    xq = f.quantize_mxfp8(step.x, f.ROWWISE, off, status=st)
    wq = f.quantize_mxfp8(step.w_gu, f.ROWWISE, status=st)
    hq = f.quantize_mxfp8(step.h, f.ROWWISE, off, status=st)
    wdq = f.quantize_mxfp8(step.w_d, f.ROWWISE, status=st)
    out = {}
    hbm = float(load_peaks()[0]["hbm_gbs"])
    h_out = torch.empty_like(step.h)
    sw_bytes = R * (2 * 2 * I + 2 * I + I // 2 + I // 16 + 4)  # gate/up in; h, codes, scales, row scale out
    fn = lambda: f.swiglu_quantize_nvfp4(step.y_gu, off, codes=step.hq[0], sf=step.hq[1],  # noqa: E731
                                         row_scale=step.hq[2], h=h_out, status=st)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    gbs = sw_bytes / (ms * 1e-3) / 1e9
    out["swiglu_quantize_nvfp4"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3)}
    del h_out
    for name, fn, flops in (
            ("gemm_fwd_gate_up_mxfp8",
             lambda: f.grouped_gemm_fwd_mxfp8(*xq, *wq, off, 2 * I, H, y=step.y_gu, status=st), 2 * R * 2 * I * H),
            ("gemm_fwd_down_mxfp8",
             lambda: f.grouped_gemm_fwd_mxfp8(*hq, *wdq, off, H, I, y=step.y_d, status=st), 2 * R * H * I)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.steps
        ach = flops / (ms * 1e-3) / 1e12
        out[name] = {"ms": round(ms, 4), "TFLOP/s": round(ach, 1), "frac_fp8": round(ach / (bf16_peak * 2), 3)}
    del xq, wq, hq, wdq
    out.update(run_routing_extras(step, args, hbm))
    # the down projection's wgrad added into an fp32 gradient buffer (accumulation)
    acc = torch.zeros((E, H, I), dtype=torch.float32, device=step.dev)
    ms = _time_call(lambda: f.grouped_gemm_wgrad_mxfp8_accumulate(step.dyc[0], step.dyc[1], step.ld_r, step.hc[0],
                                                                  step.hc[1], step.ld_r, step.dyc[2], H, I, acc,
                                                                  status=st), args.steps)
    ach = 2 * R * H * I / (ms * 1e-3) / 1e12
    out["gemm_wgrad_accumulate_fp32"] = {"ms": round(ms, 4), "TFLOP/s": round(ach, 1),
                                         "frac_fp8": round(ach / (bf16_peak * 2), 3)}
    del acc
    out.update(run_gate_up_bwd_extras(step, args, hbm, bf16_peak))  # reuses the dY column-wise buffers
    h_out = torch.empty_like(step.h)
    # f1's variant, timed last (its FP4 GEMMs run at full power, and the calls timed
    # after them would start power-capped): SwiGLU in the gate/up GEMM's epilogue (bf16 h out, half the
    # bytes of gate/up), then the per-token NVFP4 quantization of h; its chain
    # against the gate/up GEMM followed by the fused SwiGLU + NVFP4 quantization
    fl_gu = 2 * R * 2 * I * H
    calls_f1 = {
        "fused": lambda: f.grouped_gemm_fwd_nvfp4_swiglu(*step.xq, *step.wguq, off, 2 * I, H, h=h_out, status=st),
        "quant_h": lambda: f.quantize_nvfp4_pertoken(h_out, off, codes=step.hq[0], sf=step.hq[1],
                                                     row_scale=step.hq[2], status=st),
        "plain": lambda: f.grouped_gemm_fwd_nvfp4(*step.xq, *step.wguq, off, 2 * I, H, y=step.y_gu, status=st),
        "swiglu_quant": lambda: f.swiglu_quantize_nvfp4(step.y_gu, off, codes=step.hq[0], sf=step.hq[1],
                                                        row_scale=step.hq[2], status=st),
    }
    # the four calls interleaved, each bracketed by its own events, so that both chains
    # see the same clocks; medians over args.steps rounds
    for fn in calls_f1.values():
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    evs = {k: [] for k in calls_f1}
    for _ in range(args.steps):
        for k, fn in calls_f1.items():
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            evs[k].append((e0, e1))
    torch.cuda.synchronize()
    med = {k: statistics.median(e0.elapsed_time(e1) for e0, e1 in v) for k, v in evs.items()}
    ach = fl_gu / (med["fused"] * 1e-3) / 1e12
    out["gemm_fwd_gate_up_swiglu"] = {"ms": round(med["fused"], 4), "TFLOP/s": round(ach, 1),
                                      "frac_fp4": round(ach / (bf16_peak * 6), 3),
                                      "chain_ms": round(med["fused"] + med["quant_h"], 4),
                                      "unfused_chain_ms": round(med["plain"] + med["swiglu_quant"], 4),
                                      "plain_gemm_ms": round(med["plain"], 4)}
    del h_out
    return out


def run_gate_up_bwd_extras(step, args, hbm, bf16_peak):
    """The gate/up half of the backward on the same rows: the fused SwiGLU backward
    + MXFP8 row/column quantization of d(gate/up) [R x 2I] from the forward's
    gate/up output and dh, the column-wise quantization of X and of W_gu, and the
    gate/up dgrad (contraction over 2I = 4096) and wgrad (dW_gu [E x 2I x H])."""
    import torch

    f, off, st = step.fme, step.offsets, step.status
    R, H, I, E = step.R, step.H, step.I, step.E
    out = {}
    sb = f.swiglu_backward_quantize_mxfp8(step.y_gu, step.dh, off, status=st)
    rc, rs, cc, cs, poff, ld = sb[:6]
    sb_bytes = R * (2 * 2 * I + 2 * I + 2 * I + 2 * I + 2 * (2 * I // 32))
    ms = _time_call(lambda: f.swiglu_backward_quantize_mxfp8(step.y_gu, step.dh, off, row_codes=rc, row_sf=rs,
                                                             col_codes=cc, col_sf=cs, padded_offsets=poff,
                                                             status=st), args.steps)
    gbs = sb_bytes / (ms * 1e-3) / 1e9
    out["swiglu_backward_quantize_mxfp8"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                             "frac_hbm": round(gbs / hbm, 3)}
    xc = f.quantize_mxfp8(step.x, f.COLWISE, off, codes=step.dyc[0], sf=step.dyc[1], padded_offsets=step.dyc[2],
                          status=st)
    ld_w = f.colwise_ld(E * 2 * I, 1)
    wc = f.quantize_mxfp8(step.w_gu, f.COLWISE, status=st)
    dx = torch.empty((R, H), dtype=torch.bfloat16, device=step.dev)
    dw = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=step.dev)
    flops = 2 * R * 2 * I * H
    for name, fn in (
            ("gemm_dgrad_gate_up",
             lambda: f.grouped_gemm_dgrad_mxfp8(rc, rs, wc[0], wc[1], ld_w, off, H, 2 * I, y=dx, status=st)),
            ("gemm_wgrad_gate_up",
             lambda: f.grouped_gemm_wgrad_mxfp8(cc, cs, ld, xc[0], xc[1], xc[3], poff, 2 * I, H, y=dw, status=st))):
        ms = _time_call(fn, args.steps)
        ach = flops / (ms * 1e-3) / 1e12
        out[name] = {"ms": round(ms, 4), "TFLOP/s": round(ach, 1), "frac_fp8": round(ach / (bf16_peak * 2), 3)}
    code, raw = f.read_device_status(st)
    if code != 0:
        raise RuntimeError(f"gate/up backward extras: device status {code} ({raw:#x})")
    del sb, rc, rs, cc, cs, xc, wc, dx, dw
    return out


def _time_call(fn, steps):
    import torch

    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def run_routing_extras(step, args, hbm):
    """Routing around the expert GEMMs on the same rows: R = tokens x top-8 routed
    rows of 32768 tokens over the 32 experts (synthetic Zipf-popular choices).
    Grouping (3 launches), the grouped NVFP4 and MXFP8 quantizations that gather
    the tokens' rows, and the weighted combine of the down projection's output.
    GB/s counts every grouped row read once (the gather reads each token top_k
    times; L2 may serve some of those) and every output written once."""
    import torch

    from fp8_moe_expert_gb300 import synth

    f, st = step.fme, step.status
    R, H, E = step.R, step.H, step.E
    top_k = 8
    tokens = R // top_k
    ids_np, w_np = synth.topk_routing(tokens=tokens, top_k=top_k, experts=E)
    ids = torch.from_numpy(ids_np).to(step.dev)
    weights = torch.from_numpy(w_np).to(step.dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=step.dev)
    row_of = torch.empty((tokens, top_k), dtype=torch.int32, device=step.dev)
    src = torch.empty(R, dtype=torch.int32, device=step.dev)
    ws = torch.empty(f.route_workspace_bytes(tokens, top_k, E), dtype=torch.uint8, device=step.dev)
    x_tok = step.x[:tokens]
    out_tok = torch.empty((tokens, H), dtype=torch.bfloat16, device=step.dev)
    out = {}
    ms = _time_call(lambda: f.moe_route(ids, E, offsets=off, row_of=row_of, src_row=src, workspace=ws, status=st),
                    args.steps)
    out["moe_route"] = {"ms": round(ms, 4), "tokens": tokens, "top_k": top_k}
    q_bytes = R * (2 * H + H // 2 + H // 16 + 4)
    ms = _time_call(lambda: f.permute_quantize_nvfp4(x_tok, src, top_k, off, codes=step.xq[0], sf=step.xq[1],
                                                     row_scale=step.xq[2], status=st), args.steps)
    gbs = q_bytes / (ms * 1e-3) / 1e9
    out["permute_quantize_nvfp4"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3)}
    m_bytes = R * (2 * H + H + H // 32)
    ms = _time_call(lambda: f.permute_quantize_mxfp8(x_tok, src, top_k, off, codes=step.dyr[0], sf=step.dyr[1],
                                                     status=st), args.steps)
    gbs = m_bytes / (ms * 1e-3) / 1e9
    out["permute_quantize_mxfp8"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3)}
    c_bytes = R * (2 * H + 8) + tokens * 2 * H
    ms = _time_call(lambda: f.moe_combine(step.y_d, row_of, weights, out=out_tok, status=st), args.steps)
    gbs = c_bytes / (ms * 1e-3) / 1e9
    out["moe_combine"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3)}
    code, raw = f.read_device_status(st)
    if code != 0:
        raise RuntimeError(f"routing extras: device status {code} ({raw:#x})")
    del ids, weights, off, row_of, src, ws, out_tok
    return out


INPUT_NAMES = ("x", "w_gu", "h", "w_d", "dy")
OUTPUT_NAMES = ("y_gu", "y_d", "dh", "dw")


def run_e2e(step, calls, args, world):
    """Same metric through the public API with host buffers: every step copies its
    inputs from pinned host memory and every output back to pinned host memory.
    Steps are pipelined the way a user would run them: two device sets of inputs
    and outputs, copies in on one stream, the 11 calls on another, copies out on a
    third, ordered by events (step i's uploads overlap step i-1's calls and
    downloads).  The 19.3 GB of copies per step, not the kernels, set the pace:
    splitting each direction over two streams measured the same.  At least 3
    (and at least `args.warmup`) pipelined warm-up steps run first; the clock
    covers all three streams from the first timed upload to the last download."""
    import torch

    sets = [{n: getattr(step, n) for n in INPUT_NAMES + OUTPUT_NAMES}]
    sets.append({n: torch.empty_like(t) for n, t in sets[0].items()})
    h_in = {n: torch.empty(sets[0][n].shape, dtype=sets[0][n].dtype, pin_memory=True) for n in INPUT_NAMES}
    h_out = [{n: torch.empty(sets[0][n].shape, dtype=sets[0][n].dtype, pin_memory=True) for n in OUTPUT_NAMES}
             for _ in range(2)]
    for n in INPUT_NAMES:
        h_in[n].copy_(sets[0][n])
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    uploaded = [ev(), ev()]   # inputs of the set are on the device
    consumed = [ev(), ev()]   # the set's calls are done (inputs free, outputs ready)
    drained = [ev(), ev()]    # the set's outputs are on the host
    started = [False, False]

    def one(i):
        k = i % 2
        if started[k]:
            s_in.wait_event(consumed[k])
        with torch.cuda.stream(s_in):
            for n in INPUT_NAMES:
                sets[k][n].copy_(h_in[n], non_blocking=True)
            uploaded[k].record(s_in)
        s_run.wait_event(uploaded[k])
        if started[k]:
            s_run.wait_event(drained[k])
        for n, t in sets[k].items():
            setattr(step, n, t)
        with torch.cuda.stream(s_run):
            for c in calls:
                c()
            consumed[k].record(s_run)
        s_out.wait_event(consumed[k])
        with torch.cuda.stream(s_out):
            for n in OUTPUT_NAMES:
                h_out[k][n].copy_(sets[k][n], non_blocking=True)
            drained[k].record(s_out)
        started[k] = True

    steps = max(2, min(args.steps, 8))
    warm = max(3, args.warmup)
    for i in range(warm):
        one(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    cur = torch.cuda.current_stream()
    start.record(cur)
    for s_ in (s_in, s_run, s_out):
        s_.wait_event(start)
    for i in range(warm, warm + steps):
        one(i)
    for s_ in (s_in, s_run, s_out):
        cur.wait_stream(s_)
    end.record(cur)
    torch.cuda.synchronize()
    for n, t in sets[0].items():
        setattr(step, n, t)
    ms = max_over_ranks(start.elapsed_time(end) / steps, world, step.dev)
    bi = sum(t.numel() * t.element_size() for t in h_in.values())
    bo = sum(t.numel() * t.element_size() for t in h_out[0].values())
    return {"value": round(job_value(world, step.gemm_flops(), ms), 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 3), "steps": steps, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "pipelined": "uploads, calls and downloads on three streams, two device buffer sets"}


# --------------------------------------------------------- oracle (CPU) timing --
def oracle_host_sample(step, counts, rows_per_gemm, cols, rng_seed=0):
    """Host inputs of one oracle sample of the step: `rows_per_gemm` token rows of
    one expert through every GEMM (all output columns if cols is None, else `cols`
    sampled output columns; only the weight rows or columns those need), plus
    `rows_per_gemm` channel rows of that expert's wgrad.  Returns (host arrays,
    column selections, description)."""
    import numpy as np
    import torch

    from fp8_moe_expert_gb300.synth import bf16_bits_np

    E, H, I = step.E, step.H, step.I
    off = np.concatenate([[0], np.cumsum(counts)])
    live = [g for g, c in enumerate(counts) if c >= 2 * rows_per_gemm]
    g = min(live, key=lambda e: counts[e])  # smallest expert that holds the sample
    rng = np.random.default_rng(rng_seed)
    r = np.sort(rng.choice(np.arange(off[g], off[g + 1]), size=rows_per_gemm, replace=False))
    ri = torch.from_numpy(r).to(step.dev)

    def colsel(n):
        return np.arange(n) if cols is None else np.sort(rng.choice(n, size=min(cols, n), replace=False))

    sel = {"gu": colsel(2 * I), "d": colsel(H), "dg": colsel(I), "wg": colsel(I),
           "ch": np.sort(rng.choice(H, size=rows_per_gemm, replace=False))}
    host = {
        "x": bf16_bits_np(step.x[ri]), "h": bf16_bits_np(step.h[ri]), "dy": bf16_bits_np(step.dy[ri]),
        "wgu": bf16_bits_np(step.w_gu[g * 2 * I:(g + 1) * 2 * I][torch.from_numpy(sel["gu"]).to(step.dev)]),
        "wd": bf16_bits_np(step.w_d[g * H:(g + 1) * H]),
        "dy_e": bf16_bits_np(step.dy[off[g]:off[g + 1]]), "h_e": bf16_bits_np(step.h[off[g]:off[g + 1]]),
        "H": H,
    }
    n_e = int(counts[g])
    desc = (f"expert {g} ({n_e} rows): {len(r)} token rows through gate/up ({len(sel['gu'])} cols), down "
            f"({len(sel['d'])} cols), dgrad ({len(sel['dg'])} cols); wgrad {len(sel['ch'])} x {len(sel['wg'])} "
            f"over {n_e} rows; quantization of every operand row/column those need included")
    return host, sel, desc


def oracle_run_sample(task):
    """The oracle on one host sample (oracle_host_sample's arrays), on this process's
    core: every quantization those GEMM rows need, then the GEMMs.  Returns
    (seconds, gemm flops).  Module level, so that a spawned pool can run it."""
    import numpy as np

    import oracle

    host, sel = task
    orc = oracle.Oracle()
    H = host["H"]
    n_e = host["dy_e"].shape[0]
    t0 = time.perf_counter()
    # forward, NVFP4
    a = orc.dequant_nvfp4(*orc.quant_nvfp4(host["x"]))
    b = orc.dequant_nvfp4(*orc.quant_nvfp4(host["wgu"]))
    orc.gemm_abt(a, b)
    a = orc.dequant_nvfp4(*orc.quant_nvfp4(host["h"]))
    b = orc.dequant_nvfp4(*orc.quant_nvfp4(np.ascontiguousarray(host["wd"][sel["d"]])))
    orc.gemm_abt(a, b)
    # backward, MXFP8: dgrad (W_down column-wise along the hidden axis)
    a = orc.dequant_mxfp8(*orc.quant_mxfp8_rows(host["dy"]))
    ct, st, _ = orc.quant_mxfp8_cols(np.ascontiguousarray(host["wd"][:, sel["dg"]]), np.array([0, H]))
    orc.gemm_abt(a, orc.dequant_mxfp8(ct, st)[:, :H])
    # wgrad: dY_e and H_e column-wise over the expert's rows
    e_off = np.array([0, n_e])
    ca, sa, _ = orc.quant_mxfp8_cols(np.ascontiguousarray(host["dy_e"][:, sel["ch"]]), e_off)
    cb, sb, _ = orc.quant_mxfp8_cols(np.ascontiguousarray(host["h_e"][:, sel["wg"]]), e_off)
    orc.gemm_abt(orc.dequant_mxfp8(ca, sa), orc.dequant_mxfp8(cb, sb))
    secs = time.perf_counter() - t0
    k = host["x"].shape[0]
    I = host["h"].shape[1]
    flops = (2 * k * (len(sel["gu"]) * H + len(sel["d"]) * I + len(sel["dg"]) * H)
             + 2 * len(sel["ch"]) * len(sel["wg"]) * n_e)
    return secs, flops


def oracle_sample(step, counts, rows_per_gemm, cols, rng_seed=0):
    """Time the CPU oracle on one sample of the step, in this process (inputs are
    on the host before the clock starts).  Returns (seconds, gemm_flops, description)."""
    host, sel, desc = oracle_host_sample(step, counts, rows_per_gemm, cols, rng_seed)
    secs, flops = oracle_run_sample((host, sel))
    return secs, flops, desc


def oracle_quantize(task):
    """One oracle quantizer over a block of rows (bf16 bits); returns seconds.
    Column-wise blocks run along rows: a block of a multiple of 32 rows is
    quantized exactly as those rows of the whole tensor."""
    import numpy as np

    import oracle

    kind, x = task
    orc = oracle.Oracle()
    t0 = time.perf_counter()
    if kind == "nvfp4":
        orc.quant_nvfp4(x)
    elif kind == "mxfp8_rows":
        orc.quant_mxfp8_rows(x)
    else:
        orc.quant_mxfp8_cols(x, np.array([0, x.shape[0]]))
    return time.perf_counter() - t0


def _pool_ready(_):
    import oracle

    oracle.Oracle()
    return os.getpid()


def host_info():
    """The host the CPU numbers were taken on: usable cores, CPU model, architecture."""
    import platform

    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as fh:
                for line in fh:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    try:
        usable = len(os.sched_getaffinity(0))
    except AttributeError:
        usable = os.cpu_count()
    return {"nproc": usable, "cpu_count": os.cpu_count(), "cpu_model": model, "arch": platform.machine()}


QUANT_KINDS = ("nvfp4", "mxfp8_rows", "mxfp8_cols")


def quant_bytes(kind, rows, cols):
    """Algorithmic bytes of one quantizer call: bf16 in, codes, scales (and the
    per-token fp32 scale of NVFP4) out, as the GPU breakdown counts them."""
    if kind == "nvfp4":
        return rows * (2 * cols + cols // 2 + cols // 16 + 4)
    return rows * (2 * cols + cols + cols // 32)


def gpu_quantizer_batch(x_bits):
    """The three quantizers on the GPU over the whole quantizer batch (bf16 bits,
    uploaded once; larger than L2): GB/s by CUDA events, median of 5."""
    import numpy as np
    import torch

    import fp8_moe_expert_gb300 as fme

    rows, cols = x_bits.shape
    x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q4 = fme.quantize_nvfp4_pertoken(x, status=st)
    q8r = fme.quantize_mxfp8(x, fme.ROWWISE, status=st)
    q8c = fme.quantize_mxfp8(x, fme.COLWISE, status=st)
    calls = {
        "nvfp4": lambda: fme.quantize_nvfp4_pertoken(x, codes=q4[0], sf=q4[1], row_scale=q4[2], status=st),
        "mxfp8_rows": lambda: fme.quantize_mxfp8(x, fme.ROWWISE, codes=q8r[0], sf=q8r[1], status=st),
        "mxfp8_cols": lambda: fme.quantize_mxfp8(x, fme.COLWISE, codes=q8c[0], sf=q8c[1], padded_offsets=q8c[2],
                                                 status=st),
    }
    out = {}
    for kind, fn in calls.items():
        fn()
        ts = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        out[kind] = quant_bytes(kind, rows, cols) / (statistics.median(ts) * 1e-3) / 1e9
    code, raw = fme.read_device_status(st)
    if code != 0:
        raise RuntimeError(f"device status {raw:#x} in the quantizer-batch timing")
    return out


def oracle_rows_sample(step):
    """The oracle on a small sample of each NEXT row, on one host core, in the units
    the bench reports that row in (GB/s over the same per-row bytes; grouping in
    million assignments per second).  Inputs are copied to the host first."""
    import numpy as np

    import oracle
    from fp8_moe_expert_gb300 import synth
    from fp8_moe_expert_gb300.synth import bf16_bits_np

    orc = oracle.Oracle()
    H, I, E = step.H, step.I, step.E
    rows = 64
    gu = bf16_bits_np(step.y_gu[:rows])
    dh = bf16_bits_np(step.dh[:rows])
    x = bf16_bits_np(step.x[:rows])
    y = bf16_bits_np(step.y_d[:rows * 8])
    ids, w = synth.topk_routing(tokens=4096, top_k=8, experts=E)
    out = {}

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    s = timed(lambda: orc.quant_nvfp4(orc_bits(orc.swiglu(gu))))
    out["swiglu_quantize_nvfp4"] = rows * (2 * 2 * I + 2 * I + I // 2 + I // 16 + 4) / s / 1e9
    def swiglu_bwd_both():
        d = orc_bits(orc.swiglu_bwd(gu, dh))
        orc.quant_mxfp8_rows(d)
        orc.quant_mxfp8_cols(d, np.array([0, rows]))

    s = timed(swiglu_bwd_both)
    out["swiglu_backward_quantize_mxfp8"] = rows * (2 * 2 * I + 2 * I + 2 * I + 2 * I + 2 * (2 * I // 32)) / s / 1e9
    s = timed(lambda: orc.route(ids, E))
    out["moe_route_massign_per_s"] = ids.size / s / 1e6
    ro = np.arange(rows * 8, dtype=np.int32).reshape(rows, 8)
    s = timed(lambda: orc.combine(y, ro, w[:rows]))
    out["moe_combine"] = rows * (8 * (2 * H + 8) + 2 * H) / s / 1e9
    s = timed(lambda: orc.quant_nvfp4_pertensor(x))
    out["quantize_nvfp4_pertensor"] = rows * (2 * H + H // 2 + H // 16 + 4) / s / 1e9
    return {k: round(v, 4) for k, v in out.items()}


def orc_bits(v):
    """fp64 values -> bf16 bit patterns (nearest even), the oracle's inputs."""
    from fp8_moe_expert_gb300 import synth

    return synth.bf16_bits(v.astype("float32"))


def cpu_baseline(step, counts):
    """The oracle, as it stands, on the host's cores: the step's GEMM sample on one
    core and on every usable core (a spawned process pool, one sample per core),
    and the three quantizers on the whole 16384 x 7168 quantizer batch (one core:
    a 1024-row slice; every core: the whole tensor in row blocks), next to the
    GPU's GB/s on the same tensor.  About 15-30 s of host time."""
    import multiprocessing as mp

    from fp8_moe_expert_gb300 import synth

    info = host_info()
    cores = max(1, int(info["nproc"] or 1))
    s1, f1, desc = oracle_sample(step, counts, rows_per_gemm=16, cols=None)
    tasks = []
    for i in range(cores):
        host, sel, _ = oracle_host_sample(step, counts, rows_per_gemm=16, cols=None, rng_seed=100 + i)
        tasks.append((host, sel))
    x_bits, _, _ = synth.quantizer_batch()
    rows, cols = x_bits.shape
    blk = (-(-rows // cores) + 31) // 32 * 32  # ceil(rows / cores), a multiple of 32
    blocks = [x_bits[i:i + blk] for i in range(0, rows, blk)]
    single, allcore = {}, {}
    for kind in QUANT_KINDS:
        part = x_bits[:1024]
        single[kind] = quant_bytes(kind, part.shape[0], cols) / oracle_quantize((kind, part)) / 1e9
    with mp.get_context("spawn").Pool(cores) as pool:
        pool.map(_pool_ready, range(cores), chunksize=1)  # workers started and the oracle loaded
        t0 = time.perf_counter()
        res = pool.map(oracle_run_sample, tasks, chunksize=1)
        wall = time.perf_counter() - t0
        all_value = sum(f for _, f in res) / wall / 1e12
        for kind in QUANT_KINDS:
            t0 = time.perf_counter()
            pool.map(oracle_quantize, [(kind, b) for b in blocks], chunksize=1)
            allcore[kind] = quant_bytes(kind, rows, cols) / (time.perf_counter() - t0) / 1e9
    gpu = gpu_quantizer_batch(x_bits)
    return {
        "value": all_value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
        "sample": f"{cores} samples in parallel, one per core, each: {desc}",
        "single_core": {"value": f1 / s1 / 1e12, "unit": "TFLOP/s", "cores": 1, "seconds": round(s1, 3),
                        "sample": desc},
        "all_core_seconds": round(wall, 3),
        "host": info,
        "quantizers_16384x7168_gbs": {
            kind: {"oracle_1_core": round(single[kind], 4), f"oracle_{cores}_cores": round(allcore[kind], 4),
                   "gpu": round(gpu[kind], 1)} for kind in QUANT_KINDS},
        "quantizer_samples": "one core: rows 0-1023 of the batch; every core: the whole batch in blocks of "
                             f"{blk} rows (wall clock, transfer to the workers included); GPU: the whole batch",
        "next_rows_gbs": oracle_rows_sample(step),
    }


def run_reference(args, rank, world, local_rank):
    """Reference arm: the CPU oracle, as it stands, on bounded samples of the workload."""
    import torch

    if rank != 0:
        return None
    torch.cuda.set_device(local_rank)
    wl = WORKLOADS[args.workload]
    counts = counts_for(wl)
    step = MoEStep(counts, wl["seed"], f"cuda:{local_rank}", inputs_only=True)
    for i in range(args.warmup):
        oracle_sample(step, counts, rows_per_gemm=4, cols=64, rng_seed=i)
    total_s, total_f, desc = 0.0, 0, ""
    for i in range(args.steps):
        s, f, desc = oracle_sample(step, counts, rows_per_gemm=4, cols=64, rng_seed=1000 + i)
        total_s += s
        total_f += f
    value = total_f / total_s / 1e12
    ms = total_s / args.steps * 1e3
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 GEMM on exactly dequantized operands; fp32 quantizers",
        "data": "synthetic (same seeded workload as the CUDA arm)",
        "config": {"workload": args.workload, "experts": step.E, "hidden": step.H, "intermediate": step.I,
                   "routed_rows": step.R},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": desc,
                         "host": host_info()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------- traffic --
def lookup_traffic(call, workload):
    """ncu DRAM bytes per launch for `call`, from profiles/ncu_traffic.json, or None
    when absent or taken on a kernel source that has changed since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        table = json.load(fh)
    entry = table.get(workload, {}).get(call)
    if not entry:
        return None
    if entry.get("source_sha256") != source_digest():
        return None
    return entry.get("dram_bytes_per_launch")


def source_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_moe_expert_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip timing the calls outside the step")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local_rank = dist_env()
    if world > 1 and args.impl == "ours":
        import torch

        torch.distributed.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    line = run_reference(args, rank, world, local_rank) if args.impl == "reference" else \
        run_ours(args, rank, world, local_rank)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        import torch

        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
