#!/usr/bin/env python
"""Forward + backward of the pre-norm residual ReLU² MLP block on GB300.

One step = the whole hot path over one batch of synthetic input: forward and
backward of every microbatch with fp32 gradient accumulation, then scale_grads
where the workload has one.  The gradients start either from a zero_grads launch
at the step's start or from the first microbatch's backward setting them
(mlpblk_backward_overwrite, its FP8 form, mlpblk_moe_backward_overwrite: the
weight-gradient GEMMs store the tiles they sum whole and only their split tiles
are cleared first).  --grads auto (default) sets them in the backward for the
routed experts and for dense blocks with over 64 MB of gradients (not the
recompute variant), and zeroes them otherwise;
--grads overwrite|zero forces either form.  Prints one JSON line (rank 0).
The default run times the large block (d 4096, ffn 16384, 2 x 8192 tokens) and,
in a `secondary` object of the same line, the 120M-class block (d 768, ffn
3072, 8192 tokens).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

--impl reference times the float64 oracle on the host cores on a bounded token
sample of the same workload (the only other place this script runs the oracle
is the cpu_baseline leg).  Under torchrun each rank runs an independent replica
(the block has no cross-rank step); the time is the max over ranks.
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "fwd+bwd block TFLOP/s & tokens/s at 1 GB300; % of BF16 tensor peak / HBM BW"
DEFAULT_WORKLOAD = "large_accum2"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "source": "fallback"}
GEMM_KINDS = ("gemm_fwd_w1", "gemm_fwd_w2", "gemm_dgrad_h", "gemm_wgrad_w2", "gemm_dgrad_n",
              "gemm_wgrad_w1")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.CONFIGS) + sorted(synth.MOE_CONFIGS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-graph", action="store_true", help="time eager launches instead of a CUDA graph")
    p.add_argument("--grads", default="auto", choices=["auto", "zero", "overwrite"],
                   help="zero: zero_grads at the start of each step, every backward adds; overwrite: the first "
                        "microbatch's backward sets the gradients; auto: overwrite for the routed experts and for "
                        "dense blocks with over 64 MB of gradients, zero otherwise")
    p.add_argument("--no-secondary", action="store_true",
                   help="skip the 120M-class block that the default run also times")
    p.add_argument("--optimizer", action="store_true",
                   help="end each step with the optimizer-side kernels: global gradient norm, "
                        "clip scale, fused AdamW on float32 master weights")
    p.add_argument("--rmsnorm", default="stats", choices=["stats", "prologue"],
                   help="stats: rstd from one statistics pass ahead of the W1 GEMM (default); prologue: "
                        "rstd summed inside the W1 GEMM from its staged x tiles")
    p.add_argument("--precision", default="bf16", choices=["bf16", "fp8"],
                   help="bf16: the block's GEMMs on bf16 operands; fp8: the E4M3-operand variant "
                        "(per-tensor scales, fp32 accumulators)")
    p.add_argument("--variant", default="saving", choices=["saving", "recompute"],
                   help="saving: h and a saved by the forward; recompute: x and rstd saved, h and a "
                        "rebuilt by one more W1 GEMM in the backward")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


# ----------------------------------------------------------------- distributed

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo", rank=self.rank, world_size=self.world)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v):
        if not self.pg:
            return v
        import torch
        t = torch.tensor([float(v)], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """SM clock, power and clock-event reasons sampled DURING the timed region.

    A background thread reads NVML (the driver's libnvidia-ml, through ctypes)
    every 5 ms; `mark(True)` / `mark(False)` bracket the timed region on the
    host clock, and only the samples between the two marks are reported.  The
    GPU is found by its UUID as torch reports it, so the sampled device is the
    one the run uses whatever CUDA_VISIBLE_DEVICES maps.  Where NVML cannot be
    loaded the `nvidia-smi -lms` sampler (100 ms, all samples of the region)
    stands in.  Only readings: no clock or other setting is changed."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    # nvmlClocksEventReason* bits (nvml.h)
    REASON_BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
                   0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}
    PERIOD_S = 0.005

    def __init__(self, index, uuid=None):
        self.index = index
        self.uuid = uuid
        self.samples = []          # (host time, sm MHz, power W, reasons bitmask)
        self.window = [None, None]
        self.max_mhz = None
        self.source = None
        self._stop = None
        self._thread = None
        self._smi = None

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        rc = 1
        if self.uuid:
            rc = lib.nvmlDeviceGetHandleByUUID(("GPU-" + self.uuid).encode(), ctypes.byref(h))
        if rc != 0:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h))
        if rc != 0:
            raise OSError("no NVML handle")
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        return lib, h, reasons_fn

    def start(self):
        import ctypes
        import threading
        try:
            lib, h, reasons_fn = self._nvml()
        except (OSError, AttributeError):
            self._start_smi()
            return
        self.source = "nvml (5 ms)"
        self._stop = threading.Event()
        clk, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()

        def run():
            while not self._stop.is_set():
                t = time.perf_counter()
                if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                    p = mw.value / 1e3 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0 else 0.0
                    r = rs.value if reasons_fn(h, ctypes.byref(rs)) == 0 else 0
                    self.samples.append((t, float(clk.value), p, r))
                time.sleep(self.PERIOD_S)

        self._thread = threading.Thread(target=run, daemon=True)
        self._thread.start()
        time.sleep(0.05)

    def _start_smi(self):
        fd, path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.source = "nvidia-smi (100 ms)"
        try:
            self._smi = (subprocess.Popen(
                ["nvidia-smi", f"--id={self.uuid and 'GPU-' + self.uuid or self.index}",
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(path, "w"), stderr=subprocess.DEVNULL), path)
        except OSError:
            self._smi = None
        time.sleep(0.3)

    def mark(self, begin):
        self.window[0 if begin else 1] = time.perf_counter()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
            t0, t1 = self.window
            inside = [s for s in self.samples if t0 is not None and t1 is not None and t0 <= s[0] <= t1]
            return self._summary([s[1] for s in inside], [s[2] for s in inside],
                                 {n for s in inside for b, n in self.REASON_BITS.items() if s[3] & b},
                                 len(inside), self.max_mhz)
        if self._smi is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampler unavailable"]}
        proc, path = self._smi
        time.sleep(0.25)
        proc.terminate()
        proc.wait()
        rows = []
        with open(path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 7:
                    rows.append(parts)
        os.unlink(path)

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        return self._summary([num(r[0]) for r in rows if num(r[0]) is not None],
                             [num(r[2]) or 0.0 for r in rows],
                             {names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"},
                             len(rows), num(rows[0][1]) if rows else None)

    def _summary(self, sm, power, reasons, n, max_mhz):
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": max_mhz, "reasons": sorted(reasons) or ["no samples"],
                    "samples": 0, "source": self.source}
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": max_mhz,
                "reasons": sorted(reasons), "samples": n, "power_w_max": round(max(power), 1),
                "source": self.source, "window": "samples taken while the timed region ran"}


def device_uuid(index):
    import torch
    try:
        return str(torch.cuda.get_device_properties(index).uuid)
    except Exception:
        return None


# ---------------------------------------------------------------- our arm

# the CUDA sources that hold each kernel's device code and its launch choices
KERNEL_SOURCES = {
    **{k: ("gemm_tc.cuh", "ptx.cuh", "gemm_fwd.cu") for k in ("gemm_fwd_w1", "gemm_fwd_w2")},
    **{k: ("gemm_tc.cuh", "ptx.cuh", "gemm_bwd.cu")
       for k in ("gemm_wgrad_w2", "gemm_dgrad_h", "gemm_dgrad_n", "gemm_wgrad_w1")},
    **{k: ("rowops.cu",) for k in ("norm_bwd", "fold_gamma", "dgamma_reduce")},
}


def _code_text(src):
    """The code of a C/CUDA source without its comments and with every run of
    white space as one space: an edit to comments or layout leaves it unchanged."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def csrc_hash(kernel=None):
    """Hash of the code (comments and layout aside) of the kernel's sources
    (KERNEL_SOURCES), else of every CUDA source."""
    csrc = os.path.join(ROOT, "mlp_block_backprop_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel)
    paths = [os.path.join(csrc, n) for n in names] if names else sorted(glob.glob(os.path.join(csrc, "*")))
    h = hashlib.sha256()
    for p in paths:
        with open(p, encoding="utf-8") as f:
            h.update(_code_text(f.read()).encode("utf-8"))
    return h.hexdigest()[:12]


def recorded_traffic(workload, kernel):
    """DRAM bytes per launch from the committed ncu record, if it was taken on
    the current kernel sources (profiles/traffic.tsv: kernel, workload, bytes
    per launch, csrc_hash(kernel) at the time of the capture)."""
    path = os.path.join(ROOT, "profiles", "traffic.tsv")
    if not os.path.exists(path):
        return None
    cur = csrc_hash(kernel)
    with open(path) as f:
        for line in f:
            col = line.rstrip("\n").split("\t")
            if len(col) == 4 and col[0] == kernel and col[1] == workload and col[3] == cur:
                return float(col[2])
    return None


def algorithmic_work(kind, T, d, F, parts, prefold=False, dn_bytes=2):
    """(amount, unit) per launch: FLOP for the GEMMs, bytes for the HBM-bound kernels.
    dn_bytes: the element size of dn_s (bf16 on the bf16 path, fp32 on the FP8 path)."""
    if kind in GEMM_KINDS:
        return 2.0 * T * d * F, "flop"
    if kind == "norm_bwd":
        # x, dy (bf16) and dn_s read, dx (bf16) written, rstd and gamma read; the
        # dgamma partial rows (a few MB of scratch) are not counted
        return T * d * (2 + 2 + dn_bytes + 2) + 4.0 * T + 2.0 * d, "byte"
    if kind == "fold_gamma":
        if prefold:  # once per step: W1 read, W1*gamma written
            return 2.0 * F * d * 2 + 2.0 * d, "byte"
        # statistics pass: x read, rstd written, W1 read and W1*gamma written
        return 2.0 * T * d + 4.0 * T + 2.0 * F * d * 2 + 2.0 * d, "byte"
    if kind == "rstd":  # statistics pass alone: x read, rstd written
        return 2.0 * T * d + 4.0 * T, "byte"
    if kind == "zero_grads":
        return 4.0 * (2 * F * d + d), "byte"
    if kind == "scale_grads":
        return 8.0 * (2 * F * d + d), "byte"
    if kind == "dgamma_reduce":
        return 4.0 * parts * d + 8.0 * d, "byte"
    if kind in ("quant_amax", "quant_scale", "quant_apply"):
        return None, None  # one launch per quantised tensor, of different sizes
    if kind == "norm_quant":
        return 2.0 * T * d + 1.0 * T * d + 4.0 * T, "byte"
    if kind == "grad_norm":
        return 4.0 * (2 * F * d + d), "byte"
    if kind == "clip_grads":
        return 8.0 * (2 * F * d + d), "byte"
    if kind == "adamw":
        # master, grad, m, v read; master, m, v written (fp32); bf16 working copy written
        return 30.0 * (2 * F * d + d), "byte"
    return None, None


def run_ours(args, dist, peaks):
    import torch

    import mlp_block_backprop_gb300 as mb

    torch.cuda.set_device(dist.local_rank)
    inp = synth.config_inputs(args.workload)
    T, d, F, n_mb = inp.tokens, inp.d, inp.ffn, inp.n_mb
    dt = torch.bfloat16 if inp.dtype == "bf16" else torch.float32
    dev = "cuda"
    to = lambda a: torch.from_numpy(a).to(dev).to(dt)
    recompute = args.variant == "recompute"
    mb.mlpblk_set_rmsnorm_mode(mb.MLPBLK_RMSNORM_IN_W1_PROLOGUE if args.rmsnorm == "prologue"
                               else mb.MLPBLK_RMSNORM_STATS_PASS)
    fp8 = args.precision == "fp8"
    if fp8 and (recompute or inp.dtype != "bf16"):
        raise SystemExit("--precision fp8 needs a bf16 workload and the saving variant")
    bb = mb.BlockBuffers(T, d, F, dtype=inp.dtype, eps=inp.eps, recompute=recompute, fp8=fp8)
    bb.gamma.copy_(to(inp.gamma))
    bb.w1.copy_(to(inp.w1))
    bb.w2.copy_(to(inp.w2))
    xs = [to(x) for x in inp.x]
    dys = [to(g) for g in inp.dy]
    desc = bb.desc
    if args.optimizer:
        # float32 master weights and AdamW moments; the bf16 weights are the working copy
        masters = {k: torch.from_numpy(a.astype("float32")).to(dev) for k, a in
                   (("gamma", inp.gamma), ("w1", inp.w1), ("w2", inp.w2))}
        moments = {k: (torch.zeros_like(t), torch.zeros_like(t)) for k, t in masters.items()}
        norm_scale = torch.zeros(2, dtype=torch.float32, device=dev)
        hp = mb.AdamW(1e-4, 0.9, 0.95, 1e-8, 0.1)
        opt_params = [(masters["gamma"], bb.gamma, bb.dgamma, *moments["gamma"], False),
                      (masters["w1"], bb.w1, bb.dw1, *moments["w1"], True),
                      (masters["w2"], bb.w2, bb.dw2, *moments["w2"], True)]

    # with several microbatches, W1 * gamma is made once per step (the weights do
    # not change between microbatches) and every forward reads it
    prefold = n_mb > 1 and not fp8 and not recompute
    if prefold:
        bb.w1g = torch.empty_like(bb.w1)

    # the first microbatch's backward sets the gradients (--grads overwrite, or auto
    # where zero_grads would clear more than 64 MB: there the weight-gradient GEMMs
    # store the tiles they sum whole and only their split tiles are cleared; a small
    # block's zero_grads at the step's start costs less than a clearing launch
    # between the forward and the backward)
    grad_bytes = 4 * (2 * F * d + d)
    overwrite = (args.grads == "overwrite" or (args.grads == "auto" and grad_bytes > (64 << 20))) \
        and not recompute

    def step(x_list, dy_list, dx_list=None, after_mb=None):
        if not overwrite:
            mb.mlpblk_zero_grads(desc, bb.dgamma, bb.dw1, bb.dw2)
        if fp8:
            # the weights' E4M3 codes once per step: they do not change between microbatches
            mb.mlpblk_fp8_quantize_weights(desc, bb.gamma, bb.w1, bb.w2, bb.wq, bb.ws)
        if prefold:
            mb.mlpblk_fold_weights(desc, bb.gamma, bb.w1, bb.w1g)
        for i in range(n_mb):
            dx = bb.dx if dx_list is None else dx_list[i]
            if fp8:
                mb.mlpblk_forward_fp8_prequant(desc, x_list[i], bb.wq, bb.y, bb.h, bb.a8, bb.n8, bb.rstd, bb.scales,
                                               bb.ws)
                mb.mlpblk_backward_fp8_prequant(desc, dy_list[i], x_list[i], bb.gamma, bb.wq, bb.h, bb.a8, bb.n8,
                                                bb.rstd, bb.scales, dx, bb.dgamma, bb.dw1, bb.dw2, bb.ws,
                                                overwrite=overwrite and i == 0)
            elif recompute:
                mb.mlpblk_forward_recompute(desc, x_list[i], bb.gamma, bb.w1, bb.w2, bb.y, bb.rstd, bb.ws)
                mb.mlpblk_backward_recompute(desc, dy_list[i], x_list[i], bb.gamma, bb.w1, bb.w2, bb.rstd,
                                             dx, bb.dgamma, bb.dw1, bb.dw2, bb.ws)
            else:
                if prefold:
                    mb.mlpblk_forward_prefolded(desc, x_list[i], bb.w1g, bb.w2, bb.y, bb.h, bb.a, bb.rstd, bb.ws)
                else:
                    mb.mlpblk_forward(desc, x_list[i], bb.gamma, bb.w1, bb.w2, bb.y, bb.h, bb.a, bb.rstd, bb.ws)
                mb.mlpblk_backward(desc, dy_list[i], x_list[i], bb.gamma, bb.w1, bb.w2, bb.h, bb.a, bb.rstd,
                                   dx, bb.dgamma, bb.dw1, bb.dw2, bb.ws, overwrite=overwrite and i == 0)
            if after_mb is not None:
                after_mb(i)
        if inp.grad_scale is not None:
            mb.mlpblk_scale_grads(desc, bb.dgamma, bb.dw1, bb.dw2, inp.grad_scale)
        if args.optimizer:
            # a CUDA graph keeps the step number it was captured with; the update's
            # cost does not depend on it
            mb.mlpblk_grad_norm(desc, bb.dgamma, bb.dw1, bb.dw2, 1.0, norm_scale[0:1], norm_scale[1:2], bb.ws)
            mb.mlpblk_adamw_step(opt_params, hp, 1, bb.code, grad_scale=norm_scale[1:2])

    for _ in range(args.warmup):
        step(xs, dys)
    torch.cuda.synchronize()
    if mb.mlpblk_last_error() != mb.MLPBLK_OK:
        raise RuntimeError("device error during warm-up")

    launches_per_step = (1 + (9 if fp8 else 0) + (1 if prefold else 0) + n_mb * (16 if fp8 else 11 if recompute else 9)
                         + (1 if inp.grad_scale is not None else 0) + (3 if args.optimizer else 0))
    trace = mb.KernelTrace(args.steps * launches_per_step + 8)
    clocks = ClockSampler(dist.local_rank, device_uuid(dist.local_rank))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launch_mode = "eager"
    plain = traced = None
    if not args.no_graph:
        # the K timed steps captured as one CUDA graph, and the same K steps again
        # with an event pair around every launch for the per-kernel breakdown;
        # the library allocates nothing, so capture needs no memory pool set-up
        try:
            plain = torch.cuda.CUDAGraph()
            with torch.cuda.graph(plain):
                for _ in range(args.steps):
                    step(xs, dys)
            traced = torch.cuda.CUDAGraph()
            with torch.cuda.graph(traced):
                with trace:
                    for _ in range(args.steps):
                        step(xs, dys)
            plain.replay()  # untimed: warms the graphs themselves
            traced.replay()
            torch.cuda.synchronize()
            launch_mode = "cuda_graph"
        except Exception as exc:  # capture unsupported here: time eager launches
            plain = traced = None
            launch_mode = f"eager (graph capture failed: {type(exc).__name__})"
            trace = mb.KernelTrace(args.steps * launches_per_step + 8)
    dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    clocks.mark(True)
    start.record()
    if plain is not None:
        plain.replay()
    else:
        for _ in range(args.steps):
            step(xs, dys)
    end.record()
    torch.cuda.synchronize()
    clocks.mark(False)
    dist.barrier()
    clk = clocks.stop()
    # the per-kernel pass: same steps, every launch bracketed by CUDA events
    t_start.record()
    if traced is not None:
        traced.replay()
    else:
        with trace:
            for _ in range(args.steps):
                step(xs, dys)
    t_end.record()
    torch.cuda.synchronize()
    ms_total = dist.max(start.elapsed_time(end))
    ms_traced = t_start.elapsed_time(t_end)
    if mb.mlpblk_last_error() != mb.MLPBLK_OK:
        raise RuntimeError("device error in the timed region")
    ms_step = ms_total / args.steps
    flop_step = synth.block_flops(T, d, F, n_mb)
    value = dist.world * flop_step / (ms_step * 1e-3) / 1e12
    tokens_s = dist.world * T * n_mb / (ms_step * 1e-3)

    # per-kernel breakdown from the trace (CUDA events on the launch stream)
    per = {}
    for kind, ms in trace.durations():
        e = per.setdefault(kind, [0, 0.0])
        e[0] += 1
        e[1] += ms
    # every step ran the whole path: each of the six GEMMs once per microbatch
    missing = [k for k in GEMM_KINDS if per.get(k, [0])[0] < args.steps * n_mb]
    if missing:
        raise RuntimeError(f"the traced steps did not launch {missing} once per microbatch")
    total_k = sum(v[1] for v in per.values())
    kernels = {k: {"launches": v[0], "total_ms": round(v[1], 4), "mean_us": round(1e3 * v[1] / v[0], 2),
                   "share": round(v[1] / total_k, 4)} for k, v in sorted(per.items(), key=lambda kv: -kv[1][1])}
    import ctypes  # noqa: F401
    parts = min(max(1, (T + 15) // 16), 512, 2 * torch.cuda.get_device_properties(0).multi_processor_count)

    def roofline(kind):
        if kind not in per:
            return None
        amount, unit = algorithmic_work(kind, T, d, F, parts, prefold, dn_bytes=4 if fp8 else 2)
        if amount is None:  # a launch with no bandwidth or FLOP roof of its own (a scalar finalize)
            return None
        mean_s = per[kind][1] / per[kind][0] * 1e-3
        # the record holds captures of the bf16 kernels; the E4M3 GEMMs are other kernels
        traffic = None if fp8 else recorded_traffic(args.workload, kind)
        if unit == "flop":
            # the burst figure: the timed region is a fraction of a second, not
            # the seconds-long loop of the sustained measurement
            peak = peaks.get("bf16_tflops", peaks.get("bf16_tflops_sustained"))
            sus = peaks.get("bf16_tflops_sustained", peak)
            src = f"{peaks['source']} burst bf16"
            if fp8:  # E4M3 contractions: the bf16 measurement times the nominal 4.5 / 2.25 ratio
                peak, sus = 2.0 * peak, 2.0 * sus
                src += " x 2 (nominal fp8 / bf16 dense ratio)"
            ach = amount / mean_s / 1e12
            return {"kernel": kind, "bound": "tensor", "achieved": round(ach, 1), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(ach / peak, 4), "frac_of_sustained": round(ach / sus, 4),
                    "traffic": traffic, "algorithmic_per_launch": amount, "peak_source": src,
                    "mean_launch_us": round(mean_s * 1e6, 2)}
        peak = peaks["hbm_gbs"]
        ach = amount / mean_s / 1e9
        return {"kernel": kind, "bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "traffic": traffic, "algorithmic_per_launch": amount,
                "peak_source": f"{peaks['source']} copy bandwidth", "mean_launch_us": round(mean_s * 1e6, 2)}

    dominant = max(per, key=lambda k: per[k][1])
    pk_mul = 2.0 if fp8 else 1.0
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": inp.dtype,
        "data": "synthetic (seeded numpy normals, bf16-rounded; no dataset)",
        "config": {"workload": args.workload, "tokens_per_microbatch": T, "microbatches": n_mb,
                   "d_model": d, "ffn": F, "shape": synth.CONFIGS[args.workload]["shape"],
                   "flop_per_step": flop_step,
                   "variant": args.variant,
                   "precision": args.precision + (" (E4M3 GEMM operands, per-tensor scales; the weights' codes made once "
                                                  "per step for all microbatches)" if fp8 else ""),
                   "rmsnorm": args.rmsnorm,
                   "w1_gamma_fold": "once per step (mlpblk_fold_weights + mlpblk_forward_prefolded)" if prefold
                                    else "inside every forward",
                   "gradients": ("written by the first microbatch's backward (mlpblk_backward"
                                 + ("_fp8_prequant" if fp8 else "") + "_overwrite), added by the others"
                                 if overwrite else "zero_grads, then every backward adds"),
                   "optimizer": "grad norm + clip + AdamW (fp32 masters)" if args.optimizer else None,
                   # the recompute variant runs one more W1 GEMM per microbatch; the
                   # metric stays the algorithmic 12*T*d*F per microbatch
                   "executed_flop_per_step": flop_step * 7 // 6 if recompute else flop_step,
                   "saved_activation_bytes_per_microbatch": (
                       T * d * (2 if inp.dtype == "bf16" else 4) + 4 * T
                       + (3 * T * F + T * d + 16 if fp8 else 0 if recompute else
                          2 * T * F * (2 if inp.dtype == "bf16" else 4))),
                   "l2": "inputs larger than L2 (working set %.1f GB per replica)" % (
                       (bb.ws.numel() + sum(t.numel() * t.element_size() for t in
                        [bb.w1, bb.w2, bb.h, bb.a, bb.dw1, bb.dw2] + xs + dys if t is not None)) / 1e9),
                   "parallelism": "replicas" if dist.world > 1 else "single",
                   "launch": launch_mode},
        "tokens_per_s": round(tokens_s, 1),
        "frac_of_peak": {"sustained": round(value / dist.world / (pk_mul * peaks.get("bf16_tflops_sustained", 1.0)), 4),
                         "burst": round(value / dist.world / (pk_mul * peaks.get("bf16_tflops", 1.0)), 4),
                         "peak": "fp8 = 2 x measured bf16 (nominal ratio)" if fp8 else "measured bf16"},
        "roofline": roofline(dominant),
        "roofline_hbm": roofline("norm_bwd"),
        # every kernel kind against its own roof: tensor peak for the GEMMs, copy
        # bandwidth for the HBM-bound kernels (same live event durations)
        "roofline_per_kernel": {k: {f: r[f] for f in ("bound", "achieved", "unit", "frac", "mean_launch_us")}
                                for k in per for r in [roofline(k)] if r is not None},
        "kernels": kernels,
        "kernel_trace": {"how": "second replay of the same K steps with a CUDA event pair around "
                                "every launch (on the launch stream)",
                         "ms_per_step": round(ms_traced / args.steps, 4),
                         "overhead": round(ms_traced / ms_total - 1.0, 4)},
        "gpu_launches": trace.count,
        "clocks": clk,
    }

    if not args.no_e2e:
        k_e2e = max(3, args.steps)  # the same K steps as the device number
        hx = [torch.from_numpy(x).to(dt).pin_memory() for x in inp.x]
        hdy = [torch.from_numpy(g).to(dt).pin_memory() for g in inp.dy]
        hdx = [torch.empty(T, d, dtype=dt).pin_memory() for _ in range(n_mb)]
        sets = [([torch.empty_like(x) for x in xs], [torch.empty_like(g) for g in dys],
                 [torch.empty_like(bb.dx) for _ in range(n_mb)]) for _ in range(2)]

        def run_e2e(k):
            return pipelined_e2e(k, sets, hx, hdy, hdx, lambda st, after: step(st[0], st[1], st[2], after),
                                 lambda st, i: st[2][i])

        run_e2e(1)
        torch.cuda.synchronize()
        dist.barrier()
        ms_e2e_dev, wall = run_e2e(k_e2e)
        dist.barrier()
        ms_e2e = dist.max(max(ms_e2e_dev, wall * 1e3)) / k_e2e
        elt = 2 if inp.dtype == "bf16" else 4
        result["e2e"] = {"value": round(dist.world * flop_step / (ms_e2e * 1e-3) / 1e12, 2),
                         "unit": "TFLOP/s", "ms_per_step": round(ms_e2e, 4), "steps": k_e2e,
                         "h2d_bytes_per_step": n_mb * 2 * T * d * elt,
                         "d2h_bytes_per_step": n_mb * T * d * elt,
                         "path": "pinned host x, dy -> device; mlpblk_forward/backward; dx -> pinned host "
                                 "(copies on a second stream, double-buffered: the next step's inputs "
                                 "and this step's dx move while the GPU computes; each buffer set's step "
                                 "of public calls captured once as a CUDA graph and replayed)"}
    return result, inp


SECONDARY_WORKLOAD = "block_120m"
SECONDARY_MIN_STEPS = 100


def secondary_block(args, dist, peaks):
    """The 120M-class block (8192 tokens, d 768, ffn 3072), the other block the
    targets name, timed in the same run and the same way as the main workload
    (a CUDA graph of K steps, a traced replay for the per-kernel times).  Its
    step is ~0.2 ms, so it runs at least SECONDARY_MIN_STEPS steps to give the
    events and the clock sampler a timed region of some length."""
    import copy
    sub = copy.copy(args)
    sub.workload = SECONDARY_WORKLOAD
    sub.steps = max(args.steps, SECONDARY_MIN_STEPS)
    sub.no_e2e = True
    res, _ = run_ours(sub, dist, peaks)
    keep = ("value", "unit", "steps", "warmup", "ms_per_step", "tokens_per_s", "frac_of_peak", "roofline",
            "roofline_hbm", "roofline_per_kernel", "clocks", "gpu_launches", "kernel_trace")
    out = {"workload": SECONDARY_WORKLOAD, "config": res["config"]}
    out.update({k: res[k] for k in keep if k in res})
    return out


def pipelined_e2e(k, sets, host_in, host_in2, host_out, compute, out_of, use_graphs=True):
    """Times k steps end to end: every step's inputs go host -> device and its
    outputs device -> host inside the timed region, on two copy streams (one per
    direction), into two
    alternating device buffer sets, so step s+1's inputs and step s's outputs
    move while step s computes.  `compute(set, after_mb)` enqueues one step on the
    current stream (calling after_mb(i) once microbatch i's output is written);
    `out_of(set, i)` is that output.  With use_graphs, each set's step (the same
    public calls) is captured once as a CUDA graph and replayed, and the outputs
    leave after the step.  Returns (device ms, wall seconds)."""
    import torch
    graphs = None
    if use_graphs:
        graphs = []
        for st in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                compute(sets[st], None)
            graphs.append(g)
        torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    cs = torch.cuda.Stream()   # host -> device
    co = torch.cuda.Stream()   # device -> host (the two directions overlap)
    in_ev = [torch.cuda.Event() for _ in range(2)]
    free_ev = [torch.cuda.Event() for _ in range(2)]
    out_ev = [torch.cuda.Event() for _ in range(2)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def h2d(s):
        st = s % 2
        cs.wait_event(free_ev[st])  # step s-2 no longer reads this set's inputs
        with torch.cuda.stream(cs):
            for i in range(len(host_in)):
                sets[st][0][i].copy_(host_in[i], non_blocking=True)
                sets[st][1][i].copy_(host_in2[i], non_blocking=True)
        in_ev[st].record(cs)

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    start.record(main)
    cs.wait_event(start)
    h2d(0)
    for s in range(k):
        st = s % 2
        if s + 1 < k:
            h2d(s + 1)
        main.wait_event(in_ev[st])
        main.wait_event(out_ev[st])  # step s-2's outputs have left this set

        def after(i, st=st):
            ev = torch.cuda.Event()
            ev.record(main)
            co.wait_event(ev)
            with torch.cuda.stream(co):
                host_out[i].copy_(out_of(sets[st], i), non_blocking=True)

        if graphs is not None:
            graphs[st].replay()
            ev = torch.cuda.Event()
            ev.record(main)
            co.wait_event(ev)
            with torch.cuda.stream(co):
                for i in range(len(host_out)):
                    host_out[i].copy_(out_of(sets[st], i), non_blocking=True)
        else:
            compute(sets[st], after)
        free_ev[st].record(main)
        out_ev[st].record(co)
    main.wait_stream(cs)
    main.wait_stream(co)
    end.record(main)
    torch.cuda.synchronize()
    return start.elapsed_time(end), time.perf_counter() - t0


# --------------------------------------------------------- oracle on the host

def run_moe(args, dist, peaks):
    """The routed ReLU^2 expert block: forward + backward (writing the gradients) per step,
    timed like run_ours (CUDA graph of the K steps, then a traced replay)."""
    import torch

    import mlp_block_backprop_gb300 as mb

    torch.cuda.set_device(dist.local_rank)
    inp = synth.moe_config_inputs(args.workload)
    T, d, F, E, k = inp.tokens, inp.d, inp.ffn, inp.experts, inp.top_k
    bb = mb.MoeBuffers(T, d, F, E, k, eps=inp.eps)
    bf = torch.bfloat16
    to = lambda a, dt=bf: torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dt)
    bb.gamma.copy_(to(inp.gamma))
    bb.w1s.copy_(to(inp.w1s))
    bb.w2s.copy_(to(inp.w2s))
    bb.x.copy_(to(inp.x))
    bb.dy.copy_(to(inp.dy))
    bb.idx.copy_(to(inp.idx, torch.int32))
    bb.p.copy_(to(inp.p, torch.float32))

    overwrite = args.grads != "zero"

    def step():
        if not overwrite:
            bb.zero_grads()
        bb.forward()
        bb.backward(overwrite=overwrite)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    launches = 1 + 7 + 7   # zero_grads; forward; backward
    trace = mb.KernelTrace(args.steps * launches + 8)
    plain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(plain):
        for _ in range(args.steps):
            step()
    traced = torch.cuda.CUDAGraph()
    with torch.cuda.graph(traced):
        with trace:
            for _ in range(args.steps):
                step()
    plain.replay()
    traced.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(dist.local_rank, device_uuid(dist.local_rank))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    clocks.mark(True)
    start.record()
    plain.replay()
    end.record()
    torch.cuda.synchronize()
    clocks.mark(False)
    dist.barrier()
    clk = clocks.stop()
    traced.replay()
    torch.cuda.synchronize()
    if mb.mlpblk_last_error() != mb.MLPBLK_OK:
        raise RuntimeError("device error in the timed region")
    ms_step = dist.max(start.elapsed_time(end)) / args.steps
    flop_step = synth.moe_flops(T, d, F, k)
    value = dist.world * flop_step / (ms_step * 1e-3) / 1e12
    per = {}
    for kind, ms in trace.durations():
        e = per.setdefault(kind, [0, 0.0])
        e[0] += 1
        e[1] += ms
    total_k = sum(v[1] for v in per.values())
    kernels = {kk: {"launches": v[0], "mean_us": round(1e3 * v[1] / v[0], 2), "share": round(v[1] / total_k, 4)}
               for kk, v in sorted(per.items(), key=lambda kv: -kv[1][1])}
    peak = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
    gemm = {kk: round(2.0 * T * k * d * F / (per[kk][1] / per[kk][0] * 1e-3) / 1e12 / peak, 4)
            for kk in per if kk.startswith("gemm_")}
    # host x, dy, routing in; dx, d_routing_weights out; public calls (copies on a
    # second stream into two alternating buffer sets, as for the dense block)
    hx, hdy = torch.from_numpy(inp.x).to(bf).pin_memory(), torch.from_numpy(inp.dy).to(bf).pin_memory()
    hidx = torch.from_numpy(np.ascontiguousarray(inp.idx, dtype=np.int32)).pin_memory()
    hp = torch.from_numpy(np.ascontiguousarray(inp.p, dtype=np.float32)).pin_memory()
    hdx = torch.empty(T, d, dtype=bf).pin_memory()
    hdp = torch.empty(T, k, dtype=torch.float32).pin_memory()
    k_e2e = max(3, args.steps)  # the same K steps as the device number
    sets = [([torch.empty_like(bb.x), torch.empty_like(bb.idx)], [torch.empty_like(bb.dy), torch.empty_like(bb.p)],
             [torch.empty_like(bb.dx), torch.empty_like(bb.dp)]) for _ in range(2)]

    def moe_compute(st, after):
        bb.x, bb.idx = st[0]
        bb.dy, bb.p = st[1]
        bb.dx, bb.dp = st[2]
        step()
        if after is not None:
            after(0)
            after(1)

    pipelined_e2e(1, sets, [hx, hidx], [hdy, hp], [hdx, hdp], moe_compute, lambda st, i: st[2][i])
    ms_dev, wall = pipelined_e2e(k_e2e, sets, [hx, hidx], [hdy, hp], [hdx, hdp], moe_compute,
                                 lambda st, i: st[2][i])
    ms_e2e = max(ms_dev, wall * 1e3) / k_e2e
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded numpy normals, bf16-rounded; uniform random top-k routing; no dataset)",
        "config": {"workload": args.workload, "tokens": T, "d_model": d, "ffn_per_expert": F, "experts": E,
                   "top_k": k, "flop_per_step": flop_step, "launch": "cuda_graph",
                   "gradients": ("written by the backward (mlpblk_moe_backward_overwrite)" if overwrite
                                 else "zero_grads, then the backward adds"),
                   "parallelism": "replicas" if dist.world > 1 else "single"},
        "tokens_per_s": round(dist.world * T / (ms_step * 1e-3), 1),
        "frac_of_peak": {"sustained": round(value / dist.world / peak, 4)},
        "gemm_frac_of_sustained_peak": gemm,
        "kernels": kernels,
        "gpu_launches": trace.count,
        "e2e": {"value": round(dist.world * flop_step / (ms_e2e * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": 2 * T * d * 2 + T * k * 8, "d2h_bytes_per_step": T * d * 2 + T * k * 4},
        "clocks": clk,
    }
    return result, None


def oracle_sample(inp, tokens, steps=1):
    """Times the float64 oracle on the first `tokens` tokens of every microbatch
    (all weights, all gradient buffers).  Returns seconds per step."""
    import oracle
    t0 = time.perf_counter()
    for _ in range(steps):
        grads = oracle.new_grads(inp.d, inp.ffn)
        for x, dy in zip(inp.x, inp.dy):
            xs, dys = x[:tokens], dy[:tokens]
            y, h, a, r = oracle.forward(xs, inp.gamma, inp.w1, inp.w2, inp.eps)
            oracle.backward(dys, xs, inp.gamma, inp.w1, inp.w2, h, r, grads)
        if inp.grad_scale is not None:
            oracle.scale_grads(grads, inp.grad_scale)
    return (time.perf_counter() - t0) / steps


def host_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def calibrate_tokens(inp, target_s, lo=8):
    n = min(lo, inp.tokens)
    t = oracle_sample(inp, n)
    while t < target_s / 4 and n < inp.tokens:
        n = min(inp.tokens, n * 4)
        t = oracle_sample(inp, n)
    # cost ~ fixed + per-token; extrapolate linearly from the last measurement
    want = int(n * target_s / max(t, 1e-6))
    return max(lo, min(inp.tokens, want))


def cpu_baseline(inp, target_s=15.0):
    tok = calibrate_tokens(inp, target_s)
    sec = oracle_sample(inp, tok)
    flop = synth.block_flops(tok, inp.d, inp.ffn, inp.n_mb)
    return {"value": round(flop / sec / 1e12, 6), "unit": "TFLOP/s", "cores": host_threads(),
            "kind": "oracle", "seconds": round(sec, 3),
            "sample": f"first {tok} tokens of each of the {inp.n_mb} microbatch(es), all weights "
                      f"(float64 numpy, block FLOP of the sample / wall time)",
            "tokens_per_s": round(tok * inp.n_mb / sec, 2)}


def run_reference(args, dist):
    inp = synth.config_inputs(args.workload)
    budget = 120.0
    per_step = budget / max(1, args.steps + args.warmup)
    tok = calibrate_tokens(inp, per_step)
    for _ in range(args.warmup):
        oracle_sample(inp, tok)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample(inp, tok)
    sec = (time.perf_counter() - t0) / args.steps
    flop = synth.block_flops(tok, inp.d, inp.ffn, inp.n_mb)
    value = flop / sec / 1e12
    sample = (f"first {tok} tokens of each of the {inp.n_mb} microbatch(es) per step, all weights "
              f"(float64 numpy oracle on the host)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy normals)",
            "config": {"workload": args.workload, "tokens_per_microbatch_sampled": tok,
                       "microbatches": inp.n_mb, "d_model": inp.d, "ffn": inp.ffn},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": host_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    args = parse_args()
    if args.impl == "reference":
        # host-only arm: rank 0 runs it, the other ranks have nothing to do
        if int(os.environ.get("RANK", "0")) == 0:
            class _Solo:
                world = int(os.environ.get("WORLD_SIZE", "1"))
            print(json.dumps(run_reference(args, _Solo())), flush=True)
        return
    dist = Dist()
    peaks = load_peaks()
    if args.workload in synth.MOE_CONFIGS:
        result, inp = run_moe(args, dist, peaks)
    else:
        result, inp = run_ours(args, dist, peaks)
        if args.workload == DEFAULT_WORKLOAD and not args.no_secondary:
            result["secondary"] = secondary_block(args, dist, peaks)
    if dist.rank == 0:
        if dist.world == 1 and not args.no_cpu_baseline and inp is not None:
            result["cpu_baseline"] = cpu_baseline(inp)
        print(json.dumps(result), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
