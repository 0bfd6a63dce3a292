#!/usr/bin/env python
"""Benchmark of the LUT-multiplier contractions on one GB300 (or N replicas).

Default workload: the square GEMM C = A B with A, B 4096 x 4096 ~ U[-1, 1],
every product through the Mitchell M=7 LUT (68,719,476,736 approximate MACs
per step), the largest single-GPU configuration of the path.  Other workloads
(--workload: the MLP step, convolutions, attention, depthwise layers, the
elementwise product; --mantissa for the M sweep) print the same line.

Prints one JSON line (rank 0).  Timing: W warm-up steps, then K steps, each
bracketed by CUDA events on the launching stream; before each timed step the
L2 is flushed (256 MiB write) and the GPU is held by a short sleep kernel so
that all launches of the step are queued before it starts (neither is inside
the events).  ``--impl reference`` times the CPU oracle instead (rank 0 only).
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "approx-GMAC/s for LUT-multiplier GEMM/conv at M=7"
UNIT = "approx-GMAC/s"
LOOKUPS_PER_CLK_PER_SM = 32     # one 4-byte shared-memory wavefront per clock per SM
# Closed-form products per clock per SM (no table): Mitchell's costs an integer
# add, half a paired fp32 multiply and half a paired fp32 add -- two issue
# slots of the SM's four warp instructions per clock -> 64; the exact one half
# a paired FMA on the 128 fp32 lanes -> 128.
CLOSED_FORM_PER_CLK_PER_SM = {"mitchell": 64, "exact": 128}

WORKLOADS = ("mlp", "mlp_layers", "conv3x3", "conv3x3_exact", "gemm4096", "attention", "conv1x1", "dwconv3x3",
             "dwconv3x3_s2", "dwconv5x5", "gemm64", "mul")


def measured_peaks():
    """Measured peaks of this machine's GPUs, else the recipe's fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback"


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


# ---------------------------------------------------------------- workloads
def workload_name(name, M=7, kind="mitchell"):
    """The descriptive name both arms print as config.workload."""
    names = {
        "mlp": "mlp_784-1000-500-10_b256_fwd+dX+dW_mitchell_M7",
        "mlp_layers": "mlp_784-1000-500-10_b256_autograd_AMDense_layers_mitchell_M7",
        "conv3x3": "conv3x3_nhwc_128x32x32x64_k64_fwd+bwd_data+bwd_filter_mitchell_M7",
        "conv3x3_exact": "conv3x3_nhwc_128x32x32x64_k64_fwd+bwd_data+bwd_filter_exact_M7",
        "gemm4096": f"gemm_4096^3_{kind}_M{M}",
        "attention": "attention_32x16x512x64_mitchell_M7",
        "conv1x1": "conv1x1_nhwc_64x56x56x256_k256_fwd_mitchell_M7",
        "dwconv3x3": "dwconv3x3_nhwc_64x56x56x128_d1_fwd+bwd_data+bwd_filter_mitchell_M7",
        "dwconv3x3_s2": "dwconv3x3_stride2_nhwc_64x112x112x64_d1_fwd+bwd_data+bwd_filter_mitchell_M7",
        "dwconv5x5": "dwconv5x5_nhwc_64x28x28x240_d1_fwd+bwd_data+bwd_filter_mitchell_M7",
        "mul": "elementwise_2^28_pairs_special_mix_mitchell_M7",
        "gemm64": "gemm_64x128x64_mitchell_M7",
    }
    if name not in names:
        raise SystemExit(f"unknown workload {name}")
    return names[name]


def make_step(name, lut_for, M=7, kind="mitchell"):
    from approximate_multiplier_dnn_gb300 import steps
    from approximate_multiplier_dnn_gb300 import workloads as wl
    wname = workload_name(name, M, kind)
    if name == "mlp":
        return steps.MLPStep(wl.mlp(), lut_for("mitchell", 7)), wname
    if name == "mlp_layers":
        return steps.LayersMLPStep(wl.mlp(), lut_for("mitchell", 7)), wname
    if name == "conv3x3":
        return steps.ConvStep(wl.conv3x3(), wl.CONV3X3, lut_for("mitchell", 7)), wname
    if name == "conv3x3_exact":
        return steps.ConvStep(wl.conv3x3(), wl.CONV3X3, lut_for("exact", 7)), wname
    if name == "gemm4096":
        # the mantissa-width sweep runs this workload at M = 4 .. 11
        return steps.SquareGemmStep(wl.square_gemm(4096), lut_for(kind, M)), wname
    if name == "attention":
        return steps.AttentionStep(wl.attention(), lut_for("mitchell", 7)), wname
    if name == "conv1x1":
        return steps.ConvStep(wl.conv1x1(), wl.CONV1X1, lut_for("mitchell", 7), passes=(0,)), wname
    if name == "dwconv3x3":
        return steps.DwConvStep(wl.dwconv3x3(), wl.DWCONV3X3, lut_for("mitchell", 7)), wname
    if name == "dwconv3x3_s2":
        return steps.DwConvStep(wl.dwconv3x3_s2(), wl.DWCONV3X3_S2, lut_for("mitchell", 7)), wname
    if name == "dwconv5x5":
        return steps.DwConvStep(wl.dwconv5x5(), wl.DWCONV5X5, lut_for("mitchell", 7)), wname
    if name == "mul":
        return steps.MulStep(wl.elementwise_pairs(1 << 28, seed=5), lut_for("mitchell", 7)), wname
    if name == "gemm64":
        return steps.SquareGemmStep(wl.gemm_small(), lut_for("mitchell", 7)), wname
    raise SystemExit(f"unknown workload {name}")


def oracle_parts(name, kind="mitchell", M=7):
    """(oracle callable over a row subset, rows, MACs per row) for the reference
    leg: the same contractions the GPU step runs, one row range at a time
    (kind and M apply to the gemm4096 sweep)."""
    import numpy as np
    import oracle
    from approximate_multiplier_dnn_gb300 import workloads as wl
    out = []
    if name == "mlp":
        d = wl.mlp()
        # layers 2 and 3 take synthetic activations of the right shape here
        # (the oracle's cost does not depend on the values)
        xs = [d["X"], wl.normal((256, 1000), 1.0, 90), wl.normal((256, 500), 1.0, 91)]
        for l in range(3):
            W, dY = d[f"W{l + 1}"], d[f"dY{l + 1}"]
            X = xs[l]
            out.append((lambda rows, X=X, W=W: oracle.gemm("mitchell", 7, X, W, rows=rows), X.shape[0],
                        W.shape[0] * W.shape[1]))
            out.append((lambda rows, dY=dY, W=W: oracle.gemm("mitchell", 7, dY, W, transB=True, rows=rows),
                        dY.shape[0], W.shape[0] * W.shape[1]))
            out.append((lambda rows, X=X, dY=dY: oracle.gemm("mitchell", 7, X, dY, transA=True, rows=rows),
                        X.shape[1], dY.shape[0] * dY.shape[1]))
        return out
    if name == "gemm4096":
        d = wl.square_gemm(4096)
        return [(lambda rows: oracle.gemm(kind, M, d["A"], d["B"], rows=rows), 4096, 4096 * 4096)]
    if name in ("dwconv3x3", "dwconv3x3_s2", "dwconv5x5"):
        # a "row" is a block of 64 consecutive outputs (forward, data gradient)
        # or one filter-gradient element (a sum over every N*P*Q pixel)
        d, g = {"dwconv3x3": (wl.dwconv3x3, wl.DWCONV3X3), "dwconv3x3_s2": (wl.dwconv3x3_s2, wl.DWCONV3X3_S2),
                "dwconv5x5": (wl.dwconv5x5, wl.DWCONV5X5)}[name]
        d = d()
        desc = oracle.conv_desc(g["N"], g["H"], g["W"], g["C"], g["C"] * g["D"], g["R"], g["S"], g["stride"],
                                g["pad"], g["dil"])
        P, Q = oracle.conv_out_hw(desc)
        ny = g["N"] * P * Q * g["C"] * g["D"]
        nx = g["N"] * g["H"] * g["W"] * g["C"]
        taps = g["R"] * g["S"]

        def blocks(rows):
            return (rows.astype(np.int64)[:, None] * 64 + np.arange(64)).reshape(-1)

        out.append((lambda rows: oracle.dwconv2d_fwd("mitchell", 7, desc, d["x"], d["w"], blocks(rows)),
                    ny // 64, 64 * taps))
        # the pass's useful MACs (those the GPU step counts) spread over its dx blocks
        out.append((lambda rows: oracle.dwconv2d_bwd_data("mitchell", 7, desc, d["dy"], d["w"], blocks(rows)),
                    nx // 64, int(round(64 * taps * ny / nx))))
        out.append((lambda rows: oracle.dwconv2d_bwd_filter("mitchell", 7, desc, d["x"], d["dy"],
                                                            rows.astype(np.int64)),
                    taps * g["C"] * g["D"], g["N"] * P * Q))
        return out
    raise SystemExit(f"no oracle sampler for workload {name}")


def run_oracle_sample(parts, target_s, nthreads, start=0):
    """Run row chunks of each contraction round-robin until target_s has
    elapsed; returns (MACs done, seconds)."""
    import numpy as np
    t0 = time.perf_counter()
    macs = 0
    i = start
    while True:
        for fn, nrows, per_row in parts:
            r = np.arange(i * nthreads, (i + 1) * nthreads) % nrows
            fn(r.astype(np.int32))
            macs += per_row * r.size
        i += 1
        if time.perf_counter() - t0 >= target_s:
            break
    return macs, time.perf_counter() - t0


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 50 ms; stop() keeps those stamped inside the
    window passed to it (the timed region) when there are any."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu_id)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    @staticmethod
    def _stamp(text):
        from datetime import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.strptime(text.strip(), fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self, window=None):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        rows = [[x.strip() for x in ln.split(",")] for ln in self.lines]
        rows = [f for f in rows if len(f) >= 10]
        scope = "whole sampling period"
        if window:
            inside = [f for f in rows if (t := self._stamp(f[9])) is not None and window[0] <= t <= window[1]]
            if inside:
                rows, scope = inside, "timed region"
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for f in rows:
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "scope": scope}


def gpu_id_for_smi(torch):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    try:
        uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        if uuid:
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    if vis:
        return vis.split(",")[torch.cuda.current_device()]
    return torch.cuda.current_device()


def lut_residency(lut):
    """Where the LUT-GEMM keeps the table: shared memory up to 160 KB of
    narrowed entries, else global memory read through L2 (then the lookup
    roofline above is an upper bound, not the bound)."""
    info = lut.info()
    nbytes = (1 << (2 * info["M"])) * info["width_bits"] // 8
    return "shared" if nbytes <= 160 * 1024 else "global (L2 gather)"


# ---------------------------------------------------------------- tables in global memory
# A table too large for shared memory (M >= 9) is read through L1TEX and L2.
# The unit that binds is the L1TEX data pipe, one wavefront per clock per SM
# (ncu: l1tex__data_pipe_lsu_wavefronts.sum.peak_sustained is 1 per SM; the
# 4096^3 GEMM at M = 9 keeps it 98 % busy, while the tag stage's 16 sectors
# per clock per SM run at 28 %; profiles/lutgemm_global_table_l2.md).  A
# warp-lookup gathers 32 random columns of one table row, and a gather that
# hits L1 is served like a shared-memory access: one wavefront per distinct
# 4-byte word in the busiest of the 32 banks (bank_degree).  Misses cost more
# (ncu: 4.27 wavefronts per lookup at M = 9 with 82 % of sectors hitting, 10.5
# at M = 11 with 33 %), so the fraction below 1 is the miss cost.  The
# operands' two-plane loads add their wavefronts (1/TN + 2/TM = 0.25 per lookup
# on 128 x 256 tiles).  Misses go to L2, whose sector rate ncu reports as 564
# per L2 clock at 2.016 GHz (lts__t_sectors.sum.peak_sustained).
L1TEX_WAVEFRONTS_PER_CLK_PER_SM = 1
GL_OPERAND_WAVEFRONTS_PER_LOOKUP = 0.25
L2_SECTORS_PER_CLK = 564
L2_CLK_HZ = 2.016e9


def distinct_sectors_per_warp_lookup(M, width_bits):
    R = max(1.0, (1 << M) * width_bits / 8 / 32)
    return R * (1.0 - (1.0 - 1.0 / R) ** 32)


def bank_degree(M, width_bits, trials=20000):
    """Expected wavefronts of one warp's gather: the most distinct 4-byte words
    that any of the 32 banks holds among 32 uniformly random columns of a row
    of 2^M entries of width_bits (rows start on 128-byte boundaries).  Monte
    Carlo with a fixed seed."""
    import numpy as np
    rng = np.random.default_rng(12345)
    words = np.sort(rng.integers(0, 1 << M, size=(trials, 32)) * (width_bits // 8) // 4, axis=1)
    first = np.ones_like(words, dtype=bool)
    first[:, 1:] = words[:, 1:] != words[:, :-1]
    t = np.repeat(np.arange(trials), 32).reshape(trials, 32)
    per_bank = np.bincount((t * 32 + words % 32)[first], minlength=trials * 32).reshape(trials, 32)
    return float(per_bank.max(axis=1).mean())


def global_table_roofline(lut, lut_macs, lut_ms, sms, mhz, smem_roofline):
    """Roofline of a LUT-GEMM whose table is read from global memory: its
    gathers' and operand loads' L1TEX data-pipe wavefronts (the bound it runs
    closest to), with the L2 sector rate beside it."""
    info = lut.info()
    deg = bank_degree(info["M"], info["width_bits"])
    wpl = deg + GL_OPERAND_WAVEFRONTS_PER_LOOKUP
    lookups_s = lut_macs / 32.0 / (lut_ms * 1e-3)
    peak = sms * L1TEX_WAVEFRONTS_PER_CLK_PER_SM * mhz * 1e6
    spw = distinct_sectors_per_warp_lookup(info["M"], info["width_bits"])
    sectors_s = lookups_s * spw
    l2_peak = L2_SECTORS_PER_CLK * L2_CLK_HZ
    return {"bound": "l1tex", "pipe": "L1TEX data pipe, 1 wavefront per clock per SM: a warp-lookup's gather costs "
                                      "its bank degree, plus the operand loads",
            "achieved": lookups_s * wpl / 1e9, "peak": peak / 1e9, "unit": "Gwavefront/s",
            "frac": lookups_s * wpl / peak, "traffic": None,
            "wavefronts_per_warp_lookup": {"gather_bank_degree": round(deg, 3),
                                           "operands": GL_OPERAND_WAVEFRONTS_PER_LOOKUP},
            "l2": {"achieved": sectors_s * 32 / 1e9, "peak": l2_peak * 32 / 1e9, "unit": "GB/s",
                   "frac_if_every_sector_missed_l1": sectors_s / l2_peak,
                   "sectors_per_warp_lookup": spw,
                   "note": "ncu measures the sectors that reach L2 per launch (profiles/lutgemm_global_table_l2.md)"},
            "lookup_roofline_frac": smem_roofline["frac"], "lut_residency": "global (L1TEX/L2 gathers)",
            "kernel": smem_roofline["kernel"], "sms": sms, "sm_mhz": mhz}


def path_names(am, bits):
    """amsim_last_path bits of a part's last library call, as names."""
    names = [n[len("AMSIM_PATH_"):].lower() for n in dir(am) if n.startswith("AMSIM_PATH_")]
    return sorted(n for n in names if bits & getattr(am, "AMSIM_PATH_" + n.upper()))


# ---------------------------------------------------------------- traffic record
# sources of the LUT-GEMM kernels (the kernel the traffic records measure);
# a record holds for one version of them
KERNEL_SOURCES = ("gemm_kernel.cuh", "gemm_ws.cuh", "gemm_tma.cuh", "gemm_raw.cuh")
DW_KERNEL_SOURCES = ("gemm_kernel.cuh", "dwconv_kernel.cuh")   # the tiled kernel's own sources
DW_S2_KERNEL_SOURCES = ("gemm_kernel.cuh", "dwconv_kernel.cuh", "dwconv_s2.cu")


def kernel_sha(sources=KERNEL_SOURCES):
    csrc = os.path.join(ROOT, "approximate_multiplier_dnn_gb300", "csrc")
    h = hashlib.sha1()
    for f in sources:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:12]


def recorded_traffic(workload, sources=KERNEL_SOURCES):
    """Per-launch DRAM bytes of the dominant kernel from a committed ncu
    summary, if it was taken on the current kernel source; else None."""
    try:
        sha = kernel_sha(sources)
        with open(os.path.join(ROOT, "profiles", "traffic.txt")) as f:
            for line in f:
                kv = dict(x.split("=", 1) for x in line.split() if "=" in x)
                if kv.get("workload") == workload and kv.get("kernel_sha1") == sha:
                    return float(kv["bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


# ---------------------------------------------------------------- replicas
def slowest_rank_ms(total_ms, world, device):
    """The job's timed total: the largest of the ranks' totals (every rank runs
    one replica of the workload on its own GPU; the slowest sets the time)."""
    if world <= 1:
        return total_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(macs_per_step, steps, total_ms, world):
    """Whole-job approx-GMAC/s: the MACs every rank processed over the job time."""
    return world * macs_per_step * steps / (total_ms * 1e-3) / 1e9


# ---------------------------------------------------------------- reference arm
def reference_arm(args, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    parts = oracle_parts(args.workload, args.kind, args.mantissa)
    cores = os.cpu_count() or 1
    # warm-up then K bounded steps: each step one row chunk per contraction
    for w in range(args.warmup):
        run_oracle_sample(parts, 0.0, cores, start=w)
    macs = 0
    secs = 0.0
    for s in range(args.steps):
        m, t = run_oracle_sample(parts, 0.0, cores, start=args.warmup + s)
        macs += m
        secs += t
    value = macs / secs / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64-accumulate",
        "data": "synthetic",
        "config": {"workload": workload_name(args.workload, args.mantissa, args.kind),
                   "sample": f"{cores} rows of each contraction per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{cores} output rows of each contraction per step, {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gemm4096", choices=WORKLOADS)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mantissa", type=int, default=7, help="LUT mantissa bits M (gemm4096 only: the M sweep)")
    ap.add_argument("--kind", default="mitchell", choices=["mitchell", "exact"], help="multiplier (gemm4096 only)")
    ap.add_argument("--closed-form", action="store_true",
                    help="compute the built-in multipliers' products in registers instead of reading the LUT")
    args = ap.parse_args()
    if (args.mantissa != 7 or args.kind != "mitchell") and args.workload != "gemm4096":
        ap.error("--mantissa and --kind apply to --workload gemm4096 only")
    if args.closed_form and args.workload == "mul":
        ap.error("--closed-form applies to the contractions")
    if not 1 <= args.mantissa <= 11:
        ap.error("--mantissa must be in 1..11")
    args.warmup = max(args.warmup, 3)

    rank, world = env_int("RANK", 0), env_int("WORLD_SIZE", 1)
    local = env_int("LOCAL_RANK", 0)

    if args.impl == "reference":
        reference_arm(args, rank)
        return

    import torch
    import torch.distributed as dist
    import approximate_multiplier_dnn_gb300 as am

    am.build()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    luts = {}

    def lut_for(kind, M):
        if (kind, M) not in luts:
            luts[(kind, M)] = am.Lut.build(kind, M).set_closed_form(args.closed_form)
        return luts[(kind, M)]

    step, wname = make_step(args.workload, lut_for, args.mantissa, args.kind)
    if args.closed_form:
        wname += "_closed_form"
    stream = torch.cuda.current_stream()
    parts = step.parts()
    props = torch.cuda.get_device_properties(local)
    sms = props.multi_processor_count

    # warm-up (also sets kernel attributes) and enqueue-time estimate
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    part_paths = {}
    for _ in range(5):
        for p in parts:
            p[1]()
            # (amsim_last_path reports GEMM and convolution calls; parts with
            # no approximate MACs, the softmax, keep no path of their own)
            part_paths[p[0]] = path_names(am, am.amsim_last_path()) if p[2] else []
    enqueue_s = (time.perf_counter() - t0) / 5
    torch.cuda.synchronize()
    sleep_cycles = int(min(max(2.0 * enqueue_s, 50e-6), 20e-3) * 2.1e9)

    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    K = args.steps

    def timed_loop(nsteps, per_part):
        """nsteps steps, L2 flushed and the queue pre-filled before each; events
        around the step (and around every call when per_part)."""
        nev = len(parts) + 1 if per_part else 2
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(nsteps)]
        torch.cuda.synchronize()
        for s in range(nsteps):
            flush.fill_(float(s))
            torch.cuda._sleep(sleep_cycles)
            evs[s][0].record(stream)
            for i, p in enumerate(parts):
                p[1]()
                if per_part:
                    evs[s][i + 1].record(stream)
            if not per_part:
                evs[s][1].record(stream)
        torch.cuda.synchronize()
        return evs

    sampler = ClockSampler(gpu_id_for_smi(torch))
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    epoch0 = time.time()
    launches0 = am.amsim_kernel_launches()
    evs = timed_loop(K, per_part=False)
    launches_timed = am.amsim_kernel_launches() - launches0
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    time.sleep(0.1)
    clocks = sampler.stop(window=(epoch0, epoch0 + wall))
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]

    # per-call times (events between calls stop launches from overlapping, so
    # these come from a separate, shorter pass)
    P = max(3, min(K, 50))
    pevs = timed_loop(P, per_part=True)
    part_ms = [sum(pevs[s][i].elapsed_time(pevs[s][i + 1]) for s in range(P)) / P for i in range(len(parts))]
    total_ms = slowest_rank_ms(sum(step_ms), world, "cuda")
    macs = step.macs
    value = job_throughput(macs, K, total_ms, world)
    ms_per_step = total_ms / K

    # dominant kernel: the LUT-GEMM (every part with MACs), lookups = MACs
    # its time per step = the timed step time x its share of the per-call pass
    lut_parts = [i for i, p in enumerate(parts) if p[2] > 0]
    lut_share = sum(part_ms[i] for i in lut_parts) / max(1e-12, sum(part_ms))
    lut_ms = ms_per_step * lut_share
    lut_macs = sum(parts[i][2] for i in lut_parts)
    launches_lut = sum(1 for _ in lut_parts)
    achieved = lut_macs / (lut_ms * 1e-3) / 1e9 if lut_ms > 0 else 0.0   # Glookup/s
    mhz = clocks["sm_mhz"] or props.clock_rate / 1e3
    peak = sms * LOOKUPS_PER_CLK_PER_SM * mhz * 1e6 / 1e9   # Glookup/s
    traffic = recorded_traffic(wname)
    roofline = {"bound": "alu", "pipe": "shared-memory LUT lookups: SMs x 32 per clock x SM clock",
                "achieved": achieved, "peak": peak, "unit": "Glookup/s", "frac": achieved / peak,
                "traffic": traffic,
                "kernel": "LUT-GEMM calls: lutgemm_raw_kernel, or predecode + lutgemm_tma_kernel "
                          "(lutgemm_ws_kernel for gathers); see paths",
                "calls_per_step": launches_lut, "kernel_launches_per_step": launches_timed / K,
                "lut_residency": lut_residency(step.lut),
                "lut_share_of_step": round(lut_share, 4), "sms": sms,
                "sm_mhz": mhz}
    if lut_residency(step.lut) != "shared" and not args.closed_form:
        roofline = global_table_roofline(step.lut, lut_macs, lut_ms, sms, mhz, roofline)
    if args.closed_form:
        kinds = sorted({k for k, _ in luts})
        per_clk = min(CLOSED_FORM_PER_CLK_PER_SM[k] for k in kinds)
        cpeak = sms * per_clk * mhz * 1e6 / 1e9
        roofline = dict(roofline, pipe=f"closed-form {'/'.join(kinds)} products: SMs x {per_clk} per clock x "
                        "SM clock (issue slots / fp32 lanes)", peak=cpeak, unit="Gproduct/s",
                        frac=achieved / cpeak, lookup_roofline_frac=achieved / peak,
                        kernel="lutgemm_raw_kernel<1|2> (closed forms, no table); see amsim_last_path")
        roofline.pop("lut_residency", None)
    if args.workload in ("dwconv3x3", "dwconv3x3_s2", "dwconv5x5"):
        # a stencil: each pass reads its operands once and writes its output
        # once, with 9 products per output element.  Every pass's two lower
        # bounds (compulsory DRAM bytes at the measured copy bandwidth, lookups
        # at the shared-memory pipe's rate) are reported; the roofline is that
        # of the pass that takes longest, against the larger of its bounds.
        hbm, src = measured_peaks()
        per = {}
        for i, p in enumerate(parts):
            t_ms = ms_per_step * part_ms[i] / max(1e-12, sum(part_ms))
            nbytes = step.pass_bytes(step.passes[i])
            per[p[0]] = {"ms": t_ms, "bytes": nbytes, "macs": p[2],
                         "hbm_gbs": nbytes / (t_ms * 1e-3) / 1e9, "hbm_frac": nbytes / (t_ms * 1e-3) / 1e9 / hbm,
                         "glookups": p[2] / (t_ms * 1e-3) / 1e9,
                         "lookup_frac": p[2] / (t_ms * 1e-3) / 1e9 / peak,
                         "bound": "hbm" if nbytes / (hbm * 1e9) >= p[2] / (peak * 1e9) else "alu"}
        dom = max(per, key=lambda k: per[k]["ms"])
        d = per[dom]
        kern = step.kernel_name(step.passes[list(per).index(dom)])
        if d["bound"] == "hbm":
            roofline = {"bound": "hbm", "achieved": d["hbm_gbs"], "peak": hbm, "peak_source": src, "unit": "GB/s",
                        "frac": d["hbm_frac"], "lookup_frac": d["lookup_frac"]}
        else:
            roofline = {"bound": "alu", "pipe": "shared-memory LUT lookups: SMs x 32 per clock x SM clock",
                        "achieved": d["glookups"], "peak": peak, "unit": "Glookup/s", "frac": d["lookup_frac"],
                        "hbm_frac": d["hbm_frac"]}
        srcs = DW_S2_KERNEL_SOURCES if args.workload == "dwconv3x3_s2" else DW_KERNEL_SOURCES
        roofline.update({"traffic": recorded_traffic(f"{wname}:{dom}", srcs),
                         "kernel": f"{kern} ({dom} pass)", "passes": per, "sms": sms, "sm_mhz": mhz})
        if args.closed_form:
            roofline["products"] = "closed form in registers (no table lookups): lookup_frac is lookups avoided"
    if args.workload == "mul":
        # HBM-bound: 12 bytes per product (two operands in, one result out)
        hbm, src = measured_peaks()
        gbs = 12.0 * macs / (ms_per_step * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": gbs, "peak": hbm, "peak_source": src, "unit": "GB/s",
                    "frac": gbs / hbm, "traffic": traffic, "kernel": "amsim_mul_kernel"}

    # native fp32 on the same shapes (TF32 off), timed the same way: the pages
    # put the simulated GEMM beside the native one (ApproxTrain Sec. V-C)
    native = None
    if hasattr(step, "native"):
        torch.backends.cuda.matmul.allow_tf32 = False
        torch.backends.cudnn.allow_tf32 = False
        nf = step.native()
        for _ in range(3):
            nf()
        NN = max(3, min(50, K))
        nev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(NN)]
        torch.cuda.synchronize()
        for s in range(NN):
            flush.fill_(float(s))
            torch.cuda._sleep(sleep_cycles)
            nev[s][0].record(stream)
            nf()
            nev[s][1].record(stream)
        torch.cuda.synchronize()
        native_ms = sum(a.elapsed_time(b) for a, b in nev) / NN
        native = {"impl": "torch fp32 (cuBLAS / cuDNN), TF32 off, same shapes, L2 flushed before each step",
                  "ms_per_step": native_ms, "value": macs / (native_ms * 1e-3) / 1e9, "unit": "GMAC/s",
                  "approx_time_over_native": ms_per_step / native_ms}

    # end to end through the library's calls with host buffers: every step's
    # inputs go from pinned host memory to the device and its outputs come back,
    # inside the timed region.  E steps run back to back as a stream of batches:
    # two step instances alternate, step s's inputs go up on one copy stream
    # while step s-1 computes and step s-1's outputs come down on another, so
    # the throughput is that of the slowest of the three.  A serial pass (copy
    # in, compute, copy out, one step at a time) is reported beside it.
    def step_inputs(st):
        if hasattr(st, "inputs"):
            return st.inputs
        if hasattr(st, "x"):
            return {k: getattr(st, k) for k in ("x", "w", "dy") if getattr(st, k, None) is not None}
        if hasattr(st, "a"):
            return {"a": st.a, "b": st.b}
        if hasattr(st, "Q"):
            return {"Q": st.Q, "K": st.K, "V": st.V}
        return {"A": st.A, "B": st.B}

    pair = [step, make_step(args.workload, lut_for, args.mantissa, args.kind)[0]]
    for _ in range(args.warmup):
        pair[1].run()
    ins = [step_inputs(st) for st in pair]
    outs = [st.outputs() for st in pair]
    host_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v.cpu()) for k, v in ins[0].items()}
    host_out = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs[j]] for j in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(o.numel() * o.element_size() for o in outs[0])
    E = max(3, min(args.e2e_steps, K))
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record(stream)
    up.wait_event(t_start)
    down.wait_event(t_start)
    for s in range(E):
        j = s % 2
        if s >= 2:
            up.wait_event(ev_comp[j])           # step s-2 is done reading instance j's inputs
        with torch.cuda.stream(up), torch.no_grad():
            for k, v in ins[j].items():
                v.copy_(host_in[k], non_blocking=True)
        ev_up[j].record(up)
        stream.wait_event(ev_up[j])
        if s >= 2:
            stream.wait_event(ev_down[j])       # step s-2's outputs are on the host
        pair[j].run(stream)
        ev_comp[j].record(stream)
        down.wait_event(ev_comp[j])
        with torch.cuda.stream(down):
            for o, h in zip(outs[j], host_out[j]):
                h.copy_(o, non_blocking=True)
        ev_down[j].record(down)
    for j in range(2):
        stream.wait_event(ev_down[j])
    t_end.record(stream)
    torch.cuda.synchronize()
    e2e_ms = t_start.elapsed_time(t_end) / E

    # serial: one step at a time, its copies and compute in sequence
    ES = max(1, min(10, E))
    e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ES)]
    torch.cuda.synchronize()
    for s in range(ES):
        torch.cuda._sleep(sleep_cycles * 2)
        e_ev[s][0].record(stream)
        with torch.no_grad():
            for k, v in ins[0].items():
                v.copy_(host_in[k], non_blocking=True)
        step.run()
        for o, h in zip(outs[0], host_out[0]):
            h.copy_(o, non_blocking=True)
        e_ev[s][1].record(stream)
    torch.cuda.synchronize()
    serial_ms = sum(a.elapsed_time(b) for a, b in e_ev) / ES
    # the better of the two ways of running the stream (pipelining only pays
    # when a step is longer than the stream synchronisation it adds)
    best_ms, mode = (e2e_ms, "pipelined") if e2e_ms <= serial_ms else (serial_ms, "serial")
    e2e = {"value": world * macs / (best_ms * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": best_ms, "mode": mode, "steps": E,
           "pipeline": "two step instances alternate; inputs up and outputs down on two copy streams",
           "pipelined_ms_per_step": e2e_ms,
           "pipelined_value": world * macs / (e2e_ms * 1e-3) / 1e9,
           "serial_ms_per_step": serial_ms,
           "serial_value": world * macs / (serial_ms * 1e-3) / 1e9}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == "gemm4096":
        # the oracle on a seeded sample of 64 output rows (all 4096 columns,
        # all of k): its time, and the GPU's rows checked against it
        import numpy as np
        import oracle
        oracle.build()
        cores = os.cpu_count() or 1
        rows = np.sort(np.random.default_rng(0).choice(4096, size=64, replace=False)).astype(np.int32)
        A, B = step.A.cpu().numpy(), step.B.cpu().numpy()
        step.run()
        torch.cuda.synchronize()
        got = step.C.cpu().numpy()[rows].astype(np.float64)
        t0 = time.perf_counter()
        ref, sa = oracle.gemm(args.kind, args.mantissa, A, B, rows=rows, nthreads=cores)
        secs = time.perf_counter() - t0
        m = rows.size * 4096 * 4096
        ratio = np.abs(got - ref) / np.maximum(1e-5 * sa, 1e-300)
        cpu = {"value": m / secs / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"64 seeded output rows (numpy default_rng(0)) x 4096 columns x k = 4096: {m} MACs, "
                         f"{secs:.1f} s wall",
               "parity": {"rows": int(rows.size), "max_err_over_tol": float(ratio.max()),
                          "tol": "1e-5 * sum_k |AMSim product| per element", "ok": bool(ratio.max() <= 1.0)}}
    elif rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload in ("mlp", "dwconv3x3",
                                                                                    "dwconv3x3_s2", "dwconv5x5"):
        import oracle
        oracle.build()
        cores = os.cpu_count() or 1
        m, secs = run_oracle_sample(oracle_parts(args.workload), args.cpu_seconds, cores)
        cpu = {"value": m / secs / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{m} MACs: round-robin chunks of {cores} output rows over every contraction, "
                         f"{secs:.1f} s wall"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": wname, "macs_per_step": macs, "l2": "flushed before every timed step "
                       "(256 MiB write, outside the timed events)", "parallelism": f"replicas{world}"},
            "roofline": roofline,
            "parts_ms": {p[0]: round(t, 5) for p, t in zip(parts, part_ms)},
            "paths": part_paths,
            "e2e": e2e,
            "native_fp32": native,
            "gpu_launches": launches_timed,
            "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"], "reasons": clocks["reasons"],
                       "samples": clocks["samples"], "scope": clocks.get("scope")},
            "wall_s": wall,
        }
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
