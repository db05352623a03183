#!/usr/bin/env python
"""Benchmark of the MoE layer forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one moe_layer_forward (router, dispatch, gather, up-projection,
down-projection, combine, aux loss) over the Mixtral-shaped prefill workload
(T=4096, d=4096, d_ff=14336, E=8, top-2, SwiGLU, bf16, dropless), inputs and
weights resident in HBM.  Prints one JSON line on rank 0.

Under torchrun (N > 1) every rank runs an independent replica of the layer on
its own GPU (the layer has no cross-GPU step); value = all ranks' tokens / the
slowest rank's time.

--impl reference times the CPU oracle (the plain fp64 C implementation under
oracle/) on a bounded sample of the same workload, as the baseline arm.
"""
import argparse
import json
import os
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_mixture_experts_59_b300 import binding, workloads  # noqa: E402

METRIC = "MoE-layer tokens/s at Mixtral shape bf16; grouped-GEMM % BF16 peak; decode HBM GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}

def kernels_per_step(cfg):
    """The library's kernel launches for one layer call of `cfg`: a
    decode-sized batch routes and dispatches in one launch (T <= 256,
    T*k <= 512, T*E <= 2048), else router logits, top-k, dispatch rank and
    dispatch scatter; then gather, up, down, combine."""
    T, E, k = cfg["T"], cfg["E"], cfg["k"]
    front = 1 if (T <= 256 and T * k <= 512 and T * E <= 2048) else 4
    return front + 4


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixtral_prefill")
    ap.add_argument("--decode-workload", default="mixtral_decode")
    ap.add_argument("--tokens", type=int, default=None, help="override T (profiling cases)")
    ap.add_argument("--experts", type=int, default=None, help="override E (profiling cases)")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch without programmatic dependent launch (MOE_PDL=0)")
    ap.add_argument("--gemm", default=None, choices=["tc1", "pair", "swap"],
                    help="force the expert GEMM kernel (default: the library's choice)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    low = ap.add_mutually_exclusive_group()
    low.add_argument("--fp8", action="store_true",
                     help="the main workload with FP8 E4M3 expert weights (profiling cases)")
    low.add_argument("--fp4", action="store_true",
                     help="the main workload with packed 4-bit (E2M1) expert weights")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the fine-grained, Switch-skewed and tiny fp32 workloads")
    ap.add_argument("--sustained-seconds", type=float, default=2.5,
                    help="length of the back-to-back loop timed against the sustained peak "
                         "(0 = skip)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--sweep", default=None,
                    help="comma-separated token counts: time the layer at each T on the "
                         "workload's weights for every GEMM kernel (prefill/decode crossover) "
                         "and print one JSON line with the table instead of the bench line")
    return ap.parse_args()


# --------------------------------------------------------------- plumbing
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


TRAFFIC_SOURCES = ("ffn_swap.cu", "ffn_tc.cu", "ffn_tc2.cu", "ffn_tc_common.cuh", "tc_ptx.cuh")


def kernel_sources_digest():
    """sha256 over the GEMM kernel sources: a recorded DRAM-traffic figure is
    reported only while the sources it was measured on are unchanged."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_mixture_experts_59_b300", "csrc")
    for name in TRAFFIC_SOURCES:
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, kernel):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)
    recorded under profiles/ for (workload, kernel), if the kernel sources
    still match the digest recorded with it; else None."""
    path = os.path.join(ROOT, "profiles", "traffic_%s.txt" % workload)
    if not os.path.exists(path):
        return None, None
    digest = kernel_sources_digest()
    with open(path) as fh:
        for line in fh:
            parts = line.split()
            if len(parts) >= 4 and parts[0] == "traffic" and parts[1] == kernel:
                if parts[3] == digest:
                    return int(parts[2]), digest
                return None, digest
    return None, digest


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


_REASON_BITS = (("gpu_idle", 0x1), ("sw_power_cap", 0x4), ("hw_slowdown", 0x8),
                ("sw_thermal_slowdown", 0x20), ("hw_thermal_slowdown", 0x40),
                ("hw_power_brake_slowdown", 0x80))


class _Nvml:
    """Read-only NVML queries through ctypes (libnvidia-ml ships with the
    driver; the Python wrapper may be absent): SM clock, its maximum, power
    draw and the active clock-event reasons of one device."""
    NVML_CLOCK_SM = 1

    def __init__(self, cuda_index):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.lib = lib
        self.dev = ctypes.c_void_p()
        uuid = str(torch.cuda.get_device_properties(cuda_index).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) != 0:
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(cuda_index), ctypes.byref(self.dev)) != 0:
                raise RuntimeError("no NVML handle for the device")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _uint(self, fn, *args):
        v = self.ct.c_uint(0)
        if fn(self.dev, *args, self.ct.byref(v)) != 0:
            raise RuntimeError("NVML query failed")
        return v.value

    def sm_mhz(self):
        return self._uint(self.lib.nvmlDeviceGetClockInfo, self.ct.c_int(self.NVML_CLOCK_SM))

    def sm_max_mhz(self):
        return self._uint(self.lib.nvmlDeviceGetMaxClockInfo, self.ct.c_int(self.NVML_CLOCK_SM))

    def power_w(self):
        return self._uint(self.lib.nvmlDeviceGetPowerUsage) / 1000.0

    def reasons(self):
        v = self.ct.c_ulonglong(0)
        if self.reasons_fn(self.dev, self.ct.byref(v)) != 0:
            raise RuntimeError("NVML reasons query failed")
        return v.value


class ClockSampler:
    """SM clock, power and clock-event reasons of one GPU, sampled about every
    2 ms through NVML in a background thread while a timed region runs (a
    timed region of 20 layer calls lasts ~40 ms, so a 100 ms nvidia-smi poll
    would mostly see the idle GPU around it).  The summary's sm_mhz is the
    median over samples taken while the GPU was busy (NVML's gpu_idle reason
    clear); without NVML the summary only says why."""

    def __init__(self, device_index, period_s=0.002):
        self.idx = device_index
        self.period = period_s
        self.rows = []
        self.thread = None
        self.error = None
        self.windows = []

    def mark(self, t0, t1):
        """A host-time window [t0, t1] (time.perf_counter) that covered GPU
        work: the summary uses only samples taken inside such windows."""
        self.windows.append((t0, t1))

    def start(self):
        import threading
        self.rows = []
        self.error = None
        try:
            self.nv = _Nvml(self.idx)
            self.max_mhz = float(self.nv.sm_max_mhz())
        except Exception as e:          # no NVML: the summary says why
            self.error = "NVML unavailable: %s" % e
            return
        self.stop_flag = threading.Event()

        def loop():
            n = 0
            while not self.stop_flag.is_set():
                try:
                    sm = self.nv.sm_mhz()
                    rs = self.nv.reasons()
                    pw = self.nv.power_w() if n % 4 == 0 else None
                    self.rows.append((time.perf_counter(), float(sm), int(rs), pw))
                except Exception as e:
                    self.error = "NVML query failed: %s" % e
                n += 1
                time.sleep(self.period)

        self.thread = threading.Thread(target=loop, daemon=True)
        self.thread.start()

    def stop(self):
        if self.thread is None:
            return {"error": self.error} if self.error else None
        self.stop_flag.set()
        self.thread.join(timeout=5)
        self.thread = None
        rows = self.rows
        if not rows:
            return {"error": self.error or "no samples"}
        if self.windows:
            rows = [r for r in rows if any(a <= r[0] <= b for a, b in self.windows)]
            if not rows:
                return {"error": "no samples inside the timed windows"}
        busy = [r for r in rows if not (r[2] & 0x1)]
        use = busy if busy else rows
        sm = np.array([r[1] for r in use])
        reasons = set()
        for r in use:
            for name, bit in _REASON_BITS:
                if name != "gpu_idle" and (r[2] & bit):
                    reasons.add(name)
        power = [r[3] for r in rows if r[3] is not None]
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": self.max_mhz,
                "sm_mhz_p10": float(np.percentile(sm, 10)), "sm_mhz_p90": float(np.percentile(sm, 90)),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": float(max(power)) if power else None,
                "source": "NVML (ctypes), ~2 ms period, samples inside the timed passes only"}


# ------------------------------------------------------------ our path
def algorithmic(cfg, R):
    """FLOPs and weight bytes of one layer call with R kept assignments."""
    T, d, F, E, k = cfg["T"], cfg["d"], cfg["F"], cfg["E"], cfg["k"]
    Fs = cfg.get("F_shared", 0) or 0
    up_mult = 2 if cfg["act"] == "swiglu" else 1
    up = 2.0 * R * d * F * up_mult + 2.0 * T * d * Fs * 2
    down = 2.0 * R * F * d + 2.0 * T * Fs * d
    router = 2.0 * T * d * E
    return dict(up=up, down=down, router=router, total=up + down + router)


def time_layer(layer, x, steps, warmup, world, outputs, clocks=None, settle_s=1.0):
    """Times `steps` plain layer calls (the step time), then the same number of
    calls that record CUDA events at every stage boundary on the launching
    stream (the per-kernel times: events between kernels can keep a kernel
    from starting early, so they stay out of the step time).  Each pass starts
    after `settle_s` of idle GPU: under the 1.1 kW cap a B300 running these
    GEMMs back to back lowers its SM clock after about 40 ms, so two passes
    timed one after the other would see different clocks; with the pause both
    see the same state (the sustained leg measures the capped state)."""
    for _ in range(warmup):
        layer.forward(x, outputs=outputs)
    torch.cuda.synchronize()
    st = binding.device_status(layer.ws)
    if st != 0:
        raise RuntimeError("device status %d after warm-up" % st)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    time.sleep(settle_s)            # both passes start from an idle GPU (see docstring)
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    h0 = time.perf_counter()
    start.record()
    for _ in range(steps):
        layer.forward(x, outputs=outputs)
    end.record()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark(h0, time.perf_counter())
    ms = start.elapsed_time(end) / steps
    # profiled pass: stage boundaries
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(steps)]
    for row in evs:
        for e in row:
            e.record()
    pstart, pend = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    time.sleep(settle_s)
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    pstart.record()
    for i in range(steps):
        layer.forward(x, outputs=outputs, events=evs[i])
    pend.record()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark(h0, time.perf_counter())
    clk = clocks.stop() if clocks else None
    barrier(world)
    torch.cuda.synchronize()
    ms_prof = pstart.elapsed_time(pend) / steps
    stages = np.array([[row[j].elapsed_time(row[j + 1]) for j in range(6)] for row in evs])
    names = ("router", "dispatch", "gather", "up_gemm", "down_gemm", "combine")
    st = binding.device_status(layer.ws)
    if st != 0:
        raise RuntimeError("device status %d after timed steps" % st)
    out = {n: float(stages[:, j].mean()) for j, n in enumerate(names)}
    out["step_profiled"] = float(ms_prof)
    return ms, out, clk


def workload_config(args):
    over = {}
    if args.tokens is not None:
        over["T"] = args.tokens
    if args.experts is not None:
        over["E"] = args.experts
    if args.gemm:
        over["gemm_kernel"] = args.gemm
    return workloads.config(args.workload, **over)


def weight_bytes(cfg, counts_kept):
    """Bytes of expert weights a layer call must stream: every routed expert
    that kept at least one assignment (its W1, W3, W2 and biases; codes,
    block and row scales for low-bit weights) plus the shared expert."""
    d, F = cfg["d"], cfg["F"]
    mats = 3 if cfg["act"] == "swiglu" else 2
    if cfg.get("weight_fp4"):
        per = int(mats * d * F * 80 / 128) + (2 * F + d) * 4
    elif cfg.get("weight_fp8"):
        per = mats * d * F + (2 * F + d) * 4
    else:
        es = 4 if cfg["dtype"] == "f32" else 2
        per = (mats * d * F + ((F + d) if cfg["has_bias"] else 0)) * es
    hit = int((np.asarray(counts_kept) > 0).sum())
    Fs = cfg.get("F_shared", 0) or 0
    return hit * per + 3 * d * Fs * (4 if cfg["dtype"] == "f32" else 2), hit


REJECT_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clock_rejection(clk, low_frac=0.85):
    """Why a timed pass's clock record disqualifies its number, or None.
    Two things disqualify it: a hardware or thermal slowdown seen during the
    pass, or a median SM clock well below the maximum with no reason reported
    (a clock lock left by an earlier user). The power cap alone is kept,
    since it is the normal state of a long dense run."""
    if not clk or "sm_mhz" not in clk:
        return None
    bad = [r for r in clk.get("reasons", []) if r in REJECT_REASONS]
    if bad:
        return "clock-event reasons during the pass: " + ", ".join(bad)
    mx = clk.get("sm_max_mhz")
    if mx and clk["sm_mhz"] < low_frac * mx and not clk.get("reasons"):
        return "median SM clock %.0f of %.0f MHz with no reason reported" % (clk["sm_mhz"], mx)
    return None


def pick_tensor_peak(burst, sustained, region_ms, clk):
    """The bf16 tensor peak a timed pass is judged against: the burst figure
    for a pass of up to 100 ms at full clock, the sustained (power-capped)
    figure for a longer pass or one whose median SM clock sat below 90% of the
    maximum.  Returns (peak, name, reason)."""
    mhz = clk.get("sm_mhz") if clk else None
    mx = clk.get("sm_max_mhz") if clk else None
    if region_ms > 100.0:
        return sustained, "bf16_tflops_sustained", "the timed region is %.0f ms of back-to-back " \
            "layer calls" % region_ms
    if mhz and mx and mhz < 0.9 * mx:
        return sustained, "bf16_tflops_sustained", "median SM clock %.0f of %.0f MHz in the " \
            "timed region" % (mhz, mx)
    return burst, "bf16_tflops", "burst: the timed region is %.0f ms at a median %s MHz" % (
        region_ms, "%.0f" % mhz if mhz else "unknown")


def gemm_roofline(alg, wbytes, gemm_s, peaks):
    """The grouped GEMMs' roofline time max(flop / tensor peak, weight bytes /
    HBM peak) at the burst tensor peak (the GEMMs are timed over tens of
    milliseconds), and the fraction of it the measured time reaches."""
    tf = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    bw = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    t_c = (alg["up"] + alg["down"]) / (tf * 1e12)
    t_m = wbytes / (bw * 1e9)
    t_r = max(t_c, t_m)
    return {"bound": "tensor" if t_c >= t_m else "hbm", "roofline_ms": round(t_r * 1e3, 4),
            "compute_ms": round(t_c * 1e3, 4), "bytes_ms": round(t_m * 1e3, 4),
            "frac": round(t_r / gemm_s, 4), "tensor_peak_tflops": tf, "hbm_peak_gbs": bw}


def run_ours(args, world, rank, local):
    dev = torch.device("cuda", local)
    peaks, peak_src = measured_peaks()
    cfg = workload_config(args)
    inp = workloads.make_inputs(cfg, device=dev)
    bf16_inp = inp
    if args.fp8 or args.fp4:
        inp = (workloads.quantize_experts_fp4 if args.fp4 else workloads.quantize_experts_fp8)(inp)
        cfg = inp["cfg"]
        if args.no_decode:
            bf16_inp = None                      # only the low-bit copy stays on the device
    layer = binding.MoeLayer(cfg, inp, device=dev)
    x = inp["x"]
    outputs = {"y": torch.empty_like(x), "counts_kept": torch.empty(cfg["E"], dtype=torch.int32,
                                                                   device=dev)}
    clocks = ClockSampler(local)
    ms_local, stages, clk = time_layer(layer, x, args.steps, args.warmup, world, outputs, clocks)
    # a pass whose clock record disqualifies it is taken once more after a
    # longer idle; every rank takes part when any rank's record asks for it
    why = clock_rejection(clk)
    remeasured = None
    if max_over_ranks(1.0 if why else 0.0, world) > 0:
        remeasured = {"first_ms_per_step": round(ms_local, 4), "first_clocks": clk,
                      "why": why or "another rank's clock record"}
        time.sleep(5.0)
        clocks = ClockSampler(local)
        ms_local, stages, clk = time_layer(layer, x, args.steps, args.warmup, world, outputs,
                                           clocks)
    ms = max_over_ranks(ms_local, world)
    R = int(outputs["counts_kept"].sum().item())
    alg = algorithmic(cfg, R)
    value = cfg["T"] * world / (ms / 1e3)

    up_s = stages["up_gemm"] / 1e3
    dn_s = stages["down_gemm"] / 1e3
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    peak, peak_kind, peak_why = pick_tensor_peak(burst, sustained, ms * args.steps, clk)
    up_tf = alg["up"] / up_s / 1e12
    kname = "up_gemm/%s" % (args.gemm or "auto")
    traffic, digest = recorded_traffic(args.workload, kname) if args.tokens is None and \
        args.experts is None else (None, None)
    mhz = clk.get("sm_mhz") if clk else None      # absent when no sample fell inside the passes
    roof = {"kernel": "up-projection grouped GEMM (SwiGLU epilogue)", "bound": "tensor",
            "achieved": round(up_tf, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(up_tf / peak, 4), "traffic": traffic,
            "frac_of_burst_peak": round(up_tf / burst, 4),
            "frac_of_sustained_peak": round(up_tf / sustained, 4),
            "traffic_note": "ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, "
                            "profiles/traffic_%s.txt; null if the kernel sources changed "
                            "since (sources digest %s)" % (args.workload, digest),
            "peak_source": "%s %s (%s)" % (peak_src, peak_kind, peak_why),
            "algorithmic_flop_per_launch": alg["up"], "launch_ms": round(stages["up_gemm"], 4),
            "launch_mcycles_at_median_sm_clock": round(stages["up_gemm"] * mhz / 1e3, 4)
            if mhz else None}
    gg_tf = (alg["up"] + alg["down"]) / (up_s + dn_s) / 1e12
    wbytes, hit = weight_bytes(cfg, outputs["counts_kept"].cpu().numpy())
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("bf16, e2m1 expert weights" if args.fp4 else
                  "bf16, e4m3 expert weights" if args.fp8 else "bf16"),
        "data": "synthetic: seeded x~N(0,1), expert weights~N(0,0.02), router~N(0,1/sqrt(d)); bf16",
        "config": {"workload": args.workload, "T": cfg["T"], "d_model": cfg["d"], "d_ff": cfg["F"],
                   "experts": cfg["E"], "top_k": cfg["k"], "act": cfg["act"],
                   "capacity": "dropless" if not cfg["capacity_factor"] else cfg["capacity_factor"],
                   "l2": "inputs larger than L2 (expert weights %.2f GB vs 126 MB L2); no flush"
                         % (sum(inp[k].numel() * inp[k].element_size() for k in ("W1", "W3", "W2")
                                if inp.get(k) is not None) / 1e9),
                   "parallelism": "replicas" if world > 1 else "single",
                   "gemm_kernel": args.gemm or "auto"},
        "roofline": roof,
        "grouped_gemm": {"tflops": round(gg_tf, 1), "frac_of_peak": round(gg_tf / peak, 4),
                         "peak": peak, "up_ms": round(stages["up_gemm"], 4),
                         "down_ms": round(stages["down_gemm"], 4),
                         "down_tflops": round(alg["down"] / dn_s / 1e12, 1),
                         "roofline": gemm_roofline(alg, wbytes, up_s + dn_s, peaks)},
        "stage_ms": {k: round(v, 4) for k, v in stages.items()},
        "timing": "value from %d plain layer calls; stage_ms and the roofline's launch_ms from "
                  "%d more calls with CUDA events at the stage boundaries" % (args.steps, args.steps),
        "layer_tflops": round(alg["total"] / (ms / 1e3) / 1e12, 1),
        "gpu_launches": kernels_per_step(cfg) * args.steps,
        "pdl": os.environ.get("MOE_PDL", "1") != "0",
        "clocks": clk,
        **({"remeasured": remeasured} if remeasured else {}),
    }
    if args.sustained_seconds > 0:
        result["sustained"] = run_sustained(layer, x, outputs, cfg, alg, args, world, peaks,
                                            peak_src, local)
    if not args.no_e2e:
        result["e2e"] = run_e2e(layer, cfg, x, args, world, dev)
    del layer
    if not args.no_decode:
        result["decode"] = run_decode(args, bf16_inp, world, dev, peaks, peak_src)
        result["decode_fp8"] = run_decode(args, bf16_inp, world, dev, peaks, peak_src, low="fp8")
        result["decode_fp4"] = run_decode(args, bf16_inp, world, dev, peaks, peak_src, low="fp4")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(inp, cfg, args.cpu_seconds)
    del inp, bf16_inp
    torch.cuda.empty_cache()
    if not args.no_configs:
        for name in ("fine_grained", "switch_skewed", "tiny_fp32"):
            result[name] = run_workload(name, args, world, dev, peaks, local)
            torch.cuda.empty_cache()
    return result


def run_sustained(layer, x, outputs, cfg, alg, args, world, peaks, peak_src, local):
    """Back-to-back layer calls for about args.sustained_seconds, each with
    stage events, with their own clock record: the up-projection against the
    sustained bf16 peak (a seconds-long loop under the power cap), and its
    time in SM cycles at the median clock so the clock dependence shows."""
    probe = time.perf_counter()
    layer.forward(x, outputs=outputs)
    torch.cuda.synchronize()
    one = max(time.perf_counter() - probe, 1e-4)
    n = int(min(5000, max(50, args.sustained_seconds / one)))
    time.sleep(1.0)                 # start from an idle GPU, like the timed passes
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(n)]
    for row in evs:                 # torch creates the CUDA event at its first record
        for e in row:
            e.record()
    clocks = ClockSampler(local)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    clocks.start()
    h0 = time.perf_counter()
    start.record()
    for i in range(n):
        layer.forward(x, outputs=outputs, events=evs[i])
    end.record()
    torch.cuda.synchronize()
    clocks.mark(h0, time.perf_counter())
    clk = clocks.stop()
    if binding.device_status(layer.ws) != 0:
        raise RuntimeError("device status after the sustained loop")
    total_ms = start.elapsed_time(end)
    up = np.array([r[3].elapsed_time(r[4]) for r in evs])
    dn = np.array([r[4].elapsed_time(r[5]) for r in evs])
    peak = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    up_tf = alg["up"] / (up.mean() / 1e3) / 1e12
    mhz = clk.get("sm_mhz") if clk else None      # absent when no sample fell inside the passes
    return {"seconds": round(total_ms / 1e3, 3), "steps": n, "ms_per_step": round(total_ms / n, 4),
            "tokens_per_s": round(cfg["T"] * n / (total_ms / 1e3), 1),
            "up_gemm_ms": round(float(up.mean()), 4), "down_gemm_ms": round(float(dn.mean()), 4),
            "up_tflops": round(up_tf, 1), "peak": peak, "frac": round(up_tf / peak, 4),
            "peak_source": "%s bf16_tflops_sustained" % peak_src,
            "up_gemm_mcycles_at_median_sm_clock": round(float(up.mean()) * mhz / 1e3, 4) if mhz else None,
            "timing": "every call records events at its stage boundaries", "clocks": clk}


def time_layer_graph(layer, x, steps, warmup, outputs, flush):
    """The layer call captured once in a CUDA graph and replayed: mean device
    time per layer over `steps` back-to-back replays (warm L2), and over
    `steps` replays each after an L2 flush (only the replay inside its
    events).  Returns the keys to add, or the capture error."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            layer.forward(x, outputs=outputs)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer.forward(x, outputs=outputs)
    except Exception as e:           # report, do not fail the bench
        return {"graph_error": str(e)[:200]}
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    warm = a.elapsed_time(b) / steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for e0, e1 in evs:
        flush.fill_(1)
        e0.record()
        g.replay()
        e1.record()
    torch.cuda.synchronize()
    cold = float(np.mean([e0.elapsed_time(e1) for e0, e1 in evs]))
    if binding.device_status(layer.ws) != 0:
        raise RuntimeError("device status after the graph replays")
    del g
    return {"us_per_layer_graph": round(warm * 1e3, 2),
            "us_per_layer_graph_l2_flushed": round(cold * 1e3, 2),
            "graph_timing": "the layer call captured in one CUDA graph; %d replays back to "
                            "back, and %d each after a 256 MB L2 flush" % (steps, steps)}


def run_workload(name, args, world, dev, peaks, local):
    """Another of the five workloads at its full size: layer time, tokens/s,
    the grouped GEMMs against their roofline (flop at the burst tensor peak,
    weight bytes of the experts hit at the HBM peak), drops and aux loss."""
    cfg = workloads.config(name)
    inp = workloads.make_inputs(cfg, device=dev)
    layer = binding.MoeLayer(cfg, inp, device=dev)
    x = inp["x"]
    outputs = {"y": torch.empty_like(x),
               "counts_kept": torch.empty(cfg["E"], dtype=torch.int32, device=dev),
               "stats": torch.empty(2, dtype=torch.float32, device=dev)}
    steps = max(10, min(args.steps, 20))
    clocks = ClockSampler(local)
    ms, stages, clk = time_layer(layer, x, steps, args.warmup, world, outputs, clocks)
    out = {"workload": name, "T": cfg["T"], "d_model": cfg["d"], "d_ff": cfg["F"],
           "experts": cfg["E"], "top_k": cfg["k"], "act": cfg["act"],
           "F_shared": cfg.get("F_shared", 0), "dtype": cfg["dtype"],
           "capacity": "dropless" if not cfg["capacity_factor"] else cfg["capacity_factor"]}
    wbytes, hit = weight_bytes(cfg, outputs["counts_kept"].cpu().numpy())
    if wbytes < 2 * 126e6:
        # a layer this small takes less GPU time than the host needs to issue
        # it through Python, so the plain loop times the host: time it again
        # as CUDA-graph replays (device time), warm and with an L2 flush
        # (a write larger than L2) before each replay
        flush = torch.empty(256 * 2 ** 20 // 4, dtype=torch.float32, device=dev)
        out.update(time_layer_graph(layer, x, steps, args.warmup, outputs, flush))
        del flush
    R = int(outputs["counts_kept"].sum().item())
    stats = outputs["stats"].cpu().numpy()
    alg = algorithmic(cfg, R)
    gemm_s = (stages["up_gemm"] + stages["down_gemm"]) / 1e3
    out.update({
        "ms_per_step": round(ms, 4), "tokens_per_s": round(cfg["T"] * world / (ms / 1e3), 1),
        "steps": steps, "kept_rows": R, "experts_hit": hit, "weight_bytes": wbytes,
        "drop_fraction": round(float(stats[1]), 6), "aux_loss": round(float(stats[0]), 6),
        "gemm_ms": round(gemm_s * 1e3, 4),
        "gemm_tflops": round((alg["up"] + alg["down"]) / gemm_s / 1e12, 1),
        "up_tflops": round(alg["up"] / (stages["up_gemm"] / 1e3) / 1e12, 1),
        "down_tflops": round(alg["down"] / (stages["down_gemm"] / 1e3) / 1e12, 1),
        "weight_gbs": round(wbytes / gemm_s / 1e9, 1),
        "layer_tflops": round(alg["total"] / (ms / 1e3) / 1e12, 2),
        "stage_ms": {k: round(v, 4) for k, v in stages.items()},
        "clocks": clk})
    if cfg["dtype"] == "bf16":
        out["gemm_roofline"] = gemm_roofline(alg, wbytes, gemm_s, peaks)
    del layer, inp, outputs
    return out


def run_e2e(layer, cfg, x, args, world, dev):
    """Same metric through the public API with host buffers: every step copies
    its x from pinned host memory to the device, runs the layer and copies its
    y back to pinned host memory.  The copies run on their own streams with
    double-buffered device x / y, ordered by events, so step i+1's input copy
    and step i-1's output copy overlap step i's layer (the usual way to feed a
    layer from the host); the timed region spans all copies of all steps,
    including the first step's input copy and the last step's output copy,
    which nothing overlaps."""
    x_host = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    x_host.copy_(x.cpu())
    y_host = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    y_dev = [torch.empty_like(x) for _ in range(2)]
    comp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]      # x_dev[b] loaded
    ev_comp = [torch.cuda.Event() for _ in range(2)]    # layer done with x_dev[b], y_dev[b] ready
    ev_out = [torch.cuda.Event() for _ in range(2)]     # y_dev[b] copied out

    def step(i):
        b = i % 2
        with torch.cuda.stream(h2d):
            if i >= 2:
                h2d.wait_event(ev_comp[b])
            x_dev[b].copy_(x_host, non_blocking=True)
            ev_in[b].record(h2d)
        comp.wait_event(ev_in[b])
        if i >= 2:
            comp.wait_event(ev_out[b])
        layer.forward(x_dev[b], outputs={"y": y_dev[b]}, stream=comp)
        ev_comp[b].record(comp)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_comp[b])
            y_host[b].copy_(y_dev[b], non_blocking=True)
            ev_out[b].record(d2h)

    steps = max(10, args.steps)     # as many layer calls as the device-timed pass
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(comp)
    h2d.wait_stream(comp)
    d2h.wait_stream(comp)
    for i in range(steps):
        step(i)
    comp.wait_stream(d2h)
    end.record(comp)
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end) / steps, world)
    nbytes = x.numel() * x.element_size()
    return {"value": round(cfg["T"] * world / (ms / 1e3), 1), "unit": "tokens/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
            "steps": steps, "overlap": "input copy of step i+1 and output copy of step i-1 "
                                       "overlap the layer of step i (double-buffered, own streams)"}


def run_decode(args, prefill_inp, world, dev, peaks, peak_src, low=None):
    """Decode-shaped layer (T=32) on the same expert weights: weight streaming
    of the experts that got tokens, against the HBM roofline.  low="fp8": the
    same weights quantised to E4M3 with per-row scales (half the bytes);
    low="fp4": packed 4-bit (80 bytes per 128 values, 0.3125 of the bytes)."""
    cfg = workloads.config(args.decode_workload)
    inp = dict(prefill_inp)
    inp["x"] = workloads.make_x(cfg, dev)
    inp["cfg"] = cfg
    if low == "fp8":
        inp = workloads.quantize_experts_fp8(inp)
        cfg = inp["cfg"]
    elif low == "fp4":
        inp = workloads.quantize_experts_fp4(inp)
        cfg = inp["cfg"]
    layer = binding.MoeLayer(cfg, inp, device=dev)
    outputs = {"y": torch.empty_like(inp["x"]),
               "counts_kept": torch.empty(cfg["E"], dtype=torch.int32, device=dev)}
    steps = max(20, args.steps)
    ms, stages, _ = time_layer(layer, inp["x"], steps, args.warmup, world, outputs)
    ms = max_over_ranks(ms, world)
    wbytes, hit = weight_bytes(cfg, outputs["counts_kept"].cpu().numpy())
    gemm_s = (stages["up_gemm"] + stages["down_gemm"]) / 1e3
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    gbs = wbytes / gemm_s / 1e9
    del layer
    tag = {None: "", "fp8": " (FP8 E4M3 expert weights)",
           "fp4": " (packed 4-bit E2M1 expert weights, E4M3 block scales)"}[low]
    return {"workload": args.decode_workload + tag,
            "T": cfg["T"], "experts_hit": hit,
            "tokens_per_s": round(cfg["T"] * world / (ms / 1e3), 1), "ms_per_step": round(ms, 4),
            "weight_bytes": wbytes, "gemm_ms": round(gemm_s * 1e3, 4),
            "hbm_gbs": round(gbs, 1), "hbm_peak_gbs": hbm, "frac_of_hbm": round(gbs / hbm, 4),
            "layer_gbs": round(wbytes / (ms / 1e3) / 1e9, 1),
            "peak_source": "%s hbm_gbs" % peak_src, "stage_ms": {k: round(v, 4) for k, v in stages.items()}}


# ---------------------------------------------------------- CPU oracle
def _oracle_sample(oracle, inp_cpu, cfg, n):
    """The oracle's whole layer for the first n tokens: own router logits,
    softmax/top-k, dispatch with capacity, experts, combine."""
    toks = np.arange(n, dtype=np.int32)
    logits = oracle.router_logits(inp_cpu["x"], inp_cpu["Wr"], inp_cpu.get("logit_bias"), tokens=toks)
    idx, w, probs = oracle.topk(logits, cfg["k"])
    cap = oracle.capacity(n, cfg["k"], cfg["E"], cfg["capacity_factor"])
    disp = oracle.dispatch(idx, cfg["E"], cap)
    sub = dict(inp_cpu)
    sub["x"] = inp_cpu["x"][:n]
    sub["cfg"] = dict(cfg, T=n)
    oracle.layer_tokens(sub, idx, w, disp["drop_mask"], toks)
    oracle.aux_loss(disp["counts_pre"], probs)


def _host_inputs(inp):
    return {k: (v.detach().cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def cpu_baseline(inp, cfg, seconds):
    import oracle
    inp_cpu = _host_inputs(inp)
    oracle.set_threads(0)
    cores = oracle.get_threads()
    t0 = time.perf_counter()
    _oracle_sample(oracle, inp_cpu, cfg, cores)
    per = (time.perf_counter() - t0) / cores
    n = int(max(cores, min(cfg["T"], seconds / max(per, 1e-9))))
    n = max(cores, (n // cores) * cores)
    t0 = time.perf_counter()
    _oracle_sample(oracle, inp_cpu, cfg, n)
    dt = time.perf_counter() - t0
    return {"value": round(n / dt, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "first %d of %d tokens of %s, whole layer (router, top-k, dispatch, "
                      "experts, combine, aux) in fp64; %.1f s" % (n, cfg["T"], cfg["name"], dt)}


def run_reference(args, world, rank, local):
    """The CPU oracle as the baseline arm, timed on the host cores."""
    import oracle
    cfg = workload_config(args)
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    inp_cpu = _host_inputs(workloads.make_inputs(cfg, device=dev))
    if dev.type == "cuda":
        torch.cuda.empty_cache()
    oracle.set_threads(0)
    cores = oracle.get_threads()
    # size one step at about 2-3 s of host time so the whole run stays short
    t0 = time.perf_counter()
    _oracle_sample(oracle, inp_cpu, cfg, cores)
    per = (time.perf_counter() - t0) / cores
    budget = max(1.0, min(3.0, 120.0 / max(1, args.steps + args.warmup)))
    n = max(cores, int(budget / max(per, 1e-9)) // cores * cores)
    n = min(n, cfg["T"])
    for _ in range(args.warmup):
        _oracle_sample(oracle, inp_cpu, cfg, n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_sample(oracle, inp_cpu, cfg, n)
    dt = (time.perf_counter() - t0) / args.steps
    value = n / dt
    sample = ("first %d of %d tokens of %s per step, whole layer in fp64 (oracle/)"
              % (n, cfg["T"], cfg["name"]))
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64",
            "data": "synthetic: same seeded inputs as the GPU arm",
            "config": {"workload": args.workload, "T": cfg["T"], "d_model": cfg["d"],
                       "d_ff": cfg["F"], "experts": cfg["E"], "top_k": cfg["k"]},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def run_sweep(args, world, local):
    """Prefill/decode crossover: the same layer and weights at several T, each
    GEMM kernel forced in turn, plus the library's automatic choice."""
    dev = torch.device("cuda", local)
    peaks, _ = measured_peaks()
    base = workload_config(args)
    weights = workloads.make_weights(base, dev)
    per_expert = (3 if base["act"] == "swiglu" else 2) * base["d"] * base["F"] * 2
    rows = []
    for T in [int(v) for v in args.sweep.split(",")]:
        cfg = dict(base, T=T)
        inp = dict(weights)
        inp["x"] = workloads.make_x(cfg, dev)
        inp["cfg"] = cfg
        entry = {"T": T}
        for g in ("auto", "tc1", "swap", "pair"):
            cfg = dict(base, T=T, gemm_kernel=g)
            layer = binding.MoeLayer(cfg, inp, device=dev)
            outputs = {"y": torch.empty_like(inp["x"]),
                       "counts_kept": torch.empty(cfg["E"], dtype=torch.int32, device=dev)}
            steps = max(10, min(args.steps, 50))
            ms, stages, _ = time_layer(layer, inp["x"], steps, args.warmup, world, outputs,
                                       settle_s=0.25)
            R = int(outputs["counts_kept"].sum().item())
            hit = int((outputs["counts_kept"] > 0).sum().item())
            alg = algorithmic(cfg, R)
            gemm_ms = stages["up_gemm"] + stages["down_gemm"]
            entry[g] = {"ms": round(ms, 4), "tokens_per_s": round(T / (ms / 1e3), 1),
                        "gemm_ms": round(gemm_ms, 4),
                        "gemm_tflops": round((alg["up"] + alg["down"]) / (gemm_ms / 1e3) / 1e12, 1),
                        "weight_gbs": round(hit * per_expert / (gemm_ms / 1e3) / 1e9, 1)}
            del layer
        rows.append(entry)
    return {"sweep": args.workload, "d_model": base["d"], "d_ff": base["F"], "experts": base["E"],
            "top_k": base["k"], "hbm_peak_gbs": peaks.get("hbm_gbs"),
            "bf16_peak_tflops_sustained": peaks.get("bf16_tflops_sustained"), "rows": rows}


def main():
    args = parse_args()
    if args.sweep:
        world, rank, local = dist_init()
        res = run_sweep(args, world, local)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    if args.no_pdl:
        os.environ["MOE_PDL"] = "0"
    world, rank, local = dist_init()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world, rank, local)), flush=True)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    res = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
