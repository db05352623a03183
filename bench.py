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
import subprocess
import sys
import tempfile
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
    ap.add_argument("--steps", type=int, default=200)
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


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9 or parts[0] != str(self.idx):
                    continue
                rows.append(parts)
        os.remove(self.path)
        if not rows:
            return None

        def num(s):
            try:
                return float(s)
            except ValueError:
                return float("nan")
        sm = np.array([num(r[1]) for r in rows])
        mx = np.array([num(r[2]) for r in rows])
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() in ("active", "1"):
                    reasons.add(name)
        busy = sm[sm >= np.nanmedian(sm) * 0.5] if len(sm) else sm
        return {"sm_mhz": float(np.nanmedian(busy)) if len(busy) else None,
                "sm_max_mhz": float(np.nanmax(mx)) if len(mx) else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": float(np.nanmax([num(r[3]) for r in rows]))}


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


def time_layer(layer, x, steps, warmup, world, outputs, clocks=None):
    """Times `steps` plain layer calls (the step time), then the same number of
    calls that record CUDA events at every stage boundary on the launching
    stream (the per-kernel times: events between kernels can keep a kernel
    from starting early, so they stay out of the step time)."""
    for _ in range(warmup):
        layer.forward(x, outputs=outputs)
    torch.cuda.synchronize()
    st = binding.device_status(layer.ws)
    if st != 0:
        raise RuntimeError("device status %d after warm-up" % st)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    start.record()
    for _ in range(steps):
        layer.forward(x, outputs=outputs)
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    # profiled pass: stage boundaries
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(steps)]
    for row in evs:
        for e in row:
            e.record()
    pstart, pend = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    pstart.record()
    for i in range(steps):
        layer.forward(x, outputs=outputs, events=evs[i])
    pend.record()
    torch.cuda.synchronize()
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
    return workloads.config(args.workload, **over)


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
    ms = max_over_ranks(ms_local, world)
    R = int(outputs["counts_kept"].sum().item())
    alg = algorithmic(cfg, R)
    value = cfg["T"] * world / (ms / 1e3)

    up_s = stages["up_gemm"] / 1e3
    dn_s = stages["down_gemm"] / 1e3
    peak_tf = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    up_tf = alg["up"] / up_s / 1e12
    kname = "up_gemm/%s" % (args.gemm or "auto")
    traffic, digest = recorded_traffic(args.workload, kname) if args.tokens is None and \
        args.experts is None else (None, None)
    roof = {"kernel": "up-projection grouped GEMM (SwiGLU epilogue)", "bound": "tensor",
            "achieved": round(up_tf, 1), "peak": peak_tf, "unit": "TFLOP/s",
            "frac": round(up_tf / peak_tf, 4), "traffic": traffic,
            "traffic_note": "ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, "
                            "profiles/traffic_%s.txt; null if the kernel sources changed "
                            "since (sources digest %s)" % (args.workload, digest),
            "peak_source": "%s bf16_tflops_sustained" % peak_src,
            "algorithmic_flop_per_launch": alg["up"], "launch_ms": round(stages["up_gemm"], 4),
            "frac_of_burst_peak": round(up_tf / peaks.get("bf16_tflops", 1816.0), 4)}
    gg_tf = (alg["up"] + alg["down"]) / (up_s + dn_s) / 1e12
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
        "grouped_gemm": {"tflops": round(gg_tf, 1), "frac_of_peak": round(gg_tf / peak_tf, 4),
                         "peak": peak_tf, "up_ms": round(stages["up_gemm"], 4),
                         "down_ms": round(stages["down_gemm"], 4)},
        "stage_ms": {k: round(v, 4) for k, v in stages.items()},
        "timing": "value from %d plain layer calls; stage_ms and the roofline's launch_ms from "
                  "%d more calls with CUDA events at the stage boundaries" % (args.steps, args.steps),
        "layer_tflops": round(alg["total"] / (ms / 1e3) / 1e12, 1),
        "gpu_launches": kernels_per_step(cfg) * args.steps,
        "pdl": os.environ.get("MOE_PDL", "1") != "0",
        "clocks": clk,
    }

    if not args.no_e2e:
        result["e2e"] = run_e2e(layer, cfg, x, args, world, dev)
    if not args.no_decode:
        result["decode"] = run_decode(args, bf16_inp, world, dev, peaks, peak_src)
        result["decode_fp8"] = run_decode(args, bf16_inp, world, dev, peaks, peak_src, low="fp8")
        result["decode_fp4"] = run_decode(args, bf16_inp, world, dev, peaks, peak_src, low="fp4")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(inp, cfg, args.cpu_seconds)
    del layer
    return result


def run_e2e(layer, cfg, x, args, world, dev):
    """Same metric through the public API with host buffers: every step copies
    its x from pinned host memory to the device, runs the layer and copies its
    y back to pinned host memory.  The copies run on their own streams with
    double-buffered device x / y, ordered by events, so step i+1's input copy
    and step i-1's output copy overlap step i's layer (the usual way to feed a
    layer from the host); the timed region spans all copies of all steps."""
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

    steps = max(10, args.steps // 4)
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
    counts = outputs["counts_kept"].cpu().numpy()
    hit = int((counts > 0).sum())
    # weight bytes per routed expert: codes (+ block scales) + fp32 row scales
    code_bytes = {None: 2.0, "fp8": 1.0, "fp4": 80.0 / 128.0}[low]
    per_expert = int(3 * cfg["d"] * cfg["F"] * code_bytes) + \
        (2 * cfg["F"] + cfg["d"]) * 4 * (low is not None)
    wbytes = hit * per_expert
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
            if g == "auto":
                os.environ.pop("MOE_GEMM_KERNEL", None)
            else:
                os.environ["MOE_GEMM_KERNEL"] = g
            layer = binding.MoeLayer(cfg, inp, device=dev)
            outputs = {"y": torch.empty_like(inp["x"]),
                       "counts_kept": torch.empty(cfg["E"], dtype=torch.int32, device=dev)}
            steps = max(10, min(args.steps, 50))
            ms, stages, _ = time_layer(layer, inp["x"], steps, args.warmup, world, outputs)
            R = int(outputs["counts_kept"].sum().item())
            hit = int((outputs["counts_kept"] > 0).sum().item())
            alg = algorithmic(cfg, R)
            gemm_ms = stages["up_gemm"] + stages["down_gemm"]
            entry[g] = {"ms": round(ms, 4), "tokens_per_s": round(T / (ms / 1e3), 1),
                        "gemm_ms": round(gemm_ms, 4),
                        "gemm_tflops": round((alg["up"] + alg["down"]) / (gemm_ms / 1e3) / 1e12, 1),
                        "weight_gbs": round(hit * per_expert / (gemm_ms / 1e3) / 1e9, 1)}
            del layer
        os.environ.pop("MOE_GEMM_KERNEL", None)
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
    if args.gemm:
        os.environ["MOE_GEMM_KERNEL"] = args.gemm
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
