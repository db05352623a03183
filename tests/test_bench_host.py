"""Host-side arithmetic of bench.py, on CPU: the algorithmic work its
roofline divides by, and the kernel launches it claims per step.  The flop
counts are checked against the workloads' published totals (the Mixtral
prefill layer is 2.886e12 flop with its router; the fine-grained layer
6.524e12) and against a count of multiply-adds written out per expert."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_mixture_experts_59_b300 import workloads  # noqa: E402


def _macs_by_expert(cfg, rows_per_expert):
    """Multiply-adds counted expert by expert: each kept row of an expert
    multiplies d inputs by F outputs in the up projection (twice for SwiGLU's
    gate and up), F by d in the down projection; the shared expert does the
    same for all T tokens; the router d by E per token."""
    d, F, E, T = cfg["d"], cfg["F"], cfg["E"], cfg["T"]
    Fs = cfg.get("F_shared", 0) or 0
    gates = 2 if cfg["act"] == "swiglu" else 1
    up = sum(r * d * F * gates for r in rows_per_expert)
    down = sum(r * F * d for r in rows_per_expert)
    up += T * d * Fs * 2          # shared expert is SwiGLU
    down += T * Fs * d
    return up, down, T * d * E


@pytest.mark.parametrize("name", ["mixtral_prefill", "mixtral_decode", "fine_grained",
                                  "switch_skewed", "tiny_fp32"])
def test_algorithmic_flops_are_twice_the_macs(name):
    cfg = workloads.config(name)
    A = cfg["T"] * cfg["k"]
    rows = [A // cfg["E"]] * cfg["E"]          # any split of the kept rows
    rows[0] += A - sum(rows)
    up, down, router = _macs_by_expert(cfg, rows)
    alg = bench.algorithmic(cfg, sum(rows))
    assert alg["up"] == 2 * up
    assert alg["down"] == 2 * down
    assert alg["router"] == 2 * router
    assert alg["total"] == 2 * (up + down + router)


def test_published_totals():
    """Mixtral prefill: 2.886e12 flop in the experts and router; the
    fine-grained layer with its shared expert: 6.524e12."""
    c1 = workloads.config("mixtral_prefill")
    assert bench.algorithmic(c1, c1["T"] * c1["k"])["total"] == pytest.approx(2.886e12, rel=1e-3)
    c3 = workloads.config("fine_grained")
    assert bench.algorithmic(c3, c3["T"] * c3["k"])["total"] == pytest.approx(6.524e12, rel=1e-3)


@pytest.mark.parametrize("name,launches", [("mixtral_prefill", 8), ("mixtral_decode", 5),
                                           ("fine_grained", 8), ("switch_skewed", 8),
                                           ("tiny_fp32", 5)])
def test_kernel_launches_per_step(name, launches):
    """Decode-sized batches route and dispatch in one launch; larger ones in
    four.  Then gather, up, down, combine."""
    assert bench.kernels_per_step(workloads.config(name)) == launches


def test_weight_bytes_of_the_decode_layers():
    """Bytes streamed when all 8 Mixtral experts are hit: 3 bf16 matrices of
    4096 x 14336 each (352 MB per expert); E4M3 codes are one byte each plus
    fp32 row scales (2F + d per expert); packed 4-bit rows are 80 bytes per
    128 values plus the same row scales."""
    cfg = workloads.config("mixtral_decode")
    d, F = cfg["d"], cfg["F"]
    counts = [4] * 8
    assert bench.weight_bytes(cfg, counts) == (8 * 3 * d * F * 2, 8)
    c8 = dict(cfg, weight_fp8=True)
    assert bench.weight_bytes(c8, counts)[0] == 8 * (3 * d * F + (2 * F + d) * 4)
    c4 = dict(cfg, weight_fp4=True)
    assert bench.weight_bytes(c4, counts)[0] == 8 * (3 * d * F // 128 * 80 + (2 * F + d) * 4)
    # experts without kept rows stream nothing; the shared expert always streams
    c3 = workloads.config("fine_grained")
    got, hit = bench.weight_bytes(c3, [0, 3] + [0] * 254)
    assert hit == 1 and got == 3 * 7168 * 2048 * 2 * 2
    # fp32 GELU experts with biases
    c0 = workloads.config("tiny_fp32")
    assert bench.weight_bytes(c0, [1] * 8)[0] == 8 * (2 * 128 * 256 + 256 + 128) * 4


def test_gemm_roofline_takes_the_slower_roof():
    peaks = {"bf16_tflops": 1000.0, "hbm_gbs": 5000.0}
    alg = {"up": 2e12, "down": 1e12}
    r = bench.gemm_roofline(alg, 5e9, 4e-3, peaks)         # 3 ms of flop, 1 ms of bytes
    assert r["bound"] == "tensor" and r["roofline_ms"] == pytest.approx(3.0)
    assert r["frac"] == pytest.approx(0.75)
    r = bench.gemm_roofline(alg, 25e9, 10e-3, peaks)       # 5 ms of bytes
    assert r["bound"] == "hbm" and r["frac"] == pytest.approx(0.5)


def test_tensor_peak_follows_the_timed_region():
    """A short pass at full clock is judged against the burst peak; a long pass,
    or one whose clock sat well below its maximum (the power cap), against the
    sustained peak."""
    full = {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0}
    capped = {"sm_mhz": 1342.0, "sm_max_mhz": 2032.0}
    assert bench.pick_tensor_peak(1772.9, 1366.0, 40.0, full)[0] == 1772.9
    assert bench.pick_tensor_peak(1772.9, 1366.0, 497.0, full)[0] == 1366.0
    assert bench.pick_tensor_peak(1772.9, 1366.0, 40.0, capped)[0] == 1366.0
    assert bench.pick_tensor_peak(1772.9, 1366.0, 40.0, None)[0] == 1772.9
    assert bench.pick_tensor_peak(1772.9, 1366.0, 40.0, {"error": "no samples"})[0] == 1772.9


def test_recorded_traffic_needs_the_digest_it_was_taken_on(tmp_path, monkeypatch):
    """The DRAM-traffic figure in a profile is reported only while the GEMM
    kernel sources hash to the digest recorded beside it. After an edit the
    figure is withheld (None), and so is one for a kernel the file does not
    list."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic_demo.txt").write_text(
        "# header line\ntraffic up_gemm/swap 123456 abcdef0123456789\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_sources_digest", lambda: "abcdef0123456789")
    assert bench.recorded_traffic("demo", "up_gemm/swap") == (123456, "abcdef0123456789")
    assert bench.recorded_traffic("demo", "up_gemm/tc1")[0] is None
    assert bench.recorded_traffic("other", "up_gemm/swap") == (None, None)
    monkeypatch.setattr(bench, "kernel_sources_digest", lambda: "0000000000000000")
    assert bench.recorded_traffic("demo", "up_gemm/swap") == (None, "0000000000000000")



def test_clock_records_that_disqualify_a_pass():
    """A hardware or thermal slowdown, or a clock held well below its maximum
    with no reason given, sends the pass to be taken again. The power cap
    alone, a full clock, or a record with no samples does not."""
    ok = {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": []}
    capped = {"sm_mhz": 1320.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"]}
    assert bench.clock_rejection(ok) is None
    assert bench.clock_rejection(capped) is None
    assert bench.clock_rejection(None) is None
    assert bench.clock_rejection({"error": "no samples"}) is None
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        why = bench.clock_rejection(dict(ok, reasons=["sw_power_cap", r]))
        assert why is not None and r in why
    locked = {"sm_mhz": 1400.0, "sm_max_mhz": 2032.0, "reasons": []}
    assert "no reason" in bench.clock_rejection(locked)
    assert bench.clock_rejection(dict(locked, sm_mhz=1900.0)) is None
