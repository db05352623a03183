"""GPU edge cases: tiny and ragged token counts, one expert, k = E, an
all-ties router, capacity 1, dispatch over many look-back blocks, bad expert
indices (reported as a device status; the context stays usable), bounded
waits that run out in dispatch and in each expert GEMM kernel (status
MOE_ERR_DEVICE_TIMEOUT, then a clean call), and guard regions around every
output buffer."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_AUX, TOL_Y, f64, max_rel, moe_rel
from sparse_mixture_experts_59_b300 import binding, workloads

pytestmark = pytest.mark.gpu


def _layer_vs_oracle(cfg, zero_router=False):
    inp_cpu = workloads.make_inputs(cfg, device="cpu")
    if zero_router:
        inp_cpu["Wr"] = torch.zeros_like(inp_cpu["Wr"])
    inp = workloads.to_device(inp_cpu, "cuda")
    layer = binding.MoeLayer(cfg, inp)
    out = layer.forward(inp["x"], want=("logits", "topk_idx", "drop_mask", "stats", "counts_kept"))
    torch.cuda.synchronize()
    assert binding.device_status(layer.ws) == 0
    ref = oracle.layer_forward(inp_cpu, logits_in=f64(out["logits"]))
    np.testing.assert_array_equal(out["topk_idx"].cpu().numpy(), ref["topk_idx"])
    np.testing.assert_array_equal(out["drop_mask"].cpu().numpy(), ref["drop_mask"])
    np.testing.assert_array_equal(out["counts_kept"].cpu().numpy(), ref["counts_kept"])
    assert max_rel(f64(out["y"]), ref["y"]) < TOL_Y[cfg["dtype"]]
    assert moe_rel(f64(out["y"]), ref["y"], f64(inp_cpu["x"]), cfg["dtype"]) < TOL_Y[cfg["dtype"]]
    return out, ref


@pytest.mark.parametrize("T,E,k", [(256, 8, 2), (257, 8, 2), (64, 32, 8), (65, 32, 8)],
                         ids=["one-launch-T256", "four-kernels-T257", "one-launch-TE2048",
                              "four-kernels-TE2080"])
def test_route_dispatch_at_the_one_launch_limits(T, E, k):
    """Decode-sized batches route and dispatch in one launch up to T = 256,
    T*k = 512, T*E = 2048; one token past a limit the four-kernel path takes
    over.  Both sides of each limit match the oracle, aux loss included."""
    cfg = workloads.config("mixtral_prefill", T=T, d=256, F=128, E=E, k=k, seed=3700 + T)
    out, ref = _layer_vs_oracle(cfg)
    aux = float(out["stats"][0].cpu())
    assert abs(aux - ref["aux"]) <= TOL_AUX * abs(ref["aux"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 7, 129])
def test_small_and_ragged_token_counts(T, dtype):
    cfg = workloads.config("mixtral_prefill", T=T, d=136, F=200, E=8, k=2, dtype=dtype, seed=3000 + T)
    _layer_vs_oracle(cfg)


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
def test_single_expert_is_dense_ffn(act):
    cfg = workloads.config("switch_skewed" if act == "gelu" else "mixtral_prefill", T=150, d=128,
                           F=256, E=1, k=1, capacity_factor=0.0, skew=False, seed=3100)
    out, ref = _layer_vs_oracle(cfg)
    assert np.all(out["topk_idx"].cpu().numpy() == 0)


def test_k_equals_E():
    cfg = workloads.config("mixtral_prefill", T=64, d=128, F=128, E=4, k=4, seed=3200)
    _layer_vs_oracle(cfg)


@pytest.mark.parametrize("cf", [0.0, 1.0, 0.3])
def test_all_ties_router_takes_lowest_experts(cf):
    """Wr = 0: every token picks experts 0..k-1, aux = k, and with a capacity
    the tokens past it keep y = x."""
    cfg = workloads.config("tiny_fp32", T=200, E=8, k=2, dtype="bf16", capacity_factor=cf, seed=3300)
    out, ref = _layer_vs_oracle(cfg, zero_router=True)
    assert np.all(out["topk_idx"].cpu().numpy() == np.arange(2)[None, :])
    assert float(out["stats"][0]) == pytest.approx(2.0, rel=1e-6)


def test_capacity_one():
    cfg = workloads.config("switch_skewed", T=100, d=64, F=128, E=64, k=1, capacity_factor=0.01,
                           seed=3400)
    out, ref = _layer_vs_oracle(cfg)
    assert ref["cap"] == 1
    assert int(out["counts_kept"].max()) <= 1


@pytest.mark.parametrize("A,E,k,cap", [(70001 * 1, 64, 1, -1), (40000 * 2, 256, 2, 300),
                                       (2049, 3, 1, 100), (65536, 256, 8, -1)])
def test_dispatch_many_blocks(A, E, k, cap):
    """Dispatch over many decoupled look-back blocks, with skewed expert
    choices, against the oracle bit for bit."""
    T = A // k
    g = np.random.default_rng(A + E)
    # Zipf-like skew: low expert ids much more frequent; distinct per token
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    idx = np.stack([g.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    cf = 0.0 if cap < 0 else cap * E / (T * k) + 1e-9
    cfg = workloads.config("mixtral_prefill", T=T, d=64, F=64, E=E, k=k, capacity_factor=cf)
    c = binding.make_config(cfg)
    want_cap = binding.capacity(c)
    ref = oracle.dispatch(idx, E, want_cap)
    do = binding.dispatch(c, torch.from_numpy(idx).cuda())
    torch.cuda.synchronize()
    for key in ("counts_pre", "counts_kept", "offsets", "dest", "drop_mask"):
        np.testing.assert_array_equal(do[key].cpu().numpy()[:len(ref[key])], ref[key], err_msg=key)
    np.testing.assert_array_equal(do["perm_src"].cpu().numpy()[:ref["R"]], ref["perm_src"])
    # again on the same workspace (the look-back state must have been cleared)
    ws = binding.new_workspace(c)
    for _ in range(2):
        do = binding.dispatch(c, torch.from_numpy(idx).cuda(), ws=ws)
        np.testing.assert_array_equal(do["dest"].cpu().numpy(), ref["dest"])
    assert binding.device_status(ws) == 0


def test_out_of_range_expert_index_is_reported():
    """A corrupted top-k index is left out of every count and reported as
    MOE_ERR_DEVICE_BOUNDS; the next call on a re-initialised workspace works."""
    cfg = workloads.config("mixtral_prefill", T=300, d=64, F=64, E=8, k=2)
    c = binding.make_config(cfg)
    idx = torch.randint(0, 8, (300, 2), dtype=torch.int32)
    idx[:, 1] = (idx[:, 0] + 1) % 8
    bad = idx.clone()
    bad[17, 0] = 8
    bad[200, 1] = -3
    ws = binding.new_workspace(c)
    do = binding.dispatch(c, bad.cuda(), ws=ws)
    assert binding.device_status(ws) == 6          # MOE_ERR_DEVICE_BOUNDS
    assert int(do["counts_pre"].sum()) == 600 - 2
    ws = binding.new_workspace(c)
    do = binding.dispatch(c, idx.cuda(), ws=ws)
    ref = oracle.dispatch(idx.numpy(), 8, -1)
    np.testing.assert_array_equal(do["dest"].cpu().numpy(), ref["dest"])
    assert binding.device_status(ws) == 0


def test_lookback_wait_times_out_and_reports():
    """Failure path of dispatch's bounded waits: with one look-back block held
    back (its flag is never set), the blocks after it give up after about a
    second, the device status reads MOE_ERR_DEVICE_TIMEOUT, and the context
    stays usable for the next call."""
    import time
    cfg = workloads.config("mixtral_prefill", T=2048, d=64, F=64, E=8, k=2)   # 8 blocks
    c = binding.make_config(cfg)
    g = torch.Generator().manual_seed(9)
    idx = torch.stack([torch.randperm(8, generator=g)[:2] for _ in range(2048)]).to(torch.int32)
    ws = binding.new_workspace(c)
    binding.test_hold_lookback_block(ws, 2)
    t0 = time.time()
    binding.dispatch(c, idx.cuda(), ws=ws)
    status = binding.device_status(ws)
    assert status == 5                                 # MOE_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 60
    ws = binding.new_workspace(c)
    do = binding.dispatch(c, idx.cuda(), ws=ws)
    ref = oracle.dispatch(idx.numpy(), 8, -1)
    np.testing.assert_array_equal(do["dest"].cpu().numpy(), ref["dest"])
    assert binding.device_status(ws) == 0


@pytest.mark.parametrize("kern,low,hold", [("tc1", None, 0), ("tc1", None, 5), ("pair", None, 0),
                                           ("pair", None, 5), ("swap", None, 0), ("swap", None, 5),
                                           ("auto", "fp8", 0), ("auto", "fp8", 3),
                                           ("auto", "fp4", 3)])
def test_gemm_wait_times_out_and_reports(kern, low, hold):
    """Failure path of the expert GEMMs' bounded waits: with the up-projection's
    weight producer stopped before ring iteration `hold` (the copy never
    arrives), the MMA issuer (low-bit weights: the converters) gives up after about a
    second, the device status reads MOE_ERR_DEVICE_TIMEOUT, the kernel drains
    its own copies and MMAs, frees its tensor memory and returns, and a clean
    call on a fresh workspace reproduces the earlier output bit for bit.
    d = 1024 gives every CTA with a tile 16 K blocks, so iteration 5 falls
    inside the first tile (after loads and MMAs are in flight)."""
    import time
    cfg = workloads.config("mixtral_prefill", T=300, d=1024, F=384, E=4, k=2, seed=77,
                           gemm_kernel=kern)
    inp = workloads.make_inputs(cfg, device="cuda")
    if low == "fp8":
        inp = workloads.quantize_experts_fp8(inp)
        cfg = inp["cfg"]
    elif low == "fp4":
        inp = workloads.quantize_experts_fp4(inp)
        cfg = inp["cfg"]
    layer = binding.MoeLayer(cfg, inp)
    ref = layer.forward(inp["x"])["y"].clone()
    assert binding.device_status(layer.ws) == 0
    binding.test_hold_gemm_stage(layer.ws, hold)
    t0 = time.time()
    layer.forward(inp["x"])
    assert binding.device_status(layer.ws) == 5        # MOE_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 60
    layer.ws = binding.new_workspace(layer.c)
    y = layer.forward(inp["x"])["y"]
    assert binding.device_status(layer.ws) == 0
    assert torch.equal(y, ref)


GUARD = 4096            # guard bytes before and after each output


def _guarded(shape, dtype, fill=0):
    """A tensor of `shape` inside a larger byte buffer whose GUARD bytes before
    and after it hold 0xA5, so a write past either end shows.  Returns (view,
    check) where check() asserts that both guards are intact."""
    n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
    raw = torch.full((GUARD + n + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    view = raw[GUARD:GUARD + n].view(dtype).view(*shape)
    view.fill_(fill)

    def check():
        torch.cuda.synchronize()
        assert bool((raw[:GUARD] == 0xA5).all()), "guard before the buffer overwritten"
        assert bool((raw[GUARD + n:] == 0xA5).all()), "guard after the buffer overwritten"
    return view, check


@pytest.mark.parametrize("kern", ["tc1", "pair", "swap"])
@pytest.mark.parametrize("name,over", [("mixtral_prefill", dict(T=129, d=264, F=392, E=6, k=2)),
                                       ("fine_grained", dict(T=77, d=192, F=136, E=16, k=4,
                                                             F_shared=72)),
                                       ("switch_skewed", dict(T=300, d=128, F=264, E=8, k=1))])
def test_outputs_stay_inside_their_buffers(name, over, kern):
    """Canary check: every output of the layer call and of the four stage calls
    sits between guard regions; ragged shapes (T, d, F and segment lengths off
    every tile size) must leave the guards untouched."""
    cfg = workloads.config(name, seed=321, gemm_kernel=kern, **over)
    inp = workloads.make_inputs(cfg, device="cuda")
    T, d, E, k = cfg["T"], cfg["d"], cfg["E"], cfg["k"]
    A = T * k
    dt = inp["x"].dtype
    i32, f32, u8 = torch.int32, torch.float32, torch.uint8
    outs, checks = {}, []
    for key, shape, t in (("y", (T, d), dt), ("logits", (T, E), f32), ("topk_idx", (T, k), i32),
                          ("topk_w", (T, k), f32), ("counts_pre", (E,), i32),
                          ("counts_kept", (E,), i32), ("drop_mask", (A,), u8), ("stats", (2,), f32)):
        outs[key], chk = _guarded(shape, t)
        checks.append(chk)
    layer = binding.MoeLayer(cfg, inp)
    layer.forward(inp["x"], outputs=outs)
    assert binding.device_status(layer.ws) == 0
    for chk in checks:
        chk()
    # the stage calls, each output guarded
    c = binding.make_config(cfg)
    ws = binding.new_workspace(c)
    ro = binding.route(c, inp["x"], inp["Wr"], inp.get("logit_bias"), ws=ws)
    do = binding.dispatch(c, ro["topk_idx"], ro["prob_mean"], ws=ws)
    Ys, chk_ys = _guarded((A, d), dt)
    Sh, chk_sh = (_guarded((T, d), dt) if cfg.get("F_shared") else (None, None))
    w = binding._weights_struct(inp)
    binding._check(binding.lib().moe_expert_ffn(
        ctypes.byref(c), binding._p(inp["x"]), binding._p(do["perm_src"]), binding._p(do["offsets"]),
        binding._p(ro["topk_w"]), ctypes.byref(w), binding._p(Ys), binding._p(Sh), binding._p(ws),
        ws.numel(), binding._stream()))
    y2, chk_y2 = _guarded((T, d), dt)
    binding._check(binding.lib().moe_combine(
        ctypes.byref(c), binding._p(inp["x"]), binding._p(Ys), binding._p(do["drop_mask"]),
        binding._p(Sh), binding._p(y2), binding._stream()))
    assert binding.device_status(ws) == 0
    chk_ys()
    chk_y2()
    if chk_sh:
        chk_sh()
    assert torch.equal(y2, outs["y"])
