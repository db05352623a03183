"""GPU parity of the packed 4-bit expert-weight path (E2M1 codes, E4M3 scales
per 16 values, fp32 row scales) against the oracle, which decodes the same
bytes from the E2M1 and E4M3 definitions and applies the scales in double.
Routing, counts and drops are exact; slot outputs and layer outputs within
the bf16 tolerance."""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_Y, f64, max_rel, moe_rel
from sparse_mixture_experts_59_b300 import binding, workloads

pytestmark = pytest.mark.gpu

# d and F are multiples of 128 (one 80-byte chunk per 128 values)
CASES = {
    "swiglu_ragged": dict(base="mixtral_prefill", T=333, d=512, F=1408, seed=6001),
    "swiglu_decode": dict(base="mixtral_decode", T=5, d=256, F=384, seed=6002, weight_seed=6002),
    "gelu_capacity": dict(base="switch_skewed", T=512, d=256, F=512, E=16, k=1, seed=6003),
    "swiglu_k4": dict(base="mixtral_prefill", T=200, d=384, F=256, E=16, k=4, seed=6004),
    "one_token": dict(base="mixtral_decode", T=1, d=128, F=128, E=8, k=2, seed=6005),
    "dense_e1": dict(base="mixtral_prefill", T=40, d=256, F=256, E=1, k=1, seed=6010),
}


def _case(name):
    spec = dict(CASES[name])
    base = spec.pop("base")
    return workloads.config(base, **spec)


@pytest.mark.parametrize("name", list(CASES))
def test_fp4_layer_matches_oracle(name):
    cfg = _case(name)
    inp_cpu = workloads.quantize_experts_fp4(workloads.make_inputs(cfg, device="cpu"))
    inp = workloads.to_device(inp_cpu, "cuda")
    layer = binding.MoeLayer(inp_cpu["cfg"], inp)
    out = layer.forward(inp["x"], want=("logits", "topk_idx", "topk_w", "drop_mask", "counts_kept"))
    torch.cuda.synchronize()
    assert binding.device_status(layer.ws) == 0
    ref = oracle.layer_forward(inp_cpu, logits_in=f64(out["logits"]), want_slots=True)
    np.testing.assert_array_equal(out["topk_idx"].cpu().numpy(), ref["topk_idx"])
    np.testing.assert_array_equal(out["drop_mask"].cpu().numpy(), ref["drop_mask"])
    np.testing.assert_array_equal(out["counts_kept"].cpu().numpy(), ref["counts_kept"])
    x = f64(inp_cpu["x"])
    assert max_rel(f64(out["y"]), ref["y"]) < TOL_Y["bf16"]
    assert moe_rel(f64(out["y"]), ref["y"], x, "bf16") < TOL_Y["bf16"]
    c = binding.make_config(inp_cpu["cfg"])
    ws = binding.new_workspace(c)
    ro = binding.route(c, inp["x"], inp["Wr"], inp.get("logit_bias"), ws=ws)
    do = binding.dispatch(c, ro["topk_idx"], ro["prob_mean"], ws=ws)
    Ys, _ = binding.expert_ffn(c, inp["x"], do["perm_src"], do["offsets"], ro["topk_w"], inp, ws=ws)
    torch.cuda.synchronize()
    kept = np.nonzero(ref["drop_mask"] == 0)[0]
    assert max_rel(f64(Ys)[kept], ref["slots"].reshape(-1, cfg["d"])[kept]) < TOL_Y["bf16"]


def test_fp4_single_nibble_positions():
    """Each weight row holds one nonzero value at a chosen position, so a
    swapped nibble order or block-scale index moves the output to another
    column: the slot outputs must match the oracle exactly in position."""
    cfg = workloads.config("mixtral_decode", T=4, d=256, F=256, E=8, k=2, seed=6006, weight_seed=6006)
    inp_cpu = workloads.make_inputs(cfg, device="cpu")
    g = torch.Generator().manual_seed(6006)
    for key in ("W1", "W3", "W2"):
        w = inp_cpu[key]
        E, R, K = w.shape
        pos = torch.randint(0, K, (E, R), generator=g)
        val = torch.randn(E, R, generator=g)
        z = torch.zeros(E, R, K, dtype=w.dtype)
        z.scatter_(2, pos[..., None], val[..., None].to(w.dtype))
        inp_cpu[key] = z
    inp_cpu = workloads.quantize_experts_fp4(inp_cpu)
    inp = workloads.to_device(inp_cpu, "cuda")
    layer = binding.MoeLayer(inp_cpu["cfg"], inp)
    out = layer.forward(inp["x"], want=("logits",))
    torch.cuda.synchronize()
    assert binding.device_status(layer.ws) == 0
    ref = oracle.layer_forward(inp_cpu, logits_in=f64(out["logits"]))
    x = f64(inp_cpu["x"])
    assert moe_rel(f64(out["y"]), ref["y"], x, "bf16") < TOL_Y["bf16"]
    assert max_rel(f64(out["y"]) - x, ref["y"] - x) < 4 * TOL_Y["bf16"]


def test_fp4_full_size_decode_sampled():
    """The Mixtral-shaped decode layer (T=32, d=4096, d_ff=14336) with packed
    4-bit expert weights: routing in full, outputs of two tokens against the
    oracle (which copies only those tokens' experts)."""
    cfg = workloads.config("mixtral_decode")
    inp = workloads.quantize_experts_fp4(workloads.make_inputs(cfg, device="cuda"))
    layer = binding.MoeLayer(inp["cfg"], inp)
    out = layer.forward(inp["x"], want=("logits", "topk_idx", "topk_w", "drop_mask"))
    torch.cuda.synchronize()
    assert binding.device_status(layer.ws) == 0
    idx, w, _ = oracle.topk(f64(out["logits"]), cfg["k"])
    np.testing.assert_array_equal(out["topk_idx"].cpu().numpy(), idx)
    tokens = [3, 17]
    used = sorted(set(int(e) for t in tokens for e in idx[t]))
    pos = {e: i for i, e in enumerate(used)}
    sel = torch.tensor(used, device="cuda")
    sub = dict(cfg=dict(inp["cfg"], T=len(tokens), E=len(used)))
    sub["x"] = inp["x"][tokens].cpu()
    for key in ("W1", "W3", "W2", "s1", "s3", "s2"):
        sub[key] = inp[key].index_select(0, sel).cpu()
    sidx = np.array([[pos[int(e)] for e in idx[t]] for t in tokens], np.int32)
    ref = oracle.layer_tokens(sub, sidx, f64(out["topk_w"])[tokens],
                              np.zeros(len(tokens) * cfg["k"], np.uint8), np.arange(len(tokens)))["y"]
    y = f64(out["y"])[tokens]
    assert max_rel(y, ref) < TOL_Y["bf16"]
    assert moe_rel(y, ref, f64(sub["x"]), "bf16") < TOL_Y["bf16"]
