"""GPU parity of the FP8-expert-weight path (E4M3 codes with per-row fp32
scales) against the oracle, which decodes the same codes from the E4M3
definition and applies the scales in double.  Routing, counts and drops are
exact; slot outputs and layer outputs within the bf16 tolerance."""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_Y, f64, max_rel, moe_rel
from sparse_mixture_experts_59_b300 import binding, workloads

pytestmark = pytest.mark.gpu

CASES = {
    "swiglu_ragged": dict(base="mixtral_prefill", T=333, d=528, F=1392, seed=5001),
    "swiglu_decode": dict(base="mixtral_decode", T=5, d=256, F=384, seed=5002, weight_seed=5002),
    "gelu_capacity": dict(base="switch_skewed", T=512, d=256, F=512, E=16, k=1, seed=5003),
    "swiglu_k4": dict(base="mixtral_prefill", T=200, d=256, F=256, E=16, k=4, seed=5004),
    "dense_e1": dict(base="mixtral_prefill", T=40, d=256, F=256, E=1, k=1, seed=5010),
}


def _case(name):
    spec = dict(CASES[name])
    base = spec.pop("base")
    return workloads.config(base, **spec)


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_layer_matches_oracle(name):
    cfg = _case(name)
    inp_cpu = workloads.quantize_experts_fp8(workloads.make_inputs(cfg, device="cpu"))
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
    # slot outputs through the stage calls
    c = binding.make_config(inp_cpu["cfg"])
    ws = binding.new_workspace(c)
    ro = binding.route(c, inp["x"], inp["Wr"], inp.get("logit_bias"), ws=ws)
    do = binding.dispatch(c, ro["topk_idx"], ro["prob_mean"], ws=ws)
    Ys, _ = binding.expert_ffn(c, inp["x"], do["perm_src"], do["offsets"], ro["topk_w"], inp, ws=ws)
    torch.cuda.synchronize()
    kept = np.nonzero(ref["drop_mask"] == 0)[0]
    assert max_rel(f64(Ys)[kept], ref["slots"].reshape(-1, cfg["d"])[kept]) < TOL_Y["bf16"]


def test_fp8_full_size_decode_sampled():
    """The Mixtral-shaped decode layer (T=32, d=4096, d_ff=14336) with FP8
    expert weights: routing in full, outputs of two tokens against the oracle
    (which copies only those tokens' experts)."""
    cfg = workloads.config("mixtral_decode")
    inp = workloads.quantize_experts_fp8(workloads.make_inputs(cfg, device="cuda"))
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
