"""GPU parity of the whole path against the CPU oracle, element by element, on
scaled-down copies of each workload (sizes that span several tiles and leave
ragged row, column and reduction tails).  Calls go through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from helpers import (MARGIN, moe_rel, SMALL, TOL_AUX, TOL_LOGITS, TOL_W, TOL_Y, f64, margins, max_rel,
                     small_cfg, to_cpu)
from sparse_mixture_experts_59_b300 import binding, workloads

pytestmark = pytest.mark.gpu
WANT = ("logits", "topk_idx", "topk_w", "counts_pre", "counts_kept", "drop_mask", "stats")


def _params():
    """Each small workload with the library's own GEMM choice, and the bf16
    ones again with each tensor-core GEMM kernel forced (1-SM tokens-on-M,
    2-SM tokens-on-M, 2-SM weights-on-M)."""
    out = list(SMALL)
    for kern in ("tc1", "pair", "swap"):
        out += [n + "@" + kern for n in SMALL if small_cfg(n)["dtype"] == "bf16"]
    return out


@pytest.fixture(scope="module", params=_params())
def run(request):
    name, _, kern = request.param.partition("@")
    return _run(name, kern or "auto")


def _run(name, kern="auto"):
    cfg = small_cfg(name)
    cfg["gemm_kernel"] = kern
    inp_cpu = workloads.make_inputs(cfg, device="cpu")
    inp = workloads.to_device(inp_cpu, "cuda")
    layer = binding.MoeLayer(cfg, inp)
    out = layer.forward(inp["x"], want=WANT)
    torch.cuda.synchronize()
    assert binding.device_status(layer.ws) == 0
    gpu = {k: v.cpu() for k, v in out.items()}
    # the oracle routes on the GPU's fp32 logits so that routing is identical
    ref = oracle.layer_forward(inp_cpu, logits_in=f64(gpu["logits"]))
    return dict(cfg=cfg, inp_cpu=inp_cpu, inp=inp, layer=layer, gpu=gpu, ref=ref)


def test_routing_indices_bit_exact(run):
    g, r = run["gpu"], run["ref"]
    np.testing.assert_array_equal(g["topk_idx"].numpy(), r["topk_idx"])


def test_gate_weights(run):
    g, r = run["gpu"], run["ref"]
    assert max_rel(f64(g["topk_w"]), r["topk_w"]) < TOL_W
    if run["cfg"].get("renorm", True):
        np.testing.assert_allclose(f64(g["topk_w"]).sum(axis=1), 1.0, atol=1e-6)


def test_router_logits_against_own_oracle_logits(run):
    cfg, inp, g = run["cfg"], run["inp_cpu"], run["gpu"]
    own = oracle.router_logits(inp["x"], inp["Wr"], inp.get("logit_bias"))
    assert max_rel(f64(g["logits"]), own) < TOL_LOGITS[cfg["dtype"]]
    idx_own, _, _ = oracle.topk(own, cfg["k"])
    clear = margins(own, cfg["k"]) >= MARGIN
    np.testing.assert_array_equal(g["topk_idx"].numpy()[clear], idx_own[clear])


def test_counts_and_drops_bit_exact(run):
    g, r = run["gpu"], run["ref"]
    np.testing.assert_array_equal(g["counts_pre"].numpy(), r["counts_pre"])
    np.testing.assert_array_equal(g["counts_kept"].numpy(), r["counts_kept"])
    np.testing.assert_array_equal(g["drop_mask"].numpy(), r["drop_mask"])


def test_aux_loss_and_drop_fraction(run):
    g, r = run["gpu"], run["ref"]
    stats = g["stats"].numpy().astype(np.float64)
    assert abs(stats[0] - r["aux"]) <= TOL_AUX * abs(r["aux"])
    assert stats[1] == pytest.approx(r["drop_frac"], abs=1e-7)


def test_layer_output(run):
    cfg, g, r, inp = run["cfg"], run["gpu"], run["ref"], run["inp_cpu"]
    y = f64(g["y"])
    x = f64(inp["x"])
    tol = TOL_Y[cfg["dtype"]]
    assert max_rel(y, r["y"]) < tol
    assert moe_rel(y, r["y"], x, cfg["dtype"]) < tol
    # tokens whose every slot was dropped come back unchanged
    T, k = cfg["T"], cfg["k"]
    full_drop = r["drop_mask"].reshape(T, k).all(axis=1)
    if full_drop.any() and not cfg.get("F_shared"):
        fd = torch.from_numpy(full_drop)
        assert torch.equal(g["y"][fd], inp["x"][fd])


def test_stage_calls_match_layer_forward(run):
    """moe_route -> moe_dispatch -> moe_expert_ffn -> moe_combine give the same
    bits as moe_layer_forward, and the standalone dispatch's permutation is
    the oracle's."""
    cfg, inp, g, r = run["cfg"], run["inp"], run["gpu"], run["ref"]
    c = binding.make_config(cfg)
    ws = binding.new_workspace(c)
    ro = binding.route(c, inp["x"], inp["Wr"], inp.get("logit_bias"), ws=ws)
    do = binding.dispatch(c, ro["topk_idx"], ro["prob_mean"], ws=ws)
    Ys, Sh = binding.expert_ffn(c, inp["x"], do["perm_src"], do["offsets"], ro["topk_w"], inp, ws=ws)
    y = binding.combine(c, inp["x"], Ys, do["drop_mask"], Sh)
    torch.cuda.synchronize()
    assert binding.device_status(ws) == 0
    assert torch.equal(ro["logits"].cpu(), g["logits"])
    assert torch.equal(y.cpu(), g["y"])
    R = r["R"]
    np.testing.assert_array_equal(do["offsets"].cpu().numpy(), r["offsets"])
    np.testing.assert_array_equal(do["perm_src"].cpu().numpy()[:R], r["perm_src"])
    np.testing.assert_array_equal(do["dest"].cpu().numpy(), r["dest"])
    # prob_mean and the slot outputs
    P = r["probs"].mean(axis=0)
    assert max_rel(f64(ro["prob_mean"]), P) < TOL_W
    slots = oracle.layer_tokens(run["inp_cpu"], r["topk_idx"], r["topk_w"], r["drop_mask"],
                                np.arange(cfg["T"]), want_slots=True)["slots"]
    kept = np.nonzero(r["drop_mask"] == 0)[0]
    Ys_k = f64(Ys)[kept]
    ref_k = slots.reshape(-1, cfg["d"])[kept]
    assert max_rel(Ys_k, ref_k) < TOL_Y[cfg["dtype"]]


def test_repeatable(run):
    """Two calls give identical bits (no float atomics on the data path)."""
    out = run["layer"].forward(run["inp"]["x"], want=("logits",))
    torch.cuda.synchronize()
    assert torch.equal(out["y"].cpu(), run["gpu"]["y"])
