"""GPU parity of the aux-loss backward through the router (router gradients
of grad_aux * aux) against the oracle's chain-rule gradient, which is itself
pinned to central finite differences on the CPU."""
import numpy as np
import pytest
import torch

import oracle
from helpers import f64, max_rel, small_cfg
from sparse_mixture_experts_59_b300 import binding, workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny_fp32", "mixtral_small", "sigmoid_shared_small",
                                  "fine_small", "switch_small"])
def test_aux_router_backward(name):
    cfg = small_cfg(name)
    inp_cpu = workloads.make_inputs(cfg, device="cpu")
    inp = workloads.to_device(inp_cpu, "cuda")
    layer = binding.MoeLayer(cfg, inp)
    out = layer.forward(inp["x"], want=("logits", "counts_pre"))
    g = binding.aux_loss_backward(cfg, inp["x"], inp["Wr"], out["logits"], out["counts_pre"],
                                  grad_aux=0.01)
    torch.cuda.synchronize()
    gl, gW, gx = oracle.aux_router_backward(inp_cpu["x"], inp_cpu["Wr"], f64(out["logits"]),
                                            out["counts_pre"].cpu().numpy(), grad_aux=0.01,
                                            scoring=cfg.get("scoring", "softmax"))
    assert max_rel(f64(g["grad_logits"]), gl) < 1e-5
    assert max_rel(f64(g["grad_Wr"]), gW) < 1e-4
    assert max_rel(f64(g["grad_x"]), gx) < 1e-4
