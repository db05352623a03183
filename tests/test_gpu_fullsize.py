"""GPU parity at the full workload sizes, in the launch configuration the bench
times.  Integer outputs (routing, counts, permutation, drops) are compared in
full; the aux loss in full; router logits on sampled tokens; layer outputs on
a stratified sample of tokens that reaches every tile the expert GEMMs
compute: for every expert segment its first and last row and a row in each
128-row tile (the token tiles of every GEMM kernel are 128 rows or multiples
of them, and each sampled token's output covers all output columns), plus
fully dropped tokens where there are any.  The oracle computes the sampled
tokens one by one from copies of just the experts they use."""
import numpy as np
import pytest
import torch

import oracle
from helpers import MARGIN, moe_rel, TOL_AUX, TOL_LOGITS, TOL_W, TOL_Y, f64, margins, max_rel
from sparse_mixture_experts_59_b300 import binding, workloads

pytestmark = pytest.mark.gpu
WANT = ("logits", "topk_idx", "topk_w", "counts_pre", "counts_kept", "drop_mask", "stats")
TILE_ROWS = 128
DROPPED_SAMPLES = 8


def _subset_inputs(inp, cfg, tokens, idx, drop):
    """CPU copy of x[tokens] and of the experts those tokens keep, with the
    routing remapped to the copied experts."""
    k = cfg["k"]
    used = sorted(set(int(e) for t in tokens for s in range(k) if not drop[t * k + s]
                      for e in [idx[t, s]]))
    if not used:
        used = [0]
    pos = {e: i for i, e in enumerate(used)}
    sel = torch.tensor(used, dtype=torch.long, device=inp["W1"].device)
    sub = dict(cfg=dict(cfg, T=len(tokens), E=len(used)))
    tok = torch.tensor(tokens, dtype=torch.long, device=inp["x"].device)
    sub["x"] = inp["x"].index_select(0, tok).cpu()
    for key in ("W1", "W3", "W2", "b1", "b2"):
        sub[key] = None if inp.get(key) is None else inp[key].index_select(0, sel).cpu()
    for key in ("S1", "S3", "S2"):
        sub[key] = None if inp.get(key) is None else inp[key].cpu()
    sidx = np.array([[pos.get(int(idx[t, s]), 0) for s in range(k)] for t in tokens], np.int32)
    sdrop = np.array([drop[t * k + s] for t in tokens for s in range(k)], np.uint8)
    return sub, sidx, sdrop


@pytest.fixture(scope="module", params=["mixtral_prefill", "mixtral_decode", "fine_grained",
                                                "switch_skewed"])
def full(request):
    name = request.param
    cfg = workloads.config(name)
    inp = workloads.make_inputs(cfg, device="cuda")
    layer = binding.MoeLayer(cfg, inp)
    out = layer.forward(inp["x"], want=WANT)
    torch.cuda.synchronize()
    status = binding.device_status(layer.ws)
    gpu = {k: v.cpu() for k, v in out.items() if k != "y"}
    res = dict(name=name, cfg=cfg, inp=inp, out=out, gpu=gpu, status=status)
    yield res
    del layer, inp, out
    torch.cuda.empty_cache()


def test_full_size_routing_dispatch_aux(full):
    cfg, g = full["cfg"], full["gpu"]
    assert full["status"] == 0
    T, E, k = cfg["T"], cfg["E"], cfg["k"]
    idx, w, probs = oracle.topk(f64(g["logits"]), k)
    np.testing.assert_array_equal(g["topk_idx"].numpy(), idx)
    assert max_rel(f64(g["topk_w"]), w) < TOL_W
    cap = oracle.capacity(T, k, E, cfg["capacity_factor"])
    disp = oracle.dispatch(idx, E, cap)
    np.testing.assert_array_equal(g["counts_pre"].numpy(), disp["counts_pre"])
    np.testing.assert_array_equal(g["counts_kept"].numpy(), disp["counts_kept"])
    np.testing.assert_array_equal(g["drop_mask"].numpy(), disp["drop_mask"])
    aux = oracle.aux_loss(disp["counts_pre"], probs)
    assert abs(float(g["stats"][0]) - aux) <= TOL_AUX * abs(aux)
    A = T * k
    assert float(g["stats"][1]) == pytest.approx((A - disp["R"]) / A, abs=1e-6)
    # standalone dispatch on the same indices: the permutation itself
    c = binding.make_config(cfg)
    do = binding.dispatch(c, full["out"]["topk_idx"])
    np.testing.assert_array_equal(do["dest"].cpu().numpy(), disp["dest"])
    np.testing.assert_array_equal(do["perm_src"].cpu().numpy()[:disp["R"]], disp["perm_src"])


def test_full_size_sampled_logits(full):
    cfg, g, inp = full["cfg"], full["gpu"], full["inp"]
    rng = np.random.default_rng(11)
    tokens = np.sort(rng.choice(cfg["T"], size=min(64, cfg["T"]), replace=False)).astype(np.int32)
    tok = torch.from_numpy(tokens).long().cuda()
    x_s = inp["x"].index_select(0, tok).cpu()
    own = oracle.router_logits(x_s, inp["Wr"].cpu(),
                               None if inp.get("logit_bias") is None else inp["logit_bias"].cpu())
    gl = f64(g["logits"])[tokens]
    assert max_rel(gl, own) < TOL_LOGITS[cfg["dtype"]]
    idx_own, _, _ = oracle.topk(own, cfg["k"])
    clear = margins(own, cfg["k"]) >= MARGIN
    np.testing.assert_array_equal(g["topk_idx"].numpy()[tokens][clear], idx_own[clear])


def stratified_tokens(disp, T, k, tile=TILE_ROWS):
    """Tokens whose kept rows include, for every expert segment [offsets[e],
    offsets[e+1]) of the permuted rows, its first row, its last row and at
    least one row of each `tile`-row tile.  Greedy: a cell not yet covered by
    an earlier token's rows takes the token of its middle row (or of the named
    row)."""
    offs, perm, dest = disp["offsets"], disp["perm_src"], disp["dest"]
    cells = []
    for e in range(len(offs) - 1):
        a, b = int(offs[e]), int(offs[e + 1])
        if b == a:
            continue
        cells += [(a, a + 1), (b - 1, b)]
        cells += [(r0, min(b, r0 + tile)) for r0 in range(a, b, tile)]
    covered = np.zeros(int(offs[-1]), bool)
    chosen = []
    for lo, hi in cells:
        if covered[lo:hi].any():
            continue
        t = int(perm[(lo + hi - 1) // 2]) // k
        chosen.append(t)
        rows = dest[t * k:(t + 1) * k]
        covered[rows[rows >= 0]] = True
    assert all(covered[lo:hi].any() for lo, hi in cells)
    return sorted(set(chosen))


def test_full_size_layer_output_on_every_tile(full):
    cfg, g, inp, out = full["cfg"], full["gpu"], full["inp"], full["out"]
    T, E, k = cfg["T"], cfg["E"], cfg["k"]
    idx = g["topk_idx"].numpy()
    drop = g["drop_mask"].numpy()
    disp = oracle.dispatch(idx, E, oracle.capacity(T, k, E, cfg["capacity_factor"]))
    tokens = stratified_tokens(disp, T, k)
    full_drop = np.nonzero(drop.reshape(T, k).all(axis=1))[0]
    if len(full_drop):
        rng = np.random.default_rng(12)
        extra = rng.choice(full_drop, min(DROPPED_SAMPLES, len(full_drop)), replace=False)
        tokens = sorted(set(tokens) | set(int(t) for t in extra))
    # every expert with kept rows is reached
    reached = {int(idx[t, s]) for t in tokens for s in range(k) if not drop[t * k + s]}
    assert reached == {e for e in range(E) if disp["counts_kept"][e] > 0}
    sub, sidx, sdrop = _subset_inputs(inp, cfg, tokens, idx, drop)
    w = f64(g["topk_w"])[tokens]
    ref = oracle.layer_tokens(sub, sidx, w, sdrop, np.arange(len(tokens)))["y"]
    y = f64(out["y"].index_select(0, torch.tensor(tokens, device="cuda")))
    x = f64(sub["x"])
    assert max_rel(y, ref) < TOL_Y[cfg["dtype"]]
    assert moe_rel(y, ref, x, cfg["dtype"]) < TOL_Y[cfg["dtype"]]
