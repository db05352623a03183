"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test fixes one part of the oracle with brute force, a closed form, a
library routine (numpy matmul, scipy softmax/expit/ndtr) or a special case of
the method, so that a plausible mistake (a dropped term, a wrong sign, index or
tie rule, a transposed operand, slot-major instead of token-major drops) fails
at least one of them.  CPU only.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit, ndtr, softmax

import oracle
from sparse_mixture_experts_59_b300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------- routing
@pytest.mark.parametrize("E,k", [(2, 1), (3, 2), (5, 2), (8, 2), (8, 3), (6, 6)])
def test_topk_matches_subset_enumeration(E, k):
    """Top-k equals the max-sum subset of size k; on ties the lexicographically
    smallest index set wins (ties go to the lower expert index), and slots are
    ordered by logit descending then index ascending."""
    r = _rng(E * 10 + k)
    T = 300
    # integer-valued logits force many exact ties; half the rows are continuous
    logits = np.where(r.random((T, 1)) < 0.5,
                      r.integers(-2, 3, size=(T, E)).astype(np.float64),
                      r.normal(size=(T, E)))
    idx, w, probs = oracle.topk(logits, k)
    for t in range(T):
        l = logits[t]
        best = None
        for sub in itertools.combinations(range(E), k):
            s = sum(l[list(sub)])
            if best is None or s > best[0] + 0.0 or (s == best[0] and sub < best[1]):
                best = (s, sub)
        chosen = sorted(best[1], key=lambda e: (-l[e], e))
        assert list(idx[t]) == chosen, (t, l, idx[t], chosen)


def test_weights_equal_softmax_over_selected_logits():
    """Renormalised top-k softmax probabilities equal a softmax taken over the
    k selected logits only (the form on the hassanahmed.net page); the full
    probabilities equal scipy's softmax."""
    r = _rng(7)
    logits = r.normal(scale=3.0, size=(500, 16))
    for k in (1, 2, 4, 8, 16):
        idx, w, probs = oracle.topk(logits, k)
        sel = np.take_along_axis(logits, idx.astype(np.int64), axis=1)
        np.testing.assert_allclose(w, softmax(sel, axis=1), rtol=1e-12, atol=0)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert np.all(np.diff(w, axis=1) <= 0)
        np.testing.assert_allclose(probs, softmax(logits, axis=1), rtol=1e-12, atol=1e-300)


def test_router_logits_match_numpy_matmul():
    """Router logits = x @ Wr^T + bias with Wr in nn.Linear layout [E, d]
    (non-square, so a transposed operand cannot pass)."""
    r = _rng(3)
    T, d, E = 37, 24, 5
    x = r.normal(size=(T, d)).astype(np.float32)
    Wr = r.normal(size=(E, d)).astype(np.float32)
    b = r.normal(size=E).astype(np.float32)
    got = oracle.router_logits(x, Wr, b)
    ref = x.astype(np.float64) @ Wr.astype(np.float64).T + b.astype(np.float64)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    sub = oracle.router_logits(x, Wr, None, tokens=[5, 0, 36])
    np.testing.assert_allclose(sub, (x.astype(np.float64) @ Wr.astype(np.float64).T)[[5, 0, 36]],
                               rtol=1e-12, atol=1e-12)


def test_bf16_inputs_widen_exactly():
    """bf16 storage is widened exactly (compared with torch's own bf16->f64)."""
    r = torch.Generator().manual_seed(5)
    x = torch.randn(9, 16, generator=r).to(torch.bfloat16)
    Wr = torch.randn(3, 16, generator=r).to(torch.bfloat16)
    got = oracle.router_logits(x, Wr)
    ref = x.double().numpy() @ Wr.double().numpy().T
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- capacity
def test_capacity_formula():
    """max(int(T*k/E*cf), 1) from "The Capacity Factor"; <= 0 means dropless."""
    assert oracle.capacity(64, 2, 8, 1.25) == 20          # tiny fp32 workload
    assert oracle.capacity(16384, 1, 64, 1.0) == 256      # switch_skewed workload
    assert oracle.capacity(10, 1, 3, 1.0) == 3            # floor, not round
    assert oracle.capacity(10, 2, 3, 1.0) == 6            # 6.67 -> 6
    assert oracle.capacity(1, 1, 8, 1.0) == 1             # at least one
    assert oracle.capacity(100, 2, 8, 0.0) == -1          # dropless
    assert oracle.capacity(100, 2, 8, -1.0) == -1


# ---------------------------------------------------------------- dispatch
def _brute_dispatch(idx, E, cap):
    """Sort-based construction: per expert, the (token, slot) pairs that chose
    it in token order; the first `cap` are kept."""
    T, k = idx.shape
    kept_lists, counts = [], []
    drop = np.zeros(T * k, np.uint8)
    for e in range(E):
        pairs = sorted((t, s) for t in range(T) for s in range(k) if idx[t, s] == e)
        counts.append(len(pairs))
        kept = pairs if cap < 0 else pairs[:cap]
        for (t, s) in pairs[len(kept):]:
            drop[t * k + s] = 1
        kept_lists.append([t * k + s for (t, s) in kept])
    perm = [a for lst in kept_lists for a in lst]
    offsets = np.concatenate([[0], np.cumsum([len(l) for l in kept_lists])]).astype(np.int32)
    dest = np.full(T * k, -1, np.int32)
    for r_, a in enumerate(perm):
        dest[a] = r_
    return dict(counts_pre=np.array(counts, np.int32),
                counts_kept=np.array([len(l) for l in kept_lists], np.int32),
                offsets=offsets, perm_src=np.array(perm, np.int32), dest=dest, drop_mask=drop)


def _random_idx(r, T, E, k):
    return np.stack([r.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k,cap", [(1, 4, 2, -1), (7, 3, 2, 1), (50, 8, 2, 5),
                                       (200, 16, 4, 40), (333, 8, 2, -1), (97, 5, 5, 10),
                                       (64, 8, 2, 20)])
def test_dispatch_matches_sort_construction(T, E, k, cap):
    r = _rng(T * 131 + E)
    idx = _random_idx(r, T, E, k)
    got = oracle.dispatch(idx, E, cap)
    ref = _brute_dispatch(idx, E, cap)
    for key in ("counts_pre", "counts_kept", "offsets", "perm_src", "dest", "drop_mask"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    # invariants
    A = T * k
    assert got["counts_pre"].sum() == A
    assert got["counts_kept"].sum() == A - int(got["drop_mask"].sum()) == got["R"]
    assert np.all(np.diff(got["offsets"]) >= 0) and got["offsets"][-1] == got["R"]
    kept = np.nonzero(got["drop_mask"] == 0)[0]
    assert sorted(got["dest"][kept].tolist()) == list(range(got["R"]))     # bijection
    for e in range(E):
        seg = got["perm_src"][got["offsets"][e]:got["offsets"][e + 1]]
        assert np.all(np.diff(seg // k) > 0)                               # token order


def test_drop_order_is_token_major_not_slot_major():
    """Expert 0 is slot 1 of token 0 and slot 0 of token 1; with capacity 1
    token 0 keeps it (token order), although token 1 ranks it first."""
    idx = np.array([[1, 0], [0, 2]], np.int32)
    got = oracle.dispatch(idx, 3, 1)
    assert got["drop_mask"].tolist() == [0, 0, 1, 0]
    assert got["perm_src"].tolist() == [1, 0, 3]


# ------------------------------------------------------ activations / FFN
def test_activation_closed_forms():
    """GELU is the erf form z*Phi(z) (Phi from scipy's ndtr; gelu(1)=Phi(1));
    SwiGLU with unit weights gives silu(z)*z = z^2 * expit(z)."""
    one = np.ones((1, 1), np.float32)
    zero = np.zeros(1, np.float32)
    for z in (-3.0, -1.0, -0.25, 0.0, 0.5, 1.0, 2.5):
        g = oracle.expert_ffn([z], one, None, one, zero, zero, act="gelu")[0]
        assert g == pytest.approx(z * ndtr(z), rel=1e-14, abs=1e-300)
        s = oracle.expert_ffn([z], one, one, one, act="swiglu")[0]
        assert s == pytest.approx(z * z * expit(z), rel=1e-14, abs=1e-300)
    assert oracle.expert_ffn([1.0], one, None, one, zero, zero, act="gelu")[0] == \
        pytest.approx(0.8413447460685429, rel=1e-14)


def _np_ffn(x, W1, W3, W2, b1, b2, act):
    x = x.astype(np.float64)
    if act == "swiglu":
        g = x @ W1.T
        u = x @ W3.T
        h = g * expit(g) * u
        return h @ W2.T
    z = x @ W1.T + b1
    h = z * ndtr(z)
    return h @ W2.T + b2


def _small_inputs(act, E, k, T=11, d=16, F=24, cf=0.0, shared=0, seed=0, has_bias=None):
    r = _rng(seed)
    hb = (act == "gelu") if has_bias is None else has_bias
    inp = dict(
        x=r.normal(size=(T, d)).astype(np.float32),
        Wr=r.normal(size=(E, d)).astype(np.float32),
        W1=(r.normal(size=(E, F, d)) / math.sqrt(d)).astype(np.float32),
        W3=(r.normal(size=(E, F, d)) / math.sqrt(d)).astype(np.float32) if act == "swiglu" else None,
        W2=(r.normal(size=(E, d, F)) / math.sqrt(F)).astype(np.float32),
        b1=r.normal(size=(E, F)).astype(np.float32) if hb else None,
        b2=r.normal(size=(E, d)).astype(np.float32) if hb else None,
        S1=(r.normal(size=(shared, d)) / math.sqrt(d)).astype(np.float32) if shared else None,
        S3=(r.normal(size=(shared, d)) / math.sqrt(d)).astype(np.float32) if shared else None,
        S2=(r.normal(size=(d, shared)) / math.sqrt(shared)).astype(np.float32) if shared else None,
        logit_bias=None,
        cfg=dict(T=T, d=d, F=F, E=E, k=k, act=act, capacity_factor=cf, F_shared=shared,
                 dtype="f32"))
    return inp


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
@pytest.mark.parametrize("shared", [0, 20])
def test_single_expert_layer_is_dense_ffn_plus_residual(act, shared):
    """E=1, k=1, dropless: y = x + FFN(x) (+ shared FFN(x)) by numpy matmuls."""
    inp = _small_inputs(act, E=1, k=1, shared=shared if act == "swiglu" else 0, seed=11)
    out = oracle.layer_forward(inp, want_slots=True, want_shared=True)
    ref = _np_ffn(inp["x"], inp["W1"][0], None if inp["W3"] is None else inp["W3"][0],
                  inp["W2"][0], None if inp["b1"] is None else inp["b1"][0],
                  None if inp["b2"] is None else inp["b2"][0], act)
    assert np.all(out["topk_idx"] == 0) and np.all(out["topk_w"] == 1.0)
    if inp["S1"] is not None:
        sh = _np_ffn(inp["x"], inp["S1"], inp["S3"], inp["S2"], None, None, "swiglu")
        np.testing.assert_allclose(out["shared"], sh, rtol=1e-12, atol=1e-12)
        ref = ref + sh
    np.testing.assert_allclose(out["y"], inp["x"].astype(np.float64) + ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
def test_k_equals_E_is_soft_mixture(act):
    """k = E, dropless: y = x + sum_e p_e FFN_e(x), the dense soft mixture."""
    E = 4
    inp = _small_inputs(act, E=E, k=E, seed=12)
    out = oracle.layer_forward(inp)
    l = inp["x"].astype(np.float64) @ inp["Wr"].astype(np.float64).T
    p = softmax(l, axis=1)
    ref = inp["x"].astype(np.float64).copy()
    for e in range(E):
        fe = _np_ffn(inp["x"], inp["W1"][e], None if inp["W3"] is None else inp["W3"][e],
                     inp["W2"][e], None if inp["b1"] is None else inp["b1"][e],
                     None if inp["b2"] is None else inp["b2"][e], act)
        ref += p[:, e:e + 1] * fe
    np.testing.assert_allclose(out["y"], ref, rtol=1e-11, atol=1e-11)


def test_partly_dropped_token_keeps_surviving_weight():
    """A token that loses one slot to capacity keeps the other slot's original
    weight (no re-normalisation) and gets nothing from the dropped one."""
    inp = _small_inputs("swiglu", E=3, k=2, T=2, seed=13)
    # token 0 prefers experts (0, 1); token 1 prefers (0, 2); capacity 1
    inp["Wr"] = np.zeros_like(inp["Wr"])
    x = inp["x"]
    x[:, 0] = 1.0
    inp["Wr"][:, 0] = [2.0, 1.0, 0.0]
    x[0, 1] = 0.0
    x[1, 1] = 3.0
    inp["Wr"][:, 1] = [0.0, -1.0, 0.5]      # logits: token 0 [2, 1, 0], token 1 [2, -2, 1.5]
    inp["cfg"]["capacity_factor"] = 0.75       # cap = int(2*2/3*0.75) = 1
    out = oracle.layer_forward(inp, want_slots=True)
    assert out["cap"] == 1
    assert out["topk_idx"].tolist() == [[0, 1], [0, 2]]
    s_e0, s_e2 = 0, 1
    assert out["drop_mask"][2 + s_e0] == 1 and out["drop_mask"][2 + s_e2] == 0
    f2 = _np_ffn(x[1:2], inp["W1"][2], inp["W3"][2], inp["W2"][2], None, None, "swiglu")[0]
    w = out["topk_w"][1, s_e2]
    np.testing.assert_allclose(out["y"][1], x[1].astype(np.float64) + w * f2, rtol=1e-12, atol=1e-12)
    assert np.all(out["slots"][1, s_e0] == 0.0)


# ---------------------------------------------------------- special cases
@pytest.mark.parametrize("E,k,cf", [(8, 2, 1.25), (4, 1, 1.0), (6, 3, 0.0), (8, 2, 0.5)])
def test_all_ties_router(E, k, cf):
    """Wr = 0: every logit ties, so every token picks experts 0..k-1 in order
    with weight 1/k, P_e = 1/E and f_e = 1 for e < k, hence aux = k exactly.
    With a capacity, tokens t >= cap lose every slot and y = x exactly."""
    T = 40
    inp = _small_inputs("gelu", E=E, k=k, T=T, cf=cf, seed=14)
    inp["Wr"] = np.zeros_like(inp["Wr"])
    out = oracle.layer_forward(inp)
    assert np.all(out["topk_idx"] == np.arange(k)[None, :])
    np.testing.assert_allclose(out["topk_w"], 1.0 / k, rtol=0, atol=1e-15)
    np.testing.assert_allclose(out["probs"], 1.0 / E, rtol=0, atol=1e-15)
    assert out["aux"] == pytest.approx(float(k), rel=1e-14)
    cap = out["cap"]
    n_keep = T if cap < 0 else min(T, cap)
    assert out["counts_kept"].tolist() == [n_keep] * k + [0] * (E - k)
    dm = out["drop_mask"].reshape(T, k)
    assert np.all(dm[:n_keep] == 0) and np.all(dm[n_keep:] == 1)
    np.testing.assert_array_equal(out["y"][n_keep:], inp["x"][n_keep:].astype(np.float64))
    assert out["drop_frac"] == pytest.approx((T - n_keep) / T)


def test_aux_loss_closed_forms():
    """Two-token, two-expert, top-1 examples with probabilities 1/4 and 3/4:
    balanced routing gives aux = 2*(0.5*0.5 + 0.5*0.5) = 1; both tokens on
    expert 0 gives aux = 2*(1*0.75 + 0*0.25) = 1.5."""
    ln3 = math.log(3.0)
    idx, w, probs = oracle.topk([[0.0, ln3], [ln3, 0.0]], 1)
    d = oracle.dispatch(idx, 2, -1)
    assert idx.ravel().tolist() == [1, 0]
    assert oracle.aux_loss(d["counts_pre"], probs) == pytest.approx(1.0, rel=1e-14)
    idx, w, probs = oracle.topk([[ln3, 0.0], [ln3, 0.0]], 1)
    d = oracle.dispatch(idx, 2, -1)
    np.testing.assert_allclose(probs[0], [0.75, 0.25], rtol=1e-14)
    assert oracle.aux_loss(d["counts_pre"], probs) == pytest.approx(1.5, rel=1e-14)
    # f counts every top-k slot (sum f = k): uniform routing with k = 2 gives 2
    idx, w, probs = oracle.topk(np.zeros((4, 4)), 2)
    d = oracle.dispatch(idx, 4, -1)
    assert oracle.aux_loss(d["counts_pre"], probs) == pytest.approx(2.0, rel=1e-14)


# ----------------------------------------------------------- page values
def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if line:
                key, val = [s.strip() for s in line.split("=", 1)]
                vals[key] = val
    return vals


def test_page_example_shapes_and_parameter_counts():
    """The example layer's printed shapes (input and output (2,16,512)) and the
    page's parameter counts: ~25M expert parameters for 8 SwiGLU experts at
    d=512, d_ff=2048; 32,768 router and ~176M per-expert, ~1.41B per-layer
    FFN parameters at the Mixtral shape."""
    g = _golden("nybble_moe_example.txt")
    d, F, E, k = (int(g["example." + s]) for s in ("d_model", "d_ff", "num_experts", "top_k"))
    inp = workloads.make_inputs(workloads.config("mixtral_prefill", T=32, d=d, F=F, E=E, k=k,
                                                 dtype="f32", seed=77))
    assert tuple(int(v) for v in g["example.input_shape"].split(",")) == (2, 16, d)
    out = oracle.layer_forward(inp)
    assert out["y"].reshape(2, 16, d).shape == tuple(int(v) for v in g["example.output_shape"].split(","))
    n_exp = sum(inp[key].numel() for key in ("W1", "W3", "W2"))
    assert abs(n_exp - float(g["example.expert_params.approx"])) / float(g["example.expert_params.approx"]) < 0.01
    m = workloads.config("mixtral_prefill")
    assert (m["d"], m["F"], m["E"]) == (int(g["mixtral.d_model"]), int(g["mixtral.d_ff"]),
                                        int(g["mixtral.num_experts"]))
    assert m["d"] * m["E"] == int(g["mixtral.router_params"])
    per_expert = 3 * m["d"] * m["F"]
    assert abs(per_expert - float(g["mixtral.expert_params.approx"])) / 176e6 < 0.005
    assert abs(m["E"] * per_expert - float(g["mixtral.layer_ffn_params.approx"])) / 1.41e9 < 0.005



def test_mixtral_shape_against_the_pages_parameter_totals():
    """The pages give Mixtral 8x7B as 46.7B parameters held and 12.9B active
    per token. Attention, embeddings and norms count in both totals, so the
    difference is the (E - k) unused expert FFNs of every layer:
    layers x (E - k) x 3 d F, with each total rounded to 0.1B. The layer-wise
    breakdown (32 x (8 experts + ~67M attention) ~ 47B; 32 x (2 experts +
    attention) ~ 13B) must also hold for the Mixtral workload's d, F, E and k.
    A wrong k, E, d or F misses the difference by whole billions."""
    g = _golden("mixtral_param_counts.txt")
    m = workloads.config("mixtral_prefill")
    layers = int(g["mixtral.layers"])
    per_expert = 3 * m["d"] * m["F"]
    idle = layers * (m["E"] - m["k"]) * per_expert
    printed = float(g["mixtral.total_params"]) - float(g["mixtral.active_params"])
    assert abs(idle - printed) <= 0.1e9
    attn = float(g["mixtral.attention_params_per_layer.approx"])
    total = layers * (m["E"] * per_expert + attn)
    active = layers * (m["k"] * per_expert + attn)
    assert abs(total - float(g["mixtral.total_params_layerwise.approx"])) / 47e9 < 0.01
    assert abs(active - float(g["mixtral.active_params_layerwise.approx"])) / 13e9 < 0.05
    # the decode workload streams the same weights
    assert workloads.config("mixtral_decode")["E"] == m["E"]

def test_workload_capacities_and_skew():
    """The tiny workload has capacity 20 and the skewed Switch workload 256;
    the skew offsets fall with expert index as -1.8 ln(e+1)."""
    c0 = workloads.config("tiny_fp32")
    assert oracle.capacity(c0["T"], c0["k"], c0["E"], c0["capacity_factor"]) == 20
    c4 = workloads.config("switch_skewed")
    assert oracle.capacity(c4["T"], c4["k"], c4["E"], c4["capacity_factor"]) == 256
    b = workloads.skew_bias(64).numpy()
    np.testing.assert_allclose(b, -1.8 * np.log(np.arange(1, 65)), rtol=1e-6, atol=1e-6)


# ------------------------------------------------------- scoring variants
def test_sigmoid_scores_and_unrenormalised_weights():
    """Sigmoid scoring gives scipy's expit of every logit; without
    renormalisation the kept weights are the kept scores themselves; the
    selected experts are those of the softmax router (both are monotone)."""
    r = _rng(21)
    logits = r.normal(scale=2.0, size=(300, 12))
    k = 3
    idx_soft, w_soft, p_soft = oracle.topk(logits, k)
    idx_sig, w_sig, p_sig = oracle.topk(logits, k, scoring="sigmoid", renorm=True)
    np.testing.assert_array_equal(idx_sig, idx_soft)
    np.testing.assert_allclose(p_sig, expit(logits), rtol=1e-14, atol=0)
    sel = np.take_along_axis(p_sig, idx_sig.astype(np.int64), axis=1)
    np.testing.assert_allclose(w_sig, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13)
    _, w_raw, _ = oracle.topk(logits, k, scoring="sigmoid", renorm=False)
    np.testing.assert_allclose(w_raw, sel, rtol=0, atol=0)
    _, w_soft_raw, _ = oracle.topk(logits, k, scoring="softmax", renorm=False)
    np.testing.assert_allclose(w_soft_raw, np.take_along_axis(p_soft, idx_soft.astype(np.int64), axis=1),
                               rtol=0, atol=0)
    # unrenormalised softmax weights sum to less than one unless k = E
    assert np.all(w_soft_raw.sum(axis=1) < 1.0)


def test_sigmoid_layer_single_expert_is_scaled_dense_ffn():
    """E=1, k=1 with sigmoid scoring and no renormalisation: y = x +
    sigmoid(l) * FFN(x) (numpy)."""
    inp = _small_inputs("swiglu", E=1, k=1, seed=22)
    inp["cfg"]["scoring"] = "sigmoid"
    inp["cfg"]["renorm"] = False
    out = oracle.layer_forward(inp)
    l = inp["x"].astype(np.float64) @ inp["Wr"].astype(np.float64).T
    ref = _np_ffn(inp["x"], inp["W1"][0], inp["W3"][0], inp["W2"][0], None, None, "swiglu")
    np.testing.assert_allclose(out["y"], inp["x"].astype(np.float64) + expit(l) * ref,
                               rtol=1e-12, atol=1e-12)


# ------------------------------------------------------ aux loss backward
@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
def test_aux_gradient_matches_central_differences(scoring):
    """The analytic logit gradient of the aux loss equals central finite
    differences of the oracle's own aux loss with the counts held fixed."""
    r = _rng(31)
    T, E, k = 6, 5, 2
    logits = r.normal(size=(T, E))
    idx, _, probs = oracle.topk(logits, k, scoring=scoring)
    counts = oracle.dispatch(idx, E, -1)["counts_pre"]
    g = oracle.aux_grad_logits(logits, counts, grad_aux=0.7, scoring=scoring)
    h = 1e-6
    for t in range(T):
        for j in range(E):
            lp, lm = logits.copy(), logits.copy()
            lp[t, j] += h
            lm[t, j] -= h
            ap = oracle.aux_loss(counts, oracle.topk(lp, k, scoring=scoring)[2])
            am = oracle.aux_loss(counts, oracle.topk(lm, k, scoring=scoring)[2])
            assert g[t, j] == pytest.approx(0.7 * (ap - am) / (2 * h), rel=1e-6, abs=1e-10)


def _dyadic(r, shape, lo, hi, bits=8):
    """fp32 values that are multiples of 2^-bits in [lo, hi): adding or
    subtracting 2^-20 to one of them stays exact in fp32 (|v| < 8 needs at
    most 23 significant bits), so a finite-difference step perturbs exactly
    the one input it names."""
    scale = 2 ** bits
    return (r.integers(int(lo * scale), int(hi * scale), size=shape) / scale).astype(np.float32)


@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
def test_aux_router_backward_matches_central_differences(scoring):
    """g_Wr and g_x of the oracle's router backward equal central finite
    differences of the forward aux loss taken through the oracle's own
    router (logits from x and Wr), scores and aux loss, with the pre-drop
    counts f_e held fixed (they are piecewise constant).  Non-square shapes
    (T=7, d=5, E=4), so a transposed product or a swapped operand fails; every
    entry of Wr and of x is perturbed on its own."""
    r = _rng(32)
    T, d, E, k = 7, 5, 4, 2
    x = _dyadic(r, (T, d), -4, 4)
    Wr = _dyadic(r, (E, d), -0.75, 0.75)
    logits = oracle.router_logits(x, Wr)
    idx, _, _ = oracle.topk(logits, k, scoring=scoring)
    counts = oracle.dispatch(idx, E, -1)["counts_pre"]
    g, gW, gx = oracle.aux_router_backward(x, Wr, logits, counts, grad_aux=0.7, scoring=scoring)
    assert gW.shape == (E, d) and gx.shape == (T, d)

    def aux(xv, wv):
        return oracle.aux_loss(counts, oracle.topk(oracle.router_logits(xv, wv), k,
                                                   scoring=scoring)[2])

    h = np.float32(2.0 ** -20)
    fd_W = np.empty((E, d))
    for e in range(E):
        for i in range(d):
            wp, wm = Wr.copy(), Wr.copy()
            wp[e, i] += h
            wm[e, i] -= h
            assert wp[e, i] - Wr[e, i] == h and Wr[e, i] - wm[e, i] == h
            fd_W[e, i] = 0.7 * (aux(x, wp) - aux(x, wm)) / (2.0 * float(h))
    fd_x = np.empty((T, d))
    for t in range(T):
        for i in range(d):
            xp, xm = x.copy(), x.copy()
            xp[t, i] += h
            xm[t, i] -= h
            assert xp[t, i] - x[t, i] == h and x[t, i] - xm[t, i] == h
            fd_x[t, i] = 0.7 * (aux(xp, Wr) - aux(xm, Wr)) / (2.0 * float(h))
    np.testing.assert_allclose(gW, fd_W, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(gx, fd_x, rtol=1e-6, atol=1e-9)
    # the differences are not vacuous: the gradients are far from zero
    assert np.abs(fd_W).max() > 1e-3 and np.abs(fd_x).max() > 1e-3


# ----------------------------------------------------- FP8 expert weights
def test_e4m3_decoding_matches_torch_for_every_code():
    """The oracle's E4M3 decoding (from the format's definition) equals
    torch's float8_e4m3fn -> float64 conversion for all 256 codes (NaN codes
    compared as NaN)."""
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


def test_fp8_expert_layer_equals_dequantised_fp64_layer():
    """A layer with E4M3 expert weights and row scales equals the same layer
    with the weights dequantised exactly (code * scale in double) by numpy."""
    inp = workloads.make_inputs(workloads.config("mixtral_prefill", T=5, d=32, F=48, E=3, k=2,
                                                 seed=41))
    q = workloads.quantize_experts_fp8(inp)
    tokens = np.arange(5)
    routed = oracle.layer_forward(q, tokens=tokens)
    xf = inp["x"].double().numpy()
    for r, t in enumerate(tokens):
        ref = xf[t].copy()
        for s in range(2):
            e = routed["topk_idx"][t, s]
            W1 = q["W1"][e].view(torch.uint8).numpy()
            deq = lambda key, skey: (np.vectorize(oracle.e4m3_value)(q[key][e].view(torch.uint8).numpy())
                                     * q[skey][e].double().numpy()[:, None])
            g = deq("W1", "s1") @ xf[t]
            u = deq("W3", "s3") @ xf[t]
            h = g * expit(g) * u
            ref += routed["topk_w"][t, s] * (deq("W2", "s2") @ h)
        np.testing.assert_allclose(routed["y"][r], ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------- 4-bit expert weights
def test_e2m1_decoding_matches_the_format_value_set():
    """E2M1 (1 sign, 2 exponent, 1 mantissa bit) has the eight magnitudes
    0, 0.5, 1, 1.5, 2, 3, 4, 6 on codes 0..7 and their negatives on 8..15 (the
    OCP microscaling format's value table); the oracle decodes its codes from
    the bit fields."""
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = [oracle.e2m1_value(c) for c in range(16)]
    assert got[:8] == table
    assert got[8:] == [-v for v in table]
    assert np.signbit(got[8])                    # code 8 is -0


def test_fp4_quantiser_error_bound():
    """Every element of a 4-bit matrix decodes to within one block-scale step of
    the weight it came from: |w - q b s| <= b s (the largest E2M1 gap is 2,
    between 4 and 6), plus the saturation of |w| / (b s) above 6 when the
    block scale rounded down."""
    torch.manual_seed(3)
    w = (torch.randn(7, 384) * 0.02).to(torch.bfloat16)
    packed, rs = workloads.quantize_rows_fp4(w)
    deq = workloads.dequantize_rows_fp4(packed, rs)
    bs = packed.view(7, -1, 80)[:, :, 64:72].contiguous().view(torch.float8_e4m3fn).double()
    step = (bs * rs.double()[:, None, None]).repeat_interleave(16, dim=2).view(7, -1)
    excess = (w.double().abs() - 6.0 * step).clamp(min=0)
    assert torch.all((deq - w.double()).abs() <= step + excess + 1e-30)
    assert torch.all(packed.view(7, -1, 80)[:, :, 72:] == 0)


def test_fp4_expert_layer_equals_dequantised_fp64_layer():
    """A layer with packed 4-bit expert weights and row scales equals the same
    layer on the weights decoded by an independent (torch) decoder of the
    packed layout, computed with numpy in float64."""
    inp = workloads.make_inputs(workloads.config("mixtral_prefill", T=5, d=128, F=256, E=3, k=2,
                                                 seed=43))
    q = workloads.quantize_experts_fp4(inp)
    tokens = np.arange(5)
    routed = oracle.layer_forward(q, tokens=tokens)
    xf = inp["x"].double().numpy()
    deq = lambda key, skey, e: workloads.dequantize_rows_fp4(q[key][e], q[skey][e]).numpy()
    for r, t in enumerate(tokens):
        ref = xf[t].copy()
        for s in range(2):
            e = routed["topk_idx"][t, s]
            g = deq("W1", "s1", e) @ xf[t]
            u = deq("W3", "s3", e) @ xf[t]
            h = g * expit(g) * u
            ref += routed["topk_w"][t, s] * (deq("W2", "s2", e) @ h)
        np.testing.assert_allclose(routed["y"][r], ref, rtol=1e-12, atol=1e-12)
