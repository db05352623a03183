"""Shared helpers of the parity tests: seeded inputs, CPU copies for the
oracle, error metrics and tolerances."""
import numpy as np
import torch

from sparse_mixture_experts_59_b300 import workloads

# Tolerances (max relative error, normalised by the reference's largest |value|):
#  - layer outputs: 1e-5 for fp32 layers, 2e-2 for bf16 layers, against the
#    fp64 oracle (bf16 rounds x, W, H and the slot outputs to 8 mantissa bits);
#  - aux loss, P_e and gate weights: 1e-5;
#  - router logits against the oracle's own: 1e-5 (fp32), 1e-3 (bf16 inputs
#    are exact; only the fp32 accumulation order differs).
TOL_Y = {"f32": 1e-5, "bf16": 2e-2}
TOL_LOGITS = {"f32": 1e-5, "bf16": 1e-3}
TOL_W = 1e-5
TOL_AUX = 1e-5
MARGIN = 1e-3          # near-tie exclusion of the index check on own logits

# Scaled-down parity workloads: the structure of each named workload with
# sizes the oracle finishes in seconds, chosen to span several tiles and to
# leave ragged tails in rows (segments), columns (N) and reduction (K).
SMALL = {
    "tiny_fp32": dict(base="tiny_fp32"),
    "mixtral_small": dict(base="mixtral_prefill", T=333, d=520, F=1400, seed=2001),
    "mixtral_decode_small": dict(base="mixtral_decode", T=5, d=264, F=392, seed=2002,
                                 weight_seed=2002),
    "fine_small": dict(base="fine_grained", T=200, d=256, F=128, E=32, k=8, F_shared=256,
                       seed=2003),
    "switch_small": dict(base="switch_skewed", T=1024, d=256, F=512, E=16, k=1, seed=2004),
    "gelu_cap_small": dict(base="tiny_fp32", T=300, d=264, F=320, E=6, k=2, dtype="bf16",
                           capacity_factor=1.25, seed=2005),
    "swiglu_fp32_shared": dict(base="fine_grained", T=70, d=96, F=64, E=5, k=2, F_shared=48,
                               dtype="f32", seed=2006),
    "sigmoid_shared_small": dict(base="fine_grained", T=160, d=192, F=128, E=16, k=4,
                                 F_shared=128, scoring="sigmoid", seed=2007),
    "softmax_norenorm_cap": dict(base="mixtral_prefill", T=400, d=256, F=384, E=8, k=2,
                                 renorm=False, capacity_factor=1.0, seed=2008),
    "sigmoid_fp32_norenorm": dict(base="tiny_fp32", T=90, scoring="sigmoid", renorm=False,
                                  seed=2009),
    # decode-sized layers (T*k <= 512, T*E <= 2048): the one-launch route +
    # dispatch, with 2, 8 and 4 router values per lane, k up to 8, a logit
    # bias, capacity drops and d below one 128-wide K-slice
    "decode_e64_k8": dict(base="fine_grained", T=32, d=256, F=128, E=64, k=8, F_shared=128,
                          seed=2010),
    "decode_e256_k8": dict(base="fine_grained", T=8, d=192, F=128, E=256, k=8, F_shared=128,
                           seed=2011),
    "decode_e128_sigmoid_cap": dict(base="mixtral_prefill", T=16, d=64, F=128, E=128, k=6,
                                    scoring="sigmoid", renorm=False, capacity_factor=1.0,
                                    seed=2012),
    "decode_switch_bias": dict(base="switch_skewed", T=64, d=128, F=256, E=16, k=1, seed=2013),
    # segments of ~440 rows (two 256-row tiles each, the second ragged) and a
    # 1100-row shared expert over several tiles
    "long_segments_shared": dict(base="fine_grained", T=1100, d=320, F=192, E=5, k=2,
                                 F_shared=192, seed=2014),
}


def small_cfg(name):
    spec = dict(SMALL[name])
    base = spec.pop("base")
    cfg = workloads.config(base, **spec)
    cfg["name"] = name
    return cfg


def to_cpu(inp):
    return {k: (v.detach().cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def max_rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    if scale == 0.0:
        return float(np.max(np.abs(got - ref))) if ref.size else 0.0
    return float(np.max(np.abs(got - ref)) / scale)


def moe_rel(y, y_ref, x, dtype):
    """Error of the MoE contribution y - x, relative to max|y_ref - x|, after
    allowing each output element its own rounding to the output dtype (half a
    bf16 ulp is at most 2^-8 |y|).  With x of order 1 and an MoE
    contribution of order 0.05, that rounding alone would otherwise exceed the
    tolerance, so the residual cannot hide an MoE error either way."""
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    x = np.asarray(x, np.float64)
    slack = (2.0 ** -8) * np.abs(y_ref) if dtype == "bf16" else 0.0
    excess = np.maximum(np.abs(y - y_ref) - slack, 0.0)
    scale = np.max(np.abs(y_ref - x)) if y_ref.size else 0.0
    return float(np.max(excess) / scale) if scale > 0 else float(np.max(excess, initial=0.0))


def f64(t):
    return t.detach().double().cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def margins(logits, k):
    """Gap between the k-th and (k+1)-th largest logit per token (inf if k == E)."""
    l = np.sort(np.asarray(logits, np.float64), axis=1)[:, ::-1]
    if l.shape[1] <= k:
        return np.full(l.shape[0], np.inf)
    return l[:, k - 1] - l[:, k]
