"""CPU oracle for the sparse top-k MoE layer forward (test infrastructure).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import
this package.  It wraps the plain C oracle in moe_oracle.c (fp64 arithmetic)
with numpy marshalling and shares nothing with the CUDA path.

Each function cites the passage it follows in its docstring; the C source
carries the same citations.
"""
import ctypes
import os

import numpy as np

from . import build as _build

ORC_F32, ORC_BF16, ORC_E4M3, ORC_E2M1P = 0, 1, 2, 3
ORC_GELU_ERF, ORC_SWIGLU = 0, 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P, I, D, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_longlong
        lib.oracle_router_logits.argtypes = [I, P, I, I, I, P, P, P, P]
        lib.oracle_topk.argtypes = [I, I, I, P, P, P, P]
        lib.oracle_topk_ex.argtypes = [I, I, I, I, I, P, P, P, P]
        lib.oracle_capacity.argtypes = [LL, I, I, D]
        lib.oracle_capacity.restype = LL
        lib.oracle_dispatch.argtypes = [I, I, I, LL, P, P, P, P, P, P, P, P]
        lib.oracle_dispatch.restype = I
        lib.oracle_expert_ffn.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P]
        lib.oracle_layer_tokens.argtypes = [I, P, I, I, I, I, I, I, P, P, P, P, P, P,
                                            I, P, P, P, P, P, P, P, P, P]
        lib.oracle_layer_tokens_q.argtypes = [I, P, I, I, I, I, I, I, I, P, P, P, P, P, P,
                                              P, P, P, I, P, P, P, P, P, P, P, P, P]
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint]
        lib.oracle_e2m1_value.argtypes = [ctypes.c_uint]
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.restype = D
        lib.oracle_aux_loss.argtypes = [I, I, P, P]
        lib.oracle_aux_loss.restype = D
        lib.oracle_aux_grad_logits.argtypes = [I, I, I, P, P, D, P]
        lib.oracle_set_threads.argtypes = [I]
        lib.oracle_get_threads.restype = I
        _lib = lib
    return _lib


def set_threads(n: int) -> None:
    """Number of host threads the oracle uses (0 = all online cores)."""
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def _buf(a):
    """(contiguous numpy array, dtype code) for fp32 or bf16 data.

    Accepts numpy float32, numpy uint16 holding bf16 bit patterns, or CPU torch
    tensors of dtype float32 / bfloat16 (viewed, not converted); float8_e4m3fn
    tensors are E4M3 codes and uint8 tensors the packed 4-bit weight layout."""
    if a is None:
        return None, None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().contiguous().cpu()
            if a.dtype == torch.bfloat16:
                return np.ascontiguousarray(a.view(torch.int16).numpy().view(np.uint16)), ORC_BF16
            if a.dtype == torch.float32:
                return np.ascontiguousarray(a.numpy()), ORC_F32
            if a.dtype == torch.float8_e4m3fn:
                return np.ascontiguousarray(a.view(torch.uint8).numpy()), ORC_E4M3
            if a.dtype == torch.uint8:
                return np.ascontiguousarray(a.numpy()), ORC_E2M1P
            raise TypeError("oracle takes float32 or bfloat16 tensors, got %s" % a.dtype)
    except ImportError:
        pass
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, ORC_F32
    if a.dtype == np.uint16:
        return a, ORC_BF16
    if a.dtype == np.uint8:
        return a, ORC_E2M1P
    raise TypeError("oracle takes float32 or bf16 (uint16 bits) arrays, got %s" % a.dtype)


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def e2m1_value(code: int) -> float:
    """The oracle's decoding of one E2M1 nibble (from the format's definition)."""
    return float(_load().oracle_e2m1_value(int(code)))


def e4m3_value(code: int) -> float:
    """The oracle's decoding of one E4M3 byte (its own, from the format's
    definition)."""
    return float(_load().oracle_e4m3_value(int(code)))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(a) -> np.ndarray:
    """Exact float64 copy of fp32/bf16 data (numpy or torch)."""
    arr, code = _buf(a)
    return bf16_bits_to_f64(arr) if code == ORC_BF16 else arr.astype(np.float64)


def router_logits(x, Wr, bias=None, tokens=None) -> np.ndarray:
    """Router logits l[t,e] = sum_i x[t,i] Wr[e,i] (+ bias[e]) in double.

    "How Mixture of Experts Works", section "The Gating Mechanism" (bias-free
    linear router); "Mixture of Experts (MoE)", section "The router".  Wr has
    the nn.Linear layout [E, d]; bias is an optional fixed fp32 logit offset."""
    xa, xc = _buf(x)
    wa, wc = _buf(Wr)
    assert xc == wc, "x and Wr must share a storage type"
    T, d = xa.shape
    E = wa.shape[0]
    assert wa.shape[1] == d
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = T if tok is None else len(tok)
    b = None if bias is None else np.ascontiguousarray(np.asarray(bias, dtype=np.float32))
    out = np.empty((n, E), dtype=np.float64)
    _load().oracle_router_logits(n, _ptr(tok), d, E, xc, _ptr(xa), _ptr(wa), _ptr(b), _ptr(out))
    return out


def topk(logits, k: int, scoring: str = "softmax", renorm: bool = True):
    """Scores, top-k on the logits (ties to the lower index), kept weights.
    Default: softmax over all experts and renormalised weights ("How Mixture
    of Experts Works", section "The Gating Mechanism").  scoring="sigmoid"
    scores each expert independently and renorm=False keeps the raw kept
    scores ("Mixture-of-Experts routing", "The knobs").  Returns (idx int32
    [T,k], w float64 [T,k], probs float64 [T,E] = the scores)."""
    l = np.ascontiguousarray(np.asarray(logits, dtype=np.float64))
    T, E = l.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    probs = np.empty((T, E), dtype=np.float64)
    sc = 1 if scoring == "sigmoid" else 0
    _load().oracle_topk_ex(T, E, k, sc, 1 if renorm else 0, _ptr(l), _ptr(idx), _ptr(w),
                           _ptr(probs))
    return idx, w, probs


def capacity(T: int, k: int, E: int, cf: float) -> int:
    """max(int(T*k/E * cf), 1), or -1 (dropless) when cf <= 0.  "How Mixture
    of Experts Works", section "The Capacity Factor"."""
    return int(_load().oracle_capacity(int(T), int(k), int(E), float(cf)))


def dispatch(topk_idx, E: int, cap: int):
    """Per-expert counts, token-order ranks, capacity drops and the stable
    permutation grouped by expert.  "How Mixture of Experts Works", MoELayer
    listing and "The Capacity Factor"; "Mixture-of-Experts Routing", capacity
    check in token (nonzero) order."""
    idx = np.ascontiguousarray(np.asarray(topk_idx, dtype=np.int32))
    T, k = idx.shape
    A = T * k
    out = dict(
        counts_pre=np.empty(E, np.int32), counts_kept=np.empty(E, np.int32),
        offsets=np.empty(E + 1, np.int32), rank=np.empty(A, np.int32),
        dest=np.empty(A, np.int32), perm_src=np.full(max(A, 1), -1, np.int32),
        drop_mask=np.empty(A, np.uint8))
    R = _load().oracle_dispatch(T, k, E, int(cap), _ptr(idx), _ptr(out["counts_pre"]),
                                _ptr(out["counts_kept"]), _ptr(out["offsets"]), _ptr(out["rank"]),
                                _ptr(out["dest"]), _ptr(out["perm_src"]), _ptr(out["drop_mask"]))
    out["perm_src"] = out["perm_src"][:R]
    out["R"] = int(R)
    return out


def expert_ffn(xv, W1, W3, W2, b1=None, b2=None, act: str = "swiglu") -> np.ndarray:
    """One expert on one token vector, in double.  GELU MLP: "Mixture-of-Experts
    Routing" (nn.GELU, erf form, with biases); SwiGLU: "Mixture of Experts
    (MoE)", section "Implementing a complete MoE layer".  W1/W3 are [F, d],
    W2 is [d, F] (nn.Linear layout)."""
    w1, c = _buf(W1)
    w3, _ = _buf(W3)
    w2, _ = _buf(W2)
    bb1, _ = _buf(b1)
    bb2, _ = _buf(b2)
    F, d = w1.shape
    x = np.ascontiguousarray(np.asarray(xv, dtype=np.float64))
    h = np.empty(F, np.float64)
    out = np.empty(d, np.float64)
    a = ORC_SWIGLU if act == "swiglu" else ORC_GELU_ERF
    _load().oracle_expert_ffn(d, F, a, c, _ptr(x), _ptr(w1), _ptr(w3), _ptr(w2),
                              _ptr(bb1), _ptr(bb2), _ptr(h), _ptr(out))
    return out


def layer_tokens(inp, topk_idx, topk_w, drop_mask, tokens, want_slots=False,
                 want_shared=False):
    """Layer output y[t] = x[t] + sum over kept slots of w * FFN_e(x[t])
    (+ shared expert) for the listed tokens.  "Mixture-of-Experts Routing"
    (weighted sum plus residual); "Mixture of Experts (MoE)", "The shared
    expert pattern".  `inp` is a workload dict (see the package's workloads
    module).  Returns dict with y [n,d] and optionally slots [n,k,d], shared
    [n,d]."""
    cfg = inp["cfg"]
    xa, c = _buf(inp["x"])
    W1, wc = _buf(inp["W1"])
    W3, _ = _buf(inp.get("W3"))
    W2, _ = _buf(inp["W2"])
    b1, _ = _buf(inp.get("b1"))
    b2, _ = _buf(inp.get("b2"))
    S1, _ = _buf(inp.get("S1"))
    S3, _ = _buf(inp.get("S3"))
    S2, _ = _buf(inp.get("S2"))
    scales = []
    for key in ("s1", "s3", "s2"):
        v = inp.get(key)
        if v is not None and wc in (ORC_E4M3, ORC_E2M1P):
            try:
                import torch
                if isinstance(v, torch.Tensor):
                    v = v.detach().cpu().float().numpy()
            except ImportError:
                pass
            scales.append(np.ascontiguousarray(np.asarray(v, dtype=np.float32)))
        else:
            scales.append(None)
    tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    n = len(tok)
    d, F, E, k = cfg["d"], cfg["F"], cfg["E"], cfg["k"]
    F_sh = cfg.get("F_shared", 0) if S1 is not None else 0
    idx = np.ascontiguousarray(np.asarray(topk_idx, dtype=np.int32))
    w = np.ascontiguousarray(np.asarray(topk_w, dtype=np.float64))
    dm = np.ascontiguousarray(np.asarray(drop_mask, dtype=np.uint8))
    y = np.empty((n, d), np.float64)
    slots = np.empty((n, k, d), np.float64) if want_slots else None
    sh = np.empty((n, d), np.float64) if (want_shared and F_sh > 0) else None
    act = ORC_SWIGLU if cfg["act"] == "swiglu" else ORC_GELU_ERF
    _load().oracle_layer_tokens_q(n, _ptr(tok), d, F, E, k, act, c, wc, _ptr(xa), _ptr(W1),
                                  _ptr(W3), _ptr(W2), _ptr(b1), _ptr(b2), _ptr(scales[0]),
                                  _ptr(scales[1]), _ptr(scales[2]), F_sh, _ptr(S1), _ptr(S3),
                                  _ptr(S2), _ptr(idx), _ptr(w), _ptr(dm), _ptr(y), _ptr(slots),
                                  _ptr(sh))
    out = {"y": y}
    if slots is not None:
        out["slots"] = slots
    if sh is not None:
        out["shared"] = sh
    return out


def aux_loss(counts_pre, probs) -> float:
    """E * sum_e f_e P_e, f_e = counts_pre[e]/T, P_e = mean_t probs[t,e].
    "How Mixture of Experts Works", "The Load Balancing Problem"; "Mixture of
    Experts (MoE)", "Load balancing and expert collapse" (alpha left out)."""
    cp = np.ascontiguousarray(np.asarray(counts_pre, dtype=np.int32))
    p = np.ascontiguousarray(np.asarray(probs, dtype=np.float64))
    T, E = p.shape
    return float(_load().oracle_aux_loss(T, E, _ptr(cp), _ptr(p)))


def layer_forward(inp, logits_in=None, tokens=None, want_slots=False, want_shared=False):
    """The whole layer: router logits (or the given ones), top-k, dispatch with
    capacity, outputs for `tokens` (default: all) and the aux loss.

    logits_in lets the oracle take the routing logits from elsewhere (e.g. the
    GPU's fp32 logits for the bit-exact routing check); the oracle's own logits
    are still returned as logits_own for the listed tokens when it is given."""
    cfg = inp["cfg"]
    T, E, k = cfg["T"], cfg["E"], cfg["k"]
    if logits_in is None:
        logits = router_logits(inp["x"], inp["Wr"], inp.get("logit_bias"))
    else:
        logits = np.asarray(logits_in, dtype=np.float64)
    idx, w, probs = topk(logits, k, cfg.get("scoring", "softmax"), cfg.get("renorm", True))
    cap = capacity(T, k, E, cfg.get("capacity_factor", 0.0))
    disp = dispatch(idx, E, cap)
    toks = np.arange(T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    lay = layer_tokens(inp, idx, w, disp["drop_mask"], toks, want_slots, want_shared)
    out = dict(logits=logits, topk_idx=idx, topk_w=w, probs=probs, cap=cap, tokens=toks, **disp, **lay)
    out["aux"] = aux_loss(disp["counts_pre"], probs)
    A = T * k
    out["drop_frac"] = (A - disp["R"]) / A if A else 0.0
    return out


def aux_grad_logits(logits, counts_pre, grad_aux=1.0, scoring="softmax"):
    """Gradient of grad_aux * aux with respect to the router logits, f_e held
    fixed (counts are piecewise constant): the chain rule through P_e, see
    oracle_aux_grad_logits.  "How Mixture of Experts Works", "The Load
    Balancing Problem" (the aux term is trained as alpha * aux)."""
    l = np.ascontiguousarray(np.asarray(logits, dtype=np.float64))
    T, E = l.shape
    cp = np.ascontiguousarray(np.asarray(counts_pre, dtype=np.int32))
    g = np.empty((T, E), np.float64)
    _load().oracle_aux_grad_logits(T, E, 1 if scoring == "sigmoid" else 0, _ptr(l), _ptr(cp),
                                   float(grad_aux), _ptr(g))
    return g


def aux_router_backward(x, Wr, logits, counts_pre, grad_aux=1.0, scoring="softmax"):
    """Router gradients of grad_aux * aux: (g_logits [T,E], g_Wr [E,d] =
    g_logits^T x, g_x [T,d] = g_logits Wr), in double; the two products are
    library matmuls of the exactly widened inputs."""
    g = aux_grad_logits(logits, counts_pre, grad_aux, scoring)
    xf = to_f64(x)
    wf = to_f64(Wr)
    return g, g.T @ xf, g @ wf
