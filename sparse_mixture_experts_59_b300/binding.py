"""ctypes binding of the C ABI in include/moe.h.

Argument marshalling only: every stage runs in the CUDA kernels of
libmoe_b300.so.  torch supplies device memory and the current stream.  The
library is loaded on first use; if it is missing the call raises -- there is
no other implementation to fall back to.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_F32, MOE_BF16 = 0, 1
MOE_GELU_ERF, MOE_SWIGLU = 0, 1
MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_TIMEOUT", 6: "MOE_ERR_DEVICE_BOUNDS",
          7: "MOE_ERR_NO_DEVICE"}
EXPORTS = ("moe_status_string", "moe_last_error", "moe_capacity", "moe_workspace_size",
           "moe_workspace_init", "moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine",
           "moe_layer_forward", "moe_layer_forward_profiled", "moe_get_device_status",
           "moe_dispatch_noalloc", "moe_test_hold_lookback_block", "moe_test_hold_gemm_stage",
           "moe_aux_loss_backward")


class MoeError(RuntimeError):
    def __init__(self, code, detail=""):
        self.code = code
        super().__init__("%s%s" % (STATUS.get(code, "MOE_ERR_%d" % code),
                                   (": " + detail) if detail else ""))


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("F", ctypes.c_int),
                ("E", ctypes.c_int), ("k", ctypes.c_int), ("F_shared", ctypes.c_int),
                ("dtype", ctypes.c_int), ("act", ctypes.c_int), ("has_bias", ctypes.c_int),
                ("capacity_factor", ctypes.c_float), ("scoring", ctypes.c_int),
                ("no_renorm", ctypes.c_int), ("weight_fp8", ctypes.c_int),
                ("weight_fp4", ctypes.c_int), ("gemm_kernel", ctypes.c_int),
                ("route_path", ctypes.c_int)]


GEMM_KERNELS = {"auto": 0, "tc1": 1, "pair": 2, "swap": 3}
ROUTE_PATHS = {"auto": 0, "separate": 1}


WEIGHT_KEYS = ("W1", "W3", "W2", "b1", "b2", "S1", "S3", "S2", "s1", "s3", "s2")


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_KEYS]


class MoeLayerOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("y", "logits", "topk_idx", "topk_w", "counts_pre",
                                               "counts_kept", "drop_mask", "stats")]


_lib = None


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmoe_b300.so not found at %s; build it with "
                               "`python -m sparse_mixture_experts_59_b300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [I]
        L.moe_last_error.restype = ctypes.c_char_p
        L.moe_last_error.argtypes = []
        L.moe_capacity.restype = ctypes.c_longlong
        L.moe_capacity.argtypes = [P]
        L.moe_workspace_size.argtypes = [P, ctypes.POINTER(S)]
        L.moe_workspace_init.argtypes = [P, P, S, P]
        L.moe_route.argtypes = [P, P, P, P, P, P, P, P, P, S, P]
        L.moe_dispatch.argtypes = [P, P, P, P, P, P, P, P, P, P, P, S, P]
        L.moe_expert_ffn.argtypes = [P, P, P, P, P, P, P, P, P, S, P]
        L.moe_combine.argtypes = [P, P, P, P, P, P, P]
        L.moe_layer_forward.argtypes = [P, P, P, P, P, P, P, S, P]
        L.moe_layer_forward_profiled.argtypes = [P, P, P, P, P, P, P, S, P, P]
        L.moe_get_device_status.argtypes = [P, S, P, ctypes.POINTER(I)]
        L.moe_dispatch_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P]
        L.moe_test_hold_lookback_block.argtypes = [P, S, I, P]
        L.moe_test_hold_gemm_stage.argtypes = [P, S, I, P]
        L.moe_aux_loss_backward.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, P, P]
        for name in EXPORTS:
            getattr(L, name).restype = getattr(L, name).restype or I
        _lib = L
    return _lib


def _check(rc):
    if rc != 0:
        raise MoeError(rc, lib().moe_last_error().decode(errors="replace"))


def make_config(cfg: dict) -> MoeConfig:
    """C config from a workload dict (keys T, d, F, E, k, act, dtype, ...;
    optional gemm_kernel "auto" | "tc1" | "pair" | "swap" and route_path
    "auto" | "separate")."""
    return MoeConfig(
        T=int(cfg["T"]), d=int(cfg["d"]), F=int(cfg["F"]), E=int(cfg["E"]), k=int(cfg["k"]),
        F_shared=int(cfg.get("F_shared", 0) or 0),
        dtype=MOE_F32 if cfg.get("dtype", "bf16") in ("f32", torch.float32) else MOE_BF16,
        act=MOE_SWIGLU if cfg.get("act", "swiglu") == "swiglu" else MOE_GELU_ERF,
        has_bias=int(bool(cfg.get("has_bias", False))),
        capacity_factor=float(cfg.get("capacity_factor", 0.0) or 0.0),
        scoring=MOE_SCORE_SIGMOID if cfg.get("scoring", "softmax") == "sigmoid" else MOE_SCORE_SOFTMAX,
        no_renorm=0 if cfg.get("renorm", True) else 1,
        weight_fp8=int(bool(cfg.get("weight_fp8", False))),
        weight_fp4=int(bool(cfg.get("weight_fp4", False))),
        gemm_kernel=GEMM_KERNELS[cfg.get("gemm_kernel", "auto") or "auto"],
        route_path=ROUTE_PATHS[cfg.get("route_path", "auto") or "auto"])


def _p(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def capacity(cfg) -> int:
    c = cfg if isinstance(cfg, MoeConfig) else make_config(cfg)
    return int(lib().moe_capacity(ctypes.byref(c)))


def workspace_size(cfg) -> int:
    c = cfg if isinstance(cfg, MoeConfig) else make_config(cfg)
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(c), ctypes.byref(n)))
    return int(n.value)


def new_workspace(cfg, device="cuda"):
    """A zero-initialised workspace tensor for `cfg` (allocated by torch)."""
    c = cfg if isinstance(cfg, MoeConfig) else make_config(cfg)
    ws = torch.zeros(max(workspace_size(c), 256), dtype=torch.uint8, device=device)
    _check(lib().moe_workspace_init(ctypes.byref(c), _p(ws), ws.numel(), _stream()))
    return ws


def _weights_struct(w: dict) -> MoeWeights:
    return MoeWeights(*[None if w.get(n) is None else w[n].data_ptr() for n in WEIGHT_KEYS])


def route(cfg, x, Wr, logit_bias=None, ws=None, stream=None):
    """moe_route: logits [T,E] fp32, topk_idx [T,k] int32, topk_w [T,k] fp32,
    prob_mean [E] fp32."""
    c = cfg if isinstance(cfg, MoeConfig) else make_config(cfg)
    dev = x.device
    ws = ws if ws is not None else new_workspace(c, dev)
    out = dict(logits=torch.empty(c.T, c.E, dtype=torch.float32, device=dev),
               topk_idx=torch.empty(c.T, c.k, dtype=torch.int32, device=dev),
               topk_w=torch.empty(c.T, c.k, dtype=torch.float32, device=dev),
               prob_mean=torch.empty(c.E, dtype=torch.float32, device=dev))
    _check(lib().moe_route(ctypes.byref(c), _p(x), _p(Wr), _p(logit_bias), _p(out["logits"]),
                           _p(out["topk_idx"]), _p(out["topk_w"]), _p(out["prob_mean"]),
                           _p(ws), ws.numel(), _stream(stream)))
    return out


def dispatch(cfg, topk_idx, prob_mean=None, ws=None, stream=None):
    """moe_dispatch: counts_pre, counts_kept [E], offsets [E+1], perm_src, dest,
    drop_mask [T*k], stats [2] (aux loss, dropped fraction)."""
    c = cfg if isinstance(cfg, MoeConfig) else make_config(cfg)
    dev = topk_idx.device
    ws = ws if ws is not None else new_workspace(c, dev)
    A = c.T * c.k
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(counts_pre=torch.empty(c.E, **i32), counts_kept=torch.empty(c.E, **i32),
               offsets=torch.empty(c.E + 1, **i32), perm_src=torch.full((max(A, 1),), -1, **i32),
               dest=torch.empty(max(A, 1), **i32),
               drop_mask=torch.empty(max(A, 1), dtype=torch.uint8, device=dev),
               stats=torch.zeros(2, dtype=torch.float32, device=dev))
    _check(lib().moe_dispatch(ctypes.byref(c), _p(topk_idx), _p(prob_mean), _p(out["counts_pre"]),
                              _p(out["counts_kept"]), _p(out["offsets"]), _p(out["perm_src"]),
                              _p(out["dest"]), _p(out["drop_mask"]),
                              _p(out["stats"]) if prob_mean is not None else None,
                              _p(ws), ws.numel(), _stream(stream)))
    return out


def dispatch_noalloc(cfg, topk_idx, prob_mean=None, stream=None):
    """moe_dispatch_noalloc: the outputs of dispatch() plus device_status [1]
    int32, with no workspace (the library's fixed scratch array is used;
    T*k <= 65536)."""
    c = cfg if isinstance(cfg, MoeConfig) else make_config(cfg)
    dev = topk_idx.device
    A = c.T * c.k
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(counts_pre=torch.empty(c.E, **i32), counts_kept=torch.empty(c.E, **i32),
               offsets=torch.empty(c.E + 1, **i32), perm_src=torch.full((max(A, 1),), -1, **i32),
               dest=torch.empty(max(A, 1), **i32),
               drop_mask=torch.empty(max(A, 1), dtype=torch.uint8, device=dev),
               stats=torch.zeros(2, dtype=torch.float32, device=dev),
               device_status=torch.full((1,), -1, **i32))
    _check(lib().moe_dispatch_noalloc(ctypes.byref(c), _p(topk_idx), _p(prob_mean),
                                      _p(out["counts_pre"]), _p(out["counts_kept"]),
                                      _p(out["offsets"]), _p(out["perm_src"]), _p(out["dest"]),
                                      _p(out["drop_mask"]),
                                      _p(out["stats"]) if prob_mean is not None else None,
                                      _p(out["device_status"]), _stream(stream)))
    return out


def expert_ffn(cfg, x, perm_src, offsets, topk_w, weights: dict, ws=None, stream=None):
    """moe_expert_ffn: Ys [T*k, d] (rows of dropped slots unwritten) and the
    shared expert's output [T, d] (None without one)."""
    c = cfg if isinstance(cfg, MoeConfig) else make_config(cfg)
    dev = x.device
    ws = ws if ws is not None else new_workspace(c, dev)
    Ys = torch.zeros(max(c.T * c.k, 1), c.d, dtype=x.dtype, device=dev)
    Sh = torch.empty(c.T, c.d, dtype=x.dtype, device=dev) if c.F_shared > 0 else None
    w = _weights_struct(weights)
    _check(lib().moe_expert_ffn(ctypes.byref(c), _p(x), _p(perm_src), _p(offsets), _p(topk_w),
                                ctypes.byref(w), _p(Ys), _p(Sh), _p(ws), ws.numel(),
                                _stream(stream)))
    return Ys, Sh


def combine(cfg, x, Ys, drop_mask, shared_out=None, stream=None):
    """moe_combine: y [T, d]."""
    c = cfg if isinstance(cfg, MoeConfig) else make_config(cfg)
    y = torch.empty_like(x)
    _check(lib().moe_combine(ctypes.byref(c), _p(x), _p(Ys), _p(drop_mask), _p(shared_out), _p(y),
                             _stream(stream)))
    return y


def layer_forward(cfg, x, Wr, weights: dict, logit_bias=None, ws=None, outputs=None,
                  want=("y",), stream=None, events=None):
    """moe_layer_forward.  `want` names the outputs to return besides y (logits,
    topk_idx, topk_w, counts_pre, counts_kept, drop_mask, stats); `outputs` may
    pass preallocated tensors for any of them.  `events`: seven recorded-once
    torch.cuda.Event(enable_timing=True) objects to be recorded at the stage
    boundaries (moe_layer_forward_profiled)."""
    c = cfg if isinstance(cfg, MoeConfig) else make_config(cfg)
    dev = x.device
    ws = ws if ws is not None else new_workspace(c, dev)
    o = dict(outputs or {})
    A = c.T * c.k
    shapes = dict(logits=((c.T, c.E), torch.float32), topk_idx=((c.T, c.k), torch.int32),
                  topk_w=((c.T, c.k), torch.float32), counts_pre=((c.E,), torch.int32),
                  counts_kept=((c.E,), torch.int32), drop_mask=((max(A, 1),), torch.uint8),
                  stats=((2,), torch.float32))
    if "y" not in o:
        o["y"] = torch.empty_like(x)
    for name in want:
        if name != "y" and name not in o:
            shp, dt = shapes[name]
            o[name] = torch.empty(shp, dtype=dt, device=dev)
    out_s = MoeLayerOut(*[None if o.get(n) is None else o[n].data_ptr()
                          for n in ("y", "logits", "topk_idx", "topk_w", "counts_pre",
                                    "counts_kept", "drop_mask", "stats")])
    w = _weights_struct(weights)
    if events is None:
        _check(lib().moe_layer_forward(ctypes.byref(c), _p(x), _p(Wr), _p(logit_bias),
                                       ctypes.byref(w), ctypes.byref(out_s), _p(ws), ws.numel(),
                                       _stream(stream)))
    else:
        ev = (ctypes.c_void_p * 7)(*[e.cuda_event for e in events])
        _check(lib().moe_layer_forward_profiled(ctypes.byref(c), _p(x), _p(Wr), _p(logit_bias),
                                                ctypes.byref(w), ctypes.byref(out_s), _p(ws),
                                                ws.numel(), _stream(stream), ev))
    return o


def aux_loss_backward(cfg, x, Wr, logits, counts_pre, grad_aux=1.0, want_Wr=True, want_x=True,
                      stream=None):
    """moe_aux_loss_backward: router gradients of grad_aux * aux.  Returns
    dict(grad_logits [T,E], grad_Wr [E,d] or None, grad_x [T,d] or None),
    all fp32."""
    c = cfg if isinstance(cfg, MoeConfig) else make_config(cfg)
    dev = logits.device
    out = dict(grad_logits=torch.empty(c.T, c.E, dtype=torch.float32, device=dev),
               grad_Wr=torch.empty(c.E, c.d, dtype=torch.float32, device=dev) if want_Wr else None,
               grad_x=torch.empty(c.T, c.d, dtype=torch.float32, device=dev) if want_x else None)
    _check(lib().moe_aux_loss_backward(ctypes.byref(c), _p(x), _p(Wr), _p(logits), _p(counts_pre),
                                       float(grad_aux), _p(out["grad_logits"]), _p(out["grad_Wr"]),
                                       _p(out["grad_x"]), _stream(stream)))
    return out


def test_hold_lookback_block(ws, block, stream=None):
    """Test hook: the next dispatch on `ws` runs with look-back block `block`
    never publishing, so later blocks time out (MOE_ERR_DEVICE_TIMEOUT)."""
    _check(lib().moe_test_hold_lookback_block(_p(ws), ws.numel(), int(block), _stream(stream)))


def test_hold_gemm_stage(ws, iteration, stream=None):
    """Test hook: from the next layer call on `ws`, the up-projection GEMM's
    weight producer stops before ring iteration `iteration`, so the kernel's
    bounded waits run out (MOE_ERR_DEVICE_TIMEOUT) until the workspace is
    re-initialised."""
    _check(lib().moe_test_hold_gemm_stage(_p(ws), ws.numel(), int(iteration), _stream(stream)))


def device_status(ws, stream=None) -> int:
    """The workspace's device status word (synchronises the stream)."""
    v = ctypes.c_int(0)
    _check(lib().moe_get_device_status(_p(ws), ws.numel(), _stream(stream), ctypes.byref(v)))
    return int(v.value)


class MoeLayer:
    """A layer bound to its weights and a workspace: forward(x) -> dict."""

    def __init__(self, cfg: dict, weights: dict, device="cuda"):
        self.cfg = dict(cfg)
        self.c = make_config(cfg)
        self.weights = weights
        self.ws = new_workspace(self.c, device)

    def forward(self, x, want=("y",), outputs=None, stream=None, events=None):
        assert x.shape[0] == self.c.T, "layer was built for T=%d tokens" % self.c.T
        return layer_forward(self.c, x, self.weights["Wr"], self.weights,
                             logit_bias=self.weights.get("logit_bias"), ws=self.ws,
                             outputs=outputs, want=want, stream=stream, events=events)
