"""Seeded synthetic inputs for the MoE layer workloads.

This module is shared by the CUDA path's tests/bench and by the CPU oracle.  It
draws random numbers and lays out tensors; it holds none of the method's
arithmetic (no routing, no expert maths).

Weight layout is the nn.Linear one used by the pages' listings:
  Wr [E, d]      router ("gate") weight, no bias
  W1 [E, F, d]   SwiGLU gate projection, or the GELU MLP's first Linear
  W3 [E, F, d]   SwiGLU up projection (None for GELU)
  W2 [E, d, F]   down projection / second Linear
  b1 [E, F], b2 [E, d]   GELU MLP biases (None for SwiGLU)
  S1, S3 [F_sh, d], S2 [d, F_sh]   shared SwiGLU expert (fine-grained workload)
  logit_bias [E] fp32    fixed per-expert router-logit offset (skewed workload)

Workloads (sizes from the pages' Mixtral / DeepSeek-V3 / Switch descriptions):
  tiny_fp32        T=64  d=128  E=8   k=2 GELU(erf)+biases, cf 1.25, fp32
  mixtral_prefill  T=4096 d=4096 F=14336 E=8 k=2 SwiGLU, dropless, bf16
  mixtral_decode   same weights, T=32
  fine_grained     T=8192 d=7168 F=2048 E=256 k=8 SwiGLU + shared F=2048, bf16
  switch_skewed    T=16384 d=2048 F=8192 E=64 k=1 GELU+biases, cf 1.0, bf16,
                   logit bias b_e = 1.5*ln(1/(e+1)^1.2)
"""
import math

import torch

WORKLOADS = {
    "tiny_fp32": dict(T=64, d=128, F=256, E=8, k=2, act="gelu", has_bias=True,
                      dtype="f32", capacity_factor=1.25, F_shared=0, seed=1000,
                      init="uniform", router_scale=4.0, router_init="uniform", skew=False),
    "mixtral_prefill": dict(T=4096, d=4096, F=14336, E=8, k=2, act="swiglu", has_bias=False,
                            dtype="bf16", capacity_factor=0.0, F_shared=0, seed=1001,
                            init="normal", router_scale=1.0, router_init="normal", skew=False),
    "mixtral_decode": dict(T=32, d=4096, F=14336, E=8, k=2, act="swiglu", has_bias=False,
                           dtype="bf16", capacity_factor=0.0, F_shared=0, seed=1002,
                           weight_seed=1001, init="normal", router_scale=1.0,
                           router_init="normal", skew=False),
    "fine_grained": dict(T=8192, d=7168, F=2048, E=256, k=8, act="swiglu", has_bias=False,
                         dtype="bf16", capacity_factor=0.0, F_shared=2048, seed=1003,
                         init="normal", router_scale=1.0, router_init="normal", skew=False),
    "switch_skewed": dict(T=16384, d=2048, F=8192, E=64, k=1, act="gelu", has_bias=True,
                          dtype="bf16", capacity_factor=1.0, F_shared=0, seed=1004,
                          init="uniform", router_scale=1.0, router_init="normal", skew=True),
}

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def config(name: str, **overrides) -> dict:
    """The named workload's configuration, with optional size overrides (the
    parity tests use scaled-down copies that keep the structure)."""
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    cfg["name"] = name
    return cfg


def skew_bias(E: int) -> torch.Tensor:
    """Fixed per-expert logit offset b_e = 1.5*ln(1/rank_e^1.2), rank_e = e+1
    (expert 0 is the hottest), giving a Zipf-like load."""
    return torch.tensor([1.5 * math.log(1.0 / (e + 1) ** 1.2) for e in range(E)],
                        dtype=torch.float32)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, g, device, dtype, chunk_rows=None):
    """N(0, std^2) drawn in fp32 and rounded once to `dtype`; drawn in chunks
    along dim 0 to bound the fp32 temporary."""
    out = torch.empty(shape, dtype=dtype, device=device)
    n0 = shape[0]
    step = chunk_rows or n0
    for i in range(0, n0, step):
        sl = out[i:i + step]
        tmp = torch.randn(sl.shape, generator=g, device=device, dtype=torch.float32)
        sl.copy_(tmp.mul_(std))
    return out


def _uniform(shape, bound, g, device, dtype, chunk_rows=None):
    out = torch.empty(shape, dtype=dtype, device=device)
    n0 = shape[0]
    step = chunk_rows or n0
    for i in range(0, n0, step):
        sl = out[i:i + step]
        tmp = torch.rand(sl.shape, generator=g, device=device, dtype=torch.float32)
        sl.copy_(tmp.mul_(2.0 * bound).sub_(bound))
    return out


def make_weights(cfg: dict, device="cpu") -> dict:
    """Expert, router and shared-expert weights for `cfg`, seeded by
    cfg['weight_seed'] (default cfg['seed'])."""
    d, F, E = cfg["d"], cfg["F"], cfg["E"]
    dt = _TORCH_DTYPE[cfg["dtype"]]
    g = _gen(cfg.get("weight_seed", cfg["seed"]) * 7919 + 17, device)
    w = {}
    # router
    if cfg["router_init"] == "uniform":
        w["Wr"] = _uniform((E, d), 1.0 / math.sqrt(d), g, device, torch.float32)
    else:
        w["Wr"] = _normal((E, d), 1.0 / math.sqrt(d), g, device, torch.float32)
    if cfg.get("router_scale", 1.0) != 1.0:
        w["Wr"].mul_(cfg["router_scale"])
    w["Wr"] = w["Wr"].to(dt)
    # experts
    if cfg["init"] == "uniform":   # nn.Linear default: U(+-1/sqrt(fan_in))
        w["W1"] = _uniform((E, F, d), 1.0 / math.sqrt(d), g, device, dt, 1)
        w["W2"] = _uniform((E, d, F), 1.0 / math.sqrt(F), g, device, dt, 1)
        w["W3"] = (_uniform((E, F, d), 1.0 / math.sqrt(d), g, device, dt, 1)
                   if cfg["act"] == "swiglu" else None)
        if cfg["has_bias"]:
            w["b1"] = _uniform((E, F), 1.0 / math.sqrt(d), g, device, dt)
            w["b2"] = _uniform((E, d), 1.0 / math.sqrt(F), g, device, dt)
    else:
        w["W1"] = _normal((E, F, d), 0.02, g, device, dt, 1)
        w["W3"] = _normal((E, F, d), 0.02, g, device, dt, 1) if cfg["act"] == "swiglu" else None
        w["W2"] = _normal((E, d, F), 0.02, g, device, dt, 1)
        if cfg["has_bias"]:
            w["b1"] = _normal((E, F), 0.02, g, device, dt)
            w["b2"] = _normal((E, d), 0.02, g, device, dt)
    if not cfg["has_bias"]:
        w["b1"] = None
        w["b2"] = None
    Fs = cfg.get("F_shared", 0)
    if Fs:
        w["S1"] = _normal((Fs, d), 0.02, g, device, dt)
        w["S3"] = _normal((Fs, d), 0.02, g, device, dt)
        w["S2"] = _normal((d, Fs), 0.02, g, device, dt)
    else:
        w["S1"] = w["S3"] = w["S2"] = None
    w["logit_bias"] = skew_bias(E).to(device) if cfg.get("skew") else None
    return w


def make_x(cfg: dict, device="cpu") -> torch.Tensor:
    """Token activations x ~ N(0, 1) [T, d], seeded by cfg['seed']."""
    g = _gen(cfg["seed"], device)
    return _normal((cfg["T"], cfg["d"]), 1.0, g, device, _TORCH_DTYPE[cfg["dtype"]])


def make_inputs(name_or_cfg, device="cpu", **overrides) -> dict:
    """All inputs of one workload as a dict: cfg, x, Wr, logit_bias, W1, W3,
    W2, b1, b2, S1, S3, S2."""
    cfg = config(name_or_cfg, **overrides) if isinstance(name_or_cfg, str) else dict(name_or_cfg)
    inp = make_weights(cfg, device)
    inp["x"] = make_x(cfg, device)
    inp["cfg"] = cfg
    return inp


def to_device(inp: dict, device) -> dict:
    """Copy of a workload dict with every tensor moved to `device`."""
    out = {}
    for key, v in inp.items():
        out[key] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out


FP8_MAX = 448.0     # largest finite E4M3 magnitude


def quantize_experts_fp8(inp: dict) -> dict:
    """Copy of a workload whose routed expert weights W1, W3, W2 are FP8 E4M3
    codes with one fp32 scale per output row (s1, s3 [E,F], s2 [E,d]):
    s = max|row| / 448 and code = E4M3(w / s), rounded to nearest-even by
    torch's float8_e4m3fn conversion.  The dequantised weights are code * s.
    Sets cfg['weight_fp8'].  Input preparation only, like drawing the weights."""
    out = dict(inp)
    cfg = dict(inp["cfg"])
    cfg["weight_fp8"] = True
    out["cfg"] = cfg
    for key, skey in (("W1", "s1"), ("W3", "s3"), ("W2", "s2")):
        w = inp.get(key)
        if w is None:
            out[key] = None
            out[skey] = None
            continue
        codes = torch.empty(w.shape, dtype=torch.float8_e4m3fn, device=w.device)
        scales = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
        for e in range(w.shape[0]):          # one expert at a time bounds the fp32 temporary
            wf = w[e].float()
            sc = wf.abs().amax(dim=-1) / FP8_MAX
            sc = torch.where(sc > 0, sc, torch.ones_like(sc))
            scales[e] = sc
            codes[e] = (wf / sc[:, None]).to(torch.float8_e4m3fn)
        out[key] = codes
        out[skey] = scales
    return out


def dequantize_experts_fp8(inp: dict) -> dict:
    """fp32 copy of code * scale for each FP8 expert weight of `inp` (exact:
    an E4M3 value times an fp32 scale is one fp32 rounding away at most, and
    none at all when the product is representable; the oracle takes these
    fp32 values as the weights)."""
    out = dict(inp)
    for key, skey in (("W1", "s1"), ("W3", "s3"), ("W2", "s2")):
        if inp.get(key) is not None:
            out[key] = inp[key].float() * inp[skey][..., None]
    return out


FP4_MAX = 6.0       # largest E2M1 magnitude
FP4_CHUNK = 128     # values per packed chunk: 64 code bytes + 8 E4M3 block scales + 8 zero bytes
FP4_CHUNK_BYTES = 80


def _e2m1_round(q: torch.Tensor) -> torch.Tensor:
    """E2M1 codes (sign bit 3, magnitude index 0..7 for 0, .5, 1, 1.5, 2, 3,
    4, 6) of q, |q| <= 6, rounded to nearest with ties to the even mantissa."""
    a = q.abs()
    idx = ((a > 0.25).to(torch.uint8) + (a >= 0.75).to(torch.uint8) + (a > 1.25).to(torch.uint8)
           + (a >= 1.75).to(torch.uint8) + (a > 2.5).to(torch.uint8) + (a >= 3.5).to(torch.uint8)
           + (a > 5.0).to(torch.uint8))
    return idx | ((q < 0).to(torch.uint8) << 3)


def quantize_rows_fp4(w: torch.Tensor):
    """One [R, K] weight matrix (K a multiple of 128) -> (packed uint8
    [R, K/128 * 80], row scales fp32 [R]).  Row scale s = max|row| / (6*448);
    block scale b (E4M3, per 16 values) = E4M3(max|block| / (6 s)), rounded to
    nearest even; code = E2M1(w / (b s)) saturated to +-6.  Stored value of an
    element: code * b, times s."""
    R, K = w.shape
    assert K % FP4_CHUNK == 0, "4-bit weights need rows of a multiple of 128 values"
    wf = w.float()
    rs = wf.abs().amax(dim=1) / (FP4_MAX * FP8_MAX)
    rs = torch.where(rs > 0, rs, torch.ones_like(rs))
    wb = wf.view(R, K // 16, 16)
    bs_code = (wb.abs().amax(dim=2) / (FP4_MAX * rs[:, None])).to(torch.float8_e4m3fn)
    denom = bs_code.float() * rs[:, None]
    q = torch.where(denom[..., None] > 0, wb / denom[..., None], torch.zeros_like(wb))
    codes = _e2m1_round(q.clamp(-FP4_MAX, FP4_MAX)).view(R, K // FP4_CHUNK, FP4_CHUNK)
    packed = torch.zeros(R, K // FP4_CHUNK, FP4_CHUNK_BYTES, dtype=torch.uint8, device=w.device)
    packed[:, :, :64] = codes[:, :, 0::2] | (codes[:, :, 1::2] << 4)
    packed[:, :, 64:72] = bs_code.view(torch.uint8).view(R, K // FP4_CHUNK, 8)
    return packed.view(R, -1), rs


def quantize_experts_fp4(inp: dict) -> dict:
    """Copy of a workload whose routed expert weights W1, W3, W2 are packed
    4-bit weights (E2M1 codes with E4M3 scales per 16 values, see
    quantize_rows_fp4) with one fp32 scale per output row (s1, s3 [E,F],
    s2 [E,d]).  Sets cfg['weight_fp4'].  Input preparation only."""
    out = dict(inp)
    cfg = dict(inp["cfg"])
    cfg["weight_fp4"] = True
    out["cfg"] = cfg
    for key, skey in (("W1", "s1"), ("W3", "s3"), ("W2", "s2")):
        w = inp.get(key)
        if w is None:
            out[key] = None
            out[skey] = None
            continue
        E, R, K = w.shape
        packed = torch.empty(E, R, K // FP4_CHUNK * FP4_CHUNK_BYTES, dtype=torch.uint8,
                             device=w.device)
        scales = torch.empty(E, R, dtype=torch.float32, device=w.device)
        for e in range(E):                   # one expert at a time bounds the fp32 temporaries
            packed[e], scales[e] = quantize_rows_fp4(w[e])
        out[key] = packed
        out[skey] = scales
    return out


def dequantize_rows_fp4(packed: torch.Tensor, rs: torch.Tensor) -> torch.Tensor:
    """float64 [R, K] of a packed 4-bit matrix: code value * block scale * row
    scale, each factor exact in float64."""
    R = packed.shape[0]
    chunks = packed.view(R, -1, FP4_CHUNK_BYTES).to(torch.int64)
    lo, hi = chunks[:, :, :64] & 15, chunks[:, :, :64] >> 4
    codes = torch.stack([lo, hi], dim=3).view(R, -1, FP4_CHUNK)
    mag = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float64,
                       device=packed.device)
    vals = mag[codes & 7] * torch.where(codes >= 8, -1.0, 1.0).to(torch.float64)
    bs = chunks[:, :, 64:72].to(torch.uint8).contiguous().view(torch.float8_e4m3fn).double()
    vals = vals.view(R, -1, 8, 16) * bs[..., None]
    return vals.view(R, -1) * rs.double()[:, None]
