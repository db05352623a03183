"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function include/moe.h declares, and rejects bad arguments before it touches
the device."""
import ctypes
import os
import re

import pytest

from sparse_mixture_experts_59_b300 import binding, build, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_header_declares_the_stage_calls():
    names = _declared()
    for n in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_layer_forward",
              "moe_workspace_size", "moe_workspace_init", "moe_get_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) <= set(binding.EXPORTS) | {"moe_status_string", "moe_last_error"}


def test_status_strings(lib):
    assert lib.moe_status_string(0) == b"MOE_OK"
    assert lib.moe_status_string(6) == b"MOE_ERR_DEVICE_BOUNDS"


def test_capacity_matches_formula(lib):
    assert binding.capacity(workloads.config("tiny_fp32")) == 20
    assert binding.capacity(workloads.config("switch_skewed")) == 256
    assert binding.capacity(workloads.config("mixtral_prefill")) == -1
    assert binding.capacity(dict(T=1, d=8, F=8, E=8, k=1, capacity_factor=0.5)) == 1


def test_workspace_size_grows_with_tokens(lib):
    a = binding.workspace_size(workloads.config("mixtral_prefill", T=64))
    b = binding.workspace_size(workloads.config("mixtral_prefill", T=128))
    assert 0 < a < b
    # the gathered rows, hidden rows and slot outputs dominate
    c = workloads.config("mixtral_prefill")
    A = c["T"] * c["k"]
    assert binding.workspace_size(c) >= A * (2 * c["d"] + c["F"]) * 2


@pytest.mark.parametrize("bad,code", [
    (dict(d=12), 1), (dict(F=0), 1), (dict(E=0), 1), (dict(E=300), 1), (dict(k=0), 1),
    (dict(k=9, E=16), 1), (dict(k=3, E=2), 1), (dict(T=-1), 1), (dict(F_shared=4), 1),
    (dict(act="swiglu", has_bias=True), 2), (dict(act="gelu", F_shared=64), 2),
    # weight rows past 32-bit coordinates
    (dict(E=256, F=1 << 23), 1), (dict(E=2, k=2, d=1 << 30), 1),
    # packed 4-bit weights: 128-value chunks, not with FP8 or an fp32 layer
    (dict(weight_fp4=True), 1), (dict(weight_fp4=True, d=128, F=192), 1),
    (dict(weight_fp4=True, weight_fp8=True, d=128, F=128), 1),
    (dict(weight_fp4=True, dtype="f32", d=128, F=128), 2),
])
def test_invalid_configs_are_rejected(lib, bad, code):
    cfg = workloads.config("mixtral_prefill", T=16, d=64, F=64)
    cfg.update(bad)
    with pytest.raises(binding.MoeError) as ei:
        binding.workspace_size(cfg)
    assert ei.value.code == code


def test_calls_check_arguments_before_launching(lib):
    """NULL or misaligned pointers and a short workspace come back as error
    codes from the host side (no device is touched: this runs without a GPU)."""
    c = binding.make_config(workloads.config("mixtral_prefill", T=16, d=64, F=64))
    need = binding.workspace_size(c)
    fake = ctypes.c_void_p(1 << 40)        # never dereferenced: checks fail first
    mis = ctypes.c_void_p((1 << 40) + 8)
    P = ctypes.c_void_p
    L = lib
    assert L.moe_route(ctypes.byref(c), None, fake, None, fake, fake, fake, None, fake, need, None) == 1
    assert L.moe_route(ctypes.byref(c), mis, fake, None, fake, fake, fake, None, fake, need, None) == 1
    assert L.moe_route(ctypes.byref(c), fake, fake, None, fake, fake, fake, None, fake, need - 1, None) == 3
    assert L.moe_route(ctypes.byref(c), fake, fake, None, fake, fake, fake, None, None, need, None) == 1
    w = binding.MoeWeights(W1=fake.value, W3=None, W2=fake.value)
    assert L.moe_expert_ffn(ctypes.byref(c), fake, fake, fake, fake, ctypes.byref(w), fake, None,
                            fake, need, None) == 1          # W3 missing for SwiGLU
    assert b"W3" in L.moe_last_error()
    assert L.moe_combine(ctypes.byref(c), fake, fake, None, None, fake, None) == 1
    out = binding.MoeLayerOut(y=None)
    w = binding.MoeWeights(W1=fake.value, W3=fake.value, W2=fake.value)
    assert L.moe_layer_forward(ctypes.byref(c), fake, fake, None, ctypes.byref(w), ctypes.byref(out),
                               fake, need, None) == 1       # y missing
    # T = 0 is a no-op that succeeds without touching anything
    z = binding.make_config(workloads.config("mixtral_prefill", T=0, d=64, F=64))
    nz = binding.workspace_size(z)
    assert L.moe_route(ctypes.byref(z), None, None, None, None, None, None, None, fake, nz, None) == 0
    assert L.moe_combine(ctypes.byref(z), None, None, None, None, None, None) == 0


def test_noalloc_dispatch_rejects_misaligned_pointers_before_launching(lib):
    """moe_dispatch_noalloc checks its pointers as moe_dispatch does: a NULL or
    misaligned int / float buffer returns MOE_ERR_INVALID_ARG naming it, before
    any CUDA call (the addresses below are never dereferenced)."""
    c = binding.make_config(workloads.config("mixtral_prefill", T=64, d=64, F=64, E=8, k=2))
    good = [0x100000 + 0x1000 * i for i in range(11)]
    names = ("topk_idx", "prob_mean", "counts_pre", "counts_kept", "offsets", "perm_src", "dest",
             "drop_mask", "stats", "device_status")
    for j, name in enumerate(names):
        if name == "drop_mask":
            continue                       # bytes: any address is aligned
        args = list(good[:10])
        args[j] = good[j] + 2
        rc = lib.moe_dispatch_noalloc(ctypes.byref(c), *[ctypes.c_void_p(a) for a in args], None)
        assert rc == 1, name
        assert name in lib.moe_last_error().decode(), name
    args = list(good[:10])
    args[names.index("dest")] = 0
    rc = lib.moe_dispatch_noalloc(ctypes.byref(c), *[ctypes.c_void_p(a) for a in args], None)
    assert rc == 1 and "dest" in lib.moe_last_error().decode()


def test_dispatch_rejects_misaligned_prob_mean(lib):
    c = binding.make_config(workloads.config("mixtral_prefill", T=64, d=64, F=64, E=8, k=2))
    ws_bytes = binding.workspace_size(c)
    p = [ctypes.c_void_p(0x100000 + 0x1000 * i) for i in range(10)]
    p[1] = ctypes.c_void_p(0x100000 + 0x1000 + 1)          # prob_mean
    rc = lib.moe_dispatch(ctypes.byref(c), *p[:9], ctypes.c_void_p(0x200000), ws_bytes, None)
    assert rc == 1 and "prob_mean" in lib.moe_last_error().decode()


def test_config_kernel_choice_fields_are_validated(lib):
    """gemm_kernel and route_path sit at the end of moe_cfg; out-of-range
    values are refused by name (which also shows the binding's field layout
    matches the header's)."""
    base = workloads.config("mixtral_prefill", T=64, d=64, F=64, E=8, k=2)
    for kern in ("auto", "tc1", "pair", "swap"):
        assert binding.workspace_size(dict(base, gemm_kernel=kern)) > 0
    c = binding.make_config(base)
    c.gemm_kernel = 4
    n = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(n)) == 1
    assert "gemm_kernel" in lib.moe_last_error().decode()
    c = binding.make_config(dict(base, route_path="separate"))
    assert c.route_path == 1 and lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(n)) == 0
    c.route_path = 2
    assert lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(n)) == 1
    assert "route_path" in lib.moe_last_error().decode()


def test_a_missing_library_fails_loudly(tmp_path, monkeypatch):
    """Without the built CUDA library the binding raises on the first call
    that needs it. No stage has a CPU path to fall back to."""
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "libmoe_b300.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="not found"):
        binding.lib()
    cfg = workloads.config("tiny_fp32")
    with pytest.raises(RuntimeError, match="not found"):
        binding.capacity(binding.make_config(cfg))
    with pytest.raises(RuntimeError, match="not found"):
        binding.workspace_size(binding.make_config(cfg))
