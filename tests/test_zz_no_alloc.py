"""moe_dispatch_noalloc: dispatch for callers that cannot allocate device memory.

Such a caller passes only its inputs and outputs; the entry point keeps its
scratch in a fixed device array inside the library.  These tests call it
through the C ABI and check, on two calls in a row with different inputs, that
its outputs equal moe_dispatch's (which uses a caller-allocated workspace) bit
for bit, and that a size beyond its fixed maximum is refused.  The file sorts
last so that a run stopping at the first failure has run every other test.
"""
import numpy as np
import pytest
import torch

from sparse_mixture_experts_59_b300 import binding, workloads

pytestmark = pytest.mark.gpu
KEYS = ("counts_pre", "counts_kept", "offsets", "perm_src", "dest", "drop_mask", "stats")


def _indices(T, E, k, seed):
    g = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1) ** 1.2          # skewed load, so capacity drops happen
    p /= p.sum()
    idx = np.stack([g.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return torch.from_numpy(idx).cuda()


@pytest.mark.parametrize("T,E,k,cf", [(3000, 64, 2, 1.25), (8192, 256, 8, 0.0), (700, 8, 1, 1.0)])
def test_noalloc_dispatch_matches_workspace_dispatch_twice(T, E, k, cf):
    cfg = binding.make_config(workloads.config("mixtral_prefill", T=T, d=64, F=64, E=E, k=k,
                                               capacity_factor=cf))
    ws = binding.new_workspace(cfg)
    for call in range(2):
        idx = _indices(T, E, k, seed=T + 31 * call)
        pm = torch.rand(E, device="cuda")
        pm /= pm.sum()
        ref = binding.dispatch(cfg, idx, pm, ws=ws)
        got = binding.dispatch_noalloc(cfg, idx, pm)
        torch.cuda.synchronize()
        assert binding.device_status(ws) == 0
        assert int(got["device_status"].item()) == 0
        R = int(ref["offsets"][-1].item())
        for key in KEYS:
            a, b = got[key].cpu(), ref[key].cpu()
            if key == "perm_src":
                a, b = a[:R], b[:R]
            assert torch.equal(a, b), (call, key)


def test_noalloc_dispatch_refuses_sizes_beyond_its_scratch():
    cfg = binding.make_config(workloads.config("mixtral_prefill", T=32769, d=64, F=64, E=8, k=2))
    idx = torch.zeros(32769, 2, dtype=torch.int32, device="cuda")
    idx[:, 1] = 1
    with pytest.raises(binding.MoeError) as ei:
        binding.dispatch_noalloc(cfg, idx)
    assert ei.value.code == 1 and "65536" in str(ei.value)


def test_noalloc_dispatch_reports_a_device_error_then_recovers():
    """A call given an expert index outside [0, E) reports MOE_ERR_DEVICE_BOUNDS
    in its device_status output (the kernel leaves that assignment out of every
    count); the next call clears the shared scratch itself, returns status 0
    and matches moe_dispatch bit for bit."""
    T, E, k = 300, 8, 2
    cfg = binding.make_config(workloads.config("mixtral_prefill", T=T, d=64, F=64, E=E, k=k))
    idx = torch.randint(0, E, (T, k), dtype=torch.int32)
    idx[:, 1] = (idx[:, 0] + 1) % E
    bad = idx.clone()
    bad[17, 0] = E
    got = binding.dispatch_noalloc(cfg, bad.cuda())
    torch.cuda.synchronize()
    assert int(got["device_status"].item()) == 6          # MOE_ERR_DEVICE_BOUNDS
    assert int(got["counts_pre"].sum().item()) == T * k - 1
    ws = binding.new_workspace(cfg)
    ref = binding.dispatch(cfg, idx.cuda(), ws=ws)
    got = binding.dispatch_noalloc(cfg, idx.cuda())
    torch.cuda.synchronize()
    assert int(got["device_status"].item()) == 0
    assert binding.device_status(ws) == 0
    R = int(ref["offsets"][-1].item())
    for key in KEYS:
        a, b = got[key].cpu(), ref[key].cpu()
        if key == "perm_src":
            a, b = a[:R], b[:R]
        assert torch.equal(a, b), key
