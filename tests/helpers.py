"""Shared helpers for the GPU parity tests: device weights from the seeded
generator, their host copies for the oracle, and the tolerance rule."""
import numpy as np
import torch

from moe_expert_nvfp4_gb300 import ops, synth

# |gpu - ref| <= 8e-3 |ref| + 2e-3 rms(ref), rms over the whole output of a call
REL_TOL = 8e-3
RMS_TOL = 2e-3


def tolerance_violations(gpu, ref):
    """Return (number of violating elements, worst ratio err / allowed)."""
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(r * r)))
    allowed = REL_TOL * np.abs(r) + RMS_TOL * rms
    err = np.abs(g - r)
    bad = ~(err <= allowed)
    ratio = float(np.max(err / np.maximum(allowed, 1e-300)))
    return int(bad.sum()), ratio


def assert_close(gpu, ref, what=""):
    n, ratio = tolerance_violations(gpu, ref)
    assert n == 0, f"{what}: {n} elements outside tolerance (worst {ratio:.3f}x allowed)"
    return ratio


def device_weight(seed, n, k, *ids, device="cuda"):
    """(ops.NVFP4Weight on device, (codes, scales, g) on host) of one matrix."""
    c, s = synth.nvfp4_weight(seed, n, k, *ids, device=device)
    g = torch.full((1,), synth.GLOBAL_SCALE, dtype=torch.float32, device=device)
    return ops.NVFP4Weight(c, s, g)


def host_weight(seed, n, k, *ids, row_lo=0, row_hi=None):
    c, s = synth.nvfp4_weight(seed, n, k, *ids, row_lo=row_lo, row_hi=row_hi)
    return c.numpy(), s.numpy(), synth.GLOBAL_SCALE


def device_experts(seed, layer, num_experts, hidden, inter, device="cuda"):
    gc, gs, dc, ds = synth.expert_stack(seed, layer, range(num_experts), hidden, inter, device)
    g = torch.full((num_experts,), synth.GLOBAL_SCALE, dtype=torch.float32, device=device)
    return ops.ExpertStack(gc, gs, dc, ds, g, g.clone())


def device_shared(seed, layer, num_experts, hidden, inter, device="cuda"):
    gc, gs, dc, ds = synth.expert_stack(seed, layer, [num_experts], hidden, inter, device)
    g = torch.full((1,), synth.GLOBAL_SCALE, dtype=torch.float32, device=device)
    return ops.ExpertStack(gc, gs, dc, ds, g, g.clone())


def host_expert_fn(seed, layer, hidden, inter):
    cache = {}

    def get(e):
        if e not in cache:
            cache[e] = synth.expert_host(seed, layer, e, hidden, inter)
        return cache[e]
    return get


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()
