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


# ------------------------------------------------------------------ argmax

# Relative error allowed between the kernel's FP32 logit (before its one BF16
# rounding) and the float64 logit.  The kernel sums K <= 4096 exact products
# in FP32; rounding errors of random sign over K additions amount to about
# 2^-19 of a logit, so 2^-16 is a wide margin that is still 2^-8 below one
# BF16 step: a flip across a real BF16 gap is not tolerated.
ARGMAX_FP32_REL = 2.0 ** -16


def _bf16_roundings(v, rel):
    """The BF16 values a number within rel * |v| of v can round to (the two
    ends of the interval bound them: rounding is monotone)."""
    lo = v - rel * abs(v)
    hi = v + rel * abs(v)
    import oracle as O
    return float(O.bf16_round(np.array([lo]))[0]), float(O.bf16_round(np.array([hi]))[0])


def check_argmax(ids, gpu_logits, ref64, id_map=None, what="argmax"):
    """Argmax of BF16 logits, ties to the lowest index.

    * ids must equal the first maximum of the GPU's own BF16 logits, exactly;
    * where they differ from the first maximum of the oracle's BF16 logits
      (float64 rounded once), both disputed logits written by the GPU must be
      a BF16 rounding of a value within ARGMAX_FP32_REL of the float64 logit:
      the float64 logit then straddles a BF16 rounding boundary by less than
      the FP32 accumulation error, the only case where the two sides may
      rightly differ.

    id_map: the reported ids are id_map[column] (hot-vocabulary head).
    Returns the number of rows tolerated under the second rule (also
    reported as a warning)."""
    import warnings

    import oracle as O
    ids = np.asarray(ids)
    gl = np.asarray(gpu_logits, dtype=np.float64)
    ref64 = np.asarray(ref64, dtype=np.float64)
    own = O.argmax_first(gl, axis=1)
    mapped = own if id_map is None else np.asarray(id_map)[own]
    assert np.array_equal(ids, mapped), f"{what}: ids differ from the GPU's own logits' argmax"
    ref_col = O.argmax_first(O.bf16_round(ref64), axis=1)
    tolerated = 0
    for r in np.nonzero(own != ref_col)[0]:
        for col in (own[r], ref_col[r]):
            lo, hi = _bf16_roundings(ref64[r, col], ARGMAX_FP32_REL)
            assert lo <= gl[r, col] <= hi, (
                f"{what}: row {r} col {col}: GPU logit {gl[r, col]!r} is not a rounding of "
                f"{ref64[r, col]!r} within the FP32 accumulation error")
        tolerated += 1
    if tolerated:
        warnings.warn(f"{what}: {tolerated} row(s) whose top-1 pair straddles a BF16 rounding "
                      f"boundary within FP32 accumulation error")
    return tolerated


# ------------------------------------------------------------------ routing

def route_weight_bound(logits, ids, k, renormalize=True):
    """Per-element bound on the relative error of the GPU's FP32 routing
    weights against float64, for float32 logits:
      - l - l_max rounds once in FP32: exp's argument moves by at most
        2^-24 |l - l_max|, a relative change of the same size;
      - expf: within 2 ulp (2 * 2^-23);
      - the FP32 sum of n terms: at most (n - 1) 2^-24 of the sum;
      - the division: 2^-24.
    A weight divides one exp by the sum, so the two exps' argument errors
    (its own and the largest in the sum) and their expf errors add up."""
    lg = np.asarray(logits, dtype=np.float64)
    ids = np.asarray(ids)
    lmax = lg.max(axis=1, keepdims=True)
    d = np.abs(np.take_along_axis(lg, ids, axis=1) - lmax)
    n = k if renormalize else lg.shape[1]
    dmax = d.max(axis=1, keepdims=True) if renormalize else np.abs(lg - lmax).max(axis=1, keepdims=True)
    u = 2.0 ** -24
    return (d + dmax) * u + 2 * (4 * u) + (n - 1) * u + u


def check_route_weights(w_gpu, w_ref, logits, ids, k, renormalize=True, what="route"):
    bound = route_weight_bound(logits, ids, k, renormalize)
    w_gpu = np.asarray(w_gpu, dtype=np.float64)
    w_ref = np.asarray(w_ref, dtype=np.float64)
    rel = np.abs(w_gpu - w_ref) / np.abs(w_ref)
    assert np.all(rel <= bound), f"{what}: worst {float(np.max(rel / bound)):.3f}x the bound"
