"""Seeded synthetic inputs for the NVFP4 decode path.

This module only draws random inputs; it holds none of the computation being
tested.  Both the CUDA path and the float64 oracle receive what it produces.

Every tensor is a pure function of (seed, stream ids, element index): element
i of a stream is derived from a counter hash of i, so any slice (a row range,
one expert) can be regenerated on the host without drawing the rest, and the
integer-only draws (NVFP4 codes and scales) give the same bytes on the CPU and
on a CUDA device.  Floating-point draws (activations, router logits) are made
on the host only.

Distributions (the workload recipe):
* activations ~ N(0, 1), rounded to BF16 (via float32, by torch);
* router logits ~ N(0, 1), float32;
* E2M1 codes uniform over all 16 codes, two per byte;
* E4M3 block scales RNE(2^u), u ~ U(-4, 2) on a 2^24-point grid, i.e.
  log-uniform in [2^-4, 2^2];
* the FP32 per-tensor scale is the constant 0.5.

Hash: "lowbias32" (C. Wellons, "Prospecting for Hash Functions", 2018), a
bijection on 32-bit words, applied twice with a per-stream key.  It is written
with int64 torch ops whose partial products stay below 2^63.
"""
from __future__ import annotations

import math
from typing import Iterable

import numpy as np
import torch

GLOBAL_SCALE = 0.5
_M32 = 0xFFFFFFFF

# stream roles
ROLE_ACT = 1
ROLE_LOGITS = 2
ROLE_CODES = 3
ROLE_SCALES = 4


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for x in [0, 2^32) without int64 overflow."""
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & _M32


def _lowbias32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    return x ^ (x >> 16)


def _py_lowbias32(x: int) -> int:
    x &= _M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & _M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & _M32
    return x ^ (x >> 16)


def stream_key(seed: int, *ids: int) -> tuple[int, int]:
    """Two 32-bit keys for the stream named by (seed, ids...)."""
    h = _py_lowbias32(0x9E3779B9 ^ (seed & _M32))
    for v in ids:
        h = _py_lowbias32(h ^ (v & _M32))
    return h, _py_lowbias32(h ^ 0x632BE5AB)


def bits32(key: tuple[int, int], start: int, count: int, device="cpu") -> torch.Tensor:
    """Words start .. start+count-1 of a stream, as int64 in [0, 2^32)."""
    if start < 0 or start + count > 2 ** 32:
        raise ValueError("stream counter out of range")
    i = torch.arange(start, start + count, dtype=torch.int64, device=device)
    return _lowbias32(_lowbias32((i + key[0]) & _M32) ^ key[1])


# ----------------------------------------------------------------- floats

def _uniform01(w: torch.Tensor) -> torch.Tensor:
    """(top 24 bits + 0.5) / 2^24, exact in float64, in (0, 1)."""
    return ((w >> 8).to(torch.float64) + 0.5) * (1.0 / 16777216.0)


def normal(key, count: int) -> torch.Tensor:
    """count N(0,1) float64 draws (Box-Muller, one pair of words each), host."""
    w = bits32(key, 0, 2 * count).view(count, 2)
    u1, u2 = _uniform01(w[:, 0]), _uniform01(w[:, 1])
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * math.pi * u2)


def activations_bf16(seed: int, rows: int, cols: int, *ids: int) -> torch.Tensor:
    """BF16 [rows, cols] ~ N(0,1) on the host.  Row r depends only on r, so a
    prefix of rows is the same for every ``rows``."""
    z = normal(stream_key(seed, ROLE_ACT, cols, *ids), rows * cols)
    return z.to(torch.float32).to(torch.bfloat16).view(rows, cols)


def router_logits(seed: int, rows: int, experts: int, *ids: int) -> torch.Tensor:
    """float32 [rows, experts] ~ N(0,1) on the host."""
    z = normal(stream_key(seed, ROLE_LOGITS, experts, *ids), rows * experts)
    return z.to(torch.float32).view(rows, experts)


# ----------------------------------------------------------------- NVFP4

def _scale_thresholds() -> torch.Tensor:
    """Integer thresholds on the 24-bit grid r for the nearest E4M3 value to
    2^u, u = -4 + 6 (r + 0.5) / 2^24.  Candidates are the E4M3 bytes 0x18
    (0.0625) .. 0x48 (4.0), decoded by torch."""
    cand = torch.arange(0x18, 0x49, dtype=torch.int32).to(torch.uint8)
    vals = cand.view(torch.float8_e4m3fn).to(torch.float64).tolist()
    out = []
    for a, b in zip(vals[:-1], vals[1:]):
        x = ((math.log2(0.5 * (a + b)) + 4.0) / 6.0) * 16777216.0 - 0.5
        frac = x - math.floor(x)
        assert min(frac, 1.0 - frac) > 1e-6
        out.append(math.ceil(x))
    return torch.tensor(out, dtype=torch.int64)


_THRESH = _scale_thresholds()
_SCALE_BASE = 0x18


def nvfp4_codes(key, rows: int, k: int, row_lo: int = 0, row_hi: int | None = None,
                device="cpu") -> torch.Tensor:
    """uint8 [row_hi-row_lo, k/2] packed E2M1 codes of rows row_lo..row_hi-1
    of a [rows, k] matrix: 32 random bits per 4 bytes (8 uniform codes)."""
    row_hi = rows if row_hi is None else row_hi
    wpr = k // 8                              # 32-bit words per row
    w = bits32(key, row_lo * wpr, (row_hi - row_lo) * wpr, device)
    w = torch.where(w >= 2 ** 31, w - 2 ** 32, w)      # same bits, in int32 range
    return w.to(torch.int32).view(torch.uint8).view(row_hi - row_lo, k // 2)


def nvfp4_scales(key, rows: int, k: int, row_lo: int = 0, row_hi: int | None = None,
                 device="cpu") -> torch.Tensor:
    """uint8 [row_hi-row_lo, k/16] E4M3 block scales, log-uniform in [2^-4, 4]."""
    row_hi = rows if row_hi is None else row_hi
    bpr = k // 16
    r = bits32(key, row_lo * bpr, (row_hi - row_lo) * bpr, device) >> 8
    idx = torch.searchsorted(_THRESH.to(r.device), r, right=True)
    return (idx + _SCALE_BASE).to(torch.uint8).view(row_hi - row_lo, bpr)


def weight_keys(seed: int, *ids: int):
    return stream_key(seed, ROLE_CODES, *ids), stream_key(seed, ROLE_SCALES, *ids)


def nvfp4_weight(seed: int, n: int, k: int, *ids: int, row_lo: int = 0,
                 row_hi: int | None = None, device="cpu"):
    """(codes uint8 [rows, k/2], scales uint8 [rows, k/16]) for the NVFP4
    matrix [n, k] named by (seed, ids...), rows row_lo..row_hi-1."""
    if k % 32:
        raise ValueError("K must be a multiple of 32")
    ck, sk = weight_keys(seed, n, k, *ids)
    return (nvfp4_codes(ck, n, k, row_lo, row_hi, device),
            nvfp4_scales(sk, n, k, row_lo, row_hi, device))


# ----------------------------------------------------------------- FP8 / BF16 weights

ROLE_FP8 = 13
ROLE_BF16W = 14
FP8_SCALE = 1.0 / 64.0


def fp8_weight(seed: int, n: int, k: int, *ids: int) -> torch.Tensor:
    """uint8 [n, k] FP8-E4M3 ("fn") bytes of N(0, 1) * 8 draws, rounded to
    nearest by torch's float8_e4m3fn conversion (no NaN: |x| < 448 for every
    draw the generator can make); the matrix's one scale is FP8_SCALE."""
    z = normal(stream_key(seed, ROLE_FP8, n, k, *ids), n * k) * 8.0
    return z.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).view(n, k)


def bf16_weight(seed: int, n: int, k: int, *ids: int) -> torch.Tensor:
    """BF16 [n, k] weights ~ N(0, 1) / 16 on the host."""
    z = normal(stream_key(seed, ROLE_BF16W, n, k, *ids), n * k) / 16.0
    return z.to(torch.float32).to(torch.bfloat16).view(n, k)


# ----------------------------------------------------------------- MoE experts

ROLE_GATE_UP = 11
ROLE_DOWN = 12


def expert_weight(seed: int, layer: int, e: int, hidden: int, inter: int, device="cpu"):
    """(gu_codes, gu_scales, dn_codes, dn_scales) of expert e of a layer.
    Expert index ``num_experts`` names the shared expert."""
    gc, gs = nvfp4_weight(seed, 2 * inter, hidden, ROLE_GATE_UP, layer, e, device=device)
    dc, ds = nvfp4_weight(seed, hidden, inter, ROLE_DOWN, layer, e, device=device)
    return gc, gs, dc, ds


def _keyed_bits(k0: torch.Tensor, k1: torch.Tensor, count: int, device) -> torch.Tensor:
    """Words 0..count-1 of several streams at once: k0, k1 int64 [S, 1]."""
    i = torch.arange(count, dtype=torch.int64, device=device).view(1, -1)
    return _lowbias32(_lowbias32((i + k0) & _M32) ^ k1)


def _stack_matrices(seed: int, role: int, layer: int, experts: list, n: int, k: int,
                    codes_out: torch.Tensor, scales_out: torch.Tensor, group: int = 16):
    """Fill codes_out [E, n, k/2] and scales_out [E, n, k/16] with the
    matrices (seed, n, k, role, layer, e) for e in ``experts``; identical to
    drawing each with nvfp4_weight, but generated ``group`` experts at once."""
    dev = codes_out.device
    for g0 in range(0, len(experts), group):
        ids = experts[g0:g0 + group]
        ck = [weight_keys(seed, n, k, role, layer, e) for e in ids]
        c0 = torch.tensor([c[0][0] for c in ck], dtype=torch.int64, device=dev).view(-1, 1)
        c1 = torch.tensor([c[0][1] for c in ck], dtype=torch.int64, device=dev).view(-1, 1)
        s0 = torch.tensor([c[1][0] for c in ck], dtype=torch.int64, device=dev).view(-1, 1)
        s1 = torch.tensor([c[1][1] for c in ck], dtype=torch.int64, device=dev).view(-1, 1)
        w = _keyed_bits(c0, c1, n * k // 8, dev)
        w = torch.where(w >= 2 ** 31, w - 2 ** 32, w)
        codes_out[g0:g0 + len(ids)].copy_(
            w.to(torch.int32).view(torch.uint8).view(len(ids), n, k // 2))
        r = _keyed_bits(s0, s1, n * k // 16, dev) >> 8
        idx = torch.searchsorted(_THRESH.to(dev), r.contiguous(), right=True)
        scales_out[g0:g0 + len(ids)].copy_((idx + _SCALE_BASE).to(torch.uint8)
                                           .view(len(ids), n, k // 16))
        del w, r, idx


def expert_stack(seed: int, layer: int, experts: Iterable[int], hidden: int, inter: int,
                 device="cpu"):
    """Stacked weights of the listed experts: gu_codes [E, 2I, H/2],
    gu_scales [E, 2I, H/16], dn_codes [E, H, I/2], dn_scales [E, H, I/16],
    generated on ``device``; expert e's slices equal expert_weight(..., e)."""
    experts = list(experts)
    ne = len(experts)
    gu_c = torch.empty(ne, 2 * inter, hidden // 2, dtype=torch.uint8, device=device)
    gu_s = torch.empty(ne, 2 * inter, hidden // 16, dtype=torch.uint8, device=device)
    dn_c = torch.empty(ne, hidden, inter // 2, dtype=torch.uint8, device=device)
    dn_s = torch.empty(ne, hidden, inter // 16, dtype=torch.uint8, device=device)
    _stack_matrices(seed, ROLE_GATE_UP, layer, experts, 2 * inter, hidden, gu_c, gu_s)
    _stack_matrices(seed, ROLE_DOWN, layer, experts, hidden, inter, dn_c, dn_s)
    return gu_c, gu_s, dn_c, dn_s


def expert_host(seed: int, layer: int, e: int, hidden: int, inter: int,
                gscale: float = GLOBAL_SCALE):
    """Expert e as numpy arrays in the tuple order the oracle takes:
    (gu_codes, gu_scales, gu_global, dn_codes, dn_scales, dn_global)."""
    gc, gs, dc, ds = expert_weight(seed, layer, e, hidden, inter)
    return (gc.numpy(), gs.numpy(), gscale, dc.numpy(), ds.numpy(), gscale)


def to_numpy_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a (BF16 / float32) tensor, on the host."""
    return t.detach().to("cpu", torch.float64).numpy()
