"""Plain float64 oracle for NVFP4 skinny GEMM, top-k routing and the MoE decode layer.

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Nothing here is tuned:
every function is the plain definition written out, vectorised with numpy
where that does not change the arithmetic (a float64 matmul is used as a
library step; rows are processed in chunks only to bound memory, which does
not change any result).

Sources.  The pages this library follows name NVFP4 and describe the
workload but do not define the bit layout, the routing rule or SwiGLU:

* "Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)", section "Making decode
  faster", paragraph "Skinny matrix multiplies": decode matmuls are 4-16 rows
  of 16-bit activations times a large 4-bit weight matrix (W4A16), and
  expanding 4-bit weights to BF16 is numerically identical.
* same page, "FR-Spec, and a silent bug": a 4-bit head costs 37 MB for 32K
  rows versus 290 MB for 248K rows (pins 0.5625 byte per parameter).
* "One config is the weakest card's config", section "The numbers": the decode
  roofline is bandwidth divided by the weight bytes.

The format details come from the library's specification of NVFP4: E2M1 codes
packed two per byte (low nibble = even k), one FP8-E4M3 ("fn" variant, OCP MX
v1.0) scale per 16 consecutive k, one FP32 per-tensor scale, dequantised value
= code * block scale * tensor scale.  Routing is softmax over router logits,
top-k by descending logit with ties to the lower expert index, renormalised
over the chosen k.  The expert is SwiGLU: rows [0, I) of gate_up are the gate,
rows [I, 2I) the up projection, silu(z) = z / (1 + exp(-z)).

Parity status: every function below is pinned in tests/test_oracle_pins.py
against the format tables of independent libraries, exact rational brute
force, closed forms, invariants, or the pages' printed figures.
"""
from __future__ import annotations

import math
from typing import Callable, Sequence, Tuple

import numpy as np

__all__ = [
    "dec_e2m1", "dec_e4m3", "E2M1_TABLE", "E4M3_TABLE", "bf16_round",
    "dequant", "gemm64", "gemm_bf16", "topk_softmax_route", "silu",
    "expert_ffn64", "moe_decode64", "moe_decode_bf16", "argmax_first",
    "lm_head_argmax", "hot_vocab_head_argmax", "rms_scale", "round_to_e2m1",
    "round_to_e4m3", "nvfp4_quantize", "fp8_gemm64", "fp8_gemm_bf16", "bf16w_gemm64",
    "bf16w_gemm_bf16", "nvfp4_weight_bytes",
    "moe_weight_bytes", "decode_roofline_tok_s", "roofline_share",
    "RMS_EPS",
]

# --------------------------------------------------------------------------
# Formats
# --------------------------------------------------------------------------

def dec_e2m1(code: int) -> float:
    """Value of one 4-bit E2M1 code.

    Bit 3 is the sign, bits 2..1 the exponent (bias 1), bit 0 the mantissa.
    Exponent field 0 is subnormal (value 0.5*m); otherwise 2^(e-1)*(1+m/2).
    Code 8 is -0.  (OCP Microscaling Formats v1.0, FP4 E2M1.)
    """
    code = int(code)
    if not 0 <= code < 16:
        raise ValueError("E2M1 code out of range")
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return -mag if s else mag


def dec_e4m3(byte: int) -> float:
    """Value of one FP8 E4M3 byte, OCP "fn" variant (no infinities).

    Bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa.  Exponent
    field 0 is subnormal (m/8 * 2^-6).  0x7F and 0xFF are NaN; the largest
    finite magnitude is 448.
    """
    byte = int(byte)
    if not 0 <= byte < 256:
        raise ValueError("E4M3 byte out of range")
    s = (byte >> 7) & 1
    e = (byte >> 3) & 15
    m = byte & 7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        mag = (m / 8.0) * 2.0 ** -6
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


E2M1_TABLE = np.array([dec_e2m1(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([dec_e4m3(b) for b in range(256)], dtype=np.float64)

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_round(x) -> np.ndarray:
    """Round float64 values once, to nearest-even, onto the BF16 grid.

    BF16 keeps 8 significant bits for normal numbers (|x| >= 2^-126) and a
    fixed quantum of 2^-133 below that.  Values whose rounded magnitude
    reaches 2^128 become infinities; NaN and infinities pass through.
    Returns float64 arrays holding exactly representable BF16 values.
    """
    x = np.asarray(x, dtype=np.float64)
    finite = np.isfinite(x)
    xf = np.where(finite, x, 0.0)
    _, e = np.frexp(xf)                      # xf = m * 2^e, 0.5 <= |m| < 1
    q = np.where(e - 1 >= -126, e - 8, -133)  # exponent of one unit in the last place
    y = np.ldexp(np.rint(np.ldexp(xf, -q)), q)  # np.rint rounds half to even
    y = np.where(np.abs(y) > _BF16_MAX, np.copysign(np.inf, xf), y)
    return np.where(finite, y, x)


# --------------------------------------------------------------------------
# NVFP4 weights and the skinny GEMM
# --------------------------------------------------------------------------

def dequant(codes: np.ndarray, scales: np.ndarray, global_scale: float) -> np.ndarray:
    """Decode an NVFP4 matrix to float64.

    codes  uint8 [N, K/2]: byte j of row n holds k = 2j in its low nibble and
           k = 2j+1 in its high nibble.
    scales uint8 [N, K/16]: E4M3 scale of block k // 16.
    global_scale: the FP32 per-tensor scale.
    W[n, k] = E2M1(nibble(n, k)) * E4M3(scales[n, k // 16]) * global_scale,
    exact in float64 (at most 6 + 24 significant bits).
    """
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    n, kh = codes.shape
    k = 2 * kh
    if scales.shape != (n, k // 16):
        raise ValueError("scales must be [N, K/16]")
    q = np.empty((n, k), dtype=np.float64)
    q[:, 0::2] = E2M1_TABLE[codes & 0x0F]
    q[:, 1::2] = E2M1_TABLE[codes >> 4]
    s = np.repeat(E4M3_TABLE[scales], 16, axis=1)
    return q * s * float(np.float32(global_scale))


def gemm64(a: np.ndarray, codes: np.ndarray, scales: np.ndarray,
           global_scale: float, row_chunk: int = 8192) -> np.ndarray:
    """C[m, n] = sum_k A[m, k] * W[n, k] in float64, unrounded.

    A holds the BF16 activation values as float64 [M, K]; W is the NVFP4
    matrix [N, K].  Rows of W are decoded in chunks so a large head is never
    expanded whole; each output element is computed independently, so the
    chunking does not change any result.
    """
    a = np.asarray(a, dtype=np.float64)
    n = codes.shape[0]
    out = np.empty((a.shape[0], n), dtype=np.float64)
    for r0 in range(0, n, row_chunk):
        r1 = min(n, r0 + row_chunk)
        w = dequant(codes[r0:r1], scales[r0:r1], global_scale)
        out[:, r0:r1] = a @ w.T
    return out


def gemm_bf16(a, codes, scales, global_scale) -> np.ndarray:
    """The skinny GEMM's BF16 output: gemm64 rounded once to BF16."""
    return bf16_round(gemm64(a, codes, scales, global_scale))


def argmax_first(v: np.ndarray, axis: int = -1) -> np.ndarray:
    """Index of the first maximum along ``axis`` (ties go to the lowest index)."""
    return np.argmax(np.asarray(v), axis=axis).astype(np.int32)


def lm_head_argmax(a, codes, scales, global_scale) -> Tuple[np.ndarray, np.ndarray]:
    """Greedy token choice from a 4-bit head: logits rounded to BF16, then the
    first maximum per row.  Returns (ids int32 [M], bf16 logits [M, N])."""
    logits = gemm_bf16(a, codes, scales, global_scale)
    return argmax_first(logits, axis=1), logits


def hot_vocab_head_argmax(a, codes, scales, global_scale,
                          vocab_ids) -> Tuple[np.ndarray, np.ndarray]:
    """Greedy draft token through a hot-vocabulary head ("Qwen3.6-35B-A3B
    NVFP4 on an RTX 5090 (Elsa)", section "Making decode faster", paragraph
    "FR-Spec, and a silent bug"): the 4-bit head restricted to the rows of a
    list of likely tokens, those rows taken from the full head [N, K] itself.
    The listed rows' logits are rounded to BF16; the first maximum in list
    order is reported as its vocabulary id.  A listed id outside [0, N)
    stands for an all-zero row.  Returns (ids int32 [M], bf16 logits
    [M, len(vocab_ids)])."""
    vocab_ids = np.asarray(vocab_ids, dtype=np.int64)
    ok = (vocab_ids >= 0) & (vocab_ids < codes.shape[0])
    hot_codes = np.zeros((vocab_ids.size, codes.shape[1]), dtype=np.uint8)
    hot_scales = np.zeros((vocab_ids.size, scales.shape[1]), dtype=np.uint8)
    hot_codes[ok] = codes[vocab_ids[ok]]
    hot_scales[ok] = scales[vocab_ids[ok]]
    logits = gemm_bf16(a, hot_codes, hot_scales, global_scale)
    return vocab_ids[argmax_first(logits, axis=1)].astype(np.int32), logits


# --------------------------------------------------------------------------
# Other weight formats of the skinny GEMM
# --------------------------------------------------------------------------

def fp8_gemm64(a: np.ndarray, w: np.ndarray, scale: float,
               row_chunk: int = 8192) -> np.ndarray:
    """C[m, n] = sum_k A[m, k] * e4m3(W[n, k]) * scale in float64, unrounded:
    FP8-E4M3 weights [N, K] (one byte each) with ONE per-tensor float32 scale
    and 16-bit activations ("Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)",
    section "Making decode faster", paragraph "An FP8 fast path that never
    ran": the small-batch FP8 kernel engages for a single per-tensor weight
    scale)."""
    a = np.asarray(a, dtype=np.float64)
    w = np.asarray(w, dtype=np.uint8)
    s = float(np.float32(scale))
    out = np.empty((a.shape[0], w.shape[0]), dtype=np.float64)
    for r0 in range(0, w.shape[0], row_chunk):
        r1 = min(w.shape[0], r0 + row_chunk)
        out[:, r0:r1] = a @ (E4M3_TABLE[w[r0:r1]] * s).T
    return out


def fp8_gemm_bf16(a, w, scale) -> np.ndarray:
    """The FP8-weight skinny GEMM's BF16 output: fp8_gemm64 rounded once."""
    return bf16_round(fp8_gemm64(a, w, scale))


def bf16w_gemm64(a: np.ndarray, w: np.ndarray) -> np.ndarray:
    """C = A W^T in float64 for 16-bit activations and BF16 weights [N, K]
    (their values as floats): the split-K skinny GEMM of the 2048 -> 64
    projections and of 4-bit shared experts expanded to BF16 at load
    ("Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)", section "Making decode
    faster", paragraph "Skinny matrix multiplies")."""
    return np.asarray(a, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T


def bf16w_gemm_bf16(a, w) -> np.ndarray:
    """The BF16-weight skinny GEMM's BF16 output: bf16w_gemm64 rounded once."""
    return bf16_round(bf16w_gemm64(a, w))


# --------------------------------------------------------------------------
# Quantisation BF16 -> NVFP4
# --------------------------------------------------------------------------
#
# "Qwen3.8-27B-NVFP4-lmhead4-recipe" (model card), section "Files": the head
# is converted from BF16 to NVFP4 by a quantisation tool, without the rule.
# The reading taken: the usual NVFP4 recipe.  Per-tensor scale
# g = amax / (6 * 448) (so the largest block scale is E4M3's maximum); per
# 16-element block t = amax_b / (6 g), scale byte = t rounded to E4M3; each
# element's code = |x| / (scale * g) rounded to E2M1, with the element's sign
# when the code is not zero.  Every quotient and product is one float32
# operation rounded to nearest (the precision the quantised codes are decided
# in); roundings onto the E4M3 / E2M1 grids are to nearest, ties to the even
# code, saturating at 448 / 6.  An all-zero matrix gets g = 1.

def _round_to_grid(v: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the grid point nearest each non-negative value (grid ascending,
    indices are the codes), ties to the even index, saturating at the top."""
    v = np.minimum(np.asarray(v, dtype=np.float64), grid[-1])
    hi = np.clip(np.searchsorted(grid, v, side="left"), 0, grid.size - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = v - grid[lo], grid[hi] - v
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    return np.where(take_hi, hi, lo).astype(np.uint8)


def round_to_e2m1(v) -> np.ndarray:
    """Non-negative values to E2M1 codes 0..7 (nearest, ties to even, > 6 -> 6)."""
    return _round_to_grid(v, E2M1_TABLE[:8])


def round_to_e4m3(v) -> np.ndarray:
    """Non-negative values to E4M3 bytes 0..0x7E (nearest, ties to even,
    > 448 -> 448)."""
    return _round_to_grid(v, E4M3_TABLE[:127])


def nvfp4_quantize(w) -> Tuple[np.ndarray, np.ndarray, float]:
    """BF16 matrix [N, K] (its values as float64 or float32) -> (codes uint8
    [N, K/2], scales uint8 [N, K/16], global scale float32), by the recipe
    above."""
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    f32 = np.float32
    amax = f32(np.abs(w).max()) if w.size else f32(0)
    g = f32(1.0) if amax == 0 else f32(amax / f32(6 * 448))
    blocks = np.abs(w).reshape(n, k // 16, 16)
    amax_b = blocks.max(axis=2)
    t = (amax_b / f32(f32(6) * g)).astype(np.float32)
    scales = round_to_e4m3(t)
    d = (E4M3_TABLE[scales].astype(np.float32) * g).astype(np.float32)  # [n, k/16]
    dd = np.repeat(d, 16, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = np.where(dd > 0, np.abs(w) / np.where(dd > 0, dd, f32(1)), f32(0)).astype(np.float32)
    mag = round_to_e2m1(v)
    code = np.where((w < 0) & (mag != 0), mag | 8, mag).astype(np.uint8)
    codes = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return codes, scales.astype(np.uint8), float(g)


# --------------------------------------------------------------------------
# Routing
# --------------------------------------------------------------------------

def topk_softmax_route(logits: np.ndarray, k: int, renormalize: bool = True):
    """Top-k softmax routing of T tokens over E experts.

    logits float32 [T, E].  The k experts with the largest logits are chosen
    by comparing the float32 logits themselves; equal logits go to the lower
    expert index; ids are listed in that order (descending logit).  Weights
    are softmax probabilities in float64: with renormalisation
    w_j = exp(l_j - l_max) / sum over the chosen i of exp(l_i - l_max),
    otherwise the full-softmax probability of each chosen expert.
    Returns (ids int32 [T, k], weights float64 [T, k]).
    """
    logits = np.asarray(logits, dtype=np.float32)
    t, e = logits.shape
    if not 1 <= k <= e:
        raise ValueError("need 1 <= k <= E")
    ids = np.empty((t, k), dtype=np.int32)
    w = np.empty((t, k), dtype=np.float64)
    idx = np.arange(e)
    for r in range(t):
        order = np.lexsort((idx, -logits[r]))   # primary: logit descending; then index
        sel = order[:k]
        l64 = logits[r].astype(np.float64)
        lmax = l64[sel[0]]
        ex = np.exp(l64[sel] - lmax)
        den = ex.sum() if renormalize else np.exp(l64 - lmax).sum()
        ids[r] = sel
        w[r] = ex / den
    return ids, w


# --------------------------------------------------------------------------
# SwiGLU expert and the MoE layer
# --------------------------------------------------------------------------

def silu(z) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z)) in float64."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


RMS_EPS = 1e-6


def rms_scale(x) -> np.ndarray:
    """Weightless RMS scaling x / sqrt(mean(x^2) + 1e-6) per row, float64,
    unrounded: the glue this library places before each projection block of
    its stacked decode step (the pages do not describe one; it keeps 40
    unnormalised random layers inside the BF16 range)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + RMS_EPS)


ExpertWeights = Tuple[np.ndarray, np.ndarray, float, np.ndarray, np.ndarray, float]


def expert_ffn64(x: np.ndarray, expert: ExpertWeights) -> np.ndarray:
    """One SwiGLU expert in float64: W_d (silu(W_g x) * (W_u x)).

    expert = (gu_codes [2I, H/2], gu_scales [2I, H/16], gu_global,
              dn_codes [H, I/2],  dn_scales [H, I/16],  dn_global);
    rows [0, I) of gate_up are the gate, rows [I, 2I) the up projection.
    """
    gu_c, gu_s, gu_g, dn_c, dn_s, dn_g = expert
    gu = gemm64(x, gu_c, gu_s, gu_g)
    i = gu.shape[1] // 2
    h = silu(gu[:, :i]) * gu[:, i:]
    return gemm64(h, dn_c, dn_s, dn_g)


def moe_decode64(x: np.ndarray, ids: np.ndarray, w: np.ndarray,
                 experts: Callable[[int], ExpertWeights] | Sequence[ExpertWeights],
                 num_experts: int, shared: ExpertWeights | None = None) -> np.ndarray:
    """y[t] = sum_j w[t, j] * E_{ids[t, j]}(x[t]) + E_shared(x[t]), float64, unrounded.

    ``experts(e)`` (or ``experts[e]``) returns the weights of routed expert e.
    Slots whose id lies outside [0, num_experts) contribute nothing.  Repeated
    ids in one row are each counted.  The shared expert, when given, is always
    on with weight 1.  Tokens routed to the same expert are evaluated together;
    every output row is still computed independently.
    """
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(ids)
    w = np.asarray(w, dtype=np.float64)
    get = experts if callable(experts) else (lambda e: experts[e])
    y = np.zeros_like(x)
    valid = (ids >= 0) & (ids < num_experts)
    for e in np.unique(ids[valid]):
        rows, slots = np.nonzero((ids == e) & valid)
        out = expert_ffn64(x[rows], get(int(e)))
        for r, s, o in zip(rows, slots, out):
            y[r] += w[r, s] * o
    if shared is not None:
        y += expert_ffn64(x, shared)
    return y


def moe_decode_bf16(x, ids, w, experts, num_experts, shared=None) -> np.ndarray:
    """The MoE layer's BF16 output: moe_decode64 rounded once to BF16."""
    return bf16_round(moe_decode64(x, ids, w, experts, num_experts, shared))


# --------------------------------------------------------------------------
# Byte accounting and the decode roofline
# --------------------------------------------------------------------------

def nvfp4_weight_bytes(n: int, k: int) -> int:
    """Bytes one read of an NVFP4 [N, K] matrix moves: N*K/2 code bytes plus
    N*K/16 scale bytes (0.5625 byte per parameter; the 4-byte tensor scale is
    not counted)."""
    return n * k // 2 + n * k // 16


def moe_weight_bytes(ids: np.ndarray, num_experts: int, hidden: int,
                     inter: int, shared: bool = True) -> int:
    """Weight bytes one MoE call must read: every distinct routed expert in
    range (gate_up [2I, H] + down [H, I]) once, plus the shared expert."""
    ids = np.asarray(ids)
    u = np.unique(ids[(ids >= 0) & (ids < num_experts)]).size + (1 if shared else 0)
    return u * (nvfp4_weight_bytes(2 * inter, hidden) + nvfp4_weight_bytes(hidden, inter))


def decode_roofline_tok_s(bandwidth_bytes_per_s: float, weight_bytes: float) -> float:
    """Decode ceiling when every token reads all weights once: bandwidth /
    weight bytes ("One config is the weakest card's config", "The numbers")."""
    return bandwidth_bytes_per_s / weight_bytes


def roofline_share(measured: float, roofline: float) -> float:
    """Measured throughput as a fraction of the roofline."""
    return measured / roofline
