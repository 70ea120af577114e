"""Pins of the float64 oracle against things other than itself.

Each check ties an oracle function to an independent fact: another library's
format table, an exact rational brute force, a closed form, an invariant of
the mathematics, or a figure the pages print.  They are chosen so that a
dropped term, a swapped nibble, a wrong sign, a transposed operand or an
off-by-one block index fails at least one of them.  CPU only.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O

RNG = np.random.default_rng(12345)


# ---------------------------------------------------------------- helpers

def _golden_table(path):
    out = {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a, b = line.split()
        out[int(a, 0)] = float(b)
    return out


def _torch_e4m3_values():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return b.view(torch.float8_e4m3fn).to(torch.float64).numpy()


_BF16_GRID = None


def _bf16_grid():
    """All finite BF16 values, sorted, decoded by torch (not by the oracle)."""
    global _BF16_GRID
    if _BF16_GRID is None:
        bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
        v = bits.view(torch.bfloat16).to(torch.float64).numpy()
        m = np.asarray(bits.numpy().astype(np.uint16))
        keep = np.isfinite(v)
        v, m = v[keep], m[keep]
        order = np.lexsort((m, v))
        _BF16_GRID = (v[order], m[order])
    return _BF16_GRID


def _nearest_bf16_exact(r: Fraction) -> float:
    """Nearest BF16 value to the rational r, ties to the even mantissa bit,
    by search over the enumerated grid with exact rational comparisons."""
    vals, bits = _bf16_grid()
    x = float(r)
    i = int(np.searchsorted(vals, x))
    cands = set()
    for j in range(max(0, i - 3), min(len(vals), i + 3)):
        cands.add(j)
    best = None
    for j in sorted(cands):
        d = abs(Fraction(float(vals[j])) - r)
        key = (d, int(bits[j]) & 1)  # ties: prefer the even last mantissa bit
        if best is None or key < best[0]:
            best = (key, float(vals[j]))
    return best[1]


def _rand_nvfp4(n, k, rng=RNG, scale_lo=0x18, scale_hi=0x48):
    codes = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    scales = rng.integers(scale_lo, scale_hi + 1, size=(n, k // 16), dtype=np.uint8)
    return codes, scales


def _rand_bf16(shape, rng=RNG, scale=1.0):
    x = torch.from_numpy(rng.standard_normal(shape) * scale).to(torch.float32)
    return x.to(torch.bfloat16).to(torch.float64).numpy()


# ---------------------------------------------------------------- formats

def test_e2m1_table_matches_spec_table(golden_dir):
    spec = _golden_table(os.path.join(golden_dir, "e2m1_ocp_mx.txt"))
    for c in range(16):
        assert O.E2M1_TABLE[c] == spec[c]
        assert math.copysign(1.0, O.E2M1_TABLE[c]) == math.copysign(1.0, spec[c])


def test_e2m1_table_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    # float4_e2m1fn values in code order, decoded by the library
    ref = np.array([float(np.array(c, dtype=np.uint8).view(ml.float4_e2m1fn)) for c in range(16)])
    assert np.array_equal(ref, O.E2M1_TABLE)


def test_e4m3_table_matches_torch_all_256():
    ref = _torch_e4m3_values()
    nan_ref = np.isnan(ref)
    nan_o = np.isnan(O.E4M3_TABLE)
    assert np.array_equal(nan_ref, nan_o)
    assert np.array_equal(ref[~nan_ref], O.E4M3_TABLE[~nan_o])
    assert nan_o.sum() == 2 and nan_o[0x7F] and nan_o[0xFF]


def test_e4m3_landmarks_from_spec(golden_dir):
    pts = _golden_table(os.path.join(golden_dir, "e4m3_ocp_points.txt"))
    for b, v in pts.items():
        got = O.dec_e4m3(b)
        if math.isnan(v):
            assert math.isnan(got)
        else:
            assert got == v and math.copysign(1, got) == math.copysign(1, v)


def test_code_times_scale_is_exact_in_bf16_and_f16():
    """Every E2M1 x E4M3 product is exactly representable in BF16 and in FP16,
    which is what makes expanding 4-bit weights to 16 bits numerically
    identical ('Skinny matrix multiplies')."""
    prods = np.outer(O.E2M1_TABLE, O.E4M3_TABLE).ravel()
    prods = prods[np.isfinite(prods)]
    assert np.array_equal(O.bf16_round(prods), prods)
    f16 = torch.from_numpy(prods).to(torch.float16).to(torch.float64).numpy()
    assert np.array_equal(f16, prods)


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_round_matches_torch_on_float32_inputs():
    x = np.concatenate([
        RNG.standard_normal(20000) * 10.0 ** RNG.integers(-30, 30, 20000),
        RNG.standard_normal(2000) * 1e-39,          # bf16 subnormal range
        np.array([3.3e38, -3.3e38, 1e-45, 0.0, -0.0]),
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_round(x.astype(np.float64))
    assert np.array_equal(np.isinf(ref), np.isinf(got))
    fin = np.isfinite(ref)
    assert np.array_equal(ref[fin], got[fin])


def test_bf16_round_is_single_rounding_of_float64():
    """Inputs with more than float32 precision: compare with the exactly
    nearest grid value (ties to even), found by enumeration."""
    xs = list(RNG.standard_normal(300) * 10.0 ** RNG.integers(-5, 5, 300))
    one = 1.0
    xs += [one + 2 ** -8, one + 3 * 2 ** -8, one + 2 ** -8 + 2 ** -40,
           -(one + 2 ** -8), 2.0 ** -126 * (1 + 2 ** -8)]
    for x in xs:
        assert O.bf16_round(np.array([x]))[0] == _nearest_bf16_exact(Fraction(x)), x


def test_bf16_round_ties_to_even_examples():
    assert O.bf16_round(1 + 2 ** -8) == 1.0                    # tie, even is 1.0
    assert O.bf16_round(1 + 3 * 2 ** -8) == 1 + 2 ** -6         # tie, rounds up to even
    assert O.bf16_round(1 + 2 ** -8 + 2 ** -30) == 1 + 2 ** -7  # just above tie


# ---------------------------------------------------------------- dequant + GEMM

def test_dequant_nibble_order_and_block_index():
    n, k = 2, 64
    codes = np.zeros((n, k // 2), np.uint8)
    scales = np.full((n, k // 16), 0x38, np.uint8)       # 1.0
    codes[0, 3] = 0x02        # k = 6 (low nibble) -> 1.0
    codes[1, 9] = 0x70        # k = 19 (high nibble) -> 6.0
    scales[1, 1] = 0x40       # block of k 16..31 -> 2.0
    w = O.dequant(codes, scales, 0.5)
    expect = np.zeros((n, k))
    expect[0, 6] = 0.5
    expect[1, 19] = 6.0 * 2.0 * 0.5
    assert np.array_equal(w, expect)


def _brute_force_gemm(a, codes, scales, g, spec_e2m1):
    """Exact rational C = A W^T, weights decoded from the spec table and
    torch's E4M3 table (independent of the oracle's decoders)."""
    e4 = _torch_e4m3_values()
    m, k = a.shape
    n = codes.shape[0]
    out = [[Fraction(0)] * n for _ in range(m)]
    gf = Fraction(float(np.float32(g)))
    for j in range(n):
        wrow = []
        for kk in range(k):
            byte = int(codes[j, kk // 2])
            nib = byte & 0xF if kk % 2 == 0 else byte >> 4
            wrow.append(Fraction(spec_e2m1[nib]) * Fraction(float(e4[scales[j, kk // 16]])) * gf)
        for i in range(m):
            out[i][j] = sum((Fraction(float(a[i, kk])) * wrow[kk] for kk in range(k)), Fraction(0))
    return out


@pytest.mark.parametrize("m,n,k", [(1, 1, 16), (2, 3, 32), (3, 4, 64), (3, 2, 48)])
def test_gemm_matches_exact_rational_brute_force(golden_dir, m, n, k):
    spec = _golden_table(os.path.join(golden_dir, "e2m1_ocp_mx.txt"))
    rng = np.random.default_rng(m * 100 + n * 10 + k)
    a = _rand_bf16((m, k), rng)
    codes, scales = _rand_nvfp4(n, k, rng, 0x01, 0x7E)
    g = 0.5
    exact = _brute_force_gemm(a, codes, scales, g, spec)
    c64 = O.gemm64(a, codes, scales, g)
    cb = O.gemm_bf16(a, codes, scales, g)
    for i in range(m):
        for j in range(n):
            bound = sum(abs(float(a[i, kk])) for kk in range(k)) * 6 * 448 * 0.5 * k * 2 ** -52
            assert abs(Fraction(c64[i, j]) - exact[i][j]) <= Fraction(bound) + Fraction(2) ** -1070
            assert cb[i, j] == _nearest_bf16_exact(exact[i][j])


def test_gemm_identity_case():
    k, n = 2048, 8
    a = np.ones((4, k))
    codes = np.full((n, k // 2), 0x22, np.uint8)   # both nibbles = 1.0
    scales = np.full((n, k // 16), 0x38, np.uint8)  # 1.0
    c = O.gemm64(a, codes, scales, 1.0)
    assert np.array_equal(c, np.full((4, n), float(k)))


def test_gemm_one_hot_recovers_weight_column():
    k, n = 256, 5
    codes, scales = _rand_nvfp4(n, k)
    w = O.dequant(codes, scales, 0.5)
    for kstar in (0, 1, 17, 255):
        a = np.zeros((1, k))
        a[0, kstar] = 1.0
        assert np.array_equal(O.gemm64(a, codes, scales, 0.5)[0], w[:, kstar])


def test_gemm_zero_codes_give_zero():
    codes = np.zeros((3, 32), np.uint8)
    codes[1] = 0x88            # -0 in both nibbles
    scales = np.full((3, 4), 0x7E, np.uint8)
    c = O.gemm64(_rand_bf16((2, 64)), codes, scales, 0.5)
    assert np.all(c == 0.0)


def test_gemm_chunking_does_not_change_results():
    codes, scales = _rand_nvfp4(37, 128)
    a = _rand_bf16((3, 128))
    assert np.array_equal(O.gemm64(a, codes, scales, 0.5, row_chunk=5),
                          O.gemm64(a, codes, scales, 0.5))


# ---------------------------------------------------------------- routing

def _route_brute(row, k, renorm):
    e = len(row)
    order = sorted(range(e), key=lambda i: (-float(row[i]), i))[:k]
    ex = [math.exp(float(row[i]) - float(row[order[0]])) for i in order]
    den = sum(ex) if renorm else sum(math.exp(float(v) - float(row[order[0]])) for v in row)
    return order, [v / den for v in ex]


@pytest.mark.parametrize("renorm", [True, False])
def test_route_matches_brute_force_sort(renorm):
    logits = RNG.standard_normal((20, 256)).astype(np.float32)
    ids, w = O.topk_softmax_route(logits, 8, renorm)
    for t in range(20):
        bi, bw = _route_brute(logits[t], 8, renorm)
        assert list(ids[t]) == bi
        np.testing.assert_allclose(w[t], bw, rtol=1e-14)


def test_route_ties_go_to_lower_index():
    logits = np.zeros((1, 16), np.float32)
    logits[0, [3, 7, 11]] = 2.0
    logits[0, [5, 9]] = 1.0
    ids, w = O.topk_softmax_route(logits, 5)
    assert list(ids[0]) == [3, 7, 11, 5, 9]
    logits = np.zeros((1, 8), np.float32)
    ids, _ = O.topk_softmax_route(logits, 4)
    assert list(ids[0]) == [0, 1, 2, 3]


def test_route_closed_form_and_sum():
    logits = np.log(np.array([[1.0, 2.0, 3.0, 4.0, 0.5, 0.25]], np.float32))
    ids, w = O.topk_softmax_route(logits, 4)
    assert list(ids[0]) == [3, 2, 1, 0]
    l = logits[0].astype(np.float64)
    expect = np.exp(l[[3, 2, 1, 0]]) / np.exp(l[[3, 2, 1, 0]]).sum()
    np.testing.assert_allclose(w[0], expect, rtol=1e-15)
    np.testing.assert_allclose(w[0], [0.4, 0.3, 0.2, 0.1], rtol=1e-6)
    x = RNG.standard_normal((50, 256)).astype(np.float32)
    _, w = O.topk_softmax_route(x, 8)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-14)


def test_route_k_equals_e_is_permutation_and_full_softmax():
    scipy_special = pytest.importorskip("scipy.special")
    x = RNG.standard_normal((4, 32)).astype(np.float32)
    ids, w = O.topk_softmax_route(x, 32, renormalize=False)
    for t in range(4):
        assert sorted(ids[t]) == list(range(32))
        p = scipy_special.softmax(x[t].astype(np.float64))
        np.testing.assert_allclose(w[t], p[ids[t]], rtol=1e-13)
    _, w8 = O.topk_softmax_route(x, 8, renormalize=False)
    ids8, _ = O.topk_softmax_route(x, 8)
    for t in range(4):
        p = scipy_special.softmax(x[t].astype(np.float64))
        np.testing.assert_allclose(w8[t], p[ids8[t]], rtol=1e-13)


# ---------------------------------------------------------------- SwiGLU / MoE

def test_silu_against_library_sigmoid():
    sp = pytest.importorskip("scipy.special")
    z = np.concatenate([RNG.standard_normal(1000) * 5, [0.0, 40.0, -40.0, -800.0]])
    np.testing.assert_allclose(O.silu(z), z * sp.expit(z), rtol=1e-14, atol=1e-300)
    assert O.silu(0.0) == 0.0


def _expert(rng, h, i, gu_scale=0.5, dn_scale=0.5):
    gc, gs = _rand_nvfp4(2 * i, h, rng)
    dc, ds = _rand_nvfp4(h, i, rng)
    return (gc, gs, gu_scale, dc, ds, dn_scale)


def test_expert_is_swiglu_with_gate_first():
    """Compose the expert by hand from library-free pieces: weights decoded via
    the spec table + torch E4M3, numpy matmul, and expit."""
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(7)
    h, i = 64, 32
    ex = _expert(rng, h, i)
    x = _rand_bf16((3, h), rng)
    e4 = _torch_e4m3_values()
    spec = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])

    def dec(c, s, g):
        q = np.stack([spec[c & 15], spec[c >> 4]], axis=-1).reshape(c.shape[0], -1)
        return q * np.repeat(e4[s], 16, axis=1) * g

    wgu = dec(ex[0], ex[1], ex[2])
    wd = dec(ex[3], ex[4], ex[5])
    gate = x @ wgu[:i].T
    up = x @ wgu[i:].T
    ref = (gate * sp.expit(gate) * up) @ wd.T
    got = O.expert_ffn64(x, ex)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-9 * np.abs(ref).max())
    # swapping gate and up must change the answer (silu is not symmetric)
    swapped = ((up * sp.expit(up)) * gate) @ wd.T
    assert np.abs(swapped - got).max() > 1e-3 * np.abs(ref).max()


def _moe_setup(seed, e=8, h=64, i=32, t=5, k=3):
    rng = np.random.default_rng(seed)
    experts = [_expert(rng, h, i) for _ in range(e)]
    shared = _expert(rng, h, i)
    x = _rand_bf16((t, h), rng)
    logits = rng.standard_normal((t, e)).astype(np.float32)
    ids, w = O.topk_softmax_route(logits, k)
    return experts, shared, x, ids, w


def test_moe_single_token_single_expert_is_two_gemms_and_swiglu():
    experts, shared, x, _, _ = _moe_setup(1)
    ids = np.array([[5]])
    w = np.array([[0.75]])
    got = O.moe_decode64(x[:1], ids, w, experts, 8, shared)
    ref = 0.75 * O.expert_ffn64(x[:1], experts[5]) + O.expert_ffn64(x[:1], shared)
    np.testing.assert_allclose(got, ref, rtol=1e-13)


def test_moe_expert_relabelling_invariance():
    experts, shared, x, ids, w = _moe_setup(2)
    perm = np.random.default_rng(3).permutation(8)
    relabelled = [None] * 8
    for old, new in enumerate(perm):
        relabelled[new] = experts[old]
    a = O.moe_decode64(x, ids, w, experts, 8, shared)
    b = O.moe_decode64(x, perm[ids], w, relabelled, 8, shared)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-12 * np.abs(a).max())


def test_moe_routed_part_is_linear_in_weights_and_shared_is_additive():
    experts, shared, x, ids, w = _moe_setup(4)
    routed = O.moe_decode64(x, ids, w, experts, 8, None)
    both = O.moe_decode64(x, ids, w, experts, 8, shared)
    np.testing.assert_allclose(O.moe_decode64(x, ids, 2.5 * w, experts, 8, None), 2.5 * routed,
                               rtol=1e-13, atol=1e-12 * np.abs(routed).max())
    np.testing.assert_allclose(both - routed, O.expert_ffn64(x, shared),
                               rtol=1e-10, atol=1e-10 * np.abs(both).max())
    zero_shared = (np.zeros_like(shared[0]),) + shared[1:]
    np.testing.assert_array_equal(O.moe_decode64(x, ids, w, experts, 8, zero_shared), routed)


def test_moe_out_of_range_ids_skipped_and_duplicates_summed():
    experts, shared, x, ids, w = _moe_setup(5)
    ids2 = ids.copy()
    ids2[:, -1] = 99
    ids2[0, 0] = -1
    a = O.moe_decode64(x, ids2, w, experts, 8, None)
    w2 = w.copy()
    w2[:, -1] = 0.0
    w2[0, 0] = 0.0
    b = O.moe_decode64(x, ids, w2, experts, 8, None)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13 * np.abs(b).max())
    dup = np.array([[2, 2]])
    c = O.moe_decode64(x[:1], dup, np.array([[0.25, 0.5]]), experts, 8, None)
    d = O.moe_decode64(x[:1], np.array([[2]]), np.array([[0.75]]), experts, 8, None)
    np.testing.assert_allclose(c, d, rtol=1e-13)


def test_rms_scale_closed_forms():
    x = np.full((2, 100), 3.0)
    np.testing.assert_allclose(O.rms_scale(x), 3.0 / math.sqrt(9.0 + 1e-6), rtol=1e-15)
    y = O.rms_scale(RNG.standard_normal((4, 2048)) * 50)
    np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-9)
    assert np.all(O.rms_scale(np.zeros((1, 8))) == 0.0)


# ---------------------------------------------------------------- argmax

def test_argmax_first_and_lm_head_ties():
    assert O.argmax_first(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    rng = np.random.default_rng(9)
    codes, scales = _rand_nvfp4(10, 64, rng)
    codes[7] = codes[2]
    scales[7] = scales[2]
    a = _rand_bf16((3, 64), rng)
    ids, logits = O.lm_head_argmax(a, codes, scales, 0.5)
    assert np.array_equal(logits[:, 2], logits[:, 7])
    for r in range(3):
        row = logits[r]
        assert ids[r] == min(j for j in range(10) if row[j] == row.max())
    codes[:] = 0
    ids, _ = O.lm_head_argmax(a, codes, scales, 0.5)
    assert np.all(ids == 0)


def test_hot_vocab_head_whole_list_is_the_head():
    """Listing every row in order reduces the hot head to the full head."""
    rng = np.random.default_rng(21)
    codes, scales = _rand_nvfp4(40, 64, rng)
    a = _rand_bf16((3, 64), rng)
    ids, logits = O.hot_vocab_head_argmax(a, codes, scales, 0.5, np.arange(40))
    ref_ids, ref_logits = O.lm_head_argmax(a, codes, scales, 0.5)
    assert np.array_equal(ids, ref_ids) and np.array_equal(logits, ref_logits)


def test_hot_vocab_head_rows_and_ids_come_from_the_full_head():
    """The listed rows' logits are the full head's logits of those rows (each
    dot product is independent), and the answer is a vocabulary id: the
    listed id with the largest logit, the first in list order on a tie."""
    rng = np.random.default_rng(22)
    codes, scales = _rand_nvfp4(60, 96, rng)
    a = _rand_bf16((4, 96), rng)
    _, full = O.lm_head_argmax(a, codes, scales, 0.5)
    full_ids = O.argmax_first(full, axis=1)
    for lst in (rng.permutation(60)[:17], np.array([full_ids[0], 3, 59, 0]),
                np.setdiff1d(np.arange(60), full_ids)[::-1]):
        ids, logits = O.hot_vocab_head_argmax(a, codes, scales, 0.5, lst)
        assert np.array_equal(logits, full[:, lst])
        for r in range(4):
            best = max(range(len(lst)), key=lambda j: (full[r, lst[j]], -j))
            assert ids[r] == lst[best]
    # the full head's choice, when listed, is the hot head's choice
    ids, _ = O.hot_vocab_head_argmax(a, codes, scales, 0.5, np.array([full_ids[1], 7, 8]))
    assert ids[1] == full_ids[1]


def test_hot_vocab_head_ties_go_to_list_order_and_bad_ids_are_zero_rows():
    rng = np.random.default_rng(23)
    codes, scales = _rand_nvfp4(12, 64, rng)
    a = _rand_bf16((2, 64), rng)
    _, full = O.lm_head_argmax(a, codes, scales, 0.5)
    # a head whose only non-zero rows are two identical rows 9 and 4, with a
    # positive logit (the activations' sign flipped where needed): the first
    # of the two in list order wins, whichever vocabulary id is lower
    tied, tied_s = np.zeros_like(codes), scales.copy()
    tied[9], tied[4], tied_s[9] = codes[4], codes[4], scales[4]
    a = a * np.where(full[:, 4] < 0, -1.0, 1.0)[:, None]
    lg = O.gemm_bf16(a, tied, tied_s, 0.5)
    assert np.array_equal(lg[:, 9], lg[:, 4]) and np.all(lg[:, 4] > 0)
    ids, _ = O.hot_vocab_head_argmax(a, tied, tied_s, 0.5, np.array([0, 9, 4]))
    assert np.array_equal(ids, [9, 9])
    ids, _ = O.hot_vocab_head_argmax(a, tied, tied_s, 0.5, np.array([0, 4, 9]))
    assert np.array_equal(ids, [4, 4])
    # ids outside [0, N) are all-zero rows: logit exactly 0
    _, full = O.lm_head_argmax(a, codes, scales, 0.5)
    ids, logits = O.hot_vocab_head_argmax(a, codes, scales, 0.5, np.array([-1, 3, 12]))
    assert np.all(logits[:, 0] == 0.0) and np.all(logits[:, 2] == 0.0)
    assert np.array_equal(logits[:, 1], full[:, 3])


# ---------------------------------------------------------------- FP8 and BF16 weights

@pytest.mark.parametrize("m,n,k", [(1, 1, 16), (2, 3, 40), (3, 2, 64)])
def test_fp8_gemm_matches_exact_rational_brute_force(m, n, k):
    """FP8 weights decoded by torch's E4M3 table (not the oracle's), exact
    rational sums, one rounding to BF16."""
    e4 = _torch_e4m3_values()
    rng = np.random.default_rng(50 + k)
    a = _rand_bf16((m, k), rng)
    w = rng.integers(0, 256, size=(n, k), dtype=np.uint8)
    w[(w & 0x7F) == 0x7F] = 0x38  # no NaN bytes
    scale = 0.0078125 * 3  # float32-exact
    c64 = O.fp8_gemm64(a, w, scale)
    cb = O.fp8_gemm_bf16(a, w, scale)
    for i in range(m):
        for j in range(n):
            exact = sum((Fraction(float(a[i, kk])) * Fraction(float(e4[w[j, kk]])) * Fraction(scale)
                         for kk in range(k)), Fraction(0))
            bound = sum(abs(float(a[i, kk])) for kk in range(k)) * 448 * scale * k * 2 ** -52
            assert abs(Fraction(c64[i, j]) - exact) <= Fraction(bound) + Fraction(2) ** -1070
            assert cb[i, j] == _nearest_bf16_exact(exact)


def test_fp8_gemm_closed_forms():
    """All weights 1.0 (byte 0x38): each output is the row sum times the
    scale; a one-hot activation reads back one weight column; the per-tensor
    scale is linear (a power of two exactly)."""
    rng = np.random.default_rng(51)
    a = _rand_bf16((3, 64), rng)
    ones = np.full((5, 64), 0x38, dtype=np.uint8)
    assert np.allclose(O.fp8_gemm64(a, ones, 0.5), a.sum(axis=1, keepdims=True) * 0.5 * np.ones((1, 5)),
                       rtol=1e-14, atol=0)
    w = rng.integers(0, 0x7E, size=(7, 64), dtype=np.uint8)
    hot = np.zeros((1, 64))
    hot[0, 9] = 1.0
    assert np.array_equal(O.fp8_gemm64(hot, w, 1.0)[0], O.E4M3_TABLE[w[:, 9]])
    assert np.array_equal(O.fp8_gemm64(a, w, 0.25) * 4, O.fp8_gemm64(a, w, 1.0))


def test_bf16_weight_gemm_brute_force_and_expanded_nvfp4_identity():
    """BF16 weights: exact rational brute force; and the page's claim that 4-bit
    weights expanded to BF16 at load give identical numbers: every NVFP4 weight
    (code x scale x 0.5) is a BF16 value, so the BF16-weight GEMM of the
    expansion equals the NVFP4 GEMM."""
    rng = np.random.default_rng(52)
    a = _rand_bf16((2, 48), rng)
    w = _rand_bf16((3, 48), rng)
    cb = O.bf16w_gemm_bf16(a, w)
    for i in range(2):
        for j in range(3):
            exact = sum((Fraction(float(a[i, kk])) * Fraction(float(w[j, kk])) for kk in range(48)),
                        Fraction(0))
            assert cb[i, j] == _nearest_bf16_exact(exact)
    codes, scales = _rand_nvfp4(64, 256, rng, 0x01, 0x7E)
    wx = O.dequant(codes, scales, 0.5)
    assert np.array_equal(wx, O.bf16_round(wx))
    a = _rand_bf16((4, 256), rng)
    assert np.array_equal(O.bf16w_gemm64(a, wx), O.gemm64(a, codes, scales, 0.5))


# ---------------------------------------------------------------- quantiser BF16 -> NVFP4

def _grid_probe(grid, rng, top):
    """Every grid point and midpoint, the float32 neighbours of each
    midpoint, and random values, all within [0, top]."""
    g32 = grid.astype(np.float32)
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    vals = np.concatenate([g32, mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(1e9)),
                           rng.uniform(0, top, 3000).astype(np.float32),
                           (2.0 ** rng.uniform(-12, np.log2(top), 3000)).astype(np.float32)])
    return vals[vals <= top]


def test_e4m3_rounding_matches_torch_conversion():
    vals = _grid_probe(O.E4M3_TABLE[:127], np.random.default_rng(31), 448.0)
    want = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.round_to_e4m3(vals), want)
    assert np.all(O.round_to_e4m3([448.0, 449.0, 464.0, 1e6]) == 0x7E)  # saturates


def test_e2m1_rounding_matches_ml_dtypes_conversion():
    ml = pytest.importorskip("ml_dtypes")
    vals = _grid_probe(O.E2M1_TABLE[:8], np.random.default_rng(32), 6.0)
    want = vals.astype(ml.float4_e2m1fn).view(np.uint8) & 0xF
    assert np.array_equal(O.round_to_e2m1(vals), want)
    assert np.all(O.round_to_e2m1([6.0, 6.5, 100.0]) == 7)  # saturates


@pytest.mark.parametrize("g", [1.0, 2.0 ** -5])
def test_quantize_recovers_an_nvfp4_matrix_exactly(g):
    """A matrix that is exactly an NVFP4 matrix whose blocks each hold a +-6
    and whose largest scale is 448 quantises back to the same bytes."""
    rng = np.random.default_rng(33)
    n, k = 12, 128
    codes = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    lo, hi = codes & 0xF, codes >> 4
    lo = np.where(lo == 8, 0, lo)                       # no -0 (quantises to +0)
    lo[:, ::8] = np.where(rng.random((n, k // 16)) < 0.5, 7, 15)  # a +-6 in every block
    codes = (lo | (np.where(hi == 8, 0, hi) << 4)).astype(np.uint8)
    scales = rng.integers(0x08, 0x7E, size=(n, k // 16), dtype=np.uint8)
    scales[3, 5] = 0x7E
    w = O.dequant(codes, scales, g)
    assert np.array_equal(w, O.bf16_round(w))          # a BF16 matrix
    c2, s2, g2 = O.nvfp4_quantize(w)
    assert g2 == g and np.array_equal(s2, scales) and np.array_equal(c2, codes)


def test_quantize_error_bound_and_scale_cover():
    """Random BF16 weights (normal, and magnitudes spread over 2^-20 .. 2^6):
    every element is within half an E2M1 step of |x| / (scale * g), except
    where the block maximum saturates at 6 because its E4M3 scale rounded
    down (by at most 2^-4 relative), and the round trip has the right sign."""
    rng = np.random.default_rng(34)
    for w in (_rand_bf16((64, 256), rng),
              O.bf16_round(rng.choice([-1, 1], (64, 256)) * 2.0 ** rng.uniform(-20, 6, (64, 256)))):
        codes, scales, g = O.nvfp4_quantize(w)
        d = np.repeat(O.E4M3_TABLE[scales] * np.float32(g), 16, axis=1)
        q = O.dequant(codes, scales, g)
        ok = d > 0
        v = np.abs(w[ok]) / d[ok]
        step = np.where(v < 2, 0.5, np.where(v < 4, 1.0, 2.0))
        err = np.abs(np.abs(q[ok]) / d[ok] - v)
        sat = v > 6
        assert np.all(err[~sat] <= step[~sat] / 2 * (1 + 1e-6))
        assert np.all(v[sat] <= 6 / (1 - 2.0 ** -4) * (1 + 1e-6))
        assert np.all((np.sign(q) == np.sign(w)) | (q == 0))
        amax_b = np.abs(w).reshape(64, 16, 16).max(axis=2)
        assert np.all(O.E4M3_TABLE[scales] * g * 6 >= amax_b * (1 - 2.0 ** -4) * (1 - 1e-6))


def test_quantize_zero_matrix_and_signless_zeros():
    codes, scales, g = O.nvfp4_quantize(np.zeros((2, 32)))
    assert g == 1.0 and not codes.any() and not scales.any()
    w = np.zeros((1, 32))
    w[0, 0] = -6.0
    w[0, 1], w[0, 2] = -1e-3, 1e-3  # round to zero: code 0, never -0 (8)
    codes, scales, g = O.nvfp4_quantize(w)
    assert codes[0, 0] == (15 | (0 << 4)) and codes[0, 1] == 0
    q = O.dequant(codes, scales, g)[0, :3]
    assert abs(q[0] + 6.0) < 1e-5 and q[1] == 0.0 and q[2] == 0.0


# ---------------------------------------------------------------- bytes + roofline (pages)

def _figs(golden_dir):
    return json.load(open(os.path.join(golden_dir, "pages_worked_figures.json")))


def test_weight_bytes_definition():
    assert O.nvfp4_weight_bytes(64, 2048) == 73728
    assert O.nvfp4_weight_bytes(4096, 2048) == 4718592
    assert O.nvfp4_weight_bytes(151936, 2048) == 175030272


def test_hot_vocab_head_bytes_match_page(golden_dir):
    f = _figs(golden_dir)["hot_vocab_head"]
    full = O.nvfp4_weight_bytes(f["full_rows"], f["hidden"]) / 1e6
    hot = O.nvfp4_weight_bytes(f["hot_rows"], f["hidden"]) / 1e6
    assert abs(full - f["full_printed_mb"]) <= f["printed_mb_resolution"]["full"] / 2
    assert abs(hot - f["hot_printed_mb"]) <= f["printed_mb_resolution"]["hot"] / 2
    # the scale overhead matters: 4 bits alone, or one byte per 32, miss the figures
    assert abs(f["hot_rows"] * f["hidden"] * 0.5 / 1e6 - f["hot_printed_mb"]) > 0.5
    assert abs(f["hot_rows"] * f["hidden"] * (0.5 + 1 / 32) / 1e6 - f["hot_printed_mb"]) > 0.5


def test_skinny_projection_bf16_bytes_match_page(golden_dir):
    f = _figs(golden_dir)["skinny_projection_bf16"]
    assert f["rows"] * f["k"] * 2 == f["printed_kib"] * 1024
    # the NVFP4 copy of the same projection moves 0.5625 / 2 of those bytes
    assert O.nvfp4_weight_bytes(f["rows"], f["k"]) / (f["printed_kib"] * 1024) == 0.5625 / 2


def test_decode_roofline_matches_page(golden_dir):
    f = _figs(golden_dir)["decode_roofline"]
    wbytes = f["weight_gb"] * 1e9
    # RTX 5090: about 1.8 TB/s over 18.7 GB of weights -> 95.8 tok/s (printed)
    roof = O.decode_roofline_tok_s(f["rtx5090_bandwidth_tb_s"] * 1e12, wbytes)
    assert abs(roof - 95.8) / 95.8 < 0.03
    # the bandwidth implied by the printed roofline is 'about 1.8 TB/s'
    assert abs(95.8 * wbytes / 1e12 - 1.8) < 0.05
    consistent = [r for r in f["rows"] if r["card"] != "RTX 5090, before"]
    for r in consistent:
        share = 100 * O.roofline_share(r["measured_tok_s"], r["roofline_tok_s"])
        assert abs(share - r["printed_share_pct"]) <= 0.5, r
    # the 'before' row prints 8% where 6.4 / 95.8 gives 6.7%: a slip on the page
    before = [r for r in f["rows"] if r["card"] == "RTX 5090, before"][0]
    share = 100 * O.roofline_share(before["measured_tok_s"], before["roofline_tok_s"])
    assert 6.0 < share < 7.0 and before["printed_share_pct"] == 8
    m = f["mtp"]
    assert abs(m["forwards_per_s"] * m["tokens_per_forward"] - m["measured_tok_s"]) < 0.5


def test_moe_weight_bytes_counts_unique_experts():
    ids = np.array([[1, 2, 3], [3, 2, 9], [300, -1, 1]])
    per = O.nvfp4_weight_bytes(1024, 2048) + O.nvfp4_weight_bytes(2048, 512)
    assert per == 1769472
    assert O.moe_weight_bytes(ids, 256, 2048, 512) == (4 + 1) * per
    assert O.moe_weight_bytes(ids, 256, 2048, 512, shared=False) == 4 * per
