"""The K order of the warp-MMA gate/up kernel (``moe_mma_gate_up_kernel`` in
``csrc/moe_fma.cu``) checked as host logic.

Per 128-K chunk, lane (g, q) = (lane // 4, lane % 4) loads 16 bytes of codes
of tile rows g and g + 8 (elements 32 q .. 32 q + 31 of the chunk) and the
token's 32 activations of the same range.  Byte j of a row's 16 bytes holds
elements 2 j, 2 j + 1 (low nibble first) and goes to k-step j // 2: as the
A register of K slots {2q, 2q + 1} when j is even, of {2q + 8, 2q + 9} when
odd; the activation words go to the B registers of the same K slots.  With
the register layout the PTX ISA gives for mma.m16n8k16 (f16 A and B, f32
C / D), the eight k-steps of a chunk must add every product of the chunk
exactly once, in every column.
"""
import numpy as np


def _a_fragment(lane):
    """(row, K slot pair) of the A registers a0..a3 of a lane."""
    g, q = lane // 4, lane % 4
    return [(g, 2 * q), (g + 8, 2 * q), (g, 2 * q + 8), (g + 8, 2 * q + 8)]


def _b_fragment(lane):
    """(K slot pair, column) of the B registers b0, b1 of a lane."""
    g, q = lane // 4, lane % 4
    return [(2 * q, g), (2 * q + 8, g)]


def _kernel_elements(lane, step):
    """Chunk elements the kernel puts into a lane's registers at k-step
    ``step``: A registers a0..a3 (row g: bytes 2 step, 2 step + 1 of the
    lane's 16; row g + 8 likewise) and B registers b0, b1 (the token's
    elements in the same order)."""
    q = lane % 4
    base = 32 * q + 4 * step          # byte 2 step -> elements base, base + 1
    a = [base, base, base + 2, base + 2]   # a0 (row g), a1 (row g+8), a2, a3
    b = [base, base + 2]
    return a, b


def _emulate(W, x, elements=_kernel_elements):
    """D (16 x 8) after the eight k-steps of one chunk, FP64."""
    D = np.zeros((16, 8))
    for step in range(8):
        A = np.full((16, 16), np.nan)
        B = np.full((16, 8), np.nan)
        for lane in range(32):
            ea, eb = elements(lane, step)
            for (row, ks), e in zip(_a_fragment(lane), ea):
                A[row, ks], A[row, ks + 1] = W[row, e], W[row, e + 1]
            for (ks, col), e in zip(_b_fragment(lane), eb):
                B[ks, col], B[ks + 1, col] = x[e], x[e + 1]
        assert not np.isnan(A).any() and not np.isnan(B).any()
        D += A @ B
    return D


def test_every_product_of_a_chunk_added_once():
    rng = np.random.default_rng(0)
    W = rng.standard_normal((16, 128))
    x = rng.standard_normal(128)
    D = _emulate(W, x)
    want = W @ x
    for col in range(8):
        np.testing.assert_allclose(D[:, col], want, rtol=1e-12, atol=1e-12)


def test_each_element_in_exactly_one_k_step():
    for row_half in (0, 1):
        seen = np.zeros((8, 128), int)   # (row g, element) uses over the k-steps
        for step in range(8):
            for lane in range(32):
                g = lane // 4
                ea, _ = _kernel_elements(lane, step)
                for r in range(4):
                    if (r % 2) == row_half:
                        seen[g, ea[r]] += 1
                        seen[g, ea[r] + 1] += 1
        assert (seen == 1).all()


def test_a_dropped_offset_is_caught():
    """The check fails for a plausible slip: both A halves from the same
    element pair."""
    rng = np.random.default_rng(1)
    W = rng.standard_normal((16, 128))
    x = rng.standard_normal(128)

    def slipped(lane, step):
        a, b = _kernel_elements(lane, step)
        return [a[0], a[1], a[0], a[1]], b

    D = _emulate(W, x, slipped)
    assert not np.allclose(D[:, 0], W @ x)
