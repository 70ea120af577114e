"""GPU parity of the BF16 -> NVFP4 quantiser ("Qwen3.8-27B-NVFP4-lmhead4-recipe",
section "Files": a BF16 head converted to NVFP4): codes, E4M3 block scales and
the per-tensor scale bit-exact against the oracle (the codes are decided in
float32 on both sides), on normal weights from a few rows up to a
32,768 x 2048 head slice, magnitudes spread over 2^-30 .. 2^20 (subnormal and
zero block scales), an exact NVFP4 matrix (which must come back byte for
byte), the all-zero matrix and strided rows; then the quantised matrix
through the skinny GEMM against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, f64
from moe_expert_nvfp4_gb300 import ops, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_nvfp4_gb300 import build
    build.build()
    ops.load()
    assert ops.device_check(torch.cuda.current_device()) == 0, ops.last_error()


def _bf16(x) -> torch.Tensor:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def _check(w_cpu: torch.Tensor, w_dev: torch.Tensor = None) -> ops.NVFP4Weight:
    q = ops.quantize(w_cpu.cuda() if w_dev is None else w_dev)
    torch.cuda.synchronize()
    assert ops.last_dispatch().startswith("amax_kernel, quantize_kernel")
    codes, scales, g = O.nvfp4_quantize(w_cpu.float().numpy())
    assert np.float32(q.global_scale.item()) == np.float32(g)
    assert np.array_equal(q.scales.cpu().numpy(), scales)
    assert np.array_equal(q.codes.cpu().numpy(), codes)
    return q


@pytest.mark.parametrize("n,k", [(1000, 2048), (37, 4096), (5, 32), (32768, 2048)])
def test_quantize_normal_weights(n, k):
    _check(synth.activations_bf16(40, n, k))


def test_quantize_wide_magnitude_range():
    rng = np.random.default_rng(41)
    w = rng.choice([-1.0, 1.0], (300, 1024)) * 2.0 ** rng.uniform(-30, 20, (300, 1024))
    w[7, :16] = 0.0  # an all-zero block
    _check(_bf16(w))


def test_quantize_recovers_an_nvfp4_matrix_exactly():
    rng = np.random.default_rng(42)
    n, k = 64, 512
    codes = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    lo, hi = codes & 0xF, codes >> 4
    lo = np.where(lo == 8, 0, lo)
    lo[:, ::8] = np.where(rng.random((n, k // 16)) < 0.5, 7, 15)  # a +-6 in every block
    codes = (lo | (np.where(hi == 8, 0, hi) << 4)).astype(np.uint8)
    scales = rng.integers(0x08, 0x7E, size=(n, k // 16), dtype=np.uint8)
    scales[10, 3] = 0x7E
    g = 2.0 ** -7
    q = _check(_bf16(O.dequant(codes, scales, g)))
    assert np.array_equal(q.codes.cpu().numpy(), codes)
    assert np.array_equal(q.scales.cpu().numpy(), scales)
    assert q.global_scale.item() == g


def test_quantize_zero_matrix_and_strided_rows():
    q = _check(torch.zeros(8, 64, dtype=torch.bfloat16))
    assert q.global_scale.item() == 1.0
    full = synth.activations_bf16(43, 64, 2048 + 64)
    _check(full[:, :2048].contiguous(), full.cuda()[:, :2048])  # ldw = 2112


@pytest.mark.parametrize("m", [1, 8, 32])
def test_quantized_matrix_through_the_gemm(m):
    w = synth.activations_bf16(44, 4096, 2048)
    q = _check(w)
    a = synth.activations_bf16(45, m, 2048)
    c = ops.gemm(a.cuda(), q)
    torch.cuda.synchronize()
    ref = O.gemm_bf16(f64(a), q.codes.cpu().numpy(), q.scales.cpu().numpy(),
                      float(q.global_scale.item()))
    assert_close(f64(c), ref, "gemm of the quantised matrix")
