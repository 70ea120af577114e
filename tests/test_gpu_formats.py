"""GPU parity of the dense path with the other two weight formats, against the
float64 oracle:

* FP8-E4M3 weights with one per-tensor scale, BF16 activations (W8A16;
  "Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)", section "Making decode
  faster", paragraph "An FP8 fast path that never ran"): the attention-like
  projection shapes (QKV 2048 -> 5120, O 4096 -> 2048) at M = 1..32, ragged
  shapes, RMS-scaled input, argmax, determinism;
* BF16 weights (same page, paragraph "Skinny matrix multiplies": the
  2048 -> 64 projection and 4-bit shared experts expanded to BF16 at load):
  the 2048 -> 64 projection at M = 4, larger shapes, and the expansion
  identity on the GPU -- an NVFP4 matrix expanded to BF16 gives the NVFP4
  GEMM's result.

Inputs: seeded synthetic weights (FP8 bytes of N(0,1) * 8 draws with scale
1/64; BF16 N(0,1)/16 draws) and N(0,1) BF16 activations."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, check_argmax, device_weight, f64, host_weight
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


def _fp8(seed, n, k):
    codes = synth.fp8_weight(seed, n, k)
    scale = torch.full((1,), synth.FP8_SCALE, dtype=torch.float32, device="cuda")
    return ops.FP8Weight(codes.cuda(), scale), codes.numpy()


def _fp8_case(seed, m, n, k, rms=False, argmax=False):
    W, host = _fp8(seed, n, k)
    a = synth.activations_bf16(seed, m, k, 50)
    res = ops.fp8_gemm(a.cuda(), W, rms_input=rms, argmax=argmax)
    disp = ops.last_dispatch()
    torch.cuda.synchronize()
    a64 = f64(a)
    ref = O.fp8_gemm64(O.rms_scale(a64) if rms else a64, host, synth.FP8_SCALE)
    return res, ref, disp


@pytest.mark.parametrize("m", [1, 4, 8, 16, 32])
@pytest.mark.parametrize("n,k", [(5120, 2048), (2048, 4096)])
def test_fp8_projection_shapes(m, n, k):
    c, ref, disp = _fp8_case(51, m, n, k)
    assert disp.startswith("stream_tc_kernel<dense> weight=fp8")
    assert_close(f64(c), O.bf16_round(ref), f"fp8 M={m} N={n} K={k}")


@pytest.mark.parametrize("m,n,k", [(3, 200, 768), (27, 1000, 256), (1, 64, 256), (32, 129, 2304),
                                   (9, 7, 512), (17, 3000, 6144)])
def test_fp8_ragged_shapes(m, n, k):
    c, ref, _ = _fp8_case(52, m, n, k)
    assert_close(f64(c), O.bf16_round(ref), f"fp8 ragged M={m} N={n} K={k}")


def test_fp8_rms_input_and_argmax():
    (c, am), ref, disp = _fp8_case(53, 8, 3000, 2048, rms=True, argmax=True)
    assert "rms=1" in disp and "argmax=1" in disp
    assert_close(f64(c), O.bf16_round(ref), "fp8 rms + argmax")
    check_argmax(am.cpu().numpy(), f64(c), ref, what="fp8 argmax")


def test_fp8_deterministic():
    W, _ = _fp8(54, 4096, 2048)
    a = synth.activations_bf16(54, 16, 2048).cuda()
    ws = ops.Workspace(ops.load().fp8_gemm_skinny_workspace(16, 4096, 2048))
    outs = [ops.fp8_gemm(a, W, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    assert ws.status() == 0


def _bf16_case(seed, m, n, k, rms=False, argmax=False, ld=None):
    w = synth.bf16_weight(seed, n, ld or k)
    a = synth.activations_bf16(seed, m, k, 60)
    wd = w.cuda()[:, :k]
    res = ops.bf16w_gemm(a.cuda(), wd, rms_input=rms, argmax=argmax)
    disp = ops.last_dispatch()
    torch.cuda.synchronize()
    a64 = f64(a)
    ref = O.bf16w_gemm64(O.rms_scale(a64) if rms else a64, f64(w[:, :k]))
    return res, ref, disp


def test_bf16_projection_2048_to_64_m4():
    c, ref, disp = _bf16_case(61, 4, 64, 2048)
    assert disp.startswith("stream_tc_kernel<dense> weight=bf16")
    assert_close(f64(c), O.bf16_round(ref), "bf16 2048->64")


@pytest.mark.parametrize("m", [1, 8, 32])
@pytest.mark.parametrize("n,k", [(4096, 2048), (2048, 4096)])
def test_bf16_shapes(m, n, k):
    c, ref, _ = _bf16_case(62, m, n, k)
    assert_close(f64(c), O.bf16_round(ref), f"bf16 M={m} N={n} K={k}")


@pytest.mark.parametrize("m,n,k,ld", [(3, 200, 768, None), (27, 1000, 256, None),
                                      (32, 129, 2304, 2312), (9, 7, 512, None),
                                      (17, 3000, 6144, None)])
def test_bf16_ragged_and_strided(m, n, k, ld):
    c, ref, _ = _bf16_case(63, m, n, k, ld=ld)
    assert_close(f64(c), O.bf16_round(ref), f"bf16 ragged M={m} N={n} K={k}")


def test_bf16_rms_input_and_argmax():
    (c, am), ref, _ = _bf16_case(64, 8, 3000, 2048, rms=True, argmax=True)
    assert_close(f64(c), O.bf16_round(ref), "bf16 rms + argmax")
    check_argmax(am.cpu().numpy(), f64(c), ref, what="bf16 argmax")


@pytest.mark.parametrize("m", [4, 16])
def test_nvfp4_expanded_to_bf16_gives_the_nvfp4_result(m):
    """The pages' claim, on the GPU: the 4-bit matrix expanded to BF16 (exact:
    each code x block scale x tensor scale has at most 6 significant bits)
    through the BF16-weight kernel agrees with the NVFP4 kernel on the 4-bit
    matrix, and both with the oracle."""
    n, k = 2048, 2048
    W = device_weight(65, n, k)
    codes, scales, g = host_weight(65, n, k)
    wexp = O.dequant(codes, scales, g)
    wb = torch.from_numpy(wexp.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(f64(wb), wexp)          # the expansion is exact
    a = synth.activations_bf16(65, m, k).cuda()
    c4 = ops.gemm(a, W)
    cb = ops.bf16w_gemm(a, wb.cuda())
    torch.cuda.synchronize()
    ref = O.gemm64(f64(a), codes, scales, g)
    assert_close(f64(c4), O.bf16_round(ref), "nvfp4")
    assert_close(f64(cb), O.bf16_round(ref), "expanded bf16")
    # the two GPU results differ only by FP32 summation order: at most one
    # BF16 rounding step apart
    d = np.abs(f64(c4) - f64(cb))
    step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(f64(c4)), 1e-30))) - 7)
    assert np.all(d <= step), float(np.max(d / step))
