"""GPU parity of the dense NVFP4 skinny GEMM against the float64 oracle."""
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


def _case(seed, m, n, k, *ids, rms=False, argmax=False, lda=None):
    W = device_weight(seed, n, k, *ids)
    a_full = synth.activations_bf16(seed, m, lda or k, 900, *ids)
    a = a_full.cuda()[:, :k] if lda else a_full.cuda()
    ws = ops.Workspace(ops.gemm_workspace_bytes(m, n, k))
    res = ops.gemm(a, W, argmax=argmax, rms_input=rms, workspace=ws)
    disp = ops.last_dispatch()
    torch.cuda.synchronize()
    assert ws.status() == 0
    a64 = f64(a_full[:, :k])
    ref64 = O.gemm64(O.rms_scale(a64) if rms else a64, *host_weight(seed, n, k, *ids))
    return res, ref64, disp, (W, a, ws)


def test_generator_bytes_identical_on_device_and_host():
    c, s = synth.nvfp4_weight(3, 300, 2048, 5, device="cuda")
    ch, sh = synth.nvfp4_weight(3, 300, 2048, 5)
    assert torch.equal(c.cpu(), ch) and torch.equal(s.cpu(), sh)


def test_projection_2048_to_64_m4():
    c, ref, disp, (W, a, _) = _case(0, 4, 64, 2048)
    assert_close(f64(c), O.bf16_round(ref), "2048->64")
    assert disp.startswith("fma_kernel")                 # small: the CUDA-core kernel
    # the tensor-core kernel on the same call (a one-op program with every
    # op split as its tensor-core call would be: 1 tile x 2 K splits)
    out = torch.empty_like(c)
    prog = ops.Program([ops.gemm_op(a, W, out, all_sms=True)])
    prog.launch()
    torch.cuda.synchronize()
    assert prog.workspace.status() == 0
    assert_close(f64(out), O.bf16_round(ref), "2048->64 tensor cores")


@pytest.mark.parametrize("m,n,k,kernel", [(1, 4096, 2048, "fma_kernel"),
                                          (1, 151936, 2048, "stream_tc_kernel"),
                                          (2, 16384, 2048, "fma_kernel"),
                                          (2, 32768, 2048, "stream_tc_kernel"),
                                          (4, 8192, 2048, "fma_kernel"),
                                          (4, 16384, 2048, "stream_tc_kernel"),
                                          (3, 16384, 2048, "fma_kernel"),
                                          (8, 800, 2048, "fma_kernel"),
                                          (8, 2048, 4096, "fma_kernel"),
                                          (8, 4096, 2048, "stream_tc_kernel"),
                                          (9, 64, 2048, "fma_kernel"),
                                          (16, 1024, 2048, "fma_kernel"),
                                          (16, 2048, 4096, "stream_tc_kernel"),
                                          (17, 64, 2048, "stream_tc_kernel")])
def test_dispatch_by_shape(m, n, k, kernel):
    """The CUDA cores take weights up to 128 MiB at M = 1, 20 MiB at M = 2,
    3, 10 MiB at M = 4, and at M = 5..16 weights up to 5 MiB whose four-row
    CTAs fit one wave (ceil(N / 16) * ceil(M / 4) <= 2 x 152); the tensor
    cores the rest (K % 256 == 0)."""
    ws = ops.Workspace(ops.gemm_workspace_bytes(m, n, k))
    W = device_weight(30, n, k)
    a = synth.activations_bf16(30, m, k).cuda()
    ops.gemm(a, W, workspace=ws)
    assert ops.last_dispatch().startswith(kernel)
    torch.cuda.synchronize()


@pytest.mark.parametrize("m", [1, 4, 8, 16, 32])
@pytest.mark.parametrize("seed,n,k", [(1, 4096, 2048), (2, 8192, 2048), (3, 2048, 4096)])
def test_dense_sweep(seed, n, k, m):
    c, ref, disp, _ = _case(seed, m, n, k)
    assert_close(f64(c), O.bf16_round(ref), f"M={m} N={n} K={k}")


@pytest.mark.parametrize("m,n,k", [(3, 200, 768), (13, 200, 768), (27, 1000, 256), (1, 64, 256),
                                   (32, 129, 2304), (9, 7, 512), (32, 1000, 4096),
                                   (17, 3000, 6144), (11, 300, 2080), (32, 64, 1056)])
def test_ragged_shapes(m, n, k):
    c, ref, _, _ = _case(7, m, n, k)
    assert_close(f64(c), O.bf16_round(ref), f"ragged M={m} N={n} K={k}")


def test_strided_activation_rows():
    c, ref, _, _ = _case(8, 5, 320, 1024, lda=1536)
    assert_close(f64(c), O.bf16_round(ref), "lda > K")


def test_rms_input_flag():
    c, ref, disp, _ = _case(9, 8, 512, 2048, rms=True)
    assert "rms=1" in disp
    assert_close(f64(c), O.bf16_round(ref), "rms input")


def test_deterministic_split_k():
    c1, _, disp, (W, a, ws) = _case(1, 16, 4096, 2048)
    assert "grid=152" in disp or "grid=" in disp
    c2 = ops.gemm(a, W, workspace=ws)
    c3 = ops.gemm(a, W, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2) and torch.equal(c2, c3)


def test_lm_head_151936_argmax_m32():
    (c, am), ref, disp, _ = _case(5, 32, 151936, 2048, 1, argmax=True)
    assert "argmax=1" in disp and "tiles=1187" in disp
    assert_close(f64(c), O.bf16_round(ref), "lm-head")
    check_argmax(am.cpu().numpy(), f64(c), ref, what="lm-head")


def test_argmax_ties_go_to_lowest_index():
    n, k = 300, 512
    c, s = synth.nvfp4_weight(10, n, k, device="cuda")
    c[250] = c[17]
    s[250] = s[17]
    c[299] = c[3]
    s[299] = s[3]
    W = ops.NVFP4Weight(c, s, torch.full((1,), 0.5, device="cuda"))
    a = synth.activations_bf16(10, 6, k).cuda()
    C, am = ops.gemm(a, W, argmax=True)
    gl = f64(C)
    assert np.array_equal(gl[:, 250], gl[:, 17])
    assert np.array_equal(am.cpu().numpy(), O.argmax_first(gl, axis=1))
    # force a tie at the top: make row 299 (a copy of row 3) the maximum
    c[:] = 0
    c[3] = 0x22
    c[299] = 0x22
    a1 = torch.ones(2, k, dtype=torch.bfloat16, device="cuda")
    C, am = ops.gemm(a1, W, argmax=True)
    assert am.tolist() == [3, 3]


# ------------------------------------------------------------------ K % 256 != 0
# These shapes run on the CUDA-core kernel (whole rows per warp); the same
# tolerance and argmax rules hold.

@pytest.mark.parametrize("m", [1, 2, 4, 17, 32])
@pytest.mark.parametrize("n,k", [(64, 32), (1000, 96), (4096, 2080)])
def test_k_multiple_of_32(m, n, k):
    c, ref, disp, _ = _case(15, m, n, k)
    assert disp.startswith("fma_kernel")
    assert_close(f64(c), O.bf16_round(ref), f"K={k} M={m} N={n}")


def test_k_multiple_of_32_rms_and_argmax():
    (c, am), ref, disp, _ = _case(16, 8, 3000, 2080, rms=True, argmax=True)
    assert disp.startswith("fma_kernel") and "rms=1" in disp and "argmax=1" in disp
    assert_close(f64(c), O.bf16_round(ref), "K=2080 rms + argmax")
    check_argmax(am.cpu().numpy(), f64(c), ref, what="K=2080 argmax")


def test_k_multiple_of_32_deterministic_and_strided():
    c1, ref, _, (W, a, ws) = _case(17, 5, 700, 1056, lda=1200)
    assert_close(f64(c1), O.bf16_round(ref), "K=1056 lda=1200")
    c2 = ops.gemm(a, W, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)
