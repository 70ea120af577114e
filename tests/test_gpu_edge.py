"""GPU parity where the kernels' arithmetic departs from plain BF16: the
activation rows are staged as FP16 after a power-of-two shift per row (the
row's largest magnitude moved to [2^14, 2^15)), and the weights are decoded
to FP16 as code x block scale.  These cases reach the corners of that
scheme:

* all-zero activation rows (no shift; an RMS-scaled zero row stays zero);
* rows at the ends of BF16's range (2^110, 2^-120, BF16 subnormals);
* one row spanning 2^60 of dynamic range (its smallest elements fall below
  FP16 after the shift and are lost: a relative error under 2^-40 of the
  row's largest term);
* E4M3 block scales over every finite code 0x01..0x7E (subnormals 0x01..0x07
  and the maximum 448 = 0x7E) with codes +-6 and all 16 codes;
* MoE experts whose gate rows are all zero (h = silu(0) * u = 0: the down
  projection stages all-zero rows), and a token whose activation row is
  zero.

Every expected value comes from the float64 oracle on the same inputs."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, check_argmax, device_experts, device_shared, f64, host_expert_fn
from moe_expert_nvfp4_gb300 import ops, synth

pytestmark = pytest.mark.gpu
E, H, I, TOPK = 256, 2048, 512, 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_nvfp4_gb300 import build
    build.build()
    ops.load()
    assert ops.device_check(torch.cuda.current_device()) == 0, ops.last_error()


def _bf16(x: np.ndarray) -> torch.Tensor:
    """float64 values -> BF16 tensor (round to nearest even)."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def _gemm_case(a_host: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, rms=False,
               argmax=False, what="", path="call"):
    """path "call": the single call (these small shapes dispatch to the
    CUDA-core kernel); "tc": the same GEMM as a one-op program, which always
    runs on the tensor cores."""
    g = torch.full((1,), synth.GLOBAL_SCALE, dtype=torch.float32, device="cuda")
    W = ops.NVFP4Weight(codes.cuda(), scales.cuda(), g)
    a = a_host.cuda()
    if path == "call":
        ws = ops.Workspace(ops.gemm_workspace_bytes(a.shape[0], W.n, W.k))
        res = ops.gemm(a, W, rms_input=rms, argmax=argmax, workspace=ws)
        assert ops.last_dispatch().startswith("fma_kernel")
    else:
        c = torch.empty(a.shape[0], W.n, dtype=torch.bfloat16, device="cuda")
        am = torch.empty(a.shape[0], dtype=torch.int32, device="cuda") if argmax else None
        prog = ops.Program([ops.gemm_op(a, W, c, argmax_out=am, rms_input=rms, all_sms=True)])
        prog.launch()
        ws = prog.workspace
        res = (c, am) if argmax else c
    torch.cuda.synchronize()
    assert ws.status() == 0
    a64 = f64(a_host)
    ref = O.gemm64(O.rms_scale(a64) if rms else a64, codes.numpy(), scales.numpy(),
                   synth.GLOBAL_SCALE)
    c = res[0] if argmax else res
    assert np.all(np.isfinite(f64(c))), what
    assert_close(f64(c), O.bf16_round(ref), what)
    if argmax:
        check_argmax(res[1].cpu().numpy(), f64(c), ref, what=what)
    return f64(c), ref


PATHS = ["call", "tc"]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("rms", [False, True])
def test_zero_activation_rows(rms, path):
    m, n, k = 6, 640, 2048
    codes, scales = synth.nvfp4_weight(41, n, k)
    a = synth.activations_bf16(41, m, k)
    a[1] = 0
    a[4] = 0
    c, _ = _gemm_case(a, codes, scales, rms=rms, what=f"zero rows rms={rms} {path}", path=path)
    assert np.all(c[1] == 0) and np.all(c[4] == 0)


@pytest.mark.parametrize("path", PATHS)
def test_rows_at_the_ends_of_bf16_range(path):
    m, n, k = 5, 384, 2048
    codes, scales = synth.nvfp4_weight(42, n, k)
    base = f64(synth.activations_bf16(42, m, k))
    a = np.stack([base[0] * 2.0 ** 110,        # large: outputs near 2^117
                  base[1] * 2.0 ** -120,       # small: some elements BF16 subnormal
                  base[2] * 2.0 ** -128,       # most elements BF16 subnormal
                  base[3],
                  base[4] * 2.0 ** 60])
    _gemm_case(_bf16(a), codes, scales, what=f"2^110 / 2^-120 / 2^-128 rows {path}", path=path)
    _gemm_case(_bf16(a), codes, scales, rms=True, what=f"extreme rows, RMS input {path}",
               path=path)


@pytest.mark.parametrize("path", PATHS)
def test_row_with_2_pow_60_dynamic_range(path):
    m, n, k = 3, 512, 2048
    codes, scales = synth.nvfp4_weight(43, n, k)
    base = f64(synth.activations_bf16(43, m, k))
    tiers = 2.0 ** (-np.arange(k) % 61)          # magnitudes 2^0 .. 2^-60 along the row
    a = base * tiers[None, :]
    _gemm_case(_bf16(a), codes, scales, what=f"2^60 range {path}", path=path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("codes_kind", ["pm6", "all16"])
def test_every_finite_e4m3_scale(codes_kind, path):
    """Scales cycle through 0x01..0x7E (126 finite positive codes, subnormal
    to 448); codes are +-6 (0x7 / 0xF) or all 16 codes."""
    m, n, k = 8, 800, 2048
    codes, _ = synth.nvfp4_weight(44, n, k)
    nb = k // 16
    idx = (np.arange(n)[:, None] * 7 + np.arange(nb)[None, :]) % 126
    scales = torch.from_numpy((idx + 1).astype(np.uint8))
    if codes_kind == "pm6":
        sign = torch.from_numpy(np.random.default_rng(44).integers(0, 2, size=(n, k // 2, 2),
                                                                   dtype=np.uint8))
        lo = 0x7 | (sign[..., 0] << 3)
        hi = 0x7 | (sign[..., 1] << 3)
        codes = (lo | (hi << 4)).to(torch.uint8)
    _gemm_case(synth.activations_bf16(44, m, k), codes, scales, argmax=True,
               what=f"all E4M3 scales, codes {codes_kind} {path}", path=path)


@pytest.fixture(scope="module")
def layer_zero_gates():
    """The seed-4 layer with the gate rows of experts 0..127 set to code 0
    (+0), and the same for the shared expert."""
    ex = device_experts(4, 0, E, H, I)
    sh = device_shared(4, 0, E, H, I)
    ex.gu_codes[:128, :I] = 0
    sh.gu_codes[:, :I] = 0
    get = host_expert_fn(4, 0, H, I)

    def host(e):
        gc, gs, gg, dc, ds, dg = get(e)
        if e < 128 or e == E:
            gc = gc.copy()
            gc[:I] = 0
        return gc, gs, gg, dc, ds, dg
    return ex, sh, host


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("t", [1, 8, 32])
def test_moe_all_zero_h_rows(layer_zero_gates, t, path):
    """path "call": the single call (the CUDA-core kernels, in batches of 16
    tokens); "tc": a one-op program (the tensor-core kernels)."""
    ex, sh, get = layer_zero_gates
    x = synth.activations_bf16(45, t, H)
    ids, w = ops.route(synth.router_logits(45, t, E).cuda(), TOPK)
    if path == "call":
        ws = ops.Workspace(ops.moe_workspace_bytes(t, TOPK, ex))
        out = ops.moe(x.cuda(), ids, w, ex, sh, workspace=ws)
    else:
        out = torch.empty(t, H, dtype=torch.bfloat16, device="cuda")
        prog = ops.Program([ops.moe_op(x.cuda(), ids, w, ex, out, shared=sh)])
        prog.launch()
        ws = prog.workspace
    torch.cuda.synchronize()
    assert ws.status() == 0
    ref = O.moe_decode_bf16(f64(x), ids.cpu().numpy(), w.cpu().double().numpy(), get, E, get(E))
    assert_close(f64(out), ref, f"zero-gate experts T={t}")


@pytest.mark.parametrize("rms", [False, True])
def test_moe_zero_token_row(rms):
    """(8 tokens: the CUDA-core MoE kernels.)"""
    ex = device_experts(4, 0, E, H, I)
    sh = device_shared(4, 0, E, H, I)
    get = host_expert_fn(4, 0, H, I)
    t = 8
    x = synth.activations_bf16(46, t, H)
    x[2] = 0
    ids, w = ops.route(synth.router_logits(46, t, E).cuda(), TOPK)
    out = ops.moe(x.cuda(), ids, w, ex, sh, rms_input=rms)
    torch.cuda.synchronize()
    x64 = f64(x)
    ref = O.moe_decode_bf16(O.rms_scale(x64) if rms else x64, ids.cpu().numpy(),
                            w.cpu().double().numpy(), get, E, get(E))
    assert_close(f64(out), ref, f"zero token row rms={rms}")
    assert np.all(f64(out)[2] == 0)


def test_extreme_rows_on_the_cuda_core_kernel():
    """The same extreme rows with K = 2080 (the CUDA-core kernel)."""
    m, n, k = 5, 384, 2080
    codes, scales = synth.nvfp4_weight(47, n, k)
    base = f64(synth.activations_bf16(47, m, k))
    a = np.stack([base[0] * 2.0 ** 110, base[1] * 2.0 ** -120, base[2] * 2.0 ** -128, base[3],
                  base[4] * 2.0 ** 60])
    _gemm_case(_bf16(a), codes, scales, what="K=2080 extreme rows")
    _gemm_case(_bf16(a), codes, scales, rms=True, what="K=2080 extreme rows, RMS input")
