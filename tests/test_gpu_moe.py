"""GPU parity of top-k routing and the NVFP4 MoE decode layer (35B-A3B shape:
hidden 2048, 256 experts of intermediate 512, top-8, one shared expert)
against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import (assert_close, check_argmax, check_route_weights, device_experts,
                     device_shared, device_weight, f64, host_expert_fn, host_weight)
from moe_expert_nvfp4_gb300 import ops, synth

pytestmark = pytest.mark.gpu
E, H, I, K = 256, 2048, 512, 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_nvfp4_gb300 import build
    build.build()
    ops.load()
    assert ops.device_check(torch.cuda.current_device()) == 0, ops.last_error()


@pytest.fixture(scope="module")
def layer4():
    """The seed-4 expert layer on the device, and its host accessor."""
    ex = device_experts(4, 0, E, H, I)
    sh = device_shared(4, 0, E, H, I)
    get = host_expert_fn(4, 0, H, I)
    return ex, sh, get


# ------------------------------------------------------------------ routing

def _check_route(logits, k, renorm=True):
    ids, w = ops.route(logits.cuda(), k, renorm)
    rid, rw = O.topk_softmax_route(logits.numpy(), k, renorm)
    assert np.array_equal(ids.cpu().numpy(), rid)
    check_route_weights(w.cpu().numpy(), rw, logits.numpy(), rid, k, renorm)
    return ids, w


@pytest.mark.parametrize("t", [1, 4, 8, 16, 32, 1280])
def test_route_top8_of_256(t):
    _check_route(synth.router_logits(4, t, E), K)


def test_route_without_renormalisation_and_wide_shapes():
    _check_route(synth.router_logits(5, 64, 256), 8, renorm=False)
    _check_route(synth.router_logits(5, 40, 512), 32)
    _check_route(synth.router_logits(5, 9, 37), 32)
    _check_route(synth.router_logits(5, 3, 1), 1)
    with pytest.raises(RuntimeError, match="unsupported shape"):
        ops.route(synth.router_logits(5, 2, 40).cuda(), 33)


def test_route_ties_lowest_index_first():
    l = torch.zeros(3, 256, dtype=torch.float32)
    l[0, [200, 5, 77]] = 1.0
    l[1, :] = 0.5
    l[2, 255] = 3.0
    l[2, 0] = 3.0
    ids, _ = _check_route(l, 8)
    assert ids[0, :3].tolist() == [5, 77, 200]
    assert ids[1].tolist() == list(range(8))
    assert ids[2, :2].tolist() == [0, 255]


# ------------------------------------------------------------------ MoE

def _moe_case(layer4, t, shared=True, rms=False, ids=None, w=None, seed=4):
    ex, sh, get = layer4
    x = synth.activations_bf16(seed, 32, H, 1)[:t]
    if ids is None:
        ids, w = ops.route(synth.router_logits(seed, 32, E, 1)[:t].cuda(), K)
    ws = ops.Workspace(ops.moe_workspace_bytes(t, ids.shape[1], ex))
    out = ops.moe(x.cuda(), ids, w, ex, sh if shared else None, rms_input=rms, workspace=ws)
    disp = ops.last_dispatch()
    status = ws.status()
    x64 = f64(x)
    ref64 = O.moe_decode64(O.rms_scale(x64) if rms else x64, ids.cpu().numpy(),
                           w.cpu().double().numpy(), get, E, get(E) if shared else None)
    return out, ref64, disp, status, (x, ids, w, ws)


@pytest.mark.parametrize("t", [1, 4, 8, 16, 32])
def test_moe_layer_35b_shape(layer4, t):
    out, ref, disp, status, _ = _moe_case(layer4, t)
    assert status == 0
    # the CUDA-core kernels at every T up to 32 (in batches of 16 tokens);
    # gate/up by warp MMAs for 4 to 8 tokens (H a multiple of 512)
    gate_up = "moe_mma_gate_up_kernel" if 4 <= t <= 8 else "moe_fma_gate_up_kernel"
    assert "shared=1" in disp and disp.startswith(gate_up)
    assert "moe_fma_down_kernel" in disp
    assert_close(f64(out), O.bf16_round(ref), f"MoE T={t}")


@pytest.mark.parametrize("t", [1, 4, 8, 16, 32])
def test_moe_layer_on_the_tensor_cores_few_tokens(layer4, t):
    """The tensor-core MoE kernels at few tokens (a one-op program, which
    always runs them), against the oracle."""
    ex, sh, get = layer4
    x = synth.activations_bf16(4, 32, H, 1)[:t].cuda()
    ids, w = ops.route(synth.router_logits(4, 32, E, 1)[:t].cuda(), K)
    out = torch.empty(t, H, dtype=torch.bfloat16, device="cuda")
    prog = ops.Program([ops.moe_op(x, ids, w, ex, out, shared=sh)])
    prog.launch()
    torch.cuda.synchronize()
    assert prog.workspace.status() == 0
    ref = O.moe_decode64(f64(x), ids.cpu().numpy(), w.cpu().double().numpy(), get, E, get(E))
    assert_close(f64(out), O.bf16_round(ref), f"tensor-core MoE T={t}")


@pytest.mark.parametrize("e,h,i,k,t,shared", [(64, 1024, 256, 16, 3, True),   # 8 chunks a row, R = 5
                                              (64, 1024, 1024, 8, 2, True),   # 32 chunks, R = 9
                                              (64, 2048, 512, 4, 8, False),   # R = 2
                                              (32, 768, 256, 1, 5, True),     # k = 1
                                              (64, 4096, 512, 16, 8, True)])  # 64 KB of x rows
def test_moe_cuda_core_kernels_other_shapes(e, h, i, k, t, shared):
    ex = device_experts(6, 1, e, h, i)
    sh = device_shared(6, 1, e, h, i) if shared else None
    get = host_expert_fn(6, 1, h, i)
    x = synth.activations_bf16(6, t, h, 2)
    ids, w = ops.route(synth.router_logits(6, t, e, 2).cuda(), k)
    out = ops.moe(x.cuda(), ids, w, ex, sh, rms_input=True)
    gate_up = "moe_mma_gate_up_kernel" if h % 512 == 0 and 4 <= t <= 8 else "moe_fma_gate_up_kernel"
    assert ops.last_dispatch().startswith(gate_up)
    torch.cuda.synchronize()
    ref = O.moe_decode64(O.rms_scale(f64(x)), ids.cpu().numpy(), w.cpu().double().numpy(), get, e,
                         get(e) if shared else None)
    assert_close(f64(out), O.bf16_round(ref), f"CUDA-core MoE E={e} H={h} I={i} k={k} T={t}")


def test_moe_without_shared_expert(layer4):
    out, ref, _, status, _ = _moe_case(layer4, 8, shared=False)
    assert status == 0
    assert_close(f64(out), O.bf16_round(ref), "MoE no shared")


def test_moe_rms_input(layer4):
    out, ref, disp, _, _ = _moe_case(layer4, 4, rms=True)
    assert "rms=1" in disp
    assert_close(f64(out), O.bf16_round(ref), "MoE rms")


def test_moe_ids_ready_flag_same_result(layer4):
    ex, sh, _ = layer4
    out, _, _, _, (x, ids, w, ws) = _moe_case(layer4, 8)
    again = ops.moe(x.cuda(), ids, w, ex, sh, workspace=ws, ids_ready=True)
    assert "ids_ready=1" in ops.last_dispatch()
    torch.cuda.synchronize()
    assert torch.equal(again, out)


def test_moe_shared_expert_is_additive(layer4):
    """The fused layer equals routed-only plus the shared expert on its own
    (the failure mode of fusing the shared expert into the main MoE)."""
    ex, sh, get = layer4
    t = 6
    x = synth.activations_bf16(4, t, H, 7).cuda()
    ids, w = ops.route(synth.router_logits(4, t, E, 7).cuda(), K)
    both = f64(ops.moe(x, ids, w, ex, sh))
    routed = f64(ops.moe(x, ids, w, ex, None))
    ref_sh = O.expert_ffn64(f64(x), get(E))
    ref_both = O.moe_decode64(f64(x), ids.cpu().numpy(), w.cpu().double().numpy(), get, E, get(E))
    assert_close(both, O.bf16_round(ref_both), "both")
    # |both - routed - shared| within the sum of the two outputs' tolerances
    rms = np.sqrt(np.mean(ref_both ** 2))
    assert np.all(np.abs(both - routed - ref_sh) <= 1.6e-2 * np.abs(ref_both) + 6e-3 * rms)


def test_moe_bad_ids_are_skipped_and_flagged(layer4):
    ex, sh, get = layer4
    t = 4
    ids, w = ops.route(synth.router_logits(4, t, E, 9).cuda(), K)
    ids[1, 3] = 300
    ids[2, 0] = -5
    out, ref, _, status, _ = _moe_case(layer4, t, ids=ids, w=w)
    assert status & ops.STATUS_BAD_EXPERT_ID
    assert_close(f64(out), O.bf16_round(ref), "bad ids")


def test_moe_duplicate_ids_are_summed(layer4):
    ids = torch.tensor([[3, 3, 9, 9, 9, 1, 2, 200]], dtype=torch.int32, device="cuda")
    w = torch.full((1, 8), 0.125, dtype=torch.float32, device="cuda")
    out, ref, _, status, _ = _moe_case(layer4, 1, ids=ids, w=w)
    assert status == 0
    assert_close(f64(out), O.bf16_round(ref), "duplicates")


def test_moe_all_tokens_one_expert(layer4):
    t = 32
    ids = torch.arange(K, dtype=torch.int32, device="cuda").repeat(t, 1)
    w = torch.full((t, K), 1.0 / K, dtype=torch.float32, device="cuda")
    out, ref, _, status, _ = _moe_case(layer4, t, ids=ids, w=w)
    assert status == 0
    assert_close(f64(out), O.bf16_round(ref), "all tokens on experts 0..7")


@pytest.mark.parametrize("t", [8, 16])
def test_moe_deterministic(layer4, t):
    out, _, _, _, (x, ids, w, ws) = _moe_case(layer4, t)
    ex, sh, _ = layer4
    again = [ops.moe(x.cuda(), ids, w, ex, sh, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    for a in again:
        assert torch.equal(a, out)


def test_moe_reads_only_routed_experts(layer4):
    """Poison every expert that no token routes to: the output must not change."""
    ex, sh, get = layer4
    t = 2
    x = synth.activations_bf16(4, t, H, 3).cuda()
    ids, w = ops.route(synth.router_logits(4, t, E, 3).cuda(), K)
    ref = ops.moe(x, ids, w, ex, sh)
    used = set(ids.flatten().tolist())
    unused = torch.tensor([e for e in range(E) if e not in used], device="cuda")
    poisoned = ops.ExpertStack(ex.gu_codes.clone(), ex.gu_scales.clone(), ex.dn_codes.clone(),
                               ex.dn_scales.clone(), ex.gu_global, ex.dn_global)
    poisoned.gu_scales[unused] = 0x7F   # E4M3 NaN
    poisoned.dn_scales[unused] = 0x7F
    out = ops.moe(x, ids, w, poisoned, sh)
    assert torch.equal(out, ref)


# ------------------------------------------------------------------ MTP-verify batch

def test_mtp_verify_batch_moe_then_lm_head_argmax():
    """32 rows (8 requests x 4 draft tokens) through a seed-5 MoE layer, then
    the 151,936-row 4-bit head with argmax; the head is checked from the
    GPU's own BF16 MoE output (teacher forcing)."""
    ex = device_experts(5, 0, E, H, I)
    sh = device_shared(5, 0, E, H, I)
    get = host_expert_fn(5, 0, H, I)
    t = 32
    x = synth.activations_bf16(5, t, H, 1)
    logits = synth.router_logits(5, t, E, 1)
    ids, w = _check_route(logits, K)
    y = ops.moe(x.cuda(), ids, w, ex, sh)
    ref = O.moe_decode64(f64(x), ids.cpu().numpy(), w.cpu().double().numpy(), get, E, get(E))
    assert_close(f64(y), O.bf16_round(ref), "MTP MoE")
    del ex, sh
    lm = device_weight(5, 151936, H, 2)
    logits_out, am = ops.gemm(y, lm, argmax=True)
    ref_logits = O.gemm64(f64(y), *host_weight(5, 151936, H, 2))
    assert_close(f64(logits_out), O.bf16_round(ref_logits), "MTP head")
    check_argmax(am.cpu().numpy(), f64(logits_out), ref_logits, what="MTP head")


def test_one_workspace_serves_moe_then_split_k_gemm(layer4):
    """A dense split-K GEMM after an MoE call on the same workspace: the MoE
    scratch must not disturb the GEMM's tile counters (T = 16: the MoE layer
    on the CUDA cores, the GEMM on the tensor cores)."""
    ex, sh, _ = layer4
    t = 16
    W = device_weight(21, 5120, H)
    ws = ops.Workspace(max(ops.gemm_workspace_bytes(t, 5120, H), ops.moe_workspace_bytes(t, K, ex)))
    x = synth.activations_bf16(21, t, H).cuda()
    ids, w = ops.route(synth.router_logits(21, t, E).cuda(), K)
    for _ in range(2):
        ops.moe(x, ids, w, ex, sh, workspace=ws)
        c = ops.gemm(x, W, workspace=ws)
        assert "units_per_cta" in ops.last_dispatch()
    torch.cuda.synchronize()
    assert ws.status() == 0
    ref = O.gemm_bf16(f64(x), *host_weight(21, 5120, H))
    assert_close(f64(c), ref, "gemm after moe")
