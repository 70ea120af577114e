"""GPU checks of programs (a chain of GEMM / MoE calls in one persistent
launch).  With every op spread over every SM (NVFP4_FLAG_ALL_SMS; MoE ops
always are) a program splits the work exactly like the single calls, and its
results are bit-identical to the same calls issued one by one (which the
other files check against the float64 oracle).  With the default placement (small dense
ops on a rotating subset of SMs, fewer split-K partial sums) results are
checked against the oracle, teacher-forced op by op.  The workspace counters
are back at zero after every launch."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import (assert_close, device_experts, device_shared, device_weight, f64,
                     host_weight)
from moe_expert_nvfp4_gb300 import ops, synth
from moe_expert_nvfp4_gb300.decode_step import DecodeStep, StepShape

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_nvfp4_gb300 import build
    build.build()
    ops.load()
    assert ops.device_check(torch.cuda.current_device()) == 0, ops.last_error()


def _counters_zero(ws):
    torch.cuda.synchronize()
    hdr = ws.buf[:256 + 4 * 16384].view(torch.int32)
    return int(hdr[1:].abs().sum().item()) == 0 and int(hdr[0].item()) == 0


def test_single_gemm_program_equals_call():
    """An ALL_SMS program op against the same call on the tensor cores (8192
    x 2048 at M = 8 is past the CUDA-core dispatch bound)."""
    W = device_weight(11, 8192, 2048)
    a = synth.activations_bf16(11, 8, 2048).cuda()
    ref = ops.gemm(a, W)
    assert ops.last_dispatch().startswith("stream_tc_kernel<dense>")
    out = torch.empty_like(ref)
    prog = ops.Program([ops.gemm_op(a, W, out, all_sms=True)])
    prog.launch()
    torch.cuda.synchronize()
    assert ops.last_dispatch().startswith("stream_tc_kernel program ops=1")
    assert torch.equal(out, ref)
    assert _counters_zero(prog.workspace)


@pytest.mark.parametrize("m", [8, 16, 32])
def test_gemm_chain_equals_calls_and_oracle(m):
    """x -> (rms) W1 [4096 x 2048] -> (rms) W2 [2560 x 4096] -> W3 [8192 x 2560]
    + argmax; every call on the tensor cores (M = 1, and weights up to 5 MiB
    at M <= 16 that fit one wave of four-row CTAs, go to the CUDA-core
    kernel: the chain at M = 1 is checked against the oracle below)."""
    W1 = device_weight(12, 4096, 2048)
    W2 = device_weight(13, 2560, 4096)
    W3 = device_weight(14, 8192, 2560)
    x = synth.activations_bf16(12, m, 2048).cuda()
    h1 = ops.gemm(x, W1, rms_input=True)
    assert ops.last_dispatch().startswith("stream_tc_kernel<dense>")
    h2 = ops.gemm(h1, W2, rms_input=True)
    h3, am = ops.gemm(h2, W3, argmax=True)
    assert ops.last_dispatch().startswith("stream_tc_kernel<dense>")
    torch.cuda.synchronize()
    p1, p2, p3 = torch.empty_like(h1), torch.empty_like(h2), torch.empty_like(h3)
    pam = torch.empty_like(am)
    prog = ops.Program([ops.gemm_op(x, W1, p1, rms_input=True, all_sms=True),
                        ops.gemm_op(p1, W2, p2, rms_input=True, all_sms=True),
                        ops.gemm_op(p2, W3, p3, argmax_out=pam, all_sms=True)])
    for _ in range(3):   # repeated launches reuse the zeroed counters
        prog.launch()
    torch.cuda.synchronize()
    assert torch.equal(p1, h1) and torch.equal(p2, h2) and torch.equal(p3, h3)
    assert torch.equal(pam, am)
    assert prog.workspace.status() == 0
    assert _counters_zero(prog.workspace)
    # teacher-forced oracle check of the chain's middle link
    ref2 = O.gemm_bf16(O.rms_scale(f64(p1)), *host_weight(13, 2560, 4096))
    assert_close(f64(p2), ref2, f"chain M={m}")


@pytest.fixture(scope="module")
def layer():
    """Intermediate size 768: outside the CUDA-core MoE kernels' shapes, so
    the single MoE calls run on the tensor cores like the program ops."""
    E, H, I = 64, 2048, 768
    return device_experts(21, 0, E, H, I), device_shared(21, 0, E, H, I)


@pytest.mark.parametrize("t", [12, 32])
def test_moe_in_program_equals_call(layer, t):
    """(12 and 32 rows: the 2048 x 2048 calls run on the tensor cores too; at
    M = 5..8 that weight goes to the CUDA-core kernel.)"""
    ex, sh = layer
    x = synth.activations_bf16(21, t, 2048).cuda()
    ids, w = ops.route(synth.router_logits(21, t, 64).cuda(), 8)
    W = device_weight(22, 2048, 2048)
    # GEMM -> MoE -> GEMM, so the MoE reads a program-written input and its
    # output feeds a later op
    g1 = ops.gemm(x, W, rms_input=True)
    y = ops.moe(g1, ids, w, ex, sh, rms_input=True, ids_ready=True)
    g2 = ops.gemm(y, W, rms_input=True)
    torch.cuda.synchronize()
    pg1, py, pg2 = torch.empty_like(g1), torch.empty_like(y), torch.empty_like(g2)
    prog = ops.Program([ops.gemm_op(x, W, pg1, rms_input=True, all_sms=True),
                        ops.moe_op(pg1, ids, w, ex, py, shared=sh, rms_input=True),
                        ops.gemm_op(py, W, pg2, rms_input=True, all_sms=True)])
    prog.launch()
    prog.launch()
    torch.cuda.synchronize()
    assert torch.equal(pg1, g1) and torch.equal(py, y) and torch.equal(pg2, g2)
    assert prog.workspace.status() == 0
    assert _counters_zero(prog.workspace)


def test_two_moe_layers_share_schedule_slots(layer):
    """Four MoE layers in a row cycle both schedule slots twice."""
    ex, sh = layer
    t = 32
    x = synth.activations_bf16(23, t, 2048).cuda()
    lg = synth.router_logits(23, 4 * t, 64).cuda()
    ids, w = ops.route(lg, 8)
    outs, cur = [], x
    for l in range(4):
        cur = ops.moe(cur, ids[l * t:(l + 1) * t], w[l * t:(l + 1) * t], ex,
                      sh if l % 2 == 0 else None, rms_input=True, ids_ready=True)
        outs.append(cur)
    torch.cuda.synchronize()
    pouts = [torch.empty_like(o) for o in outs]
    chain, src = [], x
    for l in range(4):
        chain.append(ops.moe_op(src, ids[l * t:(l + 1) * t], w[l * t:(l + 1) * t], ex, pouts[l],
                                shared=sh if l % 2 == 0 else None, rms_input=True))
        src = pouts[l]
    prog = ops.Program(chain)
    prog.launch()
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(pouts, outs))
    assert _counters_zero(prog.workspace)


@pytest.mark.parametrize("tokens", [32])
def test_decode_step_program_equals_calls(tokens):
    """(32 tokens and intermediate size 768: every call of the step runs on
    the tensor cores, as the program's ops do.)"""
    m = DecodeStep(seed=6, shape=StepShape(layers=3, inter=768))
    b = m.buffers(tokens, keep=True)
    x, lg = m.inputs(tokens)
    b["x"].copy_(x)
    b["logits"].copy_(lg)
    m.run(b)
    torch.cuda.synchronize()
    ref = {k: [t.clone() for t in b[k]] for k in ("q", "o", "y")}
    ref_head, ref_am = b["head"].clone(), b["argmax"].clone()
    for k in ("q", "o", "y"):
        for t in b[k]:
            t.zero_()
    b["head"].zero_()
    b["argmax"].zero_()
    prog = m.program(b, all_sms=True)
    g = m.capture(b, prog=prog)
    g.replay()
    torch.cuda.synchronize()
    for k in ("q", "o", "y"):
        assert all(torch.equal(a, c) for a, c in zip(b[k], ref[k])), k
    assert torch.equal(b["head"], ref_head) and torch.equal(b["argmax"], ref_am)
    assert b["ws"].status() == 0
    assert _counters_zero(b["ws"])


@pytest.mark.parametrize("m", [1, 8, 17, 32])
def test_default_placement_chain_against_oracle(m):
    """Default placement: QKV-, O- and head-shaped GEMMs chained, each checked
    against the oracle from its own (program-written) input."""
    W1 = device_weight(31, 5120, 2048)
    W2 = device_weight(32, 2048, 4096)
    W3 = device_weight(33, 3000, 2048)
    x = synth.activations_bf16(31, m, 2048).cuda()
    p1 = torch.empty(m, 5120, dtype=torch.bfloat16, device="cuda")
    p2 = torch.empty(m, 2048, dtype=torch.bfloat16, device="cuda")
    p3 = torch.empty(m, 3000, dtype=torch.bfloat16, device="cuda")
    am = torch.empty(m, dtype=torch.int32, device="cuda")
    prog = ops.Program([ops.gemm_op(x, W1, p1, rms_input=True),
                        ops.gemm_op(p1[:, :4096], W2, p2, rms_input=True),
                        ops.gemm_op(p2, W3, p3, argmax_out=am, rms_input=True)])
    prog.launch()
    prog.launch()
    torch.cuda.synchronize()
    assert prog.workspace.status() == 0
    assert _counters_zero(prog.workspace)
    assert_close(f64(p1), O.gemm_bf16(O.rms_scale(f64(x)), *host_weight(31, 5120, 2048)), "QKV")
    assert_close(f64(p2), O.gemm_bf16(O.rms_scale(f64(p1)[:, :4096]), *host_weight(32, 2048, 4096)),
                 "O")
    assert_close(f64(p3), O.gemm_bf16(O.rms_scale(f64(p2)), *host_weight(33, 3000, 2048)), "head")
    assert np.array_equal(am.cpu().numpy(), O.argmax_first(f64(p3), axis=1))


def test_default_placement_decode_step_against_oracle():
    """Default placement, 3-layer step at T=8: every layer's QKV, O and MoE
    from its own inputs, and the head, against the oracle."""
    from helpers import host_expert_fn
    from moe_expert_nvfp4_gb300.decode_step import ROLE_HEAD, ROLE_O, ROLE_QKV
    t = 8
    m = DecodeStep(seed=6, shape=StepShape(layers=3))
    s = m.s
    b = m.buffers(t, keep=True)
    x, lg = m.inputs(t)
    b["x"].copy_(x)
    b["logits"].copy_(lg)
    prog = m.program(b)
    m.run_program(b, prog)
    torch.cuda.synchronize()
    assert b["ws"].status() == 0
    for l in range(s.layers):
        xin = f64(b["x"] if l == 0 else b["y"][l - 1])
        q = f64(b["q"][l])
        assert_close(q, O.gemm_bf16(O.rms_scale(xin), *host_weight(6, s.qkv_out, s.hidden, ROLE_QKV, l)),
                     f"layer {l} QKV")
        o = f64(b["o"][l])
        assert_close(o, O.gemm_bf16(O.rms_scale(q[:, :s.o_in]),
                                    *host_weight(6, s.hidden, s.o_in, ROLE_O, l)), f"layer {l} O")
        get = host_expert_fn(6, l, s.hidden, s.inter)
        ids = b["ids"][l * t:(l + 1) * t].cpu().numpy()
        w = b["w"][l * t:(l + 1) * t].cpu().double().numpy()
        y_ref = O.moe_decode_bf16(O.rms_scale(o), ids, w, get, s.num_experts, get(s.num_experts))
        assert_close(f64(b["y"][l]), y_ref, f"layer {l} MoE")
    head = f64(b["head"])
    assert np.array_equal(b["argmax"].cpu().numpy(), O.argmax_first(head, axis=1))
