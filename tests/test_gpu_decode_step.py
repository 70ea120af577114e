"""GPU parity of the full stacked decode step (40 layers of QKV 2048->5120,
O 4096->2048 and the 256+1-expert MoE layer, then the 151,936-row head with
argmax), both ways the library runs it: routing of every layer, then the
whole chain as one program launch replayed from a CUDA graph; and call by
call (the benchmark's path at every token count: the MoE layers and the
small dense calls on the CUDA cores, the rest on the tensor cores).

Checked: routing of every layer (ids bit-exact, weights within the FP32
bound), sampled layers op by op from the GPU's own BF16 inputs (teacher
forcing), the head's logits and argmax; then the same step issued call by
call, checked the same way on a sampled layer and the head."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, check_argmax, check_route_weights, f64, host_expert_fn
from moe_expert_nvfp4_gb300 import ops, synth
from moe_expert_nvfp4_gb300.decode_step import ROLE_HEAD, ROLE_O, ROLE_QKV, DecodeStep

pytestmark = pytest.mark.gpu
SAMPLED_LAYERS = (0, 17, 39)


@pytest.fixture(scope="module")
def model():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_nvfp4_gb300 import build
    build.build()
    ops.load()
    assert ops.device_check(torch.cuda.current_device()) == 0, ops.last_error()
    return DecodeStep(seed=6)


def _host_w(seed, n, k, *ids):
    c, s = synth.nvfp4_weight(seed, n, k, *ids)
    return c.numpy(), s.numpy(), synth.GLOBAL_SCALE


@pytest.mark.parametrize("tokens", [1, 2, 8, 16, 32])
def test_decode_step_program(model, tokens):
    m, s = model, model.s
    b = m.buffers(tokens, keep=True)
    x, lg = m.inputs(tokens)
    b["x"].copy_(x)
    b["logits"].copy_(lg)
    prog = m.program(b)
    g = m.capture(b, prog=prog)          # warm-up step, then the graph
    for t in b["q"] + b["o"] + b["y"] + [b["head"]]:
        t.zero_()
    b["argmax"].zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert b["ws"].status() == 0

    # routing, every layer
    rid, rw = O.topk_softmax_route(lg.numpy(), s.top_k)
    assert np.array_equal(b["ids"].cpu().numpy(), rid)
    check_route_weights(b["w"].cpu().numpy(), rw, lg.numpy(), rid, s.top_k)

    for l in SAMPLED_LAYERS:
        xin = f64(b["x"] if l == 0 else b["y"][l - 1])
        q = f64(b["q"][l])
        assert_close(q, O.gemm_bf16(O.rms_scale(xin), *_host_w(6, s.qkv_out, s.hidden, ROLE_QKV, l)),
                     f"layer {l} QKV")
        o = f64(b["o"][l])
        assert_close(o, O.gemm_bf16(O.rms_scale(q[:, :s.o_in]),
                                    *_host_w(6, s.hidden, s.o_in, ROLE_O, l)), f"layer {l} O")
        get = host_expert_fn(6, l, s.hidden, s.inter)
        ids = b["ids"][l * tokens:(l + 1) * tokens].cpu().numpy()
        w = b["w"][l * tokens:(l + 1) * tokens].cpu().double().numpy()
        y_ref = O.moe_decode_bf16(O.rms_scale(o), ids, w, get, s.num_experts, get(s.num_experts))
        assert_close(f64(b["y"][l]), y_ref, f"layer {l} MoE")

    # the head, from the last layer's output
    head64 = O.gemm64(O.rms_scale(f64(b["y"][s.layers - 1])),
                      *_host_w(6, s.vocab, s.hidden, ROLE_HEAD))
    assert_close(f64(b["head"]), O.bf16_round(head64), "head")
    check_argmax(b["argmax"].cpu().numpy(), f64(b["head"]), head64, what="step head")

    # the same step call by call, the way DecodeStep.path_for runs it (the
    # CUDA-core kernels by shape, the small tensor-core calls on fewer CTAs:
    # the two paths agree to the tolerance, not bit for bit): a sampled
    # layer and the head
    m.run(b)
    torch.cuda.synchronize()
    assert b["ws"].status() == 0
    l = 17
    o = f64(b["o"][l])
    assert_close(o, O.gemm_bf16(O.rms_scale(f64(b["q"][l])[:, :s.o_in]),
                                *_host_w(6, s.hidden, s.o_in, ROLE_O, l)), f"calls: layer {l} O")
    get = host_expert_fn(6, l, s.hidden, s.inter)
    ids = b["ids"][l * tokens:(l + 1) * tokens].cpu().numpy()
    w = b["w"][l * tokens:(l + 1) * tokens].cpu().double().numpy()
    y_ref = O.moe_decode_bf16(O.rms_scale(o), ids, w, get, s.num_experts, get(s.num_experts))
    assert_close(f64(b["y"][l]), y_ref, f"calls: layer {l} MoE")
    head64 = O.gemm64(O.rms_scale(f64(b["y"][s.layers - 1])),
                      *_host_w(6, s.vocab, s.hidden, ROLE_HEAD))
    assert_close(f64(b["head"]), O.bf16_round(head64), "calls: head")
    check_argmax(b["argmax"].cpu().numpy(), f64(b["head"]), head64, what="calls: step head")
