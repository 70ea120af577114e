"""GPU parity of the full stacked decode step (40 layers of QKV 2048->5120,
O 4096->2048 and the 256+1-expert MoE layer, then the 151,936-row head with
argmax): routing of every layer bit-exact, sampled layers checked op by op
from the GPU's own BF16 inputs (teacher forcing), the head's argmax, and the
CUDA-graph replay equal to the eager run."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, f64, host_expert_fn
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


@pytest.mark.parametrize("tokens", [1, 8, 32])
def test_decode_step(model, tokens):
    m, s = model, model.s
    b = m.buffers(tokens, keep=True)
    x, lg = m.inputs(tokens)
    b["x"].copy_(x)
    b["logits"].copy_(lg)
    m.run(b)
    torch.cuda.synchronize()
    assert b["ws"].status() == 0

    # routing, every layer
    rid, rw = O.topk_softmax_route(lg.numpy(), s.top_k)
    assert np.array_equal(b["ids"].cpu().numpy(), rid)
    np.testing.assert_allclose(b["w"].cpu().double().numpy(), rw, rtol=2e-6, atol=1e-12)

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
    am = b["argmax"].cpu().numpy()
    assert np.array_equal(am, O.argmax_first(f64(b["head"]), axis=1))
    ref_ids = O.argmax_first(O.bf16_round(head64), axis=1)
    for r in np.nonzero(am != ref_ids)[0]:
        a, c = head64[r, am[r]], head64[r, ref_ids[r]]
        assert abs(a - c) <= 2.0 ** (np.floor(np.log2(abs(c))) - 7), r

    # the captured graph reproduces the eager step bit for bit
    keep_head = b["head"].clone()
    keep_am = b["argmax"].clone()
    keep_y = [y.clone() for y in b["y"]]
    g = m.capture(b)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(b["head"], keep_head) and torch.equal(b["argmax"], keep_am)
    assert all(torch.equal(a, c) for a, c in zip(b["y"], keep_y))
    assert b["ws"].status() == 0
