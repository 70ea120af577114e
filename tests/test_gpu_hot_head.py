"""GPU parity of the hot-vocabulary head ("Qwen3.6-35B-A3B NVFP4 on an RTX
5090 (Elsa)", section "Making decode faster", paragraph "FR-Spec, and a silent
bug"): a draft head restricted to a list of likely tokens, built from the
rows of the full 4-bit head.

* nvfp4_gather_rows: the gathered codes and scales equal the listed rows of
  the head byte for byte (all-zero rows for ids outside [0, N)).
* nvfp4_hot_vocab_head: the hot rows' BF16 logits against the oracle within
  the tolerance; the reported ids bit-exact against the vocabulary ids of
  the first maxima of the GPU's own logits, and against the oracle up to a
  top-1 pair whose float64 logits straddle a BF16 rounding boundary within
  the FP32 accumulation error.
* the same head as an op of a program.

Inputs: seeded synthetic heads and token lists (a sorted random subset of
distinct ids stands for the frequency-ranked list the pages build from the
model's own output), sized from a ragged 1,000-row list up to the
32,768-row list of the 151,936-row head."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, check_argmax, device_weight, f64, host_weight
from moe_expert_nvfp4_gb300 import ops, synth

pytestmark = pytest.mark.gpu

HEAD_ROLE = 31  # stream id of the synthetic heads of this file


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_nvfp4_gb300 import build
    build.build()
    ops.load()
    assert ops.device_check(torch.cuda.current_device()) == 0, ops.last_error()


def _hot_list(seed, n_full, n_hot):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(n_full, n_hot, replace=False)).astype(np.int32)


def _check_ids(am, logits_gpu, ref_logits64, vocab_ids):
    """ids bit-exact against the GPU's own logits; against the oracle up to
    a top-1 pair straddling a BF16 rounding boundary within FP32
    accumulation error."""
    check_argmax(am.cpu().numpy(), f64(logits_gpu), ref_logits64, id_map=vocab_ids,
                 what="hot head")


@pytest.mark.parametrize("n_full,n_hot,k", [(3000, 1000, 1024), (151936, 32768, 2048)])
def test_gather_rows_is_the_listed_rows(n_full, n_hot, k):
    W = device_weight(7, n_full, k, HEAD_ROLE)
    lst = _hot_list(7, n_full, n_hot)
    lst[[1, n_hot // 2, n_hot - 1]] = [-1, n_full, 2**31 - 1]  # outside [0, N): zero rows
    hot = ops.gather_rows(W, torch.from_numpy(lst).cuda())
    torch.cuda.synchronize()
    assert ops.last_dispatch().startswith("gather_rows_kernel")
    codes, scales, _ = host_weight(7, n_full, k, HEAD_ROLE)
    ok = (lst >= 0) & (lst < n_full)
    want_c = np.zeros((n_hot, k // 2), np.uint8)
    want_s = np.zeros((n_hot, k // 16), np.uint8)
    want_c[ok], want_s[ok] = codes[lst[ok]], scales[lst[ok]]
    assert np.array_equal(hot.codes.cpu().numpy(), want_c)
    assert np.array_equal(hot.scales.cpu().numpy(), want_s)
    assert hot.global_scale.data_ptr() == W.global_scale.data_ptr()


@pytest.mark.parametrize("m", [1, 8, 32])
def test_hot_head_matches_oracle(m):
    """A ragged 1,000-row list (7 full 128-row tiles + 104) of a 3,000-row head."""
    n_full, n_hot, k = 3000, 1000, 1024
    W = device_weight(8, n_full, k, HEAD_ROLE)
    lst = _hot_list(8, n_full, n_hot)
    vid = torch.from_numpy(lst).cuda()
    hot = ops.gather_rows(W, vid)
    a = synth.activations_bf16(8, m, k).cuda()
    logits, am = ops.hot_vocab_head(a, hot, vid)
    torch.cuda.synchronize()
    # 0.6 MB of weights: the CUDA-core kernel up to M = 8
    assert ops.last_dispatch().startswith("fma_kernel" if m <= 8 else "stream_tc_kernel")
    codes, scales, g = host_weight(8, n_full, k, HEAD_ROLE)
    ref64 = O.gemm64(f64(a), codes[lst], scales[lst], g)
    assert_close(f64(logits), O.bf16_round(ref64), "hot logits")
    _, ref_logits = O.hot_vocab_head_argmax(f64(a), codes, scales, g, lst)
    assert np.array_equal(ref_logits, O.bf16_round(ref64))
    _check_ids(am, logits, ref64, lst)


def test_hot_head_full_size_draft_batch():
    """The 32,768-row list of the 151,936 x 2048 head at M = 8 (the bench's
    hot-vocabulary workload), logits and ids checked whole."""
    n_full, n_hot, k, m = 151936, 32768, 2048, 8
    W = device_weight(9, n_full, k, HEAD_ROLE)
    lst = _hot_list(9, n_full, n_hot)
    vid = torch.from_numpy(lst).cuda()
    hot = ops.gather_rows(W, vid)
    del W
    a = synth.activations_bf16(9, m, k).cuda()
    logits, am = ops.hot_vocab_head(a, hot, vid, rms_input=True)
    torch.cuda.synchronize()
    codes, scales, g = host_weight(9, n_full, k, HEAD_ROLE)
    ref64 = O.gemm64(O.rms_scale(f64(a)), codes[lst], scales[lst], g)
    assert_close(f64(logits), O.bf16_round(ref64), "hot logits, full size")
    _check_ids(am, logits, ref64, lst)


def test_hot_head_program_op_equals_call():
    """x -> (rms) W [4096 x 2048] -> hot head of a 20,000-row head; every op
    flagged to split over every SM like the calls: bit-identical (M = 16:
    both calls run on the tensor cores)."""
    W1 = device_weight(10, 4096, 2048)
    H = device_weight(10, 20000, 4096, HEAD_ROLE)
    lst = _hot_list(10, 20000, 5000)
    vid = torch.from_numpy(lst).cuda()
    hot = ops.gather_rows(H, vid)
    x = synth.activations_bf16(10, 16, 2048).cuda()
    h1 = ops.gemm(x, W1, rms_input=True)
    lg, am = ops.hot_vocab_head(h1, hot, vid, rms_input=True)
    p1, plg = torch.empty_like(h1), torch.empty_like(lg)
    pam = torch.full_like(am, -7)
    prog = ops.Program([ops.gemm_op(x, W1, p1, rms_input=True, all_sms=True),
                        ops.gemm_op(p1, hot, plg, argmax_out=pam, rms_input=True,
                                    argmax_map=vid, all_sms=True)])
    prog.launch()
    torch.cuda.synchronize()
    assert torch.equal(p1, h1) and torch.equal(plg, lg) and torch.equal(pam, am)
    assert np.all(np.isin(pam.cpu().numpy(), lst))
    assert prog.workspace.status() == 0
