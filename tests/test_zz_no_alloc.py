"""nvfp4_gemm_skinny_noalloc: the dense skinny GEMM for callers that cannot
allocate device memory (its scratch is an array built into the library).

Called through the C ABI and checked against nvfp4_gemm_skinny, the entry
point that takes a caller workspace, on two calls in a row (the built-in
scratch keeps the previous call's contents, so the second call checks that
it starts clean).  This file is collected last on purpose."""
import ctypes

import pytest
import torch

from helpers import assert_close, device_weight, f64
from moe_expert_nvfp4_gb300 import ops, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_nvfp4_gb300 import build
    build.build()
    L = ops.load()
    assert ops.device_check(torch.cuda.current_device()) == 0, ops.last_error()
    fn = L.nvfp4_gemm_skinny_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.POINTER(ops._Weight),
                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint32,
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


@pytest.mark.parametrize("m,n,k,argmax", [(4, 1000, 1024, True), (16, 4096, 2048, False),
                                          (32, 2048, 4096, True)])
def test_noalloc_matches_workspace_entry_point(lib, m, n, k, argmax):
    W = device_weight(31, n, k)
    a = synth.activations_bf16(31, m, k).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    ref = ops.gemm(a, W, argmax=argmax)
    ref_c, ref_ids = ref if argmax else (ref, None)
    wc = W.c()
    for call in range(2):
        c = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        ids = torch.full((m,), -1, dtype=torch.int32, device="cuda") if argmax else None
        rc = lib(a.data_ptr(), a.stride(0), m, ctypes.byref(wc), c.data_ptr(), c.stride(0),
                 ids.data_ptr() if argmax else None, 0, stream)
        assert rc == 0, ops.last_error()
        torch.cuda.synchronize()
        assert_close(f64(c), f64(ref_c), f"no-alloc call {call}")
        if argmax:
            assert torch.equal(ids, ref_ids)
