"""The C-ABI library without a GPU: it loads, exports every function the
public header declares, and its host-side validation returns the documented
status codes before touching a device."""
import ctypes
import os
import subprocess

import pytest

from moe_expert_nvfp4_gb300 import build as B
from moe_expert_nvfp4_gb300 import ops


@pytest.fixture(scope="module")
def lib():
    B.build()
    return ops.load()


def test_header_declares_the_boundary():
    names = ops.declared_functions()
    for n in ["nvfp4_gemm_skinny", "moe_nvfp4_decode", "topk_softmax_route",
              "nvfp4_gemm_skinny_workspace", "moe_nvfp4_decode_workspace", "nvfp4_device_check",
              "nvfp4_workspace_init", "nvfp4_read_device_status", "nvfp4_last_dispatch",
              "nvfp4_last_error", "nvfp4_gather_rows", "nvfp4_hot_vocab_head", "nvfp4_quantize",
              "nvfp4_program_create", "nvfp4_program_launch", "nvfp4_gemm_skinny_noalloc",
              "fp8_gemm_skinny", "fp8_gemm_skinny_workspace", "bf16w_gemm_skinny",
              "bf16w_gemm_skinny_workspace"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", ops.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in ops.declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def _w(codes=1 << 20, scales=1 << 20, g=1 << 20, n=64, k=2048):
    return ops._Weight(codes, scales, g, n, k)


def _gemm(lib, a=1 << 20, lda=2048, m=4, w=None, c=1 << 20, ldc=64, ws=1 << 20, wsb=1 << 30):
    w = w or _w()
    return lib.nvfp4_gemm_skinny(a, lda, m, ctypes.byref(w), c, ldc, None, 0, ws, wsb, None)


def test_gemm_validation_codes(lib):
    assert _gemm(lib, a=0) == -1
    assert _gemm(lib, m=0) == -3
    assert _gemm(lib, m=33) == -3
    assert _gemm(lib, w=_w(k=2000)) == -3           # K not a multiple of 32
    assert _gemm(lib, w=_w(codes=(1 << 20) + 8)) == -2  # misaligned weight
    assert _gemm(lib, a=(1 << 20) + 2) == -2           # misaligned A
    assert _gemm(lib, lda=2052) == -2                  # row stride not 16-byte multiple
    assert _gemm(lib, lda=1024) == -1                  # lda < K
    assert _gemm(lib, w=_w(g=0)) == -1
    assert "16-byte" in ops.last_error() or "NULL" in ops.last_error()


def test_route_validation_codes(lib):
    p = 1 << 20
    assert lib.topk_softmax_route(0, 4, 256, 8, 1, p, p, None) == -1
    assert lib.topk_softmax_route(p, 4, 8, 9, 1, p, p, None) == -1   # k > E
    assert lib.topk_softmax_route(p, 4, 1024, 8, 1, p, p, None) == -3
    assert lib.topk_softmax_route(p, 0, 256, 8, 1, p, p, None) == -1


def _stack(e=256, h=2048, i=512, base=1 << 20):
    return ops._Stack(base, base, base, base, base, base, e, h, i)


def test_moe_validation_codes(lib):
    p = 1 << 20
    st = _stack()

    def call(x=p, ldx=2048, t=4, k=8, ex=st, sh=None, out=p):
        return lib.moe_nvfp4_decode(x, ldx, t, p, p, k, ctypes.byref(ex),
                                    ctypes.byref(sh) if sh is not None else None, out, 2048, 0,
                                    p, 1 << 30, None)

    assert call(x=0) == -1
    assert call(t=33) == -3
    assert call(k=17) == -3
    assert call(ex=_stack(h=2000)) == -3
    assert call(ex=_stack(base=p + 4)) == -2
    assert call(sh=_stack(e=2)) == -1
    assert call(x=p + 2) == -2


def test_program_validation_codes(lib):
    p = 1 << 20
    h = ctypes.c_void_p()
    op = ops._Op()
    op.kind = ops.OP_GEMM
    op.A, op.lda, op.M, op.W, op.C, op.ldc = p, 2048, 4, _w(), p, 64
    assert lib.nvfp4_program_create(None, 1, p, 1 << 30, ctypes.byref(h)) == -1
    assert lib.nvfp4_program_create(ctypes.byref(op), 0, p, 1 << 30, ctypes.byref(h)) == -1
    assert lib.nvfp4_program_create(ctypes.byref(op), 1, p, 1 << 30, None) == -1
    op.M = 33
    assert lib.nvfp4_program_create(ctypes.byref(op), 1, p, 1 << 30, ctypes.byref(h)) == -3
    op.M, op.kind = 4, 7
    assert lib.nvfp4_program_create(ctypes.byref(op), 1, p, 1 << 30, ctypes.byref(h)) == -1
    moe = ops._Op()
    moe.kind = ops.OP_MOE
    moe.x, moe.ldx, moe.T, moe.topk_ids, moe.topk_w, moe.k = p, 2048, 4, p, p, 17
    moe.experts, moe.out, moe.ldo = _stack(), p, 2048
    assert lib.nvfp4_program_create(ctypes.byref(moe), 1, p, 1 << 30, ctypes.byref(h)) == -3
    assert not h.value
    assert lib.nvfp4_program_destroy(None) == 0


def test_hot_vocab_head_validation_codes(lib):
    p = 1 << 20
    w = _w()

    def call(a=p, m=4, ids=p, c=p, am=p):
        return lib.nvfp4_hot_vocab_head(a, 2048, m, ctypes.byref(w), ids, c, 64, am, 0, p, 1 << 30,
                                        None)

    assert call(ids=0) == -1        # the vocabulary ids are required
    assert call(am=0) == -1         # so is the argmax output
    assert call(a=0) == -1
    assert call(m=33) == -3
    assert call(a=p + 2) == -2


def test_gather_rows_validation_codes(lib):
    p = 1 << 20

    def call(w=None, rows=p, n=16, codes=p, scales=p):
        w = w or _w()
        return lib.nvfp4_gather_rows(ctypes.byref(w), rows, n, codes, scales, None)

    assert call(rows=0) == -1
    assert call(codes=0) == -1
    assert call(n=0) == -1
    assert call(w=_w(codes=0)) == -1
    assert call(w=_w(k=2000)) == -3
    assert call(codes=p + 8) == -2
    assert call(w=_w(scales=p + 4)) == -2


def test_quantize_validation_codes(lib):
    p = 1 << 20

    def call(w=p, ldw=2048, n=64, k=2048, codes=p, scales=p, g=p):
        return lib.nvfp4_quantize(w, ldw, n, k, codes, scales, g, None)

    assert call(w=0) == -1
    assert call(g=0) == -1
    assert call(n=0) == -1
    assert call(ldw=1024) == -1     # ldw < K
    assert call(k=48, ldw=48) == -3  # K not a multiple of 32
    assert call(w=p + 2) == -2
    assert call(ldw=2052) == -2     # row stride not a 16-byte multiple
    assert call(codes=p + 8) == -2
    assert call(g=p + 2) == -2      # the float output misaligned


def test_fp8_and_bf16_weight_validation_codes(lib):
    p = 1 << 20

    def fp8(a=p, lda=2048, m=4, codes=p, scale=p, n=64, k=2048, c=p):
        w = ops._Fp8Weight(codes, scale, n, k)
        return lib.fp8_gemm_skinny(a, lda, m, ctypes.byref(w), c, 64, None, 0, p, 1 << 30, None)

    assert fp8(codes=0) == -1
    assert fp8(scale=0) == -1
    assert fp8(a=0) == -1
    assert fp8(m=33) == -3
    assert fp8(k=2000, lda=2000) == -3       # K not a multiple of 256
    assert fp8(codes=p + 8) == -2
    assert fp8(a=p + 2) == -2
    assert lib.fp8_gemm_skinny(p, 2048, 4, None, p, 64, None, 0, p, 1 << 30, None) == -1

    def bf16(a=p, m=4, w=p, ldw=2048, n=64, k=2048):
        wt = ops._Bf16Weight(w, ldw, n, k)
        return lib.bf16w_gemm_skinny(a, 2048, m, ctypes.byref(wt), p, 64, None, 0, p, 1 << 30,
                                     None)

    assert bf16(w=0) == -1
    assert bf16(m=0) == -3
    assert bf16(ldw=1024) == -1              # ldw < K
    assert bf16(ldw=2052) == -2              # row stride not a 16-byte multiple
    assert bf16(w=p + 2) == -2
    assert bf16(k=300) == -3


def test_noalloc_refuses_before_touching_its_scratch(lib):
    """A refused call returns the same status as the workspace entry point
    and issues nothing (no device is needed to see the refusal)."""
    p = 1 << 20
    fn = lib.nvfp4_gemm_skinny_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.POINTER(ops._Weight),
                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint32,
                   ctypes.c_void_p]
    w = _w()
    assert fn(0, 2048, 4, ctypes.byref(w), p, 64, None, 0, None) == -1
    assert fn(p, 2048, 33, ctypes.byref(w), p, 64, None, 0, None) == -3
    assert fn(p + 2, 2048, 4, ctypes.byref(w), p, 64, None, 0, None) == -2
    assert fn(p, 2048, 4, None, p, 64, None, 0, None) == -1


def test_gemm_accepts_k_multiple_of_32(lib):
    """K % 32 == 0 passes the host checks (without a GPU the call then stops
    at the device query, never at the shape check)."""
    for k in (32, 96, 2080):
        rc = _gemm(lib, lda=k, w=_w(k=k))
        assert rc not in (-1, -2, -3), (k, rc, ops.last_error())
    assert lib.nvfp4_gemm_skinny_workspace(4, 64, 48) == 0   # K % 32 != 0
