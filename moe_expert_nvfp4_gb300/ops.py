"""Python binding of libnvfp4moe.so: torch tensors in, pointers and sizes out.

Argument marshalling only -- every step of the computation runs in the
library's CUDA kernels.  There is no CPU fallback: if the library is missing
or the device is not a GB300 (compute capability 10.3) the calls raise.
Names follow the C ABI in include/nvfp4moe.h.
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnvfp4moe.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "nvfp4moe.h")

NVFP4_OK = 0
ERRORS = {-1: "invalid argument", -2: "misaligned", -3: "unsupported shape",
          -4: "wrong architecture", -5: "CUDA error", -6: "workspace too small"}
FLAG_RMS_INPUT = 1
FLAG_NO_PDL = 2
FLAG_IDS_READY = 4
FLAG_ALL_SMS = 8
STATUS_BAD_EXPERT_ID = 1
STATUS_WAIT_TIMEOUT = 2


class _Weight(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("global_scale", ctypes.c_void_p), ("n", ctypes.c_int32), ("k", ctypes.c_int32)]


class _Fp8Weight(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("n", ctypes.c_int32),
                ("k", ctypes.c_int32)]


class _Bf16Weight(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("ldw", ctypes.c_int64), ("n", ctypes.c_int32),
                ("k", ctypes.c_int32)]


class _Stack(ctypes.Structure):
    _fields_ = [("gu_codes", ctypes.c_void_p), ("gu_scales", ctypes.c_void_p),
                ("dn_codes", ctypes.c_void_p), ("dn_scales", ctypes.c_void_p),
                ("gu_global", ctypes.c_void_p), ("dn_global", ctypes.c_void_p),
                ("num_experts", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("inter", ctypes.c_int32)]


OP_GEMM = 1
OP_MOE = 2


class _Op(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("A", ctypes.c_void_p), ("lda", ctypes.c_int64), ("M", ctypes.c_int32),
                ("W", _Weight), ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64),
                ("argmax_out", ctypes.c_void_p),
                ("x", ctypes.c_void_p), ("ldx", ctypes.c_int64), ("T", ctypes.c_int32),
                ("topk_ids", ctypes.c_void_p), ("topk_w", ctypes.c_void_p), ("k", ctypes.c_int32),
                ("experts", _Stack), ("shared", _Stack), ("out", ctypes.c_void_p),
                ("ldo", ctypes.c_int64), ("argmax_map", ctypes.c_void_p)]


_lib: Optional[ctypes.CDLL] = None


def declared_functions() -> list[str]:
    """Function names declared in the public header."""
    with open(HEADER) as f:
        txt = f.read()
    return sorted(set(re.findall(r"^(?:int|size_t|const char\*)\s+(\w+)\(", txt, re.M)))


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with moe_expert_nvfp4_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i32, i64, sz, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint32
    L.nvfp4_device_check.argtypes = [i32]
    L.nvfp4_workspace_init.argtypes = [vp, sz, vp]
    L.nvfp4_gemm_skinny_workspace.argtypes = [i32, i32, i32]
    L.nvfp4_gemm_skinny_workspace.restype = sz
    L.nvfp4_gemm_skinny.argtypes = [vp, i64, i32, ctypes.POINTER(_Weight), vp, i64, vp, u32, vp, sz, vp]
    L.fp8_gemm_skinny_workspace.argtypes = [i32, i32, i32]
    L.fp8_gemm_skinny_workspace.restype = sz
    L.fp8_gemm_skinny.argtypes = [vp, i64, i32, ctypes.POINTER(_Fp8Weight), vp, i64, vp, u32, vp,
                                  sz, vp]
    L.bf16w_gemm_skinny_workspace.argtypes = [i32, i32, i32]
    L.bf16w_gemm_skinny_workspace.restype = sz
    L.bf16w_gemm_skinny.argtypes = [vp, i64, i32, ctypes.POINTER(_Bf16Weight), vp, i64, vp, u32,
                                    vp, sz, vp]
    L.nvfp4_hot_vocab_head.argtypes = [vp, i64, i32, ctypes.POINTER(_Weight), vp, vp, i64, vp, u32,
                                       vp, sz, vp]
    L.nvfp4_gather_rows.argtypes = [ctypes.POINTER(_Weight), vp, i32, vp, vp, vp]
    L.nvfp4_quantize.argtypes = [vp, i64, i32, i32, vp, vp, vp, vp]
    L.topk_softmax_route.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp]
    L.moe_nvfp4_decode_workspace.argtypes = [i32, i32, ctypes.POINTER(_Stack)]
    L.moe_nvfp4_decode_workspace.restype = sz
    L.moe_nvfp4_decode.argtypes = [vp, i64, i32, vp, vp, i32, ctypes.POINTER(_Stack),
                                   ctypes.POINTER(_Stack), vp, i64, u32, vp, sz, vp]
    L.nvfp4_program_workspace.argtypes = [ctypes.POINTER(_Op), i32]
    L.nvfp4_program_workspace.restype = sz
    L.nvfp4_program_create.argtypes = [ctypes.POINTER(_Op), i32, vp, sz, ctypes.POINTER(vp)]
    L.nvfp4_program_launch.argtypes = [vp, vp]
    L.nvfp4_program_destroy.argtypes = [vp]
    L.nvfp4_read_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    L.nvfp4_last_dispatch.argtypes = [ctypes.c_char_p, sz]
    L.nvfp4_hbm_read_probe.argtypes = [vp, sz, vp, sz, vp]
    L.nvfp4_last_error.restype = ctypes.c_char_p
    for name in declared_functions():
        getattr(L, name)  # every declared symbol must resolve
    _lib = L
    return L


def last_error() -> str:
    return load().nvfp4_last_error().decode()


def last_dispatch() -> str:
    buf = ctypes.create_string_buffer(512)
    load().nvfp4_last_dispatch(buf, 512)
    return buf.value.decode()


def _check(rc: int, what: str):
    if rc != NVFP4_OK:
        raise RuntimeError(f"{what} failed ({rc}: {ERRORS.get(rc, '?')}): {last_error()}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


# ------------------------------------------------------------------ weights

@dataclass
class NVFP4Weight:
    """An NVFP4 matrix [n, k] on the device: codes uint8 [n, k/2], scales
    uint8 [n, k/16] (E4M3 bytes), global_scale float32 [1]."""
    codes: torch.Tensor
    scales: torch.Tensor
    global_scale: torch.Tensor

    @property
    def n(self) -> int:
        return self.codes.shape[0]

    @property
    def k(self) -> int:
        return self.codes.shape[1] * 2

    def c(self) -> _Weight:
        return _Weight(self.codes.data_ptr(), self.scales.data_ptr(), self.global_scale.data_ptr(),
                       self.n, self.k)


@dataclass
class ExpertStack:
    """E experts stacked: gu_codes [E, 2I, H/2], gu_scales [E, 2I, H/16],
    dn_codes [E, H, I/2], dn_scales [E, H, I/16], gu_global / dn_global
    float32 [E].  Gate rows are [0, I) of each gate_up matrix."""
    gu_codes: torch.Tensor
    gu_scales: torch.Tensor
    dn_codes: torch.Tensor
    dn_scales: torch.Tensor
    gu_global: torch.Tensor
    dn_global: torch.Tensor

    @property
    def num_experts(self) -> int:
        return self.gu_codes.shape[0]

    @property
    def hidden(self) -> int:
        return self.gu_codes.shape[2] * 2

    @property
    def inter(self) -> int:
        return self.gu_codes.shape[1] // 2

    def c(self) -> _Stack:
        return _Stack(self.gu_codes.data_ptr(), self.gu_scales.data_ptr(), self.dn_codes.data_ptr(),
                      self.dn_scales.data_ptr(), self.gu_global.data_ptr(), self.dn_global.data_ptr(),
                      self.num_experts, self.hidden, self.inter)


# ------------------------------------------------------------------ workspaces

class Workspace:
    """A zero-initialised device buffer reused across calls (one stream)."""

    def __init__(self, nbytes: int, device=None):
        self.buf = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8,
                               device=device or torch.device("cuda"))

    @property
    def nbytes(self) -> int:
        return self.buf.numel()

    def ptr(self) -> int:
        return self.buf.data_ptr()

    def status(self, stream=None) -> int:
        """Read and clear the device status bits (synchronises)."""
        v = ctypes.c_uint32(0)
        _check(load().nvfp4_read_device_status(self.ptr(), ctypes.byref(v), _stream(stream)),
               "nvfp4_read_device_status")
        return v.value


def gemm_workspace_bytes(m: int, n: int, k: int) -> int:
    return int(load().nvfp4_gemm_skinny_workspace(m, n, k))


def moe_workspace_bytes(t: int, k: int, experts: ExpertStack) -> int:
    st = experts.c()
    return int(load().moe_nvfp4_decode_workspace(t, k, ctypes.byref(st)))


def device_check(device: int = 0) -> int:
    return int(load().nvfp4_device_check(device))


# ------------------------------------------------------------------ calls

def gemm(a: torch.Tensor, w: NVFP4Weight, out: Optional[torch.Tensor] = None,
         argmax: bool = False, rms_input: bool = False, workspace: Optional[Workspace] = None,
         pdl: bool = True, stream=None, argmax_out: Optional[torch.Tensor] = None):
    """C = A W^T for BF16 A [M, >=K] (row stride a.stride(0)).  Returns C
    (BF16 [M, N]) and, with argmax=True (or an int32 [M] ``argmax_out``),
    also the row argmaxes."""
    L = load()
    m = a.shape[0]
    if out is None:
        out = torch.empty(m, w.n, dtype=torch.bfloat16, device=a.device)
    argmax = argmax or argmax_out is not None
    ids = argmax_out
    if argmax and ids is None:
        ids = torch.empty(m, dtype=torch.int32, device=a.device)
    if workspace is None:
        workspace = Workspace(gemm_workspace_bytes(m, w.n, w.k), a.device)
    flags = (FLAG_RMS_INPUT if rms_input else 0) | (0 if pdl else FLAG_NO_PDL)
    wc = w.c()
    _check(L.nvfp4_gemm_skinny(a.data_ptr(), a.stride(0), m, ctypes.byref(wc), out.data_ptr(),
                               out.stride(0), _ptr(ids), flags, workspace.ptr(), workspace.nbytes,
                               _stream(stream)), "nvfp4_gemm_skinny")
    return (out, ids) if argmax else out


@dataclass
class FP8Weight:
    """An FP8-E4M3 matrix [n, k] on the device: codes uint8 [n, k], scale
    float32 [1] (one scale for the matrix)."""
    codes: torch.Tensor
    scale: torch.Tensor

    @property
    def n(self) -> int:
        return self.codes.shape[0]

    @property
    def k(self) -> int:
        return self.codes.shape[1]

    def c(self) -> _Fp8Weight:
        assert self.codes.dtype == torch.uint8 and self.codes.is_contiguous()
        return _Fp8Weight(self.codes.data_ptr(), self.scale.data_ptr(), self.n, self.k)


def _dense_call(fn, wsfn, name, a, wc, n, k, out, argmax, argmax_out, rms_input, workspace, pdl,
                stream):
    L = load()
    m = a.shape[0]
    if out is None:
        out = torch.empty(m, n, dtype=torch.bfloat16, device=a.device)
    argmax = argmax or argmax_out is not None
    ids = argmax_out
    if argmax and ids is None:
        ids = torch.empty(m, dtype=torch.int32, device=a.device)
    if workspace is None:
        workspace = Workspace(int(wsfn(m, n, k)), a.device)
    flags = (FLAG_RMS_INPUT if rms_input else 0) | (0 if pdl else FLAG_NO_PDL)
    _check(fn(a.data_ptr(), a.stride(0), m, ctypes.byref(wc), out.data_ptr(), out.stride(0),
              _ptr(ids), flags, workspace.ptr(), workspace.nbytes, _stream(stream)), name)
    return (out, ids) if argmax else out


def fp8_gemm(a: torch.Tensor, w: FP8Weight, out: Optional[torch.Tensor] = None,
             argmax: bool = False, rms_input: bool = False, workspace: Optional[Workspace] = None,
             pdl: bool = True, stream=None, argmax_out: Optional[torch.Tensor] = None):
    """C = scale * A e4m3(W)^T for BF16 A [M, >=K] (as gemm())."""
    L = load()
    return _dense_call(L.fp8_gemm_skinny, L.fp8_gemm_skinny_workspace, "fp8_gemm_skinny", a,
                       w.c(), w.n, w.k, out, argmax, argmax_out, rms_input, workspace, pdl, stream)


def bf16w_gemm(a: torch.Tensor, w: torch.Tensor, out: Optional[torch.Tensor] = None,
               argmax: bool = False, rms_input: bool = False,
               workspace: Optional[Workspace] = None, pdl: bool = True, stream=None,
               argmax_out: Optional[torch.Tensor] = None):
    """C = A W^T for BF16 A [M, >=K] and BF16 weights W [N, K] (row stride
    w.stride(0)) (as gemm())."""
    L = load()
    assert w.dtype == torch.bfloat16 and w.stride(1) == 1
    wc = _Bf16Weight(w.data_ptr(), w.stride(0), w.shape[0], w.shape[1])
    return _dense_call(L.bf16w_gemm_skinny, L.bf16w_gemm_skinny_workspace, "bf16w_gemm_skinny", a,
                       wc, w.shape[0], w.shape[1], out, argmax, argmax_out, rms_input, workspace,
                       pdl, stream)


def hbm_read_probe(buf: torch.Tensor, sink: torch.Tensor, stream=None) -> None:
    """Read ``buf`` (device, 16-byte aligned, size a multiple of 16) once with
    the library's read-only probe kernel; ``sink`` receives one word per CTA."""
    _check(load().nvfp4_hbm_read_probe(buf.data_ptr(), buf.numel() * buf.element_size(),
                                       sink.data_ptr(), sink.numel() * sink.element_size(),
                                       _stream(stream)), "nvfp4_hbm_read_probe")


def quantize(w: torch.Tensor, stream=None) -> NVFP4Weight:
    """BF16 matrix [N, K] (row stride w.stride(0)) -> its NVFP4 weight (codes,
    E4M3 block scales, per-tensor scale), computed on the device."""
    assert w.dtype == torch.bfloat16 and w.dim() == 2 and w.stride(1) == 1
    n, k = w.shape
    codes = torch.empty(n, k // 2, dtype=torch.uint8, device=w.device)
    scales = torch.empty(n, k // 16, dtype=torch.uint8, device=w.device)
    g = torch.empty(1, dtype=torch.float32, device=w.device)
    _check(load().nvfp4_quantize(w.data_ptr(), w.stride(0), n, k, codes.data_ptr(),
                                 scales.data_ptr(), g.data_ptr(), _stream(stream)),
           "nvfp4_quantize")
    return NVFP4Weight(codes, scales, g)


def gather_rows(w: NVFP4Weight, rows: torch.Tensor, stream=None) -> NVFP4Weight:
    """The NVFP4 matrix of rows ``rows`` (int32 [n], device) of ``w``, in
    list order: the hot-vocabulary head of an output head (a row id outside
    [0, N) gives an all-zero row).  Shares w's global scale."""
    assert rows.dtype == torch.int32 and rows.is_contiguous() and rows.dim() == 1
    n = rows.numel()
    codes = torch.empty(n, w.k // 2, dtype=torch.uint8, device=w.codes.device)
    scales = torch.empty(n, w.k // 16, dtype=torch.uint8, device=w.codes.device)
    wc = w.c()
    _check(load().nvfp4_gather_rows(ctypes.byref(wc), rows.data_ptr(), n, codes.data_ptr(),
                                    scales.data_ptr(), _stream(stream)), "nvfp4_gather_rows")
    return NVFP4Weight(codes, scales, w.global_scale)


def hot_vocab_head(a: torch.Tensor, w_hot: NVFP4Weight, vocab_ids: torch.Tensor,
                   out: Optional[torch.Tensor] = None, argmax_out: Optional[torch.Tensor] = None,
                   rms_input: bool = False, workspace: Optional[Workspace] = None,
                   pdl: bool = True, stream=None):
    """Greedy draft token through a hot-vocabulary head: the hot rows' BF16
    logits C = A W_hot^T [M, n_hot] and the vocabulary id of each row's
    first maximum, vocab_ids[argmax] (int32 [M])."""
    L = load()
    m = a.shape[0]
    assert vocab_ids.dtype == torch.int32 and vocab_ids.is_contiguous()
    assert vocab_ids.numel() == w_hot.n
    if out is None:
        out = torch.empty(m, w_hot.n, dtype=torch.bfloat16, device=a.device)
    if argmax_out is None:
        argmax_out = torch.empty(m, dtype=torch.int32, device=a.device)
    if workspace is None:
        workspace = Workspace(gemm_workspace_bytes(m, w_hot.n, w_hot.k), a.device)
    flags = (FLAG_RMS_INPUT if rms_input else 0) | (0 if pdl else FLAG_NO_PDL)
    wc = w_hot.c()
    _check(L.nvfp4_hot_vocab_head(a.data_ptr(), a.stride(0), m, ctypes.byref(wc),
                                  vocab_ids.data_ptr(), out.data_ptr(), out.stride(0),
                                  argmax_out.data_ptr(), flags, workspace.ptr(), workspace.nbytes,
                                  _stream(stream)), "nvfp4_hot_vocab_head")
    return out, argmax_out


def route(logits: torch.Tensor, k: int, renormalize: bool = True,
          ids: Optional[torch.Tensor] = None, weights: Optional[torch.Tensor] = None, stream=None):
    """Top-k softmax routing of float32 logits [T, E] -> (ids int32 [T, k],
    weights float32 [T, k])."""
    L = load()
    t, e = logits.shape
    assert logits.is_contiguous() and logits.dtype == torch.float32
    if ids is None:
        ids = torch.empty(t, k, dtype=torch.int32, device=logits.device)
    if weights is None:
        weights = torch.empty(t, k, dtype=torch.float32, device=logits.device)
    _check(L.topk_softmax_route(logits.data_ptr(), t, e, k, 1 if renormalize else 0,
                                ids.data_ptr(), weights.data_ptr(), _stream(stream)),
           "topk_softmax_route")
    return ids, weights


def moe(x: torch.Tensor, ids: torch.Tensor, weights: torch.Tensor, experts: ExpertStack,
        shared: Optional[ExpertStack] = None, out: Optional[torch.Tensor] = None,
        rms_input: bool = False, workspace: Optional[Workspace] = None, pdl: bool = True,
        stream=None, ids_ready: bool = False) -> torch.Tensor:
    """MoE decode layer: BF16 x [T, >=H] -> BF16 out [T, H].  ids_ready: the
    ids/weights were complete before the previous kernel started."""
    L = load()
    t, k = ids.shape
    assert ids.is_contiguous() and weights.is_contiguous()
    if out is None:
        out = torch.empty(t, experts.hidden, dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = Workspace(moe_workspace_bytes(t, k, experts), x.device)
    flags = ((FLAG_RMS_INPUT if rms_input else 0) | (0 if pdl else FLAG_NO_PDL)
             | (FLAG_IDS_READY if ids_ready else 0))
    ec = experts.c()
    sc = shared.c() if shared is not None else None
    _check(L.moe_nvfp4_decode(x.data_ptr(), x.stride(0), t, ids.data_ptr(), weights.data_ptr(), k,
                              ctypes.byref(ec), ctypes.byref(sc) if sc is not None else None,
                              out.data_ptr(), out.stride(0), flags, workspace.ptr(),
                              workspace.nbytes, _stream(stream)), "moe_nvfp4_decode")
    return out


# ------------------------------------------------------------------ programs

def gemm_op(a: torch.Tensor, w: NVFP4Weight, out: torch.Tensor,
            argmax_out: Optional[torch.Tensor] = None, rms_input: bool = False,
            argmax_map: Optional[torch.Tensor] = None, all_sms: bool = False) -> dict:
    """One GEMM of a program: out = A W^T (as gemm()); with argmax_map (the
    vocabulary ids of a hot-vocabulary head, as hot_vocab_head()) argmax_out
    reports argmax_map[argmax].  all_sms: split the op over every SM exactly
    as the single call does (bit-identical results to it)."""
    assert argmax_map is None or (argmax_map.dtype == torch.int32 and argmax_map.is_contiguous())
    return dict(kind=OP_GEMM, a=a, w=w, out=out, argmax_out=argmax_out, rms_input=rms_input,
                argmax_map=argmax_map, all_sms=all_sms)


def moe_op(x: torch.Tensor, ids: torch.Tensor, weights: torch.Tensor, experts: ExpertStack,
           out: torch.Tensor, shared: Optional[ExpertStack] = None,
           rms_input: bool = False) -> dict:
    """One MoE layer of a program (as moe()); ids / weights must be complete
    before the program is launched."""
    return dict(kind=OP_MOE, x=x, ids=ids, weights=weights, experts=experts, out=out,
                shared=shared, rms_input=rms_input)


def _c_ops(ops: list) -> ctypes.Array:
    arr = (_Op * len(ops))()
    for i, o in enumerate(ops):
        c = arr[i]
        c.kind = o["kind"]
        c.flags = ((FLAG_RMS_INPUT if o.get("rms_input") else 0)
                   | (FLAG_ALL_SMS if o.get("all_sms") else 0))
        if o["kind"] == OP_GEMM:
            a, out = o["a"], o["out"]
            c.A, c.lda, c.M = a.data_ptr(), a.stride(0), a.shape[0]
            c.W = o["w"].c()
            c.C, c.ldc = out.data_ptr(), out.stride(0)
            c.argmax_out = _ptr(o.get("argmax_out"))
            c.argmax_map = _ptr(o.get("argmax_map"))
        else:
            x, ids, out = o["x"], o["ids"], o["out"]
            assert ids.is_contiguous() and o["weights"].is_contiguous()
            c.x, c.ldx, c.T = x.data_ptr(), x.stride(0), ids.shape[0]
            c.topk_ids, c.topk_w, c.k = ids.data_ptr(), o["weights"].data_ptr(), ids.shape[1]
            c.experts = o["experts"].c()
            if o.get("shared") is not None:
                c.shared = o["shared"].c()
            c.out, c.ldo = out.data_ptr(), out.stride(0)
    return arr


def program_workspace_bytes(ops: list) -> int:
    arr = _c_ops(ops)
    return int(load().nvfp4_program_workspace(arr, len(ops)))


class Program:
    """A fixed chain of GEMM / MoE calls run by one persistent launch.  The
    tensors of ``ops`` (and the workspace) are bound at creation: keep them
    alive and write new inputs into them in place."""

    def __init__(self, ops: list, workspace: Optional[Workspace] = None):
        L = load()
        self._keep = ops
        arr = _c_ops(ops)
        if workspace is None:
            dev = ops[0]["a"].device if ops[0]["kind"] == OP_GEMM else ops[0]["x"].device
            workspace = Workspace(L.nvfp4_program_workspace(arr, len(ops)), dev)
        self.workspace = workspace
        h = ctypes.c_void_p()
        _check(L.nvfp4_program_create(arr, len(ops), workspace.ptr(), workspace.nbytes,
                                      ctypes.byref(h)), "nvfp4_program_create")
        self._h = h

    def launch(self, stream=None):
        _check(load().nvfp4_program_launch(self._h, _stream(stream)), "nvfp4_program_launch")

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            load().nvfp4_program_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
