"""Stacked decode step: the full decode-time weight stream of a 4-bit MoE model.

L layers, each: RMS glue -> QKV projection (hidden -> qkv_out) -> RMS glue on
the first o_in columns -> O projection (o_in -> hidden) -> RMS glue ->
top-k routed MoE layer with a shared expert; then RMS glue -> 4-bit head ->
argmax.  Router logits are inputs (one [T, E] block per layer), so routing
for all layers runs first, in one launch.  Every step is a library call
(route, gemm, moe); the RMS glue is fused into the consuming call
(NVFP4_FLAG_RMS_INPUT).  The whole step is captured as one CUDA graph; with
programmatic dependent launch each kernel starts streaming its weights
while its predecessor finishes.

The glue is this library's stand-in for the model's normalisation layers
(the pages give none): without it 40 random layers leave the BF16 range.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import ops, synth

ROLE_QKV = 21
ROLE_O = 22
ROLE_HEAD = 23


def nvfp4_bytes(n: int, k: int) -> int:
    """Bytes one read of an NVFP4 [n, k] matrix moves (codes + block scales)."""
    return n * k // 2 + n * k // 16


@dataclass
class StepShape:
    layers: int = 40
    num_experts: int = 256
    hidden: int = 2048
    inter: int = 512
    top_k: int = 8
    qkv_out: int = 5120
    o_in: int = 4096
    vocab: int = 151936


class DecodeStep:
    """Weights of the stacked model on the device, generated from ``seed``."""

    def __init__(self, seed: int = 6, shape: StepShape = StepShape(), device: str = "cuda"):
        self.seed, self.s, self.device = seed, shape, device
        s = shape
        g1 = torch.full((1,), synth.GLOBAL_SCALE, dtype=torch.float32, device=device)
        gE = torch.full((s.num_experts,), synth.GLOBAL_SCALE, dtype=torch.float32, device=device)
        self.qkv, self.o, self.experts, self.shared = [], [], [], []
        for l in range(s.layers):
            c, sc = synth.nvfp4_weight(seed, s.qkv_out, s.hidden, ROLE_QKV, l, device=device)
            self.qkv.append(ops.NVFP4Weight(c, sc, g1))
            c, sc = synth.nvfp4_weight(seed, s.hidden, s.o_in, ROLE_O, l, device=device)
            self.o.append(ops.NVFP4Weight(c, sc, g1))
            gc, gs, dc, ds = synth.expert_stack(seed, l, range(s.num_experts), s.hidden, s.inter,
                                                device)
            self.experts.append(ops.ExpertStack(gc, gs, dc, ds, gE, gE))
            gc, gs, dc, ds = synth.expert_stack(seed, l, [s.num_experts], s.hidden, s.inter,
                                                device)
            self.shared.append(ops.ExpertStack(gc, gs, dc, ds, g1, g1))
        c, sc = synth.nvfp4_weight(seed, s.vocab, s.hidden, ROLE_HEAD, device=device)
        self.head = ops.NVFP4Weight(c, sc, g1)

    # ------------------------------------------------------------ inputs
    def inputs(self, tokens: int, seed: Optional[int] = None):
        """Host inputs of one step: activations BF16 [T, hidden] and router
        logits float32 [layers * T, E] (layer-major)."""
        seed = self.seed if seed is None else seed
        s = self.s
        x = synth.activations_bf16(seed, tokens, s.hidden, 31)
        lg = torch.cat([synth.router_logits(seed, tokens, s.num_experts, 32, l)
                        for l in range(s.layers)])
        return x, lg

    # ------------------------------------------------------------ buffers
    def buffers(self, tokens: int, keep: bool = False) -> dict:
        s, d, T = self.s, self.device, tokens
        ws = max(ops.gemm_workspace_bytes(T, s.qkv_out, s.hidden),
                 ops.gemm_workspace_bytes(T, s.hidden, s.o_in),
                 ops.gemm_workspace_bytes(T, s.vocab, s.hidden),
                 ops.moe_workspace_bytes(T, s.top_k, self.experts[0]))
        n_act = s.layers if keep else 1
        b = {
            "T": T,
            "x": torch.zeros(T, s.hidden, dtype=torch.bfloat16, device=d),
            "logits": torch.zeros(s.layers * T, s.num_experts, dtype=torch.float32, device=d),
            "ids": torch.zeros(s.layers * T, s.top_k, dtype=torch.int32, device=d),
            "w": torch.zeros(s.layers * T, s.top_k, dtype=torch.float32, device=d),
            "q": [torch.zeros(T, s.qkv_out, dtype=torch.bfloat16, device=d) for _ in range(n_act)],
            "o": [torch.zeros(T, s.hidden, dtype=torch.bfloat16, device=d) for _ in range(n_act)],
            "y": [torch.zeros(T, s.hidden, dtype=torch.bfloat16, device=d)
                  for _ in range(s.layers if keep else 2)],
            "head": torch.zeros(T, s.vocab, dtype=torch.bfloat16, device=d),
            "argmax": torch.zeros(T, dtype=torch.int32, device=d),
            "ws": ops.Workspace(ws, d),
            "keep": keep,
        }
        return b

    # ------------------------------------------------------------ the step
    def run(self, b: dict, pdl: bool = True) -> int:
        """Launch one step on the current stream; returns the number of
        kernel launches it made."""
        s, T, ws = self.s, b["T"], b["ws"]
        launches = 0
        ops.route(b["logits"], s.top_k, True, b["ids"], b["w"])
        launches += 1
        x = b["x"]
        for l in range(s.layers):
            i = l if b["keep"] else 0
            q, o = b["q"][i], b["o"][i]
            y = b["y"][l if b["keep"] else l % 2]
            ops.gemm(x, self.qkv[l], out=q, rms_input=True, workspace=ws, pdl=pdl)
            ops.gemm(q[:, :s.o_in], self.o[l], out=o, rms_input=True, workspace=ws, pdl=pdl)
            ops.moe(o, b["ids"][l * T:(l + 1) * T], b["w"][l * T:(l + 1) * T], self.experts[l],
                    self.shared[l], out=y, rms_input=True, workspace=ws, pdl=pdl,
                    ids_ready=True)
            # QKV, O, and the MoE layer: two CUDA-core kernels per batch of
            # 16 tokens, or three tensor-core kernels
            d = ops.last_dispatch()
            launches += 2 + (2 * int(d.split("batches=")[1].split()[0])
                             if "batches=" in d else 3)
            x = y
        ops.gemm(x, self.head, out=b["head"], argmax_out=b["argmax"], rms_input=True, workspace=ws,
                 pdl=pdl)
        launches += 1
        return launches

    # ------------------------------------------------------------ which way
    # Steps of at most this many tokens run call by call: their MoE layers
    # (and the dense calls of one or a few rows) go to the CUDA-core kernels,
    # which start in a few us, and the small tensor-core calls hold only some
    # of the SMs while the next call starts on the others; the persistent
    # program pays each op's completion wait and activation staging instead.
    # Measured on GB300, 40 layers, call by call against the program: T = 1
    # 0.93 against 2.96 ms, T = 2 1.15 / 2.83, T = 4 1.73 / 2.90, T = 8
    # 2.79 / 3.56, T = 16 4.74 / 5.32, T = 32 9.05 / 10.57: every token count
    # the library takes.
    CALLS_MAX_TOKENS = 32

    def path_for(self, tokens: int) -> str:
        """"calls" or "program": the faster way to run a step of ``tokens``."""
        return "calls" if tokens <= self.CALLS_MAX_TOKENS else "program"

    # ------------------------------------------------------------ as a program
    def program_ops(self, b: dict, all_sms: bool = False) -> list:
        """The step's projections, MoE layers and head as one op chain
        (all_sms: every op split over every SM, as the single calls)."""
        s, T = self.s, b["T"]
        chain = []
        x = b["x"]
        for l in range(s.layers):
            i = l if b["keep"] else 0
            q, o = b["q"][i], b["o"][i]
            y = b["y"][l if b["keep"] else l % 2]
            chain.append(ops.gemm_op(x, self.qkv[l], q, rms_input=True, all_sms=all_sms))
            chain.append(ops.gemm_op(q[:, :s.o_in], self.o[l], o, rms_input=True, all_sms=all_sms))
            chain.append(ops.moe_op(o, b["ids"][l * T:(l + 1) * T], b["w"][l * T:(l + 1) * T],
                                    self.experts[l], y, shared=self.shared[l], rms_input=True))
            x = y
        chain.append(ops.gemm_op(x, self.head, b["head"], argmax_out=b["argmax"], rms_input=True,
                                 all_sms=all_sms))
        return chain

    def program(self, b: dict, all_sms: bool = False) -> "ops.Program":
        """Create the step's program on the buffers ``b`` (once)."""
        chain = self.program_ops(b, all_sms)
        need = ops.program_workspace_bytes(chain)
        if b["ws"].nbytes < need:
            b["ws"] = ops.Workspace(need, self.device)
        return ops.Program(chain, b["ws"])

    def run_program(self, b: dict, prog: "ops.Program") -> int:
        """One step as two launches: routing of every layer, then the program."""
        ops.route(b["logits"], self.s.top_k, True, b["ids"], b["w"])
        prog.launch()
        return 2

    def capture(self, b: dict, pdl: bool = True, prog: "ops.Program" = None) -> torch.cuda.CUDAGraph:
        """Warm up, then capture one step (call by call, or as ``prog``) as a
        CUDA graph; b["launches"] = the kernels one step launches."""
        step = (lambda: self.run(b, pdl)) if prog is None else (lambda: self.run_program(b, prog))
        b["launches"] = step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        torch.cuda.synchronize()
        return g

    # ------------------------------------------------------------ accounting
    def step_bytes(self, ids: torch.Tensor, tokens: int) -> int:
        """Algorithmic weight bytes of one step for the given routing: every
        projection once, every distinct routed expert of each layer plus its
        shared expert once, and the head."""
        s = self.s
        per_expert = nvfp4_bytes(2 * s.inter, s.hidden) + nvfp4_bytes(s.hidden, s.inter)
        ids = ids.view(s.layers, tokens * s.top_k).cpu()
        total = 0
        for l in range(s.layers):
            valid = ids[l][(ids[l] >= 0) & (ids[l] < s.num_experts)]
            total += (torch.unique(valid).numel() + 1) * per_expert
        total += s.layers * (nvfp4_bytes(s.qkv_out, s.hidden) + nvfp4_bytes(s.hidden, s.o_in))
        total += nvfp4_bytes(s.vocab, s.hidden)
        return total
