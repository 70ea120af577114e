#!/usr/bin/env python3
"""Benchmark: the stacked NVFP4 decode step on GB300.

One step = one pass of the whole hot path over one batch of T tokens:
routing for 40 layers, then per layer the QKV (2048 -> 5120) and O
(4096 -> 2048) projections and the 256+1-expert MoE layer (hidden 2048,
intermediate 512, top-8), then the 151,936-row 4-bit head with argmax;
about 18.8 GB of NVFP4 weights resident in HBM.  The metric is the
algorithmic weight bytes one step must read (every projection, every
distinct routed expert plus the shared expert of each layer, and the head)
divided by the step time, in GB/s; the step's microseconds are reported too.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--tokens T]
  python bench.py --impl reference ...   # the float64 CPU oracle, same metric

N > 1 runs N independent replicas (one per GPU, launched by torchrun): the
path has no exchange step, so there is no collective on the data path.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 skinny-GEMM/MoE decode µs and HBM GB/s (frac of GB300 peak), M=1–32"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--tokens", type=int, default=8)
    p.add_argument("--layers", type=int, default=40,
                   help="layers of the stacked step (fewer only for small profiling runs)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-sweep", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--profile", default=None, metavar="WORKLOAD",
                   help="run one workload's calls a few times and exit (for ncu captures): "
                        "dense:N:K:M, head:M, moe:T, fp8:N:K:M, bf16w:N:K:M")
    p.add_argument("--path", default="auto", choices=["auto", "program", "calls"],
                   help="program: the step as one persistent launch after routing; calls: one "
                        "kernel launch per call; auto: the step's own choice for its token "
                        "count (DecodeStep.path_for)")
    return p.parse_args()


def workload_name(t, layers=40):
    return (f"stacked decode step, T={t} tokens: {layers} x (QKV NVFP4 2048->5120, O NVFP4 "
            f"4096->2048, MoE 256 routed + 1 shared experts, hidden 2048, inter 512, top-8) "
            f"+ NVFP4 head 151936x2048 + argmax")


# ------------------------------------------------------------------ distributed

def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n and world > 1:
        raise SystemExit(f"--gpus {n} but WORLD_SIZE={world}")
    return rank, world, local


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of the ranks' values (the slowest replica's time); x
    itself when there is one rank (dist None)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the bytes all ranks processed over the slowest
    rank's time, in GB/s."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.samples = []

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm_sorted) // 2] if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ helpers

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(kernel_key):
    """DRAM bytes per launch recorded from an ncu capture, valid only while
    the kernel's sources (the entry's ``sources``, else all of them) are
    unchanged (same hash)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    from moe_expert_nvfp4_gb300 import build as B
    ent = d.get(kernel_key)
    if not ent or ent.get("source_hash") != B.source_hash(ent.get("sources")):
        return None
    return ent.get("dram_bytes_per_launch")


def timed_replays(graph, steps, stream, spread=None):
    """Milliseconds per replay of ``graph`` over ``steps`` back-to-back
    replays (CUDA events on ``stream``).  With ``spread`` (a dict) an event
    after every replay also gives the per-replay times' mean and standard
    deviation (microseconds) and their count."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    evs[0].record(stream)
    for i in range(steps):
        graph.replay()
        if spread is not None or i == steps - 1:
            evs[i + 1].record(stream)
    evs[-1].synchronize()
    if spread is not None:
        per = np.array([evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]) * 1e3
        spread.update({"mean_us": float(per.mean()), "std_us": float(per.std(ddof=1)) if steps > 1
                       else 0.0, "n": steps, "min_us": float(per.min()), "max_us": float(per.max())})
    return evs[0].elapsed_time(evs[-1]) / steps  # ms per replay


def versions():
    """nvcc, driver, torch, the kernel sources' hash and the git commit (when
    the checkout has one) of this run."""
    import torch
    from moe_expert_nvfp4_gb300 import build as B
    out = {"torch": torch.__version__, "source_hash": B.source_hash()}
    try:
        r = subprocess.run([B._nvcc(), "--version"], capture_output=True, text=True, timeout=30)
        out["nvcc"] = r.stdout.strip().splitlines()[-1]
    except Exception:
        out["nvcc"] = None
    try:
        r = subprocess.run(["nvidia-smi", "--query-gpu=driver_version,name", "--format=csv,noheader",
                            "-i", "0"], capture_output=True, text=True, timeout=30)
        out["driver"], out["gpu"] = [v.strip() for v in r.stdout.strip().split(",")[:2]]
    except Exception:
        out["driver"] = out["gpu"] = None
    try:
        r = subprocess.run(["git", "rev-parse", "HEAD"], capture_output=True, text=True, cwd=ROOT,
                           timeout=30)
        out["git_sha"] = r.stdout.strip() or None
    except Exception:
        out["git_sha"] = None
    return out


def read_probe_gbs(reps=10):
    """Read-only HBM bandwidth of this GPU: the library's probe kernel over a
    4 GiB buffer (31x L2), best of ``reps`` timed launches."""
    import torch
    from moe_expert_nvfp4_gb300 import ops
    buf = torch.empty(4 << 30, dtype=torch.uint8, device="cuda")
    buf.fill_(1)
    sink = torch.empty(4096, dtype=torch.int32, device="cuda")
    for _ in range(2):
        ops.hbm_read_probe(buf, sink)
    torch.cuda.synchronize()
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        ops.hbm_read_probe(buf, sink)
        e1.record()
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    n = buf.numel()
    del buf
    return {"gbs": n / (best * 1e-3) / 1e9, "bytes": n, "kernel": "read_probe_kernel",
            "how": f"best of {reps} launches, CUDA events"}


class OracleSample:
    """The float64 oracle on layer 0 of the step, one op at a time: routing,
    the QKV projection, the O projection, then each expert the layer routes
    to (shared expert first).  Each ``step()`` runs the next op in that
    cycle and returns (weight bytes it read, seconds).  Host copies of the
    weights are made once, outside the timed calls."""

    def __init__(self, tokens, x_host, logits_host, layer=0):
        import oracle as O
        from moe_expert_nvfp4_gb300 import synth
        from moe_expert_nvfp4_gb300.decode_step import ROLE_O, ROLE_QKV, nvfp4_bytes
        H, I, E, k, qo, oi, seed = 2048, 512, 256, 8, 5120, 4096, 6
        self.O = O
        qkv = synth.nvfp4_weight(seed, qo, H, ROLE_QKV, layer)
        o = synth.nvfp4_weight(seed, H, oi, ROLE_O, layer)
        self.qkv = (qkv[0].numpy(), qkv[1].numpy(), synth.GLOBAL_SCALE)
        self.o = (o[0].numpy(), o[1].numpy(), synth.GLOBAL_SCALE)
        self.lg = logits_host[layer * tokens:(layer + 1) * tokens].numpy()
        self.ids, self.w = O.topk_softmax_route(self.lg, k)
        routed = sorted(set(self.ids.flatten().tolist()))
        self.experts = {e: synth.expert_host(seed, layer, e, H, I) for e in [E] + routed}
        self.x = x_host.double().numpy()
        self.k, self.E = k, E
        per_expert = nvfp4_bytes(2 * I, H) + nvfp4_bytes(H, I)
        self.ops = ([("route", 0), ("qkv", nvfp4_bytes(qo, H)), ("o", nvfp4_bytes(H, oi))]
                    + [(e, per_expert) for e in [E] + routed])
        self.i = 0

    def step(self):
        O = self.O
        name, nbytes = self.ops[self.i % len(self.ops)]
        self.i += 1
        t0 = time.perf_counter()
        if name == "route":
            O.topk_softmax_route(self.lg, self.k)
        elif name == "qkv":
            O.gemm_bf16(O.rms_scale(self.x), *self.qkv)
        elif name == "o":
            O.gemm_bf16(O.rms_scale(self.x[:, :2048].repeat(2, axis=1)), *self.o)
        else:
            rows = np.arange(self.x.shape[0]) if name == self.E else np.nonzero(
                (self.ids == name).any(axis=1))[0]
            O.expert_ffn64(O.rms_scale(self.x[rows]), self.experts[name])
        return nbytes, time.perf_counter() - t0


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [p.get("num_threads") for p in threadpool_info() if p.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


# ------------------------------------------------------------------ reference arm

def run_reference(args, rank):
    if rank != 0:
        return
    import torch
    from moe_expert_nvfp4_gb300 import synth
    t = args.tokens
    x = synth.activations_bf16(6, t, 2048, 31)
    lg = torch.cat([synth.router_logits(6, t, 256, 32, l) for l in range(1)])
    sampler = OracleSample(t, x, lg)
    for _ in range(args.warmup):
        sampler.step()
    sampler.i = 0
    tot_b, tot_s = 0, 0.0
    for _ in range(args.steps):
        b, dt = sampler.step()
        tot_b += b
        tot_s += dt
    value = tot_b / tot_s / 1e9
    cores = blas_threads()
    sample = (f"layer 0 of the T={t} step, one oracle op per timed step, cycling through "
              f"routing, QKV, O and each routed expert ({len(sampler.ops)} ops)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_name(t), "tokens": t},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ per-workload context

def graph_us(fn, reps, warmup=3):
    """Device microseconds per replay of a CUDA graph of fn() (CUDA events on
    the current stream, after warm-up replays)."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    ms = timed_replays(g, reps, torch.cuda.current_stream())
    del g
    return ms * 1e3


def workload_table(model, reps=10):
    """Microseconds and weight GB/s of the other workloads the metric is quoted
    on, each timed as a CUDA graph of back-to-back calls over weight copies
    that together exceed L2 (so every call reads HBM):

    * the 2048 -> 64 projection at M = 4 (latency-bound; its 74 KB weight
      stays in L2): one call per graph replay (the replay's own launch
      included), and per call in a graph of 32 back-to-back calls over 32
      weight copies (``proj_2048x64_M4_chain``);
    * the dense sweep: M in {1, 4, 8, 16, 32} x {4096 x 2048, 8192 x 2048,
      2048 x 4096} (seeds 1-3);
    * the MoE layer (256 routed + 1 shared experts, hidden 2048, inter 512,
      top-8) at T in {1, 2, 4, 8, 16, 32}, over the step's layer weights
      (where the call runs on the CUDA cores, the same layers on the tensor
      cores too);
    * the MTP-verify batch: the MoE layer at T = 32 then the 151,936 x 2048
      head with argmax;
    * the hot-vocabulary draft head: 32,768 listed rows of that head (the
      FR-Spec list; a seeded sorted subset of the vocabulary) with argmax at
      M in {1, 8, 32}, over 8 copies gathered from different lists, and the
      gather that builds one (bytes read + written);
    * the BF16 -> NVFP4 quantisation of a 151,936 x 2048 BF16 head (bytes:
      the BF16 matrix read twice -- the per-tensor maximum precedes every
      code -- and the NVFP4 matrix written)."""
    import torch
    from moe_expert_nvfp4_gb300 import ops, synth
    from moe_expert_nvfp4_gb300.decode_step import nvfp4_bytes
    dev = "cuda"
    g1 = torch.full((1,), synth.GLOBAL_SCALE, dtype=torch.float32, device=dev)
    out = {}

    def weights(seed, n, k, count):
        return [ops.NVFP4Weight(*synth.nvfp4_weight(seed, n, k, 40 + i, device=dev), g1)
                for i in range(count)]

    # the 2048 -> 64 projection at M = 4
    ws64 = weights(0, 64, 2048, 1)
    a = synth.activations_bf16(0, 4, 2048).to(dev)
    c = torch.empty(4, 64, dtype=torch.bfloat16, device=dev)
    wk = ops.Workspace(ops.gemm_workspace_bytes(4, 64, 2048))
    us = graph_us(lambda: ops.gemm(a, ws64[0], out=c, workspace=wk), reps)
    out["proj_2048x64_M4"] = {"us": us, "gbs": nvfp4_bytes(64, 2048) / us / 1e3}
    ws64 = weights(0, 64, 2048, 32)

    def chain():
        for w in ws64:
            ops.gemm(a, w, out=c, workspace=wk)
    us = graph_us(chain, reps) / len(ws64)
    out["proj_2048x64_M4_chain"] = {"us": us, "gbs": nvfp4_bytes(64, 2048) / us / 1e3,
                                    "kernel": ops.last_dispatch().split()[0]}
    del ws64

    # dense sweep; 24 rotating copies of each shape (>= 113 MB each set)
    for seed, (n, k) in zip((1, 2, 3), ((4096, 2048), (8192, 2048), (2048, 4096))):
        copies = weights(seed, n, k, 24 if n * k <= 4096 * 2048 else 16)
        wk = ops.Workspace(max(ops.gemm_workspace_bytes(m, n, k) for m in (1, 32)))
        for m in (1, 4, 8, 16, 32):
            a = synth.activations_bf16(seed, m, k).to(dev)
            c = torch.empty(m, n, dtype=torch.bfloat16, device=dev)

            def calls():
                for w in copies:
                    ops.gemm(a, w, out=c, workspace=wk)
            us = graph_us(calls, reps) / len(copies)
            out[f"dense_{n}x{k}_M{m}"] = {"us": us, "gbs": nvfp4_bytes(n, k) / us / 1e3}
        del copies

    # MoE layer over the step's layers (each layer's experts are distinct weights)
    s = model.s
    per_expert = nvfp4_bytes(2 * s.inter, s.hidden) + nvfp4_bytes(s.hidden, s.inter)
    L = min(16, s.layers)
    for t in (1, 2, 4, 8, 16, 32):
        x = synth.activations_bf16(4, t, s.hidden).to(dev)
        lg = torch.cat([synth.router_logits(4, t, s.num_experts, l) for l in range(L)]).to(dev)
        ids, wts = ops.route(lg, s.top_k)
        y = torch.empty(t, s.hidden, dtype=torch.bfloat16, device=dev)
        wk = ops.Workspace(ops.moe_workspace_bytes(t, s.top_k, model.experts[0]))
        idl = ids.view(L, -1).cpu()
        nbytes = sum((torch.unique(idl[l]).numel() + 1) * per_expert for l in range(L))

        def layers():
            for l in range(L):
                ops.moe(x, ids[l * t:(l + 1) * t], wts[l * t:(l + 1) * t], model.experts[l],
                        model.shared[l], out=y, workspace=wk, ids_ready=True)
        us = graph_us(layers, reps)
        out[f"moe_T{t}"] = {"us": us / L, "gbs": nbytes / us / 1e3,
                            "kernel": ops.last_dispatch().split(";")[0]}
        if "batches=" in ops.last_dispatch():  # the CUDA-core kernels
            # the same layers on the tensor-core kernels (one-op programs)
            progs = [ops.Program([ops.moe_op(x, ids[l * t:(l + 1) * t], wts[l * t:(l + 1) * t],
                                             model.experts[l], y, shared=model.shared[l])])
                     for l in range(L)]
            us = graph_us(lambda: [p.launch() for p in progs], reps)
            out[f"moe_tc_T{t}"] = {"us": us / L, "gbs": nbytes / us / 1e3,
                                   "kernel": "stream_tc_kernel (one-op program)"}
            del progs

    # MTP-verify batch: MoE layer at T = 32, then the head with argmax
    t = 32
    x = synth.activations_bf16(5, t, s.hidden).to(dev)
    lg = torch.cat([synth.router_logits(5, t, s.num_experts, l) for l in range(L)]).to(dev)
    ids, wts = ops.route(lg, s.top_k)
    y = torch.empty(t, s.hidden, dtype=torch.bfloat16, device=dev)
    logits = torch.empty(t, s.vocab, dtype=torch.bfloat16, device=dev)
    am = torch.empty(t, dtype=torch.int32, device=dev)
    wk = ops.Workspace(max(ops.moe_workspace_bytes(t, s.top_k, model.experts[0]),
                           ops.gemm_workspace_bytes(t, s.vocab, s.hidden)))
    idl = ids.view(L, -1).cpu()
    head_bytes = nvfp4_bytes(s.vocab, s.hidden)
    nbytes = sum((torch.unique(idl[l]).numel() + 1) * per_expert + head_bytes for l in range(L))

    def verify():
        for l in range(L):
            ops.moe(x, ids[l * t:(l + 1) * t], wts[l * t:(l + 1) * t], model.experts[l],
                    model.shared[l], out=y, workspace=wk, ids_ready=True)
            ops.gemm(y, model.head, out=logits, argmax_out=am, workspace=wk)
    us = graph_us(verify, reps)
    out["mtp_verify_T32"] = {"us": us / L, "gbs": nbytes / us / 1e3}
    del logits

    # hot-vocabulary draft head
    n_hot = 32768
    lists = [torch.randperm(s.vocab, generator=torch.Generator().manual_seed(60 + i))[:n_hot]
             .sort().values.to(torch.int32).to(dev) for i in range(8)]
    hots = [ops.gather_rows(model.head, lst) for lst in lists]
    hot_bytes = nvfp4_bytes(n_hot, s.hidden)
    us = graph_us(lambda: ops.gather_rows(model.head, lists[0]), reps)
    out[f"hot_head_gather_{n_hot}x{s.hidden}"] = {"us": us, "gbs": 2 * hot_bytes / us / 1e3}
    wk = ops.Workspace(ops.gemm_workspace_bytes(32, n_hot, s.hidden))
    for m in (1, 8, 32):
        a = synth.activations_bf16(61, m, s.hidden).to(dev)
        c = torch.empty(m, n_hot, dtype=torch.bfloat16, device=dev)
        am = torch.empty(m, dtype=torch.int32, device=dev)

        def drafts():
            for h, lst in zip(hots, lists):
                ops.hot_vocab_head(a, h, lst, out=c, argmax_out=am, workspace=wk)
        us = graph_us(drafts, reps) / len(hots)
        out[f"hot_head_{n_hot}x{s.hidden}_M{m}"] = {"us": us, "gbs": hot_bytes / us / 1e3}
    del hots

    # the other weight formats on the same path: FP8 W8A16 on the attention
    # projection shapes, BF16 weights on the 2048 -> 64 projection and a
    # 4096 x 2048 matrix (rotating copies > L2 for the larger shapes)
    fscale = torch.full((1,), synth.FP8_SCALE, dtype=torch.float32, device=dev)
    for n, k in ((5120, 2048), (2048, 4096)):
        copies = [ops.FP8Weight(synth.fp8_weight(70 + i, n, k).to(dev), fscale) for i in range(16)]
        wk = ops.Workspace(max(int(ops.load().fp8_gemm_skinny_workspace(m, n, k)) for m in (1, 32)))
        for m in (1, 8, 32):
            a = synth.activations_bf16(70, m, k).to(dev)
            c = torch.empty(m, n, dtype=torch.bfloat16, device=dev)

            def f8():
                for w in copies:
                    ops.fp8_gemm(a, w, out=c, workspace=wk)
            us = graph_us(f8, reps) / len(copies)
            out[f"fp8_{n}x{k}_M{m}"] = {"us": us, "gbs": n * k / us / 1e3}
        del copies
    wb64 = synth.bf16_weight(71, 64, 2048).to(dev)
    a = synth.activations_bf16(71, 4, 2048).to(dev)
    c = torch.empty(4, 64, dtype=torch.bfloat16, device=dev)
    wk = ops.Workspace(int(ops.load().bf16w_gemm_skinny_workspace(4, 64, 2048)))
    us = graph_us(lambda: ops.bf16w_gemm(a, wb64, out=c, workspace=wk), reps)
    out["bf16w_2048x64_M4"] = {"us": us, "gbs": 64 * 2048 * 2 / us / 1e3}
    copies = [synth.bf16_weight(72 + i, 4096, 2048).to(dev) for i in range(12)]
    wk = ops.Workspace(max(int(ops.load().bf16w_gemm_skinny_workspace(m, 4096, 2048)) for m in (1, 8)))
    for m in (1, 8):
        a = synth.activations_bf16(72, m, 2048).to(dev)
        c = torch.empty(m, 4096, dtype=torch.bfloat16, device=dev)

        def bw():
            for w in copies:
                ops.bf16w_gemm(a, w, out=c, workspace=wk)
        us = graph_us(bw, reps) / len(copies)
        out[f"bf16w_4096x2048_M{m}"] = {"us": us, "gbs": 4096 * 2048 * 2 / us / 1e3}
    del copies

    # CUDA cores against tensor cores on the same NVFP4 rows: N rows (enough
    # copies to exceed L2 where the matrix is small), K = 2048 through the
    # tcgen05 kernel (a one-op program when the call itself would take the
    # CUDA-core kernel) and K = 2080 through the CUDA-core kernel (every K
    # that is not a multiple of 256 takes it); GB/s counts each call's own
    # bytes
    for n, n_copies in ((64, 1), (4096, 24), (16384, 8), (s.vocab, 1)):
        tc_w = weights(73, n, 2048, n_copies)
        fm_w = weights(74, n, 2080, n_copies)
        for m in (1, 2, 4, 8):
            row = {}
            for name, ws_, k in (("tcgen05", tc_w, 2048), ("cuda_cores", fm_w, 2080)):
                a = synth.activations_bf16(75, m, k).to(dev)
                c = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
                wk = ops.Workspace(ops.gemm_workspace_bytes(m, n, k))
                ops.gemm(a, ws_[0], out=c, workspace=wk)
                kern = ops.last_dispatch().split()[0]
                if name == "tcgen05" and kern != "stream_tc_kernel<dense>":
                    progs = [ops.Program([ops.gemm_op(a, w, c, all_sms=True)]) for w in ws_]
                    us = graph_us(lambda: [p.launch() for p in progs], reps) / len(progs)
                    kern = "stream_tc_kernel (one-op program)"
                    del progs
                else:
                    def seq():
                        for w in ws_:
                            ops.gemm(a, w, out=c, workspace=wk)
                    us = graph_us(seq, reps) / len(ws_)
                row[name] = {"us": round(us, 2), "gbs": round(nvfp4_bytes(n, k) / us / 1e3, 1),
                             "kernel": kern}
            out[f"tc_vs_fma_{n}x2048_M{m}"] = row
        del tc_w, fm_w

    # BF16 -> NVFP4 quantisation of a head-sized BF16 matrix (622 MB >> L2)
    wb = torch.randn(s.vocab, s.hidden, device=dev,
                     generator=torch.Generator(device=dev).manual_seed(62)).to(torch.bfloat16)
    us = graph_us(lambda: ops.quantize(wb), reps)
    qbytes = s.vocab * s.hidden * (2 + 2) + nvfp4_bytes(s.vocab, s.hidden)
    out[f"quantize_{s.vocab}x{s.hidden}"] = {"us": us, "gbs": qbytes / us / 1e3}
    del wb
    for v in out.values():
        if "us" in v:
            v["us"] = round(v["us"], 2)
            v["gbs"] = round(v["gbs"], 1)
    return out


# ------------------------------------------------------------------ our arm

def run_ours(args, rank, world, local):
    import torch

    from moe_expert_nvfp4_gb300 import build as B
    from moe_expert_nvfp4_gb300 import ops
    from moe_expert_nvfp4_gb300.decode_step import DecodeStep, StepShape

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    B.build()
    ops.load()
    if ops.device_check(local) != 0:
        raise SystemExit(ops.last_error())
    stream = torch.cuda.current_stream()
    model = DecodeStep(seed=6, shape=StepShape(layers=args.layers))
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()

    def path_of(t):
        return model.path_for(t) if args.path == "auto" else args.path

    def one_config(t, steps, warmup, sample_clocks, path=None):
        path = path or path_of(t)
        b = model.buffers(t)
        x, lg = model.inputs(t)
        b["x"].copy_(x)
        b["logits"].copy_(lg)
        prog = model.program(b) if path == "program" else None
        g = model.capture(b, prog=prog)
        b["prog"] = prog
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        clk = ClockSampler(local) if sample_clocks else None
        if clk:
            clk.start()
            time.sleep(0.3)
        barrier()
        torch.cuda.synchronize()
        spread = {}
        ms = timed_replays(g, steps, stream, spread)
        torch.cuda.synchronize()
        barrier()
        clocks = clk.stop() if clk else None
        b["spread"] = spread
        ms = max_over_ranks(ms, dist, "cuda")
        nbytes = model.step_bytes(b["ids"], t)
        status = b["ws"].status()
        if status:
            raise SystemExit(f"device status {status} after the timed steps")
        am = b["argmax"].cpu()
        if ms <= 0 or nbytes <= 0 or int(am.min()) < 0 or int(am.max()) >= model.s.vocab:
            raise SystemExit("benchmark produced an empty or invalid result")
        return b, g, x, lg, ms, nbytes, clocks

    t = args.tokens
    b, g, x, lg, ms, nbytes, clocks = one_config(t, args.steps, args.warmup, True)
    n_launch = b["launches"]
    value = job_gbs(nbytes, world, ms)

    # ---- end to end: pinned host inputs in, argmax ids out, every step
    xh = x.pin_memory()
    lgh = lg.pin_memory()
    outh = torch.empty(t, dtype=torch.int32).pin_memory()
    e_steps = max(3, min(args.steps, 50))
    for _ in range(2):
        b["x"].copy_(xh, non_blocking=True)
        b["logits"].copy_(lgh, non_blocking=True)
        g.replay()
        outh.copy_(b["argmax"], non_blocking=True)
        stream.synchronize()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e_steps):
        b["x"].copy_(xh, non_blocking=True)
        b["logits"].copy_(lgh, non_blocking=True)
        g.replay()
        outh.copy_(b["argmax"], non_blocking=True)
        stream.synchronize()
    e_ms = (time.perf_counter() - t0) * 1e3 / e_steps
    barrier()
    e_ms = max_over_ranks(e_ms, dist, "cuda")
    e2e = {"value": job_gbs(nbytes, world, e_ms), "unit": UNIT,
           "h2d_bytes_per_step": xh.numel() * xh.element_size() + lgh.numel() * lgh.element_size(),
           "d2h_bytes_per_step": outh.numel() * outh.element_size(), "ms_per_step": e_ms,
           "steps": e_steps}

    # ---- the dominant kernel, timed alone with CUDA events on its stream
    s = model.s
    peak, peak_kind = measured_peak()
    peak_src = (f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s")
    path = path_of(t)
    probe = read_probe_gbs() if rank == 0 else None

    def family(name, key, calls_fn, nbytes_f, launches):
        """A kernel family of the step timed alone: a CUDA graph of its calls
        back to back, CUDA events on the stream."""
        kg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(kg):
            calls_fn()
        for _ in range(3):
            kg.replay()
        torch.cuda.synchronize()
        k_ms = timed_replays(kg, max(5, min(args.steps, 100)), stream)
        del kg
        achieved = nbytes_f / (k_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": profiled_traffic(key), "kernel": name,
                "bytes_per_launch": nbytes_f / launches, "us_per_launch": k_ms * 1e3 / launches,
                "ms_per_step": k_ms, "peak_source": peak_src, "frac_of_8tbs": achieved / 8000.0,
                "read_probe": probe,
                "frac_of_read_probe": achieved / probe["gbs"] if probe else None}

    families = {}
    if path == "program":
        # the program kernel: every projection, MoE layer and the head of the step
        families["program"] = family(
            f"stream_tc_kernel, program of the step ({3 * s.layers + 1} calls), per launch",
            f"program_T{t}_L{s.layers}", lambda: b["prog"].launch(), nbytes, 1)
    else:
        # the step's two kernel families, each timed alone: its MoE layer calls
        # and its dense calls (QKV, O, head)
        per_expert = 3 * 2048 * 512 * 9 // 16  # gate_up + down bytes of one expert
        ids_l = b["ids"].view(s.layers, -1).cpu()
        moe_bytes = sum((torch.unique(ids_l[l]).numel() + 1) * per_expert for l in range(s.layers))

        def moe_calls():
            for l in range(s.layers):
                ops.moe(b["o"][0], b["ids"][l * t:(l + 1) * t], b["w"][l * t:(l + 1) * t],
                        model.experts[l], model.shared[l], out=b["y"][0], rms_input=True,
                        workspace=b["ws"], ids_ready=True)
        moe_calls()
        kernels = " + ".join(w.split()[0] for w in ops.last_dispatch().split(";")[:3]
                             if w.strip() and not w.strip().startswith("T="))
        families["moe"] = family(f"moe_nvfp4_decode ({kernels}), per call", f"moe_layer_T{t}",
                                 moe_calls, moe_bytes, s.layers)

        seen = []

        def dense_calls():
            for l in range(s.layers):
                ops.gemm(b["x"], model.qkv[l], out=b["q"][0], rms_input=True, workspace=b["ws"])
                seen.append(ops.last_dispatch().split()[0])
                ops.gemm(b["q"][0][:, :s.o_in], model.o[l], out=b["o"][0], rms_input=True,
                         workspace=b["ws"])
                seen.append(ops.last_dispatch().split()[0])
            ops.gemm(b["y"][0], model.head, out=b["head"], argmax_out=b["argmax"],
                     rms_input=True, workspace=b["ws"])
            seen.append(ops.last_dispatch().split()[0])
        dense_calls()
        kernels = " + ".join(sorted(set(seen)))
        dense_bytes = nbytes - moe_bytes
        families["dense"] = family(f"nvfp4_gemm_skinny (QKV, O and head: {kernels}), per call",
                                   f"dense_T{t}_L{s.layers}", dense_calls, dense_bytes,
                                   2 * s.layers + 1)
    # the dominant family: the larger share of the device time
    tot_ms = sum(f["ms_per_step"] for f in families.values())
    for f in families.values():
        f["share"] = f["ms_per_step"] / tot_ms
    dom = max(families, key=lambda k: families[k]["ms_per_step"])
    roofline = dict(families[dom])
    roofline["family"] = dom
    roofline["other_families"] = {k: v for k, v in families.items() if k != dom}

    # ---- other token counts of the same step (context)
    sweep = {}
    if not args.no_sweep:
        for tt in (1, 2, 4, 8, 16, 32):
            if tt == t:
                sweep[str(tt)] = {"us_per_step": ms * 1e3, "gbs": nbytes / (ms * 1e-3) / 1e9,
                                  "weight_bytes": nbytes, "path": path}
                continue
            # both ways for the token counts around the switch, else the chosen one
            paths = ("calls", "program") if tt in (2, 4, 8, 16, 32) else (path_of(tt),)
            for pth in paths:
                _, g2, _, _, ms2, nb2, _ = one_config(tt, max(5, min(args.steps, 100)), 3, False,
                                                      pth)
                key = str(tt) if pth == path_of(tt) else f"{tt}_{pth}"
                sweep[key] = {"us_per_step": ms2 * 1e3, "gbs": nb2 / (ms2 * 1e-3) / 1e9,
                              "weight_bytes": nb2, "path": pth}
                del g2

    # ---- the other workloads of the metric (context: µs and GB/s per call)
    workloads = workload_table(model) if not args.no_sweep else None

    # ---- the same step issued call by call (one kernel per call), for context
    calls = None
    if not args.no_sweep:
        other = "calls" if path == "program" else "program"
        b3, g3, _, _, ms3, nb3, _ = one_config(t, max(5, min(args.steps, 100)), 3, False, other)
        calls = {"path": other, "us_per_step": ms3 * 1e3, "gbs": nb3 / (ms3 * 1e-3) / 1e9,
                 "launches_per_step": b3["launches"]}
        del g3

    # ---- CPU baseline: the oracle on one layer of the same step
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        sampler = OracleSample(t, x, lg)
        tot_b, tot_s = 0, 0.0
        while tot_s < 10.0 or sampler.i < len(sampler.ops):
            nb, dt = sampler.step()
            tot_b += nb
            tot_s += dt
        cpu = {"value": tot_b / tot_s / 1e9, "unit": UNIT, "cores": blas_threads(),
               "kind": "oracle",
               "sample": f"oracle float64 ops of layer 0 at T={t} (routing, QKV, O and the "
                         f"{len(sampler.ops) - 3} experts it reads), {sampler.i} ops, "
                         f"{tot_s:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "us_per_step": ms * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp16 mma (exact NVFP4 and BF16 operands), fp32 accumulate",
            "data": "synthetic",
            "config": {"workload": workload_name(t, args.layers), "tokens": t, "weight_bytes_per_step": nbytes,
                       "frac_of_8tbs": value / world / 8000.0,
                       "l2": "inputs larger than L2 (each step streams the weights once)",
                       "parallelism": f"{world} independent replica(s)"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": n_launch * args.steps, "clocks": clocks,
            "step_spread": b["spread"], "versions": versions(), "sweep": sweep,
            "path": path, "other_path": calls, "workloads": workloads,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_profile(spec, reps=4):
    """One workload's calls, ``reps`` times, then exit: the launches an ncu
    capture of that workload measures (the first is a warm-up).  Prints the
    workload's algorithmic weight bytes per call."""
    import torch
    from moe_expert_nvfp4_gb300 import ops, synth
    from moe_expert_nvfp4_gb300.decode_step import DecodeStep, StepShape, nvfp4_bytes
    ops.load()
    dev = "cuda"
    g1 = torch.full((1,), synth.GLOBAL_SCALE, dtype=torch.float32, device=dev)
    kind, *dims = spec.split(":")
    dims = [int(v) for v in dims]
    if kind in ("dense", "head"):
        n, k, m = dims if kind == "dense" else (151936, 2048, dims[0])
        w = ops.NVFP4Weight(*synth.nvfp4_weight(1, n, k, 90, device=dev), g1)
        a = synth.activations_bf16(1, m, k).to(dev)
        call = (lambda: ops.gemm(a, w, argmax=True)) if kind == "head" else (lambda: ops.gemm(a, w))
        nbytes = nvfp4_bytes(n, k)
    elif kind == "fp8":
        n, k, m = dims
        w = ops.FP8Weight(synth.fp8_weight(1, n, k).to(dev),
                          torch.full((1,), synth.FP8_SCALE, dtype=torch.float32, device=dev))
        a = synth.activations_bf16(1, m, k).to(dev)
        call = lambda: ops.fp8_gemm(a, w)
        nbytes = n * k
    elif kind == "bf16w":
        n, k, m = dims
        w = synth.bf16_weight(1, n, k).to(dev)
        a = synth.activations_bf16(1, m, k).to(dev)
        call = lambda: ops.bf16w_gemm(a, w)
        nbytes = 2 * n * k
    elif kind == "moe":
        t = dims[0]
        model = DecodeStep(seed=6, shape=StepShape(layers=1))
        s = model.s
        x = synth.activations_bf16(4, t, s.hidden).to(dev)
        ids, wts = ops.route(synth.router_logits(4, t, s.num_experts).to(dev), s.top_k)
        call = lambda: ops.moe(x, ids, wts, model.experts[0], model.shared[0])
        per_expert = nvfp4_bytes(2 * s.inter, s.hidden) + nvfp4_bytes(s.hidden, s.inter)
        nbytes = (torch.unique(ids).numel() + 1) * per_expert
    else:
        raise SystemExit(f"unknown workload {spec}")
    for _ in range(reps):
        call()
    torch.cuda.synchronize()
    print(json.dumps({"profile": spec, "weight_bytes_per_call": int(nbytes),
                      "dispatch": ops.last_dispatch()}))


def main():
    args = parse()
    if args.profile:
        run_profile(args.profile)
        return
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
