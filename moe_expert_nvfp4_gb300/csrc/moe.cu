// Top-k routed NVFP4 MoE decode layer with an always-on shared expert.
//
//   gate_up kernel: for every active expert e and every 32-wide block j of
//     the intermediate dimension, one work item streams gate rows
//     [32j, 32j+32) and up rows [I+32j, I+32j+32) over the full hidden K,
//     against the FP16-staged activations of the tokens routed to e, and
//     writes h = silu(gate) * up (FP32) for each (token, slot) pair.
//   down kernel: for every active expert and 64-row tile of the down matrix,
//     one item computes the expert's down output for its pairs (FP32); the
//     last item to finish a tile column (atomic counter) combines
//     out[t] = sum_j w[t][j] * y[pair(t, j)] + y[shared pair(t)] in slot
//     order and writes BF16.
//   Both kernels rebuild the same schedule from the ids in every CTA: expert
//   histogram, exclusive offsets, the ascending list of active experts (the
//   shared expert is id E, last), and for every flat slot t*k+j its pair
//   index = offset[id] + number of earlier slots with the same id.  Only
//   active experts' weights are streamed.
//
// Sources: "Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)", "Making decode
// faster" / "One environment variable" (the fused MoE finalize: weighted
// combine of the top-k expert outputs) and "What didn't work" (the shared
// expert kept as its own always-on expert).
#include <cuda_bf16.h>

#include "launch.h"
#include "sched.cuh"
#include "stream.cuh"

namespace nvfp4 {

__device__ __forceinline__ uint8_t* align1024m(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

struct MoeSmem {
  Ring ring;
  int* sig;
  float* rms;
  volatile int* abort_flag;
  volatile int* bcast;
  float* ep;
  uint8_t* xs;
  Sched sched;
};

__device__ __forceinline__ MoeSmem moe_smem(uint8_t* smem_raw, const MoeArgs& a) {
  uint8_t* smem = align1024m(smem_raw);
  MoeSmem m;
  m.ring = Ring{smem + kSmemRing, reinterpret_cast<uint64_t*>(smem + kSmemBars),
                reinterpret_cast<uint64_t*>(smem + kSmemBars) + kStages};
  m.sig = reinterpret_cast<int*>(smem + kSmemMisc);
  m.rms = reinterpret_cast<float*>(smem + kSmemMisc + 128);
  m.abort_flag = reinterpret_cast<int*>(smem + kSmemMisc + 256);
  m.bcast = reinterpret_cast<int*>(smem + kSmemMisc + 260);
  m.ep = reinterpret_cast<float*>(smem + kSmemEp);
  m.xs = smem + a.x_offset;
  m.sched = sched_layout(smem + a.sched_offset, a.E, a.T * a.k);
  return m;
}

// ---------------------------------------------------------------- gate_up
// Items: (active expert a, 32-wide block jb of the intermediate dimension).
// All T tokens are staged once per CTA; an item's MMA columns gather the
// staged rows of the tokens routed to its expert.
__global__ void __launch_bounds__(kThreads, 1)
    moe_gate_up_kernel(const __grid_constant__ CUtensorMap gu_codes,
                       const __grid_constant__ CUtensorMap gu_scales,
                       const __grid_constant__ CUtensorMap sh_codes,
                       const __grid_constant__ CUtensorMap sh_scales, const MoeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const MoeSmem S = moe_smem(smem_raw, a);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ring_init(S.ring);
    *S.abort_flag = 0;
  }
  // ids written before the previous kernel started may be read before the
  // dependency wait, so the weight stream can start during its tail
  if (!a.ids_ready) pdl_wait();
  build_schedule(a.ids, a.T, a.k, a.E, a.has_shared, S.sched, a.status);

  const int G = gridDim.x;
  const int per_e = a.I / 32;
  const int items = *S.sched.n_active * per_e;
  const int nkb = a.H / kStageK;

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      Pipe p;
      long issued = 0;
      for (int it = blockIdx.x; it < items; it += G) {
        const int e = S.sched.active[it / per_e];
        const int jb = it % per_e;
        const bool sh = (e == a.E);
        const CUtensorMap* mc = sh ? &sh_codes : &gu_codes;
        const CUtensorMap* ms = sh ? &sh_scales : &gu_scales;
        const int base = sh ? 0 : e * 2 * a.I;
        const int row0 = base + jb * 32, row1 = base + a.I + jb * 32;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!produce_stage(S.ring, p, mc, ms, row0, row1, kb, pol, a.status, S.abort_flag))
            goto drained;
          ++issued;
        }
      }
    drained:
      producer_drain(S.ring, p, issued, a.status);
    }
    return;
  }

  // ---------------- consumers
  if (a.ids_ready) pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, cw = warp, h = cw >> 2, wg = cw & 3;
  const int tpad = (a.T + 7) & ~7;
  const __nv_bfloat16* X = a.x;
  const int64_t ldx = a.ldx;
  // rows [0, tpad) hold the tokens (zeros past T); row tpad is all zeros
  stage_rows<__nv_bfloat16>([&](int q) { return X + q * ldx; }, a.T, tpad + 1, 0, a.H, a.H,
                            S.xs, a.xrow_bytes, S.sig, a.rms ? S.rms : nullptr, cw, lane);
  consumer_sync();
  const uint8_t* zero_row = S.xs + tpad * a.xrow_bytes;

  Pipe p;
  for (int it = blockIdx.x; it < items; it += G) {
    const int e = S.sched.active[it / per_e];
    const int jb = it % per_e;
    const int cnt = S.sched.cnt[e];
    const int* tok = S.sched.pair_tok + S.sched.off[e];
    const int ntiles = (cnt + 7) >> 3;
    const uint8_t* xr[4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int q = nt * 8 + (lane >> 2);
      xr[nt] = (q < cnt) ? S.xs + tok[q] * a.xrow_bytes : zero_row;
    }
    Acc acc;
    acc.zero();
    for (int kb = 0; kb < nkb; ++kb) {
      if (!*S.abort_flag) wait_or_abort(&S.ring.full[p.stage], p.phase, a.status, S.abort_flag);
      consume_half(S.ring.codes(p.stage), S.ring.scales(p.stage), h, wg, lane, xr, kb * kStageK,
                   ntiles, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.ring.empty[p.stage]);
      p.advance();
    }
    float tot[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) tot[i][j] = 0.0f;
    fold_window(acc, tot, ntiles, lane, [&](int q) { return q < cnt ? S.sig[tok[q]] : 0; });
    groups_to_ep(tot, S.ep, ntiles, cnt, cw, lane);
    // tile rows [0, 32) are gate j = 32jb + r, rows [32, 64) the matching up
    const float g = (e == a.E) ? *a.sh_gu_global : a.gu_global[e];
    const int off = S.sched.off[e];
    for (int i = tid; i < cnt * 32; i += kConsumerThreads) {
      const int q = i >> 5, r = i & 31;
      const float f = a.rms ? g * S.rms[tok[q]] : g;
      const float gt = S.ep[q * 64 + r] * f;
      const float up = S.ep[q * 64 + 32 + r] * f;
      a.h[static_cast<size_t>(off + q) * a.I + jb * 32 + r] = gt / (1.0f + expf(-gt)) * up;
    }
    consumer_sync();
  }
}

// ---------------------------------------------------------------- down + combine
// Items: (active expert a, group of m consecutive 64-row tiles), m chosen
// from the number of active experts so that there are about two items per
// CTA.  The expert's h rows are staged once per item.
__device__ __forceinline__ int down_group(int n_active, int tiles_per_e, int grid) {
  int m = 8;
  while (m > 1 && (tiles_per_e % m != 0 || n_active * (tiles_per_e / m) < 2 * grid)) m >>= 1;
  return m;
}

__global__ void __launch_bounds__(kThreads, 1)
    moe_down_kernel(const __grid_constant__ CUtensorMap dn_codes,
                    const __grid_constant__ CUtensorMap dn_scales,
                    const __grid_constant__ CUtensorMap sh_codes,
                    const __grid_constant__ CUtensorMap sh_scales, const MoeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const MoeSmem S = moe_smem(smem_raw, a);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ring_init(S.ring);
    *S.abort_flag = 0;
  }
  // The ids are complete here: the gate_up grid before this one read them
  // after its own dependency wait and only then allowed this grid to start.
  build_schedule(a.ids, a.T, a.k, a.E, a.has_shared, S.sched, a.status);

  const int G = gridDim.x;
  const int tiles_per_e = a.H / kTileRows;
  const int n_active = *S.sched.n_active;
  const int m = down_group(n_active, tiles_per_e, G);
  const int per_e = tiles_per_e / m;
  const int items = n_active * per_e;
  const int nkb = a.I / kStageK;

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      Pipe p;
      long issued = 0;
      for (int it = blockIdx.x; it < items; it += G) {
        const int e = S.sched.active[it / per_e];
        const bool sh = (e == a.E);
        const CUtensorMap* mc = sh ? &sh_codes : &dn_codes;
        const CUtensorMap* ms = sh ? &sh_scales : &dn_scales;
        const int row_base = (sh ? 0 : e * a.H) + (it % per_e) * m * kTileRows;
        for (int ti = 0; ti < m; ++ti)
          for (int kb = 0; kb < nkb; ++kb) {
            const int row0 = row_base + ti * kTileRows;
            if (!produce_stage(S.ring, p, mc, ms, row0, row0 + kBoxRows, kb, pol, a.status,
                               S.abort_flag))
              goto drained;
            ++issued;
          }
      }
    drained:
      producer_drain(S.ring, p, issued, a.status);
    }
    return;
  }

  pdl_wait();  // h comes from the gate_up grid
  pdl_launch_dependents();
  const int tid = threadIdx.x, cw = warp, h = cw >> 2, wg = cw & 3;
  if (items == 0 && blockIdx.x == 0) {
    // nothing routed and no shared expert: the layer output is zero
    for (int i = tid; i < a.T * a.H; i += kConsumerThreads)
      a.out[(i / a.H) * a.ldo + (i % a.H)] = __float2bfloat16_rn(0.0f);
  }
  Pipe p;
  for (int it = blockIdx.x; it < items; it += G) {
    const int e = S.sched.active[it / per_e];
    const int cnt = S.sched.cnt[e];
    const int off = S.sched.off[e];
    const int ntiles = (cnt + 7) >> 3;
    const float* Hs = a.h;
    const int I = a.I;
    consumer_sync();  // the previous item is done with the staged rows
    stage_rows<float>([&](int q) { return Hs + static_cast<size_t>(off + q) * I; }, cnt,
                      ntiles * 8, 0, a.I, a.I, S.xs, a.xrow_bytes, S.sig, nullptr, cw, lane);
    consumer_sync();
    const uint8_t* xr[4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) xr[nt] = S.xs + (nt * 8 + (lane >> 2)) * a.xrow_bytes;
    const float g = (e == a.E) ? *a.sh_dn_global : a.dn_global[e];
    for (int ti = 0; ti < m; ++ti) {
      const int nt_tile = (it % per_e) * m + ti;
      Acc acc;
      acc.zero();
      for (int kb = 0; kb < nkb; ++kb) {
        if (!*S.abort_flag) wait_or_abort(&S.ring.full[p.stage], p.phase, a.status, S.abort_flag);
        consume_half(S.ring.codes(p.stage), S.ring.scales(p.stage), h, wg, lane, xr,
                     kb * kStageK, ntiles, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.ring.empty[p.stage]);
        p.advance();
      }
      float tot[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) tot[i][j] = 0.0f;
      fold_window(acc, tot, ntiles, lane, [&](int q) { return S.sig[q]; });
      groups_to_ep(tot, S.ep, ntiles, cnt, cw, lane);
      for (int i = tid; i < cnt * 64; i += kConsumerThreads) {
        const int q = i >> 6, r = i & 63;
        a.y[static_cast<size_t>(off + q) * a.H + nt_tile * kTileRows + r] = S.ep[i] * g;
      }
      __threadfence();
      consumer_sync();
      if (tid == 0) {
        const uint32_t prev = atomicAdd(&a.tile_cnt[nt_tile], 1u);
        *S.bcast = (prev == static_cast<uint32_t>(n_active - 1)) ? 1 : 0;
      }
      consumer_sync();
      if (*S.bcast) {
        // last expert to finish this tile column: weighted combine in slot order
        __threadfence();
        const int* fp = S.sched.flat_pair;
        const int sh_off = S.sched.off[a.E];
        for (int i = tid; i < a.T * 64; i += kConsumerThreads) {
          const int t = i >> 6, r = i & 63;
          const int n = nt_tile * kTileRows + r;
          float s = 0.0f;
          for (int j = 0; j < a.k; ++j) {
            const int pr = fp[t * a.k + j];
            if (pr >= 0)
              s = fmaf(a.w[t * a.k + j], __ldcg(a.y + static_cast<size_t>(pr) * a.H + n), s);
          }
          if (a.has_shared) s += __ldcg(a.y + static_cast<size_t>(sh_off + t) * a.H + n);
          a.out[t * a.ldo + n] = __float2bfloat16_rn(s);
        }
        if (tid == 0) a.tile_cnt[nt_tile] = 0u;
      }
      consumer_sync();
    }
  }
}

template <typename K>
static cudaError_t launch4(K kernel, const CUtensorMap* maps, const MoeArgs& a, int grid,
                           size_t smem, cudaStream_t s, bool pdl, bool& attr_set) {
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, maps[0], maps[1], maps[2], maps[3], a);
}

cudaError_t launch_moe_gate_up(const CUtensorMap* maps, const MoeArgs& a, int grid, size_t smem,
                               cudaStream_t s, bool pdl) {
  static bool attr_set = false;
  return launch4(moe_gate_up_kernel, maps, a, grid, smem, s, pdl, attr_set);
}

cudaError_t launch_moe_down(const CUtensorMap* maps, const MoeArgs& a, int grid, size_t smem,
                            cudaStream_t s, bool pdl) {
  static bool attr_set = false;
  return launch4(moe_down_kernel, maps, a, grid, smem, s, pdl, attr_set);
}

}  // namespace nvfp4
