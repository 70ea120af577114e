// Dense NVFP4 skinny GEMM: C[M, N] = A[M, K] * W[N, K]^T, M <= 32.
//
// Work item = (64-row tile of W, K split).  A persistent grid of at most one
// CTA per SM walks items with stride gridDim.x; gridDim.x is a multiple of
// the split count, so each CTA keeps one K slice and stages its slice of A
// once.  Split partial sums go to the workspace; the last CTA to finish a
// tile (atomic counter) adds them in split order, so results do not depend
// on timing.  An optional argmax is fused the same way: per-tile (value,
// index) partials, reduced by the last tile to finish.
//
// Sources: "Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)", "Making decode
// faster" / "Skinny matrix multiplies" (split-K for 4..16-row decode
// matmuls; 4-bit weights with 16-bit activations).
#include <cuda_bf16.h>
#include <float.h>

#include "launch.h"
#include "stream.cuh"

namespace nvfp4 {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// (value, index) pair order for argmax: larger value wins, equal values go
// to the lower index; an empty slot has index INT_MAX.
__device__ __forceinline__ bool am_better(float v, int i, float bv, int bi) {
  return bi == 0x7fffffff || v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void am_warp_reduce(float& bv, int& bi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (oi != 0x7fffffff && am_better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    dense_gemm_kernel(const __grid_constant__ CUtensorMap map_codes,
                      const __grid_constant__ CUtensorMap map_scales, const DenseArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Ring ring{smem + kSmemRing, reinterpret_cast<uint64_t*>(smem + kSmemBars),
            reinterpret_cast<uint64_t*>(smem + kSmemBars) + kStages};
  int* sig = reinterpret_cast<int*>(smem + kSmemMisc);
  float* rms = reinterpret_cast<float*>(smem + kSmemMisc + 128);
  volatile int* abort_flag = reinterpret_cast<int*>(smem + kSmemMisc + 256);
  volatile int* bcast = reinterpret_cast<int*>(smem + kSmemMisc + 260);
  float* ep = reinterpret_cast<float*>(smem + kSmemEp);
  uint8_t* xs = smem + a.x_offset;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ring_init(ring);
    *abort_flag = 0;
  }
  __syncthreads();

  const int G = gridDim.x;
  const int split = blockIdx.x % a.splits;
  const int kb0 = split * a.nkb / a.splits;
  const int kb1 = (split + 1) * a.nkb / a.splits;

  if (warp == kConsumerWarps) {
    // ---------------- producer: weights never depend on the previous grid,
    // so streaming starts before the dependency wait.
    if (lane == 0) {
      prefetch_tensormap(&map_codes);
      prefetch_tensormap(&map_scales);
      const uint64_t pol = l2_policy_evict_first();
      Pipe p;
      long issued = 0;
      for (int it = blockIdx.x; it < a.items; it += G) {
        const int row0 = (it / a.splits) * kTileRows;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!produce_stage(ring, p, &map_codes, &map_scales, row0, row0 + kBoxRows, kb, pol,
                             a.status, abort_flag))
            goto drained;
          ++issued;
        }
      }
    drained:
      producer_drain(ring, p, issued, a.status);
    }
    return;
  }

  // ---------------- consumers
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  const int ntiles = (a.M + 7) >> 3;
  const int klen = (kb1 - kb0) * kStageK;
  const __nv_bfloat16* A = a.A;
  const int64_t lda = a.lda;
  stage_rows<__nv_bfloat16>([&](int q) { return A + q * lda; }, a.M, ntiles * 8, kb0 * kStageK,
                            klen, a.K, xs, a.xrow_bytes, sig, a.rms ? rms : nullptr, warp, lane);
  consumer_sync();
  const float gs = *a.gscale;

  Pipe p;
  for (int it = blockIdx.x; it < a.items; it += G) {
    const int tile = it / a.splits;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!*abort_flag) wait_or_abort(&ring.full[p.stage], p.phase, a.status, abort_flag);
      consume_stage(ring.codes(p.stage), ring.scales(p.stage), xs, a.xrow_bytes,
                    (kb - kb0) * kStageK, warp, lane, ntiles, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&ring.empty[p.stage]);
      p.advance();
    }

    // accumulators -> ep[m][row], undoing the FP16 staging shift
    int R0, R1, c0;
    acc_coords(warp, lane, R0, R1, c0);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      if (nt < ntiles) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int m = nt * 8 + c0 + (e & 1);
          const int R = (e < 2) ? R0 : R1;
          if (m < a.M) ep[m * 64 + R] = scale_pow2(acc[nt][e], -sig[m]);
        }
      }
    }
    consumer_sync();

    const int nval = a.M * 64;
    if (a.splits > 1) {
      float* part = a.partials + (static_cast<size_t>(split) * a.n_tiles + tile) * nval;
      for (int i = tid; i < nval; i += kConsumerThreads) part[i] = ep[i];
      __threadfence();
      consumer_sync();
      if (tid == 0) {
        const uint32_t prev = atomicAdd(&a.tile_cnt[tile], 1u);
        *bcast = (prev == static_cast<uint32_t>(a.splits - 1)) ? 1 : 0;
      }
      consumer_sync();
      if (!*bcast) continue;  // uniform across the consumer warps
      __threadfence();
      for (int i = tid; i < nval; i += kConsumerThreads) {
        float s = 0.0f;
        for (int sp = 0; sp < a.splits; ++sp)
          s += __ldcg(a.partials + (static_cast<size_t>(sp) * a.n_tiles + tile) * nval + i);
        ep[i] = s;
      }
      if (tid == 0) a.tile_cnt[tile] = 0u;
      consumer_sync();
    }

    // final values: x global scale (x RMS factor) -> BF16, coalesced rows
    for (int i = tid; i < nval; i += kConsumerThreads) {
      const int m = i >> 6, R = i & 63;
      const int n = tile * kTileRows + R;
      if (n < a.N) {
        float v = ep[i] * gs;
        if (a.rms) v *= rms[m];
        const __nv_bfloat16 b = __float2bfloat16_rn(v);
        a.C[m * a.ldc + n] = b;
        ep[i] = __bfloat162float(b);
      } else {
        ep[i] = -FLT_MAX;
      }
    }
    if (a.argmax_out) {
      consumer_sync();
      for (int m = warp; m < a.M; m += kConsumerWarps) {
        float bv = -FLT_MAX;
        int bi = 0x7fffffff;
        const int n0 = tile * kTileRows;
        if (n0 + lane < a.N) {
          bv = ep[m * 64 + lane];
          bi = n0 + lane;
        }
        if (n0 + lane + 32 < a.N && am_better(ep[m * 64 + lane + 32], n0 + lane + 32, bv, bi)) {
          bv = ep[m * 64 + lane + 32];
          bi = n0 + lane + 32;
        }
        am_warp_reduce(bv, bi);
        if (lane == 0) a.am_part[m * a.n_tiles + tile] = make_int2(__float_as_int(bv), bi);
      }
      __threadfence();
      consumer_sync();
      if (tid == 0) {
        const uint32_t prev = atomicAdd(a.argmax_cnt, 1u);
        *bcast = (prev == static_cast<uint32_t>(a.n_tiles - 1)) ? 1 : 0;
      }
      consumer_sync();
      if (*bcast) {
        __threadfence();
        for (int m = warp; m < a.M; m += kConsumerWarps) {
          float bv = -FLT_MAX;
          int bi = 0x7fffffff;
          for (int j = lane; j < a.n_tiles; j += 32) {
            const int2 pr = __ldcg(a.am_part + m * a.n_tiles + j);
            const float v = __int_as_float(pr.x);
            if (pr.y != 0x7fffffff && am_better(v, pr.y, bv, bi)) {
              bv = v;
              bi = pr.y;
            }
          }
          am_warp_reduce(bv, bi);
          if (lane == 0) a.argmax_out[m] = bi;
        }
        if (tid == 0) *a.argmax_cnt = 0u;
      }
    }
    consumer_sync();
  }
}

cudaError_t launch_dense(const CUtensorMap* maps, const DenseArgs& a, int grid, size_t smem,
                         cudaStream_t s, bool pdl) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(dense_gemm_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
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
  return cudaLaunchKernelEx(&cfg, dense_gemm_kernel, maps[0], maps[1], a);
}

}  // namespace nvfp4
