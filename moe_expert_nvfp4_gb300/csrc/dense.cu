// Dense NVFP4 skinny GEMM: C[M, N] = A[M, K] * W[N, K]^T, M <= 32.
//
// Stream-K work split: the (64-row tile, 256-K stage) units of the whole
// GEMM are cut into gridDim.x equal contiguous ranges, one per CTA, so every
// SM streams the same number of weight bytes whatever the shape.  A CTA's
// range covers the tail of one tile, whole tiles, and the head of another;
// whole tiles are stored directly, partial ones go to a per-CTA workspace
// slot and the last CTA to finish a tile (atomic counter) adds the slots in
// CTA order, so results do not depend on timing.  Activations are staged
// once per CTA when K fits in shared memory, else per window of stages,
// each window folded into the FP32 total with its own power-of-two shift.
// An optional argmax is fused the same way: per-tile (value, index)
// partials, reduced by the last tile to finish.
//
// Sources: "Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)", "Making decode
// faster" / "Skinny matrix multiplies" (split-K for 4..16-row decode
// matmuls that otherwise leave most SMs idle; 4-bit weights with 16-bit
// activations).
#include <cuda_bf16.h>
#include <float.h>

#include "launch.h"
#include "stream.cuh"

namespace nvfp4 {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// (value, index) order for argmax: larger value wins, equal values go to the
// lower index; an empty slot has index INT_MAX.
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

struct StreamK {
  long U;  // total units
  int G;
  __device__ __forceinline__ long begin(int b) const { return static_cast<long>(b) * U / G; }
  __device__ __forceinline__ int cta_of(long u) const {
    return static_cast<int>(((u + 1) * G - 1) / U);
  }
};

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

  const StreamK sk{static_cast<long>(a.n_tiles) * a.nkb, static_cast<int>(gridDim.x)};
  const int b = blockIdx.x;
  const long u0 = sk.begin(b), u1 = sk.begin(b + 1);

  if (warp == kConsumerWarps) {
    // ---------------- producer: weights never depend on the previous grid,
    // so streaming starts before the dependency wait.
    if (lane == 0) {
      prefetch_tensormap(&map_codes);
      prefetch_tensormap(&map_scales);
      const uint64_t pol = l2_policy_evict_first();
      Pipe p;
      long issued = 0;
      for (long u = u0; u < u1; ++u) {
        const int row0 = static_cast<int>(u / a.nkb) * kTileRows;
        if (!produce_stage(ring, p, &map_codes, &map_scales, row0, row0 + kBoxRows,
                           static_cast<int>(u % a.nkb), pol, a.status, abort_flag))
          break;
        ++issued;
      }
      producer_drain(ring, p, issued, a.status);
    }
    return;
  }

  // ---------------- consumers
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, cw = warp, h = cw >> 2, wg = cw & 3;
  const int ntiles = (a.M + 7) >> 3;
  const int mpad = ntiles * 8;
  const __nv_bfloat16* A = a.A;
  const int64_t lda = a.lda;
  auto rowp = [&](int q) { return A + q * lda; };
  const uint8_t* xr[4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) xr[nt] = xs + (nt * 8 + (lane >> 2)) * a.xrow_bytes;

  const bool full_k = a.win_stages >= a.nkb;
  int st0 = 0, st1 = 0;  // staged stage range [st0, st1)
  if (full_k) {
    stage_rows<__nv_bfloat16>(rowp, a.M, mpad, 0, a.K, a.K, xs, a.xrow_bytes, sig,
                              a.rms ? rms : nullptr, cw, lane);
    st1 = a.nkb;
  } else if (a.rms) {
    for (int q = cw; q < a.M; q += kConsumerWarps) {
      float ss = 0.0f;
      for (int v = lane; v < a.K / 8; v += 32) {
        const uint4 u = *reinterpret_cast<const uint4*>(rowp(q) + v * 8);
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(static_cast<float>(e[i]), static_cast<float>(e[i]), ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) rms[q] = rsqrtf(ss / static_cast<float>(a.K) + 1e-6f);
    }
  }
  consumer_sync();
  const float gs = *a.gscale;
  const int first_tile = static_cast<int>(u0 / a.nkb);

  Pipe p;
  for (long u = u0; u < u1;) {
    const int tile = static_cast<int>(u / a.nkb);
    const int kbs = static_cast<int>(u % a.nkb);
    const int kbe = static_cast<int>(min(static_cast<long>(a.nkb), kbs + (u1 - u)));
    float tot[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) tot[i][j] = 0.0f;
    for (int w0 = kbs; w0 < kbe; w0 += a.win_stages) {
      const int w1 = min(kbe, w0 + a.win_stages);
      if (w0 < st0 || w1 > st1) {
        consumer_sync();
        const int n1 = min(a.nkb, w0 + a.win_stages);
        stage_rows<__nv_bfloat16>(rowp, a.M, mpad, w0 * kStageK, (n1 - w0) * kStageK, a.K, xs,
                                  a.xrow_bytes, sig, nullptr, cw, lane);
        st0 = w0;
        st1 = n1;
        consumer_sync();
      }
      Acc acc;
      acc.zero();
      for (int kb = w0; kb < w1; ++kb) {
        if (!*abort_flag) wait_or_abort(&ring.full[p.stage], p.phase, a.status, abort_flag);
        consume_half(ring.codes(p.stage), ring.scales(p.stage), h, wg, lane, xr,
                     (kb - st0) * kStageK, ntiles, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&ring.empty[p.stage]);
        p.advance();
      }
      fold_window(acc, tot, ntiles, lane, [&](int q) { return sig[q]; });
    }
    groups_to_ep(tot, ep, ntiles, a.M, cw, lane);
    u += kbe - kbs;

    const int nval = a.M * 64;
    if (!(kbs == 0 && kbe == a.nkb)) {
      // partial tile: publish this CTA's slot; the last contributor reduces
      const int slot = (tile == first_tile) ? 0 : 1;
      float* part = a.partials + static_cast<size_t>(b * 2 + slot) * nval;
      for (int i = tid; i < nval; i += kConsumerThreads) part[i] = ep[i];
      __threadfence();
      consumer_sync();
      const int blo = sk.cta_of(static_cast<long>(tile) * a.nkb);
      const int bhi = sk.cta_of(static_cast<long>(tile + 1) * a.nkb - 1);
      if (tid == 0) {
        const uint32_t prev = atomicAdd(&a.tile_cnt[tile], 1u);
        *bcast = (prev == static_cast<uint32_t>(bhi - blo)) ? 1 : 0;
      }
      consumer_sync();
      if (!*bcast) continue;  // uniform across the consumer warps
      __threadfence();
      for (int i = tid; i < nval; i += kConsumerThreads) {
        float s = 0.0f;
        for (int bb = blo; bb <= bhi; ++bb) {
          const int sl = (sk.begin(bb) / a.nkb == tile) ? 0 : 1;
          s += __ldcg(a.partials + static_cast<size_t>(bb * 2 + sl) * nval + i);
        }
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
        const __nv_bfloat16 bv = __float2bfloat16_rn(v);
        a.C[m * a.ldc + n] = bv;
        ep[i] = __bfloat162float(bv);
      } else {
        ep[i] = -FLT_MAX;
      }
    }
    if (a.argmax_out) {
      consumer_sync();
      for (int m = cw; m < a.M; m += kConsumerWarps) {
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
        for (int m = cw; m < a.M; m += kConsumerWarps) {
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
          if (lane == 0) a.argmax_out[m] = (a.am_map && bi != 0x7fffffff) ? a.am_map[bi] : bi;
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
