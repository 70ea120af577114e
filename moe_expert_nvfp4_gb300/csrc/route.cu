// Top-k softmax routing: one warp per token row.
//
// The k largest logits are selected by comparing the float32 logits
// (ties to the lower expert index) in k rounds of a warp-wide arg-max, and
// listed in selection order.  Weights are exp(l - l_max) normalised over the
// chosen k (renormalised) or over all E experts.  Logits are read once; E <=
// 512 fits in 16 registers per lane.
#include <float.h>

#include "common.cuh"
#include "launch.h"

namespace nvfp4 {

constexpr int kRouteWarps = 4;
constexpr int kMaxPerLane = 16;  // E <= 512
constexpr int kMaxK = 32;

__device__ __forceinline__ bool rt_better(float v, int i, float bv, int bi) {
  return bi == 0x7fffffff || v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(const RouteArgs a) {
  __shared__ float sel_v[kRouteWarps][kMaxK];
  __shared__ int sel_i[kRouteWarps][kMaxK];
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRouteWarps + warp;
  if (row >= a.T) return;
  const float* l = a.logits + static_cast<size_t>(row) * a.E;
  float v[kMaxPerLane];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < a.E) ? l[e] : -FLT_MAX;
    if (e >= a.E) taken |= 1u << i;
  }
  for (int r = 0; r < a.k; ++r) {
    float bv = -FLT_MAX;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
      if (!(taken >> i & 1u) && rt_better(v[i], lane + 32 * i, bv, bi)) {
        bv = v[i];
        bi = lane + 32 * i;
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi != 0x7fffffff && rt_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi != 0x7fffffff && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == 0) {
      sel_v[warp][r] = bv;
      sel_i[warp][r] = bi;
    }
  }
  __syncwarp();
  const float lmax = sel_v[warp][0];
  float den;
  if (a.renorm) {
    float s = 0.0f;
    for (int r = lane; r < a.k; r += 32) s += expf(sel_v[warp][r] - lmax);
    den = warp_sum(s);
  } else {
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
      if (lane + 32 * i < a.E) s += expf(v[i] - lmax);
    den = warp_sum(s);
  }
  for (int r = lane; r < a.k; r += 32) {
    a.ids[static_cast<size_t>(row) * a.k + r] = sel_i[warp][r];
    a.w[static_cast<size_t>(row) * a.k + r] = expf(sel_v[warp][r] - lmax) / den;
  }
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.T + kRouteWarps - 1) / kRouteWarps);
  cfg.blockDim = dim3(kRouteWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, route_kernel, a);
}

}  // namespace nvfp4
