// BF16 -> NVFP4 quantisation of a weight matrix (building a 4-bit head from a
// BF16 one).
//
// "Qwen3.8-27B-NVFP4-lmhead4-recipe" (model card), section "Files": the head
// is converted from BF16 to NVFP4 by a quantisation tool; the rule is not
// given.  The rule here is the usual NVFP4 recipe:
//   g = amax / (6 * 448) over the whole matrix (1 for an all-zero matrix);
//   per 16-element block: t = amax_b / (6 g), scale byte = t rounded to E4M3
//   (nearest, ties to the even code, saturating at 448);
//   per element: v = |x| / (e4m3(scale) * g) (0 where that product is 0),
//   code = v rounded to E2M1 (nearest, ties to the even code, saturating at
//   6), with the sign bit when x < 0 and the code is not 0.
// Every quotient and product is one IEEE float32 operation rounded to
// nearest (__fdiv_rn, __fmul_rn): the codes are decided in float32.
//
// Three launches on the stream: the matrix's largest magnitude (the bits of
// |x| under atomicMax -- non-negative floats order like their bits), the
// per-block quantisation (one thread per 16-element block: two 16-byte
// loads, one 8-byte code store, one scale byte), and the per-tensor scale
// written over the maximum.  Bound by HBM: per weight 2 bytes read twice and
// 0.5625 written.
#include "common.cuh"
#include "launch.h"

namespace nvfp4 {
namespace {

constexpr int kQuantThreads = 256;

// E4M3 byte of t >= 0: nearest, ties to even, saturating at 448 (0x7E).
__device__ __forceinline__ uint32_t e4m3_rne(float t) {
  if (!(t < 448.0f)) return 0x7Eu;
  if (t < 0.015625f)  // below 2^-6: subnormal codes m * 2^-9 (t * 2^9 is exact)
    return static_cast<uint32_t>(rintf(t * 512.0f));  // 8 is the normal 2^-6
  const uint32_t bits = __float_as_uint(t);
  int e = static_cast<int>(bits >> 23) - 127;  // -6 .. 8
  uint32_t m = (bits >> 20) & 7u;              // the 3 mantissa bits kept
  const uint32_t rest = bits & 0xFFFFFu;       // the 20 dropped
  if (rest > 0x80000u || (rest == 0x80000u && (m & 1u))) ++m;
  if (m == 8u) {
    m = 0u;
    ++e;
  }
  const uint32_t code = (static_cast<uint32_t>(e + 7) << 3) | m;
  return code > 0x7Eu ? 0x7Eu : code;
}

// Value of an E4M3 byte 0 .. 0x7E (exact).
__device__ __forceinline__ float e4m3_value(uint32_t s) {
  const uint32_t e = s >> 3, m = s & 7u;
  return e == 0u ? static_cast<float>(m) * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// E2M1 code 0..7 of v >= 0: nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6; a value
// half-way between two goes to the even code; above 6 saturates.
__device__ __forceinline__ uint32_t e2m1_rne(float v) {
  return v <= 0.25f ? 0u
         : v < 0.75f ? 1u
         : v <= 1.25f ? 2u
         : v < 1.75f ? 3u
         : v <= 2.5f ? 4u
         : v < 3.5f ? 5u
         : v <= 5.0f ? 6u
                     : 7u;
}

__global__ void __launch_bounds__(kQuantThreads) amax_kernel(const QuantArgs a) {
  const long per_row = a.K / 8;  // 16-byte vectors of a row
  const long total = static_cast<long>(a.N) * per_row;
  uint32_t mx = 0u;
  for (long i = static_cast<long>(blockIdx.x) * kQuantThreads + threadIdx.x; i < total;
       i += static_cast<long>(gridDim.x) * kQuantThreads) {
    const long row = i / per_row, v = i - row * per_row;
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(a.W + row * a.ldw) + v);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) mx = max(mx, max((w[j] & 0x7FFFu) << 16, w[j] & 0x7FFF0000u));
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  if ((threadIdx.x & 31) == 0 && mx) atomicMax(a.amax_bits, mx);
}

__global__ void __launch_bounds__(kQuantThreads) quantize_kernel(const QuantArgs a) {
  const float amax = __uint_as_float(*a.amax_bits);
  const float g = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);  // 6 * 448
  const float den = __fmul_rn(6.0f, g);
  const long per_row = a.K / 16;
  const long total = static_cast<long>(a.N) * per_row;
  for (long b = static_cast<long>(blockIdx.x) * kQuantThreads + threadIdx.x; b < total;
       b += static_cast<long>(gridDim.x) * kQuantThreads) {
    const long row = b / per_row, kb = b - row * per_row;
    const uint4* src = reinterpret_cast<const uint4*>(a.W + row * a.ldw + kb * 16);
    const uint4 x0 = __ldg(src), x1 = __ldg(src + 1);
    const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    float f[16];
    float amax_b = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      f[2 * j] = __uint_as_float(w[j] << 16);
      f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      amax_b = fmaxf(amax_b, fmaxf(fabsf(f[2 * j]), fabsf(f[2 * j + 1])));
    }
    const uint32_t s = e4m3_rne(__fdiv_rn(amax_b, den));
    const float d = __fmul_rn(e4m3_value(s), g);
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      uint32_t c = d > 0.0f ? e2m1_rne(__fdiv_rn(fabsf(f[i]), d)) : 0u;
      if (f[i] < 0.0f && c) c |= 8u;
      packed[i >> 3] |= c << (4 * (i & 7));  // element 2j in byte j's low nibble
    }
    *reinterpret_cast<uint2*>(a.codes + row * (a.K / 2) + kb * 8) = make_uint2(packed[0], packed[1]);
    a.scales[row * per_row + kb] = static_cast<uint8_t>(s);
  }
}

__global__ void global_scale_kernel(const QuantArgs a) {
  const float amax = __uint_as_float(*a.amax_bits);
  *a.global_scale = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
}

}  // namespace

cudaError_t launch_quantize(const QuantArgs& a, int sms, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(a.amax_bits, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  const int grid = sms * 8;
  amax_kernel<<<grid, kQuantThreads, 0, s>>>(a);
  quantize_kernel<<<grid, kQuantThreads, 0, s>>>(a);
  global_scale_kernel<<<1, 1, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace nvfp4
