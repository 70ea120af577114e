// Read-only HBM probe: the read bandwidth a plain streaming kernel reaches
// on this GPU, the second denominator (besides a copy) for the weight
// stream's roofline fraction.  Every byte is read once with 16-byte loads
// that bypass L1, eight independent loads in flight per thread; the loaded
// words are folded with XOR into one word per CTA, written to `sink`, so no
// load can be dropped.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace nvfp4 {
namespace {

constexpr int kProbeThreads = 512;

__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const uint4* buf, size_t n16,
                                                                  uint32_t* sink) {
  uint32_t acc = 0u;
  const size_t stride = static_cast<size_t>(gridDim.x) * kProbeThreads;
  size_t i = static_cast<size_t>(blockIdx.x) * kProbeThreads + threadIdx.x;
  for (; i + 7 * stride < n16; i += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __ldcs(buf + i + j * stride);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc ^= v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = __ldcs(buf + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  __shared__ uint32_t s[kProbeThreads / 32];
  if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0u;
    for (int w = 0; w < kProbeThreads / 32; ++w) t ^= s[w];
    sink[blockIdx.x] = t;
  }
}

}  // namespace

cudaError_t launch_read_probe(const void* buf, size_t bytes, uint32_t* sink, int grid,
                              cudaStream_t s) {
  read_probe_kernel<<<grid, kProbeThreads, 0, s>>>(static_cast<const uint4*>(buf), bytes / 16,
                                                   sink);
  return cudaGetLastError();
}

}  // namespace nvfp4
