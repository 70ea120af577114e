// Row gather of an NVFP4 matrix: building the hot-vocabulary head.
//
// "Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)", section "Making decode
// faster", paragraph "FR-Spec, and a silent bug": the draft scores only a
// list of the most likely tokens (32K of the vocabulary) through a 4-bit
// head built from the checkpoint's own output head, 37 MB a draft step
// instead of 290 MB.  In the plain row-major NVFP4 layout a row's codes
// (K/2 bytes) and its scales (K/16 bytes) are each contiguous, so the hot
// head is those rows copied in list order (the pages' failure was slicing
// rows out of a head repacked for another kernel, whose rows are not
// contiguous).  Done once, when the list is built.
//
// One warp per output row, 16-byte copies (K % 256 == 0: a code row is a
// multiple of 128 bytes, a scale row of 16).  A row id outside [0, N) gives
// an all-zero row (every weight 0).  Bound by HBM: n_rows * (K/2 + K/16)
// bytes read and as many written.
#include "common.cuh"
#include "launch.h"

namespace nvfp4 {
namespace {

constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(kGatherWarps * 32) gather_rows_kernel(const GatherArgs a) {
  const int lane = threadIdx.x & 31;
  const long row = static_cast<long>(blockIdx.x) * kGatherWarps + (threadIdx.x >> 5);
  if (row >= a.n_rows) return;
  const int src = a.rows[row];
  const bool ok = src >= 0 && src < a.N;
  const size_t code_row = static_cast<size_t>(a.K) / 2, scale_row = static_cast<size_t>(a.K) / 16;
  const int cv = static_cast<int>(code_row / 16), sv = static_cast<int>(scale_row / 16);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const uint4* sc = reinterpret_cast<const uint4*>(a.src_codes + (ok ? src * code_row : 0));
  const uint4* ss = reinterpret_cast<const uint4*>(a.src_scales + (ok ? src * scale_row : 0));
  uint4* dc = reinterpret_cast<uint4*>(a.dst_codes + row * code_row);
  uint4* ds = reinterpret_cast<uint4*>(a.dst_scales + row * scale_row);
  for (int i = lane; i < cv; i += 32) dc[i] = ok ? __ldg(sc + i) : zero;
  for (int i = lane; i < sv; i += 32) ds[i] = ok ? __ldg(ss + i) : zero;
}

}  // namespace

cudaError_t launch_gather_rows(const GatherArgs& a, cudaStream_t s) {
  const long blocks = (static_cast<long>(a.n_rows) + kGatherWarps - 1) / kGatherWarps;
  gather_rows_kernel<<<static_cast<unsigned>(blocks), kGatherWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace nvfp4
