// nvfp4_gemm_skinny_noalloc: the dense skinny GEMM for callers that cannot
// allocate device memory.
//
// Some callers have no allocator to hand: a plugin inside a host runtime
// that owns every device allocation (and forbids cudaMalloc from plugins),
// code driven from a real-time loop where an allocation's latency or
// failure is not acceptable, or a process with a fixed, pre-committed
// memory budget.  nvfp4_gemm_skinny needs a caller-provided workspace; this
// entry point instead uses a scratch array that is part of the library's
// own device image, so the caller passes only inputs and outputs.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes.
// Every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address, so the first call
// on each device (made with that device current) looks the address up with
// cudaGetSymbolAddress and caches it; that first call should therefore come
// before any stream capture.  The cached address belongs to the device's
// primary context: resetting the device (cudaDeviceReset) while the library
// is loaded is not supported.  All calls share the one array and it keeps
// the previous call's contents: each call first clears, on its stream, the
// status word and tile counters that must start at zero.  Two calls that
// may run at the same time on the GPU (different streams, or graphs
// launched concurrently) race on the array and must not be issued.
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"
#include "nvfp4moe.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void* g_scratch_addr[kNoAllocMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set-up once
// per device); nullptr and *err on failure.
void* scratch_address(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kNoAllocMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int nvfp4_gemm_skinny_noalloc(const void* A, int64_t lda, int M, const nvfp4_weight* W,
                                          void* C, int64_t ldc, int32_t* argmax_out,
                                          uint32_t flags, nvfp4_stream_t stream) {
  // Every argument is checked before the shared scratch is touched: a call
  // that is going to be refused must not clear the array under a call still
  // running on another stream.
  int rc = nvfp4::check_gemm_args(A, lda, M, W, C, ldc);
  if (rc) return rc;
  // The largest need on a GB300 is the workspace header (65,792 bytes) plus
  // 32,768 bytes of split-K partials and 8 * 32 bytes of argmax partials per
  // SM: about 5.1 MB for 152 SMs, under the 8 MiB built in.
  const size_t need = nvfp4_gemm_skinny_workspace(M, W->n, W->k);
  if (need == 0) {
    nvfp4::set_last_error("nvfp4_gemm_skinny_noalloc: no plan for this shape");
    return NVFP4_ERR_SHAPE;
  }
  if (need > kNoAllocScratchBytes) {
    nvfp4::set_last_error("nvfp4_gemm_skinny_noalloc: this shape needs more than the 8 MiB "
                          "of built-in scratch; use nvfp4_gemm_skinny with a workspace");
    return NVFP4_ERR_WORKSPACE;
  }
  cudaError_t err = cudaSuccess;
  void* scratch = scratch_address(&err);
  if (!scratch) {
    nvfp4::set_last_error(cudaGetErrorString(err));
    return NVFP4_ERR_CUDA;
  }
  // status word and tile counters start at zero; the rest is overwritten
  err = cudaMemsetAsync(scratch, 0, nvfp4::kWsScratch, reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) {
    nvfp4::set_last_error(cudaGetErrorString(err));
    return NVFP4_ERR_CUDA;
  }
  return nvfp4_gemm_skinny(A, lda, M, W, C, ldc, argmax_out, flags, scratch,
                           kNoAllocScratchBytes, stream);
}
