// C-ABI entry points of libnvfp4moe.so (declared in include/nvfp4moe.h).
//
// Host side only: argument validation, the split / grid plan, TMA tensor
// maps, workspace layout, launches (with programmatic dependent launch),
// and the per-thread error and dispatch records.
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <string>

#include "nvfp4moe.h"
#include "common.cuh"
#include "launch.h"
#include "stream.cuh"

namespace {

using namespace nvfp4;

thread_local std::string g_error;
thread_local std::string g_dispatch;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(NVFP4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxDevices = 64;
constexpr size_t kSmemLimit = 232448;  // opt-in dynamic shared memory per block on sm_103

struct DevInfo {
  int checked = 0;  // 0 unknown, 1 ok, -1 wrong arch
  int sms = 0;
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Current device must be compute capability 10.3; fills *sms.
int current_device(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(NVFP4_ERR_INVALID, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.checked == 0) {
    int maj = 0, min = 0, n = 0;
    if ((e = cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.checked = (maj == 10 && min == 3) ? 1 : -1;
    d.sms = n;
  }
  if (d.checked < 0) return fail(NVFP4_ERR_ARCH, "device %d is not compute capability 10.3", dev);
  *sms = d.sms;
  return NVFP4_OK;
}

// ------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  return NVFP4_OK;
}

// uint8 matrix [rows, cols] (row stride = cols bytes) read in boxes of
// box_cols x 32 rows; codes use the 128-byte swizzle.
int make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
             bool swizzle) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {box_cols, static_cast<cuuint32_t>(kBoxRows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return NVFP4_OK;
}

int weight_maps(CUtensorMap* mc, CUtensorMap* ms, const uint8_t* codes, const uint8_t* scales,
                uint64_t rows, int k) {
  int rc = make_map(mc, codes, static_cast<uint64_t>(k) / 2, rows, kStageK / 2, true);
  if (rc) return rc;
  return make_map(ms, scales, static_cast<uint64_t>(k) / 16, rows, kStageK / 16, false);
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ------------------------------------------------------------- dense plan
struct DensePlan {
  int n_tiles, nkb, grid, mpad, win_stages, xrow_bytes;
  long units;
  size_t smem;
  size_t off_partials, off_am, ws_bytes;
};

// Stream-K: one CTA per SM (or per unit when there are fewer units), each
// with an equal contiguous range of (tile, k-stage) units; activations are
// staged in windows of at most win_stages stages.
bool plan_dense(int M, int N, int K, int sms, DensePlan* p) {
  p->n_tiles = (N + kTileRows - 1) / kTileRows;
  if (p->n_tiles > kWsMaxCounters) return false;
  p->nkb = K / kStageK;
  p->units = static_cast<long>(p->n_tiles) * p->nkb;
  p->grid = static_cast<int>(p->units < sms ? p->units : sms);
  p->mpad = (M + 7) / 8 * 8;
  const size_t x_avail = kSmemLimit - kSmemAlignPad - kSmemSched;
  int w = p->nkb;
  while (w > 1 && static_cast<size_t>(p->mpad) * xrow_stride(w * kStageK) > x_avail) --w;
  if (static_cast<size_t>(p->mpad) * xrow_stride(w * kStageK) > x_avail) return false;
  p->win_stages = w;
  p->xrow_bytes = xrow_stride(w * kStageK);
  p->smem = kSmemAlignPad + kSmemSched + static_cast<size_t>(p->mpad) * p->xrow_bytes;
  p->off_partials = kWsScratch;
  p->off_am = round_up(p->off_partials + 4ull * p->grid * 2 * M * 64, 256);
  p->ws_bytes = round_up(p->off_am + 8ull * M * p->n_tiles, 256);
  return true;
}

// ------------------------------------------------------------- MoE plan
struct MoePlan {
  int P, tpad, sched_bytes, grid_gu, grid_dn;
  int xrow_gu, xrow_dn;
  size_t smem_gu, smem_dn;
  size_t off_tile_cnt, off_h, off_y, ws_bytes;
};

bool plan_moe(int T, int k, int E, int H, int I, int sms, MoePlan* p) {
  p->P = T * k;
  p->tpad = (T + 7) / 8 * 8;
  p->sched_bytes = static_cast<int>(round_up(4ull * (4 * E + 5 + 2 * p->P + 33), 16));
  p->xrow_gu = xrow_stride(H);
  p->xrow_dn = xrow_stride(I);
  const size_t base = kSmemAlignPad + kSmemSched + p->sched_bytes;
  p->smem_gu = base + static_cast<size_t>(p->tpad + 1) * p->xrow_gu;  // + an all-zero row
  p->smem_dn = base + static_cast<size_t>(p->tpad) * p->xrow_dn;
  if (p->smem_gu > kSmemLimit || p->smem_dn > kSmemLimit) return false;
  const long max_active = (p->P < E ? p->P : E) + 1;
  const long gu_items = max_active * (I / 32), dn_items = max_active * (H / kTileRows);
  p->grid_gu = static_cast<int>(gu_items < sms ? gu_items : sms);
  p->grid_dn = static_cast<int>(dn_items < sms ? dn_items : sms);
  const size_t pairs = static_cast<size_t>(p->P + T);
  if (H / kTileRows > kWsMaxCounters) return false;
  p->off_tile_cnt = kWsCounters;
  p->off_h = kWsScratch;
  p->off_y = round_up(p->off_h + 4ull * pairs * I, 256);
  p->ws_bytes = round_up(p->off_y + 4ull * pairs * H, 256);
  return true;
}

// ------------------------------------------------------------- tcgen05 plans
// Shared memory: fixed header (barriers, misc, epilogue tile), the expert
// schedule, the staged activations [npad][win_k] f16, then as many 18 KB
// weight stages as fit (3..8).
struct TcLayout {
  int x_offset, ring_offset, n_stages;
  size_t smem;
};

bool tc_layout(int sched_bytes, size_t x_bytes, TcLayout* L) {
  L->x_offset = static_cast<int>(round_up(kTcOffSched + sched_bytes, 128));
  L->ring_offset = static_cast<int>(round_up(L->x_offset + x_bytes, 1024));
  const long room = static_cast<long>(kSmemLimit) - kSmemAlignPad - L->ring_offset;
  L->n_stages = static_cast<int>(room / kTcStageBytes);
  if (L->n_stages > kTcMaxStages) L->n_stages = kTcMaxStages;
  if (L->n_stages < 3) return false;
  L->smem = kSmemAlignPad + L->ring_offset + static_cast<size_t>(L->n_stages) * kTcStageBytes;
  return true;
}

struct TcDensePlan {
  int n_tiles, nkb, grid, npad, win_k;
  long units;
  TcLayout L;
  size_t off_partials, off_am, ws_bytes;
};

bool plan_tc_dense(int M, int N, int K, int sms, TcDensePlan* p) {
  p->n_tiles = (N + 127) / 128;
  if (p->n_tiles > kTcColCntBase) return false;
  p->nkb = K / kStageK;
  p->units = static_cast<long>(p->n_tiles) * p->nkb;
  p->grid = static_cast<int>(p->units < sms ? p->units : sms);
  p->npad = M <= 16 ? 16 : 32;
  p->win_k = K < kTcMaxWinK ? K : kTcMaxWinK;
  if (!tc_layout(0, static_cast<size_t>(p->npad) * p->win_k * 2, &p->L)) return false;
  p->off_partials = kWsScratch;
  p->off_am = round_up(p->off_partials + 4ull * p->grid * 2 * 32 * 128, 256);
  p->ws_bytes = round_up(p->off_am + 8ull * M * p->n_tiles, 256);
  return true;
}

struct TcMoePlan {
  int P, npad, sched_bytes, grid;
  TcLayout gu, dn;
  size_t off_partials, off_h, off_y, ws_bytes;
};

bool plan_tc_moe(int T, int k, int E, int H, int I, int sms, TcMoePlan* p) {
  p->P = T * k;
  p->npad = T <= 16 ? 16 : 32;
  if (H > 4096 || I > 2048) return false;  // staged rows are read once into registers
  p->sched_bytes = static_cast<int>(round_up(4ull * (4 * E + 5 + 2 * p->P + 33), 128));
  if (!tc_layout(p->sched_bytes, static_cast<size_t>(p->npad) * H * 2, &p->gu) ||
      !tc_layout(p->sched_bytes, static_cast<size_t>(p->npad) * I * 2, &p->dn))
    return false;
  const long max_active = (p->P < E ? p->P : E) + 1;
  if (max_active * (H / 128) > kTcColCntBase || H / 128 > kWsMaxCounters - kTcColCntBase) return false;
  p->grid = sms;
  const size_t pairs = static_cast<size_t>(p->P + T);
  p->off_partials = kWsScratch;
  p->off_h = round_up(p->off_partials + 4ull * p->grid * 2 * 32 * 128, 256);
  p->off_y = round_up(p->off_h + 4ull * pairs * I, 256);
  p->ws_bytes = round_up(p->off_y + 4ull * pairs * H, 256);
  return true;
}

int check_stack(const nvfp4_expert_stack* s, const char* name) {
  if (!s) return fail(NVFP4_ERR_INVALID, "%s is NULL", name);
  if (!s->gu_codes || !s->gu_scales || !s->dn_codes || !s->dn_scales || !s->gu_global ||
      !s->dn_global)
    return fail(NVFP4_ERR_INVALID, "%s has a NULL pointer", name);
  if (!aligned16(s->gu_codes) || !aligned16(s->gu_scales) || !aligned16(s->dn_codes) ||
      !aligned16(s->dn_scales))
    return fail(NVFP4_ERR_ALIGN, "%s weight pointers must be 16-byte aligned", name);
  if (s->num_experts < 1 || s->hidden < 1 || s->inter < 1)
    return fail(NVFP4_ERR_INVALID, "%s has non-positive sizes", name);
  if (s->hidden % kStageK || s->inter % kStageK)
    return fail(NVFP4_ERR_SHAPE, "%s: hidden and inter must be multiples of 256", name);
  return NVFP4_OK;
}

}  // namespace

namespace nvfp4 {
void set_last_error(const char* msg) { g_error = msg; }
}  // namespace nvfp4

// =================================================================== C ABI
extern "C" {

int nvfp4_device_check(int device) {
  int maj = 0, min = 0;
  cudaError_t e;
  if ((e = cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, device)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, device)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  if (maj != 10 || min != 3)
    return fail(NVFP4_ERR_ARCH, "device %d is compute capability %d.%d, need 10.3", device, maj,
                min);
  return NVFP4_OK;
}

int nvfp4_workspace_init(void* workspace, size_t bytes, nvfp4_stream_t stream) {
  if (!workspace || bytes == 0) return fail(NVFP4_ERR_INVALID, "workspace is empty");
  cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "cudaMemsetAsync");
}

size_t nvfp4_gemm_skinny_workspace(int M, int N, int K) {
  int sms = 0;
  if (M < 1 || M > kMaxM || N < 1 || K < kStageK || K % kStageK) return 0;
  if (current_device(&sms) != NVFP4_OK) return 0;
  DensePlan p;
  TcDensePlan t;
  const size_t a = plan_dense(M, N, K, sms, &p) ? p.ws_bytes : 0;
  const size_t b = plan_tc_dense(M, N, K, sms, &t) ? t.ws_bytes : 0;
  return a > b ? a : b;
}

int nvfp4_gemm_skinny(const void* A, int64_t lda, int M, const nvfp4_weight* W, void* C,
                      int64_t ldc, int32_t* argmax_out, uint32_t flags, void* workspace,
                      size_t workspace_bytes, nvfp4_stream_t stream) {
  if (!A || !W || !C) return fail(NVFP4_ERR_INVALID, "A, W and C must be non-NULL");
  if (!W->codes || !W->scales || !W->global_scale)
    return fail(NVFP4_ERR_INVALID, "weight has a NULL pointer");
  const int N = W->n, K = W->k;
  if (M < 1 || M > kMaxM) return fail(NVFP4_ERR_SHAPE, "M=%d outside [1, 32]", M);
  if (N < 1 || K < 1) return fail(NVFP4_ERR_INVALID, "N=%d K=%d must be positive", N, K);
  if (K % kStageK) return fail(NVFP4_ERR_SHAPE, "K=%d is not a multiple of 256", K);
  if (lda < K || ldc < N) return fail(NVFP4_ERR_INVALID, "lda < K or ldc < N");
  if (!aligned16(A) || (lda * 2) % 16 || !aligned16(W->codes) || !aligned16(W->scales))
    return fail(NVFP4_ERR_ALIGN, "A rows and weight arrays must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(C) & 1u) return fail(NVFP4_ERR_ALIGN, "C must be 2-byte aligned");
  int sms = 0;
  int rc = current_device(&sms);
  if (rc) return rc;
  if (!(flags & NVFP4_FLAG_WARP_MMA)) {
    TcDensePlan p;
    if (!plan_tc_dense(M, N, K, sms, &p))
      return fail(NVFP4_ERR_SHAPE, "N=%d, K=%d: no feasible plan", N, K);
    if (!workspace || workspace_bytes < p.ws_bytes)
      return fail(NVFP4_ERR_WORKSPACE, "workspace needs %zu bytes", p.ws_bytes);
    if ((rc = get_encoder())) return rc;
    CUtensorMap maps[4];
    if ((rc = weight_maps(&maps[0], &maps[1], W->codes, W->scales, static_cast<uint64_t>(N), K)))
      return rc;
    maps[2] = maps[0];
    maps[3] = maps[1];
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    TcArgs a = {};
    a.A = static_cast<const __nv_bfloat16*>(A);
    a.lda = lda;
    a.C = static_cast<__nv_bfloat16*>(C);
    a.ldc = ldc;
    a.argmax_out = argmax_out;
    a.gscale = W->global_scale;
    a.M = M;
    a.N = N;
    a.K = K;
    a.rms = (flags & NVFP4_FLAG_RMS_INPUT) ? 1 : 0;
    a.win_k = p.win_k;
    a.x_offset = p.L.x_offset;
    a.ring_offset = p.L.ring_offset;
    a.n_stages = p.L.n_stages;
    a.status = reinterpret_cast<uint32_t*>(ws + kWsStatus);
    a.argmax_cnt = reinterpret_cast<uint32_t*>(ws + kWsArgmaxCnt);
    a.tile_cnt = reinterpret_cast<uint32_t*>(ws + kWsCounters);
    a.partials = reinterpret_cast<float*>(ws + p.off_partials);
    a.am_part = reinterpret_cast<int2*>(ws + p.off_am);
    cudaError_t e = launch_tc(kTcDense, maps, a, p.grid, p.L.smem,
                              reinterpret_cast<cudaStream_t>(stream), !(flags & NVFP4_FLAG_NO_PDL));
    if (e != cudaSuccess) return cuda_fail(e, "stream_tc_kernel<dense> launch");
    char buf[256];
    snprintf(buf, sizeof(buf),
             "stream_tc_kernel<dense> grid=%d tiles=%d units=%ld units_per_cta=%.2f window=%d "
             "n=%d stages=%d smem=%zu argmax=%d rms=%d",
             p.grid, p.n_tiles, p.units, static_cast<double>(p.units) / p.grid, p.win_k, p.npad,
             p.L.n_stages, p.L.smem, argmax_out ? 1 : 0, a.rms);
    g_dispatch = buf;
    return NVFP4_OK;
  }
  DensePlan p;
  if (!plan_dense(M, N, K, sms, &p)) return fail(NVFP4_ERR_SHAPE, "N=%d, K=%d: no feasible plan", N, K);
  if (!workspace || workspace_bytes < p.ws_bytes)
    return fail(NVFP4_ERR_WORKSPACE, "workspace needs %zu bytes", p.ws_bytes);
  if ((rc = get_encoder())) return rc;
  CUtensorMap maps[2];
  if ((rc = weight_maps(&maps[0], &maps[1], W->codes, W->scales, static_cast<uint64_t>(N), K)))
    return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DenseArgs a = {};
  a.A = static_cast<const __nv_bfloat16*>(A);
  a.lda = lda;
  a.C = static_cast<__nv_bfloat16*>(C);
  a.ldc = ldc;
  a.argmax_out = argmax_out;
  a.gscale = W->global_scale;
  a.M = M;
  a.N = N;
  a.K = K;
  a.n_tiles = p.n_tiles;
  a.nkb = p.nkb;
  a.win_stages = p.win_stages;
  a.xrow_bytes = p.xrow_bytes;
  a.x_offset = kSmemSched;
  a.rms = (flags & NVFP4_FLAG_RMS_INPUT) ? 1 : 0;
  a.status = reinterpret_cast<uint32_t*>(ws + kWsStatus);
  a.argmax_cnt = reinterpret_cast<uint32_t*>(ws + kWsArgmaxCnt);
  a.tile_cnt = reinterpret_cast<uint32_t*>(ws + kWsCounters);
  a.partials = reinterpret_cast<float*>(ws + p.off_partials);
  a.am_part = reinterpret_cast<int2*>(ws + p.off_am);
  cudaError_t e = launch_dense(maps, a, p.grid, p.smem, reinterpret_cast<cudaStream_t>(stream),
                               !(flags & NVFP4_FLAG_NO_PDL));
  if (e != cudaSuccess) return cuda_fail(e, "dense_gemm_kernel launch");
  char buf[256];
  snprintf(buf, sizeof(buf),
           "dense_gemm_kernel grid=%d tiles=%d units=%ld units_per_cta=%.2f window=%d smem=%zu "
           "argmax=%d rms=%d",
           p.grid, p.n_tiles, p.units, static_cast<double>(p.units) / p.grid, p.win_stages,
           p.smem, argmax_out ? 1 : 0, a.rms);
  g_dispatch = buf;
  return NVFP4_OK;
}

int topk_softmax_route(const float* logits, int T, int E, int k, int renormalize,
                       int32_t* topk_ids, float* topk_w, nvfp4_stream_t stream) {
  if (!logits || !topk_ids || !topk_w) return fail(NVFP4_ERR_INVALID, "NULL pointer");
  if (T < 1 || E < 1 || k < 1) return fail(NVFP4_ERR_INVALID, "T, E, k must be positive");
  if (k > E) return fail(NVFP4_ERR_INVALID, "k=%d > E=%d", k, E);
  if (E > 512 || k > 32) return fail(NVFP4_ERR_SHAPE, "need E <= 512 and k <= 32");
  int sms = 0;
  int rc = current_device(&sms);
  if (rc) return rc;
  RouteArgs a = {logits, T, E, k, renormalize ? 1 : 0, topk_ids, topk_w};
  cudaError_t e = launch_route(a, reinterpret_cast<cudaStream_t>(stream), true);
  if (e != cudaSuccess) return cuda_fail(e, "route_kernel launch");
  char buf[128];
  snprintf(buf, sizeof(buf), "route_kernel grid=%d T=%d E=%d k=%d", (T + 3) / 4, T, E, k);
  g_dispatch = buf;
  return NVFP4_OK;
}

size_t moe_nvfp4_decode_workspace(int T, int k, const nvfp4_expert_stack* experts) {
  int sms = 0;
  if (!experts || T < 1 || T > kMaxM || k < 1 || k > 16) return 0;
  if (current_device(&sms) != NVFP4_OK) return 0;
  MoePlan p;
  TcMoePlan t;
  const size_t a = plan_moe(T, k, experts->num_experts, experts->hidden, experts->inter, sms, &p)
                       ? p.ws_bytes : 0;
  const size_t b = plan_tc_moe(T, k, experts->num_experts, experts->hidden, experts->inter, sms, &t)
                       ? t.ws_bytes : 0;
  return a > b ? a : b;
}

int moe_nvfp4_decode(const void* x, int64_t ldx, int T, const int32_t* topk_ids,
                     const float* topk_w, int k, const nvfp4_expert_stack* experts,
                     const nvfp4_expert_stack* shared, void* out, int64_t ldo, uint32_t flags,
                     void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  if (!x || !topk_ids || !topk_w || !out) return fail(NVFP4_ERR_INVALID, "NULL pointer");
  int rc = check_stack(experts, "experts");
  if (rc) return rc;
  if (shared) {
    if ((rc = check_stack(shared, "shared"))) return rc;
    if (shared->num_experts != 1 || shared->hidden != experts->hidden ||
        shared->inter != experts->inter)
      return fail(NVFP4_ERR_INVALID, "shared must be one expert of the same shape");
  }
  const int E = experts->num_experts, H = experts->hidden, I = experts->inter;
  if (T < 1 || T > kMaxM) return fail(NVFP4_ERR_SHAPE, "T=%d outside [1, 32]", T);
  if (k < 1 || k > 16 || k > E) return fail(NVFP4_ERR_SHAPE, "need 1 <= k <= min(16, E)");
  if (E > 512) return fail(NVFP4_ERR_SHAPE, "E=%d > 512", E);
  if (ldx < H || ldo < H) return fail(NVFP4_ERR_INVALID, "ldx and ldo must be >= hidden");
  if (!aligned16(x) || (ldx * 2) % 16) return fail(NVFP4_ERR_ALIGN, "x rows must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(out) & 1u) return fail(NVFP4_ERR_ALIGN, "out must be 2-byte aligned");
  int sms = 0;
  if ((rc = current_device(&sms))) return rc;
  if (!(flags & NVFP4_FLAG_WARP_MMA)) {
    TcMoePlan p;
    if (!plan_tc_moe(T, k, E, H, I, sms, &p))
      return fail(NVFP4_ERR_SHAPE, "T=%d, H=%d, E=%d: staged activations exceed shared memory",
                  T, H, E);
    if (!workspace || workspace_bytes < p.ws_bytes)
      return fail(NVFP4_ERR_WORKSPACE, "workspace needs %zu bytes", p.ws_bytes);
    if ((rc = get_encoder())) return rc;
    const nvfp4_expert_stack* sh = shared ? shared : experts;
    CUtensorMap gu[4], dn[4];
    if ((rc = weight_maps(&gu[0], &gu[1], experts->gu_codes, experts->gu_scales,
                          2ull * I * E, H)) ||
        (rc = weight_maps(&gu[2], &gu[3], sh->gu_codes, sh->gu_scales,
                          2ull * I * sh->num_experts, H)) ||
        (rc = weight_maps(&dn[0], &dn[1], experts->dn_codes, experts->dn_scales,
                          static_cast<uint64_t>(H) * E, I)) ||
        (rc = weight_maps(&dn[2], &dn[3], sh->dn_codes, sh->dn_scales,
                          static_cast<uint64_t>(H) * sh->num_experts, I)))
      return rc;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    TcArgs a = {};
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.ldx = ldx;
    a.ids = topk_ids;
    a.w = topk_w;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.ldo = ldo;
    a.gu_global = experts->gu_global;
    a.dn_global = experts->dn_global;
    a.sh_gu_global = sh->gu_global;
    a.sh_dn_global = sh->dn_global;
    a.T = T;
    a.k = k;
    a.E = E;
    a.H = H;
    a.I = I;
    a.has_shared = shared ? 1 : 0;
    a.ids_ready = (flags & NVFP4_FLAG_IDS_READY) ? 1 : 0;
    a.rms = (flags & NVFP4_FLAG_RMS_INPUT) ? 1 : 0;
    a.sched_offset = kTcOffSched;
    a.status = reinterpret_cast<uint32_t*>(ws + kWsStatus);
    a.tile_cnt = reinterpret_cast<uint32_t*>(ws + kWsCounters);
    a.partials = reinterpret_cast<float*>(ws + p.off_partials);
    a.h = reinterpret_cast<float*>(ws + p.off_h);
    a.y = reinterpret_cast<float*>(ws + p.off_y);
    const bool pdl = !(flags & NVFP4_FLAG_NO_PDL);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    a.win_k = H;
    a.x_offset = p.gu.x_offset;
    a.ring_offset = p.gu.ring_offset;
    a.n_stages = p.gu.n_stages;
    cudaError_t e = launch_tc(kTcGateUp, gu, a, p.grid, p.gu.smem, s, pdl);
    if (e != cudaSuccess) return cuda_fail(e, "stream_tc_kernel<gate_up> launch");
    a.win_k = I;
    a.x_offset = p.dn.x_offset;
    a.ring_offset = p.dn.ring_offset;
    a.n_stages = p.dn.n_stages;
    e = launch_tc(kTcDown, dn, a, p.grid, p.dn.smem, s, pdl);
    if (e != cudaSuccess) return cuda_fail(e, "stream_tc_kernel<down> launch");
    char buf[256];
    snprintf(buf, sizeof(buf),
             "stream_tc_kernel<gate_up> grid=%d stages=%d smem=%zu; stream_tc_kernel<down> grid=%d "
             "stages=%d smem=%zu; T=%d k=%d E=%d n=%d shared=%d rms=%d ids_ready=%d",
             p.grid, p.gu.n_stages, p.gu.smem, p.grid, p.dn.n_stages, p.dn.smem, T, k, E, p.npad,
             a.has_shared, a.rms, a.ids_ready);
    g_dispatch = buf;
    return NVFP4_OK;
  }
  MoePlan p;
  if (!plan_moe(T, k, E, H, I, sms, &p))
    return fail(NVFP4_ERR_SHAPE, "T=%d, H=%d: staged activations exceed shared memory", T, H);
  if (!workspace || workspace_bytes < p.ws_bytes)
    return fail(NVFP4_ERR_WORKSPACE, "workspace needs %zu bytes", p.ws_bytes);
  if ((rc = get_encoder())) return rc;
  const nvfp4_expert_stack* sh = shared ? shared : experts;
  CUtensorMap gu[4], dn[4];
  if ((rc = weight_maps(&gu[0], &gu[1], experts->gu_codes, experts->gu_scales,
                        2ull * I * E, H)) ||
      (rc = weight_maps(&gu[2], &gu[3], sh->gu_codes, sh->gu_scales, 2ull * I * sh->num_experts,
                        H)) ||
      (rc = weight_maps(&dn[0], &dn[1], experts->dn_codes, experts->dn_scales,
                        static_cast<uint64_t>(H) * E, I)) ||
      (rc = weight_maps(&dn[2], &dn[3], sh->dn_codes, sh->dn_scales,
                        static_cast<uint64_t>(H) * sh->num_experts, I)))
    return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  MoeArgs a = {};
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.ldx = ldx;
  a.ids = topk_ids;
  a.w = topk_w;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ldo = ldo;
  a.gu_global = experts->gu_global;
  a.dn_global = experts->dn_global;
  a.sh_gu_global = sh->gu_global;
  a.sh_dn_global = sh->dn_global;
  a.T = T;
  a.k = k;
  a.E = E;
  a.H = H;
  a.I = I;
  a.has_shared = shared ? 1 : 0;
  a.rms = (flags & NVFP4_FLAG_RMS_INPUT) ? 1 : 0;
  a.ids_ready = (flags & NVFP4_FLAG_IDS_READY) ? 1 : 0;
  a.x_offset = kSmemSched + p.sched_bytes;
  a.sched_offset = kSmemSched;
  a.status = reinterpret_cast<uint32_t*>(ws + kWsStatus);
  a.tile_cnt = reinterpret_cast<uint32_t*>(ws + p.off_tile_cnt);
  a.h = reinterpret_cast<float*>(ws + p.off_h);
  a.y = reinterpret_cast<float*>(ws + p.off_y);
  const bool pdl = !(flags & NVFP4_FLAG_NO_PDL);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  a.xrow_bytes = p.xrow_gu;
  cudaError_t e = launch_moe_gate_up(gu, a, p.grid_gu, p.smem_gu, s, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "moe_gate_up_kernel launch");
  a.xrow_bytes = p.xrow_dn;
  e = launch_moe_down(dn, a, p.grid_dn, p.smem_dn, s, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "moe_down_kernel launch");
  char buf[256];
  snprintf(buf, sizeof(buf),
           "moe_gate_up_kernel grid=%d smem=%zu; moe_down_kernel grid=%d smem=%zu; T=%d k=%d "
           "E=%d shared=%d rms=%d ids_ready=%d",
           p.grid_gu, p.smem_gu, p.grid_dn, p.smem_dn, T, k, E, a.has_shared, a.rms, a.ids_ready);
  g_dispatch = buf;
  return NVFP4_OK;
}

int nvfp4_read_device_status(void* workspace, uint32_t* flags, nvfp4_stream_t stream) {
  if (!workspace || !flags) return fail(NVFP4_ERR_INVALID, "NULL pointer");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(flags, workspace, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, 4, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "status read");
}

int nvfp4_last_dispatch(char* buf, size_t n) {
  if (buf && n) {
    const size_t m = g_dispatch.size() < n - 1 ? g_dispatch.size() : n - 1;
    memcpy(buf, g_dispatch.data(), m);
    buf[m] = 0;
  }
  return static_cast<int>(g_dispatch.size());
}

const char* nvfp4_last_error(void) { return g_error.c_str(); }

}  // extern "C"
