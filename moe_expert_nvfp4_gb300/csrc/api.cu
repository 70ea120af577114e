// C-ABI entry points of libnvfp4moe.so (declared in include/nvfp4moe.h).
//
// Host side only: argument validation, the split / grid plan, TMA tensor
// maps, workspace layout, launches (with programmatic dependent launch),
// and the per-thread error and dispatch records.
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdlib.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "nvfp4moe.h"
#include "common.cuh"
#include "launch.h"

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
constexpr size_t kSmemAlignPad = 1024;  // the kernel aligns its shared-memory base to 1024 bytes

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
// box_cols x box_rows; codes use the 128-byte swizzle.
int make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
             bool swizzle, uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return NVFP4_OK;
}

// Codes and scales of a weight, one 256-K stage wide; boxes of box_rows rows
// (128: one whole tile).
int weight_maps(CUtensorMap* mc, CUtensorMap* ms, const uint8_t* codes, const uint8_t* scales,
                uint64_t rows, int k, uint32_t box_rows) {
  int rc = make_map(mc, codes, static_cast<uint64_t>(k) / 2, rows, kStageK / 2, true, box_rows);
  if (rc) return rc;
  return make_map(ms, scales, static_cast<uint64_t>(k) / 16, rows, kStageK / 16, false, box_rows);
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// gate_up stack [E, 2I, K] (codes: K/2 bytes a row, scales: K/16) as a 4-D
// uint8 map (bytes of a row, row within the half, gate/up half, expert) read
// in boxes of 64 rows of both halves: one box = a 128-row gate_up tile (gate
// rows then the same up rows).  Codes use the 128-byte swizzle.
int gate_up_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t inter,
                uint64_t experts, uint32_t box_bytes, bool swizzle) {
  const cuuint64_t dims[4] = {row_bytes, inter, 2, experts};
  const cuuint64_t strides[3] = {row_bytes, row_bytes * inter, row_bytes * inter * 2};
  const cuuint32_t box[4] = {box_bytes, 64, 2, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled (gate_up) failed (%d)", (int)r);
  return NVFP4_OK;
}

int gate_up_maps(CUtensorMap* mc, CUtensorMap* ms, const uint8_t* codes, const uint8_t* scales,
                 int I, int H, int E) {
  int rc = gate_up_map(mc, codes, static_cast<uint64_t>(H) / 2, I, E, kStageK / 2, true);
  if (rc) return rc;
  return gate_up_map(ms, scales, static_cast<uint64_t>(H) / 16, I, E, kStageK / 16, false);
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
  L->x_offset = static_cast<int>(round_up(kTcOffSched + sched_bytes, 1024));
  L->ring_offset = static_cast<int>(round_up(L->x_offset + x_bytes, 1024));
  const long room = static_cast<long>(kSmemLimit) - kSmemAlignPad - L->ring_offset;
  L->n_stages = static_cast<int>(room / kTcStageBytes);
  if (L->n_stages > kTcMaxStages) L->n_stages = kTcMaxStages;
  if (L->n_stages < 3) return false;
  L->smem = kSmemAlignPad + L->ring_offset + static_cast<size_t>(L->n_stages) * kTcStageBytes;
  return true;
}

struct TcDensePlan {
  int n_tiles, nkb, grid, npad, xrows, win_k;
  size_t x_bytes;
  long units;
  TcLayout L;
  size_t off_partials, off_am, ws_bytes;
};

// 256-K stages (the weight bytes of four NVFP4 units: 8 FP8 or 16 BF16
// units) per CTA a single call with fewer 128-row tiles than SMs is cut
// into (whole tiles when K has at most this many): the call then holds only
// tiles x ceil(stages / this) SMs, and the next call's CTAs start streaming
// their weights on the others while it runs (programmatic dependent launch).
constexpr int kCallTargetStages = 4;

bool dense_mode_host(int mode) {
  return mode == kTcDense || mode == kTcDenseF8 || mode == kTcDenseBF;
}

bool plan_tc_dense(int M, int N, int K, int sms, TcDensePlan* p, int fmt = kFmtNvfp4) {
  p->n_tiles = (N + 127) / 128;
  if (p->n_tiles > kTcColCntBase) return false;
  p->nkb = K / tc_unit_k(fmt);
  p->units = static_cast<long>(p->n_tiles) * p->nkb;
  // the kernel splits units with 32-bit arithmetic (unit index x CTAs)
  if (p->units * (sms + 1) >= (1L << 31)) return false;
  p->grid = static_cast<int>(p->units < sms ? p->units : sms);
  if (p->n_tiles < sms) {
    const long target = kCallTargetStages * (kStageK / tc_unit_k(fmt));  // ~72 KB of weights
    const long splits = (p->nkb + target - 1) / target;
    const long g = static_cast<long>(p->n_tiles) * splits;
    if (g < p->grid) p->grid = static_cast<int>(g);
  }
  p->npad = M <= 16 ? 16 : 32;
  p->xrows = tc_xrows(M);
  const int cap = p->xrows == 8 ? 2 * kTcMaxWinK : kTcMaxWinK;  // 64 KB (8, 16 rows), 128 KB (32)
  p->win_k = K < cap ? K : cap;
  p->x_bytes = static_cast<size_t>(p->xrows) * p->win_k * 2;
  if (!tc_layout(0, p->x_bytes, &p->L)) return false;
  p->off_partials = kWsScratch;  // one pair of partial slots for every SM: programs
                                 // may place the op on any CTA
  p->off_am = round_up(p->off_partials + 4ull * sms * 2 * 32 * 128, 256);
  p->ws_bytes = round_up(p->off_am + 8ull * M * sms, 256);  // argmax: one partial per CTA
  return true;
}

struct TcMoePlan {
  int P, npad, xrows, sched_bytes, grid;
  size_t x_bytes;
  TcLayout gu, dn;
  size_t off_partials, off_h, off_y, ws_bytes;
};

bool plan_tc_moe(int T, int k, int E, int H, int I, int sms, TcMoePlan* p) {
  p->P = T * k;
  p->npad = T <= 16 ? 16 : 32;
  p->xrows = tc_xrows(T);
  if (H > 4096 || I > 2048) return false;  // staged rows are read once into registers
  p->sched_bytes = static_cast<int>(round_up(4ull * (4 * E + 5 + 2 * p->P + 33), 128));
  p->x_bytes = static_cast<size_t>(p->xrows) * (H > I ? H : I) * 2;
  if (!tc_layout(p->sched_bytes, static_cast<size_t>(p->xrows) * H * 2, &p->gu) ||
      !tc_layout(p->sched_bytes, static_cast<size_t>(p->xrows) * I * 2, &p->dn))
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


// Activation map of a tcgen05 op: BF16 [rows, k] with row stride ld
// elements, boxes of 64 x xrows (128 bytes x rows, 128-byte swizzle); rows
// past `rows` read as zero.
int act_map(CUtensorMap* m, const void* base, int rows, int64_t ld, int k, int xrows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(xrows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled (activations) failed (%d)", (int)r);
  return NVFP4_OK;
}

// ------------------------------------------------------------- validation
int check_gemm(const void* A, int64_t lda, int M, const nvfp4_weight* W, const void* C,
               int64_t ldc) {
  if (!A || !W || !C) return fail(NVFP4_ERR_INVALID, "A, W and C must be non-NULL");
  if (!W->codes || !W->scales || !W->global_scale)
    return fail(NVFP4_ERR_INVALID, "weight has a NULL pointer");
  const int N = W->n, K = W->k;
  if (M < 1 || M > kMaxM) return fail(NVFP4_ERR_SHAPE, "M=%d outside [1, 32]", M);
  if (N < 1 || K < 1) return fail(NVFP4_ERR_INVALID, "N=%d K=%d must be positive", N, K);
  if (K % 32) return fail(NVFP4_ERR_SHAPE, "K=%d is not a multiple of 32", K);
  if (lda < K || ldc < N) return fail(NVFP4_ERR_INVALID, "lda < K or ldc < N");
  if (!aligned16(A) || (lda * 2) % 16 || !aligned16(W->codes) || !aligned16(W->scales))
    return fail(NVFP4_ERR_ALIGN, "A rows and weight arrays must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(C) & 1u) return fail(NVFP4_ERR_ALIGN, "C must be 2-byte aligned");
  return NVFP4_OK;
}

int check_moe(const void* x, int64_t ldx, int T, const int32_t* topk_ids, const float* topk_w,
              int k, const nvfp4_expert_stack* experts, const nvfp4_expert_stack* shared,
              const void* out, int64_t ldo) {
  if (!x || !topk_ids || !topk_w || !out) return fail(NVFP4_ERR_INVALID, "NULL pointer");
  int rc = check_stack(experts, "experts");
  if (rc) return rc;
  if (shared) {
    if ((rc = check_stack(shared, "shared"))) return rc;
    if (shared->num_experts != 1 || shared->hidden != experts->hidden ||
        shared->inter != experts->inter)
      return fail(NVFP4_ERR_INVALID, "shared must be one expert of the same shape");
  }
  const int E = experts->num_experts, H = experts->hidden;
  if (T < 1 || T > kMaxM) return fail(NVFP4_ERR_SHAPE, "T=%d outside [1, 32]", T);
  if (k < 1 || k > 16 || k > E) return fail(NVFP4_ERR_SHAPE, "need 1 <= k <= min(16, E)");
  if (E > 512) return fail(NVFP4_ERR_SHAPE, "E=%d > 512", E);
  if (ldx < H || ldo < H) return fail(NVFP4_ERR_INVALID, "ldx and ldo must be >= hidden");
  if (!aligned16(x) || (ldx * 2) % 16) return fail(NVFP4_ERR_ALIGN, "x rows must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(out) & 1u) return fail(NVFP4_ERR_ALIGN, "out must be 2-byte aligned");
  return NVFP4_OK;
}

// ------------------------------------------------------------- CUDA-core path

struct FmaPlan {
  int grid, rows_per_cta, ru, ks;
  size_t smem, off_am, ws_bytes;
};

bool plan_fma(int M, int N, int K, int sms, FmaPlan* p) {
  p->rows_per_cta = fma_rows_per_cta(M, K);
  p->smem = fma_smem_bytes(p->rows_per_cta, K);
  if (p->smem > 200 * 1024) return false;
  const int ru = p->ru = fma_rows_per_warp(p->rows_per_cta, N);  // rows a warp takes at once
  const long groups = (static_cast<long>(N) + ru - 1) / ru;
  const long per_sm = p->smem <= 110 * 1024 ? 2 : 1;  // CTAs an SM holds
  // few groups: teams of warps share a group's K rounds
  p->ks = fma_k_split(groups, (K / 32 + 31) / 32, per_sm * sms * 8);
  const long ctas = (groups * p->ks + 7) / 8;   // eight warps a CTA
  p->grid = static_cast<int>(ctas < per_sm * sms ? ctas : per_sm * sms);
  const int row_groups = (M + p->rows_per_cta - 1) / p->rows_per_cta;
  if (4 + 4 * row_groups > static_cast<int>(kWsCounters)) return false;
  p->off_am = kWsScratch;
  p->ws_bytes = round_up(p->off_am + 8ull * M * p->grid, 256);
  return true;
}

// Which dense NVFP4 calls run on the CUDA cores (fma.cu) rather than the
// tensor cores: every K that is not a multiple of 256 (the tensor path
// streams 256-K stages), and the calls whose weight stream is short enough
// that the tensor-core kernel's fixed cost (about 8 to 13 us a call:
// tensor-memory allocation, ring fill, split-K drain) outweighs its faster
// streaming.  The CUDA-core kernel does one FMA per weight and activation
// row, so its rate falls as M grows; beyond four rows it runs four-row CTAs
// in ceil(M / 4) row groups, which pays while they all fit one wave of two
// CTAs an SM.  Measured on GB300, back-to-back calls in a CUDA graph with
// programmatic dependent launch, K = 2048 unless stated (CUDA cores vs
// tensor cores, us):
//   M = 1: 4096 rows 3.4 vs 14.4, 16384 rows 6.0 vs 13.5, 151,936 rows 51.6
//          vs 47.6;
//   M = 2: 16384 rows 9.8 vs 13.6, 32768 rows 18.8 vs 17.0;
//   M = 3: 8192 rows 8.5 vs 10.6, 16384 rows 13.7 vs 14.4;
//   M = 4: 8192 rows 9.6 vs 10.6, 16384 rows 15.8 vs 14.4;
//   M = 8: 64 rows 4.7 vs 9.0, 1024 rows 5.0 vs 9.5, 2048 x 4096 8.7 vs
//          11.7, 4096 rows 11.8 vs 10.0;
//   M = 12: 1024 rows 6.2 vs 11.1, 2048 x 4096 13.9 vs 13.8;
//   M = 16: 1024 rows 6.2 vs 12.2, 2048 x 4096 16.5 vs 14.9, 4096 rows
//          21.3 vs 12.7.
// Hence, by the weight bytes: M = 1 up to 128 MiB, M = 2, 3 up to 20 MiB,
// M = 4 up to 10 MiB; M = 5..16 up to 5 MiB and 2 CTAs an SM (ceil(N / 16)
// CTAs of two-row warps per row group); never beyond.
bool use_fma(int M, int N, int K, int sms) {
  if (K % kStageK) return true;
  const double mib = static_cast<double>(N) * K * 9.0 / 16.0 / (1 << 20);  // codes + block scales
  if (M == 1) return mib <= 128.0;
  if (M <= 3) return mib <= 20.0;
  if (M == 4) return mib <= 10.0;
  if (M > 16 || mib > 5.0) return false;
  const long ctas = (static_cast<long>(N) + 15) / 16 * ((M + 3) / 4);
  return ctas <= 2L * sms;
}

// MoE calls with few tokens run on the CUDA cores (moe_fma.cu): one FMA per
// weight and (token, slot) pair, no tensor-core pipeline to fill.  Measured
// on GB300 (256 experts, H = 2048, I = 512, top-8 + shared, back-to-back
// calls over 16 layers' experts; CUDA cores vs tensor cores, us a layer):
// T = 1 12.1 vs 43.4, T = 2 15.2 vs 44.6, T = 4 24.8 vs 49.4, T = 8 44.8 vs
// 62.7, T = 16 80.2 vs 96.3, T = 32 (two batches of 16) 160.0 vs 202.1: every
// T.  Shapes: I in {256, 512, 1024} (a down row is 8, 16 or 32 chunks of
// 32), a batch's staged activation rows within 96 KB of shared memory.
// Calls of more than kMoeFmaMaxT tokens run as batches of at most that many
// (the tokens are independent; each batch reads its own tokens' experts).
constexpr int kMoeFmaMaxCallT = 32;

bool use_moe_fma(int T, int k, int H, int I) {
  const int tb = T < kMoeFmaMaxT ? T : kMoeFmaMaxT;
  return T <= kMoeFmaMaxCallT && (I == 256 || I == 512 || I == 1024) &&
         static_cast<long>(tb) * H * 2 <= 96 * 1024 && moe_fma_slots(k, 1, I) != 0;
}

size_t moe_fma_ws_bytes(int T, int k, int I) {
  const int tb = T < kMoeFmaMaxT ? T : kMoeFmaMaxT;  // h of one batch
  return round_up(kWsScratch + static_cast<size_t>(tb) * (k + 1) * I * 4, 256);
}

// The MoE layer on the CUDA cores (arguments already checked).
int moe_fma(const void* x, int64_t ldx, int T, const int32_t* topk_ids, const float* topk_w, int k,
            const nvfp4_expert_stack* experts, const nvfp4_expert_stack* shared, void* out,
            int64_t ldo, uint32_t flags, void* workspace, size_t workspace_bytes, int sms,
            nvfp4_stream_t stream) {
  const int I = experts->inter;
  const size_t need = moe_fma_ws_bytes(T, k, I);
  if (!workspace || workspace_bytes < need)
    return fail(NVFP4_ERR_WORKSPACE, "workspace needs %zu bytes", need);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  MoeFmaArgs a;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.ldx = ldx;
  a.ids = topk_ids;
  a.w = topk_w;
  a.T = T;
  a.k = k;
  a.E = experts->num_experts;
  a.H = experts->hidden;
  a.I = I;
  a.gu_codes = experts->gu_codes;
  a.gu_scales = experts->gu_scales;
  a.dn_codes = experts->dn_codes;
  a.dn_scales = experts->dn_scales;
  a.gu_global = experts->gu_global;
  a.dn_global = experts->dn_global;
  a.has_shared = shared ? 1 : 0;
  a.s_gu_codes = shared ? shared->gu_codes : nullptr;
  a.s_gu_scales = shared ? shared->gu_scales : nullptr;
  a.s_dn_codes = shared ? shared->dn_codes : nullptr;
  a.s_dn_scales = shared ? shared->dn_scales : nullptr;
  a.s_gu_global = shared ? shared->gu_global : nullptr;
  a.s_dn_global = shared ? shared->dn_global : nullptr;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ldo = ldo;
  a.rms = (flags & NVFP4_FLAG_RMS_INPUT) ? 1 : 0;
  a.ids_ready = (flags & NVFP4_FLAG_IDS_READY) ? 1 : 0;
  a.h = reinterpret_cast<float*>(ws + kWsScratch);
  a.status = reinterpret_cast<uint32_t*>(ws + kWsStatus);
  // batches of at most kMoeFmaMaxT tokens, in order on the stream; a batch's
  // gate/up kernel writes h only after the previous batch's down kernel
  // ended (it waits for it before its main loop)
  int batches = 0;
  for (int t0 = 0; t0 < T; t0 += kMoeFmaMaxT, ++batches) {
    MoeFmaArgs b = a;
    b.T = T - t0 < kMoeFmaMaxT ? T - t0 : kMoeFmaMaxT;
    b.x = a.x + static_cast<size_t>(t0) * ldx;
    b.ids = a.ids + static_cast<size_t>(t0) * k;
    b.w = a.w + static_cast<size_t>(t0) * k;
    b.out = a.out + static_cast<size_t>(t0) * ldo;
    const cudaError_t e = launch_moe_fma(b, sms, reinterpret_cast<cudaStream_t>(stream),
                                         !(flags & NVFP4_FLAG_NO_PDL));
    if (e != cudaSuccess) return cuda_fail(e, "moe_fma kernels launch");
  }
  char buf[192];
  snprintf(buf, sizeof(buf),
           "%s; moe_fma_down_kernel slots=%d; T=%d k=%d E=%d shared=%d rms=%d ids_ready=%d "
           "batches=%d",
           moe_gate_up_mma(a.H, T < kMoeFmaMaxT ? T : kMoeFmaMaxT) ? "moe_mma_gate_up_kernel"
                                                                   : "moe_fma_gate_up_kernel",
           moe_fma_slots(k, a.has_shared, I), T, k, a.E, a.has_shared, a.rms, a.ids_ready,
           batches);
  g_dispatch = buf;
  return NVFP4_OK;
}


// ------------------------------------------------------------- tcgen05 ops
// K stages per CTA that a small dense op of a program is cut into (whole
// tiles when K has at most this many stages).  Measured on the 40-layer
// decode step at T = 8: 4 and 8 give the same step time; 16, and every op
// on every SM, are slower.
constexpr int kProgramTargetStages = 8;

void ws_header(TcArgs& a, uint8_t* ws) {
  a.tile_cnt = reinterpret_cast<uint32_t*>(ws + kWsCounters);
  a.argmax_cnt = reinterpret_cast<uint32_t*>(ws + kWsArgmaxCnt);
}

// A dense weight of any format: NVFP4 (codes, scales, per-tensor scale),
// FP8 E4M3 bytes [n, k] (codes) with one FP32 scale, or BF16 [n, ld] (codes).
struct DenseW {
  int fmt;
  const void* codes;
  const void* scales;
  const float* scale;
  int64_t ld;  // BF16: row stride in elements
  int n, k;
};

DenseW dense_w(const nvfp4_weight* W) {
  return DenseW{kFmtNvfp4, W->codes, W->scales, W->global_scale, W->k / 2, W->n, W->k};
}

// BF16 matrix [rows, ld] (k columns used) read in boxes of 64 x 128 rows
// (128 bytes x 128 rows, 128-byte swizzle).
int bf16_weight_map(CUtensorMap* m, const void* base, int64_t ld, int k, int rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled (bf16 weight) failed (%d)", (int)r);
  return NVFP4_OK;
}

// Dense op of a planned GEMM (arguments already checked).
int tc_dense_op(const void* A, int64_t lda, int M, const DenseW& W, void* C, int64_t ldc,
                int32_t* argmax_out, const int32_t* am_map, uint32_t flags, uint8_t* ws,
                const TcDensePlan& p, TcOp* op) {
  memset(op, 0, sizeof(*op));
  int rc;
  if (W.fmt == kFmtNvfp4) {
    rc = weight_maps(&op->maps[0], &op->maps[1], static_cast<const uint8_t*>(W.codes),
                     static_cast<const uint8_t*>(W.scales), static_cast<uint64_t>(W.n), W.k,
                     kTcTileRows);
    op->maps[2] = op->maps[0];
    op->maps[3] = op->maps[1];
  } else if (W.fmt == kFmtFp8) {
    rc = make_map(&op->maps[0], W.codes, static_cast<uint64_t>(W.k), static_cast<uint64_t>(W.n),
                  128, true, kTcTileRows);
  } else {
    rc = bf16_weight_map(&op->maps[0], W.codes, W.ld, W.k, W.n);
  }
  if (rc) return rc;
  if ((rc = act_map(&op->xmap, A, M, lda, W.k, p.xrows))) return rc;
  TcArgs& a = op->a;
  a.A = static_cast<const __nv_bfloat16*>(A);
  a.lda = lda;
  a.C = static_cast<__nv_bfloat16*>(C);
  a.ldc = ldc;
  a.argmax_out = argmax_out;
  a.am_map = am_map;
  a.gscale = W.scale;
  a.M = M;
  a.N = W.n;
  a.K = W.k;
  a.fmt = W.fmt;
  a.uk = tc_unit_k(W.fmt);
  a.rms = (flags & NVFP4_FLAG_RMS_INPUT) ? 1 : 0;
  a.win_k = p.win_k;
  a.n_ctas = p.grid;
  a.cta0 = 0;
  ws_header(a, ws);
  a.partials = reinterpret_cast<float*>(ws + p.off_partials);
  a.am_part = reinterpret_cast<int2*>(ws + p.off_am);
  op->mode = W.fmt == kFmtNvfp4 ? kTcDense : (W.fmt == kFmtFp8 ? kTcDenseF8 : kTcDenseBF);
  op->wait_prev = 1;
  return NVFP4_OK;
}

// gate_up and down ops of a planned MoE layer (arguments already checked).
int tc_moe_ops(const void* x, int64_t ldx, int T, const int32_t* topk_ids, const float* topk_w,
               int k, const nvfp4_expert_stack* experts, const nvfp4_expert_stack* shared,
               void* out, int64_t ldo, uint32_t flags, uint8_t* ws, const TcMoePlan& p,
               TcOp* gu, TcOp* dn, TcOp* cb) {
  const int E = experts->num_experts, H = experts->hidden, I = experts->inter;
  const nvfp4_expert_stack* sh = shared ? shared : experts;
  memset(gu, 0, sizeof(*gu));
  int rc;
  if ((rc = gate_up_maps(&gu->maps[0], &gu->maps[1], experts->gu_codes, experts->gu_scales, I, H,
                         E)) ||
      (rc = gate_up_maps(&gu->maps[2], &gu->maps[3], sh->gu_codes, sh->gu_scales, I, H,
                         sh->num_experts)) ||
      (rc = act_map(&gu->xmap, x, T, ldx, H, p.xrows)))
    return rc;
  TcArgs& a = gu->a;
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
  a.fmt = kFmtNvfp4;
  a.uk = kStageK;
  ws_header(a, ws);
  a.partials = reinterpret_cast<float*>(ws + p.off_partials);
  a.h = reinterpret_cast<float*>(ws + p.off_h);
  a.y = reinterpret_cast<float*>(ws + p.off_y);
  a.win_k = H;
  a.n_ctas = p.grid;
  a.cta0 = 0;
  gu->mode = kTcGateUp;
  gu->a.new_sched = 1;
  gu->wait_prev = 1;
  *dn = *gu;
  if ((rc = weight_maps(&dn->maps[0], &dn->maps[1], experts->dn_codes, experts->dn_scales,
                        static_cast<uint64_t>(H) * E, I, kTcTileRows)) ||
      (rc = weight_maps(&dn->maps[2], &dn->maps[3], sh->dn_codes, sh->dn_scales,
                        static_cast<uint64_t>(H) * sh->num_experts, I, kTcTileRows)))
    return rc;
  dn->a.win_k = I;
  dn->mode = kTcDown;
  dn->a.new_sched = 0;
  *cb = *dn;  // the combine reads the down op's per-pair outputs; no weights
  cb->mode = kTcCombine;
  cb->a.last_sched_use = 1;
  return NVFP4_OK;
}

// Shared-memory layout of a program whose largest op stages x_bytes of
// activations and whose MoE schedules take sched_bytes (slots of them).
bool tc_program_layout(size_t x_bytes, int sched_bytes, int slots, TcProgram* pr, size_t* smem) {
  TcLayout L;
  if (!tc_layout(sched_bytes * slots, x_bytes, &L)) return false;
  pr->x_offset = L.x_offset;
  pr->ring_offset = L.ring_offset;
  pr->n_stages = L.n_stages;
  pr->sched_offset = kTcOffSched;
  pr->sched_bytes = sched_bytes;
  pr->sched_slots = slots;
  *smem = L.smem;
  return true;
}

void tc_program_header(TcProgram* pr, uint8_t* ws) {
  pr->status = reinterpret_cast<uint32_t*>(ws + kWsStatus);
  pr->done = reinterpret_cast<uint32_t*>(ws + kWsCounters) + kTcDoneBase;
}

// A one-op program passed by value.
int tc_launch_one(const TcOp& op, size_t x_bytes, int sched_bytes, int grid, uint8_t* ws,
                  cudaStream_t s, bool pdl, int* n_stages, size_t* smem, const char* what) {
  TcProgram pr;
  memset(&pr, 0, sizeof(pr));
  if (!tc_program_layout(x_bytes, sched_bytes, 1, &pr, smem))
    return fail(NVFP4_ERR_SHAPE, "%s: staged activations exceed shared memory", what);
  tc_program_header(&pr, ws);
  pr.ops = nullptr;
  pr.n_ops = 1;
  pr.inline_ops[0] = op;
  const bool moe = op.mode == kTcGateUp || op.mode == kTcDown || op.mode == kTcCombine;
  pr.inline_ops[0].a.new_sched = moe ? 1 : 0;
  pr.inline_ops[0].a.last_sched_use = moe ? 1 : 0;
  *n_stages = pr.n_stages;
  cudaError_t e = launch_tc(pr, grid, *smem, s, pdl, false);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return NVFP4_OK;
}
}  // namespace

namespace nvfp4 {
void set_last_error(const char* msg) { g_error = msg; }
int check_gemm_args(const void* A, int64_t lda, int M, const nvfp4_weight* W, const void* C,
                    int64_t ldc) {
  return check_gemm(A, lda, M, W, C, ldc);
}
}  // namespace nvfp4

// A program: its op table on the device and the launch that runs it.
struct nvfp4_program {
  nvfp4::TcOp* d_ops = nullptr;
  nvfp4::TcProgram params;
  int grid = 0;
  int device = -1;
  size_t smem = 0;
  std::string desc;
};

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
  if (M < 1 || M > kMaxM || N < 1 || K < 32 || K % 32) return 0;
  if (current_device(&sms) != NVFP4_OK) return 0;
  if (use_fma(M, N, K, sms)) {
    FmaPlan f;
    return plan_fma(M, N, K, sms, &f) ? f.ws_bytes : 0;
  }
  TcDensePlan t;
  return plan_tc_dense(M, N, K, sms, &t) ? t.ws_bytes : 0;
}

// The dense skinny GEMM of any weight format (arguments already checked);
// am_map (nullable) maps the argmax's row index to the id reported.
static int dense_skinny(const char* name, const void* A, int64_t lda, int M, const DenseW& W,
                        void* C, int64_t ldc, int32_t* argmax_out, const int32_t* am_map,
                        uint32_t flags, void* workspace, size_t workspace_bytes,
                        nvfp4_stream_t stream) {
  int rc;
  const int N = W.n, K = W.k;
  int sms = 0;
  if ((rc = current_device(&sms))) return rc;
  TcDensePlan p;
  if (!plan_tc_dense(M, N, K, sms, &p, W.fmt))
    return fail(NVFP4_ERR_SHAPE, "N=%d, K=%d: no feasible plan", N, K);
  if (!workspace || workspace_bytes < p.ws_bytes)
    return fail(NVFP4_ERR_WORKSPACE, "workspace needs %zu bytes", p.ws_bytes);
  if ((rc = get_encoder())) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  TcOp op;
  if ((rc = tc_dense_op(A, lda, M, W, C, ldc, argmax_out, am_map, flags, ws, p, &op))) return rc;
  int n_stages = 0;
  size_t smem = 0;
  rc = tc_launch_one(op, p.x_bytes, 0, p.grid, ws,
                     reinterpret_cast<cudaStream_t>(stream), !(flags & NVFP4_FLAG_NO_PDL),
                     &n_stages, &smem, "stream_tc_kernel<dense> launch");
  if (rc) return rc;
  char buf[256];
  snprintf(buf, sizeof(buf),
           "stream_tc_kernel<dense> weight=%s grid=%d tiles=%d units=%ld units_per_cta=%.2f "
           "window=%d n=%d stages=%d smem=%zu argmax=%d rms=%d",
           name, p.grid, p.n_tiles, p.units, static_cast<double>(p.units) / p.grid, p.win_k,
           p.npad, n_stages, smem, argmax_out ? 1 : 0, op.a.rms);
  g_dispatch = buf;
  return NVFP4_OK;
}

// The CUDA-core kernel (arguments already checked).
static int fma_skinny(const void* A, int64_t lda, int M, const nvfp4_weight* W, void* C,
                      int64_t ldc, int32_t* argmax_out, const int32_t* am_map, uint32_t flags,
                      void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  int sms = 0, rc;
  if ((rc = current_device(&sms))) return rc;
  FmaPlan p;
  if (!plan_fma(M, W->n, W->k, sms, &p))
    return fail(NVFP4_ERR_SHAPE, "N=%d, K=%d: no feasible plan", W->n, W->k);
  if (!workspace || workspace_bytes < p.ws_bytes)
    return fail(NVFP4_ERR_WORKSPACE, "workspace needs %zu bytes", p.ws_bytes);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  FmaArgs a;
  a.A = static_cast<const __nv_bfloat16*>(A);
  a.lda = lda;
  a.codes = W->codes;
  a.scales = W->scales;
  a.gscale = W->global_scale;
  a.C = static_cast<__nv_bfloat16*>(C);
  a.ldc = ldc;
  a.argmax_out = argmax_out;
  a.am_map = am_map;
  a.M = M;
  a.N = W->n;
  a.K = W->k;
  a.rms = (flags & NVFP4_FLAG_RMS_INPUT) ? 1 : 0;
  a.argmax_cnt = reinterpret_cast<uint32_t*>(ws + kWsArgmaxCnt);
  a.am_part = reinterpret_cast<int2*>(ws + p.off_am);
  a.ks = p.ks;
  const cudaError_t e = launch_fma(a, p.grid, p.ru, reinterpret_cast<cudaStream_t>(stream),
                                   !(flags & NVFP4_FLAG_NO_PDL));
  if (e != cudaSuccess) return cuda_fail(e, "fma_kernel launch");
  char buf[192];
  snprintf(buf, sizeof(buf),
           "fma_kernel grid=%dx%d rows_per_cta=%d rows_per_warp=%d k_split=%d smem=%zu argmax=%d "
           "rms=%d",
           p.grid, (M + p.rows_per_cta - 1) / p.rows_per_cta, p.rows_per_cta, p.ru, p.ks, p.smem,
           argmax_out ? 1 : 0, a.rms);
  g_dispatch = buf;
  return NVFP4_OK;
}

static int gemm_skinny(const void* A, int64_t lda, int M, const nvfp4_weight* W, void* C,
                       int64_t ldc, int32_t* argmax_out, const int32_t* am_map, uint32_t flags,
                       void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  int rc = check_gemm(A, lda, M, W, C, ldc), sms = 0;
  if (rc) return rc;
  if ((rc = current_device(&sms))) return rc;
  if (use_fma(M, W->n, W->k, sms))
    return fma_skinny(A, lda, M, W, C, ldc, argmax_out, am_map, flags, workspace,
                      workspace_bytes, stream);
  return dense_skinny("nvfp4", A, lda, M, dense_w(W), C, ldc, argmax_out, am_map, flags,
                      workspace, workspace_bytes, stream);
}

// Checks shared by the FP8 and BF16 weight formats (K a multiple of 256, as
// for NVFP4: activations are staged in 256-K blocks).
static int check_dense_common(const void* A, int64_t lda, int M, int N, int K, const void* C,
                              int64_t ldc) {
  if (!A || !C) return fail(NVFP4_ERR_INVALID, "A and C must be non-NULL");
  if (M < 1 || M > kMaxM) return fail(NVFP4_ERR_SHAPE, "M=%d outside [1, 32]", M);
  if (N < 1 || K < 1) return fail(NVFP4_ERR_INVALID, "N=%d K=%d must be positive", N, K);
  if (K % kStageK) return fail(NVFP4_ERR_SHAPE, "K=%d is not a multiple of 256", K);
  if (lda < K || ldc < N) return fail(NVFP4_ERR_INVALID, "lda < K or ldc < N");
  if (!aligned16(A) || (lda * 2) % 16) return fail(NVFP4_ERR_ALIGN, "A rows must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(C) & 1u) return fail(NVFP4_ERR_ALIGN, "C must be 2-byte aligned");
  return NVFP4_OK;
}

int nvfp4_gemm_skinny(const void* A, int64_t lda, int M, const nvfp4_weight* W, void* C,
                      int64_t ldc, int32_t* argmax_out, uint32_t flags, void* workspace,
                      size_t workspace_bytes, nvfp4_stream_t stream) {
  return gemm_skinny(A, lda, M, W, C, ldc, argmax_out, nullptr, flags, workspace,
                     workspace_bytes, stream);
}

size_t fp8_gemm_skinny_workspace(int M, int N, int K) {
  int sms = 0;
  if (M < 1 || M > kMaxM || N < 1 || K < kStageK || K % kStageK) return 0;
  if (current_device(&sms) != NVFP4_OK) return 0;
  TcDensePlan t;
  return plan_tc_dense(M, N, K, sms, &t, kFmtFp8) ? t.ws_bytes : 0;
}

int fp8_gemm_skinny(const void* A, int64_t lda, int M, const fp8_weight* W, void* C, int64_t ldc,
                    int32_t* argmax_out, uint32_t flags, void* workspace, size_t workspace_bytes,
                    nvfp4_stream_t stream) {
  if (!W || !W->codes || !W->scale) return fail(NVFP4_ERR_INVALID, "FP8 weight has a NULL pointer");
  int rc = check_dense_common(A, lda, M, W->n, W->k, C, ldc);
  if (rc) return rc;
  if (!aligned16(W->codes)) return fail(NVFP4_ERR_ALIGN, "weight must be 16-byte aligned");
  const DenseW d{kFmtFp8, W->codes, nullptr, W->scale, W->k, W->n, W->k};
  return dense_skinny("fp8", A, lda, M, d, C, ldc, argmax_out, nullptr, flags, workspace,
                      workspace_bytes, stream);
}

size_t bf16w_gemm_skinny_workspace(int M, int N, int K) {
  int sms = 0;
  if (M < 1 || M > kMaxM || N < 1 || K < kStageK || K % kStageK) return 0;
  if (current_device(&sms) != NVFP4_OK) return 0;
  TcDensePlan t;
  return plan_tc_dense(M, N, K, sms, &t, kFmtBf16) ? t.ws_bytes : 0;
}

int bf16w_gemm_skinny(const void* A, int64_t lda, int M, const bf16_weight* W, void* C,
                      int64_t ldc, int32_t* argmax_out, uint32_t flags, void* workspace,
                      size_t workspace_bytes, nvfp4_stream_t stream) {
  if (!W || !W->w) return fail(NVFP4_ERR_INVALID, "BF16 weight has a NULL pointer");
  int rc = check_dense_common(A, lda, M, W->n, W->k, C, ldc);
  if (rc) return rc;
  if (W->ldw < W->k) return fail(NVFP4_ERR_INVALID, "ldw < K");
  if (!aligned16(W->w) || (W->ldw * 2) % 16)
    return fail(NVFP4_ERR_ALIGN, "weight rows must be 16-byte aligned");
  const DenseW d{kFmtBf16, W->w, nullptr, nullptr, W->ldw, W->n, W->k};
  return dense_skinny("bf16", A, lda, M, d, C, ldc, argmax_out, nullptr, flags, workspace,
                      workspace_bytes, stream);
}

int nvfp4_hot_vocab_head(const void* A, int64_t lda, int M, const nvfp4_weight* W_hot,
                         const int32_t* vocab_ids, void* C, int64_t ldc, int32_t* argmax_out,
                         uint32_t flags, void* workspace, size_t workspace_bytes,
                         nvfp4_stream_t stream) {
  if (!vocab_ids || !argmax_out)
    return fail(NVFP4_ERR_INVALID, "vocab_ids and argmax_out must be non-NULL");
  return gemm_skinny(A, lda, M, W_hot, C, ldc, argmax_out, vocab_ids, flags, workspace,
                     workspace_bytes, stream);
}

int nvfp4_quantize(const void* W, int64_t ldw, int N, int K, void* codes, void* scales,
                   float* global_scale, nvfp4_stream_t stream) {
  if (!W || !codes || !scales || !global_scale)
    return fail(NVFP4_ERR_INVALID, "W, codes, scales and global_scale must be non-NULL");
  if (N < 1 || K < 1 || ldw < K) return fail(NVFP4_ERR_INVALID, "N=%d, K=%d, ldw=%lld", N, K,
                                            static_cast<long long>(ldw));
  if (K % 32) return fail(NVFP4_ERR_SHAPE, "K=%d is not a multiple of 32", K);
  if (!aligned16(W) || (ldw * 2) % 16 || !aligned16(codes) ||
      (reinterpret_cast<uintptr_t>(global_scale) & 3u))
    return fail(NVFP4_ERR_ALIGN, "W rows and codes must be 16-byte aligned");
  int sms = 0, rc;
  if ((rc = current_device(&sms))) return rc;
  QuantArgs a;
  a.W = static_cast<const __nv_bfloat16*>(W);
  a.ldw = ldw;
  a.N = N;
  a.K = K;
  a.codes = static_cast<uint8_t*>(codes);
  a.scales = static_cast<uint8_t*>(scales);
  a.amax_bits = reinterpret_cast<uint32_t*>(global_scale);
  a.global_scale = global_scale;
  const cudaError_t e = launch_quantize(a, sms, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize kernels launch");
  char buf[128];
  snprintf(buf, sizeof(buf), "amax_kernel, quantize_kernel, global_scale_kernel N=%d K=%d", N, K);
  g_dispatch = buf;
  return NVFP4_OK;
}

int nvfp4_gather_rows(const nvfp4_weight* src, const int32_t* rows, int n_rows, void* codes,
                      void* scales, nvfp4_stream_t stream) {
  if (!src || !rows || !codes || !scales)
    return fail(NVFP4_ERR_INVALID, "src, rows, codes and scales must be non-NULL");
  if (!src->codes || !src->scales) return fail(NVFP4_ERR_INVALID, "src has a NULL pointer");
  if (n_rows < 1 || src->n < 1 || src->k < 1)
    return fail(NVFP4_ERR_INVALID, "n_rows=%d, N=%d, K=%d must be positive", n_rows, src->n,
                src->k);
  if (src->k % kStageK) return fail(NVFP4_ERR_SHAPE, "K=%d is not a multiple of 256", src->k);
  if (!aligned16(src->codes) || !aligned16(src->scales) || !aligned16(codes) || !aligned16(scales))
    return fail(NVFP4_ERR_ALIGN, "code and scale arrays must be 16-byte aligned");
  GatherArgs a;
  a.src_codes = src->codes;
  a.src_scales = src->scales;
  a.N = src->n;
  a.K = src->k;
  a.rows = rows;
  a.n_rows = n_rows;
  a.dst_codes = static_cast<uint8_t*>(codes);
  a.dst_scales = static_cast<uint8_t*>(scales);
  const cudaError_t e = launch_gather_rows(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gather_rows_kernel launch");
  char buf[128];
  snprintf(buf, sizeof(buf), "gather_rows_kernel rows=%d N=%d K=%d", n_rows, src->n, src->k);
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
  if (use_moe_fma(T, k, experts->hidden, experts->inter))
    return moe_fma_ws_bytes(T, k, experts->inter);
  TcMoePlan t;
  return plan_tc_moe(T, k, experts->num_experts, experts->hidden, experts->inter, sms, &t)
             ? t.ws_bytes : 0;
}

int moe_nvfp4_decode(const void* x, int64_t ldx, int T, const int32_t* topk_ids,
                     const float* topk_w, int k, const nvfp4_expert_stack* experts,
                     const nvfp4_expert_stack* shared, void* out, int64_t ldo, uint32_t flags,
                     void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  int rc = check_moe(x, ldx, T, topk_ids, topk_w, k, experts, shared, out, ldo);
  if (rc) return rc;
  const int E = experts->num_experts, H = experts->hidden, I = experts->inter;
  int sms = 0;
  if ((rc = current_device(&sms))) return rc;
  if (use_moe_fma(T, k, H, I))
    return moe_fma(x, ldx, T, topk_ids, topk_w, k, experts, shared, out, ldo, flags, workspace,
                   workspace_bytes, sms, stream);
  TcMoePlan p;
  if (!plan_tc_moe(T, k, E, H, I, sms, &p))
    return fail(NVFP4_ERR_SHAPE, "T=%d, H=%d, E=%d: staged activations exceed shared memory",
                T, H, E);
  if (!workspace || workspace_bytes < p.ws_bytes)
    return fail(NVFP4_ERR_WORKSPACE, "workspace needs %zu bytes", p.ws_bytes);
  if ((rc = get_encoder())) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  TcOp gu, dn, cb;
  if ((rc = tc_moe_ops(x, ldx, T, topk_ids, topk_w, k, experts, shared, out, ldo, flags, ws, p,
                       &gu, &dn, &cb)))
    return rc;
  const bool pdl = !(flags & NVFP4_FLAG_NO_PDL);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int st_gu = 0, st_dn = 0;
  size_t sm_gu = 0, sm_dn = 0;
  if ((rc = tc_launch_one(gu, static_cast<size_t>(p.xrows) * H * 2, p.sched_bytes, p.grid, ws,
                          s, pdl, &st_gu, &sm_gu, "stream_tc_kernel<gate_up> launch")) ||
      (rc = tc_launch_one(dn, static_cast<size_t>(p.xrows) * I * 2, p.sched_bytes, p.grid, ws,
                          s, pdl, &st_dn, &sm_dn, "stream_tc_kernel<down> launch")))
    return rc;
  int st_cb = 0;
  size_t sm_cb = 0;
  if ((rc = tc_launch_one(cb, 0, p.sched_bytes, p.grid, ws, s, pdl, &st_cb, &sm_cb,
                          "stream_tc_kernel<combine> launch")))
    return rc;
  char buf[256];
  snprintf(buf, sizeof(buf),
           "stream_tc_kernel<gate_up> grid=%d stages=%d smem=%zu; stream_tc_kernel<down> grid=%d "
           "stages=%d smem=%zu; stream_tc_kernel<combine> grid=%d; T=%d k=%d E=%d n=%d "
           "shared=%d rms=%d ids_ready=%d",
           p.grid, st_gu, sm_gu, p.grid, st_dn, sm_dn, p.grid, T, k, E, p.npad,
           gu.a.has_shared, gu.a.rms, gu.a.ids_ready);
  g_dispatch = buf;
  return NVFP4_OK;
}

size_t nvfp4_program_workspace(const nvfp4_op* ops, int n_ops) {
  int sms = 0;
  if (!ops || n_ops < 1 || n_ops > kTcMaxOps) return 0;
  if (current_device(&sms) != NVFP4_OK) return 0;
  size_t need = kWsScratch;
  for (int i = 0; i < n_ops; ++i) {
    const nvfp4_op& o = ops[i];
    size_t b = 0;
    if (o.kind == NVFP4_OP_GEMM) {
      TcDensePlan t;
      if (o.M < 1 || o.M > kMaxM || o.W.k < kStageK || o.W.k % kStageK ||
          !plan_tc_dense(o.M, o.W.n, o.W.k, sms, &t))
        return 0;
      b = t.ws_bytes;
    } else if (o.kind == NVFP4_OP_MOE) {
      TcMoePlan t;
      if (o.T < 1 || o.T > kMaxM || o.k < 1 || o.k > 16 ||
          !plan_tc_moe(o.T, o.k, o.experts.num_experts, o.experts.hidden, o.experts.inter, sms, &t))
        return 0;
      b = t.ws_bytes;
    } else {
      return 0;
    }
    if (b > need) need = b;
  }
  return need;
}

int nvfp4_program_create(const nvfp4_op* ops, int n_ops, void* workspace, size_t workspace_bytes,
                         nvfp4_program** program) {
  if (!program) return fail(NVFP4_ERR_INVALID, "program is NULL");
  *program = nullptr;
  if (!ops || n_ops < 1) return fail(NVFP4_ERR_INVALID, "no ops");
  int rc;
  // host-side checks of every op first, then the device
  for (int i = 0; i < n_ops; ++i) {
    const nvfp4_op& o = ops[i];
    if (o.kind == NVFP4_OP_GEMM)
      rc = check_gemm(o.A, o.lda, o.M, &o.W, o.C, o.ldc);
    else if (o.kind == NVFP4_OP_MOE)
      rc = check_moe(o.x, o.ldx, o.T, o.topk_ids, o.topk_w, o.k, &o.experts,
                     o.shared.num_experts ? &o.shared : nullptr, o.out, o.ldo);
    else
      rc = fail(NVFP4_ERR_INVALID, "op %d: unknown kind %d", i, o.kind);
    if (rc) return rc;
  }
  int sms = 0;
  if ((rc = current_device(&sms))) return rc;
  if ((rc = get_encoder())) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  std::vector<TcOp> table;
  size_t x_bytes = 0, need = kWsScratch;
  int sched_bytes = 0, n_gemm = 0, n_moe = 0;
  for (int i = 0; i < n_ops; ++i) {
    const nvfp4_op& o = ops[i];
    if (o.flags & ~static_cast<uint32_t>(NVFP4_FLAG_RMS_INPUT | NVFP4_FLAG_NO_PDL |
                                         NVFP4_FLAG_IDS_READY | NVFP4_FLAG_ALL_SMS))
      return fail(NVFP4_ERR_INVALID, "op %d: unsupported flags 0x%x", i, o.flags);
    if (o.kind == NVFP4_OP_GEMM) {
      if ((rc = check_gemm(o.A, o.lda, o.M, &o.W, o.C, o.ldc))) return rc;
      if (o.W.k % kStageK)
        return fail(NVFP4_ERR_SHAPE, "op %d: K=%d: program ops need K %% 256 == 0", i, o.W.k);
      TcDensePlan p;
      if (!plan_tc_dense(o.M, o.W.n, o.W.k, sms, &p))
        return fail(NVFP4_ERR_SHAPE, "op %d: N=%d, K=%d: no feasible plan", i, o.W.n, o.W.k);
      TcOp op;
      if (o.argmax_map && !o.argmax_out)
        return fail(NVFP4_ERR_INVALID, "op %d: argmax_map without argmax_out", i);
      if ((rc = tc_dense_op(o.A, o.lda, o.M, dense_w(&o.W), o.C, o.ldc, o.argmax_out,
                            o.argmax_map, o.flags, ws, p, &op)))
        return rc;
      op.all_sms = (o.flags & NVFP4_FLAG_ALL_SMS) ? 1 : 0;
      table.push_back(op);
      x_bytes = std::max(x_bytes, p.x_bytes);
      need = std::max(need, p.ws_bytes);
      ++n_gemm;
    } else if (o.kind == NVFP4_OP_MOE) {
      const nvfp4_expert_stack* sh = o.shared.num_experts ? &o.shared : nullptr;
      if ((rc = check_moe(o.x, o.ldx, o.T, o.topk_ids, o.topk_w, o.k, &o.experts, sh, o.out,
                          o.ldo)))
        return rc;
      const int E = o.experts.num_experts, H = o.experts.hidden, I = o.experts.inter;
      TcMoePlan p;
      if (!plan_tc_moe(o.T, o.k, E, H, I, sms, &p))
        return fail(NVFP4_ERR_SHAPE, "op %d: T=%d, H=%d, E=%d: no feasible plan", i, o.T, H, E);
      TcOp gu, dn, cb;
      if ((rc = tc_moe_ops(o.x, o.ldx, o.T, o.topk_ids, o.topk_w, o.k, &o.experts, sh, o.out,
                           o.ldo, o.flags | NVFP4_FLAG_IDS_READY, ws, p, &gu, &dn, &cb)))
        return rc;
      table.push_back(gu);
      table.push_back(dn);
      table.push_back(cb);
      x_bytes = std::max(x_bytes, p.x_bytes);
      sched_bytes = std::max(sched_bytes, p.sched_bytes);
      need = std::max(need, p.ws_bytes);
      ++n_moe;
    } else {
      return fail(NVFP4_ERR_INVALID, "op %d: unknown kind %d", i, o.kind);
    }
  }
  const int n = static_cast<int>(table.size());
  if (n > kTcMaxOps) return fail(NVFP4_ERR_SHAPE, "program of %d kernel ops > %d", n, kTcMaxOps);
  // CTA ranges.  A dense op with fewer 128-row tiles than SMs is spread over
  // only tiles x ceil(K stages / target) CTAs (whole tiles, or few splits per
  // tile: short reductions), placed after the previous small op's CTAs, so
  // that the other SMs stream the following ops' weights meanwhile.  Ops with
  // at least one tile per SM (and MoE ops, and ops flagged
  // NVFP4_FLAG_ALL_SMS) use every SM.
  constexpr int target = kProgramTargetStages;
  int next_cta = 0;
  for (TcOp& op : table) {
    // (a dense op flagged NVFP4_FLAG_ALL_SMS keeps its single call's CTA
    // count, set when the op was built)
    int g = (dense_mode_host(op.mode) && op.all_sms) ? op.a.n_ctas : sms;
    if (op.mode == kTcDense && !op.all_sms) {
      const int n_tiles = (op.a.N + 127) / 128, nkb = op.a.K / kStageK;
      if (n_tiles < sms) {
        const int splits = (nkb + target - 1) / target;
        g = std::min(sms, n_tiles * splits);
      }
    }
    op.a.n_ctas = g;
    op.a.cta0 = next_cta;
    next_cta = (next_cta + (g < sms ? g : 0)) % sms;
  }
  if (!workspace || workspace_bytes < need)
    return fail(NVFP4_ERR_WORKSPACE, "workspace needs %zu bytes", need);
  table[0].wait_prev = 0;
  auto* pg = new (std::nothrow) nvfp4_program();
  if (!pg) return fail(NVFP4_ERR_INVALID, "out of host memory");
  memset(&pg->params, 0, sizeof(pg->params));
  if (!tc_program_layout(x_bytes, sched_bytes, sched_bytes ? 2 : 1, &pg->params, &pg->smem)) {
    delete pg;
    return fail(NVFP4_ERR_SHAPE, "staged activations exceed shared memory");
  }
  tc_program_header(&pg->params, ws);
  cudaError_t e = cudaMalloc(&pg->d_ops, sizeof(TcOp) * n);
  if (e == cudaSuccess)
    e = cudaMemcpy(pg->d_ops, table.data(), sizeof(TcOp) * n, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    if (pg->d_ops) cudaFree(pg->d_ops);
    delete pg;
    return cuda_fail(e, "program table");
  }
  cudaGetDevice(&pg->device);
  pg->params.ops = pg->d_ops;
  pg->params.n_ops = n;
  pg->grid = sms;
  char buf[256];
  snprintf(buf, sizeof(buf),
           "stream_tc_kernel program ops=%d (gemm=%d moe=%d) grid=%d stages=%d smem=%zu "
           "sched_slots=%d cooperative=1",
           n, n_gemm, n_moe, pg->grid, pg->params.n_stages, pg->smem, pg->params.sched_slots);
  pg->desc = buf;
  *program = pg;
  return NVFP4_OK;
}

int nvfp4_program_launch(const nvfp4_program* program, nvfp4_stream_t stream) {
  if (!program) return fail(NVFP4_ERR_INVALID, "program is NULL");
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != program->device)
    return fail(NVFP4_ERR_INVALID, "program was created on device %d, current is %d",
                program->device, dev);
  cudaError_t e = launch_tc(program->params, program->grid, program->smem,
                            reinterpret_cast<cudaStream_t>(stream), false, true);
  if (e != cudaSuccess) return cuda_fail(e, "stream_tc_kernel program launch");
  g_dispatch = program->desc;
  return NVFP4_OK;
}

int nvfp4_program_destroy(nvfp4_program* program) {
  if (!program) return NVFP4_OK;
  cudaError_t e = cudaFree(program->d_ops);
  delete program;
  return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "cudaFree");
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

int nvfp4_hbm_read_probe(const void* buf, size_t bytes, void* sink, size_t sink_bytes,
                         nvfp4_stream_t stream) {
  if (!buf || !sink) return fail(NVFP4_ERR_INVALID, "buf and sink must be non-NULL");
  if (bytes == 0 || bytes % 16) return fail(NVFP4_ERR_INVALID, "bytes must be a positive multiple of 16");
  if (!aligned16(buf)) return fail(NVFP4_ERR_ALIGN, "buf must be 16-byte aligned");
  int sms = 0, rc;
  if ((rc = current_device(&sms))) return rc;
  const int grid = 2 * sms;
  if (sink_bytes < 4ull * grid)
    return fail(NVFP4_ERR_WORKSPACE, "sink needs %d bytes", 4 * grid);
  const cudaError_t e = launch_read_probe(buf, bytes, static_cast<uint32_t*>(sink), grid,
                                          reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "read_probe_kernel launch");
  char b2[96];
  snprintf(b2, sizeof(b2), "read_probe_kernel grid=%d bytes=%zu", grid, bytes);
  g_dispatch = b2;
  return NVFP4_OK;
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
