// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "nvfp4moe.h"

namespace nvfp4 {

// Workspace layout shared by every call, so that one workspace can serve a
// sequence of different calls: [0, 256) status word and the argmax counter;
// [256, kWsScratch) the tile counters (kept at zero between calls); call
// scratch (partials, h, per-pair outputs) from kWsScratch on.
constexpr size_t kWsStatus = 0;
constexpr size_t kWsArgmaxCnt = 4;
constexpr size_t kWsCounters = 256;
constexpr int kWsMaxCounters = 16384;
constexpr size_t kWsScratch = kWsCounters + 4 * kWsMaxCounters;

// ---- tcgen05 streaming kernel (stream_tc.cu) ------------------------------
// One launch runs a program: a sequence of ops (dense GEMM, MoE gate_up, MoE
// down), each reading what earlier ops wrote.  Shared memory (from a
// 1024-byte aligned base): barriers, misc, the [32][128] f32 epilogue tile,
// the expert-schedule slots, the staged activations, then the weight ring
// (1024-aligned, n_stages x 18 KB); one layout for the whole program.
constexpr int kTcTileRows = 128;                                // weight rows per tile
constexpr int kTcStageBytes = 128 * 256 / 2 + 128 * 256 / 16;  // 18432
constexpr int kTcMaxStages = 8;
constexpr int kTcOffBars = 0;                            // up to 64 mbarriers
constexpr int kTcOffMisc = 512;
constexpr int kTcOffArgs = 1024;                         // the current op's TcArgs (epilogue)
constexpr int kTcArgsBytes = 512;
constexpr int kTcOffEp = kTcOffArgs + kTcArgsBytes;
constexpr int kTcOffSched = kTcOffEp + 32 * 128 * 4;     // 17920
// four warpgroups: {producer, MMA, scheduler, idle}, 4 epilogue warps,
// 8 decode warps (registers rebalanced per warpgroup with setmaxnreg)
constexpr int kTcThreads = 512;
constexpr int kTcColCntBase = 8192;                      // tile counters stay below this index
constexpr int kTcDoneBase = 12288;                       // per-op completion counters
constexpr int kTcMaxOps = kWsMaxCounters - kTcDoneBase - 1;
constexpr int kTcMaxWinK = 2048;                         // activations staged per window
constexpr int kTcInlineOps = 1;                          // ops passed by value in the launch

// kTcCombine: the weighted top-k combine of a MoE layer's per-pair down
// outputs (no weights: only the epilogue warps work).
// kTcDenseF8 / kTcDenseBF: the dense op with FP8 or BF16 weights (kTcDense:
// NVFP4).
enum TcMode { kTcDense = 0, kTcGateUp = 1, kTcDown = 2, kTcCombine = 3, kTcDenseF8 = 4,
              kTcDenseBF = 5 };

// Weight format of a dense op.  Every format streams 128-row x 128-byte
// boxes of codes (the 128-byte swizzle), one box per unit of work:
//   NVFP4: 256 K per unit (E2M1 pairs) + a 128 x 16 box of E4M3 scales;
//   FP8:   128 K per unit, E4M3 bytes, one FP32 scale for the matrix;
//   BF16:  64 K per unit, read by the MMA from shared memory as it is.
enum TcFmt { kFmtNvfp4 = 0, kFmtFp8 = 1, kFmtBf16 = 2 };
__host__ __device__ constexpr int tc_unit_k(int fmt) {
  return fmt == kFmtNvfp4 ? 256 : (fmt == kFmtFp8 ? 128 : 64);
}

struct alignas(16) TcArgs {  // (a whole number of 16-byte words: copied by words)
  // dense
  const __nv_bfloat16* A;
  int64_t lda;
  __nv_bfloat16* C;
  int64_t ldc;
  int32_t* argmax_out;
  const int32_t* am_map;  // nullable: argmax_out reports am_map[n] instead of n
  const float* gscale;
  int M, N, K;
  // MoE
  const __nv_bfloat16* x;
  int64_t ldx;
  const int32_t* ids;
  const float* w;
  __nv_bfloat16* out;
  int64_t ldo;
  const float* gu_global;
  const float* dn_global;
  const float* sh_gu_global;
  const float* sh_dn_global;
  int T, k, E, H, I, has_shared, ids_ready;
  float* h;
  float* y;
  // common
  int fmt;              // TcFmt of a dense op's weight (MoE: NVFP4)
  int uk;               // K per unit of work: tc_unit_k(fmt)
  int rms;
  int win_k;            // staged activation window capacity (elements, multiple of 256)
  int n_ctas;           // CTAs the op's units are spread over (at most gridDim.x) ...
  int cta0;             // ... starting at this CTA (wrapping around)
  uint32_t* tile_cnt;   // counters region
  uint32_t* argmax_cnt;
  float* partials;      // [grid][2][32][128]
  int2* am_part;        // [M][CTAs of the op]: each CTA's best (value bits, index) per row
  int new_sched;        // MoE: build a new expert schedule from this op's ids
  int last_sched_use;   // MoE: no later op uses the current schedule
};

// Staged activation rows for n real rows: 8, 16 or 32 (the MMA's N is 16
// or 32; with 8 staged rows its rows 8..15 repeat rows 0..7).
__host__ __device__ constexpr int tc_xrows(int n) { return n <= 8 ? 8 : (n <= 16 ? 16 : 32); }

// One op of a program: its four weight tensor maps (dense: codes, scales of
// W, twice; MoE: routed codes, routed scales, shared codes, shared scales),
// the activation map (dense A / MoE x: BF16, boxes of 64 x tc_xrows rows with
// the 128-byte swizzle; unused by down) and its arguments.
struct TcOp {
  CUtensorMap maps[4];
  CUtensorMap xmap;
  TcArgs a;
  int mode;            // TcMode
  int wait_prev;       // read inputs only after every CTA finished the previous op
  int all_sms;         // program placement: spread over every SM (as the single call)
};

struct TcProgram {
  const TcOp* ops;     // device table of n_ops ops, or nullptr: inline_ops
  int n_ops;
  int x_offset, ring_offset, n_stages;
  int sched_offset, sched_bytes, sched_slots;
  uint32_t* status;
  uint32_t* done;      // [n_ops + 1] completion counters (zero between launches)
  TcOp inline_ops[kTcInlineOps];
};

// cooperative: the program's ops wait on each other across CTAs, so all CTAs
// must be resident at once.
cudaError_t launch_tc(const TcProgram& p, int grid, size_t smem, cudaStream_t s, bool pdl,
                      bool cooperative);

struct RouteArgs {
  const float* logits;
  int T, E, k, renorm;
  int32_t* ids;
  float* w;
};

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s, bool pdl);

// Row gather of an NVFP4 matrix [N, K]: dst row i = src row rows[i] (codes
// and scales), all-zero for a row id outside [0, N).  K % 256 == 0; every
// pointer 16-byte aligned.
struct GatherArgs {
  const uint8_t* src_codes;
  const uint8_t* src_scales;
  int N, K;
  const int32_t* rows;
  int n_rows;
  uint8_t* dst_codes;
  uint8_t* dst_scales;
};
cudaError_t launch_gather_rows(const GatherArgs& a, cudaStream_t s);

// BF16 -> NVFP4 quantisation of W [N, ldw] (K used; K % 32 == 0): codes
// [N, K/2], scales [N, K/16], and the per-tensor scale, which holds the bits
// of the matrix's largest magnitude while the kernels run (amax_bits and
// global_scale are the same 4 bytes).
struct QuantArgs {
  const __nv_bfloat16* W;
  int64_t ldw;
  int N, K;
  uint8_t* codes;
  uint8_t* scales;
  uint32_t* amax_bits;
  float* global_scale;
};
cudaError_t launch_quantize(const QuantArgs& a, int sms, cudaStream_t s);

// ---- CUDA-core NVFP4 skinny GEMM (fma.cu) ----------------------------------
// Whole rows per warp, no split-K; K % 32 == 0.  argmax: am_part [M][grid]
// partials and argmax_cnt [row groups] counters (zero between calls).
struct FmaArgs {
  const __nv_bfloat16* A;
  int64_t lda;
  const uint8_t* codes;
  const uint8_t* scales;
  const float* gscale;
  __nv_bfloat16* C;
  int64_t ldc;
  int32_t* argmax_out;
  const int32_t* am_map;
  int M, N, K;
  int rms;
  uint32_t* argmax_cnt;
  int2* am_part;
  int ks;  // warps that share a group of weight rows (K split): 1, 2 or 4
};
// activation rows per CTA for M rows of K (1, 2 or 4, fewer when the staged
// rows would not fit in shared memory); grid.y = ceil(M / that)
int fma_rows_per_cta(int M, int K);
// shared memory of its staged activation rows
size_t fma_smem_bytes(int rows_per_cta, int K);
// weight rows a warp of that kernel takes at once (its loads in flight:
// this many times 528 bytes per 32-K round at K = 2048), for N weight rows
int fma_rows_per_warp(int rows_per_cta, int N);
// Warps that split the K rounds of one group of weight rows (1, 2 or 4),
// given the groups, the 32-chunk rounds of a row and the warps the SMs hold.
int fma_k_split(long groups, int rounds, long warp_slots);
cudaError_t launch_fma(const FmaArgs& a, int grid, int ru, cudaStream_t s, bool pdl);

// MoE layer on the CUDA cores (moe_fma.cu) for T <= kMoeFmaMaxT tokens:
// gate/up + SwiGLU per (token, slot) pair into h, then down + combine.
constexpr int kMoeFmaMaxT = 16;
constexpr int kMoeFmaMaxSlots = 17;                      // k <= 16, + shared
constexpr int kMoeFmaMaxPairs = kMoeFmaMaxT * kMoeFmaMaxSlots;
struct MoeFmaArgs {
  const __nv_bfloat16* x;
  int64_t ldx;
  const int32_t* ids;  // [T, k]
  const float* w;      // [T, k]
  int T, k, E, H, I;
  const uint8_t* gu_codes;  // routed stack
  const uint8_t* gu_scales;
  const uint8_t* dn_codes;
  const uint8_t* dn_scales;
  const float* gu_global;
  const float* dn_global;
  int has_shared;
  const uint8_t* s_gu_codes;  // shared expert (when has_shared)
  const uint8_t* s_gu_scales;
  const uint8_t* s_dn_codes;
  const uint8_t* s_dn_scales;
  const float* s_gu_global;
  const float* s_dn_global;
  __nv_bfloat16* out;
  int64_t ldo;
  int rms, ids_ready;
  float* h;  // [T k + T, I] FP32 scratch
  uint32_t* status;
};
// slots of a token (k + shared) when the down kernel covers them and the
// inter size I, else 0
int moe_fma_slots(int k, int has_shared, int I);
// whether the gate/up step of a batch of T tokens runs by warp MMAs
// (moe_mma_gate_up_kernel: H a multiple of 512, 4 <= T <= 8) or by FMAs
// (moe_fma_gate_up_kernel)
bool moe_gate_up_mma(int H, int T);
cudaError_t launch_moe_fma(const MoeFmaArgs& a, int sms, cudaStream_t s, bool pdl);

// Read-only bandwidth probe (probe.cu): reads bytes (a multiple of 16) of
// buf once; writes one word per CTA (grid words) to sink.
cudaError_t launch_read_probe(const void* buf, size_t bytes, uint32_t* sink, int grid,
                              cudaStream_t s);

// Record the message returned by nvfp4_last_error() for this thread.
void set_last_error(const char* msg);

// The host-side argument checks of nvfp4_gemm_skinny (pointers, shape,
// alignment): NVFP4_OK or the status that call would return.
int check_gemm_args(const void* A, int64_t lda, int M, const struct nvfp4_weight* W,
                    const void* C, int64_t ldc);

}  // namespace nvfp4
