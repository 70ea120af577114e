// NVFP4 weight streaming on the 5th-generation tensor cores (tcgen05).
//
// One persistent kernel runs a program: a sequence of ops, each one of three
// kinds -- the dense skinny GEMM (C = A W^T, optional argmax), the MoE
// gate_up projection (h = silu(gate) * up per routed pair) and the MoE down
// projection with the weighted top-k combine.  A single call of the C ABI is
// a one-op program; a decode step is a program of a few hundred ops.
//
// Tile = 128 weight rows = the 128 lanes of tensor memory: 128 consecutive
// rows (dense, down) or, for gate_up, one 4-D box of 64 gate rows of an
// expert followed by the same 64 up rows.  Stage = one tile x 256 K: 16 KB
// of 128B-swizzled E2M1 codes + 2 KB of E4M3 scales.
// Work split: the (tile, stage) units of each op are cut into equal
// contiguous ranges, one per CTA ("stream-K"); a tile split between CTAs is
// reduced by the last CTA to finish it (atomic counter), adding the per-CTA
// partials in CTA order, so results do not depend on timing.
//
// Warp roles (512 threads, four warpgroups; setmaxnreg moves registers to
// the epilogue warpgroup), each walking the whole program:
//   warp 0       TMA producer: streams stages into a shared-memory ring of
//                3..8 stages (full/empty mbarriers), running ahead into the
//                next ops' weights while the current op finishes;
//   warp 1       allocates tensor memory; one thread issues tcgen05.mma:
//                D[128 x N] += A[128 x 16] (tensor memory) * B[N x 16] (shared
//                memory), 16 MMAs per stage, N = tokens rounded up to 16;
//   warps 8-15   decode: warp w owns lane quarter q = w % 4 (tile rows 32q ..
//                32q + 31, lane l = row 32q + l); warps 8-11 the first 128 K
//                of each stage, 12-15 the second.  E2M1 -> FP16 by the hardware convert, times the E4M3
//                block scale (exact in FP16), written to one of three
//                tensor-memory A buffers with tcgen05.st;
//   warps 4-7    epilogue: wait until every CTA finished the previous op
//                (a completion counter per op), stage the activations (B)
//                into shared memory as FP16 with a power-of-two shift per row,
//                read the FP32 accumulator with tcgen05.ld, undo the shift,
//                and run the stream-K reduction and the op's epilogue;
//   warp 2       builds the expert schedule of each MoE layer into one of
//                two shared-memory slots.
//
// Sources: "Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)", "Making decode
// faster": "Skinny matrix multiplies" (split-K decode matmuls, 4-bit weights
// with 16-bit activations), "One environment variable" (fused MoE finalize),
// "What didn't work" (the shared expert kept separate, always on).
#include <cuda_bf16.h>
#include <float.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "sched.cuh"
#include "tc.cuh"

namespace nvfp4 {
namespace {

constexpr int kRows = 128;
constexpr int kGuRows = 64;                    // gate (and up) rows of a gate_up tile
constexpr int kSK = 256;                       // K per stage
constexpr int kCodeBytes = kRows * kSK / 2;    // 16384
constexpr int kDecWarps = 8;
constexpr int kDecChunks = 8 * 4 / kDecWarps;  // 32-K chunks a decode warp converts per stage
constexpr int kEpiWarps = 4;                   // one per tensor-memory lane quarter
constexpr int kEpiThreads = kEpiWarps * 32;
// warpgroup 0: producer (warp 0), MMA (1), scheduler (2), idle (3);
// warpgroup 1: epilogue (4-7); warpgroups 2-3: decode (8-15)
constexpr int kEpiWarp0 = 4;
constexpr int kDecWarp0 = 8;
// arrivals that release a schedule slot: producer, MMA thread, 8 decode
// warps, 4 epilogue warps
constexpr int kSchedUsers = 2 + kDecWarps + kEpiWarps;
constexpr int kABufs = 3;                      // A operand buffers in tensor memory
constexpr int kACols = kSK / 2;                // tensor-memory columns per A buffer
constexpr int kDCol = kABufs * kACols;         // D buffers at columns 384, 416, 448, 480
constexpr int kDBufs = 4;                      // accumulator buffers (32 columns each)

// Operand type of the MMAs: FP16 x FP16 -> FP32.  The weights are decoded
// to FP16 exactly (a code x scale product has at most 6 significant bits and
// lies in [2^-10, 2688]); the activations are staged as FP16 after a
// power-of-two shift per row that puts the row's largest magnitude in
// [2^14, 2^15) (BF16 rows: exact for every element within 2^31 of the row's
// largest magnitude, smaller ones round to FP16 subnormals or zero; FP32 h
// rows: one rounding).
constexpr uint32_t kTmemCols = 512;

// Dense op kinds (one per weight format) and their compile-time format and
// K per unit.
__host__ __device__ constexpr bool dense_mode(int m) {
  return m == kTcDense || m == kTcDenseF8 || m == kTcDenseBF;
}
__host__ __device__ constexpr int mode_fmt(int m) {
  return m == kTcDenseF8 ? kFmtFp8 : (m == kTcDenseBF ? kFmtBf16 : kFmtNvfp4);
}

static_assert(kTcStageBytes == kCodeBytes + kRows * kSK / 16, "stage size");
static_assert(kTcThreads == (kDecWarp0 + kDecWarps) * 32, "thread count");
static_assert(kDecWarps == 8 && kEpiWarp0 == 4 && kEpiWarps == 4, "warpgroup layout");
// per-warpgroup registers after setmaxnreg: 128 x (96 + 200) + 256 x 96 =
// 62,464 <= 65,536 (512 threads x 128 at launch)
constexpr int kRegsSmall = 96;
constexpr int kRegsEpilogue = 200;
static_assert(128 * (kRegsSmall + kRegsEpilogue) + 256 * kRegsSmall <= 65536, "register split");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void esync() {  // the four epilogue warps
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint32_t* status,
                                              volatile int* abort_flag) {
  const uint32_t a = smem_u32(bar);
  if (mbar_test_wait(a, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (*abort_flag) return false;
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(status, kStatusTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

// The same on a barrier given by its shared-memory address; no abort check
// while the phase is already complete.
__device__ __forceinline__ bool wait_u32(uint32_t a, uint32_t parity, uint32_t* status,
                                         volatile int* abort_flag) {
  if (mbar_test_wait(a, parity)) return !*abort_flag;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (*abort_flag) return false;
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(status, kStatusTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void wait_bar(uint64_t* bar, uint32_t parity, uint32_t* status,
                                         volatile int* abort_flag) {
  if (!*abort_flag) wait_or_abort(bar, parity, status, abort_flag);
}

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

// One 32-row box of a tile: tensor maps and first row.
struct Box {
  const CUtensorMap* mc;
  const CUtensorMap* ms;
  int row;
  int expert;  // gate_up (4-D maps): expert coordinate
};

// Per-launch work description shared by all roles (all fields derived
// deterministically from the arguments and the schedule).
// The op's units are split over G CTAs: relative index r = the CTA
// (blockIdx.x - cta0) mod gridDim.x; r >= G has none.
struct Work {
  int n_tiles, nkb, per_e;
  int U;
  int G, cta0;
  __device__ __forceinline__ int begin(int r) const { return r * U / G; }
  __device__ __forceinline__ int cta_of(int u) const {
    return static_cast<int>(((u + 1) * G - 1) / U);
  }
  __device__ __forceinline__ int rel(int b) const {
    return (b - cta0 + static_cast<int>(gridDim.x)) % static_cast<int>(gridDim.x);
  }
  __device__ __forceinline__ int abs_cta(int r) const { return (r + cta0) % static_cast<int>(gridDim.x); }
};

template <int MODE>
struct Kernel {
  const TcArgs& a;
  const Sched& sc;
  const Work& wk;
  const CUtensorMap *m0, *m1, *m2, *m3;

  // expert of a MoE tile
  __device__ __forceinline__ int tile_expert(int tile) const { return sc.active[tile / wk.per_e]; }

  __device__ __forceinline__ void tile_boxes(int tile, Box (&bx)[4]) const {
    if (dense_mode(MODE)) {
      bx[0] = Box{m0, m1, tile * kRows, 0};  // one 128-row box
    } else if (MODE == kTcGateUp) {
      // one 4-D box: gate rows 64 j .. 64 j + 63 then the same up rows
      const int e = tile_expert(tile), j = tile % wk.per_e;
      const bool sh = (e == a.E);
      bx[0] = Box{sh ? m2 : m0, sh ? m3 : m1, kGuRows * j, sh ? 0 : e};
    } else {
      const int e = sc.active[tile / wk.per_e], nt = tile % wk.per_e;
      const bool sh = (e == a.E);
      bx[0] = Box{sh ? m2 : m0, sh ? m3 : m1, (sh ? 0 : e * a.H) + nt * kRows, 0};  // one 128-row box
    }
  }

  // B operand source of a tile: key identifies the staged rows (restage when
  // it changes), n_rows the number of real rows.
  __device__ __forceinline__ int b_key(int tile) const {
    return MODE == kTcDown ? sc.active[tile / wk.per_e] : 0;
  }
  __device__ __forceinline__ int b_rows(int tile) const {
    if (dense_mode(MODE)) return a.M;
    if (MODE == kTcGateUp) return a.T;
    return sc.cnt[sc.active[tile / wk.per_e]];
  }
  // K per unit: the dense op's format decides; MoE ops stream NVFP4
  __device__ __forceinline__ int uk() const { return tc_unit_k(mode_fmt(MODE)); }
  __device__ __forceinline__ int win_stages() const { return a.win_k / uk(); }
};

// Staged-row bookkeeping shared (identically) by the MMA thread and the
// decode warps: which rows and which stage range the shared-memory B
// operand holds.
struct XState {
  int key = -1, k0 = 0, k1 = 0;
  __device__ __forceinline__ bool covers(int key_, int w0, int w1) const {
    return key == key_ && w0 >= k0 && w1 <= k1;
  }
};

// Units per 256 K: activations are staged in 256-K blocks (one 16-byte load
// per lane and row), so a dense window starts and ends on a multiple of it.
template <int MODE>
__device__ __forceinline__ int units_per_256(const Kernel<MODE>& kk) { return kSK / kk.uk(); }

// Window [w0, w1) of a segment starting at stage w0: MoE, the whole segment
// (its K is staged once); dense, at most win_stages stages from w0 rounded
// down to a 256-K boundary (win_stages is a multiple of 256 K, so the
// rounded window still fits).
template <int MODE>
__device__ __forceinline__ int window_end(const Kernel<MODE>& kk, int w0, int kbe) {
  if (!dense_mode(MODE)) return kbe;
  const int g = units_per_256(kk);
  return min(kbe, w0 / g * g + kk.win_stages());
}

// Stage range restaged when a window is not covered: MoE, the whole K (its
// K is staged once per expert / layer); dense, exactly the window when the
// window capacity is shorter than K or when the CTA's remaining units of the
// op all lie in this tile (one_tile), else the whole K (staged once per op).
template <int MODE>
__device__ __forceinline__ void restage_range(const Kernel<MODE>& kk, int w0, int w1,
                                              bool one_tile, int& k0, int& k1) {
  if (dense_mode(MODE) && (kk.win_stages() < kk.wk.nkb || one_tile)) {
    const int g = units_per_256(kk);  // K % 256 == 0: nkb is a multiple of g
    k0 = w0 / g * g;
    k1 = (w1 + g - 1) / g * g;
  } else {
    k0 = 0;
    k1 = kk.wk.nkb;
  }
}

// Byte offset of 8 staged elements (row n, k .. k + 7, k % 8 == 0) in the
// activation layout: 64-element K-blocks of rb rows, one 128-byte line per
// row, the line's 16-byte chunks swizzled by row (the layout TMA writes with
// the 128-byte swizzle; the block base is 1024-byte aligned).
__device__ __forceinline__ uint32_t xoff(int n, int k, int rb) {
  return static_cast<uint32_t>((k >> 6) * rb * 128 + n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4));
}

// ------------------------------------------------------------ CTA context


// Shared-memory objects and program-wide constants of one CTA, derived on
// use from the aligned shared-memory base and the launch parameters (nothing
// to keep in registers).
struct Cta {
  uint8_t* base;
  const TcProgram& prog;
  uint32_t tmem;
  __device__ __forceinline__ uint64_t* bars() const { return reinterpret_cast<uint64_t*>(base + kTcOffBars); }
  __device__ __forceinline__ uint64_t* ring_full_at(int s) const { return bars() + s; }
  __device__ __forceinline__ uint64_t* ring_empty_at(int s) const { return bars() + kTcMaxStages + s; }
  __device__ __forceinline__ uint64_t* a_full_at(uint32_t b) const { return bars() + 2 * kTcMaxStages + b; }
  __device__ __forceinline__ uint64_t* a_empty_at(uint32_t b) const { return bars() + 2 * kTcMaxStages + kABufs + b; }
  __device__ __forceinline__ uint64_t* d_full_at(uint32_t b) const { return bars() + 2 * kTcMaxStages + 2 * kABufs + 12 + b; }
  __device__ __forceinline__ uint64_t* d_empty_at(uint32_t b) const { return bars() + 2 * kTcMaxStages + 2 * kABufs + 16 + b; }
  __device__ __forceinline__ uint64_t* x_full() const { return bars() + 2 * kTcMaxStages + 2 * kABufs + 4; }
  __device__ __forceinline__ uint64_t* mma_done() const { return bars() + 2 * kTcMaxStages + 2 * kABufs + 5; }
  __device__ __forceinline__ uint64_t* sched_full_at(int b) const { return bars() + 2 * kTcMaxStages + 2 * kABufs + 6 + b; }
  __device__ __forceinline__ uint64_t* sched_empty_at(int b) const { return bars() + 2 * kTcMaxStages + 2 * kABufs + 8 + b; }
  __device__ __forceinline__ uint64_t* x_tma() const { return bars() + 2 * kTcMaxStages + 2 * kABufs + 10; }
  __device__ __forceinline__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(base + kTcOffMisc); }
  __device__ __forceinline__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(base + kTcOffMisc + 4); }
  __device__ __forceinline__ volatile int* bcast() const { return reinterpret_cast<volatile int*>(base + kTcOffMisc + 8); }
  // ops whose epilogue this CTA has finished (the decode warps start an op's
  // weights only after the previous op's epilogue: its tail and the next
  // op's activation staging then run without the decode competing for issue)
  __device__ __forceinline__ volatile int* epi_done() const { return reinterpret_cast<volatile int*>(base + kTcOffMisc + 448); }
  __device__ __forceinline__ int* sig() const { return reinterpret_cast<int*>(base + kTcOffMisc + 64); }
  __device__ __forceinline__ float* rms() const { return reinterpret_cast<float*>(base + kTcOffMisc + 192); }
  __device__ __forceinline__ float* ep() const { return reinterpret_cast<float*>(base + kTcOffEp); }
  // the epilogue's copy of the current op's arguments (read from shared
  // memory instead of the device op table)
  __device__ __forceinline__ const TcArgs& args() const {
    return *reinterpret_cast<const TcArgs*>(base + kTcOffArgs);
  }
  // the current dense op's matrix scale, loaded before its completion wait
  __device__ __forceinline__ volatile float* op_scale() const {
    return reinterpret_cast<volatile float*>(base + kTcOffMisc + 456);
  }
  __device__ __forceinline__ uint8_t* xs() const { return base + prog.x_offset; }
  __device__ __forceinline__ uint8_t* ring() const { return base + prog.ring_offset; }
  __device__ __forceinline__ uint8_t* sched() const { return base + prog.sched_offset; }
  __device__ __forceinline__ int n_stages() const { return prog.n_stages; }
  __device__ __forceinline__ int sched_bytes() const { return prog.sched_bytes; }
  __device__ __forceinline__ int sched_slots() const { return prog.sched_slots; }
  __device__ __forceinline__ uint32_t* status() const { return prog.status; }
  __device__ __forceinline__ bool aborted() const { return *abort_flag() != 0; }
};
static_assert(2 * kTcMaxStages + 2 * kABufs + 12 + 2 * kDBufs <= kTcOffMisc / 8, "barrier area");
static_assert(sizeof(TcArgs) <= kTcArgsBytes && sizeof(TcArgs) % 16 == 0, "argument copy");
static_assert(alignof(TcArgs) <= 16, "argument copy");
static_assert(kDCol + 32 * kDBufs <= static_cast<int>(kTmemCols), "tensor memory columns");

__device__ __forceinline__ const TcOp& op_at(const TcProgram& p, int i) {
  return p.ops ? p.ops[i] : p.inline_ops[i];
}

// The expert schedule an MoE op uses: every role keeps the same count of
// schedules started, so all of them agree on the slot.  A slot is rebuilt
// only after all kSchedUsers arrivals released its previous schedule.
struct SchedCursor {
  int idx = -1;
  __device__ __forceinline__ Sched acquire(const Cta& c, const TcArgs& a) {
    if (a.new_sched) {
      ++idx;
      wait_bar(c.sched_full_at(idx % c.sched_slots()), (idx / c.sched_slots()) & 1, c.status(),
               c.abort_flag());
    }
    const int slot = idx < 0 ? 0 : idx % c.sched_slots();
    return sched_layout(c.sched() + slot * c.sched_bytes(), a.E, a.T * a.k);
  }
  // arrive: this thread speaks for its warp (or is the role's only thread)
  __device__ __forceinline__ void release(const Cta& c, const TcArgs& a, bool arrive) {
    if (a.last_sched_use && arrive && idx >= 0) mbar_arrive(c.sched_empty_at(idx % c.sched_slots()));
  }
};

// Units of an op and the contiguous range [u0, u1) of this CTA.  After an
// abort the schedule may be incomplete: no units then.
template <int MODE>
__device__ __forceinline__ Work make_work(const TcArgs& a, const Sched& sc, const Cta& c,
                                          int& u0, int& u1) {
  Work wk{};
  if (dense_mode(MODE)) {
    wk.n_tiles = (a.N + kRows - 1) / kRows;
    wk.nkb = a.K / tc_unit_k(mode_fmt(MODE));
  } else {
    const int na = c.aborted() ? 0 : min(max(*sc.n_active, 0), a.E + 1);
    if (MODE == kTcGateUp) {
      wk.per_e = a.I / kGuRows;
      wk.n_tiles = na * wk.per_e;
      wk.nkb = a.H / kSK;
    } else {
      wk.per_e = a.H / kRows;
      wk.n_tiles = na * wk.per_e;
      wk.nkb = a.I / kSK;
    }
  }
  wk.U = wk.n_tiles * wk.nkb;
  wk.G = min(a.n_ctas, wk.U);
  wk.cta0 = a.cta0;
  const int b = wk.rel(blockIdx.x);
  const bool active = b < wk.G && !c.aborted();
  u0 = active ? wk.begin(b) : 0;
  u1 = active ? wk.begin(b + 1) : 0;
  return wk;
}

// Wait until *ctr reaches target (every CTA finished an op), bounded; gives
// up at once if another CTA already timed out.
__device__ __forceinline__ void grid_wait(const uint32_t* ctr, uint32_t target, uint32_t* status,
                                          volatile int* abort_flag) {
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (ld_acquire_gpu(ctr) >= target) break;
    if (*abort_flag) return;
    if (*reinterpret_cast<volatile uint32_t*>(status) & kStatusTimeout) {
      *abort_flag = 1;
      return;
    }
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(status, kStatusTimeout);
      *abort_flag = 1;
      return;
    }
  }
}

// Tensor maps of the device op table were written by the host before the
// launch; order them for the tensor-map proxy before the first copy.
__device__ __forceinline__ void acquire_tensormap(const CUtensorMap* m) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(m) : "memory");
}

// BF16 activation rows staged with asynchronous copies and rolled loops
// (little code: the staging runs once per op, after other roles' code has
// passed through the instruction cache).  Rows [0, nr) of the K range
// [kbeg, kbeg + klen) land as BF16 in the staged layout, rows [nr, rb) as
// zeros; then per row the largest magnitude (and, with rms, the sum of
// squares), and unless raw the in-place conversion to FP16 times 2^sig[n].
// Each lane walks the 16-byte chunks lane, lane + 32, ... of its warp's
// rows in that order, as the register path and the dense RMS pass do (same
// sums, bit for bit).  The four epilogue warps; klen % 256 == 0.
__device__ __forceinline__ void stage_rows_async(const __nv_bfloat16* base, int64_t ld, int nr,
                                                 int rb, int kbeg, int klen, uint32_t xs,
                                                 int* sig, float* rms, int ew, int lane,
                                                 bool raw) {
  const int cpr = klen >> 3;  // 16-byte chunks per row
  const int etid = ew * 32 + lane;
#pragma unroll 1
  for (int i = etid; i < rb * cpr; i += kEpiThreads) {
    const int n = i / cpr, kc = i - n * cpr;
    const __nv_bfloat16* src = base + static_cast<size_t>(n < nr ? n : 0) * ld + kbeg + 8 * kc;
    cp_async_16(xs + xoff(n, 8 * kc, rb), src, n < nr ? 16u : 0u);
  }
  cp_async_wait_all();
  esync();
#pragma unroll 1
  for (int n = ew; n < rb; n += kEpiWarps) {
    if (n >= nr) {
      if (lane == 0) sig[n] = 0;
      continue;
    }
    uint32_t mx = 0u;
    float sq = 0.0f;
#pragma unroll 4
    for (int kc = lane; kc < cpr; kc += 32) {
      const uint4 v = ld_shared_v4(xs + xoff(n, 8 * kc, rb));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        mx = __vmaxu2(mx, w[j] & 0x7FFF7FFFu);
        if (rms) {
          const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
          sq = fmaf(lo, lo, fmaf(hi, hi, sq));
        }
      }
    }
    const float m = warp_max(fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xFFFF0000u)));
    const int sh = f16_row_shift(m);
    if (rms) {
      if (m > kSumsqSafeMax) {  // (warp-uniform, rare) the shifted squares
        const int h1 = (sh > 126 || sh < -126) ? sh / 2 : sh;
        const float f1 = exp2i(h1), f2 = exp2i(sh - h1);
        sq = 0.0f;
#pragma unroll 1
        for (int kc = lane; kc < cpr; kc += 32) {
          const uint4 v = ld_shared_v4(xs + xoff(n, 8 * kc, rb));
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(w[j] << 16) * f1 * f2;
            const float hi = __uint_as_float(w[j] & 0xFFFF0000u) * f1 * f2;
            sq = fmaf(lo, lo, fmaf(hi, hi, sq));
          }
        }
      }
      sq = warp_sum(sq);
      if (lane == 0) rms[n] = m > kSumsqSafeMax ? rms_factor(sq, sh, klen) : rms_plain(sq, klen);
    }
    if (lane == 0) sig[n] = raw ? 0 : sh;
    if (raw) continue;
    const int h1 = (sh > 126 || sh < -126) ? sh / 2 : sh;
    const float f1 = exp2i(h1), f2 = exp2i(sh - h1);
    const bool two = h1 != sh;
#pragma unroll 4
    for (int kc = lane; kc < cpr; kc += 32) {
      const uint32_t addr = xs + xoff(n, 8 * kc, rb);
      const uint4 v = ld_shared_v4(addr);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float lo = __uint_as_float(w[j] << 16) * f1, hi = __uint_as_float(w[j] & 0xFFFF0000u) * f1;
        if (two) {
          lo *= f2;
          hi *= f2;
        }
        o[j] = pack_f16x2(lo, hi);
      }
      st_shared_v4(addr, make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
}

// One row of the staged operand, held in registers: the lane's 16-byte
// loads of row n (chunks kc = lane + 32 i of 8 elements; FP32 rows take two
// loads a chunk), at most kStageSlots loads.
constexpr int kStageSlots = 16;

template <typename T>
__device__ __forceinline__ void stage_row_load(const T* row, int n, int nr, int kbeg, int ppr,
                                               int lane, uint4 (&b)[kStageSlots]) {
  constexpr int kLd = sizeof(T) == 2 ? 1 : 2;
#pragma unroll
  for (int i = 0; i < kStageSlots; ++i) {
    b[i] = make_uint4(0u, 0u, 0u, 0u);
    if (i < ppr && n < nr) {
      const int kc = lane + 32 * (i / kLd), sub = i % kLd;
      b[i] = __ldcg(reinterpret_cast<const uint4*>(row + kbeg + 8 * kc + 4 * sub));
    }
  }
}

// Largest magnitude (as a float) of a row's loads and, when want_sq, the
// plain FP32 sum of their squares (BF16 rows only).
template <typename T>
__device__ __forceinline__ float stage_row_max(const uint4 (&b)[kStageSlots], int ppr, bool want_sq,
                                               float& sq) {
  uint32_t mx = 0u;  // BF16: the largest |x| of each half as bits (|x| orders like its bits)
  float mf = 0.0f;
  sq = 0.0f;
#pragma unroll
  for (int i = 0; i < kStageSlots; ++i)
    if (i < ppr) {
      const uint32_t w[4] = {b[i].x, b[i].y, b[i].z, b[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if constexpr (sizeof(T) == 2) {
          mx = __vmaxu2(mx, w[j] & 0x7FFF7FFFu);
          if (want_sq) {
            const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
            sq = fmaf(lo, lo, fmaf(hi, hi, sq));
          }
        } else {
          mf = fmaxf(mf, fabsf(__uint_as_float(w[j])));
        }
      }
    }
  if constexpr (sizeof(T) == 2) return fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xFFFF0000u));
  return mf;
}

// Sum of the squares of a BF16 row's loads times 2^(2 sh): the row's shift
// puts its largest square near 2^29, so the sum neither overflows nor loses
// the row's significant terms, whatever the row's magnitude.  Scaling by a
// power of two commutes with the roundings, so for rows inside FP32's range
// the result is the plain sum of squares times 2^(2 sh).
__device__ __forceinline__ float stage_row_sumsq(const uint4 (&b)[kStageSlots], int ppr, int sh) {
  const int h1 = (sh > 126 || sh < -126) ? sh / 2 : sh;
  const float f1 = exp2i(h1), f2 = exp2i(sh - h1);
  float sq = 0.0f;
#pragma unroll
  for (int i = 0; i < kStageSlots; ++i)
    if (i < ppr) {
      const uint32_t w[4] = {b[i].x, b[i].y, b[i].z, b[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = __uint_as_float(w[j] << 16) * f1 * f2;
        const float hi = __uint_as_float(w[j] & 0xFFFF0000u) * f1 * f2;
        sq = fmaf(lo, lo, fmaf(hi, hi, sq));
      }
    }
  return sq;
}

// The FP16 conversion of a row's loads times 2^sh, stored into the staged
// layout: load i of lane l holds chunk kc = l + 32 i / kLd, whose 16-byte
// slot is at base(n, l) + (i / kLd) * 4 * rb * 128 (xoff with k = 8 kc).
template <typename T>
__device__ __forceinline__ void stage_row_store(const uint4 (&b)[kStageSlots], int n, int rb,
                                                int ppr, int sh, uint32_t xs, int lane, bool raw) {
  constexpr int kLd = sizeof(T) == 2 ? 1 : 2;
  if constexpr (sizeof(T) == 2) {
    if (raw) {  // BF16 operand: the loads as they are
      const uint32_t base = xs + xoff(n, 8 * lane, rb);
      const uint32_t step = static_cast<uint32_t>(4 * rb * 128);
#pragma unroll
      for (int i = 0; i < kStageSlots; ++i)
        if (i < ppr) st_shared_v4(base + static_cast<uint32_t>(i) * step, b[i]);
      return;
    }
  }
  // one factor when 2^sh is a normal float, else two steps
  const int h1 = (sh > 126 || sh < -126) ? sh / 2 : sh;
  const float f1 = exp2i(h1), f2 = exp2i(sh - h1);
  const bool two = h1 != sh;
  const uint32_t base = xs + xoff(n, 8 * lane, rb);
  const uint32_t step = static_cast<uint32_t>(4 * rb * 128);
#pragma unroll
  for (int i = 0; i < kStageSlots; i += kLd)
    if (i < ppr) {
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float lo, hi;
        if constexpr (sizeof(T) == 2) {
          const uint32_t w = j == 0 ? b[i].x : j == 1 ? b[i].y : j == 2 ? b[i].z : b[i].w;
          lo = __uint_as_float(w << 16);
          hi = __uint_as_float(w & 0xFFFF0000u);
        } else {
          const uint4& v = b[i + (j >> 1)];
          lo = __uint_as_float((j & 1) ? v.z : v.x);
          hi = __uint_as_float((j & 1) ? v.w : v.y);
        }
        lo *= f1;
        hi *= f1;
        if (two) {
          lo *= f2;
          hi *= f2;
        }
        o[j] = pack_f16x2(lo, hi);
      }
      st_shared_v4(base + static_cast<uint32_t>(i / kLd) * step, make_uint4(o[0], o[1], o[2], o[3]));
    }
}

// Rows n0 and n1 (n1 may be past rb): statistics of both, their warp
// reductions interleaved, the shifts, rms and the stores.
template <typename T>
__device__ __forceinline__ void stage_row_pair(const uint4 (&b0)[kStageSlots],
                                               const uint4 (&b1)[kStageSlots], int n0, int n1,
                                               int nr, int rb, int ppr, uint32_t xs, int* sig,
                                               float* rms, int klen, int lane, bool raw) {
  const bool has1 = n1 < rb;
  const bool want_sq = sizeof(T) == 2 && rms != nullptr;
  float s0, s1 = 0.0f;
  float m0 = stage_row_max<T>(b0, ppr, want_sq, s0);
  float m1 = has1 ? stage_row_max<T>(b1, ppr, want_sq, s1) : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    if (want_sq) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, o);
      s1 += __shfl_xor_sync(0xffffffffu, s1, o);
    }
  }
  // the FP16 shift of each row (a BF16 operand keeps its rows unshifted;
  // the RMS factors below still use the shift a row would have)
  const int sh0 = n0 < nr ? f16_row_shift(m0) : 0;
  const int sh1 = n1 < nr ? f16_row_shift(m1) : 0;
  if constexpr (sizeof(T) == 2) {
    if (want_sq) {
      // the plain sum of squares cannot overflow below kSumsqSafeMax; a row
      // above it (warp-uniform, rare) sums its shifted squares instead
      if (m0 > kSumsqSafeMax) s0 = warp_sum(stage_row_sumsq(b0, ppr, sh0));
      if (has1 && m1 > kSumsqSafeMax) s1 = warp_sum(stage_row_sumsq(b1, ppr, sh1));
      if (lane == 0) {
        if (n0 < nr) rms[n0] = m0 > kSumsqSafeMax ? rms_factor(s0, sh0, klen) : rms_plain(s0, klen);
        if (has1 && n1 < nr)
          rms[n1] = m1 > kSumsqSafeMax ? rms_factor(s1, sh1, klen) : rms_plain(s1, klen);
      }
    }
  }
  if (lane == 0) {
    sig[n0] = raw ? 0 : sh0;
    if (has1) sig[n1] = raw ? 0 : sh1;
  }
  stage_row_store<T>(b0, n0, rb, ppr, sh0, xs, lane, raw);
  if (has1) stage_row_store<T>(b1, n1, rb, ppr, sh1, xs, lane, raw);
}

// Activations staged through registers in one pass: BF16 (dense A, MoE x)
// or FP32 (MoE h) rows [0, nr) of the K range [kbeg, kbeg + klen) read with
// 16-byte loads, converted to FP16 times 2^sig[n] (the shift that puts row
// n's largest magnitude in [2^14, 2^15); exact for BF16 elements within 2^31
// of the largest (smaller ones round to FP16 subnormals), one rounding for
// FP32) into the 128-byte swizzled K-block layout, rows [nr, rb) zero; with
// rms != nullptr also rms[n] = 1/sqrt(mean x^2 + 1e-6) over the staged range.
// Warp ew takes rows ew, ew + 4, ... two at a time (their loads in flight
// together) when a row needs at most 8 loads a lane.  The four epilogue
// warps; klen / 256 * (4 / sizeof(T)) <= kStageSlots.
template <typename T, typename RowFn>
__device__ __forceinline__ void stage_rows(RowFn rowp, int nr, int rb, int kbeg, int klen,
                                           uint32_t xs, int* sig, float* rms, int ew, int lane,
                                           bool raw = false) {
  constexpr int kLd = sizeof(T) == 2 ? 1 : 2;
  const int ppr = (klen >> 8) * kLd;  // loads per lane per row
  if (ppr * 2 <= kStageSlots) {
    for (int n = ew; n < rb; n += 2 * kEpiWarps) {
      uint4 b0[kStageSlots], b1[kStageSlots];
      const int n1 = n + kEpiWarps;
      stage_row_load<T>(rowp(n < nr ? n : 0), n, nr, kbeg, ppr, lane, b0);
      stage_row_load<T>(rowp(n1 < nr ? n1 : 0), n1, nr, kbeg, ppr, lane, b1);
      stage_row_pair<T>(b0, b1, n, n1, nr, rb, ppr, xs, sig, rms, klen, lane, raw);
    }
  } else {
    for (int n = ew; n < rb; n += kEpiWarps) {
      uint4 b0[kStageSlots];
      stage_row_load<T>(rowp(n < nr ? n : 0), n, nr, kbeg, ppr, lane, b0);
      stage_row_pair<T>(b0, b0, n, rb, nr, rb, ppr, xs, sig, rms, klen, lane, raw);
    }
  }
}

// ------------------------------------------------------------ roles, per op

// (The producer and epilogue bodies are not inlined: with every role inlined
// into the kernel, nvcc 13.0's device front end crashes on this file now and
// then; the decode and MMA loops are inlined, which measurably matters.)
//
// The producer warp, one op.  Converged like the MMA warp: lane 0 waits for
// a free ring stage, one elected lane issues the copies.  Dense and down
// tiles are 128 consecutive weight rows: one box of codes and one of scales
// per stage; a gate_up tile is four 32-row boxes.
template <int MODE>
__device__ __noinline__ void produce_op(const Cta& c, const TcOp& op, bool table, int lane,
                                           SchedCursor& cur, int& stage, uint32_t& phase,
                                           int& issued, uint64_t pol) {
  const TcArgs& a = op.a;
  Sched sc{};
  if (!dense_mode(MODE)) sc = cur.acquire(c, op.a);
  int u0, u1;
  const Work wk = make_work<MODE>(a, sc, c, u0, u1);
  const Kernel<MODE> kk{a, sc, wk, &op.maps[0], &op.maps[1], &op.maps[2], &op.maps[3]};
  if (u0 < u1 && tc::elect_one()) {
    const int nm = dense_mode(MODE) ? (MODE == kTcDense ? 2 : 1) : 4;
    for (int m = 0; m < nm; ++m) {
      if (table) acquire_tensormap(&op.maps[m]);
      prefetch_tensormap(&op.maps[m]);
    }
  }
  __syncwarp();
  // everything the loop touches lives in registers: shared-memory addresses
  // as 32-bit values, the stage counters advanced without divisions
  const uint32_t ring_u = smem_u32(c.ring());
  const uint32_t full_u = smem_u32(c.ring_full_at(0));
  const uint32_t empty_u = smem_u32(c.ring_empty_at(0));
  const int n_stages = c.n_stages();
  volatile int* const abort_flag = c.abort_flag();
  uint32_t* const status = c.status();
  const int nkb = wk.nkb;
  constexpr int fmt = mode_fmt(MODE);
  int tile = u0 < u1 ? static_cast<int>(u0 / nkb) : 0;
  int kb = u0 < u1 ? u0 - tile * nkb : 0;
  int cur_tile = -1;
  Box bx[4];
  for (int u = u0; u < u1; ++u) {
    if (tile != cur_tile) {
      kk.tile_boxes(tile, bx);
      cur_tile = tile;
    }
    bool ok = true;
    if (lane == 0) ok = wait_u32(empty_u + 8u * stage, phase ^ 1u, status, abort_flag);
    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
    if (tc::elect_one()) {
      const uint32_t full = full_u + 8u * stage;
      const uint32_t st = ring_u + static_cast<uint32_t>(stage) * kTcStageBytes;
      if (fmt != kFmtNvfp4) {
        // one 128 x 128-byte box: 128 K of E4M3 bytes or 64 K of BF16
        // (the x coordinate counts elements of the map's type)
        mbar_arrive_expect_tx_u32(full, kCodeBytes);
        tma_load_2d_u32(st, bx[0].mc, kb * (fmt == kFmtFp8 ? 128 : 64), bx[0].row, full, pol);
      } else if (MODE == kTcGateUp) {
        mbar_arrive_expect_tx_u32(full, kTcStageBytes);
        tma_load_4d_u32(st, bx[0].mc, kb * (kSK / 2), bx[0].row, 0, bx[0].expert, full, pol);
        tma_load_4d_u32(st + kCodeBytes, bx[0].ms, kb * (kSK / 16), bx[0].row, 0, bx[0].expert, full,
                        pol);
      } else {
        mbar_arrive_expect_tx_u32(full, kTcStageBytes);
        tma_load_2d_u32(st, bx[0].mc, kb * (kSK / 2), bx[0].row, full, pol);
        tma_load_2d_u32(st + kCodeBytes, bx[0].ms, kb * (kSK / 16), bx[0].row, full, pol);
      }
    }
    __syncwarp();
    ++issued;
    if (++stage == n_stages) {
      stage = 0;
      phase ^= 1u;
    }
    if (++kb == nkb) {
      kb = 0;
      ++tile;
    }
  }
  if (!dense_mode(MODE)) cur.release(c, op.a, lane == 0);
}

// The MMA warp, one op.  The warp stays converged: lane 0 waits on the
// barriers, then one elected lane issues the stage's MMAs and the commits
// (a tcgen05.mma issued from a divergent single-lane loop is several times
// slower).  NVFP4 and FP8 units take A from a tensor-memory buffer the
// decode warps filled; BF16 units take A straight from the ring slot (the
// MMA then frees the slot: one commit per decode-warp arrival the slot's
// barrier counts).  The warp follows the ring position of every unit.
template <int MODE>
__device__ __forceinline__ void mma_op(const Cta& c, const TcOp& op, SchedCursor& cur, int lane,
                                       uint32_t& acount, uint32_t& dcount, uint32_t& xcount,
                                       int& rstage, uint32_t& rphase) {
  const TcArgs& a = op.a;
  Sched sc{};
  if (!dense_mode(MODE)) sc = cur.acquire(c, op.a);
  int u0, u1;
  const Work wk = make_work<MODE>(a, sc, c, u0, u1);
  const Kernel<MODE> kk{a, sc, wk, &op.maps[0], &op.maps[1], &op.maps[2], &op.maps[3]};
  XState xst;
  const uint32_t xs_addr = smem_u32(c.xs());
  constexpr int uk = tc_unit_k(mode_fmt(MODE));
  constexpr bool a_smem = MODE == kTcDenseBF;
  const uint32_t ring_u = smem_u32(c.ring());
  const int n_stages = c.n_stages();
  for (int u = u0; u < u1;) {
    if (__any_sync(0xffffffffu, c.aborted())) break;
    const int tile = static_cast<int>(u / wk.nkb);
    const int kbs = static_cast<int>(u % wk.nkb);
    const int kbe = min(wk.nkb, kbs + (u1 - u));
    const int key = kk.b_key(tile);
    const int nr = kk.b_rows(tile);
    const uint32_t idesc = tc::idesc_f16(nr <= 16 ? 16 : 32, a_smem);
    const int rb = tc_xrows(nr);
    const uint32_t sbo = rb == 8 ? 0u : 1024u;  // 8 staged rows: MMA rows 8..15 repeat 0..7
    const bool one_tile = u1 <= (tile + 1) * wk.nkb;
    for (int w0 = kbs; w0 < kbe;) {
      const int w1 = window_end(kk, w0, kbe);
      if (!xst.covers(key, w0, w1)) {
        restage_range(kk, w0, w1, one_tile, xst.k0, xst.k1);
        xst.key = key;
        if (lane == 0) wait_bar(c.x_full(), xcount & 1u, c.status(), c.abort_flag());
        __syncwarp();
        ++xcount;
      }
      const uint32_t db = dcount % kDBufs;
      if (lane == 0) wait_bar(c.d_empty_at(db), ((dcount / kDBufs) & 1u) ^ 1u, c.status(), c.abort_flag());
      __syncwarp();
      const uint32_t d_t = c.tmem + kDCol + 32u * db;
      for (int kb = w0; kb < w1; ++kb) {
        const uint32_t ab = acount % kABufs;
        const uint32_t rslot = ring_u + static_cast<uint32_t>(rstage) * kTcStageBytes;
        if (lane == 0) {
          if (a_smem)
            wait_bar(c.ring_full_at(rstage), rphase, c.status(), c.abort_flag());
          else
            wait_bar(c.a_full_at(ab), (acount / kABufs) & 1u, c.status(), c.abort_flag());
        }
        __syncwarp();
        tc::fence_after_sync();
        const bool run = !__any_sync(0xffffffffu, c.aborted());
        if (tc::elect_one()) {
          if (run) {
            // unit kb = uk / 64 K-blocks of 64 elements of rb staged rows;
            // K step j of 16: A columns + 8 j (tensor memory) or + 32 j bytes
            // (shared memory), B block j / 4 at + 32 (j % 4) bytes
            // (descriptor address field in 16-byte units; no carry: < 256 KB)
            const uint64_t b0 = tc::smem_desc_sw128(
                xs_addr + static_cast<uint32_t>((kb - xst.k0) * (uk / 64) * rb * 128), sbo);
            const uint32_t blk = static_cast<uint32_t>(rb * 128 / 16);
            // (fixed trip counts: the issue loops stay unrolled)
            if (a_smem) {  // BF16: 64 K a unit
              const uint64_t a0 = tc::smem_desc_sw128(rslot, 1024u);
              tc::mma_f16_ss(d_t, a0, b0, idesc, kb > w0 ? 1u : 0u);
#pragma unroll
              for (int j = 1; j < 4; ++j)
                tc::mma_f16_ss(d_t, a0 + static_cast<uint64_t>(2 * j),
                               b0 + static_cast<uint64_t>(2 * j), idesc, 1u);
            } else {
              const uint32_t a_t = c.tmem + kACols * ab;
              tc::mma_f16_ts(d_t, a_t, b0, idesc, kb > w0 ? 1u : 0u);
              if (uk == kSK) {  // NVFP4: 256 K a unit
#pragma unroll
                for (int j = 1; j < kSK / 16; ++j)
                  tc::mma_f16_ts(d_t, a_t + 8 * j,
                                 b0 + static_cast<uint64_t>((j >> 2) * blk + 2 * (j & 3)), idesc,
                                 1u);
              } else {  // FP8: 128 K a unit
#pragma unroll
                for (int j = 1; j < 8; ++j)
                  tc::mma_f16_ts(d_t, a_t + 8 * j,
                                 b0 + static_cast<uint64_t>((j >> 2) * blk + 2 * (j & 3)), idesc,
                                 1u);
              }
            }
          }
          if (a_smem) {
#pragma unroll
            for (int i = 0; i < kDecWarps; ++i) tc::commit(c.ring_empty_at(rstage));
          } else {
            tc::commit(c.a_empty_at(ab));
          }
        }
        __syncwarp();
        if (!a_smem) ++acount;
        if (++rstage == n_stages) {
          rstage = 0;
          rphase ^= 1u;
        }
      }
      if (tc::elect_one()) tc::commit(c.d_full_at(db));
      __syncwarp();
      ++dcount;
      w0 = w1;
    }
    u += kbe - kbs;
  }
  if (!dense_mode(MODE)) cur.release(c, op.a, lane == 0);
}

template <int MODE>
__device__ __forceinline__ void decode_op(const Cta& c, const TcOp& op, SchedCursor& cur,
                                          int warp, int lane, uint32_t& acount, int& rstage,
                                          uint32_t& rphase) {
  Sched sc{};
  if (!dense_mode(MODE)) sc = cur.acquire(c, op.a);
  int u0, u1;
  make_work<MODE>(op.a, sc, c, u0, u1);
  constexpr int fmt = mode_fmt(MODE);
  if (fmt == kFmtBf16) {
    // the MMA reads BF16 weights from the ring itself: only follow the ring
    const int n = u1 > u0 ? u1 - u0 : 0;
    rstage += static_cast<int>(n % c.n_stages());
    rphase ^= static_cast<uint32_t>((n / c.n_stages()) & 1);
    if (rstage >= c.n_stages()) {
      rstage -= c.n_stages();
      rphase ^= 1u;
    }
    return;
  }
  // warp dw decodes lane quarter q (tile rows 32q .. 32q + 31), chunks
  // [c0, c0 + kDecChunks) of the stage's 8 16-byte chunks of a row (NVFP4:
  // 32 K each; FP8: 16 K each)
  const int dw = warp - kDecWarp0, q = warp & 3, c0 = (dw >> 2) * kDecChunks;
  const uint32_t lane_addr = c.tmem + (static_cast<uint32_t>(32 * q) << 16);
  // loop constants in registers (shared-memory addresses as 32-bit values)
  const uint32_t ring_u = smem_u32(c.ring());
  const uint32_t rfull_u = smem_u32(c.ring_full_at(0));
  const uint32_t rempty_u = smem_u32(c.ring_empty_at(0));
  const uint32_t afull_u = smem_u32(c.a_full_at(0));
  const uint32_t aempty_u = smem_u32(c.a_empty_at(0));
  const int n_stages = c.n_stages();
  volatile int* const abort_flag = c.abort_flag();
  uint32_t* const status = c.status();
  // this lane's row of a stage: codes at row * 128 (16-byte chunks swizzled
  // by row % 8), its scale bytes (two per chunk) at 16 * row + 2 * c0
  const uint32_t code_off = static_cast<uint32_t>(q * (kCodeBytes / 4) + lane * 128);
  const uint32_t scale_off = static_cast<uint32_t>(kCodeBytes + q * 512 + lane * 16 + 2 * c0);
  uint32_t chunk_off[kDecChunks];
#pragma unroll
  for (int ci = 0; ci < kDecChunks; ++ci) chunk_off[ci] = code_off + (((c0 + ci) ^ (lane & 7)) << 4);
  uint32_t ab = acount % kABufs, aph = (acount / kABufs) & 1u;
  // A buffer whose tensor-memory stores are issued but not yet waited for:
  // announced (a_full) after the first chunk of the next stage is converted,
  // so the wait for the stores overlaps that conversion
  int pend = -1;
  for (int u = u0; u < u1; ++u) {
    if (!wait_u32(rfull_u + 8u * rstage, rphase, status, abort_flag)) break;
    const uint32_t st = ring_u + static_cast<uint32_t>(rstage) * kTcStageBytes;
    if (fmt == kFmtFp8) {
      // E4M3 -> FP16 (hardware convert, exact); the matrix's one scale is
      // applied to the accumulator
      uint4 cw[kDecChunks];
#pragma unroll
      for (int ci = 0; ci < kDecChunks; ++ci) cw[ci] = ld_shared_v4(st + chunk_off[ci]);
      __syncwarp();
      if (lane == 0) mbar_arrive_u32(rempty_u + 8u * rstage);
      if (!wait_u32(aempty_u + 8u * ab, aph ^ 1u, status, abort_flag)) break;
      tc::fence_after_sync();
#pragma unroll
      for (int ci = 0; ci < kDecChunks; ++ci) {
        const uint32_t wds[4] = {cw[ci].x, cw[ci].y, cw[ci].z, cw[ci].w};
        uint32_t v[8];
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) e4m3x4_to_f16x2(wds[wi], v[2 * wi], v[2 * wi + 1]);
        if (ci == 0 && pend >= 0) {
          tc::wait_st();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_u32(afull_u + 8u * static_cast<uint32_t>(pend));
          pend = -1;
        }
        tc::st_x8(lane_addr + kACols * ab + 8 * (c0 + ci), v);
      }
    } else {
    // all shared-memory reads of this stage first (their latency overlaps)
    uint32_t sbw[kDecChunks / 2];
    if (kDecChunks == 8) {
      const uint4 sb = ld_shared_v4(st + scale_off);
      sbw[0] = sb.x;
      sbw[kDecChunks / 2 > 1 ? 1 : 0] = sb.y;
      sbw[kDecChunks / 2 > 2 ? 2 : 0] = sb.z;
      sbw[kDecChunks / 2 > 3 ? 3 : 0] = sb.w;
    } else {
      const uint2 sb = ld_shared_v2(st + scale_off);
      sbw[0] = sb.x;
      sbw[kDecChunks / 2 > 1 ? 1 : 0] = sb.y;
    }
    uint4 cw[kDecChunks];
#pragma unroll
    for (int ci = 0; ci < kDecChunks; ++ci) cw[ci] = ld_shared_v4(st + chunk_off[ci]);
    __syncwarp();
    if (lane == 0) mbar_arrive_u32(rempty_u + 8u * rstage);
    if (!wait_u32(aempty_u + 8u * ab, aph ^ 1u, status, abort_flag)) break;
    tc::fence_after_sync();
    // E2M1 -> FP16 (hardware convert) times the E4M3 block scale as FP16:
    // the product is exact (at most 6 significant bits, magnitude in
    // [2^-10, 2688])
#pragma unroll
    for (int ci = 0; ci < kDecChunks; ++ci) {
      const uint32_t sw = sbw[ci >> 1] >> (16 * (ci & 1));
      const uint32_t wds[4] = {cw[ci].x, cw[ci].y, cw[ci].z, cw[ci].w};
      uint32_t s_lo, s_hi;
      e4m3x2_bcast_f16x2(sw, s_lo, s_hi);
      uint32_t v[16];
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        e2m1x8_to_f16x2(wds[wi], v[4 * wi], v[4 * wi + 1], v[4 * wi + 2], v[4 * wi + 3]);
        const uint32_t sv = wi < 2 ? s_lo : s_hi;
#pragma unroll
        for (int e = 0; e < 4; ++e) v[4 * wi + e] = hmul2(v[4 * wi + e], sv);
      }
      if (ci == 0 && pend >= 0) {
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_u32(afull_u + 8u * static_cast<uint32_t>(pend));
        pend = -1;
      }
      tc::st_x16(lane_addr + kACols * ab + 16 * (c0 + ci), v);
    }
    }
    pend = static_cast<int>(ab);
    ++acount;
    if (++ab == kABufs) {
      ab = 0;
      aph ^= 1u;
    }
    if (++rstage == n_stages) {
      rstage = 0;
      rphase ^= 1u;
    }
  }
  if (pend >= 0) {
    tc::wait_st();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive_u32(afull_u + 8u * static_cast<uint32_t>(pend));
  }
  if (!dense_mode(MODE)) cur.release(c, op.a, lane == 0);
}

// Epilogue warps, one op: activation staging, accumulator folds, stream-K
// reduction and the op's epilogue.
template <int MODE, int NC>
__device__ __forceinline__ void epilogue_op(const Cta& c, const TcOp& op, SchedCursor& cur,
                                         int ew, int lane, uint32_t& dcount,
                                         const uint32_t* wait_ctr, bool pdl_first) {
  const TcArgs& a = c.args();
  const int q = (kEpiWarp0 + ew) & 3;
  const int etid = ew * 32 + lane;
  const int r = 32 * q + lane;  // tile row = tensor-memory lane
  const uint32_t lane_addr = c.tmem + (static_cast<uint32_t>(32 * q) << 16);
  const int b = blockIdx.x;
  Sched sc{};
  if (!dense_mode(MODE)) sc = cur.acquire(c, a);
  int u0, u1;
  const Work wk = make_work<MODE>(a, sc, c, u0, u1);
  const Kernel<MODE> kk{a, sc, wk, &op.maps[0], &op.maps[1], &op.maps[2], &op.maps[3]};
  int* sig = c.sig();
  float* rms = c.rms();
  float* ep = c.ep();
  volatile int* bcast = c.bcast();

  // The wait for the previous op (its outputs are this op's inputs) comes
  // right before the first activations are read: everything before it
  // depends only on this op's arguments, weights and routing, and so runs
  // while the previous op finishes.  The first op of a launch whose inputs
  // come from the previous kernel (pdl_first) waits for that kernel here.
  bool waited = wait_ctr == nullptr && !pdl_first;
  auto wait_inputs = [&]() {
    if (!waited) {
      if (wait_ctr) {
        if (etid == 0) grid_wait(wait_ctr, gridDim.x, c.status(), c.abort_flag());
      } else {
        pdl_wait();
        pdl_launch_dependents();
      }
      esync();
      waited = true;
    }
  };
  if (u0 >= u1) wait_inputs();  // (keeps the completion order transitive)

  XState xst;
  bool rms_ready = false;
  int g_expert = -1;
  float g_tile = 0.0f;
  const int first_tile = (u0 < u1) ? static_cast<int>(u0 / wk.nkb) : 0;
  // the matrix's scale (NVFP4 per-tensor scale, FP8 scale; BF16: none),
  // loaded before the op's completion wait
  const float gs = dense_mode(MODE) ? *c.op_scale() : 0.0f;
  // dense argmax: lane i of epilogue warp ew keeps the running best of row
  // m = ew + kEpiWarps i over the CTA's finished tiles
  float am_v = -FLT_MAX;
  int am_i = 0x7fffffff;

  for (int u = u0; u < u1;) {
    if (c.aborted()) break;
    const int tile = static_cast<int>(u / wk.nkb);
    const int kbs = static_cast<int>(u % wk.nkb);
    const int kbe = min(wk.nkb, kbs + (u1 - u));
    const int key = kk.b_key(tile);
    const int nr = kk.b_rows(tile);
    const int rb = tc_xrows(nr);
    const bool one_tile = u1 <= (tile + 1) * wk.nkb;
    // the tile's expert's global scale: a global load (microseconds while the
    // weights stream) only when the expert changes, issued before the MMAs
    // are waited for
    if (MODE == kTcGateUp) {
      const int e = kk.tile_expert(tile);
      if (q < 2 && e != g_expert) {
        g_tile = (e == a.E) ? *a.sh_gu_global : a.gu_global[e];
        g_expert = e;
      }
    } else if (MODE == kTcDown) {
      const int e = sc.active[tile / wk.per_e];
      if (e != g_expert) {
        g_tile = (e == a.E) ? *a.sh_dn_global : a.dn_global[e];
        g_expert = e;
      }
    }
    float tot[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) tot[j] = 0.0f;

    for (int w0 = kbs; w0 < kbe;) {
      const int w1 = window_end(kk, w0, kbe);
      if (!xst.covers(key, w0, w1)) {
        restage_range(kk, w0, w1, one_tile, xst.k0, xst.k1);
        xst.key = key;
        // the previous window's MMAs are complete (its accumulator was read)
        const int kbeg = xst.k0 * kk.uk(), klen = (xst.k1 - xst.k0) * kk.uk();
        wait_inputs();
        if (MODE == kTcDown) {
          const float* hbase = a.h + static_cast<size_t>(sc.off[key]) * a.I;
          const int I = a.I;
          stage_rows<float>([&](int n) { return hbase + static_cast<size_t>(n) * I; }, nr, rb,
                            kbeg, klen, smem_u32(c.xs()), sig, nullptr, ew, lane);
        } else {
          // The RMS factors from the staged rows when the window is the whole
          // K (gate_up: always).  Otherwise dense ops take them from global
          // memory below.  The CTA that finishes a split tile applies its own
          // factor, so every CTA must compute it bit for bit alike: both ways
          // sum the same 16-byte chunks per lane in the same order (high half
          // of each word first) and reduce across the warp by the same
          // butterfly.
          const bool stage_rms =
              a.rms && !rms_ready && (MODE == kTcGateUp || (kbeg == 0 && klen == a.K));
          rms_ready = rms_ready || stage_rms;
          const __nv_bfloat16* xb = dense_mode(MODE) ? a.A : a.x;
          const int64_t ld = dense_mode(MODE) ? a.lda : a.ldx;
          stage_rows_async(xb, ld, nr, rb, kbeg, klen, smem_u32(c.xs()), sig,
                           stage_rms ? rms : nullptr, ew, lane, MODE == kTcDenseBF);
        }
        fence_proxy_async_smem();
        esync();
        __syncwarp();
        if (lane == 0) mbar_arrive(c.x_full());
        // dense: the RMS factor of each row over the whole K from global
        // memory, while the MMAs run
        if (dense_mode(MODE) && a.rms && !rms_ready) {
          for (int m = ew; m < a.M; m += kEpiWarps) {
            const __nv_bfloat16* row = a.A + m * a.lda;
            // the row's largest magnitude and plain sum of squares in one
            // pass; a row above kSumsqSafeMax (rare) sums its squares again,
            // shifted by its staging shift (no overflow at any magnitude)
            uint32_t mx = 0u;
            float ss = 0.0f;
            for (int v0 = 0; v0 < a.K / 8; v0 += 8 * 32) {
              uint4 buf[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int v = v0 + 32 * i + lane;
                buf[i] = v < a.K / 8 ? __ldcg(reinterpret_cast<const uint4*>(row + v * 8))
                                     : make_uint4(0u, 0u, 0u, 0u);
              }
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint32_t w[4] = {buf[i].x, buf[i].y, buf[i].z, buf[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  mx = __vmaxu2(mx, w[j] & 0x7FFF7FFFu);
                  const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
                  ss = fmaf(lo, lo, fmaf(hi, hi, ss));
                }
              }
            }
            const float mrow =
                warp_max(fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xFFFF0000u)));
            const int sh = f16_row_shift(mrow);
            if (mrow > kSumsqSafeMax) {
              const int h1 = (sh > 126 || sh < -126) ? sh / 2 : sh;
              const float f1 = exp2i(h1), f2 = exp2i(sh - h1);
              ss = 0.0f;
              for (int v = lane; v < a.K / 8; v += 32) {
                const uint4 q = __ldcg(reinterpret_cast<const uint4*>(row + v * 8));
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const float lo = __uint_as_float(w[j] << 16) * f1 * f2;
                  const float hi = __uint_as_float(w[j] & 0xFFFF0000u) * f1 * f2;
                  ss = fmaf(lo, lo, fmaf(hi, hi, ss));
                }
              }
            }
            ss = warp_sum(ss);
            if (lane == 0) rms[m] = mrow > kSumsqSafeMax ? rms_factor(ss, sh, a.K) : rms_plain(ss, a.K);
          }
          rms_ready = true;
          esync();
        }
      }
      // ---- fold the window's accumulator into the segment total
      const uint32_t db = dcount % kDBufs;
      wait_bar(c.d_full_at(db), (dcount / kDBufs) & 1u, c.status(), c.abort_flag());
      tc::fence_after_sync();
#pragma unroll
      for (int h = 0; h < NC / 16; ++h) {
        uint32_t dv[16];
        tc::ld_x16(lane_addr + kDCol + 32u * db + 16u * h, dv);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (16 * h + j < nr) tot[16 * h + j] += scale_pow2(__uint_as_float(dv[j]), -sig[16 * h + j]);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.d_empty_at(db));
      ++dcount;
      w0 = w1;
    }
    u += kbe - kbs;

    // ---- stream-K: a tile split between CTAs is reduced by its last CTA
    if (!(kbs == 0 && kbe == wk.nkb)) {
      const int slot = (tile == first_tile) ? 0 : 1;
      float* part = a.partials + static_cast<size_t>(b * 2 + slot) * (32 * kRows);
#pragma unroll
      for (int j = 0; j < NC; ++j)
        if (j < nr) part[j * kRows + r] = tot[j];
      esync();
      const int blo = wk.cta_of(tile * wk.nkb);
      const int bhi = wk.cta_of((tile + 1) * wk.nkb - 1);
      if (etid == 0) {
        // releases the CTA's partial (ordered before by the barrier); the last
        // adder acquires the others'
        const uint32_t prev = atom_add_acq_rel_gpu(&a.tile_cnt[tile], 1u);
        *bcast = (prev == static_cast<uint32_t>(bhi - blo)) ? 1 : 0;
      }
      esync();
      if (!*bcast) continue;  // uniform across the epilogue warps
      // sum in CTA order; this CTA's own partial comes from registers
      float own[NC];
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        own[j] = tot[j];
        tot[j] = 0.0f;
      }
      for (int bb = blo; bb <= bhi; ++bb) {
        if (wk.abs_cta(bb) == b) {
#pragma unroll
          for (int j = 0; j < NC; ++j) tot[j] += own[j];
          continue;
        }
        const int sl = (wk.begin(bb) / wk.nkb == tile) ? 0 : 1;
        const float* pp = a.partials + static_cast<size_t>(wk.abs_cta(bb) * 2 + sl) * (32 * kRows);
#pragma unroll
        for (int j = 0; j < NC; ++j)
          if (j < nr) tot[j] += __ldcg(pp + j * kRows + r);
      }
      if (etid == 0) a.tile_cnt[tile] = 0u;
    }

    // ---- epilogues
    if (dense_mode(MODE)) {
#pragma unroll
      for (int j = 0; j < NC; ++j)
        if (j < a.M) ep[j * kRows + r] = tot[j] * gs * (a.rms ? rms[j] : 1.0f);
      esync();
      const int n0 = tile * kRows;
      for (int m = ew; m < a.M; m += kEpiWarps) {
        float bv = -FLT_MAX;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = 4 * lane + i, n = n0 + rr;
          if (n < a.N) {
            const __nv_bfloat16 o = __float2bfloat16_rn(ep[m * kRows + rr]);
            a.C[m * a.ldc + n] = o;
            const float ov = __bfloat162float(o);
            if (am_better(ov, n, bv, bi)) {
              bv = ov;
              bi = n;
            }
          }
        }
        if (a.argmax_out) {
          am_warp_reduce(bv, bi);
          if (lane == (m - ew) / kEpiWarps && bi != 0x7fffffff && am_better(bv, bi, am_v, am_i)) {
            am_v = bv;
            am_i = bi;
          }
        }
      }
    } else if (MODE == kTcGateUp) {
      // rows 0-63: gate rows 64 j + r of expert e; rows 64-127 the same up rows
      if (q >= 2) {
#pragma unroll
        for (int j = 0; j < NC; ++j) ep[j * kRows + r] = tot[j];
      }
      esync();
      if (q < 2) {
        const int e = kk.tile_expert(tile), jb = tile % wk.per_e;
        const float g = g_tile;
        const int cnt = sc.cnt[e], off = sc.off[e];
        for (int qq = 0; qq < cnt; ++qq) {
          const int p = off + qq;
          const int t = sc.pair_tok[p];
          const float f = a.rms ? g * rms[t] : g;
          float gt = 0.0f;
#pragma unroll
          for (int j = 0; j < NC; ++j)
            if (j == t) gt = tot[j];
          gt *= f;
          const float up = ep[t * kRows + r + kGuRows] * f;
          a.h[static_cast<size_t>(p) * a.I + jb * kGuRows + r] = gt / (1.0f + expf(-gt)) * up;
        }
      }
    } else {
      const int e = sc.active[tile / wk.per_e], nt = tile % wk.per_e;
      const float g = g_tile;
      const int cnt = sc.cnt[e], off = sc.off[e];
#pragma unroll
      for (int j = 0; j < NC; ++j)
        if (j < cnt) a.y[static_cast<size_t>(off + j) * a.H + nt * kRows + r] = tot[j] * g;
    }
    esync();
  }
  // ---- argmax: one partial per CTA of the op; the last CTA to add its own
  // reduces the op's G partials per row (the order of (value, index) pairs is
  // total, so the result does not depend on which CTA finished which tile)
  if (dense_mode(MODE) && a.argmax_out && wk.rel(b) < wk.G) {  // uniform over the warps
    const int own = ew + kEpiWarps * lane;  // the row this lane's running best belongs to
    if (own < a.M) a.am_part[own * wk.G + wk.rel(b)] = make_int2(__float_as_int(am_v), am_i);
    esync();
    if (etid == 0) {
      const uint32_t prev = atom_add_acq_rel_gpu(a.argmax_cnt, 1u);
      *bcast = (prev == static_cast<uint32_t>(wk.G - 1)) ? 1 : 0;
    }
    esync();
    if (*bcast) {
      for (int m = ew; m < a.M; m += kEpiWarps) {
        float bv = -FLT_MAX;
        int bi = 0x7fffffff;
        for (int j = lane; j < wk.G; j += 32) {
          const int2 pr = __ldcg(a.am_part + m * wk.G + j);
          const float v = __int_as_float(pr.x);
          if (pr.y != 0x7fffffff && am_better(v, pr.y, bv, bi)) {
            bv = v;
            bi = pr.y;
          }
        }
        am_warp_reduce(bv, bi);
        if (lane == 0) a.argmax_out[m] = (a.am_map && bi != 0x7fffffff) ? a.am_map[bi] : bi;
      }
      if (etid == 0) *a.argmax_cnt = 0u;
    }
  }
  if (!dense_mode(MODE)) cur.release(c, a, lane == 0);
}

// The weighted combine of a MoE layer, after every CTA finished its down
// op: out[t] = sum over slots j (in order) of w[t][j] * y[pair(t, j)], the
// shared expert last (weight 1); ids outside [0, E) contribute nothing.  The
// T x H/4 four-column groups are spread over all CTAs, one per thread.
__device__ __noinline__ void combine_op(const Cta& c, const TcOp& op, SchedCursor& cur, int ew,
                                        int lane) {
  const TcArgs& a = c.args();
  const Sched sc = cur.acquire(c, a);
  const int etid = ew * 32 + lane;
  const int groups = a.H / 4;
  const int items = a.T * groups;
  const int sh_off = sc.off[a.E];
  for (int it = blockIdx.x * kEpiThreads + etid; it < items && !c.aborted();
       it += gridDim.x * kEpiThreads) {
    const int t = it / groups, n = 4 * (it - t * groups);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 <= a.k; j0 += 8) {
      float4 yv[8];
      float wv[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int j = j0 + jj;
        yv[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
        wv[jj] = 0.0f;
        int pr = -1;
        if (j < a.k) {
          pr = sc.flat_pair[t * a.k + j];
          if (pr >= 0) wv[jj] = a.w[t * a.k + j];
        } else if (j == a.k && a.has_shared) {
          pr = sh_off + t;
          wv[jj] = 1.0f;
        }
        if (pr >= 0)
          yv[jj] = __ldcg(reinterpret_cast<const float4*>(a.y + static_cast<size_t>(pr) * a.H + n));
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        acc.x = fmaf(wv[jj], yv[jj].x, acc.x);
        acc.y = fmaf(wv[jj], yv[jj].y, acc.y);
        acc.z = fmaf(wv[jj], yv[jj].z, acc.z);
        acc.w = fmaf(wv[jj], yv[jj].w, acc.w);
      }
    }
    __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(a.out + t * a.ldo + n);
    o[0] = __floats2bfloat162_rn(acc.x, acc.y);
    o[1] = __floats2bfloat162_rn(acc.z, acc.w);
  }
  cur.release(c, a, lane == 0);
}

// ------------------------------------------------------------ roles

__device__ __forceinline__ void producer_role(const TcProgram& prog, const Cta& c, int lane) {
  const uint64_t pol = l2_policy_evict_first();
  const bool table = prog.ops != nullptr;
  SchedCursor cur;
  int stage = 0;
  uint32_t phase = 0;
  int issued = 0;
  for (int i = 0; i < prog.n_ops; ++i) {
    if (__any_sync(0xffffffffu, c.aborted())) break;
    const TcOp& op = op_at(prog, i);
    switch (op.mode) {
      case kTcDense: produce_op<kTcDense>(c, op, table, lane, cur, stage, phase, issued, pol); break;
      case kTcGateUp: produce_op<kTcGateUp>(c, op, table, lane, cur, stage, phase, issued, pol); break;
      case kTcDown: produce_op<kTcDown>(c, op, table, lane, cur, stage, phase, issued, pol); break;
      case kTcDenseF8: produce_op<kTcDenseF8>(c, op, table, lane, cur, stage, phase, issued, pol); break;
      case kTcDenseBF: produce_op<kTcDenseBF>(c, op, table, lane, cur, stage, phase, issued, pol); break;
      default: cur.acquire(c, op.a); cur.release(c, op.a, lane == 0); break;  // combine: no weights
    }
  }
  // wait for the TMA writes still in flight (bounded, ignores aborts)
  if (lane == 0) {
    const int n = issued < c.n_stages() ? static_cast<int>(issued) : c.n_stages();
    for (int i = 0; i < n; ++i) {
      if (stage == 0) {
        stage = c.n_stages() - 1;
        phase ^= 1u;
      } else {
        --stage;
      }
      mbar_wait(c.ring_full_at(stage), phase, c.status());
    }
  }
  __syncwarp();
}

__device__ __forceinline__ void mma_role(const TcProgram& prog, const Cta& c, int lane) {
  SchedCursor cur;
  uint32_t acount = 0, dcount = 0, xcount = 0;
  int rstage = 0;
  uint32_t rphase = 0;
  for (int i = 0; i < prog.n_ops; ++i) {
    if (__any_sync(0xffffffffu, c.aborted())) break;
    const TcOp& op = op_at(prog, i);
    switch (op.mode) {
      case kTcDense: mma_op<kTcDense>(c, op, cur, lane, acount, dcount, xcount, rstage, rphase); break;
      case kTcGateUp: mma_op<kTcGateUp>(c, op, cur, lane, acount, dcount, xcount, rstage, rphase); break;
      case kTcDown: mma_op<kTcDown>(c, op, cur, lane, acount, dcount, xcount, rstage, rphase); break;
      case kTcDenseF8:
        mma_op<kTcDenseF8>(c, op, cur, lane, acount, dcount, xcount, rstage, rphase);
        break;
      case kTcDenseBF:
        mma_op<kTcDenseBF>(c, op, cur, lane, acount, dcount, xcount, rstage, rphase);
        break;
      default: cur.acquire(c, op.a); cur.release(c, op.a, lane == 0); break;
    }
  }
  // every MMA has completed before tensor memory is released
  if (tc::elect_one()) tc::commit(c.mma_done());
  __syncwarp();
  if (lane == 0) mbar_wait(c.mma_done(), 0, c.status());
  __syncwarp();
}

__device__ __forceinline__ void decode_role(const TcProgram& prog, const Cta& c, int warp, int lane) {
  SchedCursor cur;
  uint32_t acount = 0;
  int rstage = 0;
  uint32_t rphase = 0;
  for (int i = 0; i < prog.n_ops && !c.aborted(); ++i) {
    const TcOp& op = op_at(prog, i);
    if (i > 0 && op.mode != kTcCombine) {
      // wait (bounded) until this CTA's epilogue finished op i - 1
      const unsigned long long t0 = globaltimer();
      while (*c.epi_done() < i && !c.aborted()) {
        if (globaltimer() - t0 > kWaitLimitNs) {
          atomicOr(c.status(), kStatusTimeout);
          *c.abort_flag() = 1;
          break;
        }
        __nanosleep(64);
      }
    }
    switch (op.mode) {
      case kTcDense: decode_op<kTcDense>(c, op, cur, warp, lane, acount, rstage, rphase); break;
      case kTcGateUp: decode_op<kTcGateUp>(c, op, cur, warp, lane, acount, rstage, rphase); break;
      case kTcDown: decode_op<kTcDown>(c, op, cur, warp, lane, acount, rstage, rphase); break;
      case kTcDenseF8: decode_op<kTcDenseF8>(c, op, cur, warp, lane, acount, rstage, rphase); break;
      case kTcDenseBF: decode_op<kTcDenseBF>(c, op, cur, warp, lane, acount, rstage, rphase); break;
      default: cur.acquire(c, op.a); cur.release(c, op.a, lane == 0); break;
    }
  }
}

__device__ __forceinline__ void epilogue_role(const TcProgram& prog, const Cta& c, int warp, int lane) {
  const int ew = warp - kEpiWarp0, etid = ew * 32 + lane;
  const int n_ops = prog.n_ops;
  SchedCursor cur;
  uint32_t dcount = 0;
  // inputs may come from the previous kernel on the stream: a dense first op
  // waits for it just before it reads its activations, any other at once.
  // The next kernel is released only after that wait (released at launch,
  // its CTAs took SMs ahead of this kernel's: measured on GB300, the
  // 16- and 32-token decode steps 2 to 3 % slower).
  const bool pdl_first = n_ops > 0 && dense_mode(op_at(prog, 0).mode);
  if (!pdl_first) {
    pdl_wait();
    pdl_launch_dependents();
  }
  constexpr int kArgWords = static_cast<int>(sizeof(TcArgs)) / 16;
  for (int i = 0; i < n_ops && !c.aborted(); ++i) {
    const TcOp& op = op_at(prog, i);
    // the op's arguments (the device op table, or the launch parameters)
    // and a dense op's matrix scale are loaded before waiting for the
    // previous op (neither depends on it) and kept in shared memory: every
    // later read is local instead of a dependent trip to global memory
    uint4 av = make_uint4(0u, 0u, 0u, 0u);
    if (etid < kArgWords) av = reinterpret_cast<const uint4*>(&op.a)[etid];
    float scale = 1.0f;
    if (etid == kArgWords && dense_mode(op.mode) && op.a.gscale) scale = *op.a.gscale;
    // every CTA has finished op i - 1 once done[i - 1] == grid: its outputs
    // are complete (the ops wait for it before reading their inputs)
    const uint32_t* wait_ctr = (i > 0 && op.wait_prev) ? &prog.done[i - 1] : nullptr;
    esync();  // the previous op's readers of the copy are done
    if (etid < kArgWords) reinterpret_cast<uint4*>(c.base + kTcOffArgs)[etid] = av;
    if (etid == kArgWords) *c.op_scale() = scale;
    esync();
    switch (op.mode) {
      // accumulator columns: 16 when the op has at most 16 activation rows
      case kTcDense:
        if (c.args().M <= 16) epilogue_op<kTcDense, 16>(c, op, cur, ew, lane, dcount, wait_ctr, i == 0 && pdl_first);
        else epilogue_op<kTcDense, 32>(c, op, cur, ew, lane, dcount, wait_ctr, i == 0 && pdl_first);
        break;
      case kTcGateUp:
        if (c.args().T <= 16) epilogue_op<kTcGateUp, 16>(c, op, cur, ew, lane, dcount, wait_ctr, i == 0 && pdl_first);
        else epilogue_op<kTcGateUp, 32>(c, op, cur, ew, lane, dcount, wait_ctr, i == 0 && pdl_first);
        break;
      case kTcDown:
        if (c.args().T <= 16) epilogue_op<kTcDown, 16>(c, op, cur, ew, lane, dcount, wait_ctr, i == 0 && pdl_first);
        else epilogue_op<kTcDown, 32>(c, op, cur, ew, lane, dcount, wait_ctr, i == 0 && pdl_first);
        break;
      case kTcDenseF8:
        if (c.args().M <= 16) epilogue_op<kTcDenseF8, 16>(c, op, cur, ew, lane, dcount, wait_ctr, i == 0 && pdl_first);
        else epilogue_op<kTcDenseF8, 32>(c, op, cur, ew, lane, dcount, wait_ctr, i == 0 && pdl_first);
        break;
      case kTcDenseBF:
        if (c.args().M <= 16) epilogue_op<kTcDenseBF, 16>(c, op, cur, ew, lane, dcount, wait_ctr, i == 0 && pdl_first);
        else epilogue_op<kTcDenseBF, 32>(c, op, cur, ew, lane, dcount, wait_ctr, i == 0 && pdl_first);
        break;
      default:
        if (wait_ctr) {
          if (etid == 0) grid_wait(wait_ctr, gridDim.x, c.status(), c.abort_flag());
          esync();
        }
        combine_op(c, op, cur, ew, lane);
        break;
    }
    if (n_ops > 1) {
      esync();
      if (etid == 0) {
        red_add_release_gpu(&prog.done[i], 1u);
        *c.epi_done() = i + 1;
      }
    }
  }
  if (n_ops > 1 && etid == 0) {
    // the last CTA to leave returns the completion counters to zero
    if (atom_add_acq_rel_gpu(&prog.done[n_ops], 1u) == gridDim.x - 1) {
      for (int i = 0; i <= n_ops; ++i) prog.done[i] = 0u;
      __threadfence();
    }
  }
}

// One warp builds the expert schedule of each MoE op that starts one, into
// the slot its previous users released.
__device__ __forceinline__ void sched_role(const TcProgram& prog, const Cta& c, int lane) {
  int idx = -1;
  for (int i = 0; i < prog.n_ops && !c.aborted(); ++i) {
    const TcOp& op = op_at(prog, i);
    if (dense_mode(op.mode) || !op.a.new_sched) continue;
    ++idx;
    const int slot = idx % c.sched_slots();
    wait_bar(c.sched_empty_at(slot), ((idx / c.sched_slots()) & 1) ^ 1, c.status(), c.abort_flag());
    if (c.aborted()) break;
    // gate_up may read ids written before the previous kernel started
    // (NVFP4_FLAG_IDS_READY) before its dependency wait; down always can:
    // the gate_up grid before it read them after its own wait.
    if (op.mode == kTcGateUp && !op.a.ids_ready) pdl_wait();
    const Sched sc = sched_layout(c.sched() + slot * c.sched_bytes(), op.a.E, op.a.T * op.a.k);
    build_schedule_warp(op.a.ids, op.a.T, op.a.k, op.a.E, op.a.has_shared, sc, c.status(), lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(c.sched_full_at(slot));
  }
}

__global__ void __launch_bounds__(kTcThreads, 1)
    stream_tc_kernel(const __grid_constant__ TcProgram prog) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Cta c{smem, prog, 0u};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < c.n_stages(); ++s) {
      mbar_init(c.ring_full_at(s), 1);
      mbar_init(c.ring_empty_at(s), kDecWarps);
    }
    for (int b = 0; b < kABufs; ++b) {
      mbar_init(c.a_full_at(b), kDecWarps);
      mbar_init(c.a_empty_at(b), 1);
    }
    for (int b = 0; b < kDBufs; ++b) {
      mbar_init(c.d_full_at(b), 1);
      mbar_init(c.d_empty_at(b), kEpiWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(c.sched_full_at(b), 1);
      mbar_init(c.sched_empty_at(b), kSchedUsers);
    }
    mbar_init(c.x_full(), kEpiWarps);
    mbar_init(c.mma_done(), 1);
    mbar_init(c.x_tma(), 1);
    fence_mbarrier_init();
    *c.abort_flag() = 0;
    *c.epi_done() = 0;
  }
  if (warp == 1) tc::tmem_alloc(c.tmem_slot(), kTmemCols);
  __syncthreads();
  tc::fence_after_sync();
  c.tmem = *c.tmem_slot();

  // registers move from the warpgroups that need few (producer, MMA,
  // scheduler; decode) to the epilogue warpgroup
  if (warp < kEpiWarp0) {
    setmaxnreg_dec<kRegsSmall>();
    if (warp == 0) producer_role(prog, c, lane);
    else if (warp == 1) mma_role(prog, c, lane);
    else if (warp == 2) sched_role(prog, c, lane);
  } else if (warp < kDecWarp0) {
    setmaxnreg_inc<kRegsEpilogue>();
    epilogue_role(prog, c, warp, lane);
  } else {
    setmaxnreg_dec<kRegsSmall>();
    decode_role(prog, c, warp, lane);
  }

  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(c.tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_tc(const TcProgram& p, int grid, size_t smem, cudaStream_t s, bool pdl,
                      bool cooperative) {
  // The shared-memory opt-in is a per-device attribute of the kernel: set it
  // once per device, under a lock (several host threads may make their first
  // call at once).
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static bool attr_set[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!attr_set[dev]) {
      e = cudaFuncSetAttribute(stream_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               232448);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
  }
  // One CTA per SM: each CTA allocates all 512 tensor-memory columns, so a
  // second resident CTA would only queue on the allocation.
  const size_t kOnePerSm = 120 * 1024;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem < kOnePerSm ? kOnePerSm : smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cooperative) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, stream_tc_kernel, p);
}

}  // namespace nvfp4
