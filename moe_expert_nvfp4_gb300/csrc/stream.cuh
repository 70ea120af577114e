// The NVFP4 weight-streaming core shared by the dense and MoE kernels.
//
// One CTA = eight consumer warps + one producer warp.  The producer streams
// 64-row x 256-K stages of codes and scales (two 32-row TMA boxes each,
// codes 128B-swizzled) into a kStages-deep shared-memory ring guarded by
// full/empty mbarriers.  The consumers decode the E2M1 codes with the
// hardware E2M1->FP16 convert, multiply by the E4M3 block scale (the product
// is exact in FP16), and feed the warp MMA with FP32 accumulation against
// activations staged in shared memory as FP16.
//
// Work split of one stage.  Consumer warp w is in group h = w / 4 and owns
// tile rows [16(w%4), 16(w%4)+16); group h takes the half-stage k = 128h ..
// 128h+127.  Lane (g, t) reads the 16-byte chunk c = 4h + t of its two rows,
// which holds k = 32c .. 32c+31.  Byte 2j of the chunk feeds MMA j's k-pair
// t and byte 2j+1 its k-pair t+4, so MMA j covers k = 32c + 4j + {0..3};
// the activations are read with the same mapping (a dot product is
// invariant under a permutation of k applied to both operands).  MMA row g
// maps to tile row 16(w%4) + rho(g), rho(g) = 4(g&1) + (g>>1), so the eight
// lanes of each shared-memory phase touch distinct banks of the swizzled
// tile.  Even and odd j accumulate into separate registers (two independent
// MMA chains); the two groups' sums are added in a fixed order at the end of
// a tile, so results do not depend on timing.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace nvfp4 {

struct Ring {
  uint8_t* base;    // kStages * kStageBytes, 1024-byte aligned
  uint64_t* full;   // [kStages] producer -> consumers (TMA transaction bytes)
  uint64_t* empty;  // [kStages] consumers -> producer (one arrive per consumer warp)
  __device__ __forceinline__ uint8_t* codes(int s) const { return base + s * kStageBytes; }
  __device__ __forceinline__ uint8_t* scales(int s) const {
    return base + s * kStageBytes + kStageCodeBytes;
  }
};

struct Pipe {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void advance() {
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

// Bounded wait that also gives up as soon as another thread has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint32_t* status,
                                              volatile int* abort_flag) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
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

__device__ __forceinline__ void ring_init(const Ring& r) {
  for (int s = 0; s < kStages; ++s) {
    mbar_init(&r.full[s], 1);
    mbar_init(&r.empty[s], kConsumerWarps);
  }
  fence_mbarrier_init();
}

// Producer: issue one stage = rows [row0, row0+32) and [row1, row1+32),
// k-stage kb.  Returns false (and issues nothing) after an abort.
__device__ __forceinline__ bool produce_stage(const Ring& r, Pipe& p, const CUtensorMap* mc,
                                              const CUtensorMap* ms, int row0, int row1, int kb,
                                              uint64_t pol, uint32_t* status,
                                              volatile int* abort_flag) {
  if (*abort_flag) return false;
  if (!wait_or_abort(&r.empty[p.stage], p.phase ^ 1u, status, abort_flag)) return false;
  uint64_t* fb = &r.full[p.stage];
  mbar_arrive_expect_tx(fb, kStageBytes);
  uint8_t* c = r.codes(p.stage);
  uint8_t* s = r.scales(p.stage);
  tma_load_2d(c, mc, kb * (kStageK / 2), row0, fb, pol);
  tma_load_2d(c + kStageCodeBytes / 2, mc, kb * (kStageK / 2), row1, fb, pol);
  tma_load_2d(s, ms, kb * (kStageK / 16), row0, fb, pol);
  tma_load_2d(s + kStageScaleBytes / 2, ms, kb * (kStageK / 16), row1, fb, pol);
  p.advance();
  return true;
}

// Producer epilogue: wait (bounded, ignoring aborts) for the TMA writes of the
// last `issued` stages so that none lands after the CTA exits.
__device__ __forceinline__ void producer_drain(const Ring& r, Pipe p, long issued,
                                               uint32_t* status) {
  const int n = issued < kStages ? static_cast<int>(issued) : kStages;
  for (int i = 0; i < n; ++i) {
    if (p.stage == 0) {
      p.stage = kStages - 1;
      p.phase ^= 1u;
    } else {
      --p.stage;
    }
    mbar_wait(&r.full[p.stage], p.phase, status);
  }
}

// Accumulators of one consumer warp: [ntile][4] for even and odd MMA j.
struct Acc {
  float e[4][4];
  float o[4][4];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) e[i][j] = o[i][j] = 0.0f;
  }
};

// Consumer: accumulate this warp's half of one stage.  xr[nt] = staged FP16
// activation row that feeds MMA column g of token tile nt (lane-specific),
// kx0 = element offset of this stage within the staged rows.
__device__ __forceinline__ void consume_half(const uint8_t* codes, const uint8_t* scales, int h,
                                             int wg, int lane, const uint8_t* const (&xr)[4],
                                             int kx0, int ntiles, Acc& acc) {
  const int g = lane >> 2, t = lane & 3;
  const int R0 = wg * 16 + (((g & 1) << 2) | (g >> 1)), R1 = R0 + 8;
  const int c = 4 * h + t;
  const uint4 q0 = *reinterpret_cast<const uint4*>(codes + R0 * 128 + ((c ^ (R0 & 7)) << 4));
  const uint4 q1 = *reinterpret_cast<const uint4*>(codes + R1 * 128 + ((c ^ (R1 & 7)) << 4));
  const uint32_t sb0 = *reinterpret_cast<const uint16_t*>(scales + R0 * 16 + 2 * c);
  const uint32_t sb1 = *reinterpret_cast<const uint16_t*>(scales + R1 * 16 + 2 * c);
  const uint32_t s0[2] = {e4m3_bcast_f16x2(sb0 & 0xFFu), e4m3_bcast_f16x2(sb0 >> 8)};
  const uint32_t s1[2] = {e4m3_bcast_f16x2(sb1 & 0xFFu), e4m3_bcast_f16x2(sb1 >> 8)};
  const uint32_t w0[4] = {q0.x, q0.y, q0.z, q0.w};
  const uint32_t w1[4] = {q1.x, q1.y, q1.z, q1.w};
  const int xoff = (kx0 >> 8) * 512 + c * 16;  // fragment-ordered staging, see stage_rows
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    uint32_t d0[4], d1[4];
    e2m1x8_to_f16x2(w0[wi], d0[0], d0[1], d0[2], d0[3]);
    e2m1x8_to_f16x2(w1[wi], d1[0], d1[1], d1[2], d1[3]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      d0[e] = hmul2(d0[e], s0[wi >> 1]);
      d1[e] = hmul2(d1[e], s1[wi >> 1]);
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      if (nt < ntiles) {
        const uint4 b = *reinterpret_cast<const uint4*>(xr[nt] + xoff + 128 * wi);
        mma_16816(acc.e[nt], d0[0], d1[0], d0[1], d1[1], b.x, b.y);
        mma_16816(acc.o[nt], d0[2], d1[2], d0[3], d1[3], b.z, b.w);
      }
    }
  }
}

// Accumulator element -> (tile row R, column q) for lane (g, t) of a
// consumer warp in row group wg: element e of token tile nt is at
// R = e < 2 ? R0 : R1, q = 8nt + 2t + (e & 1).
__device__ __forceinline__ void acc_coords(int wg, int lane, int& R0, int& R1, int& c0) {
  const int g = lane >> 2, t = lane & 3;
  R0 = wg * 16 + (((g & 1) << 2) | (g >> 1));
  R1 = R0 + 8;
  c0 = 2 * t;
}

// Fold one window's accumulators into a running FP32 tile total, undoing the
// window's FP16 staging shift of each column's row: tot += (e + o) * 2^-sig.
// colsig(q) gives the shift of column q.
template <typename ColSig>
__device__ __forceinline__ void fold_window(const Acc& acc, float (&tot)[4][4], int ntiles,
                                            int lane, ColSig colsig) {
  const int c0 = 2 * (lane & 3);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    if (nt < ntiles) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        tot[nt][e] += scale_pow2(acc.e[nt][e] + acc.o[nt][e], -colsig(nt * 8 + c0 + (e & 1)));
    }
  }
}

// Sum the two warp groups' tile totals into ep[q * 64 + R] (group 1 writes,
// group 0 adds: a fixed order).  Columns q >= qmax are skipped.  Called by
// all consumer warps; ends with the consumers synchronised.
__device__ __forceinline__ void groups_to_ep(const float (&tot)[4][4], float* ep, int ntiles,
                                             int qmax, int cw, int lane) {
  int R0, R1, c0;
  acc_coords(cw & 3, lane, R0, R1, c0);
  const bool writer = (cw >> 2) == 1;
  if (writer) {
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
      if (nt < ntiles)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = nt * 8 + c0 + (e & 1);
          if (q < qmax) ep[q * 64 + (e < 2 ? R0 : R1)] = tot[nt][e];
        }
  }
  consumer_sync();
  if (!writer) {
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
      if (nt < ntiles)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = nt * 8 + c0 + (e & 1);
          if (q < qmax) ep[q * 64 + (e < 2 ? R0 : R1)] += tot[nt][e];
        }
  }
  consumer_sync();
}

// Byte offset of staged element kk (relative to the window start) inside a
// staged row: each 256-element stage block is stored fragment-ordered,
// element 32c + 8w + e at 128w + 16c + 2e, so that consume_half's 16-byte
// reads of the four lanes t of one row are consecutive.
__device__ __forceinline__ int xstage_off(int kk) {
  const int within = kk & 255;
  return (kk >> 8) * 512 + ((within >> 3) & 3) * 128 + (within >> 5) * 16 + (within & 7) * 2;
}

// Row stride of the staged activations: 2*klen + 64 bytes, a multiple of 16
// that is 64 mod 128 so that two consecutive rows use disjoint bank halves.
__host__ __device__ constexpr int xrow_stride(int klen) { return 2 * klen + 64; }

// Stage activation rows into shared memory as FP16.
//   rows <= kMaxM real rows; pad_rows >= rows rows are written (zeros past
//   rows; only rows below kMaxM get sig / rms entries);
//   src(q) = pointer to row q; elements [k0, k0+klen) are staged into
//   xs + q * xrow_bytes in fragment order (xstage_off); row q gets its own
//   power-of-two shift sig[q] (see f16_row_shift).  When rms != nullptr,
//   rms[q] = 1/sqrt(mean over [0, kfull) of x^2 + 1e-6) (FP32).  Executed by
//   the consumer warps.
template <typename T, typename RowPtr>
__device__ __forceinline__ void stage_rows(RowPtr src, int rows, int pad_rows, int k0, int klen,
                                           int kfull, uint8_t* xs, int xrow_bytes, int* sig,
                                           float* rms, int cw, int lane) {
  constexpr int kVec = 16 / sizeof(T);  // elements per 16-byte load
  for (int q = cw; q < pad_rows; q += kConsumerWarps) {
    uint8_t* dst = xs + q * xrow_bytes;
    if (q >= rows) {
      for (int v = lane; v < klen / 8; v += 32)
        *reinterpret_cast<uint4*>(dst + 16 * v) = make_uint4(0u, 0u, 0u, 0u);
      if (lane == 0 && q < kMaxM) {  // sig and rms hold kMaxM entries
        sig[q] = 0;
        if (rms) rms[q] = 0.0f;
      }
      continue;
    }
    const T* row = src(q);
    float amax = 0.0f;
    for (int v = lane; v < klen / kVec; v += 32) {
      const uint4 u = *reinterpret_cast<const uint4*>(row + k0 + v * kVec);
      const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
      for (int i = 0; i < kVec; ++i) amax = fmaxf(amax, fabsf(static_cast<float>(e[i])));
    }
    amax = warp_max(amax);
    if (rms) {
      float ss = 0.0f;
      for (int v = lane; v < kfull / kVec; v += 32) {
        const uint4 u = *reinterpret_cast<const uint4*>(row + v * kVec);
        const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int i = 0; i < kVec; ++i) {
          const float f = static_cast<float>(e[i]);
          ss = fmaf(f, f, ss);
        }
      }
      ss = warp_sum(ss);
      if (lane == 0) rms[q] = rsqrtf(ss / static_cast<float>(kfull) + 1e-6f);
    }
    const int s = f16_row_shift(amax);
    if (lane == 0) sig[q] = s;
    for (int v = lane; v < klen / 4; v += 32) {
      float f[4];
      if constexpr (sizeof(T) == 2) {
        const uint2 u = *reinterpret_cast<const uint2*>(row + k0 + v * 4);
        const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) f[i] = static_cast<float>(e[i]);
      } else {
        const uint4 u = *reinterpret_cast<const uint4*>(row + k0 + v * 4);
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) f[i] = scale_pow2(f[i], s);
      *reinterpret_cast<uint2*>(dst + xstage_off(v * 4)) =
          make_uint2(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]));
    }
  }
}

static_assert(kSmemBars == kStages * kStageBytes, "ring / mbarrier layout mismatch");
static_assert(kSmemMisc == kSmemBars + 2 * kStages * 8, "mbarrier area size");
static_assert(kSmemSched - kSmemEp == kMaxM * kTileRows * 4, "epilogue tile size");

}  // namespace nvfp4
