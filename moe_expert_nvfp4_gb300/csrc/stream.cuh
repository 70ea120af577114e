// The NVFP4 weight-streaming core shared by the dense and MoE kernels.
//
// One CTA = one producer warp + four consumer warps.  The producer streams
// 64-row x 256-K tiles of codes and scales (two 32-row TMA boxes each, codes
// 128B-swizzled) into a kStages-deep shared-memory ring guarded by
// full/empty mbarriers.  The consumers decode the E2M1 codes with the
// hardware E2M1->FP16 convert, multiply by the E4M3 block scale (the product
// is exact in FP16), and feed the warp MMA with FP32 accumulation against
// activations staged in shared memory as FP16.
//
// Weight-row tile layout per stage (consumer view).  Warp w owns rows
// [16w, 16w+16) of the 64-row tile.  In each half-stage i (128 K values)
// lane (g, t) reads the 16-byte chunk c = 4i + t of its two rows, which
// holds k = 32c .. 32c+31.  Byte 2j of the chunk feeds MMA j's k-pair t and
// byte 2j+1 its k-pair t+4, so MMA j covers k = 32c + 4j + {0..3} for every
// t; the activations are read with the same mapping.  (The dot product is
// invariant under a permutation of k applied to both operands.)  MMA row g
// maps to tile row 16w + rho(g), rho(g) = 4(g&1) + (g>>1), so that the eight
// lanes of each shared-memory phase touch distinct banks of the swizzled
// tile.
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
    // step back one stage
    if (p.stage == 0) {
      p.stage = kStages - 1;
      p.phase ^= 1u;
    } else {
      --p.stage;
    }
    mbar_wait(&r.full[p.stage], p.phase, status);
  }
}

// Consumer: accumulate one stage.  xs = staged activations (FP16 rows of
// xrow_bytes), kx0 = element offset of this stage in the staged rows,
// ntiles = number of 8-token MMA column tiles (1..4).
__device__ __forceinline__ void consume_stage(const uint8_t* codes, const uint8_t* scales,
                                              const uint8_t* xs, int xrow_bytes, int kx0,
                                              int warp, int lane, int ntiles,
                                              float (&acc)[4][4]) {
  const int g = lane >> 2, t = lane & 3;
  const int rg = ((g & 1) << 2) | (g >> 1);
  const int R0 = warp * 16 + rg, R1 = R0 + 8;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int c = 4 * i + t;
    const uint4 q0 = *reinterpret_cast<const uint4*>(codes + R0 * 128 + ((c ^ (R0 & 7)) << 4));
    const uint4 q1 = *reinterpret_cast<const uint4*>(codes + R1 * 128 + ((c ^ (R1 & 7)) << 4));
    const uint32_t sb0 = *reinterpret_cast<const uint16_t*>(scales + R0 * 16 + 2 * c);
    const uint32_t sb1 = *reinterpret_cast<const uint16_t*>(scales + R1 * 16 + 2 * c);
    const uint32_t s0[2] = {e4m3_bcast_f16x2(sb0 & 0xFFu), e4m3_bcast_f16x2(sb0 >> 8)};
    const uint32_t s1[2] = {e4m3_bcast_f16x2(sb1 & 0xFFu), e4m3_bcast_f16x2(sb1 >> 8)};
    const uint32_t w0[4] = {q0.x, q0.y, q0.z, q0.w};
    const uint32_t w1[4] = {q1.x, q1.y, q1.z, q1.w};
    const uint8_t* xrow = xs + g * xrow_bytes + (kx0 + 32 * c) * 2;
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
      for (int h = 0; h < 2; ++h) {
        const int j = 2 * wi + h;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          if (nt < ntiles) {
            const uint2 b =
                *reinterpret_cast<const uint2*>(xrow + nt * 8 * xrow_bytes + 4 * j * 2);
            mma_16816(acc[nt], d0[2 * h], d1[2 * h], d0[2 * h + 1], d1[2 * h + 1], b.x, b.y);
          }
        }
      }
    }
  }
}

// Accumulator element -> (tile row, token column) for lane (g, t):
// acc[nt][0] (R0, 8nt+2t), [1] (R0, 8nt+2t+1), [2] (R1, 8nt+2t), [3] (R1, 8nt+2t+1).
__device__ __forceinline__ void acc_coords(int warp, int lane, int& R0, int& R1, int& c0) {
  const int g = lane >> 2, t = lane & 3;
  R0 = warp * 16 + (((g & 1) << 2) | (g >> 1));
  R1 = R0 + 8;
  c0 = 2 * t;
}

// Stage activation rows into shared memory as FP16.
//   rows = number of real rows (<= kMaxM); pad_rows = rows rounded up to 8;
//   src(q) = pointer to row q; elements [k0, k0+klen) are staged; each row
//   gets its own power-of-two shift sig[q] (see f16_row_shift).  When
//   rms != nullptr, rms[q] = 1/sqrt(mean over [0, kfull) of x^2 + 1e-6)
//   (FP32).  Executed by the consumer warps only.
template <typename T, typename RowPtr>
__device__ __forceinline__ void stage_rows(RowPtr src, int rows, int pad_rows, int k0, int klen,
                                           int kfull, uint8_t* xs, int xrow_bytes, int* sig,
                                           float* rms, int warp, int lane) {
  constexpr int kVec = 16 / sizeof(T);  // elements per 16-byte load
  for (int q = warp; q < pad_rows; q += kConsumerWarps) {
    uint2* dst = reinterpret_cast<uint2*>(xs + q * xrow_bytes);
    if (q >= rows) {
      for (int v = lane; v < klen / 4; v += 32) dst[v] = make_uint2(0u, 0u);
      if (lane == 0) {
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
      dst[v] = make_uint2(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]));
    }
  }
}

}  // namespace nvfp4

namespace nvfp4 {
static_assert(kSmemBars == kStages * kStageBytes, "ring / mbarrier layout mismatch");
static_assert(kSmemMisc == kSmemBars + 2 * kStages * 8, "mbarrier area size");
static_assert(kSmemSched - kSmemEp == kMaxM * kTileRows * 4, "epilogue tile size");
}  // namespace nvfp4
