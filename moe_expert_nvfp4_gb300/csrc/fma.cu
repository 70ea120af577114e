// NVFP4 skinny GEMM on the CUDA cores: decode and dot product in registers.
//
// The other dense path (stream_tc.cu) hands the dot product to the tensor
// cores; at one or two activation rows a weight costs only one or two FMAs,
// which the CUDA cores can issue at the HBM rate.  This kernel is that
// alternative, and the path for K that is a multiple of 32 but not of 256
// (the tensor-memory path streams 256-K stages).
//
// Layout of the work: one warp computes whole rows n of C (no split-K).
// Lane l owns the 32-K chunks l, l + 32, ... of a row: per chunk it loads 16
// bytes of E2M1 codes and the chunk's two E4M3 block scales, converts the
// codes to FP16 (hardware convert, exact) and accumulates code x activation
// per 16-element block with the mixed FMA (f16 x f16 + f32 -> f32, the
// product exact), then adds block scale x block sum into the row's FP32
// total.  A warp reduction ends the row.  The activations (MB = 1, 2, 4, 8
// or 16 rows per CTA, grid.y covering the rest; from four rows each decoded
// chunk serves every row) are staged once per CTA in shared memory as FP16
// after the same power-of-two row shift as the tensor path (exact for BF16
// elements within 2^31 of the row's largest magnitude), with a
// bank-conflict-free padding of each chunk's four 16-byte slots.  (Staging
// the rows as FP32 instead, one FP32 FMA a weight, measured slower at every
// M: the shared-memory traffic doubles.)
//
// Sources: "Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)", "Making decode
// faster", "Skinny matrix multiplies" (decode matmuls of four to sixteen
// activation rows against 4-bit weights).
#include <cuda_bf16.h>
#include <float.h>

#include "common.cuh"
#include "launch.h"

namespace nvfp4 {
namespace {

constexpr int kFmaWarps = 8;
constexpr int kFmaThreads = kFmaWarps * 32;

// Staged activations: row m at m * rs bytes (rs = chunks * kChunkPitch), its
// 32-K chunk c at c * kChunkPitch (64 bytes of FP16, 16 of padding), the
// chunk's 16-byte slot q at q * 16.  The eight lanes of a shared-memory phase
// (chunks c .. c + 7, same q) hit eight different 16-byte bank groups (80 c
// mod 128 takes eight values), and every address is a per-chunk base plus
// a row offset and constants.
constexpr int kChunkPitch = 80;

// Barrier of the ks warps of team `team` (ks = 2: teams 0 .. 3, ks = 4:
// teams 0, 1; named barriers 1 .. 4).  The barrier ids are immediates: with
// an id in a register the compiler reserves all sixteen of the CTA's
// barriers.
__device__ __forceinline__ void team_sync(int team, int ks) {
  const int n = ks * 32;
  switch (team) {
    case 0: asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory"); break;
    case 1: asm volatile("bar.sync 2, %0;" ::"r"(n) : "memory"); break;
    case 2: asm volatile("bar.sync 3, %0;" ::"r"(n) : "memory"); break;
    default: asm volatile("bar.sync 4, %0;" ::"r"(n) : "memory"); break;
  }
}

__device__ __forceinline__ void ld_chunk(uint32_t a, uint32_t (&xv)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = ld_shared_v4(a + 16 * q);
    xv[4 * q] = v.x;
    xv[4 * q + 1] = v.y;
    xv[4 * q + 2] = v.z;
    xv[4 * q + 3] = v.w;
  }
}

__device__ __forceinline__ bool fm_better(float v, int i, float bv, int bi) {
  return bi == 0x7fffffff || v > bv || (v == bv && i < bi);
}

// Sum over the CTA of one float per thread (thread 0 gets it; the warps'
// sums are added in warp order).
__device__ __forceinline__ float cta_sum0(float v, float* s_w) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.0f;
  if (threadIdx.x == 0)
    for (int w = 0; w < kFmaWarps; ++w) t += s_w[w];
  __syncthreads();
  return t;
}

// MB activation rows per CTA (rows m0 .. m0 + MB - 1 of A, m0 = MB *
// blockIdx.y); grid-stride over the weight rows.  Two CTAs share an SM (the
// grid is at most twice the SM count), hence the register bound.
template <int MB, int RU>
__global__ void __launch_bounds__(kFmaThreads, 2) fma_kernel(const FmaArgs a) {
  static_assert(MB <= 4 && MB * RU <= 16, "rows per CTA, outputs per warp");
  extern __shared__ __align__(16) uint8_t fsm[];
  __shared__ int s_sh[MB];
  __shared__ float s_rms[MB];
  __shared__ float s_w[kFmaWarps];
  __shared__ float s_bv[kFmaWarps][MB];
  __shared__ float s_sq[kFmaWarps][MB];
  __shared__ int s_bi[kFmaWarps][MB];
  __shared__ int s_last;
  __shared__ float s_part[kFmaWarps * 16];  // K-split teams: each warp's row sums
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = MB * blockIdx.y;
  const int mb = min(MB, a.M - m0);
  const int chunks = a.K / 32;
  const int rs = chunks * kChunkPitch;  // bytes per staged row
  const uint32_t xs = smem_u32(fsm);

  // The weights do not depend on the previous kernel on the stream: the
  // first group's loads are issued before waiting for it.  A team of ks
  // warps (ks = a.ks: 1, 2 or 4; more when the weight has few rows) takes
  // groups of RU consecutive weight rows (group G = the team's global index
  // + t * teams); per group the lanes walk the rows' 32-K chunks in rounds
  // of 32, warp k of the team rounds k, k + ks, ... (ks <= rounds).
  // The loads of the next round (or group) are issued before the current
  // one is computed, so RU * 528 bytes per warp stay in flight.
  const int ks = a.ks, kidx = warp % ks, team = warp / ks;
  const int n_teams = gridDim.x * (kFmaWarps / ks);
  const int rounds = (chunks + 31) / 32;
  const int n_groups = (a.N + RU - 1) / RU;
  int G = blockIdx.x * (kFmaWarps / ks) + team, cr = kidx;
  uint4 cw[RU], nw[RU];
  uint32_t sb[RU], ns[RU];
  auto load = [&](int g, int round, uint4 (&w)[RU], uint32_t (&sc)[RU]) {
    const int c = round * 32 + lane;
#pragma unroll
    for (int j = 0; j < RU; ++j) {
      const int n = g * RU + j;
      w[j] = make_uint4(0u, 0u, 0u, 0u);
      sc[j] = 0u;
      if (g < n_groups && n < a.N && c < chunks) {
        w[j] = __ldcs(reinterpret_cast<const uint4*>(a.codes + static_cast<size_t>(n) * (a.K / 2) +
                                                     16 * c));
        sc[j] = *reinterpret_cast<const uint16_t*>(a.scales + static_cast<size_t>(n) * (a.K / 16) +
                                                   2 * c);
      }
    }
  };
  load(G, kidx, cw, sb);
  const float gs = *a.gscale;  // (a weight-side constant too)

  pdl_wait();
  pdl_launch_dependents();

  // ---- the CTA's activation rows.  Segment v (elements 8 v ..) of a row is
  // 16-byte slot v % 4 of chunk v / 4 of the row's staging area; thread t
  // takes segments v = t + 256 i.  The first kKeep segments of every row are
  // loaded at once, all in flight together, and stay in registers (K up to
  // 8192 for one or two rows, 4096 for four; the rest of a longer row is
  // loaded again for the conversion).
  const int segs = a.K / 8;
  auto seg_addr = [&](int r, int v) {
    return xs + static_cast<uint32_t>(r * rs + (v >> 2) * kChunkPitch + (v & 3) * 16);
  };
  constexpr int kKeep = MB == 4 ? 2 : 4;
  uint4 keep[MB][kKeep];
#pragma unroll
  for (int r = 0; r < MB; ++r) {
    const __nv_bfloat16* row = a.A + static_cast<size_t>(m0 + r) * a.lda;
#pragma unroll
    for (int i = 0; i < kKeep; ++i) {
      const int v = threadIdx.x + kFmaThreads * i;
      keep[r][i] = (r < mb && v < segs) ? __ldcg(reinterpret_cast<const uint4*>(row + 8 * v))
                                        : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // ---- per row: the largest magnitude and the plain sum of squares, one
  // reduction over the CTA; then the FP16 shift and the RMS factor (rows
  // above 2^56 sum their shifted squares in a second pass: no overflow at
  // any magnitude)
  {
    float mx[MB], sq[MB];
    auto add = [&](int r, const uint4 q) {
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
        mx[r] = fmaxf(mx[r], fmaxf(fabsf(lo), fabsf(hi)));
        sq[r] = fmaf(lo, lo, fmaf(hi, hi, sq[r]));
      }
    };
#pragma unroll
    for (int r = 0; r < MB; ++r) {
      mx[r] = 0.0f;
      sq[r] = 0.0f;
#pragma unroll
      for (int i = 0; i < kKeep; ++i) add(r, keep[r][i]);
      if (r < mb)
        for (int v = threadIdx.x + kFmaThreads * kKeep; v < segs; v += kFmaThreads)
          add(r, __ldcg(reinterpret_cast<const uint4*>(a.A + static_cast<size_t>(m0 + r) * a.lda +
                                                       8 * v)));
    }
    // the rows' warp reductions side by side (same order as warp_max / warp_sum)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int r = 0; r < MB; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], o));
        sq[r] += __shfl_xor_sync(0xffffffffu, sq[r], o);
      }
    if (lane == 0)
#pragma unroll
      for (int r = 0; r < MB; ++r) {
        s_bv[warp][r] = mx[r];
        s_sq[warp][r] = sq[r];
      }
    __syncthreads();
    if (threadIdx.x < MB) {
      const int r = threadIdx.x;
      float rmax = 0.0f, rsq = 0.0f;
      for (int w = 0; w < kFmaWarps; ++w) {
        rmax = fmaxf(rmax, s_bv[w][r]);
        rsq += s_sq[w][r];
      }
      s_sh[r] = r < mb ? f16_row_shift(rmax) : 0;
      s_rms[r] = (!a.rms || r >= mb) ? 1.0f : (rmax > kSumsqSafeMax ? -1.0f : rms_plain(rsq, a.K));
    }
    __syncthreads();
  }
  for (int r = 0; r < MB; ++r) {
    if (s_rms[r] < 0.0f) {  // uniform over the CTA (rare)
      const __nv_bfloat16* row = a.A + static_cast<size_t>(m0 + r) * a.lda;
      const int sh = s_sh[r];
      const int h1 = (sh > 126 || sh < -126) ? sh / 2 : sh;
      const float f1 = exp2i(h1), f2 = exp2i(sh - h1);
      float s3 = 0.0f;
      for (int v = threadIdx.x; v < a.K / 8; v += kFmaThreads) {
        const uint4 q = __ldcg(reinterpret_cast<const uint4*>(row + 8 * v));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = __uint_as_float(w[j] << 16) * f1 * f2;
          const float hi = __uint_as_float(w[j] & 0xFFFF0000u) * f1 * f2;
          s3 = fmaf(lo, lo, fmaf(hi, hi, s3));
        }
      }
      const float s4 = cta_sum0(s3, s_w);
      if (threadIdx.x == 0) s_rms[r] = rms_factor(s4, sh, a.K);
      __syncthreads();
    }
  }
  // the shifted FP16 rows (rows past the CTA's are zero)
  auto to_f16 = [&](const uint4 v, int sh) {
    const int h1 = (sh > 126 || sh < -126) ? sh / 2 : sh;
    const float f1 = exp2i(h1), f2 = exp2i(sh - h1);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      p[j] = pack_f16x2(__uint_as_float(w[j] << 16) * f1 * f2,
                        __uint_as_float(w[j] & 0xFFFF0000u) * f1 * f2);
    return make_uint4(p[0], p[1], p[2], p[3]);
  };
#pragma unroll
  for (int r = 0; r < MB; ++r) {
    const int sh = s_sh[r];
#pragma unroll
    for (int i = 0; i < kKeep; ++i) {
      const int v = threadIdx.x + kFmaThreads * i;
      if (v < segs) st_shared_v4(seg_addr(r, v), to_f16(keep[r][i], sh));
    }
    for (int v = threadIdx.x + kFmaThreads * kKeep; v < segs; v += kFmaThreads) {
      uint4 q = make_uint4(0u, 0u, 0u, 0u);
      if (r < mb)
        q = __ldcg(reinterpret_cast<const uint4*>(a.A + static_cast<size_t>(m0 + r) * a.lda + 8 * v));
      st_shared_v4(seg_addr(r, v), to_f16(q, sh));
    }
  }
  __syncthreads();

  // ---- rows of W
  // output = (row sum x 2^-shift) x tensor scale x RMS factor, in that order
  // (the undone shift alone could fall below FP32's range)
  float am_v[MB];
  int am_i[MB];
#pragma unroll
  for (int r = 0; r < MB; ++r) {
    am_v[r] = -FLT_MAX;
    am_i[r] = 0x7fffffff;
  }
  float acc[MB][RU];
#pragma unroll
  for (int r = 0; r < MB; ++r)
#pragma unroll
    for (int j = 0; j < RU; ++j) acc[r][j] = 0.0f;
  while (G < n_groups) {
    // the next item's loads first
    const bool last = cr + ks >= rounds;  // this warp's last round of the group
    const int nG = last ? G + n_teams : G;
    const int ncr = last ? kidx : cr + ks;
    load(nG, ncr, nw, ns);
    const int c = cr * 32 + lane;
    if (c < chunks) {
      const uint32_t cbase = xs + static_cast<uint32_t>(c * kChunkPitch);
      if constexpr (MB <= 2) {
#pragma unroll
        for (int r = 0; r < MB; ++r) {
          uint32_t xv[16];
          ld_chunk(cbase + static_cast<uint32_t>(r * rs), xv);
#pragma unroll
          for (int j = 0; j < RU; ++j) acc[r][j] = nvfp4_chunk_dot(cw[j], sb[j], xv, acc[r][j]);
        }
      } else {  // decode each weight chunk once for all the rows
        Nvfp4Chunk ch[RU];
#pragma unroll
        for (int j = 0; j < RU; ++j) ch[j] = nvfp4_decode_chunk(cw[j], sb[j]);
#pragma unroll
        for (int r = 0; r < MB; ++r) {
          if (r >= mb) break;  // (uniform) rows past M
          uint32_t xv[16];
          ld_chunk(cbase + static_cast<uint32_t>(r * rs), xv);
#pragma unroll
          for (int j = 0; j < RU; ++j) acc[r][j] = nvfp4_chunk_dot(ch[j], xv, acc[r][j]);
        }
      }
    }
    if (last) {  // the group's rows are complete
      // the warp sums of all the group's outputs side by side (the order of
      // warp_sum)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int j = 0; j < RU; ++j)
#pragma unroll
          for (int r = 0; r < MB; ++r) acc[r][j] += __shfl_xor_sync(0xffffffffu, acc[r][j], o);
      if (ks > 1) {
        // each warp's sums to shared memory; the team's first warp adds
        // them in warp order (a named barrier per team)
        if (lane == 0)
#pragma unroll
          for (int j = 0; j < RU; ++j)
#pragma unroll
            for (int r = 0; r < MB; ++r) s_part[warp * 16 + r * RU + j] = acc[r][j];
        team_sync(team, ks);
        if (kidx == 0) {
#pragma unroll
          for (int j = 0; j < RU; ++j)
#pragma unroll
            for (int r = 0; r < MB; ++r) {
              float t = 0.0f;
              for (int k = 0; k < ks; ++k) t += s_part[(warp + k) * 16 + r * RU + j];
              acc[r][j] = t;
            }
        }
      }
#pragma unroll
      for (int j = 0; j < RU; ++j) {
        const int n = G * RU + j;
#pragma unroll
        for (int r = 0; r < MB; ++r) {
          const float t = acc[r][j];
          acc[r][j] = 0.0f;
          if (kidx == 0 && r < mb && n < a.N) {
            const __nv_bfloat16 o =
                __float2bfloat16_rn(scale_pow2(t, -s_sh[r]) * gs * (a.rms ? s_rms[r] : 1.0f));
            if (lane == 0) a.C[static_cast<size_t>(m0 + r) * a.ldc + n] = o;
            const float ov = __bfloat162float(o);
            if (fm_better(ov, n, am_v[r], am_i[r])) {
              am_v[r] = ov;
              am_i[r] = n;
            }
          }
        }
      }
      if (ks > 1) team_sync(team, ks);  // (s_part is free again)
    }
    G = nG;
    cr = ncr;
#pragma unroll
    for (int j = 0; j < RU; ++j) {
      cw[j] = nw[j];
      sb[j] = ns[j];
    }
  }

  // ---- argmax: the CTA's best per row, then the last CTA of the row group
  // reduces the partials of every CTA (the order of (value, index) pairs is
  // total, so the result does not depend on arrival order)
  if (!a.argmax_out) return;
#pragma unroll
  for (int r = 0; r < MB; ++r) {
    float bv = am_v[r];
    int bi = am_i[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi != 0x7fffffff && fm_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      s_bv[warp][r] = bv;
      s_bi[warp][r] = bi;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int r = 0; r < mb; ++r) {
      float bv = -FLT_MAX;
      int bi = 0x7fffffff;
      for (int w = 0; w < kFmaWarps; ++w)
        if (s_bi[w][r] != 0x7fffffff && fm_better(s_bv[w][r], s_bi[w][r], bv, bi)) {
          bv = s_bv[w][r];
          bi = s_bi[w][r];
        }
      a.am_part[static_cast<size_t>(m0 + r) * gridDim.x + blockIdx.x] =
          make_int2(__float_as_int(bv), bi);
    }
    // releases this CTA's partials; the last adder acquires the others'
    const uint32_t prev = atom_add_acq_rel_gpu(a.argmax_cnt + blockIdx.y, 1u);
    s_last = prev == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  for (int r = warp; r < mb; r += kFmaWarps) {
    float bv = -FLT_MAX;
    int bi = 0x7fffffff;
    for (int j = lane; j < static_cast<int>(gridDim.x); j += 32) {
      const int2 pr = __ldcg(a.am_part + static_cast<size_t>(m0 + r) * gridDim.x + j);
      const float v = __int_as_float(pr.x);
      if (pr.y != 0x7fffffff && fm_better(v, pr.y, bv, bi)) {
        bv = v;
        bi = pr.y;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi != 0x7fffffff && fm_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) a.argmax_out[m0 + r] = (a.am_map && bi != 0x7fffffff) ? a.am_map[bi] : bi;
  }
  if (threadIdx.x == 0) a.argmax_cnt[blockIdx.y] = 0u;
}

template <int MB, int RU>
cudaError_t launch_mb(const FmaArgs& a, int grid, cudaStream_t s, bool pdl) {
  const size_t smem = fma_smem_bytes(MB, a.K);
  cudaError_t e = cudaFuncSetAttribute(fma_kernel<MB, RU>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem < 1024 ? 1024 : smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, (a.M + MB - 1) / MB);  // (MB = fma_rows_per_cta(M, K))
  cfg.blockDim = dim3(kFmaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fma_kernel<MB, RU>, a);
}

}  // namespace

constexpr size_t kFmaMaxSmem = 200 * 1024;

size_t fma_smem_bytes(int rows_per_cta, int K) {
  return static_cast<size_t>(rows_per_cta) * (K / 32) * kChunkPitch;
}

int fma_rows_per_cta(int M, int K) {
  // (more rows run as row groups of four: measured on GB300, eight- and
  // sixteen-row CTAs, which decode each weight chunk once for all their
  // rows, lost to row groups of four at every shape, e.g. 2048 x 4096 at M
  // = 8 17.5 vs 8.7 us, 1024 x 2048 at M = 16 22.3 vs 6.2 us)
  int mb = M <= 1 ? 1 : M <= 2 ? 2 : 4;
  while (mb > 1 && fma_smem_bytes(mb, K) > kFmaMaxSmem) mb /= 2;  // (long rows)
  return mb;
}

// Rows a warp takes at once.  More rows keep more bytes in flight per warp
// but leave fewer warps a group when N is small.  Measured on GB300 (K =
// 2048 unless stated, back-to-back calls, us for rows a warp = 2 / 4 / 8):
//   M = 1: 2048 x 4096 4.28 / 4.85 / 6.34; 4096 rows 4.02 / 3.51 / 4.62;
//          8192 rows 5.85 / 4.19 / 5.21; 16384 rows 9.13 / 6.58 / 6.43;
//          32768 rows 14.72 / 11.15 / 10.85;
//   M = 2 (1 / 2 / 4): 4096 rows 5.38 / 4.63 / 5.05; 8192 rows 8.02 / 6.83 / 6.58;
//   M = 4 (1 / 2): 4096 rows 8.29 / 7.77; 5120 rows 9.73 / 9.48.
int fma_rows_per_warp(int rows_per_cta, int N) {
  // (thresholds for GB300's 152 SMs)
  if (rows_per_cta == 1) return N < 3072 ? 2 : (N < 12288 ? 4 : 8);
  if (rows_per_cta == 2) return N < 6144 ? 2 : 4;
  return 2;
}

int fma_k_split(long groups, int rounds, long warp_slots) {
  // Rows of 4 or more rounds (K >= 4096) over few groups: the widest team
  // (4, 2 warps) that leaves each warp a round and keeps the grid within
  // 128 CTAs.  Measured on GB300, back-to-back calls, K = 4096, us for teams
  // of 1 / 2 / 4 warps: 64 rows M = 1 3.1 / 2.7 / 2.3, M = 4 7.1 / 6.6 /
  // 5.8; 1024 rows M = 1 4.3 / 3.8 / 5.5, 2048 rows M = 1 5.1 / 6.4 / 7.1.
  // At K = 2048 (two rounds) a team gains at most 0.2 us or loses.
  if (rounds < 4) return 1;
  const long cap = warp_slots < 1024 ? warp_slots : 1024;
  for (int ks = 4; ks > 1; ks >>= 1)
    if (ks <= rounds && groups * ks <= cap) return ks;
  return 1;
}

cudaError_t launch_fma(const FmaArgs& a, int grid, int ru, cudaStream_t s, bool pdl) {
  switch (fma_rows_per_cta(a.M, a.K) * 16 + ru) {
    case 16 + 8: return launch_mb<1, 8>(a, grid, s, pdl);
    case 16 + 4: return launch_mb<1, 4>(a, grid, s, pdl);
    case 16 + 2: return launch_mb<1, 2>(a, grid, s, pdl);
    case 32 + 4: return launch_mb<2, 4>(a, grid, s, pdl);
    case 32 + 2: return launch_mb<2, 2>(a, grid, s, pdl);
    case 64 + 2: return launch_mb<4, 2>(a, grid, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nvfp4
