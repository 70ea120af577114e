// MoE decode layer for a few tokens on the CUDA cores.
//
// With T tokens and top-k routing the layer is T * k (+ T shared) pairs of a
// token and an expert, each a matrix-vector product with one activation row:
// one FMA per weight, which the CUDA cores issue at several times the HBM
// rate, and no tensor-memory set-up, ring fill or split-K drain before the
// first byte.  Two launches:
//
//   gate/up: every warp takes (pair, two intermediate columns j, j + 1): the
//     gate rows j, j + 1 and the up rows I + j, I + j + 1 of the pair's
//     expert against the token's activation row, then
//     h[pair][j] = silu(gate) * up in FP32;
//   down + combine: every warp takes (token, output column n): row n of the
//     down matrix of each of the token's experts against that pair's h row,
//     then out[t][n] = bf16(sum over slots, in order, of w * y, the shared
//     expert's y added last).
//
// For batches of 4 to 8 tokens the gate/up step runs instead on the warp-
// level MMA used as a wide FMA (moe_mma_gate_up_kernel, below): the same
// exact products, without the per-element FMAs and half extractions that
// bound the FMA kernel's issue rate.
//
// Activations (BF16 x, FP32 h) are staged in shared memory as FP16 after a
// power-of-two shift per row that puts the row's largest magnitude in
// [2^14, 2^15) (exact for BF16 elements within 2^31 of it; one rounding for
// FP32 h), as on the tensor-core path; codes convert to FP16 exactly and
// every product code x activation is exact in FP32.  Each output is summed
// by one warp in a fixed order: deterministic, whatever the grid.
//
// Sources: "Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)", "Making decode
// faster" (decode is a few rows against 4-bit weights); the MoE layer's
// definition (routed experts, SwiGLU, weighted combine, shared expert) as
// the tensor-core path.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace nvfp4 {
namespace {

constexpr int kMfWarps = 8;
constexpr int kMfThreads = kMfWarps * 32;

// Expert of pair p: its routed id (-1 when outside [0, E): skipped), or E for
// the shared expert of token p - T k.
__device__ __forceinline__ int pair_expert(const MoeFmaArgs& a, int p) {
  const int tk = a.T * a.k;
  if (p >= tk) return a.E;
  const int e = __ldcg(a.ids + p);
  return (e >= 0 && e < a.E) ? e : -1;
}

__device__ __forceinline__ int pair_token(const MoeFmaArgs& a, int p) {
  const int tk = a.T * a.k;
  return p < tk ? p / a.k : p - tk;
}

// Rows [0, T) of x, shifted to FP16, into xs (act_off layout, H / 32 chunks a
// row) with s_sh[t] the shift and s_rms[t] the RMS factor (1 without RMS):
// warp w stages rows w, w + 8, ...; a lane keeps kKeepSeg 8-element segments
// of a row in registers between the statistics and the conversion (the rest
// it loads again).
template <int kKeepSeg>
__device__ __forceinline__ void stage_x_rows(const MoeFmaArgs& a, uint32_t xs, int* s_sh,
                                             float* s_rms, int warp, int lane) {
  const int segs = a.H / 8, chunks = a.H / 32;
  for (int t = warp; t < a.T; t += kMfWarps) {
    const __nv_bfloat16* row = a.x + static_cast<size_t>(t) * a.ldx;
    uint4 keep[kKeepSeg];
#pragma unroll
    for (int i = 0; i < kKeepSeg; ++i) {
      const int v = lane + 32 * i;
      keep[i] = v < segs ? __ldcg(reinterpret_cast<const uint4*>(row + 8 * v))
                         : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t mx = 0u;
    float sq = 0.0f;
    auto stats = [&](const uint4& q) {
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        mx = __vmaxu2(mx, w[j] & 0x7FFF7FFFu);
        const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
        sq = fmaf(lo, lo, fmaf(hi, hi, sq));
      }
    };
#pragma unroll
    for (int i = 0; i < kKeepSeg; ++i) stats(keep[i]);
    for (int v = lane + 32 * kKeepSeg; v < segs; v += 32)
      stats(__ldcg(reinterpret_cast<const uint4*>(row + 8 * v)));
    const float m = warp_max(fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xFFFF0000u)));
    const int sh = f16_row_shift(m);
    const int h1 = (sh > 126 || sh < -126) ? sh / 2 : sh;
    const float f1 = exp2i(h1), f2 = exp2i(sh - h1);
    if (a.rms) {
      if (m > kSumsqSafeMax) {  // (warp-uniform, rare) the shifted squares
        sq = 0.0f;
        for (int v = lane; v < segs; v += 32) {
          const uint4 q = __ldcg(reinterpret_cast<const uint4*>(row + 8 * v));
          const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(w[j] << 16) * f1 * f2;
            const float hi = __uint_as_float(w[j] & 0xFFFF0000u) * f1 * f2;
            sq = fmaf(lo, lo, fmaf(hi, hi, sq));
          }
        }
      }
      sq = warp_sum(sq);
    }
    if (lane == 0) {
      s_sh[t] = sh;
      s_rms[t] = !a.rms ? 1.0f : (m > kSumsqSafeMax ? rms_factor(sq, sh, a.H) : rms_plain(sq, a.H));
    }
    auto to_f16 = [&](const uint4& q) {
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = pack_f16x2(__uint_as_float(w[j] << 16) * f1 * f2,
                          __uint_as_float(w[j] & 0xFFFF0000u) * f1 * f2);
      return make_uint4(o[0], o[1], o[2], o[3]);
    };
#pragma unroll
    for (int i = 0; i < kKeepSeg; ++i) {
      const int v = lane + 32 * i;
      if (v < segs) st_shared_v4(xs + act_off(t, v >> 2, v & 3, chunks), to_f16(keep[i]));
    }
    for (int v = lane + 32 * kKeepSeg; v < segs; v += 32)
      st_shared_v4(xs + act_off(t, v >> 2, v & 3, chunks),
                   to_f16(__ldcg(reinterpret_cast<const uint4*>(row + 8 * v))));
  }
}

// ---------------------------------------------------------------- gate / up
__global__ void __launch_bounds__(kMfThreads, 2) moe_fma_gate_up_kernel(const MoeFmaArgs a) {
  extern __shared__ __align__(16) uint8_t msm[];
  __shared__ int s_e[kMoeFmaMaxPairs];
  __shared__ float s_g[kMoeFmaMaxPairs];
  __shared__ int s_sh[kMoeFmaMaxT];
  __shared__ float s_rms[kMoeFmaMaxT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t xs = smem_u32(msm);
  const int H = a.H, I = a.I, chunks = H / 32;
  const int rounds = (chunks + 31) / 32;
  const int P = a.T * a.k + (a.has_shared ? a.T : 0);
  const int per_p = I / 2;  // items of a pair: two intermediate columns each
  const int n_items = P * per_p;
  const int n_warps = gridDim.x * kMfWarps;
  const size_t e_codes = static_cast<size_t>(2 * I) * (H / 2);
  const size_t e_scales = static_cast<size_t>(2 * I) * (H / 16);

  // the pairs' experts and gate/up scales (a bad id sets the status bit once)
  auto read_pairs = [&]() {
    for (int p = threadIdx.x; p < P; p += kMfThreads) {
      const int e = pair_expert(a, p);
      s_e[p] = e;
      s_g[p] = e < 0 ? 0.0f : (e == a.E ? *a.s_gu_global : a.gu_global[e]);
      if (e < 0 && blockIdx.x == 0) atomicOr(a.status, kStatusBadId);
    }
    __syncthreads();
  };

  // item g: the four weight rows gate j, j + 1, up j, j + 1 of pair p's
  // expert (j = 2 (g % per_p)); round `round` of the K chunks
  constexpr int RU = 4;
  auto load = [&](int g, int round, uint4 (&w)[RU], uint32_t (&sc)[RU]) {
    const int c = round * 32 + lane;
#pragma unroll
    for (int j = 0; j < RU; ++j) {
      w[j] = make_uint4(0u, 0u, 0u, 0u);
      sc[j] = 0u;
    }
    if (g >= n_items || c >= chunks) return;
    const int p = g / per_p, j0 = 2 * (g - p * per_p);
    const int e = s_e[p];
    if (e < 0) return;
    const uint8_t* cb = e == a.E ? a.s_gu_codes : a.gu_codes + e * e_codes;
    const uint8_t* sb = e == a.E ? a.s_gu_scales : a.gu_scales + e * e_scales;
#pragma unroll
    for (int j = 0; j < RU; ++j) {
      const int r = (j < 2 ? 0 : I) + j0 + (j & 1);
      w[j] = __ldcs(reinterpret_cast<const uint4*>(cb + static_cast<size_t>(r) * (H / 2) + 16 * c));
      sc[j] = *reinterpret_cast<const uint16_t*>(sb + static_cast<size_t>(r) * (H / 16) + 2 * c);
    }
  };

  int G = blockIdx.x * kMfWarps + warp, cr = 0;
  uint4 cw[RU], nw[RU];
  uint32_t sb[RU], ns[RU];
  if (a.ids_ready) {
    read_pairs();
    load(G, 0, cw, sb);
  }
  pdl_wait();
  pdl_launch_dependents();
  if (!a.ids_ready) {
    read_pairs();
    load(G, 0, cw, sb);
  }
  stage_x_rows<8>(a, xs, s_sh, s_rms, warp, lane);
  __syncthreads();

  float acc[RU];
#pragma unroll
  for (int j = 0; j < RU; ++j) acc[j] = 0.0f;
  while (G < n_items) {
    const int nG = cr + 1 < rounds ? G : G + n_warps;
    const int ncr = cr + 1 < rounds ? cr + 1 : 0;
    load(nG, ncr, nw, ns);
    const int p = G / per_p;
    const int t = pair_token(a, p);
    const int c = cr * 32 + lane;
    if (c < chunks) {
      uint32_t xv[16];
      ld_act_chunk(xs, t, c, chunks, xv);
#pragma unroll
      for (int j = 0; j < RU; ++j) acc[j] = nvfp4_chunk_dot(cw[j], sb[j], xv, acc[j]);
    }
    if (cr + 1 == rounds) {  // the item's rows are complete
      float tot[RU];
#pragma unroll
      for (int j = 0; j < RU; ++j) {
        tot[j] = warp_sum(acc[j]);
        acc[j] = 0.0f;
      }
      if (lane == 0 && s_e[p] >= 0) {
        const int j0 = 2 * (G - p * per_p);
        const float f = s_g[p] * s_rms[t];
        float hv[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float gt = scale_pow2(tot[u], -s_sh[t]) * f;
          const float up = scale_pow2(tot[2 + u], -s_sh[t]) * f;
          hv[u] = gt / (1.0f + expf(-gt)) * up;
        }
        *reinterpret_cast<float2*>(a.h + static_cast<size_t>(p) * I + j0) = make_float2(hv[0], hv[1]);
      }
    }
    G = nG;
    cr = ncr;
#pragma unroll
    for (int j = 0; j < RU; ++j) {
      cw[j] = nw[j];
      sb[j] = ns[j];
    }
  }
}

// ---------------------------------------------------------------- gate / up by warp MMAs
// The same layer step with the warp-level MMA (m16n8k16, FP16 operands, FP32
// accumulation) as a wide FMA: the products code x scale x activation are
// exact, as above, and only the order of the FP32 additions differs.  A warp
// takes items (pair p, eight intermediate columns j0 .. j0 + 7): tile rows
// 0 .. 7 are the gate rows j0 + g and tile rows 8 .. 15 the up rows
// I + j0 + g of p's expert, and the activation operand is p's token row in
// all eight columns.  Lane (g, q) = (lane / 4, lane % 4) loads, per 128-K
// chunk c, the 32 codes 128 c + 32 q .. + 31 of its rows g and g + 8 (16
// bytes each) and their two block scales, and the same 32 staged
// activations of the token; k-step i of the chunk gives the MMA's K slots
// {2q, 2q + 1} and {2q + 8, 2q + 9} the elements 128 c + 32 q + 4 i .. + 3
// in that order in both operands, so each k-step sums 16 distinct products
// of the row's dot product.  The codes are decoded and multiplied by their
// block scales in FP16 (exact) into the A fragments; the FP32 accumulators
// of lane (g, 0) end with row g's gate and up sums, which it turns into
// h[p][j0 + g].  Loads run kMmaStages chunks ahead.
constexpr int kMmaStages = 4;

struct MmaChunk {
  uint4 w0, w1;  // codes of tile rows g and g + 8
  uint32_t sc;   // their two block scales each: row g low half, row g + 8 high half
};

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kMfThreads, 2) moe_mma_gate_up_kernel(const MoeFmaArgs a) {
  extern __shared__ __align__(16) uint8_t msm[];
  __shared__ int s_e[kMoeFmaMaxPairs];
  __shared__ float s_g[kMoeFmaMaxPairs];
  __shared__ int s_sh[kMoeFmaMaxT];
  __shared__ float s_rms[kMoeFmaMaxT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const uint32_t xs = smem_u32(msm);
  const int H = a.H, I = a.I, chunks = H / 32, nc = H / 128;
  const int P = a.T * a.k + (a.has_shared ? a.T : 0);
  const int per_p = I / 8;  // items of a pair (a power of two)
  const int per_p_log2 = __ffs(per_p) - 1;
  const int n_items = P * per_p;
  const int n_warps = gridDim.x * kMfWarps;
  const size_t e_codes = static_cast<size_t>(2 * I) * (H / 2);
  const size_t e_scales = static_cast<size_t>(2 * I) * (H / 16);

  auto read_pairs = [&]() {
    for (int p = threadIdx.x; p < P; p += kMfThreads) {
      const int e = pair_expert(a, p);
      s_e[p] = e;
      s_g[p] = e < 0 ? 0.0f : (e == a.E ? *a.s_gu_global : a.gu_global[e]);
      if (e < 0 && blockIdx.x == 0) atomicOr(a.status, kStatusBadId);
    }
    __syncthreads();
  };

  // load cursor: item lg, chunk lc, and the item's tile row g (codes, scales;
  // null: no rows, the loads give zeros); row g + 8 lies I rows further
  int lg = blockIdx.x * kMfWarps + warp, lc = 0;
  const uint8_t *c0p = nullptr, *s0p = nullptr;
  const size_t c_up = static_cast<size_t>(I) * (H / 2), s_up = static_cast<size_t>(I) * (H / 16);
  auto item_rows = [&]() {
    c0p = s0p = nullptr;
    if (lg >= n_items) return;
    const int p = lg >> per_p_log2, j0 = 8 * (lg & (per_p - 1));
    const int e = s_e[p];
    if (e < 0) return;
    const uint8_t* cb = e == a.E ? a.s_gu_codes : a.gu_codes + e * e_codes;
    const uint8_t* sb = e == a.E ? a.s_gu_scales : a.gu_scales + e * e_scales;
    const size_t r0 = j0 + g;
    c0p = cb + r0 * (H / 2) + 16 * q;
    s0p = sb + r0 * (H / 16) + 2 * q;
  };
  auto load_next = [&](MmaChunk& b) {
    b.w0 = b.w1 = make_uint4(0u, 0u, 0u, 0u);
    b.sc = 0u;
    if (c0p) {
      const uint8_t* cp = c0p + 64 * lc;
      const uint8_t* sp = s0p + 8 * lc;
      b.w0 = __ldcs(reinterpret_cast<const uint4*>(cp));
      b.w1 = __ldcs(reinterpret_cast<const uint4*>(cp + c_up));
      b.sc = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(sp)) |
             (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(sp + s_up)) << 16);
    }
    if (++lc == nc) {
      lc = 0;
      lg += n_warps;
      item_rows();
    }
  };

  MmaChunk buf[kMmaStages];
  auto prologue = [&]() {
    read_pairs();
    item_rows();
#pragma unroll
    for (int j = 0; j < kMmaStages; ++j) load_next(buf[j]);
  };
  if (a.ids_ready) prologue();
  pdl_wait();
  pdl_launch_dependents();
  if (!a.ids_ready) prologue();
  stage_x_rows<4>(a, xs, s_sh, s_rms, warp, lane);  // (fewer registers: the loads in flight)
  __syncthreads();

  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int G = blockIdx.x * kMfWarps + warp; G < n_items; G += n_warps) {
    const int p = G >> per_p_log2;
    const int t = pair_token(a, p);
    for (int cb = 0; cb < nc; cb += kMmaStages) {
#pragma unroll
      for (int j = 0; j < kMmaStages; ++j) {
        const MmaChunk cur = buf[j];
        load_next(buf[j]);  // kMmaStages chunks ahead
        uint32_t xv[16];
        ld_act_chunk(xs, t, 4 * (cb + j) + q, chunks, xv);
        uint32_t s0lo, s0hi, s1lo, s1hi;
        e4m3x2_bcast_f16x2(cur.sc & 0xFFFFu, s0lo, s0hi);
        e4m3x2_bcast_f16x2(cur.sc >> 16, s1lo, s1hi);
        const uint32_t w0[4] = {cur.w0.x, cur.w0.y, cur.w0.z, cur.w0.w};
        const uint32_t w1[4] = {cur.w1.x, cur.w1.y, cur.w1.z, cur.w1.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {  // word w: elements 8 w .. 8 w + 7 (k-steps 2 w, 2 w + 1)
          uint32_t d0, d1, d2, d3, e0, e1, e2, e3;
          e2m1x8_to_f16x2(w0[w], d0, d1, d2, d3);
          e2m1x8_to_f16x2(w1[w], e0, e1, e2, e3);
          const uint32_t sa = w < 2 ? s0lo : s0hi, sb = w < 2 ? s1lo : s1hi;
          mma_16816(acc, hmul2(d0, sa), hmul2(e0, sb), hmul2(d1, sa), hmul2(e1, sb), xv[4 * w],
                    xv[4 * w + 1]);
          mma_16816(acc, hmul2(d2, sa), hmul2(e2, sb), hmul2(d3, sa), hmul2(e3, sb),
                    xv[4 * w + 2], xv[4 * w + 3]);
        }
      }
    }
    // lane (g, 0): acc[0] = gate row j0 + g, acc[2] = up row j0 + g (column 0)
    if (q == 0 && s_e[p] >= 0) {
      const int j0 = 8 * (G & (per_p - 1));
      const float f = s_g[p] * s_rms[t];
      const float gt = scale_pow2(acc[0], -s_sh[t]) * f;
      const float up = scale_pow2(acc[2], -s_sh[t]) * f;
      a.h[static_cast<size_t>(p) * I + j0 + g] = gt / (1.0f + expf(-gt)) * up;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = 0.0f;
  }
}

// ---------------------------------------------------------------- down + combine
// A warp takes 32 / cpr output columns n of one token (cpr = I / 32 chunks
// a down row: 8, 16 or 32); lane l works on column l / cpr, K chunk l % cpr,
// of every slot's row: the loads of all the token's slots are in flight at
// once, each slot's sum is reduced over the column's cpr lanes, and the
// combine runs in every lane of the column in slot order (the shared expert
// last).  Slots go in batches of kSlotBatch (one batch for k <= 8 with the
// shared expert).
constexpr int kSlotBatch = 9;

__global__ void __launch_bounds__(kMfThreads, 2) moe_fma_down_kernel(const MoeFmaArgs a) {
  extern __shared__ __align__(16) uint8_t msm[];
  __shared__ int s_e[kMoeFmaMaxSlots];
  __shared__ float s_w[kMoeFmaMaxSlots];
  __shared__ float s_g[kMoeFmaMaxSlots];
  __shared__ float s_f1[kMoeFmaMaxSlots];
  __shared__ float s_f2[kMoeFmaMaxSlots];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t xs = smem_u32(msm);
  const int t = blockIdx.y;
  const int H = a.H, I = a.I, cpr = I / 32, cols = 32 / cpr;
  const int S = a.k + (a.has_shared ? 1 : 0);
  const int c = lane & (cpr - 1), col = lane / cpr;
  const size_t e_codes = static_cast<size_t>(H) * (I / 2);
  const size_t e_scales = static_cast<size_t>(H) * (I / 16);

  // The slots' experts, weights and scales.  The ids are complete: this
  // kernel starts only after the gate/up kernel passed its own wait for the
  // kernel before it (or, without programmatic launch, after it ended).
  if (threadIdx.x < S) {
    const int s = threadIdx.x;
    if (s < a.k) {
      const int e = pair_expert(a, t * a.k + s);
      s_e[s] = e;
      s_w[s] = __ldcg(a.w + t * a.k + s);
      s_g[s] = e < 0 ? 0.0f : a.dn_global[e];
    } else {
      s_e[s] = a.E;
      s_w[s] = 1.0f;
      s_g[s] = *a.s_dn_global;
    }
  }
  __syncthreads();

  // row n's chunk c of the down matrices of slots b .. b + kSlotBatch - 1
  auto load = [&](int n, int b, uint4 (&w)[kSlotBatch], uint32_t (&sc)[kSlotBatch]) {
#pragma unroll
    for (int j = 0; j < kSlotBatch; ++j) {
      const int s = b + j;
      w[j] = make_uint4(0u, 0u, 0u, 0u);
      sc[j] = 0u;
      const int e = (n < H && s < S) ? s_e[s] : -1;
      if (e >= 0) {
        const uint8_t* cb = e == a.E ? a.s_dn_codes : a.dn_codes + e * e_codes;
        const uint8_t* sb = e == a.E ? a.s_dn_scales : a.dn_scales + e * e_scales;
        w[j] = __ldcs(reinterpret_cast<const uint4*>(cb + static_cast<size_t>(n) * (I / 2) + 16 * c));
        sc[j] = *reinterpret_cast<const uint16_t*>(sb + static_cast<size_t>(n) * (I / 16) + 2 * c);
      }
    }
  };

  const int n_step = gridDim.x * kMfWarps * cols;
  int n = (blockIdx.x * kMfWarps + warp) * cols + col;
  uint4 cw[kSlotBatch];
  uint32_t sb[kSlotBatch];
  load(n, 0, cw, sb);
  pdl_wait();
  pdl_launch_dependents();

  // the slots' h rows, FP32 -> FP16 times 2^sh (sh from each row's largest
  // magnitude); warp w takes slots w, w + 8, ...; skipped slots stay unread
  for (int s = warp; s < S; s += kMfWarps) {
    if (s_e[s] < 0) continue;
    const int p = s < a.k ? t * a.k + s : a.T * a.k + t;
    const float* row = a.h + static_cast<size_t>(p) * I;
    float m = 0.0f;
    for (int v = lane; v < I / 4; v += 32) {
      const float4 f = __ldcg(reinterpret_cast<const float4*>(row) + v);
      m = fmaxf(m, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
    }
    const int sh = f16_row_shift(warp_max(m));
    const int h1 = (sh > 126 || sh < -126) ? sh / 2 : sh;
    const float f1 = exp2i(h1), f2 = exp2i(sh - h1);
    if (lane == 0) {  // the factors that undo the shift, in the same two steps
      const int u1 = -sh / 2;
      s_f1[s] = exp2i(u1);
      s_f2[s] = exp2i(-sh - u1);
    }
    for (int v = lane; v < I / 8; v += 32) {
      const float4 lo = __ldcg(reinterpret_cast<const float4*>(row) + 2 * v);
      const float4 hi = __ldcg(reinterpret_cast<const float4*>(row) + 2 * v + 1);
      const uint4 o = make_uint4(pack_f16x2(lo.x * f1 * f2, lo.y * f1 * f2),
                                 pack_f16x2(lo.z * f1 * f2, lo.w * f1 * f2),
                                 pack_f16x2(hi.x * f1 * f2, hi.y * f1 * f2),
                                 pack_f16x2(hi.z * f1 * f2, hi.w * f1 * f2));
      st_shared_v4(xs + act_off(s, v >> 2, v & 3, cpr), o);
    }
  }
  __syncthreads();

  while (true) {
    // (uniform over the warp: the warp's columns are consecutive)
    if (__shfl_sync(0xffffffffu, n, 0) >= H) break;
    float out = 0.0f;
    for (int b = 0; b < S; b += kSlotBatch) {
      if (b > 0) load(n, b, cw, sb);
#pragma unroll
      for (int j = 0; j < kSlotBatch; ++j) {
        const int s = b + j;
        if (s < S && s_e[s] >= 0) {  // uniform
          uint32_t xv[16];
          ld_act_chunk(xs, s, c, cpr, xv);
          float d = nvfp4_chunk_dot(cw[j], sb[j], xv, 0.0f);
          for (int o = cpr >> 1; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
          const float y = ((d * s_f1[s]) * s_f2[s]) * s_g[s];
          out = s < a.k ? fmaf(s_w[s], y, out) : out + y;
        }
      }
    }
    if (c == 0 && n < H) a.out[static_cast<size_t>(t) * a.ldo + n] = __float2bfloat16_rn(out);
    n += n_step;
    load(n, 0, cw, sb);
  }
}

cudaError_t launch_ex(const void* fn, dim3 grid, size_t smem, cudaStream_t s, bool pdl,
                      const MoeFmaArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kMfThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  void* args[] = {const_cast<MoeFmaArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// down: T rows of CTAs, two CTAs per SM in all
cudaError_t launch_down(const MoeFmaArgs& a, int sms, size_t smem, cudaStream_t s, bool pdl) {
  const void* fn = reinterpret_cast<const void*>(moe_fma_down_kernel);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem < 1024 ? 1024 : smem));
  if (e != cudaSuccess) return e;
  const int per_warp = 32 / (a.I / 32);  // columns a warp
  int gx = (2 * sms + a.T - 1) / a.T;
  const int need = (a.H + kMfWarps * per_warp - 1) / (kMfWarps * per_warp);
  if (gx > need) gx = need;
  return launch_ex(fn, dim3(gx, a.T), smem, s, pdl, a);
}

}  // namespace

int moe_fma_slots(int k, int has_shared, int I) {
  if (I != 256 && I != 512 && I != 1024) return 0;
  const int S = k + (has_shared ? 1 : 0);
  return S <= kMoeFmaMaxSlots ? S : 0;
}

// By warp MMAs for batches of 4 to 8 tokens.  Measured on GB300 (256
// experts, H = 2048, I = 512, top-8 + shared; 40-layer decode step, us, FMAs
// / MMAs): T = 4 1,727 / 1,657, T = 8 2,792 / 2,632; with fewer tokens the
// MMA kernel's items (eight columns of a pair) leave SMs idle (T = 1 925 /
// 1,068, T = 2 1,150 / 1,240), and with batches of 16 the step slowed
// although the MoE calls alone ran faster (T = 16 4,740 / 5,424, MoE calls
// alone 80.2 / 68.8 us a layer).
bool moe_gate_up_mma(int H, int T) { return H % (128 * kMmaStages) == 0 && T >= 4 && T <= 8; }

cudaError_t launch_moe_fma(const MoeFmaArgs& a, int sms, cudaStream_t s, bool pdl) {
  const int P = a.T * a.k + (a.has_shared ? a.T : 0);
  // gate/up: one warp an item (two or, by MMAs, eight intermediate columns of
  // a pair), at most two CTAs per SM
  const bool mma = moe_gate_up_mma(a.H, a.T);
  const long items = static_cast<long>(P) * (a.I / (mma ? 8 : 2));
  const long ctas = (items + kMfWarps - 1) / kMfWarps;
  const int grid_gu = static_cast<int>(ctas < 2L * sms ? ctas : 2L * sms);
  const size_t smem_gu = static_cast<size_t>(a.T) * a.H * 2;
  const void* gu = mma ? reinterpret_cast<const void*>(moe_mma_gate_up_kernel)
                       : reinterpret_cast<const void*>(moe_fma_gate_up_kernel);
  cudaError_t e = cudaFuncSetAttribute(gu, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem_gu < 1024 ? 1024 : smem_gu));
  if (e != cudaSuccess) return e;
  if ((e = launch_ex(gu, dim3(grid_gu), smem_gu, s, pdl, a)) != cudaSuccess) return e;
  const int S = a.k + (a.has_shared ? 1 : 0);
  const size_t smem_dn = static_cast<size_t>(S) * a.I * 2;
  if (!moe_fma_slots(a.k, a.has_shared, a.I)) return cudaErrorInvalidValue;
  return launch_down(a, sms, smem_dn, s, pdl);
}

}  // namespace nvfp4
