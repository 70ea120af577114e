// Device helpers shared by the NVFP4 decode kernels (sm_103a).
//
// Inline PTX for: mbarriers with bounded waits, TMA tile loads, the hardware
// E2M1 / E4M3 -> FP16 conversions, packed FP16 multiply, GPU-scope
// counters, and programmatic dependent launch.  Every wait here is bounded by a
// wall-clock limit: on expiry it records NVFP4_STATUS_WAIT_TIMEOUT and
// returns, so a kernel never hangs the GPU.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

// ------------------------------------------------------------------ limits
constexpr int kStageK = 256;                               // K values per pipeline stage
constexpr int kMaxM = 32;                                  // activation rows per call
constexpr unsigned long long kWaitLimitNs = 2000000000ull; // 2 s per wait

constexpr uint32_t kStatusBadId = 1u;
constexpr uint32_t kStatusTimeout = 2u;

// ------------------------------------------------------------------ misc
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: wait for the upstream grid's memory, and
// allow the downstream grid to start its prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_u32(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// 16-byte global -> shared copy through L2 (cp.async.cg); src_bytes 0
// writes 16 zero bytes instead.  The thread waits for its own copies with
// cp_async_wait_all.
__device__ __forceinline__ void cp_async_16(uint32_t smem_dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

__device__ __forceinline__ void mbar_arrive_expect_tx_u32(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
      : "memory");
}

// Non-blocking test of a phase (returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// kWaitLimitNs, records the timeout in *status (global) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status) {
  const uint32_t a = smem_u32(bar);
  if (mbar_test_wait(a, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (globaltimer() - t0 > kWaitLimitNs) {
      if (status) atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// ------------------------------------------------------------------ TMA
// 2-D tiled bulk tensor load into shared memory (addresses as 32-bit
// shared-memory values); completion is signalled on `bar` as transaction
// bytes.  x = innermost coordinate (bytes for uint8 maps; always a multiple
// of 16 here), y = row.
__device__ __forceinline__ void tma_load_2d_u32(uint32_t smem_dst, const CUtensorMap* map, int x,
                                                int y, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// 4-D tiled bulk tensor load (x innermost, a multiple of 16 bytes).
__device__ __forceinline__ void tma_load_4d_u32(uint32_t smem_dst, const CUtensorMap* map, int x,
                                                int y, int z, int w, uint32_t bar,
                                                uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ decode
// Four packed bytes of E2M1 pairs -> four f16x2 (low half = even k).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& d0, uint32_t& d1,
                                                uint32_t& d2, uint32_t& d3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
      : "r"(w));
}

// Four E4M3 bytes (byte i = element i) -> two f16x2: elements 0, 1 and 2, 3
// (low half = the lower element; exact).
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& d0, uint32_t& d1) {
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(d0), "=r"(d1)
      : "r"(w));
}

// Two E4M3 bytes (low byte: first block) -> each broadcast to both halves
// of an f16x2 (exact).
__device__ __forceinline__ void e4m3x2_bcast_f16x2(uint32_t two, uint32_t& lo, uint32_t& hi) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(two & 0xFFFFu)));
  lo = __byte_perm(h2, 0u, 0x1010);
  hi = __byte_perm(h2, 0u, 0x3232);
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// ------------------------------------------------------------------ scaling
// 2^e as a float for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) {
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// Power-of-two exponent s such that |max| * 2^s lies in [2^14, 2^15): the
// row then converts to FP16 exactly (BF16 carries 8 significant bits; FP16
// keeps 11 down to 2^-14 and its largest finite value is 65504).  Zero and
// non-finite maxima give s = 0.
__device__ __forceinline__ int f16_row_shift(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int e = static_cast<int>((b >> 23) & 0xFF);
  if (amax == 0.0f || e == 0xFF) return 0;
  const int ex = (e == 0) ? -127 : e - 127;  // subnormal max: exponent below -126
  int s = 14 - ex;
  if (s > 250) s = 250;
  return s;
}

// v * 2^s exactly (two steps keep each factor representable).
__device__ __forceinline__ float scale_pow2(float v, int s) {
  const int h = s / 2;
  return (v * exp2i(h)) * exp2i(s - h);
}

// Rows whose largest magnitude is at most 2^56 have a plain FP32 sum of
// squares below 4096 * 2^112 (no overflow), and their squares that underflow
// are below 2^-149 against a sum that is then either negligible next to 1e-6
// or above 2^-100: the plain sum gives their RMS factor.
constexpr float kSumsqSafeMax = 72057594037927936.0f;  // 2^56

__device__ __forceinline__ float rms_plain(float sq, int klen) {
  return rsqrtf(sq / static_cast<float>(klen) + 1e-6f);
}

// 1 / sqrt(mean(x^2) + 1e-6) of a row of klen elements from the sum of the
// squares of its elements times 2^sh (sq), sh being the row's staging shift
// (f16_row_shift of its largest magnitude, at most 250).  Rows far below 1
// (sh > 100) have a mean square below 2^-170: the 1e-6 decides alone.
__device__ __forceinline__ float rms_factor(float sq, int sh, int klen) {
  const float m = sq / static_cast<float>(klen);  // mean of the shifted squares
  if (sh >= 0) return rsqrtf((sh > 100 ? 0.0f : scale_pow2(m, -2 * sh)) + 1e-6f);
  // large rows: 2^sh / sqrt(m + 1e-6 * 2^(2 sh)); the factor stays a normal
  // float (sh >= -113 for BF16 rows)
  return exp2i(sh) * rsqrtf(m + scale_pow2(1e-6f, 2 * sh));
}

// ------------------------------------------------------------------ CUDA-core dot products
// (the CUDA-core kernels: fma.cu, moe_fma.cu)
__device__ __forceinline__ float fma_f16(uint32_t a_half_pair, uint32_t b_half_pair, bool hi,
                                         float c) {
  float d;
  if (hi)
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a1, b1, %3;\n\t}"
        : "=f"(d) : "r"(a_half_pair), "r"(b_half_pair), "f"(c));
  else
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %3;\n\t}"
        : "=f"(d) : "r"(a_half_pair), "r"(b_half_pair), "f"(c));
  return d;
}

__device__ __forceinline__ float f16_lo_to_f32(uint32_t h2) {
  float f;
  asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}"
      : "=f"(f) : "r"(h2));
  return f;
}

// Byte offset of 16-byte slot q (0..3) of chunk c of row m in the staged
// activations: chunks of 64 bytes, slot index xor-ed with (c / 2) % 4 so
// that the eight lanes of one shared-memory phase (chunks c .. c + 7, same q)
// hit eight different 16-byte bank groups.
__device__ __forceinline__ uint32_t act_off(int m, int c, int q, int chunks) {
  return static_cast<uint32_t>(((m * chunks + c) * 4 + (q ^ ((c >> 1) & 3))) * 16);
}

// The 32 staged FP16 activations of chunk c of row m (act_off layout) as 16
// f16x2 words: elements 32 c + 2 i, 2 i + 1 in word i.
__device__ __forceinline__ void ld_act_chunk(uint32_t xs, int m, int c, int chunks,
                                             uint32_t (&xv)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = ld_shared_v4(xs + act_off(m, c, q, chunks));
    xv[4 * q] = v.x;
    xv[4 * q + 1] = v.y;
    xv[4 * q + 2] = v.z;
    xv[4 * q + 3] = v.w;
  }
}

// A 32-K chunk of an NVFP4 row decoded: 32 E2M1 codes (16 bytes, low nibble
// = even k) as 16 f16x2 words and the two 16-element blocks' E4M3 scales
// (the two bytes of sb, low byte first) as floats; all exact.
struct Nvfp4Chunk {
  uint32_t code[16];
  float sc0, sc1;
};

__device__ __forceinline__ Nvfp4Chunk nvfp4_decode_chunk(const uint4& w, uint32_t sb) {
  Nvfp4Chunk ch;
  uint32_t s2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2) : "h"(static_cast<uint16_t>(sb)));
  ch.sc0 = f16_lo_to_f32(s2);
  ch.sc1 = f16_lo_to_f32(s2 >> 16);
  const uint32_t wds[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int wi = 0; wi < 4; ++wi)
    e2m1x8_to_f16x2(wds[wi], ch.code[4 * wi], ch.code[4 * wi + 1], ch.code[4 * wi + 2],
                    ch.code[4 * wi + 3]);
  return ch;
}

// acc + the chunk's dot product with the activations xv: one FP32 sum per
// 16-element block (the products code x activation are exact in FP32), each
// block sum times its scale.
__device__ __forceinline__ float nvfp4_chunk_dot(const Nvfp4Chunk& ch, const uint32_t (&xv)[16],
                                                 float acc) {
  float b0 = 0.0f, b1 = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    b0 = fma_f16(ch.code[e], xv[e], false, b0);
    b0 = fma_f16(ch.code[e], xv[e], true, b0);
    b1 = fma_f16(ch.code[8 + e], xv[8 + e], false, b1);
    b1 = fma_f16(ch.code[8 + e], xv[8 + e], true, b1);
  }
  acc = fmaf(ch.sc0, b0, acc);
  return fmaf(ch.sc1, b1, acc);
}

__device__ __forceinline__ float nvfp4_chunk_dot(const uint4& w, uint32_t sb,
                                                 const uint32_t (&xv)[16], float acc) {
  return nvfp4_chunk_dot(nvfp4_decode_chunk(w, sb), xv, acc);
}


// ------------------------------------------------------------------ gpu-scope sync
// Counter add with acquire-release semantics at GPU scope: after a CTA
// barrier, one thread's add publishes the CTA's earlier stores (release) and
// makes the stores published by the earlier adders visible (acquire).
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// The same, release only, without a result (the caller does not wait).
__device__ __forceinline__ void red_add_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace nvfp4
