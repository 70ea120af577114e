// Expert schedule of a routed MoE layer, rebuilt from the top-k ids in every
// CTA that needs it (deterministic; no host round trip).
//   cnt[e]       number of (token, slot) pairs routed to expert e (e == E is
//                the shared expert: all T tokens)
//   off[e]       exclusive prefix sum of cnt: pairs of e are off[e] ..
//                off[e] + cnt[e] - 1, ordered by flat slot t*k + j
//   active[a]    the experts with cnt > 0, ascending (shared expert last)
//   flat_pair[p] pair index of flat slot p (-1 for an id outside [0, E))
//   pair_tok[q]  token of pair q
#pragma once

#include "common.cuh"

namespace nvfp4 {

struct Sched {
  int* cnt;        // [E+1]
  int* off;        // [E+2]
  int* active;     // [E+1]
  int* run;        // [E+1]
  int* flat_pair;  // [P]
  int* pair_tok;   // [P+T]
  int* n_active;   // [1]
};

__device__ __forceinline__ Sched sched_layout(uint8_t* base, int E, int P) {
  int* p = reinterpret_cast<int*>(base);
  Sched s;
  s.cnt = p;
  s.off = s.cnt + (E + 1);
  s.active = s.off + (E + 2);
  s.run = s.active + (E + 1);
  s.flat_pair = s.run + (E + 1);
  s.pair_tok = s.flat_pair + P;
  s.n_active = s.pair_tok + P + 32;
  return s;
}

// Scan of the counts into offsets and the active list, then the pairs:
// one warp (lanes 0..31), after cnt[] holds the counts and run[] zeros.
__device__ __forceinline__ void schedule_tail_warp(const int32_t* ids, int T, int k, int E,
                                                   int has_shared, const Sched& s, int lane) {
  const int P = T * k;
  int carry = 0, acarry = 0;
  for (int base = 0; base <= E; base += 32) {
    const int i = base + lane;
    const int c = (i <= E) ? s.cnt[i] : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (i <= E) s.off[i] = carry + incl - c;
    const unsigned bal = __ballot_sync(0xffffffffu, c > 0);
    if (c > 0) s.active[acarry + __popc(bal & ((1u << lane) - 1u))] = i;
    carry += __shfl_sync(0xffffffffu, incl, 31);
    acarry += __popc(bal);
  }
  if (lane == 0) {
    s.off[E + 1] = carry;
    *s.n_active = acarry;
  }
  __syncwarp();
  for (int base = 0; base < P; base += 32) {
    const int p = base + lane;
    const int id = (p < P) ? ids[p] : -1;
    const bool valid = (p < P) && id >= 0 && id < E;
    const unsigned grp = __match_any_sync(0xffffffffu, valid ? id : -1 - lane);
    if (valid) {
      const int pr = s.off[id] + s.run[id] + __popc(grp & ((1u << lane) - 1u));
      s.flat_pair[p] = pr;
      s.pair_tok[pr] = p / k;
    } else if (p < P) {
      s.flat_pair[p] = -1;
    }
    __syncwarp();
    if (valid && lane == 31 - __clz(grp)) s.run[id] += __popc(grp);
    __syncwarp();
  }
  if (has_shared)
    for (int t = lane; t < T; t += 32) s.pair_tok[s.off[E] + t] = t;
  __syncwarp();
}

// All threads of the CTA.  Deterministic: the result does not depend on
// the order of the shared-memory atomics.
static __device__ void build_schedule(const int32_t* ids, int T, int k, int E, int has_shared,
                                      const Sched& s, uint32_t* status) {
  const int P = T * k;
  const int tid = threadIdx.x, nthr = blockDim.x;
  for (int i = tid; i <= E; i += nthr) {
    s.cnt[i] = 0;
    s.run[i] = 0;
  }
  __syncthreads();
  bool bad = false;
  for (int p = tid; p < P; p += nthr) {
    const int id = ids[p];
    if (id >= 0 && id < E)
      atomicAdd(&s.cnt[id], 1);
    else
      bad = true;
  }
  if (bad && blockIdx.x == 0) atomicOr(status, kStatusBadId);
  if (tid == 0) s.cnt[E] = has_shared ? T : 0;
  __syncthreads();
  if ((tid >> 5) == 0) schedule_tail_warp(ids, T, k, E, has_shared, s, tid & 31);
  __syncthreads();
}

// The same schedule built by one warp alone (the other warps go on working).
static __device__ void build_schedule_warp(const int32_t* ids, int T, int k, int E,
                                           int has_shared, const Sched& s, uint32_t* status,
                                           int lane) {
  const int P = T * k;
  for (int i = lane; i <= E; i += 32) {
    s.cnt[i] = 0;
    s.run[i] = 0;
  }
  __syncwarp();
  bool bad = false;
  for (int p = lane; p < P; p += 32) {
    const int id = ids[p];
    if (id >= 0 && id < E)
      atomicAdd(&s.cnt[id], 1);
    else
      bad = true;
  }
  if (bad && blockIdx.x == 0) atomicOr(status, kStatusBadId);
  __syncwarp();
  if (lane == 0) s.cnt[E] = has_shared ? T : 0;
  __syncwarp();
  schedule_tail_warp(ids, T, k, E, has_shared, s, lane);
}

}  // namespace nvfp4
