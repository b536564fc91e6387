// Per-token routing from fp32 logits by a segment of W lanes of a warp
// (W = 8, 16 or 32: the smallest that holds N experts, or 32 with several
// experts per lane); used by the routing kernel (route.cu) and by the
// tensor-core router's cluster tail (route_tc.cu).
//
// "Understanding Mixture of Experts", section "Expert and Router": the router
// activates the TopK(G(x), k) experts of each token with G(x) = softmax of the
// logits. "Capacity-Aware Inference: Mitigating the Straggler Effect in MoE",
// section 2 (2) Expanded Drop: m extra candidates from the token's own device.
//
// Lane l of the segment holds experts e = l, l + W, ... (PER of them).
//   scores: m = max L; u_e = score_exp(L_e - m); Z = u_0 + u_1 + ... (in
//           ascending e: a chain of adds through the lanes); p_e = u_e / Z
//           (correctly rounded);
//   top-k:  k passes, each a segment-wide maximum of (key, -e) over the pairs
//           below the previous pass's pair in the order key descending, expert
//           ascending (ties to the lower expert);
//   expanded: m more passes over the home group's experts, below the k-th
//           top-k pair (so the top-k experts are excluded);
//   gates:  p of the slot; with renorm divided by the slots' left-to-right sum.
//   column sums (load statistics): p_e in fixed point (units of 2^-40,
//           rounded half up, by integer operations on the fp32 bits) added in
//           u64, so the sum is exact and independent of the order of the
//           additions.
#pragma once
#include <cstdint>

#include "device_common.cuh"
#include "internal.h"

namespace moe {

// p in [0, 1] as a multiple of 2^-40, rounded half up; integer operations
// only (64-bit float conversions are slow on this part).
__device__ __forceinline__ unsigned long long fixed40(float p) {
  const uint32_t u = __float_as_uint(p);
  const int E = static_cast<int>((u >> 23) & 0xffu);  // biased exponent
  if (E == 0 || (u >> 31)) return 0ull;                // zero, subnormal (< 2^-126), negative
  const unsigned long long m = (u & 0x7fffffu) | 0x800000u;
  const int sh = E - 110;                              // p * 2^40 = m * 2^(E - 110)
  if (sh >= 0) return m << sh;
  if (sh < -25) return 0ull;                           // below half a unit
  return (m + (1ull << (-sh - 1))) >> (-sh);
}

// (key, e) packed so that a larger value is earlier in the order key
// descending, expert ascending.
__device__ __forceinline__ unsigned long long pair_of(uint32_t key, int e) {
  return (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(0xffffffffu - e);
}

template <int W>
__device__ __forceinline__ unsigned long long seg_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o, W);
    v = w > v ? w : v;
  }
  return v;
}

// Segment width and experts per lane for N experts.
__host__ __device__ constexpr int route_seg_width(int N) { return N <= 8 ? 8 : (N <= 16 ? 16 : 32); }

// Routes token t (valid: t < T; an invalid segment still takes part in the
// shuffles) whose logits the segment holds in l[0..PER) (lane l: experts
// l + W*j; entries past N are ignored). Writes scores, expert-choice gates or
// candidates and gates; adds the token's p into s_cs (shared, nullable).
template <int W, int PER>
__device__ __forceinline__ void route_token_seg(const RouteArgs& a, int t, bool valid, float (&l)[PER],
                                                unsigned long long* s_cs) {
  const int ls = static_cast<int>(threadIdx.x & 31) % W;  // lane in the segment
  const int N = a.N;
#pragma unroll
  for (int j = 0; j < PER; ++j)
    if (ls + W * j >= N) l[j] = -INFINITY;
  float mx = l[0];
#pragma unroll
  for (int j = 1; j < PER; ++j) mx = fmaxf(mx, l[j]);
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o, W));
  float u[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) u[j] = (ls + W * j < N) ? score_exp(__fsub_rn(l[j], mx)) : 0.f;
  float Z = 0.f;  // the shuffles do not depend on Z: unrolled, they are all in flight at once
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int n_here = min(W, N - W * j);
#pragma unroll
    for (int i = 0; i < W; ++i) {
      const float v = __shfl_sync(0xffffffffu, u[j], i, W);
      if (i < n_here) Z = (j == 0 && i == 0) ? v : __fadd_rn(Z, v);
    }
  }
  float p[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) p[j] = __fdiv_rn(u[j], Z);
  if (valid) {
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = ls + W * j;
      if (e < N) {
        if (a.scores) a.scores[static_cast<size_t>(t) * N + e] = p[j];
        if (a.ec) a.cand_gate[static_cast<size_t>(t) * N + e] = p[j];
        if (s_cs) atomicAdd(&s_cs[e], fixed40(p[j]));
      }
    }
  }
  if (a.ec) return;

  // candidates: passes of a segment maximum below the previous pair
  constexpr int kSlots = 32 / W;  // slots each lane keeps (kc <= 32)
  uint32_t key[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) key[j] = order_key(l[j]);
  const int k = a.k, kc = a.k + a.m;
  unsigned long long bound = ~0ull, kth = 0ull;
  int lo = 0, hi = N;
  int my_idx[kSlots];
  float my_gate[kSlots];
#pragma unroll
  for (int q = 0; q < kSlots; ++q) {
    my_idx[q] = -1;
    my_gate[q] = 0.f;
  }
  for (int jj = 0; jj < kc; ++jj) {
    if (jj == k) {  // expanded candidates: the home group, below the k-th pair
      const int G = N / a.group_size;
      const int tt = valid ? t : 0;
      const int hg = a.home_group ? a.home_group[tt]
                                  : static_cast<int>((static_cast<long long>(tt) * G) / a.T);
      lo = hg * a.group_size;
      hi = lo + a.group_size;
      bound = kth;
    }
    unsigned long long best = 0ull;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = ls + W * j;
      if (e >= lo && e < hi && e < N) {
        const unsigned long long pr = pair_of(key[j], e);
        if (pr < bound && pr > best) best = pr;
      }
    }
    best = seg_max_u64<W>(best);
    const int e_best = best ? static_cast<int>(0xffffffffu - static_cast<uint32_t>(best)) : -1;
    float pv = 0.f;
    const int jo = e_best >= 0 ? e_best / W : 0;
#pragma unroll
    for (int j = 0; j < PER; ++j)
      if (j == jo) pv = p[j];
    const float g = __shfl_sync(0xffffffffu, pv, e_best >= 0 ? e_best % W : 0, W);
    if (e_best >= 0) bound = best;
#pragma unroll
    for (int q = 0; q < kSlots; ++q)
      if (jj == ls + W * q) {
        my_idx[q] = e_best;
        my_gate[q] = e_best >= 0 ? g : 0.f;
      }
    if (jj == k - 1) kth = bound;
  }
  if (a.renorm) {  // left-to-right sum of the slot gates
    float S = 0.f;
#pragma unroll
    for (int q = 0; q < kSlots; ++q)
#pragma unroll
      for (int i = 0; i < W; ++i) {
        const int jj = q * W + i;
        if (jj < kc) {
          const float v = __shfl_sync(0xffffffffu, my_gate[q], i, W);
          S = (jj == 0) ? v : __fadd_rn(S, v);
        }
      }
#pragma unroll
    for (int q = 0; q < kSlots; ++q) my_gate[q] = __fdiv_rn(my_gate[q], S);
  }
  if (valid) {
#pragma unroll
    for (int q = 0; q < kSlots; ++q) {
      const int jj = ls + W * q;
      if (jj < kc) {
        a.cand_idx[static_cast<size_t>(t) * kc + jj] = my_idx[q];
        a.cand_gate[static_cast<size_t>(t) * kc + jj] = my_gate[q];
      }
    }
  }
}

}  // namespace moe
