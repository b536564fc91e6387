// Per-token routing from fp32 logits by a segment of W lanes of a warp;
// used by the routing kernel (route.cu) and by the tensor-core router's
// cluster tail (route_tc.cu).
//
// "Understanding Mixture of Experts", section "Expert and Router": the router
// activates the TopK(G(x), k) experts of each token with G(x) = softmax of the
// logits. "Capacity-Aware Inference: Mitigating the Straggler Effect in MoE",
// section 2 (2) Expanded Drop: m extra candidates from the token's own device.
//
// Lane l of the segment holds the contiguous experts e = l*PER ... l*PER +
// PER - 1 (route_seg_width and route_seg_per pick W and PER for N: 8 lanes up
// to 64 experts, so one warp routes 4 tokens at once).
//   scores: m = max L; u_e = score_exp(L_e - m); Z = u_0 + u_1 + ... in
//           ascending e: each lane adds its own run of experts to the running
//           sum it receives from the lane before (W shuffles, PER adds each);
//           p_e = u_e / Z (correctly rounded);
//   top-k:  k passes, each a segment-wide maximum of (key, -e) over the pairs
//           below the previous pass's pair in the order key descending, expert
//           ascending (ties to the lower expert);
//   expanded: m more passes over the home group's experts, below the k-th
//           top-k pair (so the top-k experts are excluded);
//   gates:  p of the slot; with renorm divided by the slots' left-to-right sum.
//   column sums (load statistics): the caller adds p_e in fixed point
//           (units of 2^-40, rounded half up, by integer operations on the
//           fp32 bits) in u64, so the sum is exact and independent of the
//           order of the additions; the segment leaves p in a shared row for
//           that (p_row), which avoids contended shared atomics.
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

// Column sums of p over the rows of a shared [rows, N] block: thread e adds
// fixed40(p[i][e]) over the rows (exact u64 sums, any order), four
// independent partial sums for overlap. Call after the rows are written.
__device__ __forceinline__ void colsum_rows(const float* p, int rows, int N,
                                            unsigned long long* out_row) {
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    unsigned long long c0 = 0ull, c1 = 0ull, c2 = 0ull, c3 = 0ull;
    int i = 0;
    for (; i + 3 < rows; i += 4) {
      c0 += fixed40(p[i * N + e]);
      c1 += fixed40(p[(i + 1) * N + e]);
      c2 += fixed40(p[(i + 2) * N + e]);
      c3 += fixed40(p[(i + 3) * N + e]);
    }
    for (; i < rows; ++i) c0 += fixed40(p[i * N + e]);
    out_row[e] = c0 + c1 + c2 + c3;
  }
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

// Segment width W and experts per lane PER for N experts (W * PER >= N).
__host__ __device__ constexpr int route_seg_width(int N) { return N <= 64 ? 8 : (N <= 128 ? 16 : 32); }
__host__ __device__ constexpr int route_seg_per(int N) {
  return N <= 8 ? 1 : (N <= 16 ? 2 : (N <= 32 ? 4 : 8));
}

// Routes token t (valid: t < T; an invalid segment still takes part in the
// shuffles) whose logits the segment holds in l[0..PER) (lane ls: experts
// ls*PER + j; entries past N are ignored). Writes scores, expert-choice gates
// or candidates and gates; with p_row (shared, nullable) also p_row[e] = p_e
// for a valid token.
template <int W, int PER>
__device__ __forceinline__ void route_token_seg(const RouteArgs& a, int t, bool valid, float (&l)[PER],
                                                float* p_row) {
  const int ls = static_cast<int>(threadIdx.x & 31) % W;  // lane in the segment
  const int N = a.N;
  const int e0 = ls * PER;
#pragma unroll
  for (int j = 0; j < PER; ++j)
    if (e0 + j >= N) l[j] = -INFINITY;
  float mx = l[0];
#pragma unroll
  for (int j = 1; j < PER; ++j) mx = fmaxf(mx, l[j]);
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o, W));
  float u[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) u[j] = (e0 + j < N) ? score_exp(__fsub_rn(l[j], mx)) : 0.f;
  // Z in ascending e: lane r continues the running sum of lanes < r
  float Z = 0.f;
#pragma unroll
  for (int r = 0; r < W; ++r) {
    if (ls == r) {
#pragma unroll
      for (int j = 0; j < PER; ++j)
        if (e0 + j < N) Z = (e0 + j == 0) ? u[j] : __fadd_rn(Z, u[j]);
    }
    Z = __shfl_sync(0xffffffffu, Z, r, W);
  }
  float p[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) p[j] = __fdiv_rn(u[j], Z);
  if (valid) {
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = e0 + j;
      if (e < N) {
        if (a.scores) a.scores[static_cast<size_t>(t) * N + e] = p[j];
        if (a.ec) a.cand_gate[static_cast<size_t>(t) * N + e] = p[j];
        if (p_row) p_row[e] = p[j];
      }
    }
  }
  if (a.ec) return;

  // candidates: passes of a segment maximum below the previous pair
  uint32_t key[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) key[j] = order_key(l[j]);
  const int k = a.k, kc = a.k + a.m;
  unsigned long long bound = ~0ull, kth = 0ull;
  int lo = 0, hi = N;
  float S = 0.f;  // left-to-right sum of the slot gates (every lane)
  int32_t* out_idx = a.cand_idx + static_cast<size_t>(valid ? t : 0) * kc;
  float* out_gate = a.cand_gate + static_cast<size_t>(valid ? t : 0) * kc;
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
      const int e = e0 + j;
      if (e >= lo && e < hi && e < N) {
        const unsigned long long pr = pair_of(key[j], e);
        if (pr < bound && pr > best) best = pr;
      }
    }
    best = seg_max_u64<W>(best);
    const int e_best = best ? static_cast<int>(0xffffffffu - static_cast<uint32_t>(best)) : -1;
    float pv = 0.f;
    const int jo = e_best >= 0 ? e_best % PER : 0;
#pragma unroll
    for (int j = 0; j < PER; ++j)
      if (j == jo) pv = p[j];
    // one shuffle for the whole warp (its segments may differ in e_best)
    const float g0 = __shfl_sync(0xffffffffu, pv, e_best >= 0 ? e_best / PER : 0, W);
    const float g = e_best >= 0 ? g0 : 0.f;
    if (e_best >= 0) bound = best;
    S = (jj == 0) ? g : __fadd_rn(S, g);
    if (valid && ls == jj % W) {
      out_idx[jj] = e_best;
      out_gate[jj] = g;
    }
    if (jj == k - 1) kth = bound;
  }
  if (a.renorm && valid) {
    __syncwarp();
    for (int jj = ls; jj < kc; jj += W) out_gate[jj] = __fdiv_rn(out_gate[jj], S);
  }
}

}  // namespace moe
