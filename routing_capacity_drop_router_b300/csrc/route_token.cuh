// Per-token routing from fp32 logits for one 128-token tile: used by the
// stand-alone routing kernel and by the tail of the tensor-core router.
//
// "Understanding Mixture of Experts", section "Expert and Router": the router
// activates the TopK(G(x), k) experts of each token with G(x) = softmax of the
// logits. "Capacity-Aware Inference: Mitigating the Straggler Effect in MoE",
// section 2 (2) Expanded Drop: m extra candidates from the token's own device.
//
//   logits: L = the tile's slices added in slot order (+ bias), staged in
//           shared memory with coalesced loads;
//   scores: m = max L; u_e = score_exp(L_e - m); Z = u_0 + u_1 + ... (in
//           order); p_e = u_e / Z (correctly rounded); one thread per token;
//   top-k:  k passes, each taking the largest (key, -e) pair below the
//           previous pass's pair in the order key descending, expert
//           ascending (ties to the lower expert);
//   expanded: m more passes restricted to the home group's experts;
//   gates:  p of the slot; with renorm divided by the slots' left-to-right sum.
//   column sums (load statistics): p_e in fixed point (units of 2^-40,
//           rounded half up, by integer operations on the fp32 bits) summed
//           per tile in u64, so the sum is exact and independent of the order
//           of the additions.
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

// Per-token routing of token t from its logits s_row[0..N) (shared memory),
// in compact loops over the experts (the code runs once per tile, so its size
// matters more than unrolling). Writes the token's candidates and gates and
// returns its softmax max and denominator in *mx_out, *z_out; the scores are
// recomputed from them later, bit-identically.
//
// The j-th candidate is the largest (key, -e) pair below the (j-1)-th one in
// the order "key descending, then expert ascending", so no expert needs to be
// marked as taken; the expanded candidates are the largest pairs of the home
// group below the k-th top-k pair.
__device__ __forceinline__ void route_one_token(const RouteArgs& a, int t, const float* s_row,
                                                float* mx_out, float* z_out) {
  const int N = a.N;
  float mx = s_row[0];
  for (int e = 1; e < N; ++e) mx = fmaxf(mx, s_row[e]);
  float Z = score_exp(__fsub_rn(s_row[0], mx));
  for (int e = 1; e < N; ++e) Z = __fadd_rn(Z, score_exp(__fsub_rn(s_row[e], mx)));
  *mx_out = mx;
  *z_out = Z;
  if (a.ec) return;

  const int k = a.k, kc = a.k + a.m;
  int32_t* idx_out = a.cand_idx + static_cast<size_t>(t) * kc;
  float* gate_out = a.cand_gate + static_cast<size_t>(t) * kc;
  float g[32];
  uint32_t prev_key = 0xffffffffu;  // pair bound: (prev_key, prev_e); start above all
  int prev_e = -1;
  uint32_t kth_key = 0u;
  int kth_e = -1;
  int lo = 0, hi = N;
  for (int j = 0; j < kc; ++j) {
    if (j == k) {  // expanded candidates: the home group, below the k-th pair
      const int G = N / a.group_size;
      const int hg = a.home_group ? a.home_group[t]
                                  : static_cast<int>((static_cast<long long>(t) * G) / a.T);
      lo = hg * a.group_size;
      hi = lo + a.group_size;
      prev_key = kth_key;
      prev_e = kth_e;
    }
    int best = -1;
    uint32_t bk = 0u;
    for (int e = lo; e < hi; ++e) {
      const uint32_t ke = order_key(s_row[e]);
      // below the bound in (key desc, e asc) order, and above the best so far
      const bool below = ke < prev_key || (ke == prev_key && e > prev_e);
      if (below && (best < 0 || ke > bk)) {
        bk = ke;
        best = e;
      }
    }
    idx_out[j] = best;
    g[j] = best >= 0 ? __fdiv_rn(score_exp(__fsub_rn(s_row[best], mx)), Z) : 0.f;
    if (best >= 0) {
      prev_key = bk;
      prev_e = best;
    }
    if (j == k - 1) {
      kth_key = prev_key;
      kth_e = prev_e;
    }
  }
  if (a.renorm) {
    float S = g[0];
    for (int j = 1; j < kc; ++j) S = __fadd_rn(S, g[j]);
    for (int j = 0; j < kc; ++j) g[j] = __fdiv_rn(g[j], S);
  }
  for (int j = 0; j < kc; ++j) gate_out[j] = g[j];
}

// Shared memory route_tile needs: the tile's [128, N + 1] fp32 staging array,
// N u64 column sums (8-byte aligned: 128 * (N + 1) * 4 is a multiple of 8),
// then each token's softmax max and denominator.
__host__ __device__ constexpr size_t route_tile_smem(int N) {
  return static_cast<size_t>(kRouteTile) * (N + 1) * sizeof(float) +
         static_cast<size_t>(N) * sizeof(unsigned long long) +
         2 * static_cast<size_t>(kRouteTile) * sizeof(float);
}

// Calls f(r, e, q) for every element of a [rows, N] tile (q = r * N + e), with
// consecutive threads on consecutive elements of a row.
template <typename F>
__device__ __forceinline__ void for_tile_elements(int rows, int N, F&& f) {
  const int nt = static_cast<int>(blockDim.x), tid = static_cast<int>(threadIdx.x);
  if (N <= nt) {
    const int rpi = nt / N, e = tid % N, r0 = tid / N;
    if (r0 < rpi)
      for (int r = r0; r < rows; r += rpi) f(r, e, r * N + e);
  } else {
    for (int r = 0; r < rows; ++r)
      for (int e = tid; e < N; e += nt) f(r, e, r * N + e);
  }
}

// Routes tokens [tile*128, tile*128 + 128) (blockDim.x == kRouteTile, one
// token per thread) from the tile's logit slices, writes logits_out, scores,
// candidates and gates, and (a.colsum) the tile's column sums of p.
// s_l: route_tile_smem(N) bytes of shared memory. Call uniformly from every
// thread of the block.
__device__ __forceinline__ void route_tile(const RouteArgs& a, int tile, float* s_l) {
  const int N = a.N, ld = N + 1;
  const int t0 = tile * kRouteTile;
  const int rows = min(kRouteTile, a.T - t0);
  const int nslots =
      a.seg_ctas ? router_tile_segments(tile, a.seg_kb, a.seg_ctas, a.seg_total) : 1;
  const float* base = a.partial + static_cast<size_t>(tile) * a.max_slots * kRouteTile * N;
  const size_t slot_stride = static_cast<size_t>(kRouteTile) * N;
  // 1. the tile's logits: slices added in slot order, then the bias. With
  //    N % 4 == 0 each thread sums 4-element vectors, 4 vectors x 4 slices of
  //    loads in flight per round (the slices were just written by other CTAs
  //    and are read through L2).
  if ((N & 3) == 0) {
    constexpr int kU = 4, kS = 4;
    const int nvec = rows * N / 4;
    const float4* b4 = reinterpret_cast<const float4*>(base);
    const size_t stride4 = slot_stride / 4;
    for (int v0 = threadIdx.x; v0 < nvec; v0 += blockDim.x * kU) {
      float4 acc[kU];
      for (int s0 = 0; s0 < nslots; s0 += kS) {
        float4 t[kS][kU];
#pragma unroll
        for (int ss = 0; ss < kS; ++ss)
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const int v = v0 + u * static_cast<int>(blockDim.x);
            if (s0 + ss < nslots && v < nvec) t[ss][u] = __ldcg(b4 + (s0 + ss) * stride4 + v);
          }
#pragma unroll
        for (int ss = 0; ss < kS; ++ss)
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const int v = v0 + u * static_cast<int>(blockDim.x);
            if (s0 + ss < nslots && v < nvec) {
              if (s0 + ss == 0) {
                acc[u] = t[ss][u];
              } else {
                acc[u].x = __fadd_rn(acc[u].x, t[ss][u].x);
                acc[u].y = __fadd_rn(acc[u].y, t[ss][u].y);
                acc[u].z = __fadd_rn(acc[u].z, t[ss][u].z);
                acc[u].w = __fadd_rn(acc[u].w, t[ss][u].w);
              }
            }
          }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int v = v0 + u * static_cast<int>(blockDim.x);
        if (v < nvec) {
          const int q = 4 * v, r = q / N, e = q - r * N;  // 4 elements of one row
          float4 o = acc[u];
          if (a.bias) {
            o.x = __fadd_rn(o.x, a.bias[e]);
            o.y = __fadd_rn(o.y, a.bias[e + 1]);
            o.z = __fadd_rn(o.z, a.bias[e + 2]);
            o.w = __fadd_rn(o.w, a.bias[e + 3]);
          }
          if (a.logits_out)
            *reinterpret_cast<float4*>(a.logits_out + static_cast<size_t>(t0) * N + q) = o;
          float* dst = s_l + r * ld + e;
          dst[0] = o.x;
          dst[1] = o.y;
          dst[2] = o.z;
          dst[3] = o.w;
        }
      }
    }
  } else {
    for_tile_elements(rows, N, [&](int r, int e, int q) {
      float v = __ldcg(base + q);
      for (int s = 1; s < nslots; ++s) v = __fadd_rn(v, __ldcg(base + s * slot_stride + q));
      if (a.bias) v = __fadd_rn(v, a.bias[e]);
      if (a.logits_out) a.logits_out[static_cast<size_t>(t0) * N + q] = v;
      s_l[r * ld + e] = v;
    });
  }
  __syncthreads();
  // 2. one token per thread
  unsigned long long* s_cs = reinterpret_cast<unsigned long long*>(s_l + kRouteTile * ld);
  float* s_mx = reinterpret_cast<float*>(s_cs + N);
  float* s_z = s_mx + kRouteTile;
  if (static_cast<int>(threadIdx.x) < rows)
    route_one_token(a, t0 + threadIdx.x, s_l + threadIdx.x * ld, s_mx + threadIdx.x,
                    s_z + threadIdx.x);
  for (int e = threadIdx.x; e < N; e += blockDim.x) s_cs[e] = 0ull;
  __syncthreads();
  // 3. scores p = score_exp(L - max) / Z, recomputed element-wise with
  //    coalesced stores (scores, expert-choice gates) and kept in s_l for the
  //    column sums
  for_tile_elements(rows, N, [&](int r, int e, int q) {
    const float p = __fdiv_rn(score_exp(__fsub_rn(s_l[r * ld + e], s_mx[r])), s_z[r]);
    if (a.scores) a.scores[static_cast<size_t>(t0) * N + q] = p;
    if (a.ec) a.cand_gate[static_cast<size_t>(t0) * N + q] = p;
    s_l[r * ld + e] = p;
  });
  if (a.colsum) {
    // thread (e, c) sums rows c, c + chunks, ...; the u64 partials meet in
    // shared memory (integer sums: the order does not matter)
    __syncthreads();
    const int chunks = N <= static_cast<int>(blockDim.x) ? static_cast<int>(blockDim.x) / N : 1;
    for (int e = static_cast<int>(threadIdx.x) % N; e < N; e += static_cast<int>(blockDim.x)) {
      const int c = static_cast<int>(threadIdx.x) / N;
      if (c >= chunks) break;
      unsigned long long acc = 0ull;
      for (int r = c; r < rows; r += chunks) acc += fixed40(s_l[r * ld + e]);
      atomicAdd(&s_cs[e], acc);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < N; e += blockDim.x)
      a.colsum[static_cast<size_t>(tile) * N + e] = s_cs[e];
  }
}

}  // namespace moe
