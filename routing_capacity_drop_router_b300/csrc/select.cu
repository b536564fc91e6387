// Per-expert selection: capacity-aware token drop and expert-choice top-c.
//
// "Capacity-Aware Inference: Mitigating the Straggler Effect in MoE", section
// 2 (1) Token Drop: an expert keeps at most C = gamma * N_bar candidates,
// dropping those with the lowest gating score. "MoE vs MoT: routing and
// inference cost", section "Mixture of Tokens": each expert takes the c tokens
// of the batch with the highest router score.
//
// One CTA per expert e:
//  1. ordered compaction of e's candidates (scan of the [T, kc] slot table in
//     token order) into a shared-memory list of (flat slot, gate key);
//  2. if the list is longer than the capacity, a 4-pass 8-bit radix select
//     over the 32-bit gate keys finds the capacity-th largest key K* and how
//     many candidates equal to K* survive (the first ones in token order);
//  3. an ordered pass writes each candidate's rank among the kept (ascending
//     token) or -1.
// Keys are distinct up to ties of equal gates, and ties are settled by list
// (token) order, so the kept set is unique and independent of thread timing.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelMaxTokens = 24576;  // 8 bytes of shared memory per list entry

// Exclusive prefix count of `pred` over the CTA in thread order; `total`
// receives the CTA-wide count. Contains __syncthreads: call uniformly.
__device__ __forceinline__ int cta_exclusive_count(bool pred, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const unsigned b = __ballot_sync(0xffffffffu, pred);
  if (lane == 0) warp_sums[warp] = __popc(b);
  __syncthreads();
  if (warp == 0) {
    int v = (lane < nwarps) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += n;
    }
    warp_sums[lane] = v;  // inclusive
  }
  __syncthreads();
  const int excl = (warp ? warp_sums[warp - 1] : 0) + __popc(b & ((1u << lane) - 1u));
  total = warp_sums[nwarps - 1];
  __syncthreads();
  return excl;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(
    const int32_t* __restrict__ cand_idx, const float* __restrict__ cand_gate, int T, int kc,
    int N, int expert_choice, int cap, int32_t* __restrict__ slot, uint8_t* __restrict__ keep,
    int32_t* __restrict__ demand, int32_t* __restrict__ kept) {
  extern __shared__ __align__(16) unsigned char sel_smem[];
  int32_t* lflat = reinterpret_cast<int32_t*>(sel_smem);
  uint32_t* lkey = reinterpret_cast<uint32_t*>(lflat + T);
  __shared__ int warp_sums[32];
  __shared__ unsigned hist[256];
  __shared__ int s_bin, s_need;

  const int e = blockIdx.x;
  const int total = expert_choice ? T : T * kc;

  // 1. ordered compaction of expert e's candidates
  int n = 0;
  for (int start = 0; start < total; start += blockDim.x) {
    const int i = start + threadIdx.x;
    bool pred = false;
    int flat = 0;
    float g = 0.f;
    if (i < total) {
      if (expert_choice) {
        flat = i * N + e;
        pred = true;
        g = cand_gate[flat];
      } else {
        const int ce = cand_idx[i];
        flat = i;
        pred = (ce == e);
        if (pred) {
          g = cand_gate[i];
        } else if (e == 0 && (ce < 0 || ce >= N)) {  // empty slot: claimed by CTA 0
          slot[i] = -1;
          if (keep) keep[i] = 0;
        }
      }
    }
    int tot;
    const int pos = n + cta_exclusive_count(pred, warp_sums, tot);
    if (pred) {
      if (pos < T) {
        lflat[pos] = flat;
        lkey[pos] = order_key(g);
      } else {  // only if a token lists the same expert twice: not selectable
        slot[flat] = -1;
        if (keep) keep[flat] = 0;
      }
    }
    n += tot;
  }
  __syncthreads();
  const int n_all = n;  // candidates counted, reported as demand
  if (n > T) n = T;

  if (n <= cap) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      slot[lflat[i]] = i;
      if (keep) keep[lflat[i]] = 1;
    }
  } else {
    // 2. radix select of the cap-th largest key (cap >= 1 here; cap <= 0 keeps none)
    uint32_t prefix = 0u, pmask = 0u;
    int need = cap;
    if (cap > 0) {
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
          const uint32_t kk = lkey[i];
          if ((kk & pmask) == prefix) atomicAdd(&hist[(kk >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
          // lane owns bins [8*lane, 8*lane + 8); walk down from bin 255
          const int lane = threadIdx.x;
          unsigned c[8], sum = 0u;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            c[q] = hist[8 * lane + q];
            sum += c[q];
          }
          unsigned suf = sum;  // inclusive suffix over lanes >= lane
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned v = __shfl_down_sync(0xffffffffu, suf, o);
            if (lane + o < 32) suf += v;
          }
          const unsigned above = suf - sum;  // keys in bins of higher lanes
          const bool hit = above < static_cast<unsigned>(need) && static_cast<unsigned>(need) <= suf;
          const unsigned hb = __ballot_sync(0xffffffffu, hit);
          if (lane == __ffs(hb) - 1) {
            unsigned cum = above;
            int bin = 8 * lane;
            for (int q = 7; q >= 0; --q) {
              if (cum + c[q] >= static_cast<unsigned>(need)) {
                bin = 8 * lane + q;
                break;
              }
              cum += c[q];
            }
            s_bin = bin;
            s_need = need - static_cast<int>(cum);
          }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(s_bin) << shift;
        pmask |= 255u << shift;
        need = s_need;
        __syncthreads();
      }
    }
    const uint32_t thr = prefix;
    const int need_eq = (cap > 0) ? need : 0;  // candidates equal to thr that stay

    // 3. ordered keep pass: rank among kept, ascending token
    int eq_base = 0, k_base = 0;
    for (int start = 0; start < n; start += blockDim.x) {
      const int i = start + threadIdx.x;
      const uint32_t kk = (i < n) ? lkey[i] : 0u;
      const bool is_eq = (i < n) && cap > 0 && kk == thr;
      int eq_tot;
      const int eq_rank = eq_base + cta_exclusive_count(is_eq, warp_sums, eq_tot);
      const bool kp = (i < n) && cap > 0 && (kk > thr || (is_eq && eq_rank < need_eq));
      int k_tot;
      const int r = k_base + cta_exclusive_count(kp, warp_sums, k_tot);
      if (i < n) {
        slot[lflat[i]] = kp ? r : -1;
        if (keep) keep[lflat[i]] = kp ? 1 : 0;
      }
      eq_base += eq_tot;
      k_base += k_tot;
    }
  }
  if (threadIdx.x == 0) {
    const int k_e = n < cap ? n : (cap > 0 ? cap : 0);
    // expert choice drops nothing: an expert's demand is the c tokens it takes
    demand[e] = expert_choice ? k_e : n_all;
    kept[e] = k_e;
  }
}

}  // namespace

int select_max_tokens() { return kSelMaxTokens; }

cudaError_t launch_select(const int32_t* cand_idx, const float* cand_gate, int T, int kc, int N,
                          int expert_choice, int cap, int32_t* slot, uint8_t* keep,
                          int32_t* demand, int32_t* kept, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(T) * 8;
  static bool attr_set[64] = {};  // per device; setting it twice is harmless
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    err = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSelMaxTokens * 8);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  select_kernel<<<N, kSelThreads, smem, s>>>(cand_idx, cand_gate, T, kc, N, expert_choice, cap,
                                             slot, keep, demand, kept);
  return cudaGetLastError();
}

}  // namespace moe
