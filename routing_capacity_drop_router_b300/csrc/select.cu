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
// (The layer's load statistics are written by the dispatch kernel, which
// runs next and overlaps them with its row copies.)
//
// Device-level capacity ("Capacity-Aware Inference", section 2 (3)): the
// experts of a device, a group of group_size consecutive experts, share one
// capacity. With group_size <= 16 the group's CTAs form a thread-block
// cluster: every radix pass sums the CTAs' histograms of their own lists
// through distributed shared memory, and a candidate equal to the threshold
// key learns its rank among the group's equal candidates in (token, slot)
// order by binary searches in the other CTAs' tie lists. Without a cluster
// (larger groups, or more than kTieMax ties in one CTA) every CTA of the group
// streams the candidate table through the same radix passes and finds the
// last kept equal candidate by an ordered scan of the table.
// Keys are distinct up to ties of equal gates, and ties are settled by list
// (token) order, so the kept set is unique and independent of thread timing.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using tc::cluster_rank;
using tc::cluster_sync;
using tc::map_to_rank;
using tc::smem_u32;

constexpr int kSelThreads = 1024;
constexpr int kSelRounds = 8;             // 32-entry rounds per warp per pass
constexpr int kSelPass = kSelThreads * kSelRounds;  // list entries per block pass
constexpr int kSelMaxTokens = 24576;      // 8 bytes of shared memory per list entry
constexpr int kTieMax = 4096;             // tie list of a clustered device group (4 bytes each)
constexpr int kMaxClusterGroup = 16;

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Exclusive prefix over warps of each warp's total (lane-uniform input);
// `total` receives the block's sum. Contains __syncthreads: call uniformly.
__device__ __forceinline__ int warp_exclusive_offset(int warp_total, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  if (lane == 0) warp_sums[warp] = warp_total;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < nwarps) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int excl = warp ? warp_sums[warp - 1] : 0;
  total = warp_sums[nwarps - 1];
  __syncthreads();
  return excl;
}

// The same with two barriers: `warp_sums` must alternate between two
// 32-int buffers on consecutive calls (the call after next reuses a buffer
// only after every warp has passed the intervening call's first barrier, so
// after it has read this call's sums).
__device__ __forceinline__ int warp_exclusive_offset2(int warp_total, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  if (lane == 0) warp_sums[warp] = warp_total;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < nwarps) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  total = warp_sums[nwarps - 1];
  return warp ? warp_sums[warp - 1] : 0;
}

// Warp 0: given a 256-bin histogram and `need` (>= 1) keys still to place,
// find the bin that holds the need-th largest key and how many of the keys to
// place fall in it (s_bin, s_need).
__device__ __forceinline__ void radix_pick(const unsigned* hist, int need, int* s_bin, int* s_need) {
  const int lane = threadIdx.x & 31;
  // lane owns bins [8*lane, 8*lane + 8); walk down from bin 255
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
    *s_bin = bin;
    *s_need = need - static_cast<int>(cum);
  }
}

// Warp-level pick over a 256-bin histogram (bin and need lane-uniform).
// Lane l reads bins l, l + 32, ... (no bank conflicts): the 32-bin block
// holding the need-th largest key is found from the top by warp sums, then
// the bin inside it by a suffix scan over the lanes.
__device__ __forceinline__ void radix_pick_warp(const unsigned* hist, int need, int& bin_out,
                                                int& need_out) {
  const int lane = threadIdx.x & 31;
  unsigned c[8], t[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) t[q] = c[q] = hist[32 * q + lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {  // the eight block sums side by side
#pragma unroll
    for (int q = 0; q < 8; ++q) t[q] += __shfl_xor_sync(0xffffffffu, t[q], o);
  }
  unsigned above = 0u;  // keys in the blocks above the chosen one
  int q = 0;
  unsigned cb = c[0];  // this lane's count in the chosen block
  bool found = false;
#pragma unroll
  for (int j = 7; j >= 0; --j) {
    if (!found && above + t[j] >= static_cast<unsigned>(need)) {
      found = true;
      q = j;
      cb = c[j];
    } else if (!found) {
      above += t[j];
    }
  }
  // inclusive suffix over lanes >= lane inside block q
  unsigned suf = cb;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned v = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += v;
  }
  const unsigned a = above + suf - cb;  // keys in higher bins
  const bool hit = a < static_cast<unsigned>(need) && static_cast<unsigned>(need) <= a + cb;
  const unsigned hb = __ballot_sync(0xffffffffu, hit);
  const int src = __ffs(hb) - 1;
  bin_out = 32 * q + src;
  need_out = need - static_cast<int>(__shfl_sync(0xffffffffu, a, src));
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(
    const int32_t* __restrict__ cand_idx, const float* __restrict__ cand_gate, int T, int kc,
    int N, int expert_choice, int cap, int group_size, int clustered, int32_t* __restrict__ slot,
    uint8_t* __restrict__ keep, int32_t* __restrict__ demand, int32_t* __restrict__ kept) {
  extern __shared__ __align__(16) unsigned char sel_smem[];
  int32_t* lflat = reinterpret_cast<int32_t*>(sel_smem);
  uint32_t* lkey = reinterpret_cast<uint32_t*>(lflat + T);
  __shared__ int warp_sums[32];
  __shared__ int warp_sums2[2 * 32];  // alternating buffers of warp_exclusive_offset2
  int scan_use = 0;
  __shared__ unsigned hist[256];
  __shared__ unsigned hsum[256];
  __shared__ unsigned hist3[3 * 256];  // per-expert radix: three rotating histograms
  __shared__ int s_bin, s_need, s_bound, s_fits, s_count, s_over;

  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();
  pdl_wait();

  // 1. ordered compaction of expert e's candidates into the shared list
  int n = 0;
  if (expert_choice) {
    n = T;
    for (int i0 = threadIdx.x; i0 < T; i0 += blockDim.x * kSelRounds) {
      float gv[kSelRounds];  // all loads in flight before the stores
#pragma unroll
      for (int j = 0; j < kSelRounds; ++j) {
        const int i = i0 + j * static_cast<int>(blockDim.x);
        gv[j] = i < T ? cand_gate[static_cast<size_t>(i) * N + e] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kSelRounds; ++j) {
        const int i = i0 + j * static_cast<int>(blockDim.x);
        if (i < T) {
          lflat[i] = i * N + e;
          lkey[i] = order_key(gv[j]);
        }
      }
    }
  } else {
    // pass: warp w takes entries [base + 256 w, base + 256 w + 256) in 32-entry
    // rounds (coalesced loads, conflict-free shared stores); ballots order the
    // matches inside a round, one block scan orders the warps
    const int total = T * kc;
    const unsigned lt = (1u << lane) - 1u;
    for (int base = 0; base < total; base += kSelPass) {
      const int w0 = base + (static_cast<int>(threadIdx.x) >> 5) * (32 * kSelRounds) + lane;
      int ce[kSelRounds];
      float gv[kSelRounds];  // gates loaded with the experts: every load in flight at once
      int cnt = 0;
#pragma unroll
      for (int j = 0; j < kSelRounds; ++j) {
        const int i = w0 + 32 * j;
        ce[j] = (i < total) ? cand_idx[i] : N;  // N: no expert, and not an empty slot
        gv[j] = (i < total) ? cand_gate[i] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kSelRounds; ++j) {
        const int i = w0 + 32 * j;
        cnt += __popc(__ballot_sync(0xffffffffu, ce[j] == e));
        if (e == 0 && i < total && (ce[j] < 0 || ce[j] >= N)) {  // empty slots: block 0
          slot[i] = -1;
          if (keep) keep[i] = 0;
        }
      }
      int tot;
      int pos = n + warp_exclusive_offset2(cnt, warp_sums2 + 32 * (scan_use++ & 1), tot);
#pragma unroll
      for (int j = 0; j < kSelRounds; ++j) {
        const int i = w0 + 32 * j;
        const unsigned b = __ballot_sync(0xffffffffu, ce[j] == e);
        if (ce[j] == e) {
          const int p = pos + __popc(b & lt);
          if (p < T) {
            lflat[p] = i;
            lkey[p] = order_key(gv[j]);
          } else {  // only if a token lists the same expert twice: not selectable
            slot[i] = -1;
            if (keep) keep[i] = 0;
          }
        }
        pos += __popc(b);
      }
      n += tot;
    }
  }
  __syncthreads();
  const int n_all = n;  // candidates counted, reported as demand
  if (n > T) n = T;
  int k_e = n < cap ? n : (cap > 0 ? cap : 0);  // kept by expert e

  if (group_size > 0) {
    // ---- device-level capacity: threshold of the whole group ----
    const int lo = (e / group_size) * group_size, hi = lo + group_size;
    const int total = T * kc;
    uint32_t prefix = 0u, pmask = 0u;
    int need = cap;
    bool all_kept = false;
    if (cap > 0 && clustered) {  // the group's demand: everything fits?
      if (threadIdx.x == 0) s_count = n;
      __syncthreads();
      cluster_sync();
      if (threadIdx.x == 0) {
        unsigned sum = 0u;
        for (int r = 0; r < group_size; ++r)
          sum += ld_cluster_u32(map_to_rank(smem_u32(&s_count), r));
        s_fits = sum <= static_cast<unsigned>(cap);
      }
      __syncthreads();
      all_kept = s_fits != 0;
      cluster_sync();  // s_count is reused below
    }
    if (cap > 0 && !all_kept) {
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
        __syncthreads();
        if (clustered) {  // this CTA's own list
          for (int i0 = 0; i0 < n; i0 += blockDim.x) {  // uniform trip count per warp
            const int i = i0 + static_cast<int>(threadIdx.x);
            int bin = -1;
            if (i < n) {
              const uint32_t kk = lkey[i];
              if ((kk & pmask) == prefix) bin = static_cast<int>((kk >> shift) & 255u);
            }
            const unsigned peers = __match_any_sync(0xffffffffu, bin);
            if (bin >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
          }
          __syncthreads();
          cluster_sync();  // every CTA's histogram is complete
          if (threadIdx.x < 256) {
            unsigned sum = 0u;
            for (int r = 0; r < group_size; ++r)
              sum += ld_cluster_u32(map_to_rank(smem_u32(&hist[threadIdx.x]), r));
            hsum[threadIdx.x] = sum;
          }
          __syncthreads();
          if (threadIdx.x < 32) radix_pick(hsum, need, &s_bin, &s_need);
          __syncthreads();
          cluster_sync();  // the peers have read this CTA's histogram
        } else {  // the whole candidate table
          for (int i0 = 0; i0 < total; i0 += blockDim.x * 4) {  // uniform trip count
            int ce[4];
            float gv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int i = i0 + j * static_cast<int>(blockDim.x) + static_cast<int>(threadIdx.x);
              ce[j] = i < total ? cand_idx[i] : -1;
              gv[j] = i < total ? cand_gate[i] : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              int bin = -1;
              if (ce[j] >= lo && ce[j] < hi) {
                const uint32_t kk = order_key(gv[j]);
                if ((kk & pmask) == prefix) bin = static_cast<int>((kk >> shift) & 255u);
              }
              const unsigned peers = __match_any_sync(0xffffffffu, bin);
              if (bin >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
            }
          }
          __syncthreads();
          if (shift == 24) {  // the group's demand: everything fits?
            if (threadIdx.x < 32) {
              unsigned t8 = 0u;
              for (int q = 0; q < 8; ++q) t8 += hist[8 * lane + q];
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) t8 += __shfl_xor_sync(0xffffffffu, t8, o);
              if (lane == 0) s_fits = t8 <= static_cast<unsigned>(cap);
            }
            __syncthreads();
            all_kept = s_fits != 0;
            __syncthreads();
            if (all_kept) break;
          }
          if (threadIdx.x < 32) radix_pick(hist, need, &s_bin, &s_need);
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(s_bin) << shift;
        pmask |= 255u << shift;
        need = s_need;
        __syncthreads();
      }
    }
    const uint32_t thr = prefix;
    // ties: of the group's candidates equal to thr, the first `need` in
    // (token, slot) order stay; the others are marked by a zero key
    if (cap > 0 && !all_kept) {
      bool scan_table = !clustered;
      if (clustered) {
        // ordered compaction of this CTA's equal entries (list positions)
        int32_t* ties = reinterpret_cast<int32_t*>(lkey + T);
        const unsigned lt = (1u << lane) - 1u;
        int n_eq = 0;
        for (int base = 0; base < n; base += kSelPass) {
          const int w0 = base + (static_cast<int>(threadIdx.x) >> 5) * (32 * kSelRounds) + lane;
          bool eq[kSelRounds];
          int cnt = 0;
#pragma unroll
          for (int j = 0; j < kSelRounds; ++j) {
            const int i = w0 + 32 * j;
            eq[j] = i < n && lkey[i] == thr;
            cnt += __popc(__ballot_sync(0xffffffffu, eq[j]));
          }
          int tot;
          int run = n_eq + warp_exclusive_offset(cnt, warp_sums, tot);
#pragma unroll
          for (int j = 0; j < kSelRounds; ++j) {
            const unsigned b = __ballot_sync(0xffffffffu, eq[j]);
            const int q = run + __popc(b & lt);
            if (eq[j] && q < kTieMax) ties[q] = w0 + 32 * j;
            run += __popc(b);
          }
          n_eq += tot;
        }
        if (threadIdx.x == 0) s_count = n_eq;
        __syncthreads();
        cluster_sync();
        if (threadIdx.x == 0) {
          int over = 0;
          for (int r = 0; r < group_size; ++r)
            over |= static_cast<int>(ld_cluster_u32(map_to_rank(smem_u32(&s_count), r))) > kTieMax;
          s_over = over;
        }
        __syncthreads();
        scan_table = s_over != 0;
        if (!scan_table) {
          const uint32_t me = cluster_rank();
          for (int q = threadIdx.x; q < n_eq; q += blockDim.x) {
            const int pos = ties[q];
            const int f = lflat[pos];
            int rank = q;  // equal entries of this CTA before it
            for (int r = 0; r < group_size; ++r) {
              if (r == static_cast<int>(me)) continue;
              const int n_r = static_cast<int>(ld_cluster_u32(map_to_rank(smem_u32(&s_count), r)));
              int a = 0, b = n_r;  // entries of CTA r with flat index below f
              while (a < b) {
                const int mid = (a + b) >> 1;
                const uint32_t pr = ld_cluster_u32(map_to_rank(smem_u32(&ties[mid]), r));
                const int fr = static_cast<int>(
                    ld_cluster_u32(map_to_rank(smem_u32(&lflat[pr]), r)));
                if (fr < f) a = mid + 1;
                else b = mid;
              }
              rank += a;
            }
            if (rank >= need) lkey[pos] = 0u;  // below every gate's key
          }
        }
        // the peers have finished reading this CTA's lists
        __syncthreads();
        cluster_sync();
      }
      if (scan_table) {
        // the need-th candidate equal to thr in table order is the last one kept
        if (threadIdx.x == 0) s_bound = -1;
        __syncthreads();
        const unsigned lt = (1u << lane) - 1u;
        int before = 0;
        for (int base = 0; base < total; base += kSelPass) {
          const int w0 = base + (static_cast<int>(threadIdx.x) >> 5) * (32 * kSelRounds) + lane;
          bool eq[kSelRounds];
          int cnt = 0;
#pragma unroll
          for (int j = 0; j < kSelRounds; ++j) {
            const int i = w0 + 32 * j;
            const int c = i < total ? cand_idx[i] : -1;
            const float g = i < total ? cand_gate[i] : 0.f;
            eq[j] = c >= lo && c < hi && order_key(g) == thr;
            cnt += __popc(__ballot_sync(0xffffffffu, eq[j]));
          }
          int tot;
          int run = before + warp_exclusive_offset(cnt, warp_sums, tot);
#pragma unroll
          for (int j = 0; j < kSelRounds; ++j) {
            const unsigned b = __ballot_sync(0xffffffffu, eq[j]);
            if (eq[j] && run + __popc(b & lt) + 1 == need) s_bound = w0 + 32 * j;
            run += __popc(b);
          }
          before += tot;
          if (before >= need) break;  // uniform: every thread holds the same count
        }
        __syncthreads();
        const int bound = s_bound;
        for (int i = threadIdx.x; i < n; i += blockDim.x)
          if (lkey[i] == thr && lflat[i] > bound) lkey[i] = 0u;
        __syncthreads();
      }
    }
    // ordered keep pass over the own list; slot = kept candidates before it
    const unsigned lt = (1u << lane) - 1u;
    int k_base = 0;
    for (int base = 0; base < n; base += kSelPass) {
      const int w0 = base + (static_cast<int>(threadIdx.x) >> 5) * (32 * kSelRounds) + lane;
      bool kp[kSelRounds];
      int cnt = 0;
#pragma unroll
      for (int j = 0; j < kSelRounds; ++j) {
        const int i = w0 + 32 * j;
        bool v = false;
        if (i < n && cap > 0) {
          const uint32_t kk = lkey[i];
          v = all_kept || kk >= thr;
        }
        kp[j] = v;
        cnt += __popc(__ballot_sync(0xffffffffu, v));
      }
      int tot;
      int run = k_base + warp_exclusive_offset(cnt, warp_sums, tot);
#pragma unroll
      for (int j = 0; j < kSelRounds; ++j) {
        const int i = w0 + 32 * j;
        const unsigned b = __ballot_sync(0xffffffffu, kp[j]);
        if (i < n) {
          slot[lflat[i]] = kp[j] ? run + __popc(b & lt) : -1;
          if (keep) keep[lflat[i]] = kp[j] ? 1 : 0;
        }
        run += __popc(b);
      }
      k_base += tot;
    }
    k_e = k_base;
  } else if (n <= cap) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      slot[lflat[i]] = i;
      if (keep) keep[lflat[i]] = 1;
    }
  } else {
    // 2. radix select of the cap-th largest key (cap >= 1 here; cap <= 0 keeps
    //    none); histogram counts are aggregated per warp over equal bins, since
    //    gates of one expert share their high bits
    uint32_t prefix = 0u, pmask = 0u;
    int need = cap;
    if (cap > 0) {
      // Two barriers per pass: pass p fills histogram p % 3 and clears (p+1)
      // % 3 for the next pass (last read by the pick of pass p - 2, before
      // the barriers of pass p - 1); warp 0 finds the bin and hands it over
      // at the second barrier (read by every warp before the next pass's
      // first barrier, after which warp 0 writes it again).
      for (int b = threadIdx.x; b < 256; b += blockDim.x) hist3[b] = 0u;
      __syncthreads();
      int pass = 0;
      for (int shift = 24; shift >= 0; shift -= 8, ++pass) {
        unsigned* h = hist3 + 256 * (pass % 3);
        unsigned* h_next = hist3 + 256 * ((pass + 1) % 3);
        for (int b = threadIdx.x; b < 256; b += blockDim.x) h_next[b] = 0u;
        for (int i0 = 0; i0 < n; i0 += blockDim.x) {  // uniform trip count per warp
          const int i = i0 + static_cast<int>(threadIdx.x);
          int bin = -1;
          if (i < n) {
            const uint32_t kk = lkey[i];
            if ((kk & pmask) == prefix) bin = static_cast<int>((kk >> shift) & 255u);
          }
          if (pass == 0) {
            // the top byte is shared by most gates of one expert: one
            // atomic per distinct bin of the warp
            const unsigned peers = __match_any_sync(0xffffffffu, bin);
            if (bin >= 0 && lane == __ffs(peers) - 1) atomicAdd(&h[bin], __popc(peers));
          } else if (bin >= 0) {  // lower bytes spread over the bins
            atomicAdd(&h[bin], 1u);
          }
        }
        __syncthreads();
        if (threadIdx.x < 32) {
          int bin, left;
          radix_pick_warp(h, need, bin, left);
          if (lane == 0) {
            s_bin = bin;
            s_need = left;
          }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(s_bin) << shift;
        pmask |= 255u << shift;
        need = s_need;
      }
    }
    const uint32_t thr = prefix;
    const int need_eq = (cap > 0) ? need : 0;  // candidates equal to thr that stay

    // 3. ordered keep pass: a candidate is kept if its key is above thr, or
    //    equal to it and among the first need_eq such in token order; its slot
    //    is the number of kept candidates before it. One scan carries both
    //    counts (above in the high half, equal in the low half; each < 2^16).
    const unsigned lt = (1u << lane) - 1u;
    int k_base = 0, eq_base = 0;  // kept and equal-to-thr entries before this pass
    for (int base = 0; base < n; base += kSelPass) {
      const int w0 = base + (static_cast<int>(threadIdx.x) >> 5) * (32 * kSelRounds) + lane;
      uint32_t kk[kSelRounds];
      int gt_w = 0, eq_w = 0;
#pragma unroll
      for (int j = 0; j < kSelRounds; ++j) {
        const int i = w0 + 32 * j;
        kk[j] = (i < n) ? lkey[i] : 0u;
        const bool valid = i < n && cap > 0;
        gt_w += __popc(__ballot_sync(0xffffffffu, valid && kk[j] > thr));
        eq_w += __popc(__ballot_sync(0xffffffffu, valid && kk[j] == thr));
      }
      // one scan carries both warp counts (above in the high half, equal in
      // the low half; each < 2^16)
      int tot;
      const int ex =
          warp_exclusive_offset2((gt_w << 16) | eq_w, warp_sums2 + 32 * (scan_use++ & 1), tot);
      int gt_before = (ex >> 16), eq_before = eq_base + (ex & 0xffff);
      // kept before an entry = above-thr before it + min(equal before it, need_eq)
#pragma unroll
      for (int j = 0; j < kSelRounds; ++j) {
        const int i = w0 + 32 * j;
        const bool valid = i < n && cap > 0;
        const bool is_gt = valid && kk[j] > thr;
        const bool is_eq = valid && kk[j] == thr;
        const unsigned bg = __ballot_sync(0xffffffffu, is_gt);
        const unsigned be = __ballot_sync(0xffffffffu, is_eq);
        const int g_i = gt_before + __popc(bg & lt);
        const int q_i = eq_before + __popc(be & lt);
        if (i < n) {
          const bool kp = is_gt || (is_eq && q_i < need_eq);
          slot[lflat[i]] = kp ? k_base + g_i + min(q_i, need_eq) - min(eq_base, need_eq) : -1;
          if (keep) keep[lflat[i]] = kp ? 1 : 0;
        }
        gt_before += __popc(bg);
        eq_before += __popc(be);
      }
      k_base += (tot >> 16) + min(eq_base + (tot & 0xffff), need_eq) - min(eq_base, need_eq);
      eq_base += tot & 0xffff;
    }
  }
  if (threadIdx.x == 0) {
    // expert choice drops nothing: an expert's demand is the c tokens it takes
    demand[e] = expert_choice ? k_e : n_all;
    kept[e] = k_e;
  }
}

}  // namespace

int select_max_tokens() { return kSelMaxTokens; }

namespace {

constexpr size_t kSelSmemMax = static_cast<size_t>(kSelMaxTokens) * 8 + kTieMax * 4;

// Whether a device group of `gs` selection CTAs can run as one cluster.
bool group_cluster_ok(int dev, int gs) {
  static int cached[64][kMaxClusterGroup + 1] = {};  // 0 unknown, 1 yes, 2 no
  if (dev < 0 || dev >= 64 || gs < 1 || gs > kMaxClusterGroup) return false;
  if (cached[dev][gs] == 0) {
    bool ok = true;
    if (gs > 8)
      ok = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
           cudaSuccess;
    int n = 0;
    if (ok) {
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(gs);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(gs));
      cfg.blockDim = dim3(kSelThreads);
      cfg.dynamicSmemBytes = kSelSmemMax;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      ok = cudaOccupancyMaxActiveClusters(&n, select_kernel, &cfg) == cudaSuccess && n >= 1;
    }
    if (!ok) (void)cudaGetLastError();
    cached[dev][gs] = ok ? 1 : 2;
  }
  return cached[dev][gs] == 1;
}

}  // namespace

cudaError_t launch_select(const int32_t* cand_idx, const float* cand_gate, int T, int kc, int N,
                          int expert_choice, int cap, int group_size, int32_t* slot, uint8_t* keep,
                          int32_t* demand, int32_t* kept, cudaStream_t s) {
  static bool attr_set[64] = {};  // per device; setting it twice is harmless
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    err = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSelSmemMax));
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  const int clustered = group_size > 0 && group_cluster_ok(dev, group_size) ? 1 : 0;
  const size_t smem = static_cast<size_t>(T) * 8 + (clustered ? kTieMax * 4 : 0);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = clustered ? static_cast<unsigned>(group_size) : 1u;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(N));
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = clustered ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, select_kernel, cand_idx, cand_gate, T, kc, N, expert_choice, cap,
                            group_size, clustered, slot, keep, demand, kept);
}

}  // namespace moe
