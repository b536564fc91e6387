// Dispatch: histogram -> prefix sum -> permute of the kept (token, expert)
// pairs into expert-contiguous rows, and the gather of the token rows.
//
// "MoE vs MoT: routing and inference cost", section "MoE basic structure":
// each MoE layer sends tokens to their experts (dispatch) and brings the
// results back (gather); within one GPU the dispatch is this permutation.
//
// Each CTA recomputes expert_offsets = exclusive scan of kept[0..N) in shared
// memory (N <= 256), then one warp per token:
//   row(t, j) = offsets[e] + slot[t, j] for every kept slot j;
//   tok_rows[t] = those rows sorted ascending (= ascending expert);
//   coverage[t] = how many rows token t has (the experts that took it);
//   x[t] is read once, 16 bytes per lane, and written to each of its rows
//   (skipped when xp is null: the expert GEMM then gathers the rows itself
//   through row_token).
// With load statistics requested, one extra block (after the token blocks)
// computes them from the selection's demand/kept and the router's column
// sums while the others copy rows.
#include <climits>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "stats_final.cuh"

namespace moe {
namespace {

constexpr int kDispThreads = 256;
constexpr int kDispWarps = kDispThreads / 32;
constexpr int kMaxRowsPerToken = 256;  // kc <= 32 for token slots, N <= 256 for expert choice

__device__ __forceinline__ void scan_offsets(const int32_t* __restrict__ kept, int N, int* s_off) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int v[8], sum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = lane * 8 + q;
      v[q] = (e < N) ? max(kept[e], 0) : 0;
      sum += v[q];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int run = incl - sum;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      s_off[lane * 8 + q] = run;
      run += v[q];
    }
    if (lane == 31) s_off[256] = incl;
  }
  __syncthreads();
}

template <typename E>
__global__ void __launch_bounds__(kDispThreads) dispatch_kernel(
    const E* __restrict__ x, const int32_t* __restrict__ cand_idx,
    const float* __restrict__ cand_gate, const int32_t* __restrict__ slot,
    const int32_t* __restrict__ kept, int T, int d, int N, int kc, int expert_choice,
    int rows_max,
    int32_t* __restrict__ expert_offsets, int32_t* __restrict__ row_token,
    float* __restrict__ row_gate, int32_t* __restrict__ tok_rows,
    int32_t* __restrict__ coverage, E* __restrict__ xp, int token_blocks,
    const int32_t* __restrict__ demand, const StatsArgs st) {
  __shared__ int s_off[257];
  __shared__ int s_rows[kDispWarps][kMaxRowsPerToken];
  pdl_launch_dependents();
  pdl_wait();
  if (static_cast<int>(blockIdx.x) >= token_blocks) {  // the load-statistics block
    stats_final_block(demand, kept, st.colsum, st.rows, T, N, st.stats);
    return;
  }
  scan_offsets(kept, N, s_off);
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= N; e += blockDim.x) expert_offsets[e] = s_off[e];

  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  int* rows = s_rows[wib];
  const int nvec = d * static_cast<int>(sizeof(E)) / 16;  // 16-byte vectors per row
  const int warps_total = kDispWarps * token_blocks;

  for (int t = blockIdx.x * kDispWarps + wib; t < T; t += warps_total) {
    int nrows = 0;
    if (!expert_choice) {
      int row = INT_MAX;
      float g = 0.f;
      if (lane < kc) {
        const size_t o = static_cast<size_t>(t) * kc + lane;
        const int s = slot[o];
        const int e = cand_idx[o];
        if (s >= 0 && e >= 0 && e < N && s_off[e] + s < s_off[e + 1] &&
            s_off[e] + s < rows_max) {
          row = s_off[e] + s;
          g = cand_gate[o];
        }
      }
      const bool valid = row != INT_MAX;
      int rank = 0;
      for (int j = 0; j < kc; ++j) rank += (__shfl_sync(0xffffffffu, row, j) < row);
      nrows = __popc(__ballot_sync(0xffffffffu, valid));
      if (valid) {
        rows[rank] = row;
        row_token[row] = t;
        row_gate[row] = g;
      }
    } else {
      for (int base = 0; base < N; base += 32) {
        const int e = base + lane;
        const size_t o = static_cast<size_t>(t) * N + e;
        const int s = (e < N) ? slot[o] : -1;
        const bool valid = s >= 0 && s_off[e] + s < s_off[e + 1] && s_off[e] + s < rows_max;
        const unsigned b = __ballot_sync(0xffffffffu, valid);
        if (valid) {
          const int row = s_off[e] + s;
          rows[nrows + __popc(b & ((1u << lane) - 1u))] = row;
          row_token[row] = t;
          row_gate[row] = cand_gate[o];
        }
        nrows += __popc(b);
      }
    }
    __syncwarp();
    int32_t* tr = tok_rows + static_cast<size_t>(t) * kc;
    for (int j = lane; j < kc; j += 32) tr[j] = (j < nrows) ? rows[j] : -1;
    if (coverage && lane == 0) coverage[t] = nrows;
    if (nrows == 0 || xp == nullptr) {
      __syncwarp();
      continue;
    }
    // gather: x[t] read once, 4 vectors in flight per lane
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d);
    for (int c0 = 0; c0 < nvec; c0 += 32 * 4) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < nvec) v[u] = __ldg(src + c);
      }
      for (int r = 0; r < nrows; ++r) {
        uint4* dst = reinterpret_cast<uint4*>(xp + static_cast<size_t>(rows[r]) * d);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + u * 32 + lane;
          if (c < nvec) dst[c] = v[u];
        }
      }
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_dispatch(int dtype, const void* x, const int32_t* cand_idx,
                            const float* cand_gate, const int32_t* slot, const int32_t* kept,
                            int T, int d, int N, int kc, int expert_choice, int64_t rows_max,
                            int32_t* expert_offsets, int32_t* row_token, float* row_gate,
                            int32_t* tok_rows, int32_t* coverage, void* xp, const int32_t* demand,
                            const StatsArgs& st, cudaStream_t s) {
  const int rmax = rows_max > 0x7fffffff ? 0x7fffffff : static_cast<int>(rows_max);
  int blocks = (T + kDispWarps - 1) / kDispWarps;
  const int cap = device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;  // still writes expert_offsets when T == 0
  if (st.stats && (!demand || N > 256)) return cudaErrorInvalidValue;
  const int grid = blocks + (st.stats ? 1 : 0);
  static_assert(kDispThreads >= 256, "the statistics block needs 256 threads");
  if (dtype == 1) {
    return launch_pdl(dispatch_kernel<__nv_bfloat16>, grid, kDispThreads, 0, s,
                      static_cast<const __nv_bfloat16*>(x), cand_idx, cand_gate, slot, kept, T, d,
                      N, kc, expert_choice, rmax, expert_offsets, row_token, row_gate, tok_rows,
                      coverage, static_cast<__nv_bfloat16*>(xp), blocks, demand, st);
  }
  return launch_pdl(dispatch_kernel<float>, grid, kDispThreads, 0, s,
                    static_cast<const float*>(x), cand_idx, cand_gate, slot, kept, T, d, N, kc,
                    expert_choice, rmax, expert_offsets, row_token, row_gate, tok_rows,
                    coverage, static_cast<float*>(xp), blocks, demand, st);
}

}  // namespace moe
