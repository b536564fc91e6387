// Load statistics of a routed batch: the Switch balance term
// B = sum_i f_i * P_i ("MoE vs MoT: routing and inference cost", section "MoE
// basic structure"), the straggler ratio max/mean kept load ("Capacity-Aware
// Inference: Mitigating the Straggler Effect in MoE", section 1) and the
// dropped fraction.
//
// P_i = mean_t p[t, i] comes from per-tile column sums of the scores held in
// fixed point (units of 2^-40, u64), which the routing kernels write as they
// compute p; integer sums are exact, so the result does not depend on the
// order of the additions. B itself is formed as one exact integer,
// sum_i demand_i * colsum_i, divided once in fp64. Inside the layer the final
// step (stats_final.cuh) runs in an extra block of the dispatch kernel; the
// kernels here serve moe_load_stats.
#include <cuda_runtime.h>

#include "internal.h"
#include "route_token.cuh"
#include "stats_final.cuh"

namespace moe {
namespace {

constexpr int kColsumTokens = 32;  // tokens per row of colsum_kernel

// Column sums of [T, N] fp32 scores, one block per 32-token row.
__global__ void __launch_bounds__(256) colsum_kernel(const float* __restrict__ scores, int T,
                                                     int N, unsigned long long* __restrict__ colsum) {
  pdl_launch_dependents();
  pdl_wait();
  const int tile = blockIdx.x;
  const int t0 = tile * kColsumTokens, t1 = min(T, t0 + kColsumTokens);
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    unsigned long long acc = 0ull;
    for (int t = t0; t < t1; ++t)
      acc += fixed40(scores[static_cast<size_t>(t) * N + e]);
    colsum[static_cast<size_t>(tile) * N + e] = acc;
  }
}

__global__ void __launch_bounds__(256) stats_final_kernel(const int32_t* __restrict__ demand,
                                                          const int32_t* __restrict__ kept,
                                                          const unsigned long long* __restrict__ colsum,
                                                          int rows, int T, int N,
                                                          double* __restrict__ stats) {
  pdl_launch_dependents();
  pdl_wait();
  stats_final_block(demand, kept, colsum, rows, T, N, stats);
}

}  // namespace

size_t colsum_bytes(int T, int N) {
  // the routing kernel writes at most ceil(T / 8) rows, the tensor-core
  // router at most ceil(T / 128) * 8, colsum_kernel ceil(T / 32)
  const size_t rows = (static_cast<size_t>(T) + 7) / 8 + 8;
  return rows * static_cast<size_t>(N) * sizeof(unsigned long long);
}

int colsum_kernel_rows(int T) { return (T + kColsumTokens - 1) / kColsumTokens; }

cudaError_t launch_colsum(const float* scores, int T, int N, unsigned long long* colsum,
                          cudaStream_t s) {
  const int rows = colsum_kernel_rows(T);
  if (rows > 0) return launch_pdl(colsum_kernel, rows, 256, 0, s, scores, T, N, colsum);
  return cudaSuccess;
}

cudaError_t launch_stats_final(const int32_t* demand, const int32_t* kept,
                               const unsigned long long* colsum, int rows, int T, int N,
                               double* stats, cudaStream_t s) {
  return launch_pdl(stats_final_kernel, 1, 256, 0, s, demand, kept, colsum, rows, T, N, stats);
}

}  // namespace moe
