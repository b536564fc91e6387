// Load statistics of a routed batch: the Switch balance term
// B = sum_i f_i * P_i ("MoE vs MoT: routing and inference cost", section "MoE
// basic structure"), the straggler ratio max/mean kept load ("Capacity-Aware
// Inference: Mitigating the Straggler Effect in MoE", section 1) and the
// dropped fraction. Column sums of the scores are taken in fp64 in a fixed
// order (per-CTA partials, then the partials in CTA order).
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kStatTokens = 256;  // tokens per partial-sum CTA

__global__ void __launch_bounds__(256) stats_partial_kernel(const float* __restrict__ scores, int T,
                                                            int N, double* __restrict__ partial) {
  __shared__ double red[256];
  const int nsub = 256 / N;  // N <= 256
  const int e = threadIdx.x % N, sub = threadIdx.x / N;
  const int t0 = blockIdx.x * kStatTokens;
  const int t1 = min(T, t0 + kStatTokens);
  double s = 0.0;
  if (sub < nsub)
    for (int t = t0 + sub; t < t1; t += nsub) s += static_cast<double>(scores[static_cast<size_t>(t) * N + e]);
  red[threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.x < N) {
    double acc = 0.0;
    for (int q = 0; q < nsub; ++q) acc += red[q * N + threadIdx.x];
    partial[static_cast<size_t>(blockIdx.x) * N + threadIdx.x] = acc;
  }
}

__global__ void __launch_bounds__(256) stats_final_kernel(const int32_t* __restrict__ demand,
                                                          const int32_t* __restrict__ kept,
                                                          const double* __restrict__ partial,
                                                          int nblocks, int T, int N,
                                                          double* __restrict__ stats) {
  __shared__ double psum[256];
  __shared__ double s_kept[256], s_dem[256];
  if (threadIdx.x < N) {
    // partials in block order; four independent loads in flight
    const int e = threadIdx.x;
    double acc = 0.0;
    int b = 0;
    for (; b + 4 <= nblocks; b += 4) {
      const double v0 = partial[static_cast<size_t>(b) * N + e];
      const double v1 = partial[static_cast<size_t>(b + 1) * N + e];
      const double v2 = partial[static_cast<size_t>(b + 2) * N + e];
      const double v3 = partial[static_cast<size_t>(b + 3) * N + e];
      acc += v0;
      acc += v1;
      acc += v2;
      acc += v3;
    }
    for (; b < nblocks; ++b) acc += partial[static_cast<size_t>(b) * N + e];
    psum[e] = acc;
    s_kept[e] = static_cast<double>(kept[e]);
    s_dem[e] = static_cast<double>(demand[e]);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double P = 0, D = 0, mx = 0;
    for (int e = 0; e < N; ++e) {
      P += s_kept[e];
      D += s_dem[e];
      mx = fmax(mx, s_kept[e]);
    }
    double B = 0;
    if (D > 0 && T > 0)
      for (int e = 0; e < N; ++e) B += (s_dem[e] / D) * (psum[e] / T);
    const double mean = P / N;
    stats[0] = P;
    stats[1] = D;
    stats[2] = mx;
    stats[3] = mean;
    stats[4] = mean > 0 ? mx / mean : 0.0;
    stats[5] = D > 0 ? 1.0 - P / D : 0.0;
    stats[6] = B;
    stats[7] = N * B;
  }
}

}  // namespace

size_t stats_partial_doubles(int T, int N) {
  const size_t nb = (static_cast<size_t>(T) + kStatTokens - 1) / kStatTokens;
  return (nb > 0 ? nb : 1) * static_cast<size_t>(N);
}

cudaError_t launch_stats(const int32_t* demand, const int32_t* kept, const float* scores, int T,
                         int N, double* partial, double* stats, cudaStream_t s) {
  const int nb = (T + kStatTokens - 1) / kStatTokens;
  if (nb > 0) stats_partial_kernel<<<nb, 256, 0, s>>>(scores, T, N, partial);
  stats_final_kernel<<<1, 256, 0, s>>>(demand, kept, partial, nb, T, N, stats);
  return cudaGetLastError();
}

}  // namespace moe
