// Final step of the load statistics (see stats.cu), run by one block of at
// least 256 threads (the dispatch kernel's extra block in the layer, the
// statistics kernel for moe_load_stats); reads demand, kept and the column
// sums through L2 (__ldcg), as earlier kernels of the stream wrote them.
// Everything up to the last few divisions is integer arithmetic: this part's
// fp64 pipe is narrow, and one thread does the handful of fp64 operations.
#pragma once
#include <cstdint>

#include "internal.h"

namespace moe {

__device__ __forceinline__ double u128_to_double(unsigned long long hi, unsigned long long lo) {
  return fma(static_cast<double>(hi), 18446744073709551616.0, static_cast<double>(lo));
}

__device__ __forceinline__ void stats_final_block(const int32_t* demand, const int32_t* kept,
                                                  const unsigned long long* colsum, int rows,
                                                  int T, int N, double* stats) {
  // per expert: exact column sum (u64: thread (e, c) adds rows c, c + chunks,
  // ...; integer sums, so the order does not matter) and demand_i * colsum_i
  // as 128 bits
  __shared__ unsigned long long s_sum[256], s_hi[256], s_lo[256];
  __shared__ long long s_P[256], s_D[256], s_mx[256];
  for (int e = threadIdx.x; e < 256; e += blockDim.x) s_sum[e] = 0ull;
  __syncthreads();
  const int chunks = static_cast<int>(blockDim.x) / N;  // >= 1: N <= 256 <= blockDim.x
  if (static_cast<int>(threadIdx.x) < chunks * N) {
    const int e = static_cast<int>(threadIdx.x) % N, c = static_cast<int>(threadIdx.x) / N;
    unsigned long long acc = 0ull;
    int b = c;
    for (; b + 3 * chunks < rows; b += 4 * chunks) {  // four loads in flight
      const unsigned long long v0 = __ldcg(colsum + static_cast<size_t>(b) * N + e);
      const unsigned long long v1 = __ldcg(colsum + static_cast<size_t>(b + chunks) * N + e);
      const unsigned long long v2 = __ldcg(colsum + static_cast<size_t>(b + 2 * chunks) * N + e);
      const unsigned long long v3 = __ldcg(colsum + static_cast<size_t>(b + 3 * chunks) * N + e);
      acc += v0 + v1 + v2 + v3;
    }
    for (; b < rows; b += chunks) acc += __ldcg(colsum + static_cast<size_t>(b) * N + e);
    atomicAdd(&s_sum[e], acc);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 256; e += blockDim.x) {
    unsigned long long hi = 0ull, lo = 0ull;
    long long kp = 0, dm = 0;
    if (e < N) {
      const unsigned long long acc = s_sum[e];
      kp = __ldcg(kept + e);
      dm = __ldcg(demand + e);
      const unsigned long long d = static_cast<unsigned long long>(dm);
      lo = acc * d;
      hi = __umul64hi(acc, d);
    }
    s_hi[e] = hi;
    s_lo[e] = lo;
    s_P[e] = kp;
    s_D[e] = dm;
    s_mx[e] = kp;
  }
  __syncthreads();
  if (threadIdx.x < 32) {  // one warp folds the 256 entries, 8 per lane, then a tree
    const int l = threadIdx.x;
    unsigned long long hi = 0ull, lo = 0ull;
    long long P = 0, D = 0, mx = 0;
    for (int q = 0; q < 8; ++q) {
      const int e = l * 8 + q;
      const unsigned long long nlo = lo + s_lo[e];
      hi += s_hi[e] + (nlo < lo ? 1ull : 0ull);
      lo = nlo;
      P += s_P[e];
      D += s_D[e];
      mx = s_mx[e] > mx ? s_mx[e] : mx;
    }
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long ohi = __shfl_down_sync(0xffffffffu, hi, o);
      const unsigned long long olo = __shfl_down_sync(0xffffffffu, lo, o);
      const long long oP = __shfl_down_sync(0xffffffffu, P, o);
      const long long oD = __shfl_down_sync(0xffffffffu, D, o);
      const long long omx = __shfl_down_sync(0xffffffffu, mx, o);
      const unsigned long long nlo = lo + olo;
      hi += ohi + (nlo < lo ? 1ull : 0ull);
      lo = nlo;
      P += oP;
      D += oD;
      mx = omx > mx ? omx : mx;
    }
    if (l == 0) {
      const double Pd = static_cast<double>(P), Dd = static_cast<double>(D);
      const double mean = Pd / N;
      // B = sum_i (demand_i / D) * (colsum_i * 2^-40 / T)
      const double B = (D > 0 && T > 0)
                           ? u128_to_double(hi, lo) / (Dd * static_cast<double>(T)) * 0x1p-40
                           : 0.0;
      stats[0] = Pd;
      stats[1] = Dd;
      stats[2] = static_cast<double>(mx);
      stats[3] = mean;
      stats[4] = P > 0 ? static_cast<double>(mx) * N / Pd : 0.0;
      stats[5] = D > 0 ? static_cast<double>(D - P) / Dd : 0.0;
      stats[6] = B;
      stats[7] = N * B;
    }
  }
}

}  // namespace moe
