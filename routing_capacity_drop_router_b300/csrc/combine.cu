// Gate-weighted combine, the sum of the layer equation
// y = sum_i G(x)_i E_i(x) ("Understanding Mixture of Experts", section "How
// MoE differs from the Transformer").
//
// One warp per token; the token's rows (ascending expert) and gates are staged
// in shared memory, the shared expert's row last with gate 1 (fma(1, v, acc)
// rounds v + acc once, as an add would), then each lane walks 16-byte column
// vectors (two per pass, the loads of RB rows issued before their FMAs: 2 for
// top-2 tokens, 4 when a token may have more rows): for every row an FMA into
// fp32 accumulators in a fixed order (ascending expert, shared expert last),
// one rounding to the output dtype at the end.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kCombThreads = 256;
constexpr int kCombWarps = kCombThreads / 32;
constexpr int kCombMaxRows = 257;  // up to 256 routed rows, then the shared expert's
constexpr int kShared = -2;        // row marker: the shared expert's output row
constexpr int kU = 2;   // 16-byte column vectors per lane per pass
// few registers, so that 32+ warps per SM keep enough 16-byte loads in flight
constexpr int kCombMinBlocks = 4;

template <typename E> struct Pack;  // 16 bytes of E <-> fp32
template <> struct Pack<__nv_bfloat16> {
  static constexpr int n = 8;
  static __device__ __forceinline__ void unpack(const uint4& q, float* v) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
  static __device__ __forceinline__ uint4 pack(const float* v) {
    uint4 q;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    return q;
  }
};
template <> struct Pack<float> {
  static constexpr int n = 4;
  static __device__ __forceinline__ void unpack(const uint4& q, float* v) {
    v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y);
    v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
  }
  static __device__ __forceinline__ uint4 pack(const float* v) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                      __float_as_uint(v[3]));
  }
};

template <typename E, int kRB>
__global__ void __launch_bounds__(kCombThreads, kRB > 2 ? kCombMinBlocks - 1 : kCombMinBlocks)
    combine_kernel(
    const E* __restrict__ op, const float* __restrict__ row_gate,
    const int32_t* __restrict__ tok_rows, const E* __restrict__ shared_out, E* __restrict__ y,
    int T, int d, int kc, int rows_max) {
  constexpr int V = Pack<E>::n;
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int s_row[kCombWarps][kCombMaxRows];
  __shared__ float s_gate[kCombWarps][kCombMaxRows];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int nvec = d / V;
  const int warps_total = kCombWarps * gridDim.x;
  for (int t = blockIdx.x * kCombWarps + wib; t < T; t += warps_total) {
    int nrows = 0;
    for (int base = 0; base < kc; base += 32) {
      const int j = base + lane;
      const int r = (j < kc) ? tok_rows[static_cast<size_t>(t) * kc + j] : -1;
      const bool ok = r >= 0 && r < rows_max;
      const unsigned b = __ballot_sync(0xffffffffu, ok);
      if (ok) {  // kept in list order (ascending rows)
        const int pos = nrows + __popc(b & ((1u << lane) - 1u));
        s_row[wib][pos] = r;
        s_gate[wib][pos] = row_gate[r];
      }
      nrows += __popc(b);
    }
    if (shared_out) {  // the shared expert's row, last, gate 1
      if (lane == 0) {
        s_row[wib][nrows] = kShared;
        s_gate[wib][nrows] = 1.0f;
      }
      ++nrows;
    }
    __syncwarp();
    const E* sh = shared_out ? shared_out + static_cast<size_t>(t) * d : nullptr;
    uint4* dst = reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * d);
    // kU column vectors per lane and up to kRB rows loaded before their FMAs,
    // so each lane keeps kU * kRB 16-byte loads in flight
    for (int c0 = lane; c0 < nvec; c0 += 32 * kU) {
      float acc[kU][V];
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int i = 0; i < V; ++i) acc[u][i] = 0.f;
      for (int r0 = 0; r0 < nrows; r0 += kRB) {
        uint4 q[kRB][kU];
#pragma unroll
        for (int rr = 0; rr < kRB; ++rr) {
          if (r0 + rr < nrows) {
            const int row = s_row[wib][r0 + rr];
            const uint4* src = reinterpret_cast<const uint4*>(
                row == kShared ? sh : op + static_cast<size_t>(row) * d);
#pragma unroll
            for (int u = 0; u < kU; ++u)
              if (c0 + 32 * u < nvec) q[rr][u] = __ldg(src + c0 + 32 * u);
          }
        }
#pragma unroll
        for (int rr = 0; rr < kRB; ++rr) {
          if (r0 + rr < nrows) {
            const float g = s_gate[wib][r0 + rr];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              if (c0 + 32 * u < nvec) {
                float v[V];
                Pack<E>::unpack(q[rr][u], v);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[u][i] = fmaf(g, v[i], acc[u][i]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + 32 * u;
        if (c < nvec) dst[c] = Pack<E>::pack(acc[u]);
      }
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_combine(int dtype, const void* op, const float* row_gate,
                           const int32_t* tok_rows, const void* shared_out, void* y, int T,
                           int d, int kc, int64_t rows_max, cudaStream_t s) {
  const int rmax = rows_max > 0x7fffffff ? 0x7fffffff : static_cast<int>(rows_max);
  if (T == 0) return cudaSuccess;
  int blocks = (T + kCombWarps - 1) / kCombWarps;
  const int cap = device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  // rows loaded per batch: a top-2 token's rows in one batch; more rows
  // (top-k > 2, expanded candidates, expert choice, a shared expert) in 4s
  const bool wide = kc + (shared_out ? 1 : 0) > 2;
  if (dtype == 1) {
    auto k = wide ? combine_kernel<__nv_bfloat16, 4> : combine_kernel<__nv_bfloat16, 2>;
    return launch_pdl(k, blocks, kCombThreads, 0, s, static_cast<const __nv_bfloat16*>(op),
                      row_gate, tok_rows, static_cast<const __nv_bfloat16*>(shared_out),
                      static_cast<__nv_bfloat16*>(y), T, d, kc, rmax);
  } else {
    auto k = wide ? combine_kernel<float, 4> : combine_kernel<float, 2>;
    return launch_pdl(k, blocks, kCombThreads, 0, s, static_cast<const float*>(op), row_gate,
                      tok_rows, static_cast<const float*>(shared_out), static_cast<float*>(y), T,
                      d, kc, rmax);
  }
  return cudaGetLastError();
}

}  // namespace moe
