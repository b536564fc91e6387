// Router on the fp32 FMA pipes (fp32 layers, or bf16 shapes the tensor-core
// router does not take): logits, then softmax scores, top-k / expanded
// candidates and gates.
//
// "Understanding Mixture of Experts", section "Expert and Router": the router
// scores each token against every expert and activates TopK(G(x), k).
// "Capacity-Aware Inference: Mitigating the Straggler Effect in MoE", section
// 2 (2) Expanded Drop: m extra candidates from the experts of the token's own
// device.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "route_token.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------------------
// Logits: a CTA computes 64 tokens x NE experts, streaming x and W_r through
// shared memory in k-chunks of 32 (converted to fp32), fp32 FMA accumulate.
// Thread (tt, eg): token tt = tid % 64, experts eg + 4j.
// ---------------------------------------------------------------------------
constexpr int kLogitTM = 64;
constexpr int kLogitKC = 32;

template <typename E> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* v) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};
template <> struct Vec8<float> {
  static __device__ __forceinline__ void load(const float* p, float* v) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

template <typename E, int NE>
__global__ void __launch_bounds__(256) router_logits_kernel(const E* __restrict__ x,
                                                            const E* __restrict__ W_r,
                                                            const float* __restrict__ bias,
                                                            float* __restrict__ L, int T, int d,
                                                            int N) {
  constexpr int PER = NE / 4;
  __shared__ float xs[kLogitKC][kLogitTM + 1];
  __shared__ float ws[kLogitKC][NE];
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kLogitTM;
  const int e0 = blockIdx.y * NE;
  const int tt = tid % kLogitTM;
  const int eg = tid / kLogitTM;
  float acc[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) acc[j] = 0.f;

  for (int k0 = 0; k0 < d; k0 += kLogitKC) {
    {  // x chunk: 64 rows x 32 cols, 8 per thread
      const int row = tid / 4, seg = tid % 4;
      float v[8];
      const int t = t0 + row, kk = k0 + seg * 8;
      if (t < T && kk < d) {
        Vec8<E>::load(x + static_cast<size_t>(t) * d + kk, v);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[seg * 8 + i][row] = v[i];
    }
    for (int i = tid; i < kLogitKC * NE; i += 256) {  // W_r chunk
      const int kk = i / NE, e = i % NE;
      const int gk = k0 + kk, ge = e0 + e;
      ws[kk][e] = (gk < d && ge < N) ? to_f32(W_r[static_cast<size_t>(gk) * N + ge]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kLogitKC; ++kk) {
      const float a = xs[kk][tt];
#pragma unroll
      for (int j = 0; j < PER; ++j) acc[j] = fmaf(a, ws[kk][eg + 4 * j], acc[j]);
    }
    __syncthreads();
  }
  const int t = t0 + tt;
  if (t < T) {
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = e0 + eg + 4 * j;
      if (e < N) L[static_cast<size_t>(t) * N + e] = acc[j] + (bias ? bias[e] : 0.f);
    }
  }
}

template <typename E>
cudaError_t logits_dispatch_ne(const E* x, const E* W_r, const float* bias, float* L, int T, int d,
                               int N, cudaStream_t s) {
  const dim3 block(256);
  const int gx = (T + kLogitTM - 1) / kLogitTM;
  if (N <= 8) return launch_pdl(router_logits_kernel<E, 8>, dim3(gx, 1), block, 0, s, x, W_r, bias, L, T, d, N);
  if (N <= 16) return launch_pdl(router_logits_kernel<E, 16>, dim3(gx, 1), block, 0, s, x, W_r, bias, L, T, d, N);
  if (N <= 32) return launch_pdl(router_logits_kernel<E, 32>, dim3(gx, 1), block, 0, s, x, W_r, bias, L, T, d, N);
  return launch_pdl(router_logits_kernel<E, 64>, dim3(gx, (N + 63) / 64), block, 0, s, x, W_r, bias,
                    L, T, d, N);
}

// ---------------------------------------------------------------------------
// Per-token routing from fp32 logits [T, N] (route_token.cuh): 8 warps per
// block, each warp routing 32 / W tokens at once (one W-lane segment each);
// the block writes one row of column sums of p.
// ---------------------------------------------------------------------------
constexpr int kRouteWarpsPerBlock = 8;

template <int W, int PER>
__global__ void __launch_bounds__(kRouteWarpsPerBlock * 32) route_tokens_kernel(const RouteArgs a) {
  constexpr int kTokensPerBlock = kRouteWarpsPerBlock * (32 / W);
  // p of the block's tokens for the column sums: kTokensPerBlock * W * PER <= 2048
  __shared__ float s_p[kTokensPerBlock * W * PER];
  pdl_launch_dependents();
  pdl_wait();
  const int N = a.N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ls = lane % W;
  const int slot = warp * (32 / W) + lane / W;
  const int t = blockIdx.x * kTokensPerBlock + slot;
  const bool valid = t < a.T;
  float l[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = ls * PER + j;  // a lane's experts are contiguous
    l[j] = (valid && e < N) ? a.logits[static_cast<size_t>(t) * N + e] : 0.f;
  }
  route_token_seg<W, PER>(a, t, valid, l, a.colsum ? s_p + slot * N : nullptr);
  if (a.colsum) {
    __syncthreads();
    const int rows = max(0, min(kTokensPerBlock, a.T - static_cast<int>(blockIdx.x) * kTokensPerBlock));
    colsum_rows(s_p, rows, N, a.colsum + static_cast<size_t>(blockIdx.x) * N);
  }
}

template <int W, int PER>
cudaError_t route_launch(const RouteArgs& a, cudaStream_t s) {
  constexpr int kTokensPerBlock = kRouteWarpsPerBlock * (32 / W);
  return launch_pdl(route_tokens_kernel<W, PER>, (a.T + kTokensPerBlock - 1) / kTokensPerBlock,
                    kRouteWarpsPerBlock * 32, 0, s, a);
}

}  // namespace

cudaError_t launch_router_logits(int dtype, const void* x, const void* W_r, const float* bias,
                                 float* L, int T, int d, int N, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (dtype == 1)
    return logits_dispatch_ne(static_cast<const __nv_bfloat16*>(x),
                              static_cast<const __nv_bfloat16*>(W_r), bias, L, T, d, N, s);
  return logits_dispatch_ne(static_cast<const float*>(x), static_cast<const float*>(W_r), bias, L,
                            T, d, N, s);
}

int route_tokens_colsum_rows(int T, int N) {
  const int per_block = kRouteWarpsPerBlock * (32 / route_seg_width(N));
  return (T + per_block - 1) / per_block;
}

cudaError_t launch_route_tokens(const RouteArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  // (W, PER) = (route_seg_width(N), route_seg_per(N))
  if (a.N <= 8) return route_launch<8, 1>(a, s);
  if (a.N <= 16) return route_launch<8, 2>(a, s);
  if (a.N <= 32) return route_launch<8, 4>(a, s);
  if (a.N <= 64) return route_launch<8, 8>(a, s);
  if (a.N <= 128) return route_launch<16, 8>(a, s);
  if (a.N <= 256) return route_launch<32, 8>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
