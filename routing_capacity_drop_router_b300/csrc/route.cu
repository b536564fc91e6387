// Router: logits, softmax scores, top-k / expanded candidates and gates.
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
  if (N <= 8) {
    router_logits_kernel<E, 8><<<dim3(gx, 1), block, 0, s>>>(x, W_r, bias, L, T, d, N);
  } else if (N <= 16) {
    router_logits_kernel<E, 16><<<dim3(gx, 1), block, 0, s>>>(x, W_r, bias, L, T, d, N);
  } else if (N <= 32) {
    router_logits_kernel<E, 32><<<dim3(gx, 1), block, 0, s>>>(x, W_r, bias, L, T, d, N);
  } else {
    router_logits_kernel<E, 64><<<dim3(gx, (N + 63) / 64), block, 0, s>>>(x, W_r, bias, L, T, d, N);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Per-token routing from fp32 logits, one thread per token, all N logits of
// the token in registers (NMAX >= N).
//   scores: m = max L; u_e = score_exp(L_e - m); Z = u_0 + u_1 + ... (in
//   order); p_e = u_e / Z (correctly rounded).
//   top-k: k passes of an argmax over order keys, strict '>' in ascending e,
//   so ties go to the lower expert; a chosen expert's key is cleared to 0
//   (every finite value has a key >= 0x00800000).
//   expanded: m more passes restricted to the home group's experts.
//   gates: p of the slot; with renorm divided by the slots' left-to-right sum.
// ---------------------------------------------------------------------------
template <int NMAX>
__global__ void __launch_bounds__(64) route_tokens_kernel(
    const float* __restrict__ partial, int nsplit, const float* __restrict__ bias,
    float* __restrict__ logits_out, float* __restrict__ scores, int32_t* __restrict__ cand_idx,
    float* __restrict__ cand_gate, const int32_t* __restrict__ home_group, int T, int N, int k,
    int m, int group_size, int renorm, int expert_choice) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  float l[NMAX];
  {
    const float* row = partial + static_cast<size_t>(t) * N;
#pragma unroll
    for (int e = 0; e < NMAX; ++e) l[e] = (e < N) ? row[e] : 0.f;
    for (int sp = 1; sp < nsplit; ++sp) {  // splits added in ascending order
      row += static_cast<size_t>(T) * N;
#pragma unroll
      for (int e = 0; e < NMAX; ++e)
        if (e < N) l[e] += row[e];
    }
    if (bias) {
#pragma unroll
      for (int e = 0; e < NMAX; ++e)
        if (e < N) l[e] += bias[e];
    }
    if (logits_out) {
#pragma unroll
      for (int e = 0; e < NMAX; ++e)
        if (e < N) logits_out[static_cast<size_t>(t) * N + e] = l[e];
    }
  }
  float mx = l[0];
#pragma unroll
  for (int e = 1; e < NMAX; ++e)
    if (e < N) mx = fmaxf(mx, l[e]);
  float p[NMAX];
  float Z = 0.f;
#pragma unroll
  for (int e = 0; e < NMAX; ++e) {
    p[e] = (e < N) ? score_exp(__fsub_rn(l[e], mx)) : 0.f;
    if (e == 0) Z = p[0];
    else if (e < N) Z = __fadd_rn(Z, p[e]);
  }
#pragma unroll
  for (int e = 0; e < NMAX; ++e) p[e] = __fdiv_rn(p[e], Z);

  if (expert_choice) {
    float* out = cand_gate + static_cast<size_t>(t) * N;
#pragma unroll
    for (int e = 0; e < NMAX; ++e)
      if (e < N) {
        out[e] = p[e];
        if (scores) scores[static_cast<size_t>(t) * N + e] = p[e];
      }
    return;
  }
  if (scores) {
#pragma unroll
    for (int e = 0; e < NMAX; ++e)
      if (e < N) scores[static_cast<size_t>(t) * N + e] = p[e];
  }

  uint32_t key[NMAX];
#pragma unroll
  for (int e = 0; e < NMAX; ++e) key[e] = (e < N) ? order_key(l[e]) : 0u;

  const int kc = k + m;
  int32_t* idx_out = cand_idx + static_cast<size_t>(t) * kc;
  float* gate_out = cand_gate + static_cast<size_t>(t) * kc;
  float g[32];
  for (int j = 0; j < kc; ++j) {
    int lo = 0, hi = N;  // pass range: all experts for top-k, the home group after
    if (j >= k) {
      const int G = N / group_size;
      const int hg = home_group ? home_group[t]
                                : static_cast<int>((static_cast<long long>(t) * G) / T);
      lo = hg * group_size;
      hi = lo + group_size;
    }
    int best = -1;
    uint32_t bk = 0u;
    float bp = 0.f;
#pragma unroll
    for (int e = 0; e < NMAX; ++e) {
      if (e >= lo && e < hi && key[e] > bk) {
        bk = key[e];
        best = e;
        bp = p[e];
      }
    }
#pragma unroll
    for (int e = 0; e < NMAX; ++e)
      if (e == best) key[e] = 0u;
    idx_out[j] = best;
    g[j] = (best >= 0) ? bp : 0.f;
  }
  if (renorm) {
    float S = g[0];
    for (int j = 1; j < kc; ++j) S = __fadd_rn(S, g[j]);
    for (int j = 0; j < kc; ++j) g[j] = __fdiv_rn(g[j], S);
  }
  for (int j = 0; j < kc; ++j) gate_out[j] = g[j];
}

template <int NMAX>
cudaError_t route_tokens_launch(const float* partial, int nsplit, const float* bias,
                                float* logits_out, float* scores, int32_t* cand_idx,
                                float* cand_gate, const int32_t* home_group, int T, int N, int k,
                                int m, int group_size, int renorm, int ec, cudaStream_t s) {
  const int threads = 64;
  route_tokens_kernel<NMAX><<<(T + threads - 1) / threads, threads, 0, s>>>(
      partial, nsplit, bias, logits_out, scores, cand_idx, cand_gate, home_group, T, N, k, m,
      group_size, renorm, ec);
  return cudaGetLastError();
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

cudaError_t launch_route_tokens(const float* partial, int nsplit, const float* bias,
                                float* logits_out, float* scores, int32_t* cand_idx,
                                float* cand_gate, const int32_t* home_group, int T, int N, int k,
                                int m, int group_size, int renorm, int ec, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
#define MOE_ROUTE_CASE(NM)                                                                     \
  if (N <= NM)                                                                                 \
    return route_tokens_launch<NM>(partial, nsplit, bias, logits_out, scores, cand_idx,       \
                                   cand_gate, home_group, T, N, k, m, group_size, renorm, ec, s);
  MOE_ROUTE_CASE(8)
  MOE_ROUTE_CASE(16)
  MOE_ROUTE_CASE(32)
  MOE_ROUTE_CASE(64)
  MOE_ROUTE_CASE(128)
  MOE_ROUTE_CASE(256)
#undef MOE_ROUTE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe
