// fp32 grouped expert GEMM on the FMA pipes, for fp32 layers whose 1e-5
// tolerance rules out the tensor cores' reduced-precision formats.
//
// Segment s covers rows [offsets[s], offsets[s+1]) of A and uses weight
// matrix B[s] ([K, n_out], row-major). A CTA computes a 64 x 64 output tile
// with a 4 x 4 block per thread, staging 16-wide k-chunks of A and B in shared
// memory. CTA x-index -> (segment, m-tile) through the running count of
// m-tiles per segment, so segment sizes stay on the device.
// SwiGLU variant: out = silu(A B1) * (A B3) with two accumulator sets.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kTM = 64, kTN = 64, kTK = 16;

template <bool SWIGLU>
__global__ void __launch_bounds__(256) grouped_gemm_f32_kernel(
    const float* __restrict__ A, const int32_t* __restrict__ offsets, int S, int K, int n_out,
    int rows_max, const float* __restrict__ B1, const float* __restrict__ B3,
    float* __restrict__ out) {
  __shared__ int s_seg, s_r0, s_r1;
  __shared__ float As[kTK][kTM + 4];
  __shared__ float B1s[kTK][kTN];
  __shared__ float B3s[SWIGLU ? kTK : 1][SWIGLU ? kTN : 1];
  pdl_launch_dependents();
  pdl_wait();
  if (threadIdx.x == 0) {
    int tile = blockIdx.x, acc = 0;
    s_seg = -1;
    for (int s = 0; s < S; ++s) {
      const int a = offsets[s], b = offsets[s + 1];
      const int nt = (b - a + kTM - 1) / kTM;
      if (tile < acc + nt) {
        s_seg = s;
        s_r0 = a + (tile - acc) * kTM;
        s_r1 = b < rows_max ? b : rows_max;
        break;
      }
      acc += nt;
    }
  }
  __syncthreads();
  if (s_seg < 0 || s_r0 < 0) return;
  const int seg = s_seg, r0 = s_r0, r1 = s_r1;
  const int n0 = blockIdx.y * kTN;
  const float* B1e = B1 + static_cast<size_t>(seg) * K * n_out;
  const float* B3e = SWIGLU ? B3 + static_cast<size_t>(seg) * K * n_out : nullptr;
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  float acc1[4][4] = {}, acc3[4][4] = {};

  for (int k0 = 0; k0 < K; k0 += kTK) {
    {  // A chunk: 64 rows x 16 k, 4 per thread
      const int row = tid / 4, kk = (tid % 4) * 4;
      const int r = r0 + row;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = k0 + kk + i;
        As[kk + i][row] = (r < r1 && k < K) ? A[static_cast<size_t>(r) * K + k] : 0.f;
      }
    }
    {  // B chunk: 16 k x 64 n, 4 per thread
      const int kk = tid / 16, nn = (tid % 16) * 4;
      const int k = k0 + kk;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = n0 + nn + i;
        const bool ok = k < K && n < n_out;
        B1s[kk][nn + i] = ok ? B1e[static_cast<size_t>(k) * n_out + n] : 0.f;
        if (SWIGLU) B3s[kk][nn + i] = ok ? B3e[static_cast<size_t>(k) * n_out + n] : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      float a[4], b1[4], b3[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b1[j] = B1s[kk][tx * 4 + j];
        if (SWIGLU) b3[j] = B3s[kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc1[i][j] = fmaf(a[i], b1[j], acc1[i][j]);
          if (SWIGLU) acc3[i][j] = fmaf(a[i], b3[j], acc3[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + ty * 4 + i;
    if (r >= r1) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= n_out) continue;
      out[static_cast<size_t>(r) * n_out + n] =
          SWIGLU ? silu_accurate(acc1[i][j]) * acc3[i][j] : acc1[i][j];
    }
  }
}

}  // namespace

cudaError_t launch_grouped_gemm_simt_f32(const float* A, const int32_t* offsets, int S,
                                         int64_t rows_max, int K, int n_out, const float* B1,
                                         const float* B3, float* out, bool swiglu,
                                         cudaStream_t s) {
  if (S == 0 || rows_max == 0) return cudaSuccess;
  const long long mt = (rows_max + kTM - 1) / kTM + S;  // upper bound of m-tiles
  const int rmax = rows_max > 0x7fffffff ? 0x7fffffff : static_cast<int>(rows_max);
  const dim3 grid(static_cast<unsigned>(mt), (n_out + kTN - 1) / kTN);
  if (swiglu)
    return launch_pdl(grouped_gemm_f32_kernel<true>, grid, 256, 0, s, A, offsets, S, K, n_out,
                      rmax, B1, B3, out);
  return launch_pdl(grouped_gemm_f32_kernel<false>, grid, 256, 0, s, A, offsets, S, K, n_out,
                    rmax, B1, static_cast<const float*>(nullptr), out);
}

}  // namespace moe
