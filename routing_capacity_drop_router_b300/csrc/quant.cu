// Activation rows to e4m3 with one fp32 scale per row, the operand format of
// the FP8 expert GEMMs.
//
// Quantising the expert weights lightens the weight side of a bandwidth-bound
// step ("From personas to MoE 02", section "dense was honestly heavy"); the
// tensor cores multiply e4m3 only by e4m3, so the rows that meet the weights
// (the dispatched token rows, the SwiGLU hidden rows) are quantised too:
//   scale[r] = max_j |X[r][j]| / 448   (fp32, correctly rounded; 1 for a zero row)
//   Q[r][j]  = e4m3 nearest to X[r][j] / scale[r]
//              (the quotient correctly rounded to fp32, then rounded to the
//               nearest e4m3 value, ties to even, finite overflow saturated)
// so X[r][j] ~ value(Q[r][j]) * scale[r]. Both roundings are fixed IEEE
// operations, so the codes are a fixed function of the bf16 inputs.
//
// One block per row (grid-stride over the rows); the row is read twice (the
// maximum, a block reduction, then the codes; the second read hits L2), so a
// few long rows (a decode batch's hidden rows) still spread over many SMs.
// Only rows below offsets[S] (the kept rows, read on the device) are written.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kQThreads = 256;
constexpr int kQWarps = kQThreads / 32;
constexpr float kE4m3Max = 448.0f;

__global__ void __launch_bounds__(kQThreads) quantize_rows_e4m3_kernel(
    const __nv_bfloat16* __restrict__ X, const int32_t* __restrict__ offsets, int S, int rows_max,
    int K, uint8_t* __restrict__ Q, float* __restrict__ scale) {
  __shared__ float s_max[kQWarps];
  pdl_launch_dependents();
  pdl_wait();
  const int P = min(max(offsets[S], 0), rows_max);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = K / 8;  // 16-byte vectors of 8 bf16
  for (int r = blockIdx.x; r < P; r += gridDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(X + static_cast<size_t>(r) * K);
    float amax = 0.f;
    for (int c = threadIdx.x; c < nvec; c += kQThreads) {
      const uint4 q = __ldg(src + c);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) s_max[warp] = amax;
    __syncthreads();
    amax = s_max[0];
#pragma unroll
    for (int w = 1; w < kQWarps; ++w) amax = fmaxf(amax, s_max[w]);
    const float sc = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.0f;
    uint2* dst = reinterpret_cast<uint2*>(Q + static_cast<size_t>(r) * K);
    for (int c = threadIdx.x; c < nvec; c += kQThreads) {
      const uint4 q = __ldg(src + c);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
      uint32_t w[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float2 f0 = __bfloat1622float2(h[2 * i]);
        const float2 f1 = __bfloat1622float2(h[2 * i + 1]);
        const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(f0.x, sc), __fdiv_rn(f0.y, sc)), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(f1.x, sc), __fdiv_rn(f1.y, sc)), __NV_SATFINITE, __NV_E4M3);
        w[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      }
      dst[c] = make_uint2(w[0], w[1]);
    }
    if (threadIdx.x == 0) scale[r] = sc;
    __syncthreads();  // s_max is reused by the next row
  }
}

}  // namespace

cudaError_t launch_quantize_rows_e4m3(const void* X, const int32_t* offsets, int S,
                                      int64_t rows_max, int K, uint8_t* Q, float* scale,
                                      cudaStream_t s) {
  if (S == 0 || rows_max == 0) return cudaSuccess;
  if (K <= 0 || K % 8) return cudaErrorInvalidValue;
  const int rmax = rows_max > 0x7fffffff ? 0x7fffffff : static_cast<int>(rows_max);
  const long long cap = device_sm_count() * 8;
  const int blocks = static_cast<int>(rows_max < cap ? rows_max : cap);
  return launch_pdl(quantize_rows_e4m3_kernel, blocks, kQThreads, 0, s,
                    static_cast<const __nv_bfloat16*>(X), offsets, S, rmax, K, Q, scale);
}

}  // namespace moe
