// Device helpers shared by the layer's kernels.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace moe {

// ---- element types --------------------------------------------------------
struct bf16_t { using T = __nv_bfloat16; };
struct f32_t { using T = float; };

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename E> __device__ __forceinline__ E from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// ---- router score exponential ---------------------------------------------
// exp(x) for x <= 0 by Cody-Waite range reduction (Cody & Waite, "Software
// Manual for the Elementary Functions", 1980) and the degree-7 Taylor
// polynomial of exp on |r| <= ln2/2. Every step is an explicitly rounded fp32
// operation (no contraction), so the result is a fixed function of x:
//   n = rint(x * log2e); r = (x - n*ln2_hi) - n*ln2_lo;
//   q = ((((((c7 r + c6) r + c5) r + c4) r + c3) r + c2) r + c1) r + c0;
//   exp(x) ~ q * 2^n, flushed to 0 when n < -125.
// ln2_hi is ln 2 truncated to 16 significant bits (45426 / 2^16), so n*ln2_hi
// is exact for |n| < 2^8 and x - n*ln2_hi is exact; ln2_lo is the fp32 rounding
// of ln 2 - ln2_hi; c_i the fp32 rounding of 1/i!.
__device__ __forceinline__ float score_exp(float x) {
  constexpr double kLn2 = 0.693147180559945309417232121458;
  constexpr float kLog2e = static_cast<float>(1.0 / kLn2);
  constexpr float kLn2Hi = 45426.0f / 65536.0f;
  constexpr float kLn2Lo = static_cast<float>(kLn2 - 45426.0 / 65536.0);
  constexpr float c0 = 1.0f, c1 = 1.0f, c2 = 0.5f;
  constexpr float c3 = static_cast<float>(1.0 / 6.0);
  constexpr float c4 = static_cast<float>(1.0 / 24.0);
  constexpr float c5 = static_cast<float>(1.0 / 120.0);
  constexpr float c6 = static_cast<float>(1.0 / 720.0);
  constexpr float c7 = static_cast<float>(1.0 / 5040.0);
  const float n = rintf(__fmul_rn(x, kLog2e));
  if (!(n >= -125.0f)) return 0.0f;
  float r = __fsub_rn(x, __fmul_rn(n, kLn2Hi));
  r = __fsub_rn(r, __fmul_rn(n, kLn2Lo));
  float q = c7;
  q = __fadd_rn(__fmul_rn(q, r), c6);
  q = __fadd_rn(__fmul_rn(q, r), c5);
  q = __fadd_rn(__fmul_rn(q, r), c4);
  q = __fadd_rn(__fmul_rn(q, r), c3);
  q = __fadd_rn(__fmul_rn(q, r), c2);
  q = __fadd_rn(__fmul_rn(q, r), c1);
  q = __fadd_rn(__fmul_rn(q, r), c0);
  const float scale = __int_as_float((static_cast<int>(n) + 127) << 23);  // 2^n, normal
  return __fmul_rn(q, scale);
}

// ---- ordering key ---------------------------------------------------------
// Unsigned key that orders finite fp32 values like the values, -0 == +0.
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---- programmatic dependent launch ----------------------------------------
// pdl_wait: block until the previous kernel on the stream has completed and
// its writes are visible (a no-op when the launch was not programmatic).
// pdl_launch_dependents: allow the next kernel to be scheduled now; it still
// waits in its own pdl_wait before reading anything this kernel writes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- sticky status --------------------------------------------------------
__device__ __forceinline__ void record_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// silu(z) = z / (1 + e^-z): the fast exponential for bf16 outputs, the
// accurate one where the result is stored in fp32.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }
__device__ __forceinline__ float silu_accurate(float z) { return z / (1.0f + expf(-z)); }

}  // namespace moe
