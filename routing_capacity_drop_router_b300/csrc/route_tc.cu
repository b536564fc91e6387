// Router logits on the tcgen05 tensor cores (bf16 in, fp32 accumulate).
//
// "Understanding Mixture of Experts", section "Expert and Router": the router
// scores every token against every expert, L = x W_r (+ b). The read of x
// bounds this step, so the design goal is enough bytes in flight: the d axis
// is split over `splits` CTAs per 128-token tile (split-K), each CTA streams
// its k-slice of x through a 4-stage TMA ring, and one thread issues
// 128 x (64*NB) x 16 MMAs into TMEM. W_r [d, N] is read as stored (MN-major,
// N contiguous) in 64-expert TMA boxes; experts past N load as zeros.
// Each split writes its fp32 partial logits partial[split][t][0..N); the
// per-token routing kernel adds the splits in ascending order plus the bias,
// so the result is deterministic.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kRM = 128;        // tokens per tile (MMA M)
constexpr int kRK = 64;         // k per stage
constexpr int kRStages = 4;
constexpr int kRThreads = 128;  // 4 warps: producer, MMA, then all four drain TMEM
constexpr int kRABytes = kRM * kRK * 2;
constexpr int kRBoxBytes = 64 * kRK * 2;
constexpr unsigned long long kRWaitNs = 1000000000ull;
constexpr int kErrDeviceTimeout = -7;  // MOE_ERR_DEVICE_TIMEOUT

struct __align__(8) RouterCtrl {
  unsigned long long full[kRStages];
  unsigned long long empty[kRStages];
  unsigned long long acc_full;
  unsigned long long drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <int NB>
constexpr int router_smem_bytes() {
  return 1024 + kRStages * (kRABytes + NB * kRBoxBytes) + static_cast<int>(sizeof(RouterCtrl));
}

template <int NB>
__global__ void __launch_bounds__(kRThreads) router_logits_tc_kernel(
    const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, int T,
    int N, int num_kb, int kb_per_split, float* __restrict__ partial,
    int32_t* __restrict__ status) {
  constexpr int kStageBytes = kRABytes + NB * kRBoxBytes;
  constexpr uint32_t kCols = 64u * NB;
  constexpr uint32_t kAlloc = NB == 1 ? 64u : (NB == 2 ? 128u : 256u);
  // kind::f16 instruction descriptor: D fp32, A/B bf16, A K-major, B MN-major,
  // N = 64*NB, M = 128.
  constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                              ((kCols >> 3) << 17) | (static_cast<uint32_t>(kRM >> 4) << 24);
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw);
  RouterCtrl* ctrl = reinterpret_cast<RouterCtrl*>(smem + kRStages * kStageBytes);
  volatile int* abort_flag = &ctrl->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x, split = blockIdx.y;
  const int kb0 = split * kb_per_split;
  const int kb1 = min(num_kb, kb0 + kb_per_split);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), 1);
    }
    mbar_init(smem_u32(&ctrl->acc_full), 1);
    mbar_init(smem_u32(&ctrl->drain), 1);
    ctrl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctrl->tmem_base)),
                 "r"(kAlloc)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer ----
    int stage = 0;
    uint32_t phase = 0;
    bool issued[kRStages] = {};
    uint32_t issued_phase[kRStages] = {};
    bool ok = true;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort_flag, kRWaitNs)) {
        ok = false;
        break;
      }
      const uint32_t fb = smem_u32(&ctrl->full[stage]);
      mbar_expect_tx(fb, kStageBytes);
      const uint32_t sa = base + stage * kStageBytes;
      tma_load_2d(sa, &tmX, kb * kRK, m_tile * kRM, fb);
#pragma unroll
      for (int j = 0; j < NB; ++j)
        tma_load_2d(sa + kRABytes + j * kRBoxBytes, &tmW, 64 * j, kb * kRK, fb);
      issued[stage] = true;
      issued_phase[stage] = phase;
      if (++stage == kRStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {  // drain copies in flight before the CTA can exit (bounded)
      for (int s = 0; s < kRStages; ++s) {
        if (!issued[s]) continue;
        const unsigned long long t0 = global_ns();
        while (!mbar_try(smem_u32(&ctrl->full[s]), issued_phase[s]))
          if (global_ns() - t0 > kRWaitNs / 10) break;
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(smem_u32(&ctrl->full[stage]), phase, abort_flag, kRWaitNs)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sa = base + stage * kStageBytes;
#pragma unroll
      for (int kk = 0; kk < kRK / 16; ++kk)
        tc_mma(tmem, kmajor_desc(sa, kk), mnmajor_desc(sa + kRABytes, kk, kRBoxBytes), kIdesc,
               (kb > kb0 || kk > 0) ? 1u : 0u);
      tc_commit(smem_u32(&ctrl->empty[stage]));
      if (++stage == kRStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (ok) tc_commit(smem_u32(&ctrl->acc_full));
    // every MMA issued so far completes before this arrives
    tc_commit(smem_u32(&ctrl->drain));
    const unsigned long long t0 = global_ns();
    while (!mbar_try(smem_u32(&ctrl->drain), 0u))
      if (global_ns() - t0 > kRWaitNs) {
        *abort_flag = 1;
        break;
      }
  }
  __syncwarp();

  // ---- drain: TMEM lane = token row of this tile ----
  int ok = 1;
  if (lane == 0) ok = mbar_wait(smem_u32(&ctrl->acc_full), 0u, abort_flag, kRWaitNs);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) {
    tc_fence_after();
    const int t = m_tile * kRM + warp * 32 + lane;
    float* dst = partial + (static_cast<size_t>(split) * T + t) * N;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int c = 0; c < N; c += 16) {
      uint32_t v[16];
      tc_ld16(taddr + c, v);
      tc_wait_ld();
      if (t < T) {
        if (c + 16 <= N) {  // N % 8 == 0, so dst + c is 16-byte aligned
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(dst + c + i) =
                make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                            __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c + i < N) dst[c + i] = __uint_as_float(v[i]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0 && *abort_flag) record_status(status, kErrDeviceTimeout);
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kAlloc)
                 : "memory");
  }
}

template <int NB>
cudaError_t launch_nb(const CUtensorMap& mX, const CUtensorMap& mW, int T, int N, int num_kb,
                      int kb_per_split, int splits, float* partial, int32_t* status,
                      cudaStream_t s) {
  constexpr int smem = router_smem_bytes<NB>();
  static bool attr_set[64] = {};  // per device; setting it twice is harmless
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    err = cudaFuncSetAttribute(router_logits_tc_kernel<NB>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  const dim3 grid((T + kRM - 1) / kRM, splits);
  router_logits_tc_kernel<NB><<<grid, kRThreads, smem, s>>>(mX, mW, T, N, num_kb, kb_per_split,
                                                            partial, status);
  return cudaGetLastError();
}

}  // namespace

bool router_tc_supported(int dtype, int d, int N) {
  return dtype == 1 && d % 64 == 0 && N % 8 == 0 && N <= 256;
}

RouterSplit router_split_plan(int T, int d, int N) {
  RouterSplit p;
  const int m_tiles = (T + kRM - 1) / kRM;
  const int num_kb = d / kRK;
  const int nb = (N + 63) / 64;
  const int per_sm = nb == 1 ? 2 : 1;  // CTAs whose shared memory fits on one SM
  const int target = device_sm_count() * per_sm;
  int splits = m_tiles > 0 ? target / m_tiles : 1;  // at most one wave
  if (splits > num_kb) splits = num_kb;
  if (splits < 1) splits = 1;
  p.kb_per_split = (num_kb + splits - 1) / splits;
  p.splits = (num_kb + p.kb_per_split - 1) / p.kb_per_split;
  return p;
}

cudaError_t launch_router_logits_tc(const void* x, const void* W_r, int T, int d, int N,
                                    const RouterSplit& plan, float* partial, int32_t* status,
                                    cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  CUtensorMap mX, mW;
  if (!make_tmap_2d_bf16(&mX, x, static_cast<uint64_t>(T), static_cast<uint64_t>(d), 64, kRM))
    return cudaErrorInvalidValue;
  if (!make_tmap_2d_bf16(&mW, W_r, static_cast<uint64_t>(d), static_cast<uint64_t>(N), 64, kRK))
    return cudaErrorInvalidValue;
  const int num_kb = d / kRK;
  const int kbp = plan.kb_per_split, sp = plan.splits;
  switch ((N + 63) / 64) {
    case 1: return launch_nb<1>(mX, mW, T, N, num_kb, kbp, sp, partial, status, s);
    case 2: return launch_nb<2>(mX, mW, T, N, num_kb, kbp, sp, partial, status, s);
    case 3: return launch_nb<3>(mX, mW, T, N, num_kb, kbp, sp, partial, status, s);
    case 4: return launch_nb<4>(mX, mW, T, N, num_kb, kbp, sp, partial, status, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
