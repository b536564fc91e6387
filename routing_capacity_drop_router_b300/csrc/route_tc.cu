// Router logits on the tcgen05 tensor cores (bf16 in, fp32 accumulate), with
// the per-token routing in the same launch.
//
// "Understanding Mixture of Experts", section "Expert and Router": the router
// scores every token against every expert, L = x W_r (+ b). The read of x
// bounds this step, so the design goal is an even spread of that read: the
// m_tiles * (d / 64) k-blocks (128 tokens x 64 of d each), tile-major, are cut
// into one contiguous range per CTA (2 CTAs per SM for N <= 64), so every CTA
// streams the same number of k-blocks through its 4-stage TMA ring whatever
// T and d are. A range covers at most two tiles; for each tile one thread
// issues 128 x (64*NB) x 16 MMAs into its own TMEM accumulator, and the
// accumulator is written as one fp32 segment partial[tile][slot] (slot = the
// CTA's rank among the tile's CTAs, i.e. k order). Each CTA then counts
// itself in the tile's arrival counter; the last to arrive adds the tile's
// segments in slot order plus the bias and routes its 128 tokens
// (route_token.cuh), so the logits and every decision are deterministic and
// the routing needs no second launch. W_r [d, N] is read as stored
// (MN-major, N contiguous) in 64-expert TMA boxes; experts past N load as
// zeros.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "route_token.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kRM = 128;        // tokens per tile (MMA M)
constexpr int kRK = 64;         // k per stage
constexpr int kRStages = 4;
constexpr int kRThreads = 128;  // 4 warps: producer, MMA, then all four drain TMEM
static_assert(kRM == kRouteTile && kRThreads == kRouteTile, "one routing thread per tile row");
constexpr int kRABytes = kRM * kRK * 2;
constexpr int kRBoxBytes = 64 * kRK * 2;
constexpr unsigned long long kRWaitNs = 1000000000ull;
constexpr int kErrDeviceTimeout = -7;  // MOE_ERR_DEVICE_TIMEOUT

struct __align__(8) RouterCtrl {
  unsigned long long full[kRStages];
  unsigned long long empty[kRStages];
  unsigned long long acc_full[2];
  unsigned long long drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <int NB>
constexpr int router_smem_bytes() {
  return 1024 + kRStages * (kRABytes + NB * kRBoxBytes) + static_cast<int>(sizeof(RouterCtrl));
}
// the routing tail reuses the stage buffers for its [128, N + 1] staging array
static_assert(route_tile_smem(64) <= kRStages * (kRABytes + 1 * kRBoxBytes), "stage reuse");
static_assert(route_tile_smem(128) <= kRStages * (kRABytes + 2 * kRBoxBytes), "stage reuse");
static_assert(route_tile_smem(256) <= kRStages * (kRABytes + 4 * kRBoxBytes), "stage reuse");

template <int NB>
__global__ void __launch_bounds__(kRThreads) router_tc_kernel(
    const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
    const RouteArgs ra, uint32_t* __restrict__ tile_counters, int32_t* __restrict__ status) {
  constexpr int kStageBytes = kRABytes + NB * kRBoxBytes;
  constexpr uint32_t kCols = 64u * NB;  // accumulator columns of one segment
  constexpr uint32_t kAlloc = 2u * kCols;
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
  const int T = ra.T, N = ra.N;
  const int G = static_cast<int>(gridDim.x), num_kb = ra.seg_kb;
  const long long W = ra.seg_total;

  // ---- this CTA's k-blocks, cut at the tile boundary into <= 2 segments ----
  const long long q0 = static_cast<long long>(blockIdx.x) * W / G;
  const long long q1 = static_cast<long long>(blockIdx.x + 1) * W / G;
  int nseg = 0, seg_tile[2] = {0, 0}, seg_kb0[2] = {0, 0}, seg_kb1[2] = {0, 0}, seg_slot[2] = {0, 0};
  for (long long q = q0; q < q1 && nseg < 2;) {
    const int m = static_cast<int>(q / num_kb);
    const long long tile_end = static_cast<long long>(m + 1) * num_kb;
    const long long e = q1 < tile_end ? q1 : tile_end;
    seg_tile[nseg] = m;
    seg_kb0[nseg] = static_cast<int>(q - static_cast<long long>(m) * num_kb);
    seg_kb1[nseg] = static_cast<int>(e - static_cast<long long>(m) * num_kb);
    seg_slot[nseg] = static_cast<int>(blockIdx.x) -
                     router_cta_of(static_cast<long long>(m) * num_kb, G, W);
    ++nseg;
    q = e;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), 1);
    }
    mbar_init(smem_u32(&ctrl->acc_full[0]), 1);
    mbar_init(smem_u32(&ctrl->acc_full[1]), 1);
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
  // set-up above overlaps the previous kernel; nothing global is touched before this
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 0 && lane == 0) {
    // ---- TMA producer ----
    int stage = 0;
    uint32_t phase = 0;
    bool issued[kRStages] = {};
    uint32_t issued_phase[kRStages] = {};
    bool ok = true;
    for (int sg = 0; ok && sg < nseg; ++sg) {
      for (int kb = seg_kb0[sg]; kb < seg_kb1[sg]; ++kb) {
        if (!mbar_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort_flag, kRWaitNs)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&ctrl->full[stage]);
        mbar_expect_tx(fb, kStageBytes);
        const uint32_t sa = base + stage * kStageBytes;
        tma_load_2d(sa, &tmX, kb * kRK, seg_tile[sg] * kRM, fb);
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
    // ---- MMA issuer: segment sg accumulates in TMEM columns [sg*kCols, ...) ----
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int sg = 0; ok && sg < nseg; ++sg) {
      const uint32_t d_tmem = tmem + static_cast<uint32_t>(sg) * kCols;
      for (int kb = seg_kb0[sg]; kb < seg_kb1[sg]; ++kb) {
        if (!mbar_wait(smem_u32(&ctrl->full[stage]), phase, abort_flag, kRWaitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = base + stage * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < kRK / 16; ++kk)
          tc_mma(d_tmem, kmajor_desc(sa, kk), mnmajor_desc(sa + kRABytes, kk, kRBoxBytes), kIdesc,
                 (kb > seg_kb0[sg] || kk > 0) ? 1u : 0u);
        tc_commit(smem_u32(&ctrl->empty[stage]));
        if (++stage == kRStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) tc_commit(smem_u32(&ctrl->acc_full[sg]));
    }
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

  // ---- drain: TMEM lane = token row of the tile; row r -> partial row r ----
  for (int sg = 0; sg < nseg; ++sg) {
    int ok = 1;
    if (lane == 0) ok = mbar_wait(smem_u32(&ctrl->acc_full[sg]), 0u, abort_flag, kRWaitNs);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    tc_fence_after();
    const int r = warp * 32 + lane;
    float* dst = const_cast<float*>(ra.partial) +
                 ((static_cast<size_t>(seg_tile[sg]) * ra.max_slots + seg_slot[sg]) * kRM + r) * N;
    const uint32_t taddr =
        tmem + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(sg) * kCols;
    for (int c = 0; c < N; c += 16) {
      uint32_t v[16];
      tc_ld16(taddr + c, v);
      tc_wait_ld();
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

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0 && *abort_flag) record_status(status, kErrDeviceTimeout);
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kAlloc)
                 : "memory");
  }

  // ---- arrival: the last CTA of each tile routes its tokens ----
  // Every CTA arrives (even after an expired wait), so each counter is back at
  // zero at the end of every launch.
  __shared__ int s_last[2];
  __threadfence();  // this CTA's segments are visible before it arrives
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int sg = 0; sg < nseg; ++sg) {
      const int m = seg_tile[sg];
      const uint32_t need = static_cast<uint32_t>(router_tile_segments(m, num_kb, G, W));
      const uint32_t old = atomicAdd(&tile_counters[m], 1u);
      s_last[sg] = old == need - 1;
      if (s_last[sg]) tile_counters[m] = 0u;
    }
  }
  __syncthreads();
  for (int sg = 0; sg < nseg; ++sg) {
    if (s_last[sg]) {
      __threadfence();
      // the stage buffers (last written by TMA, read by the tensor cores) are
      // reused as generic shared memory
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      route_tile(ra, seg_tile[sg], reinterpret_cast<float*>(smem));
      __syncthreads();
    }
  }
  (void)T;
}

template <int NB>
cudaError_t launch_nb(const CUtensorMap& mX, const CUtensorMap& mW, int ctas,
                      const RouteArgs& ra, uint32_t* tile_counters, int32_t* status,
                      cudaStream_t s) {
  constexpr int smem = router_smem_bytes<NB>();
  static bool attr_set[64] = {};  // per device; setting it twice is harmless
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    err = cudaFuncSetAttribute(router_tc_kernel<NB>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  return launch_pdl(router_tc_kernel<NB>, ctas, kRThreads, smem, s, mX, mW, ra, tile_counters,
                    status);
}

}  // namespace

bool router_tc_supported(int dtype, int d, int N) {
  return dtype == 1 && d % 64 == 0 && N % 8 == 0 && N <= 256;
}

RouterSplit router_split_plan(int T, int d, int N) {
  RouterSplit p;
  const int m_tiles = (T + kRM - 1) / kRM;
  p.num_kb = d / kRK;
  p.total = static_cast<long long>(m_tiles) * p.num_kb;
  const int nb = (N + 63) / 64;
  const int per_sm = nb == 1 ? 2 : 1;  // CTAs whose shared memory fits on one SM
  long long g = static_cast<long long>(device_sm_count()) * per_sm;
  if (g < m_tiles) g = m_tiles;  // keeps every range within num_kb k-blocks (<= 2 tiles)
  if (g > p.total) g = p.total;
  if (g < 1) g = 1;
  p.ctas = static_cast<int>(g);
  p.max_slots = 1;
  for (int m = 0; m < m_tiles; ++m) {
    const int n = router_tile_segments(m, p.num_kb, p.ctas, p.total);
    if (n > p.max_slots) p.max_slots = n;
  }
  return p;
}

cudaError_t launch_router_tc(const void* x, const void* W_r, int d, const RouterSplit& plan,
                             const RouteArgs& ra, uint32_t* tile_counters, int32_t* status,
                             cudaStream_t s) {
  const int T = ra.T, N = ra.N;
  if (T == 0) return cudaSuccess;
  if ((T + kRM - 1) / kRM > kMaxRouterTiles) return cudaErrorInvalidValue;
  if (ra.seg_ctas != plan.ctas || ra.seg_kb != plan.num_kb || ra.seg_total != plan.total ||
      ra.max_slots != plan.max_slots)
    return cudaErrorInvalidValue;
  CUtensorMap mX, mW;
  if (!make_tmap_2d_bf16(&mX, x, static_cast<uint64_t>(T), static_cast<uint64_t>(d), 64, kRM))
    return cudaErrorInvalidValue;
  if (!make_tmap_2d_bf16(&mW, W_r, static_cast<uint64_t>(d), static_cast<uint64_t>(N), 64, kRK))
    return cudaErrorInvalidValue;
  const int g = plan.ctas;
  if (N <= 64) return launch_nb<1>(mX, mW, g, ra, tile_counters, status, s);
  if (N <= 128) return launch_nb<2>(mX, mW, g, ra, tile_counters, status, s);
  if (N <= 256) return launch_nb<4>(mX, mW, g, ra, tile_counters, status, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
