// Router logits on the tcgen05 tensor cores (bf16 in, fp32 accumulate), and
// the per-token routing in the same launch.
//
// "Understanding Mixture of Experts", section "Expert and Router": the router
// scores every token against every expert, L = x W_r (+ b). The read of x
// bounds this step, so the design goal is an even spread of that read over
// the SMs. Each 128-token tile is one thread-block cluster of C CTAs (C a
// power of two <= 8 chosen so that all clusters are resident at once): CTA r
// of the cluster streams k-blocks [r*d/(64C), (r+1)*d/(64C)) of the tile's x
// rows and of W_r through a 4-stage TMA ring, and one thread issues
// 128 x (64*NB) x 16 MMAs into TMEM. W_r [d, N] is read as stored (MN-major,
// N contiguous) in 64-expert TMA boxes; experts past N load as zeros.
//
// Tail, through distributed shared memory: after a cluster barrier (every
// CTA's MMAs are done, so its stage buffers are free) each CTA writes TMEM
// row i of its partial logits into the stage buffer of the CTA that routes
// token i (CTA i / (128/C)), at the slot of its own rank; after a second
// cluster barrier each CTA adds, for its 128/C tokens, the C partials in rank
// order (= k order) and the bias (all threads, coalesced logit stores), then
// routes them with W-lane warp segments, 256 / W tokens per pass
// (route_token.cuh; 8 lanes of 8 contiguous experts each for N = 64, so the
// ordered softmax sum crosses 8 lanes, not 64). So the logits and every
// decision are deterministic, and no partial goes through global memory.
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
constexpr int kRThreads = 256;  // warps 0-3: producer, MMA, TMEM drain; all 8 route
constexpr int kRDrainThreads = 128;  // one TMEM lane (tile row) per drain thread
static_assert(kRM == kRouteTile && kRDrainThreads == kRM, "one drain thread per tile row");
constexpr int kRABytes = kRM * kRK * 2;
constexpr int kRBoxBytes = 64 * kRK * 2;
constexpr unsigned long long kRWaitNs = 1000000000ull;
constexpr int kErrDeviceTimeout = -7;  // MOE_ERR_DEVICE_TIMEOUT
constexpr int kMaxCluster = 8;

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
// the tail receives 128 rows x N fp32 partials into the stage buffers
static_assert(128 * 64 * 4 <= kRStages * (kRABytes + 1 * kRBoxBytes), "receive buffer");
static_assert(128 * 128 * 4 <= kRStages * (kRABytes + 2 * kRBoxBytes), "receive buffer");
static_assert(128 * 256 * 4 <= kRStages * (kRABytes + 4 * kRBoxBytes), "receive buffer");

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

template <int NB, int W, int PER>
__global__ void __launch_bounds__(kRThreads) router_tc_kernel(
    const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
    const RouteArgs ra, int num_kb, int32_t* __restrict__ status) {
  constexpr int kStageBytes = kRABytes + NB * kRBoxBytes;
  constexpr uint32_t kCols = 64u * NB;  // accumulator columns (>= 64: a valid allocation)
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
  uint32_t nrank;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(nrank));
  const int cl = static_cast<int>(nrank);
  const uint32_t rank = cluster_rank();
  const int tile = static_cast<int>(blockIdx.x) / cl;
  const int kb_per = num_kb / cl;
  const int kb0 = static_cast<int>(rank) * kb_per, kb1 = kb0 + kb_per;
  const int tpc = kRM / cl;  // tokens routed by each CTA of the cluster

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
                 "r"(kCols)
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
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort_flag, kRWaitNs)) {
        ok = false;
        break;
      }
      const uint32_t fb = smem_u32(&ctrl->full[stage]);
      mbar_expect_tx(fb, kStageBytes);
      const uint32_t sa = base + stage * kStageBytes;
      tma_load_2d(sa, &tmX, kb * kRK, tile * kRM, fb);
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
  // one thread waits for the accumulator; the others wait at the block
  // barrier, which takes no issue slots from the producer and the MMA issuer
  __shared__ int s_acc_ok;
  if (warp == 2 && lane == 0)
    s_acc_ok = mbar_wait(smem_u32(&ctrl->acc_full), 0u, abort_flag, kRWaitNs) ? 1 : 0;
  __syncthreads();
  const int acc_ok = s_acc_ok;
  // the stage buffers (written by TMA, read by the tensor cores) are about to
  // receive generic stores from the cluster
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");

  // ---- cluster barrier 1: every CTA's MMAs are done, its stage buffers free ----
  tc_fence_before();
  cluster_sync();
  tc_fence_after();

  // ---- drain: TMEM row r of this CTA's partial -> receive buffer of CTA
  //      r / tpc, slot [rank][r % tpc][0..N) ----
  if (acc_ok && warp < kRDrainThreads / 32) {
    const int r = warp * 32 + lane;
    const uint32_t owner = static_cast<uint32_t>(r / tpc);
    const uint32_t dst_local = base + static_cast<uint32_t>(((rank * tpc) + (r % tpc)) * N * 4);
    const uint32_t dst = map_to_rank(dst_local, owner);
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int c0 = 0; c0 < N; c0 += 64) {  // up to four 16-column loads, then one wait
      uint32_t v[64];
      const int nchunk = min(4, (N - c0 + 15) / 16);  // warp-uniform
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q < nchunk) tc_ld16(taddr + c0 + 16 * q, v + 16 * q);
      tc_wait_ld();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = c0 + 16 * q;
        if (q >= nchunk) break;
        const int nv = (N - c) >= 16 ? 4 : (N - c) / 4;  // N % 8 == 0
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (i < nv)
            st_cluster_v4(dst + (c + 4 * i) * 4, __uint_as_float(v[16 * q + 4 * i]),
                          __uint_as_float(v[16 * q + 4 * i + 1]),
                          __uint_as_float(v[16 * q + 4 * i + 2]),
                          __uint_as_float(v[16 * q + 4 * i + 3]));
      }
    }
  }
  tc_fence_before();
  // ---- cluster barrier 2: every partial has arrived ----
  cluster_sync();
  tc_fence_after();
  if (threadIdx.x == 0 && *abort_flag) record_status(status, kErrDeviceTimeout);
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols)
                 : "memory");
  }

  // ---- routing of this CTA's tokens t0 + i, i < tpc ----
  // (a) every thread: logits = the C partials added in rank order, plus the
  //     bias, stored to global memory and in place into rank 0's slot
  float* recv = reinterpret_cast<float*>(smem);
  const int t0 = tile * kRM + static_cast<int>(rank) * tpc;
  for (int idx = static_cast<int>(threadIdx.x); idx < tpc * N; idx += kRThreads) {
    const int i = idx / N, e = idx - (idx / N) * N;
    float v = recv[idx];
    for (int src = 1; src < cl; ++src) v = __fadd_rn(v, recv[(src * tpc + i) * N + e]);
    if (ra.bias) v = __fadd_rn(v, ra.bias[e]);
    const int t = t0 + i;
    if (ra.logits_out && t < T) ra.logits_out[static_cast<size_t>(t) * N + e] = v;
    recv[idx] = v;
  }
  __syncthreads();
  // (b) one W-lane segment per token, 256 / W tokens per pass
  const int ls = lane % W;
  constexpr int kSegs = kRThreads / W;
  for (int i0 = 0; i0 < tpc; i0 += kSegs) {
    const int i = i0 + static_cast<int>(threadIdx.x) / W;
    const int t = t0 + i;
    const bool valid = i < tpc && t < T;
    float l[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = ls * PER + j;
      l[j] = (valid && e < N) ? recv[i * N + e] : 0.f;
    }
    // p replaces the token's logits in its own row (read above by this segment)
    route_token_seg<W, PER>(ra, t, valid, l, ra.colsum ? recv + i * N : nullptr);
  }
  if (ra.colsum) {
    __syncthreads();
    colsum_rows(recv, max(0, min(tpc, T - t0)), N, ra.colsum + static_cast<size_t>(blockIdx.x) * N);
  }
}

template <int NB, int W, int PER>
cudaError_t launch_router(const CUtensorMap& mX, const CUtensorMap& mW, const RouterPlan& plan,
                          int num_kb, const RouteArgs& ra, int32_t* status, cudaStream_t s) {
  constexpr int smem = router_smem_bytes<NB>();
  static bool attr_set[64] = {};  // per device; setting it twice is harmless
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    err = cudaFuncSetAttribute(router_tc_kernel<NB, W, PER>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(plan.cluster);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.m_tiles * plan.cluster));
  cfg.blockDim = dim3(kRThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, router_tc_kernel<NB, W, PER>, mX, mW, ra, num_kb, status);
}

}  // namespace

bool router_tc_supported(int dtype, int d, int N) {
  return dtype == 1 && d % 64 == 0 && N % 8 == 0 && N <= 256;
}

RouterPlan router_plan(int T, int d, int N) {
  RouterPlan p;
  p.m_tiles = (T + kRM - 1) / kRM;
  const int num_kb = d / kRK;
  const int per_sm = N <= 64 ? 2 : 1;  // CTAs whose shared memory fits on one SM
  const int slots = device_sm_count() * per_sm;
  int c = kMaxCluster;
  while (c > 1 && (num_kb % c != 0 || p.m_tiles * c > slots)) c >>= 1;
  p.cluster = c;
  p.colsum_rows = p.m_tiles * c;
  return p;
}

cudaError_t launch_router_tc(const void* x, const void* W_r, int d, const RouterPlan& plan,
                             const RouteArgs& ra, int32_t* status, cudaStream_t s) {
  const int T = ra.T, N = ra.N;
  if (T == 0) return cudaSuccess;
  if (plan.cluster < 1 || plan.cluster > kMaxCluster || (d / kRK) % plan.cluster != 0)
    return cudaErrorInvalidValue;
  CUtensorMap mX, mW;
  if (!make_tmap_2d_bf16(&mX, x, static_cast<uint64_t>(T), static_cast<uint64_t>(d), 64, kRM))
    return cudaErrorInvalidValue;
  if (!make_tmap_2d_bf16(&mW, W_r, static_cast<uint64_t>(d), static_cast<uint64_t>(N), 64, kRK))
    return cudaErrorInvalidValue;
  const int nkb = d / kRK;
  // (W, PER) = (route_seg_width(N), route_seg_per(N))
  if (N <= 8) return launch_router<1, 8, 1>(mX, mW, plan, nkb, ra, status, s);
  if (N <= 16) return launch_router<1, 8, 2>(mX, mW, plan, nkb, ra, status, s);
  if (N <= 32) return launch_router<1, 8, 4>(mX, mW, plan, nkb, ra, status, s);
  if (N <= 64) return launch_router<1, 8, 8>(mX, mW, plan, nkb, ra, status, s);
  if (N <= 128) return launch_router<2, 16, 8>(mX, mW, plan, nkb, ra, status, s);
  if (N <= 256) return launch_router<4, 32, 8>(mX, mW, plan, nkb, ra, status, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
