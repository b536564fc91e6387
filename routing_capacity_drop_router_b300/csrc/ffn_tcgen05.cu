// Grouped expert GEMM on the 5th-generation tensor cores (tcgen05), bf16 in,
// fp32 accumulate in tensor memory.
//
// The experts are independent FFNs ("MoE vs MoT: routing and inference cost",
// section "MoE basic structure": the FFN layer replicated N times), and their
// rows are expert-contiguous after dispatch, so the expert FFN is one grouped
// GEMM over segments (the same page, section "measured figures", names grouped
// GEMM as the serving optimisation for experts).
//
//   SwiGLU (GEMM1): out[r, n] = silu(A[r] . W1[s][:, n]) * (A[r] . W3[s][:, n])
//   plain  (GEMM2): out[r, n] = A[r] . B[s][:, n]
// for rows r of segment s = [offsets[s], offsets[s+1]).
//
// Design (one CTA per SM, persistent):
//   tile = 128 rows x 256 accumulator columns; SwiGLU tiles hold 128 columns
//   of W1 and the same 128 columns of W3 side by side, so one 128x256x16 MMA
//   produces both halves of a SwiGLU output tile.
//   warp 0   : TMA producer, 4-stage ring of (A 128x64, B 64x256) bf16 tiles
//              with 128-byte swizzle; A is K-major, B is read as stored
//              ([K, n] row-major = MN-major), so weights need no repack.
//   warp 1   : allocates 512 TMEM columns (two 256-column accumulators);
//              lane 0 issues tcgen05.mma and tcgen05.commit.
//   warps 2-5: epilogue, TMEM -> registers (tcgen05.ld 32x32b), SwiGLU in
//              fp32, bf16 stores; warp w reads TMEM lanes 32*(w%4)...
//   Tiles run segment by segment, n-tile by n-tile, m fastest, so CTAs that
//   run at the same time share the weight tile in L2. Segment sizes are read
//   on the device: no host synchronisation.
//   Every mbarrier wait is bounded (1 s of globaltimer); on expiry the CTA
//   raises a shared abort flag, every role leaves its loop, outstanding TMA
//   copies and MMAs are drained (bounded), TMEM is freed and
//   MOE_ERR_DEVICE_TIMEOUT is recorded in the status word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kBM = 128;
constexpr int kBN = 256;  // accumulator columns per tile
constexpr int kBK = 64;   // one 128-byte swizzle row of bf16
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBN * kBK * 2;
constexpr int kBBoxBytes = 64 * kBK * 2;  // one 64-column TMA box of B
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kTmemCols = 512;
constexpr int kThreads = 192;
constexpr int kMaxSegments = 256;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
constexpr int kErrDeviceTimeout = -7;  // MOE_ERR_DEVICE_TIMEOUT

struct __align__(8) Ctrl {
  unsigned long long full[kStages];
  unsigned long long empty[kStages];
  unsigned long long tfull[2];
  unsigned long long tempty[2];
  unsigned long long drain;
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  int tile_base[kMaxSegments + 1];  // first tile of each segment
  int mtiles[kMaxSegments];
  int seg_row[kMaxSegments + 1];    // offsets[], so a tile decodes from shared memory
};
constexpr int kSmemBytes = 1024 /*alignment slack*/ + kStages * kStageBytes + static_cast<int>(sizeof(Ctrl));

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), A K-major (bit 15 = 0), B MN-major (bit 16 = 1),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                            (static_cast<uint32_t>(kBN >> 3) << 17) |
                            (static_cast<uint32_t>(kBM >> 4) << 24);

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_tc_kernel(
    const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB1,
    const __grid_constant__ CUtensorMap tmB3, const int32_t* __restrict__ offsets, int S, int K,
    int n_out, int rows_max, __nv_bfloat16* __restrict__ out, int32_t* __restrict__ status,
    int withhold_kb) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + kStages * kStageBytes);
  volatile int* abort_flag = &ctrl->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_n = SWIGLU ? kBN / 2 : kBN;  // output columns per tile
  const int n_tiles = (n_out + tile_n - 1) / tile_n;
  const int num_kb = (K + kBK - 1) / kBK;

  // ---- set-up: barriers, tile table, TMEM ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctrl->tfull[b]), 1);
      mbar_init(smem_u32(&ctrl->tempty[b]), 128);
    }
    mbar_init(smem_u32(&ctrl->drain), 1);
    ctrl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  // barrier set-up overlaps the previous kernel; the offsets come from it
  pdl_launch_dependents();
  pdl_wait();
  if (warp == 0) {  // tile table: running count of m-tiles x n-tiles per segment
    int run = 0;
    for (int s0 = 0; s0 < S; s0 += 32) {
      const int s = s0 + lane;
      int mt = 0;
      int r0 = 0, r1 = 0;
      if (s < S) {
        r0 = offsets[s];
        r1 = offsets[s + 1];
        mt = (r1 - r0 + kBM - 1) / kBM;
        ctrl->seg_row[s] = r0;
        if (s == S - 1) ctrl->seg_row[S] = r1;
      }
      int incl = mt * n_tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (s < S) {
        ctrl->tile_base[s] = run + incl - mt * n_tiles;
        ctrl->mtiles[s] = mt;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      ctrl->tile_base[S] = run;
      ctrl->total_tiles = run;
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctrl->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctrl->tmem_base;
  const int total = ctrl->total_tiles;

  auto decode = [&](int tile, int& seg, int& row0, int& row_end, int& col0) {
    int lo = 0, hi = S - 1;  // last segment with tile_base <= tile (empty ones skipped)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ctrl->tile_base[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    seg = lo;
    const int local = tile - ctrl->tile_base[seg];
    const int mt = ctrl->mtiles[seg];
    const int n_idx = local / mt, m_idx = local - n_idx * mt;
    row0 = ctrl->seg_row[seg] + m_idx * kBM;
    row_end = ctrl->seg_row[seg + 1];
    col0 = n_idx * tile_n;
  };

  const uint32_t stage0 = base;
  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int stage = 0;
    uint32_t phase = 0;
    int issued[kStages];
    uint32_t issued_phase[kStages];
    for (int s = 0; s < kStages; ++s) issued[s] = 0, issued_phase[s] = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      int seg, row0, row_end, col0;
      decode(tile, seg, row0, row_end, col0);
      for (int kb = 0; kb < num_kb; ++kb) {
        const uint32_t fb = smem_u32(&ctrl->full[stage]);
        if (!mbar_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        mbar_expect_tx(fb, kStageBytes);
        if (kb == withhold_kb && tile == 0) {
          // failure-detection self-test: announce the stage's bytes but load
          // nothing, so the MMA issuer's bounded wait expires
          issued[stage] = 1;
          issued_phase[stage] = phase;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        const uint32_t sa = stage0 + stage * kStageBytes;
        const uint32_t sb = sa + kABytes;
        tma_load_2d(sa, &tmA, kb * kBK, row0, fb);
        if (SWIGLU) {
          tma_load_3d(sb + 0 * kBBoxBytes, &tmB1, col0, kb * kBK, seg, fb);
          tma_load_3d(sb + 1 * kBBoxBytes, &tmB1, col0 + 64, kb * kBK, seg, fb);
          tma_load_3d(sb + 2 * kBBoxBytes, &tmB3, col0, kb * kBK, seg, fb);
          tma_load_3d(sb + 3 * kBBoxBytes, &tmB3, col0 + 64, kb * kBK, seg, fb);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) tma_load_3d(sb + j * kBBoxBytes, &tmB1, col0 + 64 * j, kb * kBK, seg, fb);
        }
        issued[stage] = 1;
        issued_phase[stage] = phase;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) {  // drain copies in flight before the CTA can exit (bounded)
      for (int s = 0; s < kStages; ++s) {
        if (!issued[s]) continue;
        const unsigned long long t0 = global_ns();
        while (!mbar_try(smem_u32(&ctrl->full[s]), issued_phase[s]))
          if (global_ns() - t0 > kWaitLimitNs / 10) break;
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++local) {
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      if (!mbar_wait(smem_u32(&ctrl->tempty[buf]), (use & 1u) ^ 1u, abort_flag, kWaitLimitNs)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kBN);
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait(smem_u32(&ctrl->full[stage]), phase, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = stage0 + stage * kStageBytes;
        const uint32_t sb = sa + kABytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          tc_mma(d_tmem, kmajor_desc(sa, kk), mnmajor_desc(sb, kk, kBBoxBytes), kIdesc, (kb | kk) != 0 ? 1u : 0u);
        tc_commit(smem_u32(&ctrl->empty[stage]));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit(smem_u32(&ctrl->tfull[buf]));
    }
    // every MMA issued so far completes before this arrives
    tc_commit(smem_u32(&ctrl->drain));
    const unsigned long long t0 = global_ns();
    while (!mbar_try(smem_u32(&ctrl->drain), 0u))
      if (global_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        break;
      }
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    int local = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      int ok = 1;
      if (lane == 0) ok = mbar_wait(smem_u32(&ctrl->tfull[buf]), use & 1u, abort_flag, kWaitLimitNs);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      int seg, row0, row_end, col0;
      decode(tile, seg, row0, row_end, col0);
      const int row = row0 + q * 32 + lane;
      const bool valid = row >= 0 && row < row_end && row < rows_max;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * kBN);
      __nv_bfloat16* orow = out + static_cast<size_t>(row) * n_out;
      if (SWIGLU) {
#pragma unroll 1
        for (int c = 0; c < kBN / 2; c += 32) {
          uint32_t a[32], g[32];
          tc_ld32(taddr + c, a);
          tc_ld32(taddr + kBN / 2 + c, g);
          tc_wait_ld();
          if (valid && col0 + c < n_out) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float h0 = silu_fast(__uint_as_float(a[2 * i])) * __uint_as_float(g[2 * i]);
              const float h1 = silu_fast(__uint_as_float(a[2 * i + 1])) * __uint_as_float(g[2 * i + 1]);
              pk[i] = pack_bf16x2(h0, h1);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + col0 + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < kBN; c += 32) {
          uint32_t a[32];
          tc_ld32(taddr + c, a);
          tc_wait_ld();
          if (valid && col0 + c < n_out) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
            uint4* dst = reinterpret_cast<uint4*>(orow + col0 + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&ctrl->tempty[buf]));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0 && *abort_flag) record_status(status, kErrDeviceTimeout);
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace

cudaError_t launch_grouped_gemm_tc_bf16(const void* A, const int32_t* offsets, int S,
                                        int64_t rows_max, int K, int n_out, const void* B1,
                                        const void* B3, void* out, bool swiglu,
                                        int32_t* status, cudaStream_t s, int withhold_kb) {
  if (S == 0 || rows_max == 0) return cudaSuccess;
  if (S > kMaxSegments) return cudaErrorInvalidValue;
  CUtensorMap mA, mB1, mB3;
  if (!make_tmap_2d_bf16(&mA, A, static_cast<uint64_t>(rows_max), static_cast<uint64_t>(K), 64, kBM))
    return cudaErrorInvalidValue;
  if (!make_tmap_3d_bf16(&mB1, B1, S, K, n_out, 64, kBK)) return cudaErrorInvalidValue;
  if (swiglu) {
    if (!make_tmap_3d_bf16(&mB3, B3, S, K, n_out, 64, kBK)) return cudaErrorInvalidValue;
  } else {
    mB3 = mB1;
  }
  const int tile_n = swiglu ? kBN / 2 : kBN;
  const long long n_tiles = (n_out + tile_n - 1) / tile_n;
  const long long m_tiles_max = (rows_max + kBM - 1) / kBM + S;
  long long grid = n_tiles * m_tiles_max;
  const int sms = device_sm_count();
  if (grid > sms) grid = sms;

  static bool attr_set[64][2] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev][swiglu ? 1 : 0]) {
    err = swiglu ? cudaFuncSetAttribute(grouped_gemm_tc_kernel<true>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)
                 : cudaFuncSetAttribute(grouped_gemm_tc_kernel<false>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_set[dev][swiglu ? 1 : 0] = true;
  }
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  const int rmax = rows_max > 0x7fffffff ? 0x7fffffff : static_cast<int>(rows_max);
  if (swiglu)
    return launch_pdl(grouped_gemm_tc_kernel<true>, static_cast<unsigned>(grid), kThreads,
                      kSmemBytes, s, mA, mB1, mB3, offsets, S, K, n_out, rmax, o, status,
                      withhold_kb);
  return launch_pdl(grouped_gemm_tc_kernel<false>, static_cast<unsigned>(grid), kThreads,
                    kSmemBytes, s, mA, mB1, mB3, offsets, S, K, n_out, rmax, o, status,
                    withhold_kb);
}

}  // namespace moe
