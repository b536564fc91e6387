// Grouped expert GEMM with e4m3 (FP8) expert weights and bf16 activations on
// the tcgen05 tensor cores.
//
// The expert FFN is the same grouped GEMM as ffn_tcgen05.cu ("MoE vs MoT:
// routing and inference cost", section "MoE basic structure"; grouped GEMM in
// section "measured figures"); here the weights of every expert are stored as
// e4m3 bytes with one fp32 scale per output column, W[k, n] = value(q[k, n]) *
// scale[n], which halves the bytes a weight-bound (decode) step streams. The
// activations stay bf16: each e4m3 value is exactly representable in bf16, so
// the weight tiles are widened to bf16 in shared memory and multiplied with
// kind::f16 MMAs; the per-column scale multiplies the fp32 accumulator in the
// epilogue (a column factor commutes with the sum over k).
//
// Design (one CTA per SM, persistent, one CTA per 128-row tile):
//   warp 0   : TMA producer of the weight bytes (two 128-column x 64-deep
//              e4m3 boxes per k-block, 128-byte swizzle) into a 6-stage ring:
//              a weight-bound step is limited by the bytes each SM keeps in
//              flight, so the bytes get the deepest ring;
//   warp 14  : TMA producer of A (128 x 64 bf16, 128-byte swizzle) into a
//              3-stage ring;
//   warps 6-13: converters: e4m3 -> bf16 of a byte stage into one of two bf16
//              operand buffers, in the MN-major 128-byte-swizzled layout the
//              MMA reads (four 64-column boxes), then a proxy fence, an
//              arrival on that buffer's barrier and the byte stage's release;
//   warp 1   : TMEM allocation (two 256-column accumulators); lane 0 issues
//              the 128x256x16 MMAs (A from its ring, B from the bf16 buffer)
//              and commits both back to their producers;
//   warps 2-5: epilogue, TMEM -> registers, column scales, SwiGLU in fp32,
//              bf16 stores.
//   SwiGLU tiles hold 128 columns of W1 next to the same 128 columns of W3.
//   Every mbarrier wait is bounded (1 s of globaltimer); on expiry the CTA
//   raises its abort flag, every role leaves its loop, copies and MMAs in
//   flight are drained, TMEM is freed and MOE_ERR_DEVICE_TIMEOUT is recorded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kBM = 128;
constexpr int kBN = 256;                   // accumulator columns per tile
constexpr int kBK = 64;
constexpr int kB8Stages = 6;  // TMA ring of e4m3 weight bytes
constexpr int kAStages = 3;   // TMA ring of A
constexpr int kBufs = 2;      // bf16 operand buffers
constexpr int kABytes = kBM * kBK * 2;     // bf16 A tile
constexpr int kB8BoxBytes = 128 * kBK;     // one 128-column e4m3 box
constexpr int kB8Bytes = 2 * kB8BoxBytes;  // 256 columns of bytes
constexpr int kB16BoxBytes = 64 * kBK * 2; // one 64-column bf16 box
constexpr int kB16Bytes = 4 * kB16BoxBytes;

constexpr int kTmemCols = 512;
constexpr int kConvWarps = 8;
constexpr int kAWarp = 6 + kConvWarps;
constexpr int kThreads = 32 * (kAWarp + 1);
constexpr int kMaxSegments = 256;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
constexpr int kErrDeviceTimeout = -7;  // MOE_ERR_DEVICE_TIMEOUT

struct __align__(8) Ctrl {
  unsigned long long b8full[kB8Stages];   // weight bytes landed
  unsigned long long b8empty[kB8Stages];  // converted: the stage may be refilled
  unsigned long long afull[kAStages];     // A landed
  unsigned long long aempty[kAStages];    // MMAs done with A
  unsigned long long bfull[kBufs];        // bf16 B written
  unsigned long long bempty[kBufs];       // MMAs done with the bf16 B
  unsigned long long tfull[2];
  unsigned long long tempty[2];
  unsigned long long drain;
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  int tile_base[kMaxSegments + 1];
  int mtiles[kMaxSegments];
  int seg_row[kMaxSegments + 1];
};
constexpr int kSmemBytes = 1024 + kB8Stages * kB8Bytes + kAStages * kABytes +
                           kBufs * kB16Bytes + static_cast<int>(sizeof(Ctrl));
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// kind::f16: D fp32, A and B bf16, A K-major, B MN-major, N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                            (static_cast<uint32_t>(kBN >> 3) << 17) |
                            (static_cast<uint32_t>(kBM >> 4) << 24);

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Two e4m3 values (low byte first) -> two bf16 (low half first): the hardware
// widens the pair to f16 and each f16 to f32, which packs to bf16; exact for
// every byte, subnormals included, since each e4m3 value is an f16 and a bf16
// value.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<unsigned short>(two)));
  const float lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xffffu)));
  const float hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
  return pack_bf16x2(lo, hi);
}

// 16 e4m3 bytes -> 16 bf16 (8 words, in order). No branch, so the compiler
// overlaps the items a thread converts. (Integer rebiasing of the f16 or e4m3
// bits measured slower on this part than the conversion instructions.)
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 v, uint32_t (&o)[8]) {
  const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    o[2 * j] = e4m3x2_to_bf16x2(wv[j] & 0xffffu);
    o[2 * j + 1] = e4m3x2_to_bf16x2(wv[j] >> 16);
  }
}

template <bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_w8_kernel(
    const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB1,
    const __grid_constant__ CUtensorMap tmB3, const float* __restrict__ sc1,
    const float* __restrict__ sc3, const int32_t* __restrict__ offsets, int S, int K, int n_out,
    int rows_max, __nv_bfloat16* __restrict__ out, int32_t* __restrict__ status) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw);
  unsigned char* b8_base = smem;
  unsigned char* a_base = b8_base + kB8Stages * kB8Bytes;
  unsigned char* b16_base = a_base + kAStages * kABytes;
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(b16_base + kBufs * kB16Bytes);
  volatile int* abort_flag = &ctrl->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_n = SWIGLU ? kBN / 2 : kBN;
  const int n_tiles = (n_out + tile_n - 1) / tile_n;
  const int num_kb = (K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kB8Stages; ++s) {
      mbar_init(smem_u32(&ctrl->b8full[s]), 1);
      mbar_init(smem_u32(&ctrl->b8empty[s]), kConvWarps);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(smem_u32(&ctrl->afull[s]), 1);
      mbar_init(smem_u32(&ctrl->aempty[s]), 1);
    }
    for (int b = 0; b < kBufs; ++b) {
      mbar_init(smem_u32(&ctrl->bfull[b]), kConvWarps);
      mbar_init(smem_u32(&ctrl->bempty[b]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctrl->tfull[b]), 1);
      mbar_init(smem_u32(&ctrl->tempty[b]), 4);
    }
    mbar_init(smem_u32(&ctrl->drain), 1);
    ctrl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  pdl_launch_dependents();
  pdl_wait();
  if (warp == 0) {  // tile table: running count of m-tiles x n-tiles per segment
    int run = 0;
    for (int s0 = 0; s0 < S; s0 += 32) {
      const int s = s0 + lane;
      int mt = 0;
      if (s < S) {
        const int r0 = offsets[s], r1 = offsets[s + 1];
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
    int lo = 0, hi = S - 1;
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

  if ((warp == 0 || warp == kAWarp) && lane == 0) {
    // ---------------- TMA producers: weight bytes (warp 0), A (kAWarp) ----------------
    const bool bytes = warp == 0;
    const int n_st = bytes ? kB8Stages : kAStages;
    unsigned long long* fullb = bytes ? ctrl->b8full : ctrl->afull;
    unsigned long long* emptyb = bytes ? ctrl->b8empty : ctrl->aempty;
    int stage = 0;
    uint32_t phase = 0;
    int issued[kB8Stages];
    uint32_t issued_phase[kB8Stages];
    for (int s = 0; s < kB8Stages; ++s) issued[s] = 0, issued_phase[s] = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      int seg, row0, row_end, col0;
      decode(tile, seg, row0, row_end, col0);
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait(smem_u32(&emptyb[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&fullb[stage]);
        mbar_expect_tx(fb, bytes ? kB8Bytes : kABytes);
        issued[stage] = 1;
        issued_phase[stage] = phase;
        if (bytes) {
          const uint32_t s8 = smem_u32(b8_base + stage * kB8Bytes);
          if (SWIGLU) {
            tma_load_3d(s8, &tmB1, col0, kb * kBK, seg, fb);
            tma_load_3d(s8 + kB8BoxBytes, &tmB3, col0, kb * kBK, seg, fb);
          } else {
            tma_load_3d(s8, &tmB1, col0, kb * kBK, seg, fb);
            tma_load_3d(s8 + kB8BoxBytes, &tmB1, col0 + 128, kb * kBK, seg, fb);
          }
        } else {
          tma_load_2d(smem_u32(a_base + stage * kABytes), &tmA, kb * kBK, row0, fb);
        }
        if (++stage == n_st) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) {  // copies in flight land before the CTA can exit (bounded)
      for (int s = 0; s < n_st; ++s) {
        if (!issued[s]) continue;
        const unsigned long long t0 = global_ns();
        while (!mbar_try(smem_u32(&fullb[s]), issued_phase[s]))
          if (global_ns() - t0 > kWaitLimitNs / 10) break;
      }
    }
  } else if (warp >= 6 && warp < kAWarp) {
    // ---------------- converters: e4m3 bytes -> bf16 MMA operand ----------------
    const int ct = threadIdx.x - 6 * 32;  // 0 .. 32 * kConvWarps - 1
    int stage = 0, buf = 0;
    uint32_t phase = 0, bphase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      for (int kb = 0; kb < num_kb; ++kb) {
        int w = 1;
        if (lane == 0) {
          w = mbar_wait(smem_u32(&ctrl->b8full[stage]), phase, abort_flag, kWaitLimitNs) &&
              mbar_wait(smem_u32(&ctrl->bempty[buf]), bphase ^ 1u, abort_flag, kWaitLimitNs);
        }
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
        const unsigned char* s8 = b8_base + stage * kB8Bytes;
        unsigned char* s16 = b16_base + buf * kB16Bytes;
        // item = (byte box, k-row r, 16-byte chunk c); 2 x 64 x 8 items
#pragma unroll
        for (int it = 0; it < (2 * 64 * 8 + kConvWarps * 32 - 1) / (kConvWarps * 32); ++it) {
          // a quarter-warp (8 lanes) takes one chunk c of 8 consecutive rows:
          // its 16-byte loads and both 16-byte stores then hit 8 distinct
          // chunk positions of the 128-byte swizzle rows (no bank conflict)
          const int item = ct + it * kConvWarps * 32;
          if (item >= 2 * 64 * 8) break;  // uniform per warp: items come in warp-sized runs
          const int ln = item & 31, rest = item >> 5;
          const int r = ((rest >> 1) & 7) * 8 + (ln & 7);
          const int c = (rest & 1) * 4 + (ln >> 3);
          const int box = rest >> 4;
          const uint4 v = *reinterpret_cast<const uint4*>(
              s8 + box * kB8BoxBytes + r * 128 + ((c ^ (r & 7)) << 4));
          uint32_t o[8];
          e4m3x16_to_bf16(v, o);
          // 16 columns n = 16c .. 16c+15 of the byte box: bf16 box 2*box + c/4,
          // 16-byte chunks q and q+1 of its 128-byte row r, q = 2*(c%4)
          unsigned char* row = s16 + (2 * box + (c >> 2)) * kB16BoxBytes + r * 128;
          const int q = 2 * (c & 3);
          *reinterpret_cast<uint4*>(row + ((q ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(row + (((q + 1) ^ (r & 7)) << 4)) =
              make_uint4(o[4], o[5], o[6], o[7]);
        }
        // the MMA reads these through the async proxy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&ctrl->bfull[buf]));
          mbar_arrive(smem_u32(&ctrl->b8empty[stage]));  // the bytes are consumed
        }
        if (++stage == kB8Stages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++buf == kBufs) {
          buf = 0;
          bphase ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    int stage = 0, bb = 0;
    uint32_t phase = 0, bphase = 0;
    int local = 0;
    bool ok = true;
    const uint32_t b16_0 = smem_u32(b16_base);
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
        // A landed and B converted
        if (!mbar_wait(smem_u32(&ctrl->afull[stage]), phase, abort_flag, kWaitLimitNs) ||
            !mbar_wait(smem_u32(&ctrl->bfull[bb]), bphase, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(a_base + stage * kABytes);
        const uint32_t sb = b16_0 + bb * kB16Bytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          tc_mma(d_tmem, kmajor_desc(sa, kk), mnmajor_desc(sb, kk, kB16BoxBytes), kIdesc,
                 (kb | kk) != 0 ? 1u : 0u);
        tc_commit(smem_u32(&ctrl->aempty[stage]));
        tc_commit(smem_u32(&ctrl->bempty[bb]));
        if (++stage == kAStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++bb == kBufs) {
          bb = 0;
          bphase ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit(smem_u32(&ctrl->tfull[buf]));
    }
    tc_commit(smem_u32(&ctrl->drain));
    const unsigned long long t0 = global_ns();
    while (!mbar_try(smem_u32(&ctrl->drain), 0u))
      if (global_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        break;
      }
  } else if (warp >= 2 && warp < 6) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;
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
      const bool valid = row < row_end && row < rows_max;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * kBN);
      __nv_bfloat16* orow = out + static_cast<size_t>(row) * n_out;
      const float* s1 = sc1 + static_cast<size_t>(seg) * n_out;
      const float* s3 = SWIGLU ? sc3 + static_cast<size_t>(seg) * n_out : nullptr;
      // 16 columns at a time keeps the epilogue's registers low enough for
      // eight converter warps next to it
      if (SWIGLU) {
#pragma unroll 1
        for (int c = 0; c < kBN / 2; c += 16) {
          uint32_t a[16], g[16];
          tc_ld16(taddr + c, a);
          tc_ld16(taddr + kBN / 2 + c, g);
          tc_wait_ld();
          if (valid && col0 + c < n_out) {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int n = col0 + c + 2 * i;
              const float a0 = __uint_as_float(a[2 * i]) * s1[n];
              const float a1 = __uint_as_float(a[2 * i + 1]) * s1[n + 1];
              const float g0 = __uint_as_float(g[2 * i]) * s3[n];
              const float g1 = __uint_as_float(g[2 * i + 1]) * s3[n + 1];
              pk[i] = pack_bf16x2(silu_fast(a0) * g0, silu_fast(a1) * g1);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + col0 + c);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < kBN; c += 16) {
          uint32_t a[16];
          tc_ld16(taddr + c, a);
          tc_wait_ld();
          if (valid && col0 + c < n_out) {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int n = col0 + c + 2 * i;
              pk[i] = pack_bf16x2(__uint_as_float(a[2 * i]) * s1[n],
                                  __uint_as_float(a[2 * i + 1]) * s1[n + 1]);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + col0 + c);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctrl->tempty[buf]));
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

cudaError_t launch_grouped_gemm_tc_w8(const void* A, const int32_t* offsets, int S,
                                      int64_t rows_max, int K, int n_out, const void* B1,
                                      const float* sc1, const void* B3, const float* sc3,
                                      void* out, bool swiglu, int32_t* status, cudaStream_t s) {
  if (S == 0 || rows_max == 0) return cudaSuccess;
  if (S > kMaxSegments || n_out % 128 != 0) return cudaErrorInvalidValue;
  CUtensorMap mA, mB1, mB3;
  if (!make_tmap_2d_bf16(&mA, A, static_cast<uint64_t>(rows_max), static_cast<uint64_t>(K), 64, kBM))
    return cudaErrorInvalidValue;
  if (!make_tmap_3d_u8(&mB1, B1, S, K, n_out, 128, kBK)) return cudaErrorInvalidValue;
  if (swiglu) {
    if (!make_tmap_3d_u8(&mB3, B3, S, K, n_out, 128, kBK)) return cudaErrorInvalidValue;
  } else {
    mB3 = mB1;
  }
  const int tile_n = swiglu ? kBN / 2 : kBN;
  const long long n_tiles = (n_out + tile_n - 1) / tile_n;
  long long grid = n_tiles * ((rows_max + kBM - 1) / kBM + S);
  const int sms = device_sm_count();
  if (grid > sms) grid = sms;
  static bool attr_set[64][2] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev][swiglu ? 1 : 0]) {
    err = swiglu ? cudaFuncSetAttribute(grouped_gemm_w8_kernel<true>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)
                 : cudaFuncSetAttribute(grouped_gemm_w8_kernel<false>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_set[dev][swiglu ? 1 : 0] = true;
  }
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  const int rmax = rows_max > 0x7fffffff ? 0x7fffffff : static_cast<int>(rows_max);
  if (swiglu)
    return launch_pdl(grouped_gemm_w8_kernel<true>, static_cast<unsigned>(grid), kThreads,
                      kSmemBytes, s, mA, mB1, mB3, sc1, sc3, offsets, S, K, n_out, rmax, o, status);
  return launch_pdl(grouped_gemm_w8_kernel<false>, static_cast<unsigned>(grid), kThreads,
                    kSmemBytes, s, mA, mB1, mB3, sc1, sc3, offsets, S, K, n_out, rmax, o, status);
}

}  // namespace moe
