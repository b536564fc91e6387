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
// Design (persistent, warp-specialised; one CTA per SM):
//   tile = 256 rows x 256 accumulator columns computed by a CTA pair (a
//   cluster of 2 CTAs, tcgen05 cta_group::2): CTA r holds rows 128r..128r+127
//   of A and columns 128r..128r+127 of B in its shared memory, and its tensor
//   memory receives its 128 rows of the 256-column accumulator. Each SM thus
//   loads 32 KiB per 64-deep k-block for 128x256x64 of MMA work instead of
//   48 KiB, and 6 stages of buffering fit in shared memory. SwiGLU tiles put
//   128 columns of W1 (CTA 0) next to the same 128 columns of W3 (CTA 1), so
//   one M=256, N=256 MMA produces both halves of a SwiGLU output tile.
//   A segment's last tile, when it has fewer than 256 rows, runs transposed
//   (out^T = W^T A^T): the weight columns become the MMA's M = 256 (MN-major,
//   loaded as before) and the tile's n token rows its N, n rounded up to 32
//   and split N/2 : N/2 over the pair, so the tail costs n/256 of a tile
//   instead of a whole one. Each product is the same sum over the same k, and
//   the outputs equal the padded form's bit for bit. The epilogue then reads
//   a TMEM lane per output column and stores rows transposed, neighbouring
//   lanes trading one value so each writes 32-bit words; under SwiGLU the
//   gate and up halves of a column sit in different lane quadrants and meet
//   through a small shared-memory exchange. Without SwiGLU (the second GEMM)
//   every pair tile runs transposed, full ones with N = 256: the same
//   products, and the transposed epilogue's stores (64 contiguous bytes of a
//   row per half-warp) load the memory system less than one 16-byte store
//   per row per lane; under SwiGLU full tiles keep the untransposed form,
//   whose epilogue needs no exchange.
//   Where clusters cannot be formed the same kernel runs one CTA per tile
//   (128 rows, both B halves, cta_group::1, 4 stages).
//   warp 0   : TMA producer of its CTA's operand tiles (128-byte swizzle); A
//              is K-major, B is read as stored ([K, n] row-major = MN-major),
//              so weights need no repack. In a pair both producers count
//              their bytes on CTA 0's full barrier.
//              Row-gather form (GATHER): A row r is row row_src[r] of the
//              token matrix x, so the dispatched copy of x is never written.
//              Four copy warps (warp 0 and warps 6-8) each copy 32 rows of
//              the A tile with 16-byte cp.async into the same swizzled layout
//              TMA would produce (lane: chunk lane % 8 of rows 32w + 4i +
//              lane / 8); each warp announces a k-block's rows on the full
//              barrier (one arrival per copy warp, after its copies land and a
//              proxy fence) while up to stages - 1 later k-blocks are in
//              flight; lane 0 of warp 0 still loads B by TMA.
//   warp 1   : allocates 512 TMEM columns (two 256-column accumulators);
//              lane 0 of CTA 0 issues tcgen05.mma and tcgen05.commit, whose
//              arrivals are multicast to both CTAs' barriers.
//   warps 2-5: epilogue, TMEM -> registers (tcgen05.ld 32x32b), SwiGLU in
//              fp32, bf16 stores; warp w reads TMEM lanes 32*(w%4)...; each
//              warp signals CTA 0's accumulator-empty barrier when done.
//   Tiles run segment by segment, n-tile by n-tile, m fastest, so units that
//   run at the same time share the weight tile in L2. Segment sizes are read
//   on the device: no host synchronisation.
//   FP8 form: A is e4m3 [rows, K] with one fp32 scale per row, B is e4m3
//   stored K-major ([n_out, K] per segment) with one fp32 scale per column;
//   a 128-byte k-block then holds 128 k, B tiles are K-major like A, the MMAs
//   are kind::f8f6f4 (e4m3 x e4m3, fp32 accumulate) and the epilogue scales
//   each accumulator by its row's and column's scales before the SwiGLU.
//   The producers' waits for a free stage and the epilogue's waits for a
//   full accumulator suspend in the barrier (try_wait with a time hint)
//   rather than spin; the MMA issuer, on the critical path, spins.
//   Every mbarrier wait is bounded (1 s of globaltimer); on expiry the CTA
//   raises a shared abort flag, every role leaves its loop, outstanding TMA
//   copies and MMAs are drained (bounded), TMEM is freed and
//   MOE_ERR_DEVICE_TIMEOUT is recorded in the status word. The cluster
//   barriers at entry and exit are reached by every thread whatever happened
//   in between (all waits before them are bounded).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>

#include "device_common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kBM = 128;  // rows per CTA (TMEM lanes)
constexpr int kBN = 256;  // accumulator columns per tile
constexpr int kBK = 64;   // one 128-byte swizzle row of bf16
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBoxBytes = 64 * kBK * 2;  // one 64-column TMA box of B
constexpr int kTmemCols = 512;
constexpr int kThreads = 192;
constexpr int kCopyWarps = 4;  // row-gather form: warp 0 and warps 6..8 copy A rows
constexpr int kThreadsGather = kThreads + 32 * (kCopyWarps - 1);
template <bool GATHER>
constexpr int threads_of() { return GATHER ? kThreadsGather : kThreads; }
constexpr int kEpiWarps = 4;
constexpr int kMaxSegments = 256;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
constexpr int kErrDeviceTimeout = -7;  // MOE_ERR_DEVICE_TIMEOUT
constexpr int kErrDeviceBounds = -8;   // MOE_ERR_DEVICE_BOUNDS

// Geometry of the pair (PAIR) and single-CTA forms.
template <bool PAIR>
struct Geo {
  static constexpr int kStages = PAIR ? 6 : 4;
  static constexpr int kBoxes = PAIR ? 2 : 4;  // 64-column B boxes this CTA loads per k-block
  static constexpr int kStageBytes = kABytes + kBoxes * kBoxBytes;
  static constexpr int kTileRows = PAIR ? 2 * kBM : kBM;
  // bytes the MMA issuer's full barrier waits for per k-block (both CTAs)
  static constexpr uint32_t kTxBytes = (PAIR ? 2u : 1u) * static_cast<uint32_t>(kStageBytes);
  // the same with A gathered by cp.async (B bytes only)
  static constexpr uint32_t kTxBytesB = (PAIR ? 2u : 1u) * static_cast<uint32_t>(kBoxes * kBoxBytes);
  // Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A bf16 (7-9 =
  // 1), B bf16 (10-12 = 1), A K-major (bit 15 = 0), B MN-major (bit 16 = 1),
  // N >> 3 in bits 17-22, M >> 4 in bits 24-28 (M = 256 for a pair).
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                                     (static_cast<uint32_t>(kBN >> 3) << 17) |
                                     (static_cast<uint32_t>(kTileRows >> 4) << 24);
};

// Transposed tail tile of a pair (see the file comment): the weight columns
// are the MMA's A operand (M = 256, MN-major as stored), the tile's n token
// rows its B operand (N = n rounded up to 32, the step of N for a CTA-pair
// MMA; K-major), so the accumulator holds out^T: TMEM lane = output column,
// TMEM column = token row.
__host__ __device__ constexpr uint32_t swap_idesc(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (0u << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>((2 * kBM) >> 4) << 24);
}
// SwiGLU epilogue of a transposed tile: gate and up values of one output
// column sit in different TMEM lane quadrants, so the epilogue warps swap
// half of each 32-token chunk through shared memory (two buffers of
// [2 column groups][2 directions][16 tokens][32 lanes] fp32).
constexpr int kXchgFloats = 2 * 2 * 16 * 32;
constexpr int kXchgBytes = 2 * kXchgFloats * 4;

template <int STAGES>
struct __align__(8) Ctrl {
  unsigned long long full[STAGES];
  unsigned long long empty[STAGES];
  unsigned long long tfull[2];
  unsigned long long tempty[2];
  unsigned long long xchg[2];  // transposed SwiGLU exchange, one per buffer
  unsigned long long drain;
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  int tile_base[kMaxSegments + 1];  // first tile of each segment
  int mtiles[kMaxSegments];
  int seg_row[kMaxSegments + 1];    // offsets[], so a tile decodes from shared memory
};
template <bool PAIR>
constexpr int xchg_bytes() { return PAIR ? kXchgBytes : 0; }
template <bool PAIR>
constexpr int smem_bytes() {
  return 1024 /*alignment slack*/ + Geo<PAIR>::kStages * Geo<PAIR>::kStageBytes +
         xchg_bytes<PAIR>() + static_cast<int>(sizeof(Ctrl<Geo<PAIR>::kStages>));
}
static_assert(smem_bytes<true>() <= 227 * 1024, "shared memory");
static_assert(smem_bytes<false>() <= 227 * 1024, "shared memory");

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Transposed-tile store: lane l of the warp holds column col (= c_base + l) of
// rows t0 .. t0 + CNT - 1 in v[]. Neighbouring lanes trade one value, so that
// the even lane writes columns (col, col + 1) of row t0 + i and the odd lane
// the same two columns of row t0 + i + 1, each as one 32-bit word. Rows at
// or beyond lim and columns at or beyond n_out (even) are not written.
template <int CNT>
__device__ __forceinline__ void store_transposed(const float* v, int t0, int col, int lim,
                                                 int n_out, __nv_bfloat16* __restrict__ out,
                                                 int lane) {
  const int odd = lane & 1;
  const int c = col & ~1;
#pragma unroll
  for (int i = 0; i < CNT; i += 2) {
    const float send = odd ? v[i] : v[i + 1];
    const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
    const int t = t0 + i + odd;
    const uint32_t w = odd ? pack_bf16x2(recv, v[i + 1]) : pack_bf16x2(v[i], recv);
    if (t < lim && c < n_out)
      *reinterpret_cast<uint32_t*>(out + static_cast<size_t>(t) * n_out + c) = w;
  }
}

template <bool PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t dst) {
  if (PAIR) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
}
template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t base) {
  if (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(kTmemCols)
                 : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(kTmemCols)
                 : "memory");
}

// Instruction descriptor of the FP8 form, kind::f8f6f4: D fp32 (bits 4-5 =
// 1), A and B e4m3 (bits 7-9 and 10-12 = 0), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
template <bool PAIR>
constexpr uint32_t fp8_idesc() {
  return (1u << 4) | (static_cast<uint32_t>(kBN >> 3) << 17) |
         (static_cast<uint32_t>(Geo<PAIR>::kTileRows >> 4) << 24);
}

template <bool SWIGLU, bool PAIR, bool GATHER, bool FP8>
__global__ void __launch_bounds__(threads_of<GATHER>(), 1) grouped_gemm_tc_kernel(
    const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB1,
    const __grid_constant__ CUtensorMap tmB3, const int32_t* __restrict__ offsets, int S, int K,
    int n_out, int rows_max, __nv_bfloat16* __restrict__ out, int32_t* __restrict__ status,
    int withhold_kb, const __nv_bfloat16* __restrict__ xg, const int32_t* __restrict__ row_src,
    int x_rows, const float* __restrict__ a_scale, const float* __restrict__ b1_scale,
    const float* __restrict__ b3_scale, int swap_tails) {
  static_assert(!(GATHER && FP8), "the row gather reads bf16 token rows");
  using G = Geo<PAIR>;
  // segment tails of a bf16 pair run transposed (swap_tails != 0)
  constexpr bool kSwap = PAIR && !GATHER && !FP8;
  constexpr int kStages = G::kStages;
  // elements of k per 128-byte k-block
  constexpr int kKE = FP8 ? 2 * kBK : kBK;
  constexpr uint32_t kIdesc = FP8 ? fp8_idesc<PAIR>() : G::kIdesc;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw);
  float* xchg = reinterpret_cast<float*>(smem + kStages * G::kStageBytes);
  Ctrl<kStages>* ctrl =
      reinterpret_cast<Ctrl<kStages>*>(smem + kStages * G::kStageBytes + xchg_bytes<PAIR>());
  volatile int* abort_flag = &ctrl->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_rank() : 0u;  // 0 issues the MMAs
  const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int n_units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int tile_n = SWIGLU ? kBN / 2 : kBN;  // output columns per tile
  const int n_tiles = (n_out + tile_n - 1) / tile_n;
  const int num_kb = (K + kKE - 1) / kKE;

  // ---- set-up: barriers, tile table, TMEM ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // GATHER: the expect_tx arrival plus one per copy warp of each CTA
      // once its rows landed
      mbar_init(smem_u32(&ctrl->full[s]), GATHER ? 1 + kCopyWarps * (PAIR ? 2 : 1) : 1);
      mbar_init(smem_u32(&ctrl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctrl->tfull[b]), 1);
      mbar_init(smem_u32(&ctrl->tempty[b]), (PAIR ? 2 : 1) * kEpiWarps);
      mbar_init(smem_u32(&ctrl->xchg[b]), 32 * kEpiWarps);  // every epilogue thread
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
        mt = (r1 - r0 + G::kTileRows - 1) / G::kTileRows;
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
  if (warp == 1) tmem_alloc<PAIR>(smem_u32(&ctrl->tmem_base));
  tc_fence_before();
  __syncthreads();
  if (PAIR) {  // the peer's barriers are initialised before anything targets them
    __syncwarp();
    cluster_sync();
  }
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
    row0 = ctrl->seg_row[seg] + m_idx * G::kTileRows;
    row_end = ctrl->seg_row[seg + 1];
    col0 = n_idx * tile_n;
  };
  // A segment's last tile with fewer rows than a pair tile runs transposed,
  // N = its rows rounded up to 32 (nsw), instead of padding the rows to 256;
  // without SwiGLU every tile does (full ones with N = 256).
  auto transposed = [&](int row0, int row_end, int& nsw) {
    const int n = min(min(row_end, rows_max) - row0, G::kTileRows);
    nsw = (n + 31) & ~31;
    return kSwap && swap_tails != 0 && n > 0 && (!SWIGLU || n < G::kTileRows);
  };

  const uint32_t stage0 = base;
  // B tiles of one k-block: CTA 0 of a pair W1 (or B) columns col0.., CTA 1
  // W3 columns col0.. (or B columns col0 + 128..); one CTA: all of them
  // A transposed SwiGLU tile gives each CTA 64 columns of W1 and the same 64
  // of W3 (col0 + 64 * rank ..), so one CTA's TMEM holds gate and up of the
  // same output columns.
  auto load_b = [&](uint32_t sb, uint32_t fb, int seg, int col0, int kb, bool sw) {
    if (FP8) {  // K-major boxes of 128 k x 128 columns (16 KiB)
      constexpr int kBox8 = 128 * 128;
      if (PAIR) {
        const CUtensorMap* mb = (SWIGLU && rank == 1) ? &tmB3 : &tmB1;
        const int c = SWIGLU ? col0 : col0 + static_cast<int>(rank) * 128;
        tma_load_3d_pair(sb, mb, kb * kKE, c, seg, fb);
      } else if (SWIGLU) {
        tma_load_3d(sb, &tmB1, kb * kKE, col0, seg, fb);
        tma_load_3d(sb + kBox8, &tmB3, kb * kKE, col0, seg, fb);
      } else {
        tma_load_3d(sb, &tmB1, kb * kKE, col0, seg, fb);
        tma_load_3d(sb + kBox8, &tmB1, kb * kKE, col0 + 128, seg, fb);
      }
      return;
    }
    if (PAIR && SWIGLU && sw) {
      const int c = col0 + 64 * static_cast<int>(rank);
      tma_load_3d_pair(sb, &tmB1, c, kb * kBK, seg, fb);
      tma_load_3d_pair(sb + kBoxBytes, &tmB3, c, kb * kBK, seg, fb);
    } else if (PAIR) {
      const CUtensorMap* mb = (SWIGLU && rank == 1) ? &tmB3 : &tmB1;
      const int c = SWIGLU ? col0 : col0 + static_cast<int>(rank) * 128;
      tma_load_3d_pair(sb, mb, c, kb * kBK, seg, fb);
      tma_load_3d_pair(sb + kBoxBytes, mb, c + 64, kb * kBK, seg, fb);
    } else if (SWIGLU) {
      tma_load_3d(sb + 0 * kBoxBytes, &tmB1, col0, kb * kBK, seg, fb);
      tma_load_3d(sb + 1 * kBoxBytes, &tmB1, col0 + 64, kb * kBK, seg, fb);
      tma_load_3d(sb + 2 * kBoxBytes, &tmB3, col0, kb * kBK, seg, fb);
      tma_load_3d(sb + 3 * kBoxBytes, &tmB3, col0 + 64, kb * kBK, seg, fb);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        tma_load_3d(sb + j * kBoxBytes, &tmB1, col0 + 64 * j, kb * kBK, seg, fb);
    }
  };
  if ((warp == 0 && (GATHER || lane == 0)) || (GATHER && warp >= 2 + kEpiWarps)) {
    // ---------------- producer ----------------
    int stage = 0;
    uint32_t phase = 0;
    int issued[kStages];
    uint32_t issued_phase[kStages];
    for (int s = 0; s < kStages; ++s) issued[s] = 0, issued_phase[s] = 0;
    bool ok = true;
    if constexpr (GATHER) {
      constexpr int kDepth = kStages - 1;  // k-blocks whose rows may still be in flight
      constexpr int kRowsPerLane = kBM / (4 * kCopyWarps);
      const int cw = warp == 0 ? 0 : warp - (1 + kEpiWarps);  // copy warp 0..3
      const int rbase = 32 * cw;                                // its 32 rows of the tile
      const int rsub = lane >> 3, ch = lane & 7;
      const int lim = min(ctrl->seg_row[S], rows_max);  // rows that have a token
      int pend = 0, pend_stage = 0;  // k-blocks copied but not yet announced; the oldest
      auto announce = [&]() {  // the oldest pending k-block's rows have landed
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          const uint32_t fb = smem_u32(&ctrl->full[pend_stage]);
          if (PAIR) mbar_arrive_cluster(map_to_rank(fb, 0));
          else mbar_arrive(fb);
        }
        pend_stage = pend_stage + 1 == kStages ? 0 : pend_stage + 1;
        --pend;
      };
      for (int tile = unit; ok && tile < total; tile += n_units) {
        int seg, row0, row_end, col0;
        decode(tile, seg, row0, row_end, col0);
        const int arow = row0 + static_cast<int>(rank) * kBM;
        int tok[kRowsPerLane];  // source row of x, -1: zero row
        bool bad = false;
#pragma unroll
        for (int i = 0; i < kRowsPerLane; ++i) {
          const int r = arow + rbase + 4 * i + rsub;
          int t = -1;
          if (r < lim) {
            t = row_src[r];
            if (t < 0 || t >= x_rows) {
              bad = true;
              t = -1;
            }
          }
          tok[i] = t;
        }
        if (bad) record_status(status, kErrDeviceBounds);
        for (int kb = 0; kb < num_kb; ++kb) {
          int w = 1;
          if (lane == 0)
            w = mbar_wait_suspend(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs);
          if (!__shfl_sync(0xffffffffu, w, 0)) {
            ok = false;
            break;
          }
          const uint32_t sa = stage0 + stage * G::kStageBytes;
          if (cw == 0 && lane == 0) {
            const uint32_t fb_local = smem_u32(&ctrl->full[stage]);
            if (rank == 0) mbar_expect_tx(fb_local, G::kTxBytesB);
            issued[stage] = 1;
            issued_phase[stage] = phase;
            load_b(sa + kABytes, PAIR ? map_to_rank(fb_local, 0) : fb_local, seg, col0, kb, false);
          }
          const __nv_bfloat16* xk = xg + kb * kBK + ch * 8;
#pragma unroll
          for (int i = 0; i < kRowsPerLane; ++i) {
            const int r = rbase + 4 * i + rsub;
            const int t = tok[i];
            cp_async16(sa + r * 128 + ((ch ^ (r & 7)) << 4),
                       xk + static_cast<size_t>(t < 0 ? 0 : t) * K, t < 0 ? 0u : 16u);
          }
          cp_async_commit();
          if (++pend == kDepth) {
            cp_async_wait<kDepth - 1>();
            announce();
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      cp_async_wait_all();  // every copy lands before its k-block is announced
      while (pend > 0) announce();
    } else {
    for (int tile = unit; ok && tile < total; tile += n_units) {
      int seg, row0, row_end, col0, nsw;
      decode(tile, seg, row0, row_end, col0);
      const bool sw = transposed(row0, row_end, nsw);
      // a transposed tile's rows are the B operand, split N/2 : N/2 over the pair
      const int arow = row0 + static_cast<int>(rank) * (sw ? nsw / 2 : kBM);
      for (int kb = 0; kb < num_kb; ++kb) {
        const uint32_t fb_local = smem_u32(&ctrl->full[stage]);
        if (!mbar_wait_suspend(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        // in a pair every copy counts on CTA 0's barrier, which expects both
        const uint32_t fb = PAIR ? map_to_rank(fb_local, 0) : fb_local;
        if (rank == 0) mbar_expect_tx(fb_local, G::kTxBytes);
        issued[stage] = 1;
        issued_phase[stage] = phase;
        if (!(kb == withhold_kb && tile == 0)) {
          // (failure-detection self-test: the withheld k-block is announced
          // but never loaded, so the MMA issuer's bounded wait expires)
          const uint32_t sa = stage0 + stage * G::kStageBytes;
          if (PAIR) tma_load_2d_pair(sa, &tmA, kb * kKE, arow, fb);
          else tma_load_2d(sa, &tmA, kb * kKE, arow, fb);
          load_b(sa + kABytes, fb, seg, col0, kb, sw);
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    }
    if (!ok && lane == 0) {  // copies in flight land before the CTA (or its pair) can exit (bounded)
      if (rank == 0) {
        for (int s = 0; s < kStages; ++s) {
          if (!issued[s]) continue;
          const unsigned long long t0 = global_ns();
          while (!mbar_try(smem_u32(&ctrl->full[s]), issued_phase[s]))
            if (global_ns() - t0 > kWaitLimitNs / 10) break;
        }
      } else {  // CTA 1 cannot observe CTA 0's barrier: give its copies 2 ms
        const unsigned long long t0 = global_ns();
        while (global_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer ----------------
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true;
    for (int tile = unit; ok && tile < total; tile += n_units, ++local) {
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      // the accumulator is free once every epilogue warp (of both CTAs) is done
      if (!mbar_wait_cluster(smem_u32(&ctrl->tempty[buf]), (use & 1u) ^ 1u, abort_flag,
                             kWaitLimitNs)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kBN);
      int seg, row0, row_end, col0, nsw;
      decode(tile, seg, row0, row_end, col0);
      const bool sw = transposed(row0, row_end, nsw);
      const uint32_t idesc = sw ? swap_idesc(nsw) : kIdesc;
      for (int kb = 0; kb < num_kb; ++kb) {
        // (row gather in a pair: CTA 1's rows are released at cluster scope)
        const bool got =
            (GATHER && PAIR)
                ? mbar_wait_cluster(smem_u32(&ctrl->full[stage]), phase, abort_flag, kWaitLimitNs)
                : mbar_wait(smem_u32(&ctrl->full[stage]), phase, abort_flag, kWaitLimitNs);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = stage0 + stage * G::kStageBytes;
        const uint32_t sb = sa + kABytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // 32 bytes of k per MMA
          // token rows (K-major) and weight columns; a transposed tile swaps them
          const uint64_t rd = kmajor_desc(sa, kk);
          const uint64_t wd = FP8 ? kmajor_desc(sb, kk) : mnmajor_desc(sb, kk, kBoxBytes);
          const uint64_t ad = sw ? wd : rd, bd = sw ? rd : wd;
          const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
          if (FP8) {
            if (PAIR) tc_mma_pair_f8(d_tmem, ad, bd, idesc, acc);
            else tc_mma_f8(d_tmem, ad, bd, idesc, acc);
          } else {
            if (PAIR) tc_mma_pair(d_tmem, ad, bd, idesc, acc);
            else tc_mma(d_tmem, ad, bd, idesc, acc);
          }
        }
        if (PAIR) tc_commit_pair_mc(smem_u32(&ctrl->empty[stage]), 0x3);
        else tc_commit(smem_u32(&ctrl->empty[stage]));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (PAIR) tc_commit_pair_mc(smem_u32(&ctrl->tfull[buf]), 0x3);
      else tc_commit(smem_u32(&ctrl->tfull[buf]));
    }
    // every MMA issued so far completes before this arrives
    if (PAIR) tc_commit_pair(smem_u32(&ctrl->drain));
    else tc_commit(smem_u32(&ctrl->drain));
    const unsigned long long t0 = global_ns();
    while (!mbar_try(smem_u32(&ctrl->drain), 0u))
      if (global_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        break;
      }
  } else if (warp >= 2 && warp < 2 + kEpiWarps) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const uint32_t tempty0 = PAIR ? map_to_rank(smem_u32(&ctrl->tempty[0]), 0) : smem_u32(&ctrl->tempty[0]);
    int local = 0;
    int xuse = 0;  // exchange rounds so far (transposed SwiGLU tiles)
    for (int tile = unit; tile < total; tile += n_units, ++local) {
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_suspend(smem_u32(&ctrl->tfull[buf]), use & 1u, abort_flag, kWaitLimitNs);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      int seg, row0, row_end, col0, nsw;
      decode(tile, seg, row0, row_end, col0);
      const uint32_t taddr_t =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * kBN);
      if (transposed(row0, row_end, nsw)) {
        // TMEM lane = output column, TMEM column = token row row0 + column
        const int lim = min(min(row_end, rows_max), row0 + G::kTileRows);
        const int ntok = lim - row0;
        if (SWIGLU) {
          // lanes 0-63: W1 (gate) columns col0 + 64 * rank ..; lanes 64-127:
          // W3 (up) of the same columns. Warp q and warp q ^ 2 hold gate and
          // up of 32 columns; per 32-token chunk each keeps 16 tokens and
          // passes the other 16 to its partner.
          const int grp = q & 1;
          const bool gate = q < 2;
          const int col = col0 + 64 * static_cast<int>(rank) + 32 * grp + lane;
          const int keep0 = gate ? 0 : 16;  // tokens of the chunk this warp stores
          for (int c0 = 0; c0 < ntok; c0 += 32) {
            uint32_t a[32];
            tc_ld32(taddr_t + c0, a);
            tc_wait_ld();
            const int b = xuse & 1;
            const uint32_t par = static_cast<uint32_t>(xuse >> 1) & 1u;
            ++xuse;
            float* xb = xchg + b * kXchgFloats + grp * 1024;
            float* put = xb + (gate ? 0 : 512);
            const float* take = xb + (gate ? 512 : 0);
            float mine[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float lo = __uint_as_float(a[i]), hi = __uint_as_float(a[16 + i]);
              put[i * 32 + lane] = gate ? hi : lo;
              mine[i] = gate ? lo : hi;
            }
            mbar_arrive(smem_u32(&ctrl->xchg[b]));
            const int got = mbar_wait(smem_u32(&ctrl->xchg[b]), par, abort_flag, kWaitLimitNs);
            if (!__all_sync(0xffffffffu, got)) {
              ok = 0;
              break;
            }
            float h[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float other = take[i * 32 + lane];
              h[i] = gate ? silu_fast(mine[i]) * other : silu_fast(other) * mine[i];
            }
            store_transposed<16>(h, row0 + c0 + keep0, col, lim, n_out, out, lane);
          }
        } else {
          const int col = col0 + 128 * static_cast<int>(rank) + 32 * q + lane;
          for (int c0 = 0; c0 < ntok; c0 += 32) {
            uint32_t a[32];
            tc_ld32(taddr_t + c0, a);
            tc_wait_ld();
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(a[i]);
            store_transposed<32>(v, row0 + c0, col, lim, n_out, out, lane);
          }
        }
        if (!ok) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          const uint32_t te = tempty0 + static_cast<uint32_t>(buf * sizeof(unsigned long long));
          if (PAIR) mbar_arrive_cluster(te);
          else mbar_arrive(te);
        }
        continue;
      }
      const int row = row0 + static_cast<int>(rank) * kBM + q * 32 + lane;
      const bool valid = row >= 0 && row < row_end && row < rows_max;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * kBN);
      __nv_bfloat16* orow = out + static_cast<size_t>(row) * n_out;
      // FP8: the row's scale times each column's scale multiplies the sum of
      // the code products
      const float sa = (FP8 && valid) ? a_scale[row] : 1.f;
      const float* sc1 = FP8 ? b1_scale + static_cast<size_t>(seg) * n_out + col0 : nullptr;
      const float* sc3 = (FP8 && SWIGLU) ? b3_scale + static_cast<size_t>(seg) * n_out + col0 : nullptr;
      if (SWIGLU) {
#pragma unroll 1
        for (int c = 0; c < kBN / 2; c += 32) {
          uint32_t a[32], g[32];
          tc_ld32(taddr + c, a);
          tc_ld32(taddr + kBN / 2 + c, g);
          tc_wait_ld();
          if (valid && col0 + c < n_out) {
            if (FP8) {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                a[i] = __float_as_uint(__uint_as_float(a[i]) * sa * __ldg(sc1 + c + i));
                g[i] = __float_as_uint(__uint_as_float(g[i]) * sa * __ldg(sc3 + c + i));
              }
            }
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
            if (FP8) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                a[i] = __float_as_uint(__uint_as_float(a[i]) * sa * __ldg(sc1 + c + i));
            }
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
      __syncwarp();
      if (lane == 0) {
        const uint32_t te = tempty0 + static_cast<uint32_t>(buf * sizeof(unsigned long long));
        if (PAIR) mbar_arrive_cluster(te);
        else mbar_arrive(te);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) {  // CTA 0's MMAs into this CTA's TMEM and shared memory are done
    __syncwarp();
    cluster_sync();
  }
  tc_fence_after();
  if (threadIdx.x == 0 && *abort_flag) record_status(status, kErrDeviceTimeout);
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc<PAIR>(tmem_base);
  }
}

// Clusters of 2 of the kernel that will be launched (its shared-memory
// attribute already set) that can be resident at once (0: pairs unavailable).
template <bool SWIGLU, bool GATHER, bool FP8>
int pair_slots(int dev) {
  static int cached[64] = {};
  static bool done[64] = {};
  if (dev < 0 || dev >= 64) return 0;
  if (done[dev]) return cached[dev];
  int n = 0;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(device_sm_count() & ~1));
  cfg.blockDim = dim3(threads_of<GATHER>());
  cfg.dynamicSmemBytes = smem_bytes<true>();
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_tc_kernel<SWIGLU, true, GATHER, FP8>, &cfg) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  cached[dev] = n;
  done[dev] = true;
  return n;
}

template <bool SWIGLU, bool PAIR, bool GATHER, bool FP8>
cudaError_t set_smem_attr(int dev) {
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (attr_set[dev]) return cudaSuccess;
  const cudaError_t err = cudaFuncSetAttribute(grouped_gemm_tc_kernel<SWIGLU, PAIR, GATHER, FP8>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               smem_bytes<PAIR>());
  if (err == cudaSuccess) attr_set[dev] = true;
  return err;
}

template <bool SWIGLU, bool GATHER, bool FP8 = false>
cudaError_t launch_gemm(const CUtensorMap& mA, const CUtensorMap& mB1, const CUtensorMap& mB3,
                        const int32_t* offsets, int S, int64_t rows_max, int K, int n_out,
                        __nv_bfloat16* o, int32_t* status, cudaStream_t s, int withhold_kb,
                        int max_sms, const __nv_bfloat16* xg, const int32_t* row_src,
                        int x_rows, const float* a_scale = nullptr,
                        const float* b1_scale = nullptr, const float* b3_scale = nullptr) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if ((err = set_smem_attr<SWIGLU, true, GATHER, FP8>(dev)) != cudaSuccess) return err;
  if ((err = set_smem_attr<SWIGLU, false, GATHER, FP8>(dev)) != cudaSuccess) return err;
  // Pairs pay off once segments average a 256-row tile; below that (decode
  // batches) half of every pair tile would be padding. The row-gather form
  // runs one CTA per tile: its pairs wait on two CTAs' copies per k-block and
  // measured about twice as slow.
  const char* env = getenv("MOE_GEMM_CTA_PAIRS");
  const bool want_pairs = env ? env[0] != '0' : (!GATHER && rows_max >= 2LL * kBM * S);
  int sms = device_sm_count();
  if (max_sms > 0 && max_sms < sms) sms = max_sms;  // confined to a slice of the GPU
  int slots = want_pairs ? pair_slots<SWIGLU, GATHER, FP8>(dev) : 0;
  if (slots > sms / 2) slots = sms / 2;
  const bool pair = slots > 0;
  const int tile_rows = pair ? 2 * kBM : kBM;
  const int tile_n = SWIGLU ? kBN / 2 : kBN;
  const long long n_tiles = (n_out + tile_n - 1) / tile_n;
  const long long m_tiles_max = (rows_max + tile_rows - 1) / tile_rows + S;
  long long units = n_tiles * m_tiles_max;
  const long long cap = pair ? slots : sms;
  if (units > cap) units = cap;
  const int rmax = rows_max > 0x7fffffff ? 0x7fffffff : static_cast<int>(rows_max);
  // pair tiles run transposed (see transposed()) unless MOE_GEMM_SWAP_TAILS=0
  const char* sw_env = getenv("MOE_GEMM_SWAP_TAILS");
  const int swap_tails = sw_env ? (sw_env[0] != '0') : 1;

  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = pair ? 2 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pair ? 2 * units : units));
  cfg.blockDim = dim3(threads_of<GATHER>());
  cfg.dynamicSmemBytes = pair ? smem_bytes<true>() : smem_bytes<false>();
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pair ? 2 : 1;
  if (pair)
    return cudaLaunchKernelEx(&cfg, grouped_gemm_tc_kernel<SWIGLU, true, GATHER, FP8>, mA, mB1,
                              mB3, offsets, S, K, n_out, rmax, o, status, withhold_kb, xg, row_src,
                              x_rows, a_scale, b1_scale, b3_scale, swap_tails);
  return cudaLaunchKernelEx(&cfg, grouped_gemm_tc_kernel<SWIGLU, false, GATHER, FP8>, mA, mB1,
                            mB3, offsets, S, K, n_out, rmax, o, status, withhold_kb, xg, row_src,
                            x_rows, a_scale, b1_scale, b3_scale, swap_tails);
}

}  // namespace

cudaError_t launch_grouped_gemm_tc_bf16(const void* A, const int32_t* offsets, int S,
                                        int64_t rows_max, int K, int n_out, const void* B1,
                                        const void* B3, void* out, bool swiglu,
                                        int32_t* status, cudaStream_t s, int withhold_kb,
                                        int max_sms, const int32_t* row_src, int a_rows) {
  if (S == 0 || rows_max == 0) return cudaSuccess;
  if (S > kMaxSegments) return cudaErrorInvalidValue;
  if (row_src && (!swiglu || a_rows < 0 || K % kBK)) return cudaErrorInvalidValue;
  CUtensorMap mA, mB1, mB3;
  if (!make_tmap_3d_bf16(&mB1, B1, S, K, n_out, 64, kBK)) return cudaErrorInvalidValue;
  if (row_src) {
    mA = mB1;  // not read: A rows are gathered
  } else if (!make_tmap_2d_bf16(&mA, A, static_cast<uint64_t>(rows_max), static_cast<uint64_t>(K),
                                64, kBM)) {
    return cudaErrorInvalidValue;
  }
  if (swiglu) {
    if (!make_tmap_3d_bf16(&mB3, B3, S, K, n_out, 64, kBK)) return cudaErrorInvalidValue;
  } else {
    mB3 = mB1;
  }
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  const __nv_bfloat16* xg = static_cast<const __nv_bfloat16*>(A);
  if (swiglu && row_src)
    return launch_gemm<true, true>(mA, mB1, mB3, offsets, S, rows_max, K, n_out, o, status, s, -1,
                                   max_sms, xg, row_src, a_rows);
  if (swiglu)
    return launch_gemm<true, false>(mA, mB1, mB3, offsets, S, rows_max, K, n_out, o, status, s,
                                    withhold_kb, max_sms, nullptr, nullptr, 0);
  return launch_gemm<false, false>(mA, mB1, mB3, offsets, S, rows_max, K, n_out, o, status, s,
                                   withhold_kb, max_sms, nullptr, nullptr, 0);
}

cudaError_t launch_grouped_gemm_tc_fp8(const void* A, const float* a_scale,
                                       const int32_t* offsets, int S, int64_t rows_max, int K,
                                       int n_out, const void* B1, const float* sc1,
                                       const void* B3, const float* sc3, void* out, bool swiglu,
                                       int32_t* status, cudaStream_t s) {
  if (S == 0 || rows_max == 0) return cudaSuccess;
  if (S > kMaxSegments || K % 128 || n_out % 128) return cudaErrorInvalidValue;
  if (!a_scale || !sc1 || (swiglu && (!B3 || !sc3))) return cudaErrorInvalidValue;
  CUtensorMap mA, mB1, mB3;
  // A: [rows_max, K] bytes in 128 x 128 boxes; B: [S, n_out, K] bytes, boxes
  // of 128 k x 128 columns
  if (!make_tmap_2d_u8(&mA, A, static_cast<uint64_t>(rows_max), static_cast<uint64_t>(K), 128,
                       kBM))
    return cudaErrorInvalidValue;
  if (!make_tmap_3d_u8(&mB1, B1, S, n_out, K, 128, 128)) return cudaErrorInvalidValue;
  if (swiglu) {
    if (!make_tmap_3d_u8(&mB3, B3, S, n_out, K, 128, 128)) return cudaErrorInvalidValue;
  } else {
    mB3 = mB1;
  }
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  if (swiglu)
    return launch_gemm<true, false, true>(mA, mB1, mB3, offsets, S, rows_max, K, n_out, o, status,
                                          s, -1, 0, nullptr, nullptr, 0, a_scale, sc1, sc3);
  return launch_gemm<false, false, true>(mA, mB1, mB3, offsets, S, rows_max, K, n_out, o, status,
                                         s, -1, 0, nullptr, nullptr, 0, a_scale, sc1, nullptr);
}

}  // namespace moe
