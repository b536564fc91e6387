// Internal launch interface between the C ABI (moe_api.cu) and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

// Launches kernel<<<grid, block, smem, s>>>(args...) with programmatic
// dependent launch allowed: the kernel may be scheduled while the previous
// kernel on the stream finishes, and every kernel of this library waits
// (griddepcontrol.wait, pdl_wait) before it touches global memory, so the
// overlap covers only launch latency and set-up.
template <typename... P, typename... A>
cudaError_t launch_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       A&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
}

// Router logits L = x W_r + b (fp32 out).
cudaError_t launch_router_logits(int dtype, const void* x, const void* W_r, const float* bias,
                                 float* L, int T, int d, int N, cudaStream_t s);

// The first kCtrlBytes of every workspace: the sticky status word (it must
// start at zero: the workspace is zeroed, or moe_clear_device_status is
// called, before first use); the rest is reserved.
constexpr size_t kCtrlBytes = 1024;
constexpr int kRouteTile = 128;          // tokens per router tile (tensor-core M)

// Per-token routing (route_token.cuh) inputs and outputs.
struct RouteArgs {
  const float* logits = nullptr;   // [T, N] input of the routing kernel (route.cu)
  const float* bias = nullptr;     // [N], added to the logits by the tensor-core router
  float* logits_out = nullptr;     // [T, N] nullable (tensor-core router)
  float* scores = nullptr;         // [T, N] nullable
  int32_t* cand_idx = nullptr;     // [T, kc] (unused under expert choice)
  float* cand_gate = nullptr;      // [T, kc]
  const int32_t* home_group = nullptr;
  unsigned long long* colsum = nullptr;  // [rows, N] fixed-point column sums of p, nullable
  int T = 0, N = 0, k = 0, m = 0, group_size = 1, renorm = 0, ec = 0;
};

// Router logits on tcgen05 (bf16, d % 64 == 0, N % 8 == 0, N <= 256): one
// thread-block cluster of `cluster` CTAs per 128-token tile splits d; the
// partial logits meet in distributed shared memory and each CTA routes
// 128 / cluster of the tile's tokens. Column sums: one row per CTA.
struct RouterPlan {
  int cluster = 1;  // CTAs per tile (a power of two dividing d / 64, <= 8)
  int m_tiles = 0;
  int colsum_rows = 0;
};
bool router_tc_supported(int dtype, int d, int N);
RouterPlan router_plan(int T, int d, int N);
cudaError_t launch_router_tc(const void* x, const void* W_r, int d, const RouterPlan& plan,
                             const RouteArgs& ra, int32_t* status, cudaStream_t s);

// Per-token scores, candidates and gates from fp32 logits [T, N] (ra.logits),
// one warp segment per token; colsum rows: route_tokens_colsum_rows(T, N).
int route_tokens_colsum_rows(int T, int N);
cudaError_t launch_route_tokens(const RouteArgs& ra, cudaStream_t s);


// Load statistics. colsum: [rows, N] fixed-point column sums of the scores
// (the routing kernels with ra.colsum, or launch_colsum with
// colsum_kernel_rows(T) rows).
struct StatsArgs {
  const unsigned long long* colsum = nullptr;
  int rows = 0;             // rows of colsum
  double* stats = nullptr;  // [MOE_STATS_LEN]
};
size_t colsum_bytes(int T, int N);  // enough rows for either router
int colsum_kernel_rows(int T);
cudaError_t launch_colsum(const float* scores, int T, int N, unsigned long long* colsum,
                          cudaStream_t s);
cudaError_t launch_stats_final(const int32_t* demand, const int32_t* kept,
                               const unsigned long long* colsum, int rows, int T, int N,
                               double* stats, cudaStream_t s);

// Per-expert selection (token choice: rank only; capacity drop: top-cap by
// gate; expert choice: top-cap tokens by score; group_size > 0: the experts of
// each group of group_size share the capacity cap).
cudaError_t launch_select(const int32_t* cand_idx, const float* cand_gate, int T, int kc, int N,
                          int expert_choice, int cap, int group_size, int32_t* slot, uint8_t* keep,
                          int32_t* demand, int32_t* kept, cudaStream_t s);
int select_max_tokens();

// Offsets, row maps, token rows, per-token coverage (nullable) and the
// gather of x into xp; with st.stats set, one extra block writes the load
// statistics from demand, kept and the column sums.
cudaError_t launch_dispatch(int dtype, const void* x, const int32_t* cand_idx,
                            const float* cand_gate, const int32_t* slot, const int32_t* kept,
                            int T, int d, int N, int kc, int expert_choice, int64_t rows_max,
                            int32_t* expert_offsets, int32_t* row_token, float* row_gate,
                            int32_t* tok_rows, int32_t* coverage, void* xp,
                            const int32_t* demand, const StatsArgs& st, cudaStream_t s);

// Grouped GEMM on e4m3 operands (tcgen05 kind::f8f6f4): A [rows_max, K]
// e4m3 bytes with one fp32 scale per row (a_scale [rows_max]); B1, B3
// [S, n_out, K] e4m3 bytes, K-major, with one fp32 scale per output column
// (sc1, sc3 [S, n_out]). The products of the codes are summed in fp32 and
// scaled in the epilogue: out = silu(sa*sc1*(A B1)) * (sa*sc3*(A B3)) or
// sa*sc1*(A B1); out bf16. K and n_out multiples of 128.
cudaError_t launch_grouped_gemm_tc_fp8(const void* A, const float* a_scale,
                                       const int32_t* offsets, int S, int64_t rows_max, int K,
                                       int n_out, const void* B1, const float* sc1,
                                       const void* B3, const float* sc3, void* out, bool swiglu,
                                       int32_t* status, cudaStream_t s);

// Rows r < offsets[S] of the bf16 matrix X [rows_max, K] to e4m3 with one
// fp32 scale per row: scale = max|X[r]| / 448 (1 for a zero row), Q[r][j] =
// nearest e4m3 of X[r][j] / scale (ties to even, saturating). K % 8 == 0.
cudaError_t launch_quantize_rows_e4m3(const void* X, const int32_t* offsets, int S,
                                      int64_t rows_max, int K, uint8_t* Q, float* scale,
                                      cudaStream_t s);

// Grouped GEMMs. SwiGLU variant: out = silu(A B1) * (A B3); plain: out = A B1.
cudaError_t launch_grouped_gemm_simt_f32(const float* A, const int32_t* offsets, int S,
                                         int64_t rows_max, int K, int n_out, const float* B1,
                                         const float* B3, float* out, bool swiglu,
                                         cudaStream_t s);
// withhold_kb >= 0 (self-test only): the first tile announces but never
// loads its k-block withhold_kb, so a bounded wait expires. max_sms > 0 caps
// the persistent grid at that many SMs. row_src (SwiGLU only): A is the
// [a_rows, K] token matrix and row r of the product reads A[row_src[r]]
// (rows at or past offsets[S] read zeros; an index outside [0, a_rows) reads
// zeros and records MOE_ERR_DEVICE_BOUNDS).
cudaError_t launch_grouped_gemm_tc_bf16(const void* A, const int32_t* offsets, int S,
                                        int64_t rows_max, int K, int n_out, const void* B1,
                                        const void* B3, void* out, bool swiglu,
                                        int32_t* status, cudaStream_t s, int withhold_kb = -1,
                                        int max_sms = 0, const int32_t* row_src = nullptr,
                                        int a_rows = 0);

// y[t] = sum_r gate_r op[r] (+ shared[t]).
cudaError_t launch_combine(int dtype, const void* op, const float* row_gate,
                           const int32_t* tok_rows, const void* shared_out, void* y, int T,
                           int d, int kc, int64_t rows_max, cudaStream_t s);

int device_sm_count();

// bf16 TMA maps with 128-byte swizzle. 2-D: [rows, cols] row-major, box
// box_cols x box_rows. 3-D: [S, K, n] row-major, box box_n x box_k x 1.
bool make_tmap_2d_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                       uint32_t box_cols, uint32_t box_rows);
bool make_tmap_3d_bf16(CUtensorMap* m, const void* ptr, uint64_t S, uint64_t K, uint64_t n,
                       uint32_t box_n, uint32_t box_k);
// Byte tensors (e4m3), 128-byte swizzle. 2-D: [rows, cols] row-major, box
// box_cols x box_rows. 3-D: [S, K, n] row-major, box box_n x box_k x 1.
bool make_tmap_2d_u8(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                     uint32_t box_cols, uint32_t box_rows);
bool make_tmap_3d_u8(CUtensorMap* m, const void* ptr, uint64_t S, uint64_t K, uint64_t n,
                     uint32_t box_n, uint32_t box_k);

}  // namespace moe
