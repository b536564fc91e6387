// Internal launch interface between the C ABI (moe_api.cu) and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

// Router logits L = x W_r + b (fp32 out).
cudaError_t launch_router_logits(int dtype, const void* x, const void* W_r, const float* bias,
                                 float* L, int T, int d, int N, cudaStream_t s);

// Router logits on tcgen05 (bf16, N % 8 == 0): split-K partials
// partial[split][T][N] fp32, summed by launch_route_tokens.
struct RouterSplit {
  int splits = 1;
  int kb_per_split = 1;
};
bool router_tc_supported(int dtype, int d, int N);
RouterSplit router_split_plan(int T, int d, int N);
cudaError_t launch_router_logits_tc(const void* x, const void* W_r, int T, int d, int N,
                                    const RouterSplit& plan, float* partial, int32_t* status,
                                    cudaStream_t s);

// Per-token scores, candidates and gates. The logits of token t are
// sum_{s < nsplit} partial[s][t][:] (+ bias), summed in ascending s; with
// logits_out they are also stored there.
cudaError_t launch_route_tokens(const float* partial, int nsplit, const float* bias,
                                float* logits_out, float* scores, int32_t* cand_idx,
                                float* cand_gate, const int32_t* home_group, int T, int N, int k,
                                int m, int group_size, int renorm, int expert_choice,
                                cudaStream_t s);

// Per-expert selection (token choice: rank only; capacity drop: top-cap by
// gate; expert choice: top-cap tokens by score).
cudaError_t launch_select(const int32_t* cand_idx, const float* cand_gate, int T, int kc, int N,
                          int expert_choice, int cap, int32_t* slot, uint8_t* keep,
                          int32_t* demand, int32_t* kept, cudaStream_t s);
int select_max_tokens();

// Offsets, row maps, token rows and the gather of x into xp.
cudaError_t launch_dispatch(int dtype, const void* x, const int32_t* cand_idx,
                            const float* cand_gate, const int32_t* slot, const int32_t* kept,
                            int T, int d, int N, int kc, int expert_choice, int64_t rows_max,
                            int32_t* expert_offsets, int32_t* row_token, float* row_gate,
                            int32_t* tok_rows, void* xp, cudaStream_t s);

// Grouped GEMMs. SwiGLU variant: out = silu(A B1) * (A B3); plain: out = A B1.
cudaError_t launch_grouped_gemm_simt_f32(const float* A, const int32_t* offsets, int S,
                                         int64_t rows_max, int K, int n_out, const float* B1,
                                         const float* B3, float* out, bool swiglu,
                                         cudaStream_t s);
cudaError_t launch_grouped_gemm_tc_bf16(const void* A, const int32_t* offsets, int S,
                                        int64_t rows_max, int K, int n_out, const void* B1,
                                        const void* B3, void* out, bool swiglu,
                                        int32_t* status, cudaStream_t s);

// y[t] = sum_r gate_r op[r] (+ shared[t]).
cudaError_t launch_combine(int dtype, const void* op, const float* row_gate,
                           const int32_t* tok_rows, const void* shared_out, void* y, int T,
                           int d, int kc, int64_t rows_max, cudaStream_t s);

// Load statistics. partial: >= stats_partial_doubles(T, N) doubles of scratch.
size_t stats_partial_doubles(int T, int N);
cudaError_t launch_stats(const int32_t* demand, const int32_t* kept, const float* scores, int T,
                         int N, double* partial, double* stats, cudaStream_t s);

int device_sm_count();

// bf16 TMA maps with 128-byte swizzle. 2-D: [rows, cols] row-major, box
// box_cols x box_rows. 3-D: [S, K, n] row-major, box box_n x box_k x 1.
bool make_tmap_2d_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                       uint32_t box_cols, uint32_t box_rows);
bool make_tmap_3d_bf16(CUtensorMap* m, const void* ptr, uint64_t S, uint64_t K, uint64_t n,
                       uint32_t box_n, uint32_t box_k);

}  // namespace moe
