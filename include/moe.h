/*
 * moe.h - C ABI of the B300 sparse Mixture-of-Experts FFN layer library.
 *
 * One MoE FFN layer forward pass, y = sum_i G(x)_i * E_i(x)
 * ("Understanding Mixture of Experts", section "How MoE differs from the
 * Transformer", layer equation), with SwiGLU experts E(x) = (silu(x W1) *
 * (x W3)) W2 and three routing modes:
 *   - token choice: each token takes its top-k experts by router score
 *     (same page, section "Expert and Router", TopK(G(x), k));
 *   - expert choice: each expert takes its top c = k*T/N tokens
 *     ("MoE vs MoT: routing and inference cost", section "Mixture of Tokens");
 *   - capacity-aware token drop: an expert over capacity C = gamma * N_bar
 *     drops the candidates with the lowest gating score, optionally with m
 *     extra local candidates per token ("Capacity-Aware Inference: Mitigating
 *     the Straggler Effect in MoE", section 2, (1) Token Drop and (2) Expanded
 *     Drop);
 *   - device-level capacity-aware drop: the experts of a device (a group of
 *     group_size consecutive experts) share one capacity, the sum of theirs,
 *     so an expert over its own share keeps its tokens while its device has
 *     room (same page, section 2, (3) Device-Level Capacity-Aware Inference).
 *
 * Conventions for every call below:
 *   - Pointers to tensors are DEVICE pointers unless a comment says host.
 *     The caller allocates and owns every buffer, including the workspace;
 *     the library never allocates, frees or synchronises inside these calls
 *     (moe_get_device_status is the one call that synchronises a stream).
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream. All work is enqueued on it asynchronously, in call order.
 *   - Tensors are dense row-major. Activations, weights and y have the
 *     config's dtype (MOE_BF16 or MOE_F32); logits, scores and gates are fp32;
 *     indices and counts are int32. Accumulation is always fp32.
 *   - Base pointers of activation/weight tensors must be 16-byte aligned.
 *     bf16 layers need d and f to be multiples of 64; fp32 layers need d to
 *     be a multiple of 8.
 *   - Return value: MOE_OK or a negative MOE_ERR_* code. Argument checks run
 *     on the host before anything is enqueued; on failure no output is touched.
 *     Conditions a kernel detects (a bounded wait that expired) are recorded in
 *     a sticky status word in the workspace, read by moe_get_device_status.
 *   - Inputs must be finite (no NaN/Inf); non-finite values give undefined
 *     routing.
 *
 * Notation: T tokens, d model width, N routed experts, f expert hidden width,
 * k experts per token, m expanded candidates, kc candidate slots per token
 * (k + m, or N under expert choice), C capacity, P kept (token, expert) pairs,
 * rows_max the upper bound of P that sizes the row buffers (moe_sizes).
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---- */
#define MOE_OK                  0
#define MOE_ERR_NULL           (-1)  /* a required pointer is NULL */
#define MOE_ERR_SHAPE          (-2)  /* a size is out of range or inconsistent */
#define MOE_ERR_ALIGN          (-3)  /* a pointer or row pitch breaks the 16-byte rule */
#define MOE_ERR_WORKSPACE      (-4)  /* workspace smaller than moe_workspace_size */
#define MOE_ERR_UNSUPPORTED    (-5)  /* valid but not implemented (see limits below) */
#define MOE_ERR_LAUNCH         (-6)  /* the CUDA runtime refused a launch */
#define MOE_ERR_DEVICE_TIMEOUT (-7)  /* a kernel's bounded wait expired (sticky, device) */
#define MOE_ERR_DEVICE_BOUNDS  (-8)  /* a kernel saw an index outside its buffer (sticky) */

/* ---- routing modes and dtypes ---- */
#define MOE_TOKEN_CHOICE   0
#define MOE_EXPERT_CHOICE  1
#define MOE_CAPACITY_DROP  2
#define MOE_CAPACITY_DROP_DEVICE 3  /* capacity per device group of group_size experts */

#define MOE_F32  0
#define MOE_BF16 1

/* flags */
#define MOE_LOGITS_GIVEN 1  /* router logits are an input; x and W_router are not read for routing */
#define MOE_FUSE_GATHER  2  /* moe_layer_forward, bf16 experts: the first expert GEMM reads each
                               token row of x through row_token (moe_expert_ffn_gather) and
                               dispatch writes no xp copy; ignored for fp32 or e4m3 experts */

/* Limits: 1 <= N <= 256, 1 <= k <= N, k + m <= 32, expert choice N <= 256,
 * T <= 24576 (per-expert candidate lists are held in shared memory),
 * expanded and device-level drop: group_size divides N. */

typedef struct moe_config {
  int32_t T;          /* tokens in the batch */
  int32_t d;          /* model width */
  int32_t N;          /* routed experts */
  int32_t f;          /* routed expert hidden width */
  int32_t k;          /* experts per token (expert choice: c = floor(k*T/N)) */
  int32_t mode;       /* MOE_TOKEN_CHOICE / MOE_EXPERT_CHOICE / MOE_CAPACITY_DROP /
                         MOE_CAPACITY_DROP_DEVICE */
  double  gamma;      /* capacity factor; C = min(T, floor(gamma * k*T/N)); INFINITY = no limit.
                         MOE_CAPACITY_DROP_DEVICE: a device holds
                         min(T * min(kc, group_size), floor(gamma * k*T/N * group_size)) */
  int32_t m;          /* expanded drop: extra local candidates per token (0 = off) */
  int32_t group_size; /* experts per device group (expanded drop, device-level drop) */
  int32_t renorm;     /* 1: gates divided by their sum over the token's candidates */
  int32_t f_shared;   /* hidden width of the always-on shared expert (0 = none) */
  int32_t dtype;      /* MOE_BF16 or MOE_F32 */
  int32_t flags;      /* MOE_LOGITS_GIVEN | MOE_FUSE_GATHER */
} moe_config;

/* Derived sizes of a config (host values). */
typedef struct moe_sizes_t {
  int32_t kc;          /* candidate slots per token */
  int32_t capacity;    /* C (capacity drop), a device's capacity (device-level drop),
                          c (expert choice) or T (token choice) */
  int64_t rows_max;    /* upper bound of P: row capacity of xp/op/row_token/row_gate */
  size_t  workspace;   /* bytes moe_layer_forward needs */
  size_t  ffn_workspace; /* bytes moe_expert_ffn needs for rows_max rows */
} moe_sizes_t;

/* Number of doubles moe_layer_forward / moe_load_stats write to `stats`. */
#define MOE_STATS_LEN 8
/* stats[0] P kept pairs        stats[1] candidate pairs before selection
 * stats[2] max kept per expert stats[3] mean kept per expert
 * stats[4] max/mean kept (the straggler ratio of "Capacity-Aware Inference", section 1)
 * stats[5] dropped fraction of candidate pairs
 * stats[6] Switch balance term B = sum_i f_i * P_i ("MoE vs MoT", section
 *          "MoE basic structure"), f_i = demand_i / sum(demand), P_i = mean_t p[t,i]
 * stats[7] N * B (1 for a perfectly even router) */

/* Fill `out` for `cfg`. Host only; no CUDA call. Returns MOE_ERR_* if the
 * config is invalid or outside the limits. */
int moe_sizes(const moe_config* cfg, moe_sizes_t* out);

/* Bytes of workspace moe_layer_forward needs (0 if the config is invalid). */
size_t moe_workspace_size(const moe_config* cfg);

/* Every workspace (moe_layer_forward, moe_route, moe_expert_ffn,
 * moe_grouped_gemm) begins with a 1024-byte control block: the sticky status
 * word, then reserved bytes. The control block must be zero before the
 * workspace's first use (allocate it zeroed, or call
 * moe_clear_device_status). Calls that share a workspace must not overlap on
 * the GPU. */
#define MOE_CTRL_BYTES 1024

/* Bytes of workspace moe_route needs (the control block). */
size_t moe_route_workspace_size(const moe_config* cfg);

/* Bytes of workspace moe_expert_ffn needs for `rows_max` rows of hidden width f. */
size_t moe_ffn_workspace_size(int64_t rows_max, int32_t f, int32_t dtype);

/*
 * Router: logits, softmax scores and each token's candidate experts.
 * "Understanding Mixture of Experts", section "Expert and Router": the router
 * decides which experts receive the token and G(x) weights them; TopK(G(x),k).
 *
 *   x        [T, d] dtype       (not read with MOE_LOGITS_GIVEN)
 *   W_router [d, N] dtype       (not read with MOE_LOGITS_GIVEN)
 *   bias     [N] fp32, nullable; added to the logits
 *   logits   [T, N] fp32: output, or input with MOE_LOGITS_GIVEN
 *   scores   [T, N] fp32 nullable: p = softmax over experts of each row,
 *            by the fixed fp32 sequence max / subtract / Cody-Waite exp /
 *            left-to-right sum / correctly rounded divide, so every decision
 *            taken from it is reproducible bit for bit
 *   cand_idx [T, kc] int32: token choice / capacity drop: the top-k experts
 *            by logit, best first, ties to the lower expert; then (m > 0) the
 *            m highest-logit experts of the token's home group not already
 *            chosen; empty slots hold -1. Unused (nullable) under expert choice.
 *   cand_gate[T, kc] fp32: gate of each slot, p or (renorm) p divided by the
 *            left-to-right sum of the token's slot probabilities. Under expert
 *            choice kc = N and cand_gate receives the scores p.
 *   home_group [T] int32 nullable: device group of each token for expanded
 *            drop; NULL = contiguous shards, group floor(t*G/T), G = N/group_size.
 *   ws       >= moe_route_workspace_size(cfg) bytes, 256-byte aligned.
 * bf16 layers with N a multiple of 8 compute the logits on the tcgen05 tensor
 * cores, one thread-block cluster per 128-token tile splitting d; the
 * cluster's fp32 partials are added in k order, then the bias, and the tokens
 * are routed in the same launch. Other shapes use fp32 FMA and a second
 * kernel for the routing. Either way L is fp32-accumulated, not the exact dot
 * product.
 */
int moe_route(const moe_config* cfg, const void* x, const void* W_router, const float* bias,
              float* logits, float* scores, int32_t* cand_idx, float* cand_gate,
              const int32_t* home_group, void* ws, size_t ws_bytes, void* stream);

/*
 * Per-expert selection over the candidates (one thread block per expert).
 * "Capacity-Aware Inference", section 2 (1) Token Drop: expert e keeps at most
 * C of its candidates, those with the highest gate (ties: the lower token),
 * and drops the rest. Under expert choice every token is a candidate of every
 * expert with gate p[t, e] and exactly c = min(T, floor(k*T/N)) are kept
 * ("MoE vs MoT", section "Mixture of Tokens"). Under token choice nothing is
 * dropped and only the ranks below are produced. Under MOE_CAPACITY_DROP_DEVICE
 * ("Capacity-Aware Inference", section 2 (3)) the candidates of the experts of
 * one device group compete for the device's capacity (moe_sizes().capacity):
 * the highest gates are kept, ties to the lower token and then to the lower
 * candidate slot; an expert may keep more than C while the device has room.
 *
 *   cand_idx  [T, kc] int32 (ignored under expert choice)
 *   cand_gate [T, kc] fp32
 *   slot      [T, kc] int32 out: for a kept slot, its rank among expert e's
 *             kept tokens in ascending token order; -1 for a dropped or empty slot
 *   keep      [T, kc] uint8 out, nullable: 1 kept, 0 not
 *   demand    [N] int32 out: candidates per expert before selection (expert
 *             choice: the c tokens the expert takes, since nothing is dropped)
 *   kept      [N] int32 out: pairs per expert after selection
 */
int moe_capacity_drop(const moe_config* cfg, const int32_t* cand_idx, const float* cand_gate,
                      int32_t* slot, uint8_t* keep, int32_t* demand, int32_t* kept, void* stream);

/*
 * Histogram -> prefix sum -> permute: the kept pairs in expert-contiguous row
 * order, and the token rows gathered into it (the dispatch step that the
 * all-to-all of "MoE vs MoT", section "MoE basic structure", performs across
 * devices; here within one GPU).
 *
 *   x              [T, d] dtype
 *   cand_idx, cand_gate, slot   as produced above ([T, kc])
 *   kept           [N] int32
 *   expert_offsets [N + 1] int32 out: exclusive prefix sum of kept; [N] = P
 *   row_token      [rows_max] int32 out: token of each row (rows < P)
 *   row_gate       [rows_max] fp32 out: gate of each row
 *   tok_rows       [T, kc] int32 out: rows of each token in ascending expert
 *                  order (= ascending row), padded with -1
 *   coverage       [T] int32 out, nullable: the number of kept pairs of each
 *                  token. Under expert choice this is how many experts took
 *                  the token: some tokens are taken by several experts and
 *                  some by none ("MoE vs MoT", section "Mixture of Tokens");
 *                  it sums to N * c. Under token choice and drop it is the
 *                  token's surviving candidates.
 *   xp             [rows_max, d] dtype out: xp[r] = x[row_token[r]]
 * Rows inside an expert are in ascending token order. Rows >= P are not written.
 */
int moe_dispatch(const moe_config* cfg, const void* x, const int32_t* cand_idx,
                 const float* cand_gate, const int32_t* slot, const int32_t* kept,
                 int32_t* expert_offsets, int32_t* row_token, float* row_gate,
                 int32_t* tok_rows, int32_t* coverage, void* xp, void* stream);

/*
 * Grouped SwiGLU experts over expert-contiguous rows ("MoE vs MoT", section
 * "MoE basic structure": the FFN is replicated N times; section "measured
 * figures": grouped GEMM for the experts).
 * For every segment s in [0, n_segments), rows r in
 * [offsets[s], offsets[s+1]):  h = silu(xp[r] W1[s]) * (xp[r] W3[s]) stored in
 * dtype, then op[r] = h W2[s] stored in dtype.
 *
 *   d, dtype     from cfg (the other cfg fields are not read)
 *   xp           [rows_max, d] dtype
 *   offsets      [n_segments + 1] int32, device-resident, non-decreasing,
 *                offsets[0] = 0, offsets[n_segments] <= rows_max
 *   f            hidden width of these experts
 *   W1, W3       [n_segments, d, f] dtype;  W2 [n_segments, f, d] dtype
 *   op           [rows_max, d] dtype out (rows >= offsets[n_segments] untouched)
 *   ws           >= moe_ffn_workspace_size(rows_max, f, dtype) bytes (control
 *                block, then the hidden activations)
 * bf16 runs on the tcgen05 tensor cores (fp32 accumulate in tensor memory);
 * fp32 runs on the fp32 FMA pipes. The bf16 GEMMs (here, in moe_grouped_gemm
 * and in moe_layer_forward) run as CTA pairs (thread-block clusters of 2
 * sharing each MMA, 256-row tiles) when rows_max >= 256 * n_segments and the
 * device can co-schedule them, otherwise one CTA per 128-row tile. The
 * environment variable MOE_GEMM_CTA_PAIRS, read at every launch, overrides
 * the choice: "0" one CTA per tile, anything else pairs. In pair form an
 * expert's last tile with fewer than 256 rows is computed transposed (the
 * weight columns as the MMA's 256 rows, the tile's rows as its columns), so
 * it costs its rows instead of a padded tile; the second GEMM (and
 * moe_grouped_gemm) computes every tile that way. The outputs are the same
 * bits. MOE_GEMM_SWAP_TAILS=0, read at every launch, computes every tile
 * untransposed, padding the last ones.
 */
int moe_expert_ffn(const moe_config* cfg, const void* xp, const int32_t* offsets,
                   int32_t n_segments, int64_t rows_max, int32_t f,
                   const void* W1, const void* W3, const void* W2, void* op,
                   void* ws, size_t ws_bytes, void* stream);

/*
 * moe_expert_ffn with the dispatch gather fused into the first GEMM: row r of
 * segment s is computed from x[row_token[r]] instead of xp[r], so the
 * expert-contiguous copy of the token rows is never written or read. Moving
 * token rows is one of the data movements the pages name as the cost of MoE
 * inference ("From personas to MoE 02", section "ugh, bandwidth"); the result
 * equals moe_expert_ffn on xp[r] = x[row_token[r]] bit for bit.
 *
 *   x            [T, d] bf16 (T = cfg->T), 16-byte aligned, non-NULL
 *   row_token    [rows_max] int32: the token of each row (as moe_dispatch
 *                writes it); read for rows below offsets[n_segments]
 *   other arguments as in moe_expert_ffn (bf16 only: MOE_ERR_UNSUPPORTED for
 *   fp32). A row_token entry outside [0, T) makes that row read zeros and
 *   records MOE_ERR_DEVICE_BOUNDS in the status word.
 * The first GEMM copies the rows with 16-byte asynchronous copies into the
 * same swizzled shared-memory tiles the TMA path fills, one CTA per 128-row
 * tile unless MOE_GEMM_CTA_PAIRS asks for pairs; the second GEMM is
 * unchanged. On a B300 these copies feed the tensor cores at about half the
 * rate of the TMA tile loads, so the first GEMM takes about twice as long as
 * on the dispatched copy, which costs far more than the copy saves:
 * MOE_FUSE_GATHER is off unless asked for.
 */
int moe_expert_ffn_gather(const moe_config* cfg, const void* x, const int32_t* row_token,
                          const int32_t* offsets, int32_t n_segments, int64_t rows_max, int32_t f,
                          const void* W1, const void* W3, const void* W2, void* op, void* ws,
                          size_t ws_bytes, void* stream);

/*
 * moe_expert_ffn for callers that cannot allocate device memory. The source
 * pages have no counterpart: this is an integration convenience, not part of
 * the method.
 *
 * Who needs it: a host framework that owns every device buffer and hands an
 * operator only its inputs and outputs (no workspace), or a latency-critical
 * loop where cudaMalloc, which may synchronise the device, is not allowed.
 * Same computation and arguments as moe_expert_ffn minus the workspace: the
 * SwiGLU hidden activations live in a library-owned static device array of
 * MOE_NOALLOC_SCRATCH_BYTES bytes that every GPU loading this library holds
 * until the process exits. The call allocates and frees nothing.
 *
 *   rows_max * f * sizeof(dtype) must not exceed MOE_NOALLOC_SCRATCH_BYTES - 256,
 *            otherwise MOE_ERR_WORKSPACE is returned and nothing is enqueued
 *            (e.g. bf16 with f = 14336 fits up to 2340 rows).
 *   device_status [1] int32 nullable, device: receives MOE_ERR_DEVICE_TIMEOUT
 *            if a bounded wait expires. The call does not clear it: the
 *            caller sets it to 0 before first use (it may share the word with
 *            earlier stages; the first error recorded wins). With NULL the
 *            call records into a word inside the library's array that no entry
 *            point reads back, so device-side errors are then lost: pass a
 *            word whenever a timeout must be observed.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, and looks it up again
 * after the device's context changes (cudaDeviceReset); make the first call
 * in each context before any stream capture. Every call on a device shares
 * the one array:
 * calls whose work overlaps on the GPU (different streams, or host threads
 * without ordering) race on it and must be serialised by the caller.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (64u << 20)
int moe_expert_ffn_noalloc(const moe_config* cfg, const void* xp, const int32_t* offsets,
                           int32_t n_segments, int64_t rows_max, int32_t f, const void* W1,
                           const void* W3, const void* W2, void* op, int32_t* device_status,
                           void* stream);

/*
 * Routed experts in FP8 ("From personas to MoE 02", section "dense was
 * honestly heavy": quantising the weights, NVFP4 for instance, lightens the
 * weight side of a bandwidth-bound step; the e4m3 format and its scales are
 * this library's choice). e4m3: 1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits, largest magnitude 448.
 *
 * Weights are stored K-major, one fp32 scale per output column:
 *   W1[e][k][n] = value(W1q[e][n][k]) * s1[e][n], likewise W3 with s3, and
 *   W2[e][j][c] = value(W2q[e][c][j]) * s2[e][c] (j < f, c < d).
 * Both operands of every expert product are e4m3 on the tensor cores
 * (tcgen05 kind::f8f6f4, fp32 accumulate): the token rows before W1/W3 and
 * the SwiGLU hidden rows (stored bf16) before W2 are quantised per row on the
 * GPU, scale = max|row| / 448 (fp32; 1 for a zero row) and each element the
 * e4m3 value nearest to element / scale (ties to even, saturating). The row
 * scale times the column scale multiplies each fp32 sum in the epilogue. The
 * expert output op, h and y stay bf16.
 */
typedef struct moe_e4m3_experts {
  const uint8_t* W1;   /* [N, f, d] e4m3 bytes (K-major) */
  const uint8_t* W3;   /* [N, f, d] */
  const uint8_t* W2;   /* [N, d, f] */
  const float*   s1;   /* [N, f] */
  const float*   s3;   /* [N, f] */
  const float*   s2;   /* [N, d] */
} moe_e4m3_experts;

/* Workspace bytes of moe_expert_ffn_e4m3 for rows_max rows, width d and
 * hidden width f: the control block, then (each 256-byte aligned) the bf16
 * hidden rows [rows_max, f], the e4m3 token rows [rows_max, d] and their
 * scales [rows_max] fp32, the e4m3 hidden rows [rows_max, f] and their scales
 * [rows_max] fp32. */
size_t moe_ffn_workspace_size_e4m3(int64_t rows_max, int32_t d, int32_t f);

/* Workspace bytes of moe_layer_forward_e4m3: moe_workspace_size plus the
 * e4m3 rows and scales above (0 if the config is invalid). */
size_t moe_workspace_size_e4m3(const moe_config* cfg);

/*
 * moe_expert_ffn with e4m3 experts (struct above; its pointers are device
 * pointers, the struct itself is read on the host). xp stays bf16 and is
 * quantised per row inside the call. bf16 configs only, d and f multiples of
 * 128; MOE_ERR_UNSUPPORTED for fp32 configs. ws >= moe_ffn_workspace_size_e4m3.
 */
int moe_expert_ffn_e4m3(const moe_config* cfg, const void* xp, const int32_t* offsets,
                        int32_t n_segments, int64_t rows_max, int32_t f,
                        const moe_e4m3_experts* experts, void* op, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * moe_layer_forward with e4m3 routed experts; the router, the shared expert
 * (Ws1, Ws3, Ws2, bf16) and everything else as in moe_layer_forward.
 * ws >= moe_workspace_size_e4m3(cfg).
 */
int moe_layer_forward_e4m3(const moe_config* cfg, const void* x, const void* W_router,
                           const float* bias, const moe_e4m3_experts* experts, const void* Ws1,
                           const void* Ws3, const void* Ws2, const int32_t* home_group,
                           float* logits, void* y, double* stats, void* ws, size_t ws_bytes,
                           void* stream);

/*
 * moe_expert_ffn confined to a slice of the GPU: its two persistent GEMMs
 * launch on at most max_sms streaming multiprocessors (bf16 only; f32 returns
 * MOE_ERR_UNSUPPORTED). Same arguments and result as moe_expert_ffn.
 * One call per device group, each on the SMs one device would have, times
 * the experts as expert parallelism would run them, where the layer waits
 * for the most loaded device ("Capacity-Aware Inference: Mitigating the
 * Straggler Effect in MoE", section 1: the straggler sets the latency).
 * offsets may point into a larger offsets array (row indices stay absolute
 * in xp); W1/W3/W2 then point at the group's first expert.
 */
int moe_expert_ffn_on_sms(const moe_config* cfg, const void* xp, const int32_t* offsets,
                          int32_t n_segments, int64_t rows_max, int32_t f, const void* W1,
                          const void* W3, const void* W2, void* op, int32_t max_sms, void* ws,
                          size_t ws_bytes, void* stream);

/*
 * One grouped GEMM, out[r] = A[r] B[s] for rows r of segment s, the second
 * half of the expert FFN on its own. A [rows_max, K], B [n_segments, K, n_out],
 * out [rows_max, n_out], all dtype; K and n_out multiples of 64 (bf16).
 * ws >= moe_ffn_workspace_size(0, 0, dtype) bytes (status word only).
 */
int moe_grouped_gemm(int32_t dtype, const void* A, const int32_t* offsets, int32_t n_segments,
                     int64_t rows_max, int32_t K, int32_t n_out, const void* B, void* out,
                     void* ws, size_t ws_bytes, void* stream);

/*
 * Failure-detection self-test (the pages have no counterpart): enqueues the
 * bf16 grouped GEMM of moe_grouped_gemm (same arguments, n_segments >= 1,
 * rows_max >= 1) with one CTA announcing but never loading one k-block of its
 * first tile, so the tensor-core issuer's bounded wait (1 s) expires. The
 * kernel then leaves every loop, drains its copies and MMAs, frees its tensor
 * memory and records MOE_ERR_DEVICE_TIMEOUT in ws's status word, where
 * moe_get_device_status reads it; `out` is left partly written. The GPU
 * context stays usable (clear the status with moe_clear_device_status).
 */
int moe_selftest_expired_wait(const void* A, const int32_t* offsets, int32_t n_segments,
                              int64_t rows_max, int32_t K, int32_t n_out, const void* B,
                              void* out, void* ws, size_t ws_bytes, void* stream);

/*
 * Gate-weighted combine, the sum of the layer equation ("Understanding
 * Mixture of Experts", y = sum_i G(x)_i E_i(x)):
 *   y[t] = sum over r in tok_rows[t] (ascending) of row_gate[r] * op[r]
 *          + shared_out[t]
 * summed in fp32 and rounded once to dtype. A token with no row outputs
 * shared_out[t] (or 0).
 *   op [rows_max, d], row_gate [rows_max] fp32, tok_rows [T, kc] int32,
 *   shared_out [T, d] nullable, y [T, d] out.
 */
int moe_combine(const moe_config* cfg, const void* op, const float* row_gate,
                const int32_t* tok_rows, const void* shared_out, void* y, void* stream);

/*
 * Load statistics of one routed batch into stats[MOE_STATS_LEN] (device
 * doubles; layout above). scores [T, N] are the router probabilities; their
 * column sums are taken in fixed point (units of 2^-40, exact u64 sums), so
 * P_i does not depend on the order of the additions.
 * ws >= 8 * N * ceil(T / 32) bytes, 16-byte aligned (scratch: one row of N
 * column sums per 32 tokens; it has no control block).
 */
int moe_load_stats(const moe_config* cfg, const int32_t* demand, const int32_t* kept,
                   const float* scores, double* stats, void* ws, size_t ws_bytes, void* stream);

/*
 * The whole layer: route -> select -> dispatch -> expert FFN (+ shared
 * expert, "How to design inference cost with MoE routing", section "how
 * routing allocates the compute budget": an always-on expert that every token
 * passes through, gate 1) -> combine -> statistics, all enqueued on `stream`
 * with no host synchronisation.
 *
 *   x [T, d]; W_router [d, N]; bias [N] fp32 nullable
 *   W1, W3 [N, d, f]; W2 [N, f, d]
 *   Ws1, Ws3 [d, f_shared]; Ws2 [f_shared, d]   (read only when f_shared > 0)
 *   home_group [T] int32 nullable (expanded drop)
 *   logits [T, N] fp32 nullable: input with MOE_LOGITS_GIVEN (required then);
 *          otherwise, when non-NULL, receives a copy of the logits
 *   y [T, d] out; stats [MOE_STATS_LEN] doubles nullable
 *   ws >= moe_workspace_size(cfg) bytes; intermediates stay readable there
 *   through moe_workspace_views until the next call that uses ws.
 */
int moe_layer_forward(const moe_config* cfg, const void* x, const void* W_router,
                      const float* bias, const void* W1, const void* W3, const void* W2,
                      const void* Ws1, const void* Ws3, const void* Ws2,
                      const int32_t* home_group, float* logits, void* y, double* stats,
                      void* ws, size_t ws_bytes, void* stream);

/*
 * Stage tracing of moe_layer_forward (profiling aid; the pages have no
 * counterpart). moe_layer_stages returns how many kernels moe_layer_forward
 * launches for `cfg` and, when `names` is non-NULL, stores up to max_names
 * static stage names in launch order: the routing ("router" for the
 * tensor-core router, which routes in the same launch; "router_logits" +
 * "route_tokens" on the FMA path; "route_tokens" alone with
 * MOE_LOGITS_GIVEN), select (which also finishes
 * the load statistics when a stats pointer is passed), dispatch,
 * expert_gemm1_swiglu, expert_gemm2, [shared_offsets, shared_gemm1_swiglu,
 * shared_gemm2 when f_shared > 0], combine. Returns a negative MOE_ERR_* for
 * an invalid config.
 *
 * moe_set_trace_events hands the library n_events cudaEvent_t handles
 * (created by the caller, which keeps ownership; n_events <= 32, 0 turns
 * tracing off; a NULL entry records nothing at that point). While set, every
 * moe_layer_forward made from the SAME host thread records events[0] on its
 * stream before the first launch and events[i + 1] right after stage i, for
 * the events it has; the elapsed time between consecutive events is the
 * device time of one stage, launch gap included. Events are re-recorded by
 * every call. The kernels are launched with programmatic dependent launch, so
 * without events a kernel's launch and set-up overlap the previous kernel; an
 * event between two stages serialises them.
 */
int moe_layer_stages(const moe_config* cfg, const char** names, int max_names);
int moe_set_trace_events(void* const* events, int n_events);

/* Device pointers to the intermediates moe_layer_forward leaves in ws. */
typedef struct moe_views_t {
  int32_t* status;         /* [1] sticky device status */
  float*   logits;         /* [T, N] */
  float*   scores;         /* [T, N] */
  int32_t* cand_idx;       /* [T, kc] */
  float*   cand_gate;      /* [T, kc] */
  int32_t* slot;           /* [T, kc] */
  uint8_t* keep;           /* [T, kc] */
  int32_t* demand;         /* [N] */
  int32_t* kept;           /* [N] */
  int32_t* expert_offsets; /* [N + 1] */
  int32_t* row_token;      /* [rows_max] */
  float*   row_gate;       /* [rows_max] */
  int32_t* tok_rows;       /* [T, kc] */
  void*    xp;             /* [rows_max, d] (not written with MOE_FUSE_GATHER) */
  void*    op;             /* [rows_max, d] */
  void*    shared_out;     /* [T, d] or NULL */
  int32_t* coverage;       /* [T] kept pairs per token (moe_dispatch's coverage) */
} moe_views_t;

/* Carve `ws` into the views above. Host only; no CUDA call. */
int moe_workspace_views(const moe_config* cfg, void* ws, moe_views_t* out);

/* Enqueue a read of the sticky device status word at ws and synchronise
 * `stream`; *out_host receives MOE_OK or the first MOE_ERR_DEVICE_* recorded.
 * `ws` is any workspace passed to the calls above; the status word is the
 * first 4 bytes of its control block. */
int moe_get_device_status(const void* ws, void* stream, int32_t* out_host);

/* Enqueue a reset of ws's control block (MOE_CTRL_BYTES, starting with the
 * status word) to zero. */
int moe_clear_device_status(void* ws, void* stream);

/* Static description of a status code. */
const char* moe_status_string(int status);

/* Release host-side caches. Tensor-map descriptors are currently encoded on
 * every call, so there is nothing to release; the entry point is kept so a
 * caller need not change when a cache is added. */
void moe_release_caches(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
