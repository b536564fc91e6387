// C ABI of the MoE layer library: argument checks, workspace layout and the
// launch sequence. Every check runs on the host before anything is enqueued.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "device_common.cuh"
#include "internal.h"

namespace moe {

int device_sm_count() {
  static int counts[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    counts[dev] = n;
  }
  return counts[dev];
}

namespace {

__global__ void write_pair_kernel(int32_t* p, int32_t a, int32_t b) {
  pdl_launch_dependents();
  pdl_wait();
  p[0] = a;
  p[1] = b;
}
// Zeroes a workspace's control block (status word and arrival counters).
__global__ void clear_ctrl_kernel(int32_t* ctrl) {
  pdl_wait();
  for (int i = threadIdx.x; i < static_cast<int>(kCtrlBytes / 4); i += blockDim.x) ctrl[i] = 0;
}

struct Derived {
  int kc = 0;
  int cap = 0;            // C, c, a device's C or T
  int device_group = 0;   // experts sharing one capacity (device-level drop), else 0
  int64_t rows_max = 0;
  int sx = 0;             // bytes per activation element
  bool ec = false;
};

constexpr int kMaxN = 256;
constexpr int kMaxSlots = 32;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A buffer of `count` elements must be present unless it is empty (framework
// tensors of size zero carry a NULL data pointer).
bool have(const void* p, int64_t count) { return p != nullptr || count == 0; }

int validate(const moe_config* c, Derived* dv) {
  if (!c) return MOE_ERR_NULL;
  if (c->T < 0 || c->d <= 0 || c->N <= 0 || c->f <= 0 || c->k <= 0) return MOE_ERR_SHAPE;
  if (c->mode != MOE_TOKEN_CHOICE && c->mode != MOE_EXPERT_CHOICE && c->mode != MOE_CAPACITY_DROP &&
      c->mode != MOE_CAPACITY_DROP_DEVICE)
    return MOE_ERR_SHAPE;
  const bool device_drop = c->mode == MOE_CAPACITY_DROP_DEVICE;
  if (c->dtype != MOE_BF16 && c->dtype != MOE_F32) return MOE_ERR_SHAPE;
  if (c->k > c->N || c->m < 0 || c->f_shared < 0) return MOE_ERR_SHAPE;
  if (std::isnan(c->gamma) || c->gamma < 0) return MOE_ERR_SHAPE;
  if ((c->m > 0 || device_drop) && (c->group_size <= 0 || c->N % c->group_size != 0))
    return MOE_ERR_SHAPE;
  if (c->N > kMaxN) return MOE_ERR_UNSUPPORTED;
  if (c->T > select_max_tokens()) return MOE_ERR_UNSUPPORTED;
  const bool ec = c->mode == MOE_EXPERT_CHOICE;
  if (ec && c->m != 0) return MOE_ERR_SHAPE;
  if (!ec && c->k + c->m > kMaxSlots) return MOE_ERR_UNSUPPORTED;
  if (c->dtype == MOE_BF16) {
    if (c->d % 64 || c->f % 64 || c->f_shared % 64) return MOE_ERR_SHAPE;
  } else {
    if (c->d % 8) return MOE_ERR_SHAPE;
  }
  Derived d;
  d.ec = ec;
  d.kc = ec ? c->N : c->k + c->m;
  d.sx = c->dtype == MOE_BF16 ? 2 : 4;
  const int64_t T = c->T, N = c->N;
  if (ec) {
    d.cap = static_cast<int>(std::min<int64_t>(T, (static_cast<int64_t>(c->k) * T) / N));
    d.rows_max = N * d.cap;
  } else if (device_drop) {
    // a device of group_size experts holds the sum of their capacities
    const int64_t gs = c->group_size;
    const int64_t most = T * std::min<int64_t>(d.kc, gs);
    int64_t cap = most;
    if (!std::isinf(c->gamma)) {
      const double nbar =
          static_cast<double>(static_cast<int64_t>(c->k) * T) / static_cast<double>(N);
      const double cf = std::floor(c->gamma * nbar * static_cast<double>(gs));
      cap = cf >= static_cast<double>(most) ? most : static_cast<int64_t>(cf);
    }
    d.cap = static_cast<int>(cap);
    d.device_group = static_cast<int>(gs);
    d.rows_max = std::min<int64_t>(T * d.kc, (N / gs) * cap);
  } else if (c->mode == MOE_CAPACITY_DROP && !std::isinf(c->gamma)) {
    const double nbar = static_cast<double>(static_cast<int64_t>(c->k) * T) / static_cast<double>(N);
    const double cf = std::floor(c->gamma * nbar);
    d.cap = cf >= static_cast<double>(T) ? static_cast<int>(T) : static_cast<int>(cf);
    d.rows_max = std::min<int64_t>(T * d.kc, N * d.cap);
  } else {
    d.cap = static_cast<int>(T);
    d.rows_max = T * d.kc;
  }
  if (dv) *dv = d;
  return MOE_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Stage timing of moe_layer_forward (moe_set_trace_events): caller-owned
// events, per host thread.
constexpr int kMaxTraceEvents = 32;
thread_local cudaEvent_t g_trace_events[kMaxTraceEvents];
thread_local int g_trace_n = 0;

// Records the trace events of one moe_layer_forward: event 0 before the first
// launch, event i + 1 after stage i (no-op when no events are set).
struct Tracer {
  cudaStream_t s;
  int next = 0;
  bool mark(int stages = 1) {
    for (int j = 0; j < stages; ++j, ++next)
      if (next < g_trace_n && g_trace_events[next] &&
          cudaEventRecord(g_trace_events[next], s) != cudaSuccess)
        return false;
    return true;
  }
};

// The kernels moe_layer_forward launches for c, in launch order.
int layer_stage_names(const moe_config& c, const char** names, int max_names) {
  const char* list[16];
  int n = 0;
  if (c.flags & MOE_LOGITS_GIVEN) {
    list[n++] = "route_tokens";
  } else if (router_tc_supported(c.dtype, c.d, c.N)) {
    list[n++] = "router";  // tensor-core logits and routing in one launch
  } else {
    list[n++] = "router_logits";
    list[n++] = "route_tokens";
  }
  list[n++] = "select";
  list[n++] = "dispatch";
  list[n++] = "expert_gemm1_swiglu";
  list[n++] = "expert_gemm2";
  if (c.f_shared > 0) {
    list[n++] = "shared_offsets";
    list[n++] = "shared_gemm1_swiglu";
    list[n++] = "shared_gemm2";
  }
  list[n++] = "combine";
  if (names)
    for (int i = 0; i < n && i < max_names; ++i) names[i] = list[i];
  return n;
}

int status_from(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// Logits (unless given) and per-token routing. logits: output buffer, or the
// input when MOE_LOGITS_GIVEN; colsum: column sums of the scores for the
// load statistics (nullable), whose row count is stored in *colsum_rows.
int run_router(const moe_config& c, bool ec, const void* x, const void* W_r, const float* bias,
               float* logits, float* scores, int32_t* cand_idx, float* cand_gate,
               const int32_t* home_group, int32_t* status, unsigned long long* colsum,
               int* colsum_rows, cudaStream_t s, Tracer* tr = nullptr) {
  const bool given = (c.flags & MOE_LOGITS_GIVEN) != 0;
  const bool tc = !given && router_tc_supported(c.dtype, c.d, c.N);
  RouteArgs ra;
  ra.logits = logits;
  ra.scores = scores;
  ra.cand_idx = cand_idx;
  ra.cand_gate = cand_gate;
  ra.home_group = home_group;
  ra.colsum = colsum;
  ra.T = c.T;
  ra.N = c.N;
  ra.k = c.k;
  ra.m = c.m;
  ra.group_size = c.group_size > 0 ? c.group_size : 1;
  ra.renorm = c.renorm;
  ra.ec = ec ? 1 : 0;
  if (tc) {
    const RouterPlan p = router_plan(c.T, c.d, c.N);
    if (colsum_rows) *colsum_rows = p.colsum_rows;
    ra.bias = bias;
    ra.logits_out = logits;
    if (c.T > 0 && launch_router_tc(x, W_r, c.d, p, ra, status, s) != cudaSuccess)
      return MOE_ERR_LAUNCH;
    return (!tr || tr->mark()) ? MOE_OK : MOE_ERR_LAUNCH;
  }
  if (colsum_rows) *colsum_rows = route_tokens_colsum_rows(c.T, c.N);
  if (!given) {
    if ((c.T > 0 &&
         launch_router_logits(c.dtype, x, W_r, bias, logits, c.T, c.d, c.N, s) != cudaSuccess) ||
        (tr && !tr->mark()))
      return MOE_ERR_LAUNCH;
  }
  if ((c.T > 0 && launch_route_tokens(ra, s) != cudaSuccess) || (tr && !tr->mark()))
    return MOE_ERR_LAUNCH;
  return MOE_OK;
}

struct Layout {
  size_t ctrl, logits, scores, cand_idx, cand_gate, slot, keep, demand, kept, offsets,
      shared_offsets, row_token, row_gate, tok_rows, coverage, xp, hp, op, shared_out, colsum,
      // e4m3 experts only: e4m3 token rows and scales, e4m3 hidden rows and scales
      xq, xs, hq, hs, total;
};

Layout layout(const moe_config& c, const Derived& d, bool e4m3 = false) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const size_t T = c.T, N = c.N, kc = d.kc, R = d.rows_max, dd = c.d;
  L.ctrl = take(kCtrlBytes);
  L.logits = take(T * N * 4);
  L.scores = take(T * N * 4);
  L.cand_idx = take(T * kc * 4);
  L.cand_gate = take(T * kc * 4);
  L.slot = take(T * kc * 4);
  L.keep = take(T * kc);
  L.demand = take(N * 4);
  L.kept = take(N * 4);
  L.offsets = take((N + 1) * 4);
  L.shared_offsets = take(2 * 4);
  L.row_token = take(R * 4);
  L.row_gate = take(R * 4);
  L.tok_rows = take(T * kc * 4);
  L.coverage = take(T * 4);
  L.xp = take(R * dd * d.sx);
  const size_t hp_rows = std::max(R * static_cast<size_t>(c.f), T * static_cast<size_t>(c.f_shared));
  L.hp = take(hp_rows * d.sx);
  L.op = take(R * dd * d.sx);
  L.shared_out = take(c.f_shared > 0 ? T * dd * d.sx : 0);
  L.colsum = take(colsum_bytes(c.T, c.N));
  L.xq = take(e4m3 ? R * dd : 0);
  L.xs = take(e4m3 ? R * 4 : 0);
  L.hq = take(e4m3 ? R * static_cast<size_t>(c.f) : 0);
  L.hs = take(e4m3 ? R * 4 : 0);
  L.total = off;
  return L;
}

// The e4m3 expert FFN's workspace after the control block: bf16 hidden rows,
// e4m3 token rows and scales, e4m3 hidden rows and scales.
struct FfnE4m3Layout {
  size_t hp, xq, xs, hq, hs, total;
};
FfnE4m3Layout ffn_e4m3_layout(int64_t rows_max, int d, int f) {
  FfnE4m3Layout L{};
  const size_t R = static_cast<size_t>(rows_max);
  size_t off = kCtrlBytes;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L.hp = take(R * f * 2);
  L.xq = take(R * d);
  L.xs = take(R * 4);
  L.hq = take(R * f);
  L.hs = take(R * 4);
  L.total = off;
  return L;
}

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<unsigned char*>(ws) + off);
}


// FFN over expert-contiguous rows; hp is scratch of rows_max * f elements;
// status is the workspace's status word. With row_src (bf16 only) xp is the
// [a_rows, d] token matrix and GEMM1 reads row r of the segments from
// xp[row_src[r]].
int run_ffn(int dtype, const void* xp, const int32_t* offsets, int S, int64_t rows_max, int d,
            int f, const void* W1, const void* W3, const void* W2, void* hp, void* op,
            int32_t* status, cudaStream_t s, Tracer* tr = nullptr, int max_sms = 0,
            const int32_t* row_src = nullptr, int a_rows = 0) {
  cudaError_t e;
  if (row_src && dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (dtype == MOE_BF16) {
    e = launch_grouped_gemm_tc_bf16(xp, offsets, S, rows_max, d, f, W1, W3, hp, true, status, s, -1,
                                    max_sms, row_src, a_rows);
    if (e != cudaSuccess || (tr && !tr->mark())) return MOE_ERR_LAUNCH;
    e = launch_grouped_gemm_tc_bf16(hp, offsets, S, rows_max, f, d, W2, nullptr, op, false, status,
                                    s, -1, max_sms);
  } else {
    e = launch_grouped_gemm_simt_f32(static_cast<const float*>(xp), offsets, S, rows_max, d, f,
                                     static_cast<const float*>(W1), static_cast<const float*>(W3),
                                     static_cast<float*>(hp), true, s);
    if (e != cudaSuccess || (tr && !tr->mark())) return MOE_ERR_LAUNCH;
    e = launch_grouped_gemm_simt_f32(static_cast<const float*>(hp), offsets, S, rows_max, f, d,
                                     static_cast<const float*>(W2), nullptr,
                                     static_cast<float*>(op), false, s);
  }
  if (e != cudaSuccess || (tr && !tr->mark())) return MOE_ERR_LAUNCH;
  return MOE_OK;
}

// Expert FFN with e4m3 experts: the bf16 rows xp are quantised per row (xq,
// xs), GEMM1 on e4m3 operands writes the bf16 hidden rows hp, which are
// quantised per row (hq, hs) for GEMM2. Trace marks: the first quantisation
// and GEMM1 count as GEMM1, the second quantisation and GEMM2 as GEMM2.
int run_ffn_e4m3(const void* xp, const int32_t* offsets, int S, int64_t rows_max, int d, int f,
                 const moe_e4m3_experts& w, void* hp, uint8_t* xq, float* xs, uint8_t* hq,
                 float* hs, void* op, int32_t* status, cudaStream_t s, Tracer* tr = nullptr) {
  cudaError_t e = launch_quantize_rows_e4m3(xp, offsets, S, rows_max, d, xq, xs, s);
  if (e == cudaSuccess)
    e = launch_grouped_gemm_tc_fp8(xq, xs, offsets, S, rows_max, d, f, w.W1, w.s1, w.W3, w.s3, hp,
                                   true, status, s);
  if (e != cudaSuccess || (tr && !tr->mark())) return MOE_ERR_LAUNCH;
  e = launch_quantize_rows_e4m3(hp, offsets, S, rows_max, f, hq, hs, s);
  if (e == cudaSuccess)
    e = launch_grouped_gemm_tc_fp8(hq, hs, offsets, S, rows_max, f, d, w.W2, w.s2, nullptr,
                                   nullptr, op, false, status, s);
  if (e != cudaSuccess || (tr && !tr->mark())) return MOE_ERR_LAUNCH;
  return MOE_OK;
}

int check_e4m3(const moe_config& c, int f, const moe_e4m3_experts* w) {
  if (c.dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (!w) return MOE_ERR_NULL;
  if (c.d % 128 || f % 128) return MOE_ERR_SHAPE;
  if (!w->W1 || !w->W3 || !w->W2 || !w->s1 || !w->s3 || !w->s2) return MOE_ERR_NULL;
  if (!aligned16(w->W1) || !aligned16(w->W3) || !aligned16(w->W2)) return MOE_ERR_ALIGN;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_sizes(const moe_config* cfg, moe_sizes_t* out) {
  if (!out) return MOE_ERR_NULL;
  Derived d;
  const int st = validate(cfg, &d);
  if (st != MOE_OK) return st;
  out->kc = d.kc;
  out->capacity = d.cap;
  out->rows_max = d.rows_max;
  out->workspace = layout(*cfg, d).total;
  out->ffn_workspace = moe_ffn_workspace_size(d.rows_max, cfg->f, cfg->dtype);
  return MOE_OK;
}

size_t moe_workspace_size(const moe_config* cfg) {
  Derived d;
  if (validate(cfg, &d) != MOE_OK) return 0;
  return layout(*cfg, d).total;
}

size_t moe_ffn_workspace_size(int64_t rows_max, int32_t f, int32_t dtype) {
  if (rows_max < 0 || f < 0) return 0;
  const size_t sx = dtype == MOE_BF16 ? 2 : 4;
  return kCtrlBytes + align256(static_cast<size_t>(rows_max) * static_cast<size_t>(f) * sx);
}

size_t moe_ffn_workspace_size_e4m3(int64_t rows_max, int32_t d, int32_t f) {
  if (rows_max < 0 || d < 0 || f < 0) return 0;
  return ffn_e4m3_layout(rows_max, d, f).total;
}

size_t moe_workspace_size_e4m3(const moe_config* cfg) {
  Derived d;
  if (validate(cfg, &d) != MOE_OK) return 0;
  return layout(*cfg, d, true).total;
}

size_t moe_route_workspace_size(const moe_config* cfg) {
  Derived d;
  if (validate(cfg, &d) != MOE_OK) return 0;
  return kCtrlBytes;
}

int moe_route(const moe_config* cfg, const void* x, const void* W_router, const float* bias,
              float* logits, float* scores, int32_t* cand_idx, float* cand_gate,
              const int32_t* home_group, void* ws, size_t ws_bytes, void* stream) {
  Derived d;
  int st = validate(cfg, &d);
  if (st != MOE_OK) return st;
  const bool given = (cfg->flags & MOE_LOGITS_GIVEN) != 0;
  const int64_t T = cfg->T;
  if (!have(logits, T) || !have(cand_gate, T) || (!d.ec && !have(cand_idx, T)) || !ws)
    return MOE_ERR_NULL;
  if (!given && (!have(x, T) || !W_router)) return MOE_ERR_NULL;
  if (!given && (!aligned16(x) || !aligned16(W_router))) return MOE_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_ALIGN;
  if (ws_bytes < moe_route_workspace_size(cfg)) return MOE_ERR_WORKSPACE;
  return run_router(*cfg, d.ec, x, W_router, bias, logits, scores, cand_idx, cand_gate,
                    home_group, static_cast<int32_t*>(ws), nullptr, nullptr, as_stream(stream));
}

int moe_capacity_drop(const moe_config* cfg, const int32_t* cand_idx, const float* cand_gate,
                      int32_t* slot, uint8_t* keep, int32_t* demand, int32_t* kept, void* stream) {
  Derived d;
  int st = validate(cfg, &d);
  if (st != MOE_OK) return st;
  const int64_t T = cfg->T;
  if (!have(cand_gate, T) || !have(slot, T) || !demand || !kept || (!d.ec && !have(cand_idx, T)))
    return MOE_ERR_NULL;
  return status_from(launch_select(cand_idx, cand_gate, cfg->T, d.kc, cfg->N, d.ec ? 1 : 0, d.cap, d.device_group,
                                   slot, keep, demand, kept, as_stream(stream)));
}

int moe_dispatch(const moe_config* cfg, const void* x, const int32_t* cand_idx,
                 const float* cand_gate, const int32_t* slot, const int32_t* kept,
                 int32_t* expert_offsets, int32_t* row_token, float* row_gate, int32_t* tok_rows,
                 int32_t* coverage, void* xp, void* stream) {
  Derived d;
  int st = validate(cfg, &d);
  if (st != MOE_OK) return st;
  const int64_t T = cfg->T, R = d.rows_max;
  if (!have(x, T) || !have(cand_gate, T) || !have(slot, T) || !kept || !expert_offsets ||
      !have(row_token, R) || !have(row_gate, R) || !have(tok_rows, T) || !have(xp, R) ||
      (!d.ec && !have(cand_idx, T)))
    return MOE_ERR_NULL;
  if (!aligned16(x) || !aligned16(xp)) return MOE_ERR_ALIGN;
  return status_from(launch_dispatch(cfg->dtype, x, cand_idx, cand_gate, slot, kept, cfg->T,
                                     cfg->d, cfg->N, d.kc, d.ec ? 1 : 0, d.rows_max, expert_offsets, row_token,
                                     row_gate, tok_rows, coverage, xp, nullptr, StatsArgs{},
                                     as_stream(stream)));
}

int moe_expert_ffn(const moe_config* cfg, const void* xp, const int32_t* offsets,
                   int32_t n_segments, int64_t rows_max, int32_t f, const void* W1,
                   const void* W3, const void* W2, void* op, void* ws, size_t ws_bytes,
                   void* stream) {
  if (!cfg) return MOE_ERR_NULL;
  if (cfg->dtype != MOE_BF16 && cfg->dtype != MOE_F32) return MOE_ERR_SHAPE;
  if (cfg->d <= 0 || f <= 0 || n_segments < 0 || rows_max < 0) return MOE_ERR_SHAPE;
  if (cfg->dtype == MOE_BF16 && (cfg->d % 64 || f % 64)) return MOE_ERR_SHAPE;
  if (n_segments > kMaxN) return MOE_ERR_UNSUPPORTED;
  if (!xp || !offsets || !W1 || !W3 || !W2 || !op || !ws) return MOE_ERR_NULL;
  if (!aligned16(xp) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(op) ||
      !aligned16(ws))
    return MOE_ERR_ALIGN;
  if (ws_bytes < moe_ffn_workspace_size(rows_max, f, cfg->dtype)) return MOE_ERR_WORKSPACE;
  void* hp = static_cast<unsigned char*>(ws) + kCtrlBytes;
  return run_ffn(cfg->dtype, xp, offsets, n_segments, rows_max, cfg->d, f, W1, W3, W2, hp, op,
                 static_cast<int32_t*>(ws), as_stream(stream));
}

int moe_expert_ffn_gather(const moe_config* cfg, const void* x, const int32_t* row_token,
                          const int32_t* offsets, int32_t n_segments, int64_t rows_max, int32_t f,
                          const void* W1, const void* W3, const void* W2, void* op, void* ws,
                          size_t ws_bytes, void* stream) {
  if (!cfg) return MOE_ERR_NULL;
  if (cfg->dtype != MOE_BF16) return cfg->dtype == MOE_F32 ? MOE_ERR_UNSUPPORTED : MOE_ERR_SHAPE;
  if (cfg->T < 0 || cfg->d <= 0 || f <= 0 || n_segments < 0 || rows_max < 0) return MOE_ERR_SHAPE;
  if (cfg->d % 64 || f % 64) return MOE_ERR_SHAPE;
  if (n_segments > kMaxN) return MOE_ERR_UNSUPPORTED;
  if (!offsets || !W1 || !W3 || !W2 || !op || !ws) return MOE_ERR_NULL;
  if (!x || (rows_max > 0 && !row_token)) return MOE_ERR_NULL;
  if (!aligned16(x) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(op) ||
      !aligned16(ws))
    return MOE_ERR_ALIGN;
  if (ws_bytes < moe_ffn_workspace_size(rows_max, f, cfg->dtype)) return MOE_ERR_WORKSPACE;
  void* hp = static_cast<unsigned char*>(ws) + kCtrlBytes;
  return run_ffn(cfg->dtype, x, offsets, n_segments, rows_max, cfg->d, f, W1, W3, W2, hp, op,
                 static_cast<int32_t*>(ws), as_stream(stream), nullptr, 0, row_token, cfg->T);
}

int moe_expert_ffn_on_sms(const moe_config* cfg, const void* xp, const int32_t* offsets,
                          int32_t n_segments, int64_t rows_max, int32_t f, const void* W1,
                          const void* W3, const void* W2, void* op, int32_t max_sms, void* ws,
                          size_t ws_bytes, void* stream) {
  if (!cfg) return MOE_ERR_NULL;
  if (cfg->dtype != MOE_BF16) return cfg->dtype == MOE_F32 ? MOE_ERR_UNSUPPORTED : MOE_ERR_SHAPE;
  if (max_sms <= 0) return MOE_ERR_SHAPE;
  if (cfg->d <= 0 || f <= 0 || n_segments < 0 || rows_max < 0) return MOE_ERR_SHAPE;
  if (cfg->d % 64 || f % 64) return MOE_ERR_SHAPE;
  if (n_segments > kMaxN) return MOE_ERR_UNSUPPORTED;
  if (!xp || !offsets || !W1 || !W3 || !W2 || !op || !ws) return MOE_ERR_NULL;
  if (!aligned16(xp) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(op) ||
      !aligned16(ws))
    return MOE_ERR_ALIGN;
  if (ws_bytes < moe_ffn_workspace_size(rows_max, f, cfg->dtype)) return MOE_ERR_WORKSPACE;
  void* hp = static_cast<unsigned char*>(ws) + kCtrlBytes;
  return run_ffn(cfg->dtype, xp, offsets, n_segments, rows_max, cfg->d, f, W1, W3, W2, hp, op,
                 static_cast<int32_t*>(ws), as_stream(stream), nullptr, max_sms);
}

int moe_grouped_gemm(int32_t dtype, const void* A, const int32_t* offsets, int32_t n_segments,
                     int64_t rows_max, int32_t K, int32_t n_out, const void* B, void* out,
                     void* ws, size_t ws_bytes, void* stream) {
  if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_SHAPE;
  if (K <= 0 || n_out <= 0 || n_segments < 0 || rows_max < 0) return MOE_ERR_SHAPE;
  if (dtype == MOE_BF16 && (K % 64 || n_out % 64)) return MOE_ERR_SHAPE;
  if (n_segments > kMaxN) return MOE_ERR_UNSUPPORTED;
  if (!A || !offsets || !B || !out || !ws) return MOE_ERR_NULL;
  if (!aligned16(A) || !aligned16(B) || !aligned16(out) || !aligned16(ws)) return MOE_ERR_ALIGN;
  if (ws_bytes < moe_ffn_workspace_size(0, 0, dtype)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  cudaError_t e;
  if (dtype == MOE_BF16)
    e = launch_grouped_gemm_tc_bf16(A, offsets, n_segments, rows_max, K, n_out, B, nullptr, out,
                                    false, static_cast<int32_t*>(ws), s);
  else
    e = launch_grouped_gemm_simt_f32(static_cast<const float*>(A), offsets, n_segments, rows_max,
                                     K, n_out, static_cast<const float*>(B), nullptr,
                                     static_cast<float*>(out), false, s);
  return status_from(e);
}

int moe_selftest_expired_wait(const void* A, const int32_t* offsets, int32_t n_segments,
                              int64_t rows_max, int32_t K, int32_t n_out, const void* B,
                              void* out, void* ws, size_t ws_bytes, void* stream) {
  if (K <= 0 || n_out <= 0 || n_segments <= 0 || rows_max <= 0) return MOE_ERR_SHAPE;
  if (K % 64 || n_out % 64) return MOE_ERR_SHAPE;
  if (n_segments > kMaxN) return MOE_ERR_UNSUPPORTED;
  if (!A || !offsets || !B || !out || !ws) return MOE_ERR_NULL;
  if (!aligned16(A) || !aligned16(B) || !aligned16(out) || !aligned16(ws)) return MOE_ERR_ALIGN;
  if (ws_bytes < moe_ffn_workspace_size(0, 0, MOE_BF16)) return MOE_ERR_WORKSPACE;
  return status_from(launch_grouped_gemm_tc_bf16(A, offsets, n_segments, rows_max, K, n_out, B,
                                                 nullptr, out, false, static_cast<int32_t*>(ws),
                                                 as_stream(stream), 0));
}

int moe_combine(const moe_config* cfg, const void* op, const float* row_gate,
                const int32_t* tok_rows, const void* shared_out, void* y, void* stream) {
  Derived d;
  int st = validate(cfg, &d);
  if (st != MOE_OK) return st;
  const int64_t T = cfg->T, R = d.rows_max;
  if (!have(op, R) || !have(row_gate, R) || !have(tok_rows, T) || !have(y, T)) return MOE_ERR_NULL;
  if (!aligned16(op) || !aligned16(y) || (shared_out && !aligned16(shared_out)))
    return MOE_ERR_ALIGN;
  return status_from(launch_combine(cfg->dtype, op, row_gate, tok_rows, shared_out, y, cfg->T,
                                    cfg->d, d.kc, d.rows_max, as_stream(stream)));
}

int moe_load_stats(const moe_config* cfg, const int32_t* demand, const int32_t* kept,
                   const float* scores, double* stats, void* ws, size_t ws_bytes, void* stream) {
  Derived d;
  int st = validate(cfg, &d);
  if (st != MOE_OK) return st;
  if (!demand || !kept || !have(scores, cfg->T) || !stats || !ws) return MOE_ERR_NULL;
  const size_t need = static_cast<size_t>(colsum_kernel_rows(cfg->T)) *
                      static_cast<size_t>(cfg->N) * sizeof(unsigned long long);
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_ALIGN;
  cudaStream_t s = as_stream(stream);
  auto* colsum = static_cast<unsigned long long*>(ws);
  if (launch_colsum(scores, cfg->T, cfg->N, colsum, s) != cudaSuccess) return MOE_ERR_LAUNCH;
  return status_from(launch_stats_final(demand, kept, colsum, colsum_kernel_rows(cfg->T), cfg->T,
                                        cfg->N, stats, s));
}

}  // extern "C"

namespace moe {
namespace {

// moe_layer_forward with bf16/fp32 experts (W1, W3, W2) or, when w8 is set,
// e4m3 experts.
int layer_forward(const moe_config* cfg, const void* x, const void* W_router, const float* bias,
                  const void* W1, const void* W3, const void* W2, const moe_e4m3_experts* w8,
                  const void* Ws1, const void* Ws3, const void* Ws2, const int32_t* home_group,
                  float* logits, void* y, double* stats, void* ws, size_t ws_bytes,
                  void* stream) {
  Derived d;
  int st = validate(cfg, &d);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  const bool given = (c.flags & MOE_LOGITS_GIVEN) != 0;
  // bf16 experts: GEMM1 gathers the token rows itself, dispatch copies none
  const bool fuse = (c.flags & MOE_FUSE_GATHER) != 0 && c.dtype == MOE_BF16 && !w8;
  if (w8) {
    if ((st = check_e4m3(c, c.f, w8)) != MOE_OK) return st;
    W1 = w8->W1;
    W3 = w8->W3;
    W2 = w8->W2;
  }
  if (!have(x, c.T) || !W1 || !W3 || !W2 || !have(y, c.T) || !ws) return MOE_ERR_NULL;
  if (given ? !have(logits, c.T) : !W_router) return MOE_ERR_NULL;
  if (c.f_shared > 0 && (!Ws1 || !Ws3 || !Ws2)) return MOE_ERR_NULL;
  if (!aligned16(x) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(y) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u) || (!given && !aligned16(W_router)))
    return MOE_ERR_ALIGN;
  if (c.f_shared > 0 && (!aligned16(Ws1) || !aligned16(Ws3) || !aligned16(Ws2))) return MOE_ERR_ALIGN;
  const Layout L = layout(c, d, w8 != nullptr);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;

  cudaStream_t s = as_stream(stream);
  Tracer tr{s};
  if (!tr.mark()) return MOE_ERR_LAUNCH;
  int32_t* ctrl = at<int32_t>(ws, L.ctrl);
  int32_t* status = ctrl;
  float* Lg = given ? logits : (logits ? logits : at<float>(ws, L.logits));
  float* scores = at<float>(ws, L.scores);
  int32_t* cand_idx = at<int32_t>(ws, L.cand_idx);
  float* cand_gate = at<float>(ws, L.cand_gate);
  int32_t* slot = at<int32_t>(ws, L.slot);
  uint8_t* keep = at<uint8_t>(ws, L.keep);
  int32_t* demand = at<int32_t>(ws, L.demand);
  int32_t* kept = at<int32_t>(ws, L.kept);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* row_token = at<int32_t>(ws, L.row_token);
  float* row_gate = at<float>(ws, L.row_gate);
  int32_t* tok_rows = at<int32_t>(ws, L.tok_rows);
  void* xp = at<void>(ws, L.xp);
  void* hp = at<void>(ws, L.hp);
  void* op = at<void>(ws, L.op);
  void* ys = c.f_shared > 0 ? at<void>(ws, L.shared_out) : nullptr;

  unsigned long long* colsum = stats ? at<unsigned long long>(ws, L.colsum) : nullptr;
  int colsum_rows = 0;
  st = run_router(c, d.ec, x, W_router, bias, Lg, scores, cand_idx, cand_gate, home_group, status,
                  colsum, &colsum_rows, s, &tr);
  if (st != MOE_OK) return st;
  StatsArgs sa;
  sa.colsum = colsum;
  sa.rows = colsum_rows;
  sa.stats = stats;
  if (launch_select(cand_idx, cand_gate, c.T, d.kc, c.N, d.ec ? 1 : 0, d.cap, d.device_group, slot, keep, demand,
                    kept, s) != cudaSuccess ||
      !tr.mark(1))
    return MOE_ERR_LAUNCH;
  if (launch_dispatch(c.dtype, x, cand_idx, cand_gate, slot, kept, c.T, c.d, c.N, d.kc,
                      d.ec ? 1 : 0, d.rows_max, offsets, row_token, row_gate, tok_rows,
                      at<int32_t>(ws, L.coverage), fuse ? nullptr : xp, demand, sa, s) !=
          cudaSuccess ||
      !tr.mark(1))
    return MOE_ERR_LAUNCH;
  if (w8)
    st = run_ffn_e4m3(xp, offsets, c.N, d.rows_max, c.d, c.f, *w8, hp, at<uint8_t>(ws, L.xq),
                      at<float>(ws, L.xs), at<uint8_t>(ws, L.hq), at<float>(ws, L.hs), op, status,
                      s, &tr);
  else if (fuse)
    st = run_ffn(c.dtype, x, offsets, c.N, d.rows_max, c.d, c.f, W1, W3, W2, hp, op, status, s,
                 &tr, 0, row_token, c.T);
  else
    st = run_ffn(c.dtype, xp, offsets, c.N, d.rows_max, c.d, c.f, W1, W3, W2, hp, op, status, s,
                 &tr);
  if (st != MOE_OK) return st;
  if (c.f_shared > 0) {
    if (c.T > 0) {
      int32_t* soff = at<int32_t>(ws, L.shared_offsets);
      if (launch_pdl(write_pair_kernel, 1, 1, 0, s, soff, 0, c.T) != cudaSuccess || !tr.mark(1))
        return MOE_ERR_LAUNCH;
      st = run_ffn(c.dtype, x, soff, 1, c.T, c.d, c.f_shared, Ws1, Ws3, Ws2, hp, ys, status, s,
                   &tr);
      if (st != MOE_OK) return st;
    } else if (!tr.mark(3)) {
      return MOE_ERR_LAUNCH;
    }
  }
  if (launch_combine(c.dtype, op, row_gate, tok_rows, ys, y, c.T, c.d, d.kc, d.rows_max, s) !=
          cudaSuccess ||
      !tr.mark(1))
    return MOE_ERR_LAUNCH;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" {

int moe_layer_forward(const moe_config* cfg, const void* x, const void* W_router,
                      const float* bias, const void* W1, const void* W3, const void* W2,
                      const void* Ws1, const void* Ws3, const void* Ws2,
                      const int32_t* home_group, float* logits, void* y, double* stats, void* ws,
                      size_t ws_bytes, void* stream) {
  return layer_forward(cfg, x, W_router, bias, W1, W3, W2, nullptr, Ws1, Ws3, Ws2, home_group,
                       logits, y, stats, ws, ws_bytes, stream);
}

int moe_layer_forward_e4m3(const moe_config* cfg, const void* x, const void* W_router,
                           const float* bias, const moe_e4m3_experts* experts, const void* Ws1,
                           const void* Ws3, const void* Ws2, const int32_t* home_group,
                           float* logits, void* y, double* stats, void* ws, size_t ws_bytes,
                           void* stream) {
  if (!experts) return MOE_ERR_NULL;
  return layer_forward(cfg, x, W_router, bias, nullptr, nullptr, nullptr, experts, Ws1, Ws3, Ws2,
                       home_group, logits, y, stats, ws, ws_bytes, stream);
}

int moe_expert_ffn_e4m3(const moe_config* cfg, const void* xp, const int32_t* offsets,
                        int32_t n_segments, int64_t rows_max, int32_t f,
                        const moe_e4m3_experts* experts, void* op, void* ws, size_t ws_bytes,
                        void* stream) {
  if (!cfg) return MOE_ERR_NULL;
  if (cfg->d <= 0 || f <= 0 || n_segments < 0 || rows_max < 0) return MOE_ERR_SHAPE;
  int st = check_e4m3(*cfg, f, experts);
  if (st != MOE_OK) return st;
  if (n_segments > kMaxN) return MOE_ERR_UNSUPPORTED;
  if (!xp || !offsets || !op || !ws) return MOE_ERR_NULL;
  if (!aligned16(xp) || !aligned16(op) || !aligned16(ws)) return MOE_ERR_ALIGN;
  const FfnE4m3Layout L = ffn_e4m3_layout(rows_max, cfg->d, f);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  return run_ffn_e4m3(xp, offsets, n_segments, rows_max, cfg->d, f, *experts, at<void>(ws, L.hp),
                      at<uint8_t>(ws, L.xq), at<float>(ws, L.xs), at<uint8_t>(ws, L.hq),
                      at<float>(ws, L.hs), op, static_cast<int32_t*>(ws), as_stream(stream));
}

int moe_layer_stages(const moe_config* cfg, const char** names, int max_names) {
  const int st = validate(cfg, nullptr);
  if (st != MOE_OK) return st;
  if (max_names < 0) return MOE_ERR_SHAPE;
  return layer_stage_names(*cfg, names, max_names);
}

int moe_set_trace_events(void* const* events, int n_events) {
  if (n_events < 0 || n_events > kMaxTraceEvents) return MOE_ERR_SHAPE;
  if (n_events > 0 && !events) return MOE_ERR_NULL;
  for (int i = 0; i < n_events; ++i) g_trace_events[i] = static_cast<cudaEvent_t>(events[i]);
  g_trace_n = n_events;
  return MOE_OK;
}

int moe_workspace_views(const moe_config* cfg, void* ws, moe_views_t* out) {
  Derived d;
  int st = validate(cfg, &d);
  if (st != MOE_OK) return st;
  if (!ws || !out) return MOE_ERR_NULL;
  const Layout L = layout(*cfg, d);
  out->status = at<int32_t>(ws, L.ctrl);
  out->logits = at<float>(ws, L.logits);
  out->scores = at<float>(ws, L.scores);
  out->cand_idx = at<int32_t>(ws, L.cand_idx);
  out->cand_gate = at<float>(ws, L.cand_gate);
  out->slot = at<int32_t>(ws, L.slot);
  out->keep = at<uint8_t>(ws, L.keep);
  out->demand = at<int32_t>(ws, L.demand);
  out->kept = at<int32_t>(ws, L.kept);
  out->expert_offsets = at<int32_t>(ws, L.offsets);
  out->row_token = at<int32_t>(ws, L.row_token);
  out->row_gate = at<float>(ws, L.row_gate);
  out->tok_rows = at<int32_t>(ws, L.tok_rows);
  out->xp = at<void>(ws, L.xp);
  out->op = at<void>(ws, L.op);
  out->shared_out = cfg->f_shared > 0 ? at<void>(ws, L.shared_out) : nullptr;
  out->coverage = at<int32_t>(ws, L.coverage);
  return MOE_OK;
}

int moe_get_device_status(const void* ws, void* stream, int32_t* out_host) {
  if (!ws || !out_host) return MOE_ERR_NULL;
  cudaStream_t s = as_stream(stream);
  int32_t v = MOE_OK;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) *out_host = v;
  return status_from(e);
}

int moe_clear_device_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_NULL;
  clear_ctrl_kernel<<<1, 256, 0, as_stream(stream)>>>(static_cast<int32_t*>(ws));
  return status_from(cudaGetLastError());
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "a required pointer is NULL";
    case MOE_ERR_SHAPE: return "a size is out of range or inconsistent";
    case MOE_ERR_ALIGN: return "a pointer breaks the 16-byte alignment rule";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_UNSUPPORTED: return "configuration outside the implemented limits";
    case MOE_ERR_LAUNCH: return "the CUDA runtime refused a launch";
    case MOE_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait expired";
    case MOE_ERR_DEVICE_BOUNDS: return "a kernel saw an index outside its buffer";
    default: return "unknown status";
  }
}

void moe_release_caches(void) {}  // tensor maps are encoded per call; nothing is cached

}  // extern "C"
