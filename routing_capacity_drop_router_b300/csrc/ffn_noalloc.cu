// Expert FFN entry point that allocates nothing and takes no workspace.
//
// Some callers cannot hand this library a workspace: a host framework that
// owns all device memory and gives an operator only its input and output
// buffers, or a latency-critical loop where cudaMalloc (which may synchronise
// the device) is not allowed. For them the SwiGLU hidden activations between
// the two expert GEMMs live in a fixed-size array of device global memory that
// the library itself owns.
//
// The array is a file-scope __device__ variable. In host code its name is only
// a host-side stand-in, not a device address, so the entry point looks up the
// real address with cudaGetSymbolAddress once per device (with that device
// current) and passes that pointer to the kernels. The address belongs to the
// device's current context: the lookup is cached together with that context's
// unique id and repeated when the id changes (after cudaDeviceReset, or when
// the primary context was released and created again while the library stayed
// loaded), so a stale address is never handed to a kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {
namespace {

constexpr size_t kScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
constexpr size_t kStatusBytes = 256;  // status word, padded to keep h 256-byte aligned

// Held by every GPU that loads the library, until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
unsigned char* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx_id[kMaxDevices] = {};  // context the address belongs to

__global__ void clear_status_word_kernel(int32_t* status) { *status = 0; }

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The driver's context queries, reached through the runtime's entry-point
// lookup so the library does not link libcuda; NULL if unavailable.
void context_queries(CtxGetCurrentFn* cur, CtxGetIdFn* id) {
  static std::once_flag once;
  static CtxGetCurrentFn f_cur = nullptr;
  static CtxGetIdFn f_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  *cur = f_cur;
  *id = f_id;
}

// Unique id of the current context (0 when it cannot be read).
unsigned long long current_context_id() {
  CtxGetCurrentFn cur = nullptr;
  CtxGetIdFn id = nullptr;
  context_queries(&cur, &id);
  CUcontext ctx = nullptr;
  unsigned long long v = 0;
  if (!cur || !id || cur(&ctx) != CUDA_SUCCESS || !ctx || id(ctx, &v) != CUDA_SUCCESS) return 0;
  return v;
}

// Device address of the scratch array in the current device's current
// context. Looked up once per device and context; without a readable context
// id it is looked up on every call (the lookup allocates nothing).
cudaError_t scratch_address(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long ctx = current_context_id();
  if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx_id[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // also makes the context current
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<unsigned char*>(p);
    g_scratch_ctx_id[dev] = current_context_id();
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" int moe_expert_ffn_noalloc(const moe_config* cfg, const void* xp,
                                      const int32_t* offsets, int32_t n_segments,
                                      int64_t rows_max, int32_t f, const void* W1,
                                      const void* W3, const void* W2, void* op,
                                      int32_t* device_status, void* stream) {
  using namespace moe;
  if (!cfg) return MOE_ERR_NULL;
  if (cfg->dtype != MOE_BF16 && cfg->dtype != MOE_F32) return MOE_ERR_SHAPE;
  if (cfg->d <= 0 || f <= 0 || n_segments < 0 || rows_max < 0) return MOE_ERR_SHAPE;
  if (cfg->dtype == MOE_BF16 && (cfg->d % 64 || f % 64)) return MOE_ERR_SHAPE;
  if (n_segments > 256) return MOE_ERR_UNSUPPORTED;
  if (!xp || !offsets || !W1 || !W3 || !W2 || !op) return MOE_ERR_NULL;
  if (!aligned16(xp) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(op) ||
      (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u)))
    return MOE_ERR_ALIGN;
  const size_t sx = cfg->dtype == MOE_BF16 ? 2 : 4;
  const double need = static_cast<double>(rows_max) * static_cast<double>(f) * sx;
  if (need > static_cast<double>(kScratchBytes - kStatusBytes)) return MOE_ERR_WORKSPACE;

  unsigned char* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_LAUNCH;
  int32_t* status = device_status ? device_status : reinterpret_cast<int32_t*>(scratch);
  void* hp = scratch + kStatusBytes;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // The array keeps the previous call's contents, so the library's own status
  // word is cleared first. A caller's word is left alone: it may already hold
  // an earlier stage's error, and the first error recorded wins.
  cudaError_t e = cudaSuccess;
  if (!device_status) {
    clear_status_word_kernel<<<1, 1, 0, s>>>(status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return MOE_ERR_LAUNCH;
  }
  if (cfg->dtype == MOE_BF16) {
    e = launch_grouped_gemm_tc_bf16(xp, offsets, n_segments, rows_max, cfg->d, f, W1, W3, hp,
                                    true, status, s);
    if (e == cudaSuccess)
      e = launch_grouped_gemm_tc_bf16(hp, offsets, n_segments, rows_max, f, cfg->d, W2, nullptr,
                                      op, false, status, s);
  } else {
    e = launch_grouped_gemm_simt_f32(static_cast<const float*>(xp), offsets, n_segments, rows_max,
                                     cfg->d, f, static_cast<const float*>(W1),
                                     static_cast<const float*>(W3), static_cast<float*>(hp), true,
                                     s);
    if (e == cudaSuccess)
      e = launch_grouped_gemm_simt_f32(static_cast<const float*>(hp), offsets, n_segments,
                                       rows_max, f, cfg->d, static_cast<const float*>(W2),
                                       nullptr, static_cast<float*>(op), false, s);
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}
