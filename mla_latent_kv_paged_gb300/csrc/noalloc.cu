// Decode entry point that allocates nothing and needs no caller workspace.
//
// Some callers cannot hand this library a device buffer for the split-KV
// plan and partial results: a serving loop that reserves all device memory
// for the KV cache up front and never calls cudaMalloc afterwards (an
// allocation there can block on the device and stall every in-flight
// request), or host code driving the GPU through an interface that exposes
// only the model's own tensors. For them this file keeps the scratch in one
// file-scope device array of fixed size, reserved by the CUDA runtime on
// every device that loads the library and held until the process exits.
//
// The array's address is fetched once per device with cudaGetSymbolAddress
// (in host code the symbol names a host-side stand-in, not device memory).
// That happens on the first call made with each device current, so the
// first call on a device should come before any stream capture. The address
// belongs to the device's context: it is kept together with the context's
// unique id, and a call made under another context (for example after
// cudaDeviceReset, which replaces the primary context and reloads the
// library's device code elsewhere) fetches it again, which again must happen
// outside stream capture. All calls share the one array: two calls whose
// kernels overlap on the GPU (different streams, or different host threads)
// race on it and give wrong results. Nothing in the array needs to start at
// zero: the plan kernel writes every entry the later kernels read.
#include <cudaTypedefs.h>

#include <mutex>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
struct ScratchEntry {
  unsigned long long ctx_id;  // unique id of the context the address belongs to (never reused)
  void* ptr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

// Unique id of the current context, through driver entry points fetched by the
// runtime (no link-time dependency on the driver library).
cudaError_t current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (!ctx) return cudaErrorContextIsDestroyed;  // none current on this thread yet
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of the scratch array in the current device's context
// (looked up on the first call under each context).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  unsigned long long id = 0;
  e = current_context_id(&id);
  const bool no_context = e == cudaErrorContextIsDestroyed;
  if (e != cudaSuccess && !no_context) return e;
  if (no_context || !g_scratch[dev].ptr || g_scratch[dev].ctx_id != id) {
    // the lookup also makes the device's primary context current if none is
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (no_context) {
      e = current_context_id(&id);
      if (e != cudaSuccess) return e;
    }
    g_scratch[dev] = ScratchEntry{id, p};
  }
  *out = g_scratch[dev].ptr;
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

size_t mla_decode_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

mla_status mla_decode_noalloc(const uint16_t* q_abs, const uint16_t* cache, const int32_t* block_table,
                              const int32_t* seq_lens, int B, int n_q, int H, int num_pages, int page_size,
                              int max_pages_per_seq, float softmax_scale, int num_splits, uint16_t* u, float* lse,
                              int32_t* err_word, void* stream) {
  if (!q_abs || !cache || !block_table || !seq_lens || !u) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_abs) || !aligned16(cache) || !aligned16(block_table) || !aligned16(seq_lens) || !aligned16(u) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || num_pages < 1 || max_pages_per_seq < 1 || num_splits < 1) return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return MLA_ERR_INVALID_ARG;
  if (B > MLA_MAX_BATCH || n_q < 1 || n_q > 2 || H < 1 || H > kMaxHeads || !page_size_ok(page_size))
    return MLA_ERR_UNSUPPORTED_SHAPE;
  if (!token_counts_ok(num_pages, page_size, max_pages_per_seq)) return MLA_ERR_UNSUPPORTED_SHAPE;
  // the plan and partials of this call must fit the fixed array
  if (plan_layout(nullptr, B, n_q, H, num_splits, nullptr) > kNoAllocScratchBytes)
    return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  Plan plan;
  plan_layout(scratch, B, n_q, H, num_splits, &plan);
  cudaStream_t s = (cudaStream_t)stream;
  // the plan waits for the kernel before it: that may be the previous call's
  // merge, still reading the plan in the shared array
  cudaError_t e = launch_plan(seq_lens, block_table, B, n_q, max_pages_per_seq, page_size, num_pages, num_splits,
                              plan, err_word, s, /*overlap=*/false);
  if (e == cudaSuccess)
    e = launch_decode(q_abs, cache, block_table, B, n_q, H, num_pages, page_size, max_pages_per_seq, softmax_scale,
                      num_splits, plan, err_word, s);
  if (e == cudaSuccess) e = launch_combine(plan, B, n_q, H, u, lse, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

}  // extern "C"
