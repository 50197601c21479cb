// C ABI entry points: argument validation on the host, then kernel launches on
// the caller's stream. Nothing here allocates, frees or synchronises.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_internal.cuh"

using namespace mla;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mla_status launch_status(cudaError_t e) {
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

bool heads_ok(int H) { return H >= 1 && H <= kMaxHeads; }

// The address a kernel uses for p: device or managed memory as it is, pinned
// host memory through its mapped device address; false for memory the device
// cannot address (pageable host memory) or when the runtime cannot tell.
bool device_address(const void* p, const void** out) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *out = p;
    return true;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer) {
    // the same offset inside the allocation
    *out = static_cast<const char*>(a.devicePointer) +
           (static_cast<const char*>(p) - static_cast<const char*>(a.hostPointer));
    return true;
  }
  return false;
}

}  // namespace

extern "C" {

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED_SHAPE: return "MLA_ERR_UNSUPPORTED_SHAPE";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "MLA_ERR_WORKSPACE_TOO_SMALL";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_BOUNDS: return "MLA_ERR_BOUNDS";
    case MLA_ERR_RANGE: return "MLA_ERR_RANGE";
    default: return "MLA_ERR_UNKNOWN";
  }
}

int mla_abi_version(void) { return MLA_ABI_VERSION; }

size_t mla_cache_bytes_per_token(int d_c, int d_r) {
  if (d_c < 0 || d_r < 0) return 0;
  return (size_t)(d_c + d_r) * 2u;
}

size_t mla_page_bytes(int page_size, int d_c, int d_r) {
  if (page_size < 0) return 0;
  return (size_t)page_size * mla_cache_bytes_per_token(d_c, d_r);
}

mla_status mla_absorb_q(const uint16_t* q_nope, const uint16_t* q_rope, const uint16_t* w_uk,
                        uint16_t* q_abs, int T, int H, int d_nope, int d_r, int d_c, void* stream) {
  if (!q_nope || !q_rope || !w_uk || !q_abs) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(q_abs))
    return MLA_ERR_INVALID_ARG;
  if (T < 1) return MLA_ERR_INVALID_ARG;
  if (d_nope != kDNope || d_r != kDR || d_c != kDC || !heads_ok(H)) return MLA_ERR_UNSUPPORTED_SHAPE;
  return launch_status(launch_absorb_q(q_nope, q_rope, w_uk, q_abs, T, H, (cudaStream_t)stream));
}

mla_status mla_merge_w_kq(const uint16_t* w_uq, const uint16_t* w_uk, uint16_t* w_kq, int d_q, int H, int d_nope,
                          int d_c, void* stream) {
  if (!w_uq || !w_uk || !w_kq) return MLA_ERR_INVALID_ARG;
  if (!aligned16(w_uq) || !aligned16(w_uk) || !aligned16(w_kq)) return MLA_ERR_INVALID_ARG;
  if (d_q < 1) return MLA_ERR_INVALID_ARG;
  if (d_nope != kDNope || d_c != kDC || !heads_ok(H) || d_q % 64 != 0 || d_q > 16384)
    return MLA_ERR_UNSUPPORTED_SHAPE;
  return launch_status(launch_merge_w_kq(w_uq, w_uk, w_kq, d_q, H, (cudaStream_t)stream));
}

mla_status mla_absorb_q_latent(const uint16_t* c_q, const uint16_t* q_rope, const uint16_t* w_kq, uint16_t* q_abs,
                               int T, int H, int d_q, int d_r, int d_c, void* stream) {
  if (!c_q || !q_rope || !w_kq || !q_abs) return MLA_ERR_INVALID_ARG;
  if (!aligned16(c_q) || !aligned16(q_rope) || !aligned16(w_kq) || !aligned16(q_abs)) return MLA_ERR_INVALID_ARG;
  if (T < 1 || d_q < 1) return MLA_ERR_INVALID_ARG;
  if (d_r != kDR || d_c != kDC || !heads_ok(H) || d_q % 64 != 0 || d_q > 16384) return MLA_ERR_UNSUPPORTED_SHAPE;
  return launch_status(launch_absorb_latent(c_q, q_rope, w_kq, q_abs, T, H, d_q, (cudaStream_t)stream));
}

namespace {
bool comb_shape_ok(int H, int d_model) { return heads_ok(H) && d_model % 128 == 0 && d_model >= 128 && d_model <= 65536; }
}  // namespace

mla_status mla_merge_w_comb(const uint16_t* w_uv, const uint16_t* w_o, uint16_t* w_comb, int H, int d_v, int d_c,
                            int d_model, void* stream) {
  if (!w_uv || !w_o || !w_comb) return MLA_ERR_INVALID_ARG;
  if (!aligned16(w_uv) || !aligned16(w_o) || !aligned16(w_comb)) return MLA_ERR_INVALID_ARG;
  if (d_model < 1) return MLA_ERR_INVALID_ARG;
  if (d_v != kDV || d_c != kDC || !comb_shape_ok(H, d_model)) return MLA_ERR_UNSUPPORTED_SHAPE;
  // w_comb[n][h][c] = sum_v w_o[n][h][v] w_uv[h][v][c]: the absorption kernel with
  // the rows of w_o in place of query rows and w_uv in place of w_uk
  return launch_status(launch_merge_w_kq(w_o, w_uv, w_comb, d_model, H, (cudaStream_t)stream));
}

size_t mla_out_comb_workspace_bytes(int T, int H, int d_model) {
  if (T < 1 || T > 2 * MLA_MAX_BATCH || !comb_shape_ok(H, d_model)) return 0;
  return out_comb_workspace_bytes(T, H, d_model);
}

mla_status mla_out_comb(const uint16_t* u, const uint16_t* w_comb, uint16_t* out, int T, int H, int d_c, int d_model,
                        void* workspace, size_t workspace_bytes, void* stream) {
  if (!u || !w_comb || !out || !workspace) return MLA_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(w_comb) || !aligned16(out) || !aligned16(workspace)) return MLA_ERR_INVALID_ARG;
  if (T < 1 || d_model < 1) return MLA_ERR_INVALID_ARG;
  if (T > 2 * MLA_MAX_BATCH || d_c != kDC || !comb_shape_ok(H, d_model)) return MLA_ERR_UNSUPPORTED_SHAPE;
  if (workspace_bytes < out_comb_workspace_bytes(T, H, d_model)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  return launch_status(launch_out_comb(u, w_comb, out, T, H, d_model, workspace, (cudaStream_t)stream));
}

int mla_decode_default_splits(int n_q) {
  if (n_q < 1) return -1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  // one wave of worker clusters, shared by the n_q query indices
  int workers = decode_max_workers();
  if (workers < 1) workers = sms / 2;
  int g = workers / n_q;
  return g < 1 ? 1 : g;
}

size_t mla_decode_workspace_bytes(int B, int n_q, int H, int num_splits) {
  if (B < 1 || B > MLA_MAX_BATCH || n_q < 1 || n_q > 2 || !heads_ok(H) || num_splits < 1) return 0;
  return plan_layout(nullptr, B, n_q, H, num_splits, nullptr);
}

namespace {
// the checks shared by the decode entry points; fills `plan` on success
mla_status decode_args(void* workspace, size_t workspace_bytes, int B, int n_q, int H, int num_pages,
                       int page_size, int max_pages_per_seq, int num_splits, Plan* plan) {
  if (!workspace || !aligned16(workspace)) return MLA_ERR_INVALID_ARG;
  if (B < 1 || num_pages < 1 || max_pages_per_seq < 1 || num_splits < 1) return MLA_ERR_INVALID_ARG;
  if (B > MLA_MAX_BATCH || n_q < 1 || n_q > 2 || !heads_ok(H) || !page_size_ok(page_size))
    return MLA_ERR_UNSUPPORTED_SHAPE;
  if (!token_counts_ok(num_pages, page_size, max_pages_per_seq)) return MLA_ERR_UNSUPPORTED_SHAPE;
  const size_t need = plan_layout(nullptr, B, n_q, H, num_splits, nullptr);
  if (workspace_bytes < need) return MLA_ERR_WORKSPACE_TOO_SMALL;
  plan_layout(workspace, B, n_q, H, num_splits, plan);
  return MLA_OK;
}
}  // namespace

mla_status mla_decode_paged(const uint16_t* q_abs, const uint16_t* cache,
                            const int32_t* block_table, const int32_t* seq_lens,
                            int B, int n_q, int H, int num_pages, int page_size,
                            int max_pages_per_seq, float softmax_scale, int num_splits,
                            void* workspace, size_t workspace_bytes, int32_t* err_word,
                            void* stream) {
  if (!q_abs || !cache || !block_table || !seq_lens) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_abs) || !aligned16(cache) || !aligned16(block_table) || !aligned16(seq_lens))
    return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return MLA_ERR_INVALID_ARG;
  Plan plan;
  mla_status st = decode_args(workspace, workspace_bytes, B, n_q, H, num_pages, page_size, max_pages_per_seq,
                              num_splits, &plan);
  if (st != MLA_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  st = launch_status(launch_plan(seq_lens, block_table, B, n_q, max_pages_per_seq, page_size, num_pages, num_splits,
                                 plan, err_word, s));
  if (st != MLA_OK) return st;
  return launch_status(launch_decode(q_abs, cache, block_table, B, n_q, H, num_pages, page_size,
                                     max_pages_per_seq, softmax_scale, num_splits, plan, err_word, s));
}

mla_status mla_quantize_fp8(const uint16_t* rows, const float* scales, uint8_t* codes, int64_t n_rows,
                            void* stream) {
  if (!rows || !scales || !codes) return MLA_ERR_INVALID_ARG;
  if (!aligned16(rows) || !aligned16(scales) || !aligned16(codes)) return MLA_ERR_INVALID_ARG;
  if (n_rows < 1 || n_rows > ((int64_t)1 << 40)) return MLA_ERR_INVALID_ARG;
  return launch_status(launch_quantize_fp8(rows, scales, codes, n_rows, (cudaStream_t)stream));
}

mla_status mla_decode_paged_fp8(const uint16_t* q_abs, const uint8_t* cache8, const float* scales,
                                const int32_t* block_table, const int32_t* seq_lens, int B, int n_q, int H,
                                int num_pages, int page_size, int max_pages_per_seq, float softmax_scale,
                                int num_splits, void* workspace, size_t workspace_bytes, int32_t* err_word,
                                void* stream) {
  if (!q_abs || !cache8 || !scales || !block_table || !seq_lens) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_abs) || !aligned16(cache8) || !aligned16(scales) || !aligned16(block_table) ||
      !aligned16(seq_lens))
    return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return MLA_ERR_INVALID_ARG;
  Plan plan;
  mla_status st = decode_args(workspace, workspace_bytes, B, n_q, H, num_pages, page_size, max_pages_per_seq,
                              num_splits, &plan);
  if (st != MLA_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  st = launch_status(launch_plan(seq_lens, block_table, B, n_q, max_pages_per_seq, page_size, num_pages, num_splits,
                                 plan, err_word, s));
  if (st != MLA_OK) return st;
  return launch_status(launch_decode_fp8(q_abs, cache8, scales, block_table, B, n_q, H, num_pages, page_size,
                                         max_pages_per_seq, softmax_scale, num_splits, plan, err_word, s));
}

mla_status mla_decode_paged_planned_fp8(const uint16_t* q_abs, const uint8_t* cache8, const float* scales,
                                        const int32_t* block_table, int B, int n_q, int H, int num_pages,
                                        int page_size, int max_pages_per_seq, float softmax_scale, int num_splits,
                                        void* workspace, size_t workspace_bytes, int32_t* err_word, void* stream) {
  if (!q_abs || !cache8 || !scales || !block_table) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_abs) || !aligned16(cache8) || !aligned16(scales) || !aligned16(block_table))
    return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return MLA_ERR_INVALID_ARG;
  Plan plan;
  mla_status st = decode_args(workspace, workspace_bytes, B, n_q, H, num_pages, page_size, max_pages_per_seq,
                              num_splits, &plan);
  if (st != MLA_OK) return st;
  return launch_status(launch_decode_fp8(q_abs, cache8, scales, block_table, B, n_q, H, num_pages, page_size,
                                         max_pages_per_seq, softmax_scale, num_splits, plan, err_word,
                                         (cudaStream_t)stream));
}

mla_status mla_decode_plan(const int32_t* seq_lens, int B, int n_q, int H, int num_pages, int page_size,
                           int max_pages_per_seq, int num_splits, void* workspace, size_t workspace_bytes,
                           int32_t* err_word, void* stream) {
  if (!seq_lens || !aligned16(seq_lens)) return MLA_ERR_INVALID_ARG;
  Plan plan;
  mla_status st = decode_args(workspace, workspace_bytes, B, n_q, H, num_pages, page_size, max_pages_per_seq,
                              num_splits, &plan);
  if (st != MLA_OK) return st;
  return launch_status(launch_plan(seq_lens, nullptr, B, n_q, max_pages_per_seq, page_size, num_pages, num_splits,
                                   plan, err_word, (cudaStream_t)stream));
}

mla_status mla_decode_paged_planned(const uint16_t* q_abs, const uint16_t* cache, const int32_t* block_table,
                                    int B, int n_q, int H, int num_pages, int page_size, int max_pages_per_seq,
                                    float softmax_scale, int num_splits, void* workspace, size_t workspace_bytes,
                                    int32_t* err_word, void* stream) {
  if (!q_abs || !cache || !block_table) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_abs) || !aligned16(cache) || !aligned16(block_table)) return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return MLA_ERR_INVALID_ARG;
  Plan plan;
  mla_status st = decode_args(workspace, workspace_bytes, B, n_q, H, num_pages, page_size, max_pages_per_seq,
                              num_splits, &plan);
  if (st != MLA_OK) return st;
  return launch_status(launch_decode(q_abs, cache, block_table, B, n_q, H, num_pages, page_size, max_pages_per_seq,
                                     softmax_scale, num_splits, plan, err_word, (cudaStream_t)stream));
}

mla_status mla_combine(const void* workspace, int B, int n_q, int H, int num_splits, uint16_t* u,
                       float* lse, void* stream) {
  if (!workspace || !u) return MLA_ERR_INVALID_ARG;
  if (!aligned16(workspace) || !aligned16(u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || num_splits < 1) return MLA_ERR_INVALID_ARG;
  if (B > MLA_MAX_BATCH || n_q < 1 || n_q > 2 || !heads_ok(H)) return MLA_ERR_UNSUPPORTED_SHAPE;
  // lse may be pinned host memory, written over the host link
  const void* lse_dev = nullptr;
  if (lse && !device_address(lse, &lse_dev)) return MLA_ERR_INVALID_ARG;
  Plan plan;
  plan_layout(const_cast<void*>(workspace), B, n_q, H, num_splits, &plan);
  return launch_status(launch_combine(plan, B, n_q, H, u, static_cast<float*>(const_cast<void*>(lse_dev)),
                                      (cudaStream_t)stream));
}

mla_status mla_out_proj(const uint16_t* u, const uint16_t* w_uv, uint16_t* out, int T, int H,
                        int d_c, int d_v, void* stream) {
  if (!u || !w_uv || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(w_uv) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
  if (T < 1) return MLA_ERR_INVALID_ARG;
  if (d_c != kDC || d_v != kDV || !heads_ok(H)) return MLA_ERR_UNSUPPORTED_SHAPE;
  // out may be pinned host memory, written over the host link
  const void* out_dev = nullptr;
  if (!device_address(out, &out_dev)) return MLA_ERR_INVALID_ARG;
  return launch_status(launch_out_proj(u, w_uv, static_cast<uint16_t*>(const_cast<void*>(out_dev)), T, H,
                                       (cudaStream_t)stream));
}

mla_status mla_copy16(const void* src, void* dst, size_t bytes, void* stream) {
  if (!src || !dst || bytes == 0 || bytes % 16 != 0) return MLA_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return MLA_ERR_INVALID_ARG;
  const void* s_dev = nullptr;
  const void* d_dev = nullptr;
  if (!device_address(src, &s_dev) || !device_address(dst, &d_dev)) return MLA_ERR_INVALID_ARG;
  return launch_status(launch_copy16(s_dev, const_cast<void*>(d_dev), bytes, (cudaStream_t)stream));
}

size_t mla_append_workspace_bytes(int T, int d_model) {
  if (T < 1 || T > 2 * MLA_MAX_BATCH || d_model < 64 || d_model % 64 != 0 || d_model > 65536) return 0;
  return append_workspace_bytes(T, d_model);
}

mla_status mla_append_kv(const uint16_t* h, const uint16_t* w_dkr, uint16_t* cache, const int32_t* block_table,
                         const int32_t* seq_lens, int B, int n_q, int d_model, int num_pages, int page_size,
                         int max_pages_per_seq, float rope_theta, void* workspace, size_t workspace_bytes,
                         int32_t* err_word, void* stream) {
  if (!h || !w_dkr || !cache || !block_table || !seq_lens || !workspace) return MLA_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w_dkr) || !aligned16(cache) || !aligned16(block_table) || !aligned16(seq_lens) ||
      !aligned16(workspace))
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || num_pages < 1 || max_pages_per_seq < 1) return MLA_ERR_INVALID_ARG;
  if (!(rope_theta > 1.f) || rope_theta != rope_theta) return MLA_ERR_INVALID_ARG;
  if (B > MLA_MAX_BATCH || n_q < 1 || n_q > 2 || !page_size_ok(page_size)) return MLA_ERR_UNSUPPORTED_SHAPE;
  if (d_model < 64 || d_model % 64 != 0 || d_model > 65536) return MLA_ERR_UNSUPPORTED_SHAPE;
  if (!token_counts_ok(num_pages, page_size, max_pages_per_seq)) return MLA_ERR_UNSUPPORTED_SHAPE;
  if (workspace_bytes < append_workspace_bytes(B * n_q, d_model)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  return launch_status(launch_append(h, w_dkr, cache, block_table, seq_lens, B, n_q, d_model, num_pages, page_size,
                                     max_pages_per_seq, (double)rope_theta, workspace, err_word,
                                     (cudaStream_t)stream));
}

}  // extern "C"
