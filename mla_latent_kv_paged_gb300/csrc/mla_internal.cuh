// Internal declarations shared by the CUDA translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <stdint.h>

#include <utility>

#include "../../include/mla.h"

namespace mla {

constexpr int kDNope = 128;
constexpr int kDR = 64;
constexpr int kDC = 512;
constexpr int kDV = 128;
constexpr int kRow = kDC + kDR;  // 576 values per cached token
constexpr int kTile = 64;  // tokens per tile, the decode kernel's unit; a page holds 1 or 2 tiles
constexpr int kMaxHeads = 128;

// ---------------------------------------------------------------- workspace
// Views into the caller's workspace; the layout is documented in mla.h.
struct Plan {
  int32_t* hdr;          // [64]
  int32_t* range_item;   // [G + 1]
  int32_t* seq_item;     // [B + 1]
  int32_t* seq_len_eff;  // [B]
  int32_t* item_seq;     // [I]
  int32_t* item_tile0;   // [I] first tile (64 tokens) of the piece within its sequence
  int32_t* item_tile1;   // [I] end tile (exclusive)
  float* lse_part;       // [I][n_q][H]
  uint16_t* o_part;      // [I][n_q][64][H][8] fp16, head-minor
  int4* range_desc;      // [G + 1] {first item, its sequence, its first tile, its end tile}
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Returns the total size; fills `p` relative to `base` when base != nullptr.
__host__ __device__ inline size_t plan_layout(void* base, int B, int n_q, int H, int G, Plan* p) {
  const size_t I = (size_t)G + (size_t)B;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  size_t o_hdr = take(64 * 4);
  size_t o_ri = take((size_t)(G + 1) * 4);
  size_t o_si = take((size_t)(B + 1) * 4);
  size_t o_sl = take((size_t)B * 4);
  size_t o_is = take(I * 4);
  size_t o_p0 = take(I * 4);
  size_t o_p1 = take(I * 4);
  size_t o_lse = take(I * n_q * H * 4);
  size_t o_o = take(I * n_q * H * (size_t)kDC * 2);
  size_t o_rd = take((size_t)(G + 1) * 16);
  if (base && p) {
    char* c = reinterpret_cast<char*>(base);
    p->hdr = reinterpret_cast<int32_t*>(c + o_hdr);
    p->range_item = reinterpret_cast<int32_t*>(c + o_ri);
    p->seq_item = reinterpret_cast<int32_t*>(c + o_si);
    p->seq_len_eff = reinterpret_cast<int32_t*>(c + o_sl);
    p->item_seq = reinterpret_cast<int32_t*>(c + o_is);
    p->item_tile0 = reinterpret_cast<int32_t*>(c + o_p0);
    p->item_tile1 = reinterpret_cast<int32_t*>(c + o_p1);
    p->lse_part = reinterpret_cast<float*>(c + o_lse);
    p->o_part = reinterpret_cast<uint16_t*>(c + o_o);
    p->range_desc = reinterpret_cast<int4*>(c + o_rd);
  }
  return off;
}

// ---------------------------------------------------------------- device helpers
__device__ inline void report_error(int32_t* err_word, int code) {
  if (err_word) atomicCAS(err_word, 0, code);
}

__device__ inline float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ inline float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ inline float bf16_to_float(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// float -> bf16 round-to-nearest-even (finite inputs; NaN stays NaN).
__device__ inline uint16_t float_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
__device__ inline uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)float_to_bf16(lo) | ((uint32_t)float_to_bf16(hi) << 16);
}

// ---------------------------------------------------------------- tensor maps
// bf16 (or, with u8, 8-bit) tensor map of `rank` dims (dims[0] innermost), byte
// strides of dims 1..rank-1, box extents, swizzle span in bytes (0, 32, 64 or 128).
bool make_tmap(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
               const uint32_t* box, int swizzle_bytes, bool u8 = false);

// ---------------------------------------------------------------- launch helper
// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel of the stream finishes; it must execute
// griddepcontrol.wait before reading anything that kernel (or earlier work)
// produced.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- shared memory limit
// Raises a kernel's dynamic shared memory limit once per device (the attribute
// belongs to the device that is current; a process may drive several).
template <auto Kernel>
cudaError_t smem_limit(size_t bytes) {
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> done[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && cached) done[dev].store(true, std::memory_order_release);
  return e;
}

// ---------------------------------------------------------------- launchers
// overlap: start beside the kernel enqueued before (programmatic dependent
// launch); it then reads seq_lens and writes the plan while that kernel runs.
// page_size: 64 or 128 tokens (1 or 2 tiles per block-table entry)
inline bool page_size_ok(int page_size) { return page_size == kTile || page_size == 2 * kTile; }
// sizes in tokens that stay in int32 (positions, and rows of the cache)
inline bool token_counts_ok(int num_pages, int page_size, int max_pages) {
  return (int64_t)max_pages * page_size <= INT32_MAX / 2 && (int64_t)num_pages * page_size <= INT32_MAX;
}
cudaError_t launch_plan(const int32_t* seq_lens, const int32_t* block_table, int B, int n_q,
                        int max_pages, int page_size, int num_pages, int G, const Plan& plan, int32_t* err_word,
                        cudaStream_t s, bool overlap = true);
cudaError_t launch_decode(const uint16_t* q_abs, const uint16_t* cache, const int32_t* block_table,
                          int B, int n_q, int H, int num_pages, int page_size, int max_pages, float scale, int G,
                          const Plan& plan, int32_t* err_word, cudaStream_t s);
// The same decode over an FP8 cache: e4m3 codes [num_pages][64][576] and one
// float scale per column (fp8_scales[576]).
cudaError_t launch_decode_fp8(const uint16_t* q_abs, const uint8_t* cache8, const float* fp8_scales,
                              const int32_t* block_table, int B, int n_q, int H, int num_pages, int page_size,
                              int max_pages, float scale, int G, const Plan& plan, int32_t* err_word,
                              cudaStream_t s);
// e4m3 codes of bf16 rows of 576 values with per-column scales
cudaError_t launch_quantize_fp8(const uint16_t* rows, const float* scales, uint8_t* codes, int64_t n_rows,
                                cudaStream_t s);
// Worker clusters (CTA pairs) of the decode kernel that fit on the device at once.
int decode_max_workers();
cudaError_t launch_combine(const Plan& plan, int B, int n_q, int H, uint16_t* u, float* lse,
                           cudaStream_t s);
cudaError_t launch_absorb_q(const uint16_t* q_nope, const uint16_t* q_rope, const uint16_t* w_uk,
                            uint16_t* q_abs, int T, int H, cudaStream_t s);
cudaError_t launch_out_proj(const uint16_t* u, const uint16_t* w_uv, uint16_t* out, int T, int H,
                            cudaStream_t s);
cudaError_t launch_merge_w_kq(const uint16_t* w_uq, const uint16_t* w_uk, uint16_t* w_kq, int d_q, int H,
                              cudaStream_t s);
size_t out_comb_workspace_bytes(int T, int H, int d_model);
cudaError_t launch_out_comb(const uint16_t* u, const uint16_t* w_comb, uint16_t* out, int T, int H, int d_model,
                            void* workspace, cudaStream_t s);
cudaError_t launch_absorb_latent(const uint16_t* c_q, const uint16_t* q_rope, const uint16_t* w_kq, uint16_t* q_abs,
                                 int T, int H, int d_q, cudaStream_t s);
size_t append_workspace_bytes(int T, int d_model);
// bytes (a multiple of 16) from src to dst, both device addresses (device
// memory, or pinned host memory through its device address)
cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, cudaStream_t s);
cudaError_t launch_append(const uint16_t* h, const uint16_t* w_dkr, uint16_t* cache, const int32_t* block_table,
                          const int32_t* seq_lens, int B, int n_q, int d_model, int num_pages, int page_size,
                          int max_pages, double theta, void* workspace, int32_t* err_word, cudaStream_t s);

}  // namespace mla
