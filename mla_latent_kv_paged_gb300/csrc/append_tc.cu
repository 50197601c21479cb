// Latent-cache append: the cache row of each new token, written into its page.
//
// What it computes (Huny's Dev Blog "MLA 아키텍처 해부" section 1.2, the joint
// low-rank compression c_t^KV = h_t W^DKV, and section 2.2, the decoupled
// positional key k^R_t = RoPE(h_t W^KR), shared by all heads and cached
// already rotated): for new row t = b * n_q + j at position pos = L_b - n_q + j,
//   row[i] = sum_k h[t][k] w_dkr[i][k]            i < 576 (w_dkr rows: W^DKV^T ; W^KR^T)
//   (row[512 + 2i], row[513 + 2i]) rotated by pos * theta^(-2i / 64)
// and row goes to cache[block_table[b][pos / 64]][pos % 64][0:576] as bf16.
//
// A weight-streaming GEMM at decode sizes (576 x d_model weights, T rows), so
// the reduction over d_model is split across CTAs: CTA (m, s, tile) of the
// first kernel multiplies output columns [128m, 128m + 128) by its slice of
// d_model on the tensor cores (tcgen05, D in tensor memory) and writes an fp32
// partial. The second kernel (one CTA per row, a thread per column pair) adds
// the partials in split order, so the sums are reproducible bit for bit,
// rotates the positional pairs and scatters the rows into their pages.
#include <math.h>

#include "mla_internal.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kThreads = 128;
constexpr int kMTiles = 5;               // 576 output columns in tiles of 128 (the last one half used)
constexpr int kPartCols = kMTiles * 128;  // 640
constexpr uint32_t kABox = 128 * 128;     // [128 rows][64 bf16], 128B swizzle
constexpr uint32_t kSmemBudget = 200 * 1024;

struct AppendShape {
  int NT, tiles, KB, S, max_kb;
};

__host__ __device__ inline int nt_for(int T) { return T <= 32 ? 32 : T <= 64 ? 64 : 128; }

// Splits of the d_model reduction: at most kTargetSplits, each at most max_kb
// 64-wide boxes (shared-memory budget). A function of (T, d_model) only.
__host__ __device__ inline AppendShape append_shape(int T, int d_model) {
  AppendShape a;
  a.NT = nt_for(T);
  a.tiles = (T + a.NT - 1) / a.NT;
  a.KB = d_model / 64;
  a.max_kb = (int)(kSmemBudget / (kABox + (uint32_t)a.NT * 128));
  const int kTargetSplits = 30;
  int S = a.KB < kTargetSplits ? a.KB : kTargetSplits;
  const int need = (a.KB + a.max_kb - 1) / a.max_kb;
  a.S = S > need ? S : need;
  return a;
}

__host__ __device__ inline size_t append_ws_bytes(int T, int d_model) {
  const AppendShape a = append_shape(T, d_model);
  return (size_t)a.tiles * a.S * a.NT * kPartCols * 4;
}

template <int kNT>
__global__ void __launch_bounds__(kThreads, 1)
append_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_h,
                   int d_model, float* __restrict__ partials, int S, int32_t* err_word) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x, s = blockIdx.y, tile = blockIdx.z;
  const int KB = d_model / 64;
  const int kb0 = (int)((int64_t)s * KB / S), kb1 = (int)((int64_t)(s + 1) * KB / S), nkb = kb1 - kb0;
  constexpr uint32_t kBBox = kNT * 128;
  const uint32_t off_b = (uint32_t)nkb * kABox;
  const uint32_t off_bar = off_b + (uint32_t)nkb * kBBox;
  const uint32_t bar_ld = sbase + off_bar, bar_d = bar_ld + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + off_bar + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + off_bar + 20);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) report_error(err_word, MLA_ERR_CUDA);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_d, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_w);
    prefetch_tmap(&map_h);
    // this CTA's weights into shared memory while the previous kernel finishes
    // (weights are never its output); the hidden states follow after the wait
    mbar_arrive_expect_tx(bar_ld, (uint32_t)nkb * (kABox + kNT * 128));
    const uint64_t pol = policy_evict_first();
    for (int k = 0; k < nkb; ++k) tma_load_2d(sbase + k * kABox, &map_w, bar_ld, (kb0 + k) * 64, m * 128, pol);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kNT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // h belongs to the previous kernel
  grid_dependency_wait();
  grid_launch_dependents();

  bool ok = true;
  if (threadIdx.x == 0) {
    const uint64_t pol = policy_evict_first();
    for (int k = 0; k < nkb; ++k)
      tma_load_2d(sbase + off_b + k * kBBox, &map_h, bar_ld, (kb0 + k) * 64, tile * kNT, pol);
    ok = wait_phase(bar_ld, 0, abort_flag, err_word);
    if (ok) {
      tc_fence_after();
      auto da = [](uint32_t addr) -> uint64_t { return (uint64_t)((addr >> 4) & 0x3FFFu); };
      const uint32_t idesc = idesc_bf16(128, kNT, false, false);
      const uint64_t adesc = smem_desc(0, 16, 1024, kSwizzle128B) + da(sbase);
      const uint64_t bdesc = smem_desc(0, 16, 1024, kSwizzle128B) + da(sbase + off_b);
      for (int k = 0; k < nkb; ++k)
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          mma_ss(tmem, adesc + ((k * kABox + k4 * 32) >> 4), bdesc + ((k * kBBox + k4 * 32) >> 4), idesc,
                 (k > 0 || k4 > 0) ? 1u : 0u);
    }
    mma_commit(bar_d);
  }
  __syncwarp();
  if (wait_phase(bar_d, 0, abort_flag, err_word)) {
    tc_fence_after();
    // D: lane = output column 128m + 32warp + lane, tensor-memory columns = rows
    const int col = m * 128 + warp * 32 + lane;
    float* part = partials + ((size_t)(tile * S + s) * kNT) * kPartCols + col;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int c0 = 0; c0 < kNT; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(taddr + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int v = 0; v < 32; ++v) part[(size_t)(c0 + v) * kPartCols] = __uint_as_float(r[v]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kNT);
  }
  (void)ok;
}

// Row t of the new tokens: the split partials added in order, the positional
// pairs rotated, the row written into its page. Thread c handles columns 2c
// and 2c + 1 (a positional pair when 2c >= 512).
__global__ void __launch_bounds__(kRow / 2)
append_finalize_kernel(const float* __restrict__ partials, uint16_t* __restrict__ cache,
                       const int32_t* __restrict__ block_table, const int32_t* __restrict__ seq_lens, int T,
                       int n_q, int num_pages, int page_size, int max_pages, double theta, int NT, int S,
                       int32_t* err_word) {
  const int t = blockIdx.x, c = threadIdx.x, col = 2 * c;
  const int b = t / n_q, j = t % n_q;
  // independent of the partials: overlaps the GEMM kernel
  const int raw = seq_lens[b];
  const int max_tokens = max_pages * page_size;
  const int L = raw < n_q ? n_q : (raw > max_tokens ? max_tokens : raw);
  const int pos = L - n_q + j;
  const int page = block_table[(size_t)b * max_pages + pos / page_size];
  const double inv_freq = col >= kDC ? pow(theta, -2.0 * (double)((col - kDC) >> 1) / kDR) : 0.0;
  sm100::grid_dependency_wait();  // the partials come from the GEMM kernel
  sm100::grid_launch_dependents();
  const float2* p = reinterpret_cast<const float2*>(partials + ((size_t)(t / NT) * S * NT + t % NT) * kPartCols + col);
  // the partials of up to 32 splits in flight at once (one L2 round trip for the
  // usual split counts), added in split order
  float x = 0.f, y = 0.f;
  constexpr int kInFlight = 32;
  for (int s0 = 0; s0 < S; s0 += kInFlight) {
    float2 v[kInFlight];
#pragma unroll
    for (int k = 0; k < kInFlight; ++k)
      if (s0 + k < S) v[k] = __ldcg(p + (size_t)(s0 + k) * NT * kPartCols / 2);
#pragma unroll
    for (int k = 0; k < kInFlight; ++k)
      if (s0 + k < S) {
        x += v[k].x;
        y += v[k].y;
      }
  }
  if (col >= kDC) {
    // the angle pos * theta^(-2i/64), reduced to [-pi, pi] in double (positions
    // reach 10^5-10^6 rad, beyond fp32's resolution); sine, cosine and the
    // rotation in fp32
    const double ang = (double)pos * inv_freq;
    const double k = rint(ang * 0.15915494309189535);  // 1 / (2 pi)
    const float r = (float)fma(-k, 6.283185307179586, ang);
    float sn, cs;
    sincosf(r, &sn, &cs);
    const float rx = x * cs - y * sn, ry = x * sn + y * cs;
    x = rx;
    y = ry;
  }
  if (c == 0 && L != raw) report_error(err_word, MLA_ERR_BOUNDS);
  if (page < 0 || page >= num_pages) {
    if (c == 0) report_error(err_word, MLA_ERR_BOUNDS);
    return;
  }
  reinterpret_cast<uint32_t*>(cache + ((size_t)page * page_size + pos % page_size) * kRow)[c] = pack_bf16x2(x, y);
}

template <int kNT>
cudaError_t launch_gemm(const CUtensorMap& mw, const CUtensorMap& mh, int d_model, float* partials,
                        const AppendShape& a, int32_t* err_word, cudaStream_t s) {
  const int max_nkb = (a.KB + a.S - 1) / a.S;
  const size_t smem = (size_t)max_nkb * (kABox + kNT * 128) + 64;
  cudaError_t e = smem_limit<append_gemm_kernel<kNT>>(kSmemBudget + 1024);
  if (e != cudaSuccess) return e;
  const dim3 grid(kMTiles, a.S, a.tiles);
  return launch_pdl(append_gemm_kernel<kNT>, grid, dim3(kThreads), smem, s, mw, mh, d_model, partials, a.S,
                    err_word);
}

}  // namespace

size_t append_workspace_bytes(int T, int d_model) { return append_ws_bytes(T, d_model); }

cudaError_t launch_append(const uint16_t* h, const uint16_t* w_dkr, uint16_t* cache, const int32_t* block_table,
                          const int32_t* seq_lens, int B, int n_q, int d_model, int num_pages, int page_size,
                          int max_pages, double theta, void* workspace, int32_t* err_word, cudaStream_t s) {
  const int T = B * n_q;
  const AppendShape a = append_shape(T, d_model);
  CUtensorMap mw, mh;
  const uint64_t dw[2] = {(uint64_t)d_model, (uint64_t)kRow}, dh[2] = {(uint64_t)d_model, (uint64_t)T};
  const uint64_t st[1] = {(uint64_t)d_model * 2};
  const uint32_t bw[2] = {64, 128}, bh[2] = {64, (uint32_t)a.NT};
  if (!make_tmap(&mw, w_dkr, 2, dw, st, bw, 128) || !make_tmap(&mh, h, 2, dh, st, bh, 128))
    return cudaErrorInvalidValue;
  float* partials = reinterpret_cast<float*>(workspace);
  cudaError_t e = a.NT == 32   ? launch_gemm<32>(mw, mh, d_model, partials, a, err_word, s)
                  : a.NT == 64 ? launch_gemm<64>(mw, mh, d_model, partials, a, err_word, s)
                               : launch_gemm<128>(mw, mh, d_model, partials, a, err_word, s);
  if (e != cudaSuccess) return e;
  return launch_pdl(append_finalize_kernel, dim3(T), dim3(kRow / 2), 0, s, (const float*)partials, cache, block_table,
                    seq_lens, T, n_q, num_pages, page_size, max_pages, theta, a.NT, a.S, err_word);
}

}  // namespace mla
