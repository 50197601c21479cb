// Per-head projections on the tcgen05 tensor cores (bf16 in, fp32 accumulate
// in tensor memory, bf16 out). Both are weight-streaming GEMMs at decode batch
// sizes: every CTA keeps one head's weight slice resident in shared memory and
// multiplies it by the query rows of that head.
//
// absorb_q (Huny's Dev Blog "MLA 아키텍처 해부" section 3.1, qt = q^C (W^UK)^T):
//   D[c][t] = sum_i W_UK[h][i][c] q_nope[t][h][i]      M = 128 latent cols, N = rows t, K = 128
//   A = W_UK[h][:, c-block] read M-major, B = q_nope rows (K-major).
//   The rotated positional query is copied to columns 512..575.
//   The same kernel merges the query-side weight (ingu627.github.io "Multi-Head
//   Latent Attention (MLA)" section 2.2, W_KQ = W_UK^T W_UQ per head): the d_q
//   rows of the input-major W_UQ [d_q][H][128] take the place of query rows,
//   giving W_KQ [d_q][H][512] (rows of 512, no positional part).
// out_proj (section 3.2, u W^UV):
//   D[v][t] = sum_c W_UV[h][v][c] u[t][h][c]            M = 128 value cols, N = rows t, K = 512
//   A = W_UV[h] (K-major), B = u rows (K-major). Each 64-wide K slice has its
//   own barrier, so the MMAs of a slice start as soon as it lands.
// The absorb path also performs the value/output merge (Huny's Dev Blog
// section 3 item 2, W_comb = W^UV W^O per head): the rows of W_O
// [d_model][H][128] in place of query rows and W_UV (stored like W_UK) give
// W_comb [d_model][H][512].
// D sits in tensor memory with one lane per output column; the epilogue puts
// the [rows][128 columns] tile through shared memory and writes each output
// row as 16-byte stores. N (rows per tile) is 32, 64 or 128, the smallest
// that holds the batch's rows.
#include "mla_internal.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kThreads = 128;
constexpr uint32_t kBoxRows = 128;  // A boxes: 128 rows x 64 bf16

template <bool kAbsorb, int kNT>
struct ProjCfg {
  static constexpr int NT = kNT;                        // rows t per tile (MMA N)
  static constexpr int K = kAbsorb ? kDNope : kDC;      // reduction length
  static constexpr int KB = K / 64;                     // 64-wide K boxes
  static constexpr uint32_t kABox = kBoxRows * 128;     // 16 KB
  static constexpr uint32_t kBBox = NT * 128;
  static constexpr uint32_t kABytes = kAbsorb ? 2 * kABox : KB * kABox;
  static constexpr uint32_t kBBytes = KB * kBBox;
  static constexpr int kBars = kAbsorb ? 1 : KB;        // load barriers
  static constexpr uint32_t kOffA = 0, kOffB = kABytes, kOffBar = kABytes + kBBytes;
  static constexpr uint32_t kSmem = kOffBar + 8 * (kBars + 1) + 16;
  static constexpr uint32_t kTmCols = NT < 32 ? 32 : NT;
};

template <bool kAbsorb, int kNT>
__global__ void __launch_bounds__(kThreads, 1)
proj_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const uint16_t* __restrict__ weights, const uint16_t* __restrict__ q_rope, uint16_t* __restrict__ out,
               int T, int H, int out_row, int32_t* err_word) {
  using C = ProjCfg<kAbsorb, kNT>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, cblk = blockIdx.y;  // cblk: 128-column block of q_abs (absorb only)
  const uint32_t bar_ld = sbase + C::kOffBar, bar_d = bar_ld + 8 * C::kBars;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 8 * (C::kBars + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + 8 * (C::kBars + 1) + 4);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) report_error(err_word, MLA_ERR_CUDA);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kBars; ++i) mbar_init(bar_ld + 8 * i, 1);
    mbar_init(bar_d, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_a);
    prefetch_tmap(&map_b);
    // this CTA's weight tiles into shared memory while the previous kernel
    // finishes (weights are never that kernel's output); the activations
    // follow after the grid dependency wait on the same barriers
    const uint64_t pol = policy_evict_first();
    if (kAbsorb) {
      mbar_arrive_expect_tx(bar_ld, C::kABytes + C::kBBytes);
      for (int m = 0; m < 2; ++m)  // W_UK[h][i][c] as boxes of [128 i][64 c]: this block's two halves
        tma_load_3d(sbase + C::kOffA + m * C::kABox, &map_a, bar_ld, cblk * 128 + m * 64, 0, h, pol);
    } else {
      for (int kb = 0; kb < C::KB; ++kb) {
        mbar_arrive_expect_tx(bar_ld + 8 * kb, C::kABox + C::kBBox);
        tma_load_3d(sbase + C::kOffA + kb * C::kABox, &map_a, bar_ld + 8 * kb, kb * 64, 0, h, pol);
      }
    }
  }
  // absorb_q: the next kernel (the decode kernel) may start now; it reads this
  // kernel's output only after its own dependency wait
  if (kAbsorb) grid_launch_dependents();
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything above overlaps the previous kernel; its outputs are read below
  grid_dependency_wait();
  // out_proj: the next kernel (the next step's split plan, which writes the
  // plan part of the workspace before its own dependency wait) starts only now,
  // when every kernel before this one has finished: none of them still reads
  // the workspace, so consecutive steps may share one
  if (!kAbsorb) grid_launch_dependents();

  const uint32_t idesc = idesc_bf16(128, C::NT, kAbsorb, false);
  auto da = [](uint32_t addr) -> uint64_t { return (uint64_t)((addr >> 4) & 0x3FFFu); };
  const uint64_t bdesc = smem_desc(0, 16, 1024, kSwizzle128B) + da(sbase + C::kOffB);
  uint32_t phase = 0;
  for (int t0 = 0; t0 < T; t0 += C::NT, phase ^= 1u) {
    if (threadIdx.x == 0) {
      const uint64_t pol = policy_evict_first();
      bool ok = true;
      if (kAbsorb) {
        if (t0 > 0) mbar_arrive_expect_tx(bar_ld, C::kBBytes);  // the first tile was armed with the weights
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(sbase + C::kOffB + kb * C::kBBox, &map_b, bar_ld, kb * 64, h, t0, pol);
        ok = wait_phase(bar_ld, phase, abort_flag, err_word);
        if (ok) {
          tc_fence_after();
          // A is M-major: 64-column halves 16 KB apart (LBO), 8-row K groups 1 KB apart (SBO)
          const uint64_t adesc = smem_desc(0, C::kABox, 1024, kSwizzle128B) + da(sbase + C::kOffA);
#pragma unroll
          for (int ks = 0; ks < C::K / 16; ++ks)
            mma_ss(tmem, adesc + (ks * 2048 >> 4), bdesc + (((ks >> 2) * C::kBBox + (ks & 3) * 32) >> 4), idesc,
                   ks > 0 ? 1u : 0u);
        }
      } else {
        for (int kb = 0; kb < C::KB; ++kb) {
          const uint32_t b = bar_ld + 8 * kb;
          if (t0 > 0) mbar_arrive_expect_tx(b, C::kBBox);  // the first tile was armed with the weights
          tma_load_3d(sbase + C::kOffB + kb * C::kBBox, &map_b, b, kb * 64, h, t0, pol);
        }
        const uint64_t adesc = smem_desc(0, 16, 1024, kSwizzle128B) + da(sbase + C::kOffA);
        for (int kb = 0; kb < C::KB && ok; ++kb) {
          ok = wait_phase(bar_ld + 8 * kb, phase, abort_flag, err_word);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            mma_ss(tmem, adesc + ((kb * C::kABox + k4 * 32) >> 4), bdesc + ((kb * C::kBBox + k4 * 32) >> 4), idesc,
                   (kb > 0 || k4 > 0) ? 1u : 0u);
        }
      }
      mma_commit(bar_d);  // arrives once the MMAs (if any) finished
    }
    // rotated positional query, copied unchanged next to the absorbed one, by
    // warps 1..3 while thread 0 waits for the tiles
    if (kAbsorb && q_rope && cblk == 0 && t0 == 0 && warp > 0) {
      for (int i = threadIdx.x - 32; i < T * (kDR / 8); i += kThreads - 32) {
        const int t = i / (kDR / 8), v = i % (kDR / 8);
        const uint4 w = reinterpret_cast<const uint4*>(q_rope + ((size_t)t * H + h) * kDR)[v];
        reinterpret_cast<uint4*>(out + ((size_t)t * H + h) * out_row + kDC)[v] = w;
      }
    }
    __syncwarp();
    if (!wait_phase(bar_d, phase, abort_flag, err_word)) break;
    tc_fence_after();
    // epilogue: lane = output column, registers = rows t. The tile goes through
    // shared memory (the B operand's space, free once the MMAs are done) as
    // [rows][128 columns] bf16, so that each output row leaves as 16-byte stores
    // of 256 contiguous bytes (one 2-byte store per column and row had queued
    // for microseconds)
    const int col = warp * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t tile = sbase + C::kOffB;
#pragma unroll 1
    for (int c0 = 0; c0 < C::NT; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(taddr + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int v = 0; v < 32; ++v)
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(tile + (uint32_t)(c0 + v) * 256u + 2u * col),
                     "h"(float_to_bf16(__uint_as_float(r[v])))
                     : "memory");
    }
    __syncthreads();
    for (int i = threadIdx.x; i < C::NT * 16; i += kThreads) {
      const int row = i >> 4, part = i & 15, t = t0 + row;
      if (t < T) {
        uint4 v;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(tile + (uint32_t)row * 256u + 16u * part));
        uint16_t* dst = kAbsorb ? out + ((size_t)t * H + h) * out_row + cblk * 128
                                : out + ((size_t)t * H + h) * kDV;
        reinterpret_cast<uint4*>(dst)[part] = v;
      }
    }
    fence_proxy_async_smem();  // the next rows' B tile is written by TMA
    tc_fence_before();
    __syncthreads();  // D and the B tile are free for the next rows
    tc_fence_after();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmCols);
  }
}

template <bool kAbsorb, int kNT>
cudaError_t launch_proj(const CUtensorMap& ma, const CUtensorMap& mb, const uint16_t* w, const uint16_t* q_rope,
                        uint16_t* out, int T, int H, int out_row, cudaStream_t s) {
  using C = ProjCfg<kAbsorb, kNT>;
  cudaError_t e = smem_limit<proj_tc_kernel<kAbsorb, kNT>>(C::kSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid(H, kAbsorb ? kDC / 128 : 1);
  return launch_pdl(proj_tc_kernel<kAbsorb, kNT>, grid, dim3(kThreads), C::kSmem, s, ma, mb, w, q_rope, out, T,
                    H, out_row, (int32_t*)nullptr);
}

bool maps(CUtensorMap* ma, CUtensorMap* mb, const uint16_t* w, const uint16_t* act, int T, int H, int K, int nt) {
  // weights [H][128][512]: boxes of 64 columns x 128 rows; activations [T][H][K]: 64 x 1 head x nt rows
  const uint64_t da[3] = {kDC, 128, (uint64_t)H}, sa[2] = {kDC * 2, (uint64_t)128 * kDC * 2};
  const uint64_t db[3] = {(uint64_t)K, (uint64_t)H, (uint64_t)T}, sb[2] = {(uint64_t)K * 2, (uint64_t)H * K * 2};
  const uint32_t ba[3] = {64, kBoxRows, 1}, bb[3] = {64, 1, (uint32_t)nt};
  return make_tmap(ma, w, 3, da, sa, ba, 128) && make_tmap(mb, act, 3, db, sb, bb, 128);
}

}  // namespace

namespace {
cudaError_t absorb_rows(const uint16_t* q_nope, const uint16_t* q_rope, const uint16_t* w_uk, uint16_t* out, int T,
                        int H, int out_row, cudaStream_t s) {
  const int nt = T <= 32 ? 32 : T <= 64 ? 64 : 128;
  CUtensorMap ma, mb;
  if (!maps(&ma, &mb, w_uk, q_nope, T, H, kDNope, nt)) return cudaErrorInvalidValue;
  if (nt == 32) return launch_proj<true, 32>(ma, mb, w_uk, q_rope, out, T, H, out_row, s);
  if (nt == 64) return launch_proj<true, 64>(ma, mb, w_uk, q_rope, out, T, H, out_row, s);
  return launch_proj<true, 128>(ma, mb, w_uk, q_rope, out, T, H, out_row, s);
}
}  // namespace

cudaError_t launch_absorb_q(const uint16_t* q_nope, const uint16_t* q_rope, const uint16_t* w_uk,
                            uint16_t* q_abs, int T, int H, cudaStream_t s) {
  return absorb_rows(q_nope, q_rope, w_uk, q_abs, T, H, kRow, s);
}

cudaError_t launch_merge_w_kq(const uint16_t* w_uq, const uint16_t* w_uk, uint16_t* w_kq, int d_q, int H,
                              cudaStream_t s) {
  return absorb_rows(w_uq, nullptr, w_uk, w_kq, d_q, H, kDC, s);
}

cudaError_t launch_out_proj(const uint16_t* u, const uint16_t* w_uv, uint16_t* out, int T, int H,
                            cudaStream_t s) {
  const int nt = T <= 32 ? 32 : 64;
  CUtensorMap ma, mb;
  if (!maps(&ma, &mb, w_uv, u, T, H, kDC, nt)) return cudaErrorInvalidValue;
  if (nt == 32) return launch_proj<false, 32>(ma, mb, w_uv, nullptr, out, T, H, kDV, s);
  return launch_proj<false, 64>(ma, mb, w_uv, nullptr, out, T, H, kDV, s);
}

}  // namespace mla
