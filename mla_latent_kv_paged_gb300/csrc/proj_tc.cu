// Per-head projections on the tcgen05 tensor cores (bf16 in, fp32 accumulate
// in tensor memory, bf16 out). Both are weight-streaming GEMMs at decode batch
// sizes: every CTA keeps one head's weight slice resident in shared memory and
// multiplies it by the query rows of that head.
//
// absorb_q (Huny's Dev Blog "MLA 아키텍처 해부" section 3.1, qt = q^C (W^UK)^T):
//   D[c][t] = sum_i W_UK[h][i][c] q_nope[t][h][i]      M = 128 latent cols, N = rows t, K = 128
//   A = W_UK[h][:, c-block] read M-major, B = q_nope rows (K-major).
//   The rotated positional query is copied to columns 512..575.
// out_proj (section 3.2, u W^UV):
//   D[v][t] = sum_c W_UV[h][v][c] u[t][h][c]            M = 128 value cols, N = rows t, K = 512
//   A = W_UV[h] (K-major), B = u rows (K-major).
// D sits in tensor memory with one lane per output column, so the epilogue
// writes each output row t with 32 consecutive columns per warp.
#include "mla_internal.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kThreads = 128;
constexpr uint32_t kBoxRows = 128;  // A boxes: 128 rows x 64 bf16

template <bool kAbsorb>
struct ProjCfg {
  static constexpr int NT = kAbsorb ? 128 : 64;        // rows t per tile (MMA N)
  static constexpr int K = kAbsorb ? kDNope : kDC;      // reduction length
  static constexpr int KB = K / 64;                     // 64-wide K boxes
  static constexpr uint32_t kABytes = kAbsorb ? 2 * kBoxRows * 128 : KB * kBoxRows * 128;
  static constexpr uint32_t kBBytes = KB * NT * 128;
  static constexpr uint32_t kOffA = 0, kOffB = kABytes, kOffBar = kABytes + kBBytes;
  static constexpr uint32_t kSmem = kOffBar + 64;
  static constexpr uint32_t kTmCols = NT < 32 ? 32 : NT;
};

template <bool kAbsorb>
__global__ void __launch_bounds__(kThreads, 1)
proj_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const uint16_t* __restrict__ q_rope, uint16_t* __restrict__ out, int T, int H, int32_t* err_word) {
  using C = ProjCfg<kAbsorb>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, cblk = blockIdx.y;  // cblk: 128-column block of q_abs (absorb only)
  const uint32_t bar_a = sbase + C::kOffBar, bar_b = bar_a + 8, bar_d = bar_a + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 24);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + 28);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) report_error(err_word, MLA_ERR_CUDA);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(bar_a, 1);
    mbar_init(bar_b, 1);
    mbar_init(bar_d, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_a);
    prefetch_tmap(&map_b);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {
    const uint64_t pol = policy_evict_first();
    mbar_arrive_expect_tx(bar_a, C::kABytes);
    if (kAbsorb) {
      // W_UK[h][i][c] as boxes of [128 i][64 c]: the two 64-column halves of this block
      for (int m = 0; m < 2; ++m)
        tma_load_3d(sbase + C::kOffA + m * kBoxRows * 128, &map_a, bar_a, cblk * 128 + m * 64, 0, h, pol);
    } else {
      for (int kb = 0; kb < C::KB; ++kb)
        tma_load_3d(sbase + C::kOffA + kb * kBoxRows * 128, &map_a, bar_a, kb * 64, 0, h, pol);
    }
  }
  // rotated positional query: copied unchanged next to the absorbed one
  if (kAbsorb && cblk == 0) {
    for (int i = threadIdx.x; i < T * (kDR / 8); i += kThreads) {
      const int t = i / (kDR / 8), v = i % (kDR / 8);
      const uint4 w = reinterpret_cast<const uint4*>(q_rope + ((size_t)t * H + h) * kDR)[v];
      reinterpret_cast<uint4*>(out + ((size_t)t * H + h) * kRow + kDC)[v] = w;
    }
  }

  const uint32_t idesc = idesc_bf16(128, C::NT, kAbsorb, false);
  auto da = [](uint32_t addr) -> uint64_t { return (uint64_t)((addr >> 4) & 0x3FFFu); };
  int phase = 0;
  for (int t0 = 0; t0 < T; t0 += C::NT, phase ^= 1) {
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(bar_b, C::kBBytes);
      for (int kb = 0; kb < C::KB; ++kb)
        tma_load_3d(sbase + C::kOffB + kb * C::NT * 128, &map_b, bar_b, kb * 64, h, t0, policy_evict_first());
      bool ok = wait_phase(bar_a, 0, abort_flag, err_word) && wait_phase(bar_b, phase, abort_flag, err_word);
      if (ok) {
        tc_fence_after();
        const uint64_t bdesc = smem_desc(0, 16, 1024, kSwizzle128B) + da(sbase + C::kOffB);
        if (kAbsorb) {
          // A is M-major: 64-column halves 16 KB apart (LBO), 8-row K groups 1 KB apart (SBO)
          const uint64_t adesc = smem_desc(0, kBoxRows * 128, 1024, kSwizzle128B) + da(sbase + C::kOffA);
#pragma unroll
          for (int ks = 0; ks < C::K / 16; ++ks)
            mma_ss(tmem, adesc + (ks * 2048 >> 4), bdesc + (((ks >> 2) * C::NT * 128 + (ks & 3) * 32) >> 4), idesc,
                   ks > 0 ? 1u : 0u);
        } else {
          const uint64_t adesc = smem_desc(0, 16, 1024, kSwizzle128B) + da(sbase + C::kOffA);
#pragma unroll
          for (int ks = 0; ks < C::K / 16; ++ks)
            mma_ss(tmem, adesc + (((ks >> 2) * kBoxRows * 128 + (ks & 3) * 32) >> 4),
                   bdesc + (((ks >> 2) * C::NT * 128 + (ks & 3) * 32) >> 4), idesc, ks > 0 ? 1u : 0u);
        }
      }
      mma_commit(bar_d);  // arrives once the MMAs (if any) finished
    }
    __syncwarp();
    if (!wait_phase(bar_d, phase, abort_flag, err_word)) break;
    tc_fence_after();
    // epilogue: lane = output column, registers = rows t
    const int col = warp * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int c0 = 0; c0 < C::NT; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(taddr + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int v = 0; v < 32; ++v) {
        const int t = t0 + c0 + v;
        if (t < T) {
          const float f = __uint_as_float(r[v]);
          if (kAbsorb)
            out[((size_t)t * H + h) * kRow + cblk * 128 + col] = float_to_bf16(f);
          else
            out[((size_t)t * H + h) * kDV + col] = float_to_bf16(f);
        }
      }
    }
    tc_fence_before();
    __syncthreads();  // D and the B tile are free for the next rows
    tc_fence_after();
  }
  // drain: the MMAs of the last tile completed before the epilogue read D
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmCols);
  }
}

template <bool kAbsorb>
cudaError_t set_smem() {
  static bool done = false;
  if (!done) {
    cudaError_t e = cudaFuncSetAttribute(proj_tc_kernel<kAbsorb>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)ProjCfg<kAbsorb>::kSmem);
    if (e != cudaSuccess) return e;
    done = true;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_absorb_q(const uint16_t* q_nope, const uint16_t* q_rope, const uint16_t* w_uk,
                            uint16_t* q_abs, int T, int H, cudaStream_t s) {
  using C = ProjCfg<true>;
  CUtensorMap ma, mb;
  // W_UK [H][128 i][512 c]: boxes of 64 c x 128 i; q_nope [T][H][128]: boxes of 64 i x 1 head x NT rows
  const uint64_t da[3] = {kDC, kDNope, (uint64_t)H}, sa[2] = {kDC * 2, (uint64_t)kDNope * kDC * 2};
  const uint64_t db[3] = {kDNope, (uint64_t)H, (uint64_t)T}, sb[2] = {kDNope * 2, (uint64_t)H * kDNope * 2};
  const uint32_t ba[3] = {64, kBoxRows, 1}, bb[3] = {64, 1, (uint32_t)C::NT};
  if (!make_tmap(&ma, w_uk, 3, da, sa, ba, 128) || !make_tmap(&mb, q_nope, 3, db, sb, bb, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem<true>();
  if (e != cudaSuccess) return e;
  proj_tc_kernel<true><<<dim3(H, kDC / 128), kThreads, C::kSmem, s>>>(ma, mb, q_rope, q_abs, T, H, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_out_proj(const uint16_t* u, const uint16_t* w_uv, uint16_t* out, int T, int H,
                            cudaStream_t s) {
  using C = ProjCfg<false>;
  CUtensorMap ma, mb;
  // W_UV [H][128 v][512 c]: boxes of 64 c x 128 v; u [T][H][512]: boxes of 64 c x 1 head x NT rows
  const uint64_t da[3] = {kDC, kDV, (uint64_t)H}, sa[2] = {kDC * 2, (uint64_t)kDV * kDC * 2};
  const uint64_t db[3] = {kDC, (uint64_t)H, (uint64_t)T}, sb[2] = {kDC * 2, (uint64_t)H * kDC * 2};
  const uint32_t ba[3] = {64, kBoxRows, 1}, bb[3] = {64, 1, (uint32_t)C::NT};
  if (!make_tmap(&ma, w_uv, 3, da, sa, ba, 128) || !make_tmap(&mb, u, 3, db, sb, bb, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem<false>();
  if (e != cudaSuccess) return e;
  proj_tc_kernel<false><<<dim3(H, 1), kThreads, C::kSmem, s>>>(ma, mb, nullptr, out, T, H, nullptr);
  return cudaGetLastError();
}

}  // namespace mla
