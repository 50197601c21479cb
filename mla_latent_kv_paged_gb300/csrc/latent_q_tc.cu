// Absorbed query straight from the compressed query latent, through the
// merged query-side weight (ingu627.github.io "Multi-Head Latent Attention
// (MLA)" section 2.2: S = C_KV^T (W_UK^T W_UQ) C_Q, merged per head):
//   q_abs[t][h][c] = sum_k c_q[t][k] w_kq[k][h][c]        c < 512
// and the rotated positional query q_rope[t][h] copied to columns 512..575.
// w_kq [d_q][H][512] is what mla_merge_w_kq writes.
//
// A weight-streaming GEMM at decode batch sizes: CTA (h, cblk) computes
// D[c][t] for the 128 columns [128 cblk, 128 cblk + 128) of head h on the
// tensor cores (tcgen05, D in tensor memory): M = 128 columns, N = rows t
// (32, 64 or 128 per tile), K = d_q in 64-wide slices streamed through a
// TMA ring. A = w_kq[k-slice][h][c-block] read M-major as two [64 k][64 c]
// boxes, B = the c_q rows of the tile (K-major). One thread issues the loads
// and the MMAs; the first slices' weight boxes are requested before the grid
// dependency wait (weights are never the previous kernel's output).
#include "mla_internal.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kThreads = 128;
constexpr int kStages = 5;
constexpr uint32_t kABox = 64 * 128;  // [64 k][64 c] bf16, 128B swizzle

template <int kNT>
struct LatentCfg {
  static constexpr uint32_t kBBox = kNT * 128;  // [kNT rows][64 k] bf16, 128B swizzle
  static constexpr uint32_t kStage = 2 * kABox + kBBox;
  static constexpr uint32_t kOffBar = kStages * kStage;
  static constexpr uint32_t kSmem = kOffBar + 8 * (2 * kStages + 1) + 16;
  static constexpr uint32_t kTmCols = kNT;
  static_assert(kStage % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(kNT * 256 <= kStage, "the epilogue tile fits the first stage");
};

template <int kNT>
__global__ void __launch_bounds__(kThreads, 1)
absorb_latent_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_c,
                     const uint16_t* __restrict__ q_rope, uint16_t* __restrict__ q_abs, int T, int H, int d_q) {
  using C = LatentCfg<kNT>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) return;  // the host checks the alignment of the dynamic shared memory base
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, cblk = blockIdx.y;
  const int KB = d_q / 64;
  auto full = [&](int s) { return sbase + C::kOffBar + 8u * (uint32_t)s; };
  auto empty = [&](int s) { return sbase + C::kOffBar + 8u * (uint32_t)(kStages + s); };
  const uint32_t bar_d = sbase + C::kOffBar + 8u * (2 * kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 8 * (2 * kStages + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + 8 * (2 * kStages + 1) + 4);
  const int wx = h * kDC + cblk * 128;  // first weight column of this CTA
  const int pre = KB < kStages ? KB : kStages;  // slices whose weights load before the dependency wait

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(bar_d, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_w);
    prefetch_tmap(&map_c);
    const uint64_t pol = policy_evict_first();
    for (int k = 0; k < pre; ++k) {
      mbar_arrive_expect_tx(full(k), C::kStage);
      for (int m = 0; m < 2; ++m)
        tma_load_2d(sbase + k * C::kStage + m * kABox, &map_w, full(k), wx + 64 * m, 64 * k, pol);
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // c_q and q_rope may be the previous kernel's output
  grid_dependency_wait();
  grid_launch_dependents();

  const uint32_t idesc = idesc_bf16(128, kNT, true, false);
  auto da = [](uint32_t addr) -> uint64_t { return (uint64_t)((addr >> 4) & 0x3FFFu); };
  uint32_t dphase = 0;
  int tile = 0;
  bool ok = true;
  for (int t0 = 0; t0 < T && ok; t0 += kNT, dphase ^= 1u, ++tile) {
    if (threadIdx.x == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_c = policy_evict_last();
      const int base = tile * KB;  // ring use of slice k of this tile: base + k
      // load slice k of this tile into its stage (the weights of the first
      // tile's first slices are already on their way)
      auto load = [&](int k) -> bool {
        const int u = base + k, s = u % kStages;
        const uint32_t st = sbase + s * C::kStage;
        if (u >= pre) {
          if (u >= kStages && !wait_phase(empty(s), ((u / kStages) - 1) & 1, abort_flag, nullptr)) return false;
          mbar_arrive_expect_tx(full(s), C::kStage);
          for (int m = 0; m < 2; ++m) tma_load_2d(st + m * kABox, &map_w, full(s), wx + 64 * m, 64 * k, pol_w);
        }
        tma_load_2d(st + 2 * kABox, &map_c, full(s), 64 * k, t0, pol_c);
        return true;
      };
      for (int k = 0; k < kStages && k < KB && ok; ++k) ok = load(k);
      for (int k = 0; k < KB && ok; ++k) {
        const int u = base + k, s = u % kStages;
        if (!wait_phase(full(s), (u / kStages) & 1, abort_flag, nullptr)) { ok = false; break; }
        tc_fence_after();
        const uint32_t st = sbase + s * C::kStage;
        // A is M-major: the two 64-column boxes 8 KB apart (LBO), 8-row K groups 1 KB apart (SBO)
        const uint64_t adesc = smem_desc(0, kABox, 1024, kSwizzle128B) + da(st);
        const uint64_t bdesc = smem_desc(0, 16, 1024, kSwizzle128B) + da(st + 2 * kABox);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_ss(tmem, adesc + ((ks * 2048) >> 4), bdesc + ((ks * 32) >> 4), idesc, (k > 0 || ks > 0) ? 1u : 0u);
        mma_commit(empty(s));
        // refill the stage of the previous slice (its MMAs have had this slice's wait to finish)
        if (k >= 1 && k - 1 + kStages < KB) ok = load(k - 1 + kStages);
      }
      mma_commit(bar_d);  // arrives once the MMAs (if any) finished
    }
    // rotated positional query, copied unchanged next to the absorbed one, by
    // warps 1..3 while thread 0 streams the weights
    if (cblk == 0 && t0 == 0 && warp > 0) {
      for (int i = threadIdx.x - 32; i < T * (kDR / 8); i += kThreads - 32) {
        const int t = i / (kDR / 8), v = i % (kDR / 8);
        const uint4 w = reinterpret_cast<const uint4*>(q_rope + ((size_t)t * H + h) * kDR)[v];
        reinterpret_cast<uint4*>(q_abs + ((size_t)t * H + h) * kRow + kDC)[v] = w;
      }
    }
    __syncwarp();
    if (!wait_phase(bar_d, dphase, abort_flag, nullptr)) break;
    tc_fence_after();
    // epilogue: lane = output column, registers = rows t. The tile goes through
    // shared memory (the first ring stage: every MMA of the tile is done) as
    // [rows][128 columns] bf16, and each row leaves as 16-byte stores
    const int col = warp * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int c0 = 0; c0 < kNT; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(taddr + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int v = 0; v < 32; ++v)
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(sbase + (uint32_t)(c0 + v) * 256u + 2u * col),
                     "h"(float_to_bf16(__uint_as_float(r[v])))
                     : "memory");
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kNT * 16; i += kThreads) {
      const int row = i >> 4, part = i & 15, t = t0 + row;
      if (t < T) {
        uint4 v;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(sbase + (uint32_t)row * 256u + 16u * part));
        reinterpret_cast<uint4*>(q_abs + ((size_t)t * H + h) * kRow + cblk * 128)[part] = v;
      }
    }
    fence_proxy_async_smem();  // the ring stages are written by TMA again for the next rows
    tc_fence_before();
    __syncthreads();  // D and the first stage are free for the next rows
    tc_fence_after();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmCols);
  }
}

template <int kNT>
cudaError_t launch_latent(const CUtensorMap& mw, const CUtensorMap& mc, const uint16_t* q_rope, uint16_t* q_abs,
                          int T, int H, int d_q, cudaStream_t s) {
  using C = LatentCfg<kNT>;
  cudaError_t e = smem_limit<absorb_latent_kernel<kNT>>(C::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(absorb_latent_kernel<kNT>, dim3(H, kDC / 128), dim3(kThreads), C::kSmem, s, mw, mc, q_rope,
                    q_abs, T, H, d_q);
}

}  // namespace

cudaError_t launch_absorb_latent(const uint16_t* c_q, const uint16_t* q_rope, const uint16_t* w_kq, uint16_t* q_abs,
                                 int T, int H, int d_q, cudaStream_t s) {
  const int nt = T <= 32 ? 32 : T <= 64 ? 64 : 128;
  // w_kq [d_q][H * 512]: boxes of 64 columns x 64 rows; c_q [T][d_q]: 64 x nt rows
  const uint64_t dw[2] = {(uint64_t)H * kDC, (uint64_t)d_q}, sw[1] = {(uint64_t)H * kDC * 2};
  const uint64_t dc[2] = {(uint64_t)d_q, (uint64_t)T}, sc[1] = {(uint64_t)d_q * 2};
  const uint32_t bw[2] = {64, 64}, bc[2] = {64, (uint32_t)nt};
  CUtensorMap mw, mc;
  if (!make_tmap(&mw, w_kq, 2, dw, sw, bw, 128) || !make_tmap(&mc, c_q, 2, dc, sc, bc, 128))
    return cudaErrorInvalidValue;
  if (nt == 32) return launch_latent<32>(mw, mc, q_rope, q_abs, T, H, d_q, s);
  if (nt == 64) return launch_latent<64>(mw, mc, q_rope, q_abs, T, H, d_q, s);
  return launch_latent<128>(mw, mc, q_rope, q_abs, T, H, d_q, s);
}

}  // namespace mla
