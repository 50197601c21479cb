// Attention-layer output through the merged value/output weight (Huny's Dev
// Blog "MLA 아키텍처 해부" section 3, item 2: HeadOut_i = u_i (W_i^UV W_i^O),
// W_i,comb = W_i^UV W_i^O; the layer output is the sum over heads):
//   out[t][n] = sum_h sum_c u[t][h][c] w_comb[n][h][c]        K = H * 512
// w_comb [d_model][H][512] is what mla_merge_w_comb writes.
//
// A weight-streaming GEMM at decode batch sizes with a long reduction, so the
// K range is split across CTAs: CTA (m, s, tile) of the first kernel
// multiplies output columns [128m, 128m + 128) by its K slices on the tensor
// cores (tcgen05, D in tensor memory), streaming 64-wide slices of the weight
// rows (A, K-major) and of the u rows (B, K-major) through a TMA ring, and
// writes an fp32 partial. The second kernel adds the partials in split order,
// so the sums are reproducible bit for bit, and rounds to bf16.
#include "mla_internal.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kThreads = 128;
constexpr int kStages = 5;
constexpr uint32_t kABox = 128 * 128;  // [128 output columns][64 k] bf16, 128B swizzle
constexpr int kMaxSplits = 16;
constexpr int kResidentSlots = 304;    // CTAs resident at once on a 152-SM GB300 with the 100 KB ring

template <int kNT>
struct CombCfg {
  static constexpr uint32_t kBBox = kNT * 128;  // [kNT rows][64 k] bf16, 128B swizzle
  static constexpr uint32_t kStage = kABox + kBBox;
  static constexpr uint32_t kOffBar = kStages * kStage;
  static constexpr uint32_t kSmem = kOffBar + 8 * (2 * kStages + 1) + 16;
  static_assert(kStage % 1024 == 0, "swizzled tiles need 1024-byte alignment");
};

struct CombShape {
  int NT, ttiles, ntiles, KB, S;
};

__host__ __device__ inline CombShape comb_shape(int T, int H, int d_model) {
  CombShape c;
  c.NT = T <= 32 ? 32 : T <= 64 ? 64 : 128;
  c.ttiles = (T + c.NT - 1) / c.NT;
  c.ntiles = d_model / 128;
  c.KB = H * (kDC / 64);
  // about one wave of CTAs; a function of (T, H, d_model) only
  int S = kResidentSlots / (c.ntiles * c.ttiles);
  S = S < 1 ? 1 : S > kMaxSplits ? kMaxSplits : S;
  c.S = S < c.KB ? S : c.KB;
  return c;
}

template <int kNT>
__global__ void __launch_bounds__(kThreads, 1)
comb_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_u, int KB,
                 int d_model, float* __restrict__ partials) {
  using C = CombCfg<kNT>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) return;  // the host checks the alignment of the dynamic shared memory base
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x, s = blockIdx.y, tile = blockIdx.z, S = gridDim.y;
  const int kb0 = (int)((int64_t)s * KB / S), kb1 = (int)((int64_t)(s + 1) * KB / S), nkb = kb1 - kb0;
  auto full = [&](int i) { return sbase + C::kOffBar + 8u * (uint32_t)i; };
  auto empty = [&](int i) { return sbase + C::kOffBar + 8u * (uint32_t)(kStages + i); };
  const uint32_t bar_d = sbase + C::kOffBar + 8u * (2 * kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 8 * (2 * kStages + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + 8 * (2 * kStages + 1) + 4);
  const int pre = nkb < kStages ? nkb : kStages;  // slices whose weights load before the dependency wait

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    mbar_init(bar_d, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_w);
    prefetch_tmap(&map_u);
    const uint64_t pol = policy_evict_first();
    for (int k = 0; k < pre; ++k) {
      mbar_arrive_expect_tx(full(k), C::kStage);
      tma_load_2d(sbase + k * C::kStage, &map_w, full(k), (kb0 + k) * 64, m * 128, pol);
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kNT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // u may be the previous kernel's output; the partials buffer may still be
  // read by the previous call's reduction
  grid_dependency_wait();
  grid_launch_dependents();

  if (threadIdx.x == 0) {
    const uint64_t pol_w = policy_evict_first(), pol_u = policy_evict_last();
    const uint32_t idesc = idesc_bf16(128, kNT, false, false);
    auto da = [](uint32_t addr) -> uint64_t { return (uint64_t)((addr >> 4) & 0x3FFFu); };
    bool ok = true;
    auto load = [&](int k) -> bool {  // slice k of this split into stage k % kStages
      const int st_i = k % kStages;
      const uint32_t st = sbase + st_i * C::kStage;
      if (k >= pre) {
        if (!wait_phase(empty(st_i), ((k / kStages) - 1) & 1, abort_flag, nullptr)) return false;
        mbar_arrive_expect_tx(full(st_i), C::kStage);
        tma_load_2d(st, &map_w, full(st_i), (kb0 + k) * 64, m * 128, pol_w);
      }
      tma_load_2d(st + kABox, &map_u, full(st_i), (kb0 + k) * 64, tile * kNT, pol_u);
      return true;
    };
    for (int k = 0; k < pre && ok; ++k) ok = load(k);
    for (int k = 0; k < nkb && ok; ++k) {
      const int st_i = k % kStages;
      if (!wait_phase(full(st_i), (k / kStages) & 1, abort_flag, nullptr)) break;
      tc_fence_after();
      const uint32_t st = sbase + st_i * C::kStage;
      const uint64_t adesc = smem_desc(0, 16, 1024, kSwizzle128B) + da(st);
      const uint64_t bdesc = smem_desc(0, 16, 1024, kSwizzle128B) + da(st + kABox);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss(tmem, adesc + ((ks * 32) >> 4), bdesc + ((ks * 32) >> 4), idesc, (k > 0 || ks > 0) ? 1u : 0u);
      mma_commit(empty(st_i));
      // refill the stage of the previous slice (its MMAs have had this slice's wait to finish)
      if (k >= 1 && k - 1 + kStages < nkb) ok = load(k - 1 + kStages);
    }
    mma_commit(bar_d);  // arrives once the MMAs (if any) finished
  }
  __syncwarp();
  const bool done = wait_phase(bar_d, 0, abort_flag, nullptr);
  tc_fence_after();
  if (done) {
    // lane = output column n, registers = rows t of the tile
    const int n = m * 128 + warp * 32 + lane;
    float* dst = partials + ((size_t)(tile * S + s) * kNT) * d_model + n;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int c0 = 0; c0 < kNT; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(taddr + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int v = 0; v < 32; ++v) dst[(size_t)(c0 + v) * d_model] = __uint_as_float(r[v]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kNT);
  }
}

// out[t][n .. n+7] = bf16(sum over splits s, in order, of the partials)
__global__ void __launch_bounds__(256)
comb_reduce_kernel(const float* __restrict__ partials, uint16_t* __restrict__ out, int T, int d_model, int NT,
                   int S) {
  grid_dependency_wait();  // the partials come from the GEMM kernel
  grid_launch_dependents();
  const int groups = d_model / 8;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)T * groups) return;
  const int t = (int)(idx / groups), n = (int)(idx % groups) * 8;
  const int tile = t / NT, tt = t % NT;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int s = 0; s < S; ++s) {
    const float4* p =
        reinterpret_cast<const float4*>(partials + ((size_t)(tile * S + s) * NT + tt) * d_model + n);
    const float4 a = __ldcg(p), b = __ldcg(p + 1);
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(out + (size_t)t * d_model + n) = o;
}

template <int kNT>
cudaError_t launch_comb_gemm(const CUtensorMap& mw, const CUtensorMap& mu, const CombShape& c, int d_model,
                             float* partials, cudaStream_t s) {
  using C = CombCfg<kNT>;
  cudaError_t e = smem_limit<comb_gemm_kernel<kNT>>(C::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(comb_gemm_kernel<kNT>, dim3(c.ntiles, c.S, c.ttiles), dim3(kThreads), C::kSmem, s, mw, mu,
                    c.KB, d_model, partials);
}

}  // namespace

size_t out_comb_workspace_bytes(int T, int H, int d_model) {
  const CombShape c = comb_shape(T, H, d_model);
  return (size_t)c.ttiles * c.S * c.NT * d_model * 4;
}

cudaError_t launch_out_comb(const uint16_t* u, const uint16_t* w_comb, uint16_t* out, int T, int H, int d_model,
                            void* workspace, cudaStream_t s) {
  const CombShape c = comb_shape(T, H, d_model);
  const uint64_t K = (uint64_t)H * kDC;
  // w_comb [d_model][K]: boxes of 64 k x 128 rows; u [T][K]: 64 k x NT rows
  const uint64_t dw[2] = {K, (uint64_t)d_model}, sw[1] = {K * 2};
  const uint64_t du[2] = {K, (uint64_t)T}, su[1] = {K * 2};
  const uint32_t bw[2] = {64, 128}, bu[2] = {64, (uint32_t)c.NT};
  CUtensorMap mw, mu;
  if (!make_tmap(&mw, w_comb, 2, dw, sw, bw, 128) || !make_tmap(&mu, u, 2, du, su, bu, 128))
    return cudaErrorInvalidValue;
  float* part = static_cast<float*>(workspace);
  cudaError_t e = c.NT == 32   ? launch_comb_gemm<32>(mw, mu, c, d_model, part, s)
                  : c.NT == 64 ? launch_comb_gemm<64>(mw, mu, c, d_model, part, s)
                               : launch_comb_gemm<128>(mw, mu, c, d_model, part, s);
  if (e != cudaSuccess) return e;
  const int64_t n = (int64_t)T * (d_model / 8);
  return launch_pdl(comb_reduce_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, (const float*)part, out,
                    T, d_model, c.NT, c.S);
}

}  // namespace mla
