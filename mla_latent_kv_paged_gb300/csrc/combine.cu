// Log-sum-exp merge of split-KV partials (the flash-decoding merge; Huny's
// Dev Blog "MLA 아키텍처 해부" section 4 table names FlashDecoding as the
// decode technique):
//   lse = ln sum_k exp(lse_k),   u = sum_k exp(lse_k - lse) * o_k
// One warp per (sequence, query, head); each lane owns 16 of the 512 latent
// columns as four float4 groups, so partial reads are 128-bit and coalesced,
// and each lane writes 8 bytes of bf16 output per group.
#include "mla_internal.cuh"

#include "sm100.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(Plan plan, int n_q, int H, uint16_t* __restrict__ u, float* __restrict__ lse_out) {
  sm100::grid_dependency_wait();  // the partials come from the decode kernel
  sm100::grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bj = blockIdx.x;  // b * n_q + j
  const int h = blockIdx.y * kWarps + warp;
  if (h >= H) return;
  const int b = bj / n_q, j = bj % n_q;
  const int k0 = plan.seq_item[b], k1 = plan.seq_item[b + 1];
  auto row_of = [&](int k) { return ((size_t)k * n_q + j) * H + h; };

  // all log-sum-exps of this row at once: lane l holds piece k0 + 32 i + l
  float m = -INFINITY;
  for (int k = k0 + lane; k < k1; k += 32) m = fmaxf(m, plan.lse_part[row_of(k)]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float4 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (m != -INFINITY) {
    for (int kc = k0; kc < k1; kc += 32) {
      const int n = min(32, k1 - kc);
      const float lk = lane < n ? plan.lse_part[row_of(kc + lane)] : -INFINITY;
      const float wl = lk == -INFINITY ? 0.f : expf(lk - m);
      float ws = wl;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
      wsum += ws;
#pragma unroll 4
      for (int k = 0; k < n; ++k) {
        const float w = __shfl_sync(0xffffffffu, wl, k);
        const float4* src = reinterpret_cast<const float4*>(plan.o_part + row_of(kc + k) * kDC);
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = src[lane + 32 * i];
        if (w != 0.f) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[i].x = fmaf(w, v[i].x, acc[i].x);
            acc[i].y = fmaf(w, v[i].y, acc[i].y);
            acc[i].z = fmaf(w, v[i].z, acc[i].z);
            acc[i].w = fmaf(w, v[i].w, acc[i].w);
          }
        }
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint2* dst = reinterpret_cast<uint2*>(u + ((size_t)bj * H + h) * kDC);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint2 o;
    o.x = pack_bf16x2(acc[i].x * inv, acc[i].y * inv);
    o.y = pack_bf16x2(acc[i].z * inv, acc[i].w * inv);
    dst[lane + 32 * i] = o;
  }
  if (lse_out && lane == 0) lse_out[(size_t)bj * H + h] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const Plan& plan, int B, int n_q, int H, uint16_t* u, float* lse,
                           cudaStream_t s) {
  dim3 grid(B * n_q, (H + kWarps - 1) / kWarps);
  return launch_pdl(combine_kernel, grid, dim3(kWarps * 32), 0, s, plan, n_q, H, u, lse);
}

}  // namespace mla
