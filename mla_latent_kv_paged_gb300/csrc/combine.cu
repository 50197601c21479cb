// Log-sum-exp merge of split-KV partials (the flash-decoding merge; Huny's
// Dev Blog "MLA 아키텍처 해부" section 4 table names FlashDecoding as the
// decode technique):
//   lse = ln sum_k exp(lse_k),   u = sum_k exp(lse_k - lse) * o_k
// One warp per (sequence, query, head); each lane owns 16 of the 512 latent
// columns as four float4 groups, so partial reads are 128-bit and coalesced,
// and each lane writes 8 bytes of bf16 output per group.
#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(Plan plan, int n_q, int H, uint16_t* __restrict__ u, float* __restrict__ lse_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bj = blockIdx.x;  // b * n_q + j
  const int h = blockIdx.y * kWarps + warp;
  if (h >= H) return;
  const int b = bj / n_q, j = bj % n_q;
  const int k0 = plan.seq_item[b], k1 = plan.seq_item[b + 1];

  float m = -INFINITY;
  for (int k = k0; k < k1; ++k) m = fmaxf(m, plan.lse_part[((size_t)k * n_q + j) * H + h]);
  float4 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (m != -INFINITY) {
    for (int k = k0; k < k1; ++k) {
      const size_t row = ((size_t)k * n_q + j) * H + h;
      const float lk = plan.lse_part[row];
      if (lk == -INFINITY) continue;
      const float w = expf(lk - m);
      wsum += w;
      const float4* src = reinterpret_cast<const float4*>(plan.o_part + row * kDC);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 v = src[lane + 32 * i];
        acc[i].x = fmaf(w, v.x, acc[i].x);
        acc[i].y = fmaf(w, v.y, acc[i].y);
        acc[i].z = fmaf(w, v.z, acc[i].z);
        acc[i].w = fmaf(w, v.w, acc[i].w);
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
  combine_kernel<<<grid, kWarps * 32, 0, s>>>(plan, n_q, H, u, lse);
  return cudaGetLastError();
}

}  // namespace mla
