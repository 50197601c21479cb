// Per-head projections on CUDA cores (fp32 accumulation, bf16 in and out).
//
// absorb_q: q_abs[t][h][c] = sum_i q_nope[t][h][i] * W_UK[h][i][c], and the
//           rotated positional query copied to columns 512..575
//           (Huny's Dev Blog "MLA 아키텍처 해부" section 3.1, qt = q^C (W^UK)^T).
// out_proj: out[t][h][v] = sum_c W_UV[h][v][c] * u[t][h][c]   (section 3.2).
#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kTT = 32;  // query rows per pass

// grid (H, d_c / 128); thread = one latent column c; W_UK rows are read
// coalesced along c, q_nope rows are staged in shared memory.
__global__ void __launch_bounds__(128)
absorb_q_simt_kernel(const uint16_t* __restrict__ q_nope, const uint16_t* __restrict__ q_rope,
                     const uint16_t* __restrict__ w_uk, uint16_t* __restrict__ q_abs, int T, int H) {
  __shared__ float qs[kTT][kDNope];
  const int h = blockIdx.x, c = blockIdx.y * 128 + threadIdx.x;
  const uint16_t* w = w_uk + (size_t)h * kDNope * kDC;
  for (int t0 = 0; t0 < T; t0 += kTT) {
    const int nt = min(kTT, T - t0);
    __syncthreads();
    for (int i = threadIdx.x; i < kTT * kDNope; i += 128) {
      const int tt = i / kDNope, e = i % kDNope;
      qs[tt][e] = tt < nt ? bf16_to_float(q_nope[((size_t)(t0 + tt) * H + h) * kDNope + e]) : 0.f;
    }
    __syncthreads();
    float acc[kTT];
#pragma unroll
    for (int tt = 0; tt < kTT; ++tt) acc[tt] = 0.f;
    for (int i = 0; i < kDNope; ++i) {
      const float wv = bf16_to_float(w[(size_t)i * kDC + c]);
#pragma unroll
      for (int tt = 0; tt < kTT; ++tt) acc[tt] = fmaf(qs[tt][i], wv, acc[tt]);
    }
    for (int tt = 0; tt < nt; ++tt)
      q_abs[((size_t)(t0 + tt) * H + h) * kRow + c] = float_to_bf16(acc[tt]);
  }
  if (blockIdx.y == 0) {
    for (int i = threadIdx.x; i < T * kDR; i += 128) {
      const int t = i / kDR, e = i % kDR;
      q_abs[((size_t)t * H + h) * kRow + kDC + e] = q_rope[((size_t)t * H + h) * kDR + e];
    }
  }
}

// grid (H); thread = one output column v; W_UV and u chunks staged in shared memory.
__global__ void __launch_bounds__(128)
out_proj_simt_kernel(const uint16_t* __restrict__ u, const uint16_t* __restrict__ w_uv,
                     uint16_t* __restrict__ out, int T, int H) {
  __shared__ float ws[kDV][65];
  __shared__ float us[kTT][64];
  const int h = blockIdx.x, v = threadIdx.x;
  const uint16_t* w = w_uv + (size_t)h * kDV * kDC;
  for (int t0 = 0; t0 < T; t0 += kTT) {
    const int nt = min(kTT, T - t0);
    float acc[kTT];
#pragma unroll
    for (int tt = 0; tt < kTT; ++tt) acc[tt] = 0.f;
    for (int c0 = 0; c0 < kDC; c0 += 64) {
      __syncthreads();
      for (int i = threadIdx.x; i < kDV * 64; i += 128) {
        const int vv = i / 64, cc = i % 64;
        ws[vv][cc] = bf16_to_float(w[(size_t)vv * kDC + c0 + cc]);
      }
      for (int i = threadIdx.x; i < kTT * 64; i += 128) {
        const int tt = i / 64, cc = i % 64;
        us[tt][cc] = tt < nt ? bf16_to_float(u[((size_t)(t0 + tt) * H + h) * kDC + c0 + cc]) : 0.f;
      }
      __syncthreads();
      for (int cc = 0; cc < 64; ++cc) {
        const float wv = ws[v][cc];
#pragma unroll
        for (int tt = 0; tt < kTT; ++tt) acc[tt] = fmaf(wv, us[tt][cc], acc[tt]);
      }
    }
    for (int tt = 0; tt < nt; ++tt) out[((size_t)(t0 + tt) * H + h) * kDV + v] = float_to_bf16(acc[tt]);
  }
}

}  // namespace

cudaError_t launch_absorb_q(const uint16_t* q_nope, const uint16_t* q_rope, const uint16_t* w_uk,
                            uint16_t* q_abs, int T, int H, cudaStream_t s) {
  absorb_q_simt_kernel<<<dim3(H, kDC / 128), 128, 0, s>>>(q_nope, q_rope, w_uk, q_abs, T, H);
  return cudaGetLastError();
}

cudaError_t launch_out_proj(const uint16_t* u, const uint16_t* w_uv, uint16_t* out, int T, int H,
                            cudaStream_t s) {
  out_proj_simt_kernel<<<H, 128, 0, s>>>(u, w_uv, out, T, H);
  return cudaGetLastError();
}

}  // namespace mla
