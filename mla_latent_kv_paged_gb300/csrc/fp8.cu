// FP8 (e4m3) latent cache: quantisation of bf16 cache rows with one scale per
// column (Huny's Dev Blog "MLA 아키텍처 해부", section 6 item 4: FP8 on the
// latent needs per-channel or per-block scales, not one per tensor).
//
// code[r][d] = e4m3(rows[r][d] / scales[d]): the quotient is one correctly
// rounded fp32 division, the conversion rounds to nearest (ties to even) and
// saturates at +-448. A streaming, HBM-bound elementwise kernel: each thread
// turns 8 values (16 bytes in) into 8 codes (8 bytes out).
#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kQuantThreads = 256;

// two fp32 values -> two e4m3 codes (lo in the low byte), nearest even, saturating
__device__ __forceinline__ uint32_t to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(kQuantThreads)
quantize_fp8_kernel(const uint4* __restrict__ rows, const float* __restrict__ scales, uint2* __restrict__ codes,
                    int64_t n8) {
  for (int64_t i = (int64_t)blockIdx.x * kQuantThreads + threadIdx.x; i < n8; i += (int64_t)gridDim.x * kQuantThreads) {
    const uint4 w = rows[i];
    const int col = (int)((i * 8) % kRow);  // rows of 576 values, groups of 8 never cross a row
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a = __fdiv_rn(bf16_lo(ww[k]), __ldg(scales + col + 2 * k));
      const float b = __fdiv_rn(bf16_hi(ww[k]), __ldg(scales + col + 2 * k + 1));
      out[k >> 1] |= to_e4m3x2(a, b) << (16 * (k & 1));
    }
    codes[i] = make_uint2(out[0], out[1]);
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const uint16_t* rows, const float* scales, uint8_t* codes, int64_t n_rows,
                                cudaStream_t s) {
  const int64_t n8 = n_rows * (kRow / 8);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t want = (n8 + kQuantThreads - 1) / kQuantThreads;
  const int blocks = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
  quantize_fp8_kernel<<<blocks, kQuantThreads, 0, s>>>(reinterpret_cast<const uint4*>(rows), scales,
                                                       reinterpret_cast<uint2*>(codes), n8);
  return cudaGetLastError();
}

}  // namespace mla
