// Log-sum-exp merge of split-KV partials (the flash-decoding merge; Huny's
// Dev Blog "MLA 아키텍처 해부" section 4 table names FlashDecoding as the
// decode technique):
//   lse = ln sum_k exp(lse_k),   u = sum_k exp(lse_k - lse) * o_k
// One block per (sequence, query) row and 64-column slice, two threads per
// head (32 columns each), so a 32-sequence batch is one wave of 256 blocks that
// leaves room on each SM for the up-projection after it; the loads of two
// partials are in flight together.
// The partials are fp16, head-minor in groups of eight columns
// (o_part[k][j][column / 8][head][column % 8]), so a warp reads 32
// consecutive heads of eight columns as one 512-byte run; the bf16 result goes
// through shared memory so the stores of u are row-contiguous.
#include "mla_internal.cuh"

#include "sm100.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;  // two per head (H <= 128): 32 columns each
constexpr int kCols = 64;      // latent columns per block
constexpr int kCPT = kCols / 2;  // columns per thread
constexpr int kKB = 2;         // partials whose loads are in flight together

__global__ void __launch_bounds__(kThreads)
combine_kernel(Plan plan, int n_q, int H, uint16_t* __restrict__ u, float* __restrict__ lse_out) {
  __shared__ uint32_t tile[128][kCols / 2 + 1];  // bf16 pairs, padded row
  // The next kernel (the up-projection) may start now and load its weights
  // while the decode kernel's last CTAs and this merge run; it reads u only
  // after its own dependency wait.
  sm100::grid_launch_dependents();
  const int h = threadIdx.x & 127, part = threadIdx.x >> 7;
  const int bj = blockIdx.x;  // b * n_q + j
  const int c0 = blockIdx.y * kCols + kCPT * part;  // this thread's first column
  const int b = bj / n_q, j = bj % n_q;
  // The plan's piece ranges were written by a kernel that had finished before
  // the decode kernel (the kernel before this one) passed its own dependency
  // wait, and that kernel lets this one start only after that wait: they can be
  // read before this kernel's wait. The partials cannot.
  const int k0 = plan.seq_item[b], k1 = plan.seq_item[b + 1];
  sm100::grid_dependency_wait();  // the partials come from the decode kernel
  auto lse_of = [&](int k) { return plan.lse_part[((size_t)k * n_q + j) * H + h]; };
  float acc[kCPT];
#pragma unroll
  for (int c = 0; c < kCPT; ++c) acc[c] = 0.f;
  float m = -INFINITY, wsum = 0.f;
  if (h < H) {
    const uint4* o16 = reinterpret_cast<const uint4*>(plan.o_part);
    auto src_of = [&](int k) { return o16 + (((size_t)k * n_q + j) * (kDC / 8) + c0 / 8) * H + h; };
    // the first eight log-sum-exps and the first two pieces' data in flight
    // together: one dependent round trip when a sequence has at most two pieces
    float l8[8];
    uint4 v[kKB][kCPT / 8];
#pragma unroll
    for (int i = 0; i < 8; ++i) l8[i] = k0 + i < k1 ? lse_of(k0 + i) : -INFINITY;
#pragma unroll
    for (int i = 0; i < kKB; ++i)
#pragma unroll
      for (int q = 0; q < kCPT / 8; ++q)
        v[i][q] = k0 + i < k1 ? src_of(k0 + i)[(size_t)q * H] : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, l8[i]);
    for (int kb = k0 + 8; kb < k1; kb += 8) {  // more than eight pieces
      float l[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) l[i] = kb + i < k1 ? lse_of(kb + i) : -INFINITY;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, l[i]);
    }
    if (m != -INFINITY) {
      for (int kb = k0; kb < k1; kb += kKB) {
        float w[kKB];
        if (kb > k0) {  // later batches: their own loads
#pragma unroll
          for (int i = 0; i < kKB; ++i)
#pragma unroll
            for (int q = 0; q < kCPT / 8; ++q)
              v[i][q] = kb + i < k1 ? src_of(kb + i)[(size_t)q * H] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kKB; ++i) {
          const int k = kb + i;
          const float lk = k >= k1 ? -INFINITY : (kb == k0 ? l8[i] : lse_of(k));
          w[i] = lk == -INFINITY ? 0.f : expf(lk - m);
        }
#pragma unroll
        for (int i = 0; i < kKB; ++i) {
          wsum += w[i];
#pragma unroll
          for (int q = 0; q < kCPT / 8; ++q) {
            const uint32_t ww[4] = {v[i][q].x, v[i][q].y, v[i][q].z, v[i][q].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = sm100::f16x2_to_f32(ww[e]);
              acc[8 * q + 2 * e] = fmaf(w[i], f.x, acc[8 * q + 2 * e]);
              acc[8 * q + 2 * e + 1] = fmaf(w[i], f.y, acc[8 * q + 2 * e + 1]);
            }
          }
        }
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int c = 0; c < kCPT / 2; ++c)
    tile[h][(kCPT / 2) * part + c] = pack_bf16x2(acc[2 * c] * inv, acc[2 * c + 1] * inv);
  __syncthreads();
  // row h of the slice is 128 contiguous bytes of u: 8 threads per row, 16 bytes each
  for (int i = threadIdx.x; i < H * 8; i += kThreads) {
    const int row = i >> 3, q = i & 7;
    uint4 o;
    o.x = tile[row][4 * q];
    o.y = tile[row][4 * q + 1];
    o.z = tile[row][4 * q + 2];
    o.w = tile[row][4 * q + 3];
    *reinterpret_cast<uint4*>(u + ((size_t)bj * H + row) * kDC + blockIdx.y * kCols + 8 * q) = o;
  }
  if (lse_out && blockIdx.y == 0 && part == 0 && h < H)
    lse_out[(size_t)bj * H + h] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const Plan& plan, int B, int n_q, int H, uint16_t* u, float* lse,
                           cudaStream_t s) {
  dim3 grid(B * n_q, kDC / kCols);
  return launch_pdl(combine_kernel, grid, dim3(kThreads), 0, s, plan, n_q, H, u, lse);
}

}  // namespace mla
