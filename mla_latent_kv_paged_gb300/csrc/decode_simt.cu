// Paged MLA decode on CUDA cores (fp32 FMA): the straightforward kernel.
//
// Per (range piece, query j, group of 16 heads) one block streams the piece's
// pages through shared memory, scores all 16 heads against each 576-value
// row (latent c^KV followed by the rotated shared k^R: Huny's Dev Blog "MLA
// 아키텍처 해부" section 2.2), runs an online softmax, and accumulates the
// weighted latents (section 3.2, u = a C^KV). Writes the normalised partial
// and its log-sum-exp.
#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kHG = 16;              // heads per block
constexpr int kThreads = 256;        // 16 threads per head
constexpr int kRowWords = kRow / 2 + 1;  // 289 32-bit words per padded tile row

__global__ void __launch_bounds__(kThreads)
decode_simt_kernel(const uint16_t* __restrict__ q_abs, const uint16_t* __restrict__ cache,
                   const int32_t* __restrict__ block_table, int n_q, int H, int num_pages,
                   int max_pages, float scale, Plan plan) {
  extern __shared__ float smem_f[];
  float* Qs = smem_f;                                            // [16][576]
  uint32_t* tile = reinterpret_cast<uint32_t*>(Qs + kHG * kRow);  // [64][289] bf16x2
  float* S = reinterpret_cast<float*>(tile + kPage * kRowWords);  // [16][64]

  const int p = blockIdx.x, j = blockIdx.y, hg = blockIdx.z;
  const int tid = threadIdx.x, hl = tid >> 4, l16 = tid & 15;
  const int h = hg * kHG + hl;
  const int it0 = plan.range_item[p], it1 = plan.range_item[p + 1];

  for (int k = it0; k < it1; ++k) {
    const int b = plan.item_seq[k];
    const int pg0 = plan.item_page0[k], pg1 = plan.item_page1[k];
    const int L = plan.seq_len_eff[b];
    const int n_att = L - n_q + j + 1;
    const size_t qrow0 = ((size_t)b * n_q + j) * H;

    __syncthreads();
    for (int i = tid; i < kHG * kRow; i += kThreads) {
      const int hh = hg * kHG + i / kRow, e = i % kRow;
      Qs[i] = hh < H ? bf16_to_float(q_abs[(qrow0 + hh) * kRow + e]) : 0.f;
    }
    float O[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) O[i] = 0.f;
    float m = -INFINITY, l = 0.f;

    for (int pg = pg0; pg < pg1; ++pg) {
      const int tok0 = pg * kPage;
      const int ntok = min(kPage, n_att - tok0);
      if (ntok <= 0) break;
      int id = block_table[(size_t)b * max_pages + pg];
      const bool ok = id >= 0 && id < num_pages;
      __syncthreads();
      const uint32_t* src = reinterpret_cast<const uint32_t*>(cache + (size_t)(ok ? id : 0) * kPage * kRow);
      for (int i = tid; i < ntok * (kRow / 2); i += kThreads) {
        const int r = i / (kRow / 2), w = i % (kRow / 2);
        tile[r * kRowWords + w] = ok ? src[r * (kRow / 2) + w] : 0u;
      }
      __syncthreads();
      // scores: this thread's head against tokens l16, l16+16, l16+32, l16+48
      float sc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int tt = l16 + 16 * q;
        float acc = -INFINITY;
        if (tt < ntok) {
          acc = 0.f;
          const uint32_t* row = tile + tt * kRowWords;
          const float* qv = Qs + hl * kRow;
          for (int w = 0; w < kRow / 2; ++w) {
            const uint32_t x = row[w];
            acc = fmaf(qv[2 * w], bf16_lo(x), acc);
            acc = fmaf(qv[2 * w + 1], bf16_hi(x), acc);
          }
          acc *= scale;
        }
        sc[q] = acc;
      }
      float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float m_new = fmaxf(m, mt);
      const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
      float ps = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float pv = (sc[q] == -INFINITY) ? 0.f : expf(sc[q] - m_new);
        ps += pv;
        S[hl * kPage + l16 + 16 * q] = pv;
      }
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l = l * alpha + ps;
      m = m_new;
      __syncwarp();
      __syncthreads();
      // latent aggregation: features f = l16 + 16 i (only the first 512 columns)
#pragma unroll
      for (int i = 0; i < 32; ++i) O[i] *= alpha;
      for (int tt = 0; tt < ntok; ++tt) {
        const float pv = S[hl * kPage + tt];
        const uint16_t* row16 = reinterpret_cast<const uint16_t*>(tile + tt * kRowWords);
#pragma unroll
        for (int i = 0; i < 32; ++i) O[i] = fmaf(pv, bf16_to_float(row16[l16 + 16 * i]), O[i]);
      }
    }
    if (h < H) {
      const size_t orow = ((size_t)k * n_q + j) * H + h;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) plan.o_part[orow * kDC + l16 + 16 * i] = O[i] * inv;
      if (l16 == 0) plan.lse_part[orow] = l > 0.f ? m + logf(l) : -INFINITY;
    }
  }
}

}  // namespace

cudaError_t launch_decode(const uint16_t* q_abs, const uint16_t* cache, const int32_t* block_table,
                          int B, int n_q, int H, int num_pages, int max_pages, float scale, int G,
                          const Plan& plan, int32_t* err_word, cudaStream_t s) {
  (void)B;
  (void)err_word;
  const size_t smem = (size_t)kHG * kRow * 4 + (size_t)kPage * kRowWords * 4 + (size_t)kHG * kPage * 4;
  cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(G, n_q, (H + kHG - 1) / kHG);
  decode_simt_kernel<<<grid, kThreads, smem, s>>>(q_abs, cache, block_table, n_q, H, num_pages,
                                                  max_pages, scale, plan);
  return cudaGetLastError();
}

}  // namespace mla
