// Split-KV work plan: cuts the 64-token tiles of all sequences (in sequence
// order; a page of 64 tokens is one tile, a page of 128 two) into G contiguous
// ranges of near-equal cost and lists the (sequence, tile range) pieces each
// range covers. A range that moves on to another sequence pays for the switch
// (the accumulator of the finished piece is written out and the next query is
// loaded), so every sequence start after the first counts as kSwitchPages extra
// tiles: the cuts are equal steps along that longer line, and a cut that falls
// inside a switch lands on the sequence start.
// Flash-decoding over a paged cache: the Huny's Dev Blog "MLA 아키텍처 해부"
// section 4 table names FlashDecoding / PagedAttention as the decode
// techniques; section 6 item 2 sets MLA pages at 64-128 tokens.
//
// One block of 256 threads. Integer work only; the output is a pure function
// of (seq_lens, n_q, max_pages * page_size, G), so repeated calls give
// identical plans.
#include "mla_internal.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

constexpr int kPlanThreads = 256;  // barriers of a smaller block are cheaper; the work is light
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kSwitchPages = 3;

// Exclusive scan of v[0..n) in place (shared memory), returns the total.
// Every thread of the block must call it.
__device__ int block_exclusive_scan(int* v, int n, int* warp_sums) {
  const int tid = threadIdx.x;
  const int per = (n + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int local = 0;
  for (int i = lo; i < hi; ++i) local += v[i];
  // inclusive scan of `local` across the block
  int x = local;
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kPlanWarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kPlanWarps) warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  int excl = x - local + (warp > 0 ? warp_sums[warp - 1] : 0);
  const int total = warp_sums[kPlanWarps - 1];
  for (int i = lo; i < hi; ++i) {
    int t = v[i];
    v[i] = excl;
    excl += t;
  }
  __syncthreads();
  return total;
}

// a / b for a >= 0, b > 0: a 32-bit division when both fit (always at serving
// sizes), a 64-bit one otherwise; the same quotient either way
__device__ inline int64_t div_nn(int64_t a, int64_t b) {
  if (((uint64_t)a | (uint64_t)b) >> 32 == 0) return (int64_t)((uint32_t)a / (uint32_t)b);
  return a / b;
}
__device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return div_nn(a + b - 1, b); }

__global__ void __launch_bounds__(kPlanThreads, 1)
plan_kernel(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table, int B,
            int n_q, int max_tokens, int num_pages, int G, Plan plan, int32_t* err_word) {
  extern __shared__ int smem_i[];
  int* s_pstart = smem_i;            // [B+1] exclusive page prefix
  int* s_istart = smem_i + (B + 1);  // [B+1] exclusive piece prefix
  __shared__ int warp_sums[32];
  __shared__ int s_items;
  const int tid = threadIdx.x;
  // the next kernel may start at once: it reads the plan only after its own
  // grid dependency wait, which covers this kernel's completion
  sm100::grid_launch_dependents();

  // 1. clamp context lengths (to the block table's max_pages * page_size tokens), count tiles
  for (int b = tid; b < B; b += kPlanThreads) {
    int L = seq_lens[b];
    if (L < n_q) {
      report_error(err_word, MLA_ERR_BOUNDS);
      L = n_q;
    }
    if (L > max_tokens) {
      report_error(err_word, MLA_ERR_BOUNDS);
      L = max_tokens;
    }
    plan.seq_len_eff[b] = L;
    s_pstart[b] = (L + kTile - 1) / kTile;
  }
  __syncthreads();
  const int total = block_exclusive_scan(s_pstart, B, warp_sums);
  if (tid == 0) {
    s_pstart[B] = total;
  }
  __syncthreads();
  const int Ge = min(G, total);  // >= 1 since every sequence has >= 1 page
  // Cost line: sequence b's pages sit at [Q_b, Q_b + n_b), Q_b = P_b + a*b,
  // after a switch of a pages for b >= 1; length V = total + a*(B-1). Cut p
  // sits at x_p = floor(p*V/Ge). The switch cost is dropped (a = 0) when a
  // step along the line would not exceed it: steps of at least a+1 keep two
  // cuts from landing on the same sequence start, so no range is empty.
  const int64_t V0 = (int64_t)total + (int64_t)kSwitchPages * (B - 1);
  const int64_t a = (div_nn(V0, Ge) >= kSwitchPages + 1) ? kSwitchPages : 0;
  const int64_t V = (int64_t)total + a * (B - 1);

  // 2. pieces per sequence: cuts strictly inside (Q_b, Q_b + n_b)
  for (int b = tid; b < B; b += kPlanThreads) {
    const int64_t Qb = s_pstart[b] + a * b, Eq = s_pstart[b + 1] + a * b;
    int64_t lo = ceil_div64((Qb + 1) * Ge, V);
    int64_t hi = ceil_div64(Eq * Ge, V) - 1;
    lo = max(lo, (int64_t)1);
    hi = min(hi, (int64_t)Ge - 1);
    s_istart[b] = 1 + (int)max((int64_t)0, hi - lo + 1);
  }
  __syncthreads();
  const int items = block_exclusive_scan(s_istart, B, warp_sums);
  if (tid == 0) {
    s_istart[B] = items;
    s_items = items;
    plan.hdr[0] = items;
    plan.hdr[1] = Ge;
    plan.hdr[2] = total;
  }
  __syncthreads();

  // 3. write the pieces of each sequence
  for (int b = tid; b < B; b += kPlanThreads) {
    const int64_t Pb = s_pstart[b], Eb = s_pstart[b + 1];
    const int64_t Qb = Pb + a * b, Eq = Eb + a * b;
    int64_t lo = max(ceil_div64((Qb + 1) * Ge, V), (int64_t)1);
    int64_t hi = min(ceil_div64(Eq * Ge, V) - 1, (int64_t)Ge - 1);
    int k = s_istart[b];
    int64_t start = Pb;
    for (int64_t p = lo; p <= hi; ++p) {
      const int64_t x = div_nn(p * V, Ge) - a * b;  // global page of the cut
      plan.item_seq[k] = b;
      plan.item_tile0[k] = (int)(start - Pb);
      plan.item_tile1[k] = (int)(x - Pb);
      ++k;
      start = x;
    }
    plan.item_seq[k] = b;
    plan.item_tile0[k] = (int)(start - Pb);
    plan.item_tile1[k] = (int)(Eb - Pb);
    plan.seq_item[b] = s_istart[b];
  }
  if (tid == 0) plan.seq_item[B] = s_items;
  __syncthreads();  // the pieces are written: step 4 copies each range's first one

  // 4. first piece of each range, and its description (one 16-byte load for the
  // decode kernel's producer instead of two dependent ones)
  for (int p = tid; p <= G; p += kPlanThreads) {
    int r;
    if (p == 0) {
      r = 0;
    } else if (p >= Ge) {
      r = s_items;
    } else {
      const int64_t x = div_nn((int64_t)p * V, Ge);
      // largest b whose stretch of the line (switch, then pages) starts at or
      // before x: Q_b - a <= x for b >= 1 (strictly increasing in b)
      int lo = 0, hi = B - 1;
      while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (s_pstart[mid] + a * (mid - 1) <= x) lo = mid; else hi = mid - 1;
      }
      const int b = lo;
      const int64_t Qb = s_pstart[b] + a * b;
      if (x <= Qb) {  // on the switch into b or on its first page
        r = s_istart[b];
      } else {
        const int64_t first = max(ceil_div64((Qb + 1) * Ge, V), (int64_t)1);
        r = s_istart[b] + (int)(p - first + 1);
      }
    }
    plan.range_item[p] = r;
    int4 d = make_int4(r, -1, 0, 0);
    if (r < s_items) {
      d.y = plan.item_seq[r];
      d.z = plan.item_tile0[r];
      d.w = plan.item_tile1[r];
    }
    plan.range_desc[p] = d;
  }

  // Page ids are checked by the decode kernel when it reads them. The plan
  // does not read anything the previous kernel wrote, so it runs beside it;
  // it waits for that kernel only before finishing, so a kernel that waits
  // for the plan also sees everything written before it.
  sm100::grid_dependency_wait();
}

// The same plan for at most 32 sequences by one warp: lane b holds sequence b,
// prefix sums are warp scans, and the lane of sequence b also writes the
// ranges whose cut falls in b's part of the cost line (no search), so the plan
// needs no block barrier and no shared memory. The cut positions and their
// arithmetic are those of plan_kernel, so the two give identical plans.
__device__ __forceinline__ int warp_exclusive_scan(int v, int lane, int* total) {
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  *total = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

__global__ void __launch_bounds__(32, 1)
plan_small_kernel(const int32_t* __restrict__ seq_lens, int B, int n_q, int max_tokens, int G, Plan plan,
                  int32_t* err_word) {
  const int lane = threadIdx.x;
  sm100::grid_launch_dependents();
  const bool live = lane < B;
  int n_b = 0;  // tiles of sequence `lane`
  if (live) {
    int L = seq_lens[lane];
    if (L < n_q) {
      report_error(err_word, MLA_ERR_BOUNDS);
      L = n_q;
    }
    if (L > max_tokens) {
      report_error(err_word, MLA_ERR_BOUNDS);
      L = max_tokens;
    }
    plan.seq_len_eff[lane] = L;
    n_b = (L + kTile - 1) / kTile;
  }
  int total;
  const int P_b = warp_exclusive_scan(n_b, lane, &total);
  const int Ge = min(G, total);
  const int64_t V0 = (int64_t)total + (int64_t)kSwitchPages * (B - 1);
  const int64_t a = (div_nn(V0, Ge) >= kSwitchPages + 1) ? kSwitchPages : 0;
  const int64_t V = (int64_t)total + a * (B - 1);
  const int64_t Qb = P_b + a * lane, Eq = (int64_t)(P_b + n_b) + a * lane;
  const int64_t lo_b = max(ceil_div64((Qb + 1) * Ge, V), (int64_t)1);
  const int64_t hi_b = min(ceil_div64(Eq * Ge, V) - 1, (int64_t)Ge - 1);
  int items;
  const int I_b = warp_exclusive_scan(live ? 1 + (int)max((int64_t)0, hi_b - lo_b + 1) : 0, lane, &items);
  if (lane == 0) {
    plan.hdr[0] = items;
    plan.hdr[1] = Ge;
    plan.hdr[2] = total;
    plan.seq_item[B] = items;
  }
  if (live) {
    // the pieces of sequence b, and the ranges whose cut falls in b's part of the
    // cost line [Q_b - a, Eq_b) (from 0 for b = 0): a cut on the switch stretch,
    // x <= Q_b, starts its range at b's first piece, a cut inside b at its own
    const int64_t t1_first = lo_b <= hi_b ? div_nn(lo_b * V, Ge) - a * lane - P_b : n_b;
    const int64_t p_first = lane == 0 ? 0 : ceil_div64((Qb - a) * Ge, V);
    for (int64_t p = p_first; p < min(lo_b, (int64_t)Ge); ++p) {
      plan.range_item[p] = I_b;
      plan.range_desc[p] = make_int4(I_b, lane, 0, (int)t1_first);
    }
    int k = I_b;
    int64_t start = P_b;
    for (int64_t p = lo_b; p <= hi_b; ++p) {
      const int64_t x = div_nn(p * V, Ge) - a * lane;
      plan.item_seq[k] = lane;
      plan.item_tile0[k] = (int)(start - P_b);
      plan.item_tile1[k] = (int)(x - P_b);
      ++k;
      start = x;
      const int64_t x1 = p + 1 <= hi_b ? div_nn((p + 1) * V, Ge) - a * lane : P_b + n_b;
      plan.range_item[p] = k;
      plan.range_desc[p] = make_int4(k, lane, (int)(x - P_b), (int)(x1 - P_b));
    }
    plan.item_seq[k] = lane;
    plan.item_tile0[k] = (int)(start - P_b);
    plan.item_tile1[k] = n_b;
    plan.seq_item[lane] = I_b;
  }
  // ranges past the last cut are empty
  for (int p = Ge + lane; p <= G; p += 32) {
    plan.range_item[p] = items;
    plan.range_desc[p] = make_int4(items, -1, 0, 0);
  }
  sm100::grid_dependency_wait();
}

}  // namespace

cudaError_t launch_plan(const int32_t* seq_lens, const int32_t* block_table, int B, int n_q,
                        int max_pages, int page_size, int num_pages, int G, const Plan& plan, int32_t* err_word,
                        cudaStream_t s, bool overlap) {
  const int max_tokens = max_pages * page_size;
  if (B <= 32) {
    if (overlap)
      return launch_pdl(plan_small_kernel, dim3(1), dim3(32), 0, s, seq_lens, B, n_q, max_tokens, G, plan, err_word);
    plan_small_kernel<<<1, 32, 0, s>>>(seq_lens, B, n_q, max_tokens, G, plan, err_word);
    return cudaGetLastError();
  }
  const size_t smem = (size_t)2 * (B + 1) * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  if (overlap)
    return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), smem, s, seq_lens, block_table, B, n_q, max_tokens,
                      num_pages, G, plan, err_word);
  // after the previous kernel has finished (its grid dependency wait then returns at once)
  plan_kernel<<<1, kPlanThreads, smem, s>>>(seq_lens, block_table, B, n_q, max_tokens, num_pages, G, plan, err_word);
  return cudaGetLastError();
}

}  // namespace mla
