// Split-KV MLA decode over the paged latent cache on the 5th-generation tensor
// cores (tcgen05, sm_103a).
//
// What it computes (Huny's Dev Blog "MLA 아키텍처 해부", sections 2.2 and 3):
// for one sequence b, query j and all heads h at once,
//   z[h][s] = scale * q_abs[h] . row_s          (row_s = [c_s (512) ; k^R_s (64)])
//   m, l    = running max / sum of exp over the tokens of a page range
//   O[h]    = sum_s exp(z[h][s] - m) c_s        (u = a C^KV, before normalisation)
// and writes o = O / l and lse = m + ln l for the range.
//
// Layout of the work. One worker = a cluster of two CTAs on two SMs; CTA r
// owns the feature half r of every cache row: latent columns [256r, 256r+256)
// and positional columns [512+32r, 512+32r+32). It TMA-loads only its half of
// each 64-token tile (36 KB; a page of 64 tokens is one tile, a page of 128
// two), so every cached byte is read from HBM once. The 128 heads share every
// tile in shared memory (the reuse the absorbed formulation creates).
//
// Scores need all 576 columns: each CTA computes a partial score
// S_r[128 heads][64 tokens] (K = 288) with tcgen05 MMAs into tensor memory.
// The softmax of a page is split by tokens: CTA r finishes tokens
// [32r, 32r+32). It sends the partial scores of the other 32 tokens to the
// peer (log2 units, as fp16 offsets from a per-head midpoint sent in fp32:
// 8.5 KB, st.async into the peer's shared memory), adds the peer's partial for
// its own tokens, and both CTAs exchange their page
// maxima so they share one exact running maximum per head. Each CTA then
// exponentiates its 32 tokens into P (bf16): its own half goes to tensor
// memory (the A operand of its value MMAs), a copy to the peer's shared
// memory (the peer's A operand for those 16-token K steps). Each CTA
// accumulates its 256-column half of O[128][512] in tensor memory with the
// value MMAs (P x C[64][256]).
//
// Tensor memory (512 columns x 128 lanes of 32 bits): O [0,256), S [256,320),
// this CTA's P half for three pages [320,368), the CTA's positional query half
// [368,384) and latent query half [384,512), the A operands of the score MMAs.
// Shared memory: 5-slot ring (180 KB) of page halves and, at the start of each
// range, the query half (TMA into two slots; the score readers move it into
// tensor memory), the peer's partial scores (one 8.5 KB
// buffer per softmax group), the peer's P half (3 x 8 KB), the exchange vectors.
//
// Warps: 0 = TMA producer, 1 = score-MMA issuer (and TMEM owner), 2 =
// value-MMA issuer, 3..6 = score readers (the peer's tokens of S, the query
// stage-in from the ring into tensor memory), 7..14 =
// softmax and epilogue in two groups of four warps that take alternate pages
// (one thread per head row, the CTA's 32 tokens of the page). The score MMAs
// of page g+1 run while the softmax of page g is in flight; the value MMAs
// trail by one page.
#include "mla_internal.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kStages = 5;
constexpr int kAWarps = 4;  // score readers: one per TMEM lane quadrant
constexpr int kBWarps = 8;  // softmax: two groups of four (one per lane quadrant), alternate pages
constexpr int kAThreads = kAWarps * 32, kBThreads = kBWarps * 32;
constexpr int kGThreads = kBThreads / 2;  // one softmax group: a thread per head row
constexpr int kThreads = 96 + kAThreads + kBThreads;
constexpr uint32_t kCBoxBytes = 64 * 128;   // [64 tokens][64 latent cols] bf16, 128B swizzle
constexpr uint32_t kKrBoxBytes = 64 * 64;   // [64 tokens][32 positional cols] bf16, 64B swizzle
constexpr uint32_t kStageBytes = 4 * kCBoxBytes + kKrBoxBytes;  // 36864
constexpr uint32_t kQrBoxBytes = 64 * 64;   // [64 heads][32 positional cols] bf16, 64B swizzle
constexpr uint32_t kQBoxBytes = 128 * 128;  // [128 heads][64 latent cols] bf16, 128B swizzle
constexpr int kQSlots = 2;                  // ring slots taken by a range's latent query half (4 boxes)
constexpr uint32_t kVecBytes = 128 * 4;     // one float per head
// peer partial scores: [4 groups of 8 tokens][128 heads] fp16 offsets from a per-head
// midpoint, then the midpoints [128 heads] fp32 (log2 units)
constexpr uint32_t kXDataBytes = 4 * 128 * 16;
constexpr uint32_t kXBytes = kXDataBytes + kVecBytes;
constexpr uint32_t kPPeerBytes = 128 * 64;  // the peer's half of P: [128 heads][32 tokens] bf16, 64B swizzle
constexpr uint32_t kPHalfBytes = kPPeerBytes;
constexpr int kPBufs = 3;  // P buffers: page g uses g % 3, so its writers wait for page g - 3
constexpr uint32_t kTokBytes = 4 * 4;       // "partial consumed" tokens: one per warp of a group
// FP8 cache: a CTA's half of a page (e4m3 codes, [64 tokens][256 latent + 32
// positional columns], rows of 64 and 32 bytes) lands in the upper half of its
// ring slot, and the score readers expand it in place into the layout of the
// 16-bit page half above (fp16 values: e4m3 converts to fp16 exactly).
constexpr uint32_t kF8CBoxBytes = 64 * 64;   // [64 tokens][64 latent cols] e4m3
constexpr uint32_t kF8KrBoxBytes = 16 * 32;  // [16 tokens][32 positional cols] e4m3, four per page half
constexpr uint32_t kF8StageBytes = 4 * kF8CBoxBytes + 4 * kF8KrBoxBytes;  // 18432
constexpr uint32_t kF8Off = kStageBytes - kF8StageBytes;              // 18432
constexpr int kF8Chunks = kF8StageBytes / 16;  // 16-byte chunks of a page half: 1152

constexpr uint32_t kOffStage = 0;
constexpr uint32_t kOffX = kOffStage + kStages * kStageBytes;  // peer partial scores, one buffer per group
constexpr uint32_t kOffP = kOffX + 2 * kXBytes;        // the peer's half of P, two pages
constexpr uint32_t kOffMX = kOffP + kPBufs * kPPeerBytes;  // peer page maxima [2 groups][128]
constexpr uint32_t kOffLX = kOffMX + 2 * kVecBytes;  // peer softmax sums [2 ranges][128]
constexpr uint32_t kOffMR = kOffLX + 2 * kVecBytes;    // reference maximum after the latest page [128]
constexpr uint32_t kOffLG = kOffMR + kVecBytes;        // handed-over group sums [2 ranges][sum, ref][128]
constexpr uint32_t kOffIV = kOffLG + 4 * kVecBytes;    // 1 / softmax sum of the range [128]
constexpr uint32_t kOffTok = kOffIV + kVecBytes;       // tokens from the peer
constexpr uint32_t kOffBar = kOffTok + kTokBytes;

// barrier indices. A barrier that completes once per page and is waited by
// only one of the two softmax groups exists once per group (index g % 2): a
// parity wait is only sound if the barrier's previous phase is one this
// waiter has already seen complete.
enum {
  FULL0 = 0, EMPTY0 = FULL0 + kStages, QCF = EMPTY0 + kStages,
  SF0 = QCF + 1, SFREE = SF0 + 2, PF0 = SFREE + 1, PVD0 = PF0 + kPBufs, XF0 = PVD0 + kPBufs, XE0 = XF0 + 2,
  MXF0 = XE0 + 2, LXF0 = MXF0 + 2, MRF = LXF0 + 2, LGF0 = MRF + 1, IVF0 = LGF0 + 2, OFREE = IVF0 + 2,
  MMAD = OFREE + 1,
  // FP8 cache only: CVF = a ring slot's 16-bit page half (or query) is in place
  // (every use of a slot completes it once, so its phases follow FULL's); CVR =
  // every score reader has read its share of the codes of the page being expanded
  CVF0 = MMAD + 1, CVR = CVF0 + kStages,
  kNumBars = CVR + 1
};
constexpr uint32_t kOffSlots = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffSlots + 16;  // the base is checked to be 1024-byte aligned
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(2 * kQBoxBytes + kQrBoxBytes <= kStageBytes, "a ring slot holds a query quarter");

// tensor memory columns: O[128][256] fp32, S[128][64] fp32, this CTA's half of P
// (bf16 pairs) for two pages, the CTA's latent half of q_abs (bf16 pairs)
constexpr uint32_t kTmO = 0, kTmS = 256, kTmP = 320, kTmQr = 368, kTmQ = 384, kTmCols = 512;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P values stay <= 256

#if MLA_DEBUG_CHECKS
// Test builds only (libmla_gb300_debug.so): counters read by the host through
// mla_debug_read_counters, and a switch that keeps the producer from loading
// anything so that the consumers' bounded waits give up.
//   [0] warps that rescaled O (the running maximum rose past the threshold)
//   [1] shared-memory or tensor-memory addresses outside this CTA's allocation
__device__ unsigned long long g_dbg_counters[4];
__device__ int g_dbg_skip_producer;
__device__ __noinline__ bool dbg_check(bool ok, int32_t* err_word) {
  if (!ok) {
    atomicAdd(&g_dbg_counters[1], 1ull);
    report_error(err_word, MLA_ERR_BOUNDS);
  }
  return ok;
}
// true when [addr, addr + bytes) lies inside this CTA's dynamic shared memory
// (for an address of the peer CTA: the same offset before mapa)
#define MLA_SMEM_OK(addr, bytes) \
  dbg_check((addr) >= sbase && (uint64_t)(addr) + (bytes) <= (uint64_t)sbase + kSmemBytes, err_word)
#define MLA_TMEM_OK(col, ncols) dbg_check((uint32_t)(col) + (ncols) <= (uint32_t)kTmCols, err_word)
#else
#define MLA_SMEM_OK(addr, bytes) true
#define MLA_TMEM_OK(col, ncols) true
#endif


// kF8: the cache holds e4m3 codes with a scale per column (fp8_scales, 576
// floats). The scales are folded into the query (scores) and into the written
// partials (values), the codes are expanded to fp16 in shared memory, and the
// MMAs run on fp16 operands (the query, P and the page, kind::f16 with fp16
// inputs); the bf16 path is unchanged.
__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr));
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
// Four e4m3 codes (byte i = value i) -> fp16 pairs: values 0,1 in lo, 2,3 in hi
// (exact: every e4m3 value is an fp16 value).
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
// bf16 pair times two scales, as an fp16 pair
__device__ __forceinline__ uint32_t scale_bf16x2_to_f16x2(uint32_t w, float s0, float s1) {
  return cvt_f16x2(bf16_lo(w) * s0, bf16_hi(w) * s1);
}

template <bool kF8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap map_c, const __grid_constant__ CUtensorMap map_kr,
                 const __grid_constant__ CUtensorMap map_qkr, const __grid_constant__ CUtensorMap map_q,
                 const int32_t* __restrict__ block_table, int n_q, int H, int max_pages, int num_pages,
                 int tile_shift, float sl2, Plan plan, const float* __restrict__ fp8_scales, int32_t* err_word) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) report_error(err_word, MLA_ERR_CUDA);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int worker = blockIdx.x >> 1, j = blockIdx.y;
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffSlots + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(FULL0 + i), 1);
      mbar_init(bar(EMPTY0 + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(LXF0 + i), 1);
      mbar_init(bar(LGF0 + i), kGThreads);  // a group's sums handed over
      mbar_init(bar(IVF0 + i), kGThreads);  // 1/l posted for helper group i
    }
    for (int i = 0; i < kPBufs; ++i) {
      mbar_init(bar(PF0 + i), kGThreads + 1);  // a group's rows + the arming arrive for the peer's half
      mbar_init(bar(PVD0 + i), 2);             // the value MMAs of the page done in both CTAs
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(SF0 + i), 1);
      mbar_init(bar(XF0 + i), 1);  // armed here, filled by the peer's st.async
      mbar_init(bar(XE0 + i), 1);  // armed here, completed by the peer's four 4-byte tokens
      mbar_init(bar(MXF0 + i), 1);
    }
    mbar_init(bar(SFREE), kAThreads + kGThreads);

    mbar_init(bar(MRF), kGThreads);  // the reference maximum of a page posted
    mbar_init(bar(QCF), kAThreads);  // the range's latent query half is in tensor memory
    mbar_init(bar(OFREE), 2 * kGThreads);        // both halves of O drained
    mbar_init(bar(MMAD), 2);  // both MMA issuers done
    if (kF8) {
      for (int i = 0; i < kStages; ++i) mbar_init(bar(CVF0 + i), kAThreads);
      mbar_init(bar(CVR), kAThreads);
    }
    *abort_flag = 0;
    fence_mbar_init();
    for (int i = 0; i < kPBufs; ++i) mbar_arrive_expect_tx(bar(PF0 + i), kPHalfBytes);
    for (int i = 0; i < 2; ++i) {
      mbar_arrive_expect_tx(bar(LXF0 + i), kVecBytes);
      mbar_arrive_expect_tx(bar(XF0 + i), kXBytes);
      mbar_arrive_expect_tx(bar(XE0 + i), kTokBytes);
      mbar_arrive_expect_tx(bar(MXF0 + i), kVecBytes);
    }
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map_c);
    prefetch_tmap(&map_kr);
    prefetch_tmap(&map_qkr);
    prefetch_tmap(&map_q);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers are initialised before any remote arrive
  const uint32_t tmem = *tmem_slot;
  // set-up above overlaps the plan kernel; the plan and q_abs are read below
  grid_dependency_wait();
  grid_launch_dependents();
  const int it0 = plan.range_item[worker], it1 = plan.range_item[worker + 1];

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Loads this CTA's half of each page into the stage ring.
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    int stage = 0;
    uint32_t ph = 0;
    int last_ph[kStages];
#pragma unroll
    for (int i = 0; i < kStages; ++i) last_ph[i] = -1;
    bool ok = true;
    // tile cursors over (range, tile): lanes hold the page ids of 32 consecutive
    // tiles (a page holds 1 << tile_shift tiles of 64 tokens)
    const int tile_mask = (1 << tile_shift) - 1;
    struct Cursor {
      int it, pg, pg1, base, id_l, pg0, seq;  // pg0, seq: the piece's first tile and its sequence
      size_t row;  // block-table row of the current range
    };
    auto cur_load = [&](Cursor& c) {
      const int mine = c.base + lane;
      c.id_l = mine < c.pg1 ? block_table[c.row + (mine >> tile_shift)] : 0;
    };
    auto cur_init = [&](Cursor& c, int it) {
      c.it = it;
      if (it < it1) {
        c.seq = plan.item_seq[it];
        c.row = (size_t)c.seq * max_pages;
        c.pg = c.base = c.pg0 = plan.item_tile0[it];
        c.pg1 = plan.item_tile1[it];
        cur_load(c);
      }
    };
    auto cur_next = [&](Cursor& c) -> int {  // page id of the tile at the cursor, then advance
      const int id = __shfl_sync(0xffffffffu, c.id_l, c.pg - c.base);
      if (++c.pg == c.pg1) {
        cur_init(c, c.it + 1);
      } else if (c.pg - c.base == 32) {
        c.base = c.pg;
        cur_load(c);
      }
      return id;
    };
    Cursor ld;
    {  // the range's first piece from its 16-byte description
      const int4 d0 = plan.range_desc[worker];
      ld.it = d0.x;
      if (d0.x < it1) {
        ld.seq = d0.y;
        ld.row = (size_t)d0.y * max_pages;
        ld.pg = ld.base = ld.pg0 = d0.z;
        ld.pg1 = d0.w;
        cur_load(ld);
      }
    }
#if MLA_DEBUG_CHECKS
    if (*reinterpret_cast<volatile int*>(&g_dbg_skip_producer)) ld.it = it1;  // load nothing
#endif
    while (ok && ld.it < it1) {
      if (ld.pg == ld.pg0) {
        // first page of a range: the CTA's half of its query into the next two
        // ring slots (the score readers move it into tensor memory). Slot q holds
        // latent boxes [128 heads][64] for columns 256r + 128q + {0, 64} and, in
        // its last 4 KB, positional rows [64q, 64q + 64) of columns 512 + 32r.
        const int qrow = (ld.seq * n_q + j) * H;
        for (int q = 0; q < kQSlots && ok; ++q) {
          if (!wait_phase(bar(EMPTY0 + stage), ph ^ 1u, abort_flag, err_word)) { ok = false; break; }
          if (lane == 0 && MLA_SMEM_OK(sbase + kOffStage + stage * kStageBytes, kStageBytes)) {
            const uint32_t fb = bar(FULL0 + stage);
            const uint32_t dst = sbase + kOffStage + stage * kStageBytes;
            mbar_arrive_expect_tx(fb, 2 * kQBoxBytes + kQrBoxBytes);
            for (int m = 0; m < 2; ++m)
              tma_load_2d(dst + m * kQBoxBytes, &map_q, fb, 256 * (int)rank + 128 * q + 64 * m, qrow, pol_keep);
            tma_load_2d(dst + 2 * kQBoxBytes, &map_qkr, fb, kDC + 32 * (int)rank, qrow + 64 * q, pol_keep);
          }
          last_ph[stage] = (int)ph;
          __syncwarp();
          if (++stage == kStages) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
      }
      const int sub = ld.pg & tile_mask;  // the tile's place in its page
      const int pid = cur_next(ld);
      // an id outside the pool loads zeros (TMA bounds) and is reported
      if (lane == 0 && (pid < 0 || pid >= num_pages)) report_error(err_word, MLA_ERR_BOUNDS);
      if (!wait_phase(bar(EMPTY0 + stage), ph ^ 1u, abort_flag, err_word)) { ok = false; break; }
      if (lane == 0 && MLA_SMEM_OK(sbase + kOffStage + stage * kStageBytes, kStageBytes)) {
        const uint32_t fb = bar(FULL0 + stage);
        const uint32_t dst = sbase + kOffStage + stage * kStageBytes;
        const int y = ((pid << tile_shift) + sub) * kTile;
        if (kF8) {
          // the codes into the upper half of the slot, unswizzled rows
          mbar_arrive_expect_tx(fb, kF8StageBytes);
#pragma unroll
          for (int cb = 0; cb < 4; ++cb)
            tma_load_2d(dst + kF8Off + cb * kF8CBoxBytes, &map_c, fb, 256 * (int)rank + 64 * cb, y, pol_stream);
          // the positional codes as four boxes of 16 rows (same bytes, same place as
          // one box of 64 rows; measured 1.5% faster per call at 32 x 4096)
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            tma_load_2d(dst + kF8Off + 4 * kF8CBoxBytes + kb * kF8KrBoxBytes, &map_kr, fb, kDC + 32 * (int)rank,
                        y + 16 * kb, pol_stream);
        } else {
          mbar_arrive_expect_tx(fb, kStageBytes);
#pragma unroll
          for (int cb = 0; cb < 4; ++cb)
            tma_load_2d(dst + cb * kCBoxBytes, &map_c, fb, 256 * (int)rank + 64 * cb, y, pol_stream);
          tma_load_2d(dst + 4 * kCBoxBytes, &map_kr, fb, kDC + 32 * (int)rank, y, pol_stream);
        }
      }
      last_ph[stage] = (int)ph;
      __syncwarp();
      if (++stage == kStages) { stage = 0; ph ^= 1u; }
    }
    if (!ok) {
      // let every issued copy land before this CTA can exit
#pragma unroll
      for (int i = 0; i < kStages; ++i) {
        if (last_ph[i] >= 0) {
          const long long t0 = clock64();
          while (!mbar_try_wait(bar(FULL0 + i), (uint32_t)last_ph[i]) && clock64() - t0 < kWaitLimitCycles) {
          }
        }
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Two threads feed the tensor pipe: warp 1 the score MMAs, warp 2 the value
    // MMAs. An MMA issue stalls at the pipe's execution rate, so with one
    // issuer the pipe idled whenever that thread waited for P or for a tile;
    // with two, whichever has work ready keeps it busy. A value MMA of a page
    // follows that page's score MMAs through S -> P, so its commit (EMPTY)
    // also covers the page's score MMAs.
    if (lane == 0) {
      constexpr uint32_t kIdQK = kF8 ? idesc_f16(128, 64, false, false) : idesc_bf16(128, 64, false, false);
      constexpr uint32_t kIdPV = kF8 ? idesc_f16(128, 256, false, true) : idesc_bf16(128, 256, false, true);
      // descriptor templates; the start address is added per use
      const uint64_t dQK_c = smem_desc(0, 16, 1024, kSwizzle128B);
      const uint64_t dQK_r = smem_desc(0, 16, 512, kSwizzle64B);
      const uint64_t dPV_a = smem_desc(0, 16, 512, kSwizzle64B);  // the peer's half of P
      const uint64_t dPV_b = smem_desc(0, kCBoxBytes, 1024, kSwizzle128B);
      // start-address field: 14 bits of (shared address >> 4). Shared
      // addresses of the second CTA of a cluster carry high bits that must
      // not spill into the neighbouring descriptor fields.
      auto da = [](uint32_t addr) -> uint64_t { return (uint64_t)((addr >> 4) & 0x3FFFu); };
      bool ok = true;
      int g = 0, stage = 0;
      uint32_t ph = 0;
      if (warp == 1) {
        // ---- score MMAs: S = q_abs half . [c ; k^R] half of the page
        for (int it = it0; it < it1 && ok; ++it) {
          const int li = it - it0;
          const int ntiles = plan.item_tile1[it] - plan.item_tile0[it];
          // the range's query: the score readers have moved the latent and
          // positional halves from their two ring slots into tensor memory (and
          // read the slots: free them)
          if (!wait_phase(bar(QCF), li & 1, abort_flag, err_word)) { ok = false; break; }
          for (int q = 0; q < kQSlots; ++q) {
            mbar_arrive(bar(EMPTY0 + stage));
            if (++stage == kStages) { stage = 0; ph ^= 1u; }
          }
          for (int i = 0; i < ntiles; ++i, ++g) {
            // an FP8 page is expanded by the score readers after it lands (CVF)
            if (!wait_phase(bar((kF8 ? CVF0 : FULL0) + stage), ph, abort_flag, err_word) ||
                !wait_phase(bar(SFREE), (g & 1) ^ 1, abort_flag, err_word)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d = tmem + kTmS;
            const uint64_t bc = dQK_c + da(sbase + kOffStage + stage * kStageBytes);
#pragma unroll
            for (int ks = 0; ks < 16; ++ks)
              mma_ts(d, tmem + kTmQ + ks * 8, bc + (((ks >> 2) * kCBoxBytes + (ks & 3) * 32) >> 4), kIdQK,
                     ks > 0 ? 1u : 0u);
            // positional part: A = the positional query half in tensor memory
            const uint64_t br = dQK_r + da(sbase + kOffStage + stage * kStageBytes + 4 * kCBoxBytes);
            mma_ts(d, tmem + kTmQr, br, kIdQK, 1u);
            mma_ts(d, tmem + kTmQr + 8, br + 2, kIdQK, 1u);
            mma_commit(bar(SF0 + (g & 1)));
            if (++stage == kStages) { stage = 0; ph ^= 1u; }
          }
        }
      } else {
        // ---- value MMAs: O += P . C half, P from tensor memory (this CTA's
        // tokens) and from shared memory (the peer's tokens)
        for (int it = it0; it < it1 && ok; ++it) {
          const int li = it - it0;
          const int ntiles = plan.item_tile1[it] - plan.item_tile0[it];
          for (int q = 0; q < kQSlots; ++q)  // the range's query slots (released by the score issuer)
            if (++stage == kStages) { stage = 0; ph ^= 1u; }
          for (int i = 0; i < ntiles; ++i, ++g) {
            const int pb = g % kPBufs;
            if (!wait_phase(bar(PF0 + pb), (g / kPBufs) & 1, abort_flag, err_word)) { ok = false; break; }
            // the first value MMA of a range overwrites O: the previous range's
            // epilogue must have read it
            if (i == 0 && li > 0 && !wait_phase(bar(OFREE), (li - 1) & 1, abort_flag, err_word)) { ok = false; break; }
            // arm the P buffer for page g+2; its peer half can only come after
            // this page's value MMAs (waited through PVD by the peer)
            mbar_arrive_expect_tx(bar(PF0 + pb), kPHalfBytes);
            tc_fence_after();
            const uint64_t ad = dPV_a + da(sbase + kOffP + pb * kPPeerBytes);
            const uint64_t bd = dPV_b + da(sbase + kOffStage + stage * kStageBytes);
            const uint32_t am = tmem + kTmP + 16 * pb;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint32_t acc = (i > 0 || ks > 0) ? 1u : 0u;
              if ((ks >> 1) == (int)rank)
                mma_ts(tmem + kTmO, am + 8 * (ks & 1), bd + (ks * 2048 >> 4), kIdPV, acc);
              else
                mma_ss(tmem + kTmO, ad + ((ks & 1) * 32 >> 4), bd + (ks * 2048 >> 4), kIdPV, acc);
            }
            mma_commit_multicast(bar(PVD0 + pb), 0x3);
            mma_commit(bar(EMPTY0 + stage));
            if (++stage == kStages) { stage = 0; ph ^= 1u; }
          }
        }
      }
      (void)ph;
      mma_commit(bar(MMAD));
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ score readers and softmax
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // head row == TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + kTmS, tO = tmem + lane_off + kTmO;
    const uint32_t r_x = mapa(sbase + kOffX, peer), r_p = mapa(sbase + kOffP, peer);
    const uint32_t r_lx = mapa(sbase + kOffLX, peer), r_mx = mapa(sbase + kOffMX, peer);
    const uint32_t r_xf = mapa(bar(XF0), peer), r_xe = mapa(bar(XE0), peer), r_pf = mapa(bar(PF0), peer);
    const uint32_t r_lxf = mapa(bar(LXF0), peer), r_mxf = mapa(bar(MXF0), peer);
    const uint32_t r_tok = mapa(sbase + kOffTok, peer);

    if (warp < 3 + kAWarps) {
      // -------------------------------------------------------- A: score readers
      // Per page: read the peer's 32 tokens of this CTA's partial scores and send
      // them (log2 units, fp16) into the peer's shared memory.
      const int atid = threadIdx.x - 96;  // 0 .. 127
      const uint32_t tQ = tmem + lane_off + kTmQ;
      int g = 0;
      bool ok = true;
      // FP8 cache: expand the codes of page gg (range li) in place into the fp16
      // page half the MMAs read. Every reader first loads its 9 of the 1152
      // 16-byte chunks (the codes sit in the upper half of the slot, which the
      // expansion overwrites), all readers meet (CVR), then each writes its
      // chunks' 16 values as two 16-byte chunks of the swizzled layout of the
      // TMA boxes of the bf16 path. Pages are expanded in order, at most two
      // ahead of the page whose scores are being read and never beyond the
      // current range (the next range's query slots come first in the ring).
      int cv_n = 0, cv_next = 0, cv_last = -1;
      auto expand = [&](int gg, int lii) -> bool {
        const int slot = gg + kQSlots * (lii + 1);
        const int st = slot % kStages;
        if (!wait_phase(bar(FULL0 + st), (slot / kStages) & 1, abort_flag, err_word)) return false;
        const uint32_t sb = sbase + kOffStage + st * kStageBytes;
        uint32_t v[9][4];
#pragma unroll
        for (int k = 0; k < 9; ++k)
          ld_shared_v4(sb + kF8Off + (uint32_t)(atid + 128 * k) * 16, v[k][0], v[k][1], v[k][2], v[k][3]);
        mbar_arrive(bar(CVR));
        if (!wait_phase(bar(CVR), cv_n & 1, abort_flag, err_word)) return false;
        ++cv_n;
#pragma unroll
        for (int k = 0; k < 9; ++k) {
          const uint32_t q = (uint32_t)atid + 128u * k;
          uint32_t a0, a1;
          if (q < 1024) {  // latent box q / 256, token row, 16 of its 64 columns
            const uint32_t cb = q >> 8, t = (q >> 2) & 63, kk = q & 3;
            const uint32_t base = sb + cb * kCBoxBytes + t * 128;
            a0 = base + (((2 * kk) ^ (t & 7)) * 16);
            a1 = base + (((2 * kk + 1) ^ (t & 7)) * 16);
          } else {  // positional box: token row, 16 of its 32 columns (64B swizzle)
            const uint32_t qq = q - 1024, t = qq >> 1, kk = qq & 1;
            const uint32_t base = sb + 4 * kCBoxBytes + t * 64;
            a0 = base + (((2 * kk) ^ ((t >> 1) & 3)) * 16);
            a1 = base + (((2 * kk + 1) ^ ((t >> 1) & 3)) * 16);
          }
          uint32_t o[8];
          e4m3x4_to_f16(v[k][0], o[0], o[1]);
          e4m3x4_to_f16(v[k][1], o[2], o[3]);
          e4m3x4_to_f16(v[k][2], o[4], o[5]);
          e4m3x4_to_f16(v[k][3], o[6], o[7]);
          if (MLA_SMEM_OK(a0, 16) && MLA_SMEM_OK(a1, 16)) {
            st_shared_v4(a0, o[0], o[1], o[2], o[3]);
            st_shared_v4(a1, o[4], o[5], o[6], o[7]);
          }
        }
        fence_proxy_async_smem();  // read by the MMAs (async proxy)
        mbar_arrive(bar(CVF0 + st));
        return true;
      };
      auto expand_upto = [&](int target, int lii) -> bool {
        if (target > cv_last) target = cv_last;
        while (cv_next <= target) {
          if (!expand(cv_next, lii)) return false;
          ++cv_next;
        }
        return true;
      };

      for (int it = it0; it < it1 && ok; ++it) {
        const int li = it - it0;
        const int pg0 = plan.item_tile0[it];
        const int ntiles = plan.item_tile1[it] - pg0;
        const int n_att = plan.seq_len_eff[plan.item_seq[it]] - n_q + j + 1;  // tokens query j attends
        // the range's latent query half: this thread's head row from the two ring
        // slots (four [128][64] boxes, 128B-swizzled: 16-byte chunk c of row r at
        // c ^ (r % 8)) into tensor memory. The previous range's score MMAs are done
        // (this warp read the S of its last page), so Q may be overwritten.
        for (int q = 0; q < kQSlots && ok; ++q) {
          const int slot = g + kQSlots * li + q;
          if (!wait_phase(bar(FULL0 + slot % kStages), (slot / kStages) & 1, abort_flag, err_word)) { ok = false; break; }
          const uint32_t sq = sbase + kOffStage + (slot % kStages) * kStageBytes + (uint32_t)row * 128;
          (void)MLA_SMEM_OK(sq + kQBoxBytes, 128);
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            uint32_t r[32];
#pragma unroll
            for (int c = 0; c < 8; ++c)
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(r[4 * c]), "=r"(r[4 * c + 1]), "=r"(r[4 * c + 2]), "=r"(r[4 * c + 3])
                           : "r"(sq + m * kQBoxBytes + ((c ^ (row & 7)) * 16)));
            if (kF8) {  // the FP8 cache's column scales fold into the query (fp16)
              const float* sc = fp8_scales + 256 * rank + 128 * q + 64 * m;
#pragma unroll
              for (int k = 0; k < 32; ++k) r[k] = scale_bf16x2_to_f16x2(r[k], __ldg(sc + 2 * k), __ldg(sc + 2 * k + 1));
            }
            tmem_st32(tQ + 64 * q + 32 * m, r);
          }
          if ((row >> 6) == q) {  // this row's positional half: 64 bytes, 64B-swizzled (warp-uniform)
            const uint32_t sr = sbase + kOffStage + (slot % kStages) * kStageBytes + 2 * kQBoxBytes;
            const int rl = row & 63;
            uint32_t r[16];
#pragma unroll
            for (int c = 0; c < 4; ++c)
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(r[4 * c]), "=r"(r[4 * c + 1]), "=r"(r[4 * c + 2]), "=r"(r[4 * c + 3])
                           : "r"(sr + rl * 64 + ((c ^ ((rl >> 1) & 3)) * 16)));
            if (kF8) {
              const float* sc = fp8_scales + kDC + 32 * rank;
#pragma unroll
              for (int k = 0; k < 16; ++k) r[k] = scale_bf16x2_to_f16x2(r[k], __ldg(sc + 2 * k), __ldg(sc + 2 * k + 1));
            }
            tmem_st16(tmem + lane_off + kTmQr, r);
          }
          // every use of a ring slot completes its CVF once (the query's too)
          if (kF8) mbar_arrive(bar(CVF0 + slot % kStages));
        }
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(QCF));
        if (kF8) {  // the range's first page, expanded before its score MMAs
          cv_next = g;
          cv_last = g + ntiles - 1;
          if (!expand_upto(g, li)) { ok = false; break; }
        }
        for (int i = 0; i < ntiles; ++i, ++g) {
          if (!wait_phase(bar(SF0 + (g & 1)), (g >> 1) & 1, abort_flag, err_word)) { ok = false; break; }
          tc_fence_after();
          uint32_t r[32];
          tmem_ld32(tS + 32 * peer, r);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(SFREE));
          // the peer has read this CTA's partial of page g-2 (same buffer)
          if (g >= 2) {
            if (!wait_phase(bar(XE0 + (g & 1)), ((g >> 1) & 1) ^ 1, abort_flag, err_word)) { ok = false; break; }
            if (atid == 0) mbar_arrive_expect_tx(bar(XE0 + (g & 1)), kTokBytes);  // arm for this page
          }
          // The partial scores go out as fp16 offsets from the midpoint of this head's
          // values (sent in fp32): the rounding error then follows the spread of the
          // scores within the 32 tokens, not their size (a score shared by the tokens
          // costs no precision). Only tokens the query attends count toward the
          // midpoint; slack rows past the context may hold any bits.
          float v[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]) * sl2;
          const int nvp = n_att - ((pg0 + i) * kTile + 32 * (int)peer);  // attended among the 32
          float hi = -INFINITY, lo = INFINITY;
          if (nvp >= 32) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              hi = fmaxf(hi, v[k]);
              lo = fminf(lo, v[k]);
            }
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (k < nvp) {
                hi = fmaxf(hi, v[k]);
                lo = fminf(lo, v[k]);
              }
          }
          const float mid = lo <= hi ? 0.5f * lo + 0.5f * hi : 0.f;
          const uint32_t xoff = (uint32_t)(g & 1) * kXBytes;
          const uint32_t xa = r_x + xoff + (uint32_t)row * 16;
          const uint32_t xf = r_xf + 8u * (uint32_t)(g & 1);
          if (MLA_SMEM_OK(sbase + kOffX + xoff + (uint32_t)row * 16 + 3 * 128 * 16, 16) &&
              MLA_SMEM_OK(sbase + kOffX + xoff + kXDataBytes + (uint32_t)row * 4, 4)) {
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
              uint4 w;
              w.x = cvt_f16x2(v[8 * q8 + 0] - mid, v[8 * q8 + 1] - mid);
              w.y = cvt_f16x2(v[8 * q8 + 2] - mid, v[8 * q8 + 3] - mid);
              w.z = cvt_f16x2(v[8 * q8 + 4] - mid, v[8 * q8 + 5] - mid);
              w.w = cvt_f16x2(v[8 * q8 + 6] - mid, v[8 * q8 + 7] - mid);
              st_async_v4(xa + q8 * 128 * 16, w, xf);
            }
            st_async_b32(r_x + xoff + kXDataBytes + (uint32_t)row * 4, __float_as_uint(mid), xf);
          }
          // FP8 cache: expand the range's pages up to two ahead of this one
          if (kF8 && !expand_upto(g + 2, li)) { ok = false; break; }
        }
      }
    } else {
      // -------------------------------------------------------- B: softmax + epilogue
      // Two groups of four warps (one per TMEM lane quadrant) take alternate
      // pages: group grp handles the pages g with g % 2 == grp, one thread per
      // head row and all 32 of this CTA's tokens of the page, so one group's
      // exchanges with the peer overlap the other group's arithmetic. Through
      // shared memory the groups pass the reference maximum of each head
      // (decided page by page, in page order) and, at the end of a range, the
      // softmax sum of the group that does not write the output.
      const int grp = (warp - 3 - kAWarps) >> 2;
      const int gwarp = (warp - 3 - kAWarps) & 3;
      const int gtid = gwarp * 32 + lane;  // 0 .. 127
      const uint32_t vec_off = (uint32_t)row * 4;
      float x[32];
      float l_g = 0.f, m_l = -INFINITY;  // this group's sum over the range so far, on reference m_l
      int g = 0, lg_n = 0, iv_n = 0;
      bool ok = true;
      // The group that does not handle a range's last page drains columns
      // [128, 256) of O at the range switch, once the other group has posted 1/l.
      // O columns [128 half, 128 half + 128) of this CTA's half, scaled by inv,
      // as fp16 into the head-minor partials o_part[item][j][column / 8][head][column % 8]
      // (each warp store is 512 contiguous bytes).
      auto drain_o = [&](int it, int half, float inv) {
        uint4* dst = reinterpret_cast<uint4*>(plan.o_part) +
                     ((size_t)(it * n_q + j) * (kDC / 8) + (256 * rank + 128 * half) / 8) * H + row;
        float amax = 0.f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tO + 128 * half + 32 * c, r);
          tmem_wait_ld();
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              f[e] = __uint_as_float(r[8 * v + e]) * inv;
              // the FP8 cache's column scale (u = s * sum p code)
              if (kF8) f[e] *= __ldg(fp8_scales + 256 * rank + 128 * half + 32 * c + 8 * v + e);
              amax = fmaxf(amax, fabsf(f[e]));
            }
            if (row < H)
              dst[(size_t)(4 * c + v) * H] = make_uint4(cvt_f16x2(f[0], f[1]), cvt_f16x2(f[2], f[3]),
                                                       cvt_f16x2(f[4], f[5]), cvt_f16x2(f[6], f[7]));
          }
        }
        // a partial beyond the fp16 range would turn into infinity
        if (row < H && !(amax <= 65504.f)) report_error(err_word, MLA_ERR_RANGE);
      };
      for (int it = it0; it < it1 && ok; ++it) {
        const int li = it - it0;
        const int b = plan.item_seq[it], pg0 = plan.item_tile0[it], pg1 = plan.item_tile1[it];
        const int L = plan.seq_len_eff[b];
        const int n_att = L - n_q + j + 1;
        const int ntiles = pg1 - pg0;
        bool fresh = true;  // no page of this range handled by this group yet
        for (int i = 0; i < ntiles && ok; ++i, ++g) {
          if ((g & 1) != grp) {
            if (i == ntiles - 1) {
              // helper at the end of the range handled by the other group
              if (!wait_phase(bar(IVF0 + grp), iv_n & 1, abort_flag, err_word)) { ok = false; break; }
              ++iv_n;
              float inv;
              asm volatile("ld.shared.f32 %0, [%1];" : "=f"(inv) : "r"(sbase + kOffIV + vec_off));
              if (!wait_phase(bar(PVD0 + g % kPBufs), (g / kPBufs) & 1, abort_flag, err_word)) { ok = false; break; }
              tc_fence_after();
              drain_o(it, 1, inv);
              tc_fence_before();
              mbar_arrive(bar(OFREE));
            }
            continue;
          }
          const int xb = g & 1;
          // this CTA's partial scores of its 32 tokens
          const int nv = n_att - ((pg0 + i) * kTile + 32 * (int)rank);  // valid tokens among these 32
          if (!wait_phase(bar(SF0 + xb), (g >> 1) & 1, abort_flag, err_word)) { ok = false; break; }
          tc_fence_after();
          {
            uint32_t r[32];
            tmem_ld32(tS + 32 * rank, r);
            tmem_wait_ld();
#pragma unroll
            for (int v = 0; v < 32; ++v) x[v] = __uint_as_float(r[v]);  // scaled below
          }
          tc_fence_before();
          mbar_arrive(bar(SFREE));
          // add the peer's partial for these tokens: its midpoint plus the fp16 offsets
          if (!wait_phase(bar(XF0 + xb), (g >> 1) & 1, abort_flag, err_word)) { ok = false; break; }
          if (gtid == 0) mbar_arrive_expect_tx(bar(XF0 + xb), kXBytes);  // arm for page g+2
          float mid_p;
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(mid_p) : "r"(sbase + kOffX + xb * kXBytes + kXDataBytes + vec_off));
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            uint4 w;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                         : "r"(sbase + kOffX + xb * kXBytes + (uint32_t)((q8 * 128 + row) * 16)));
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 f = f16x2_to_f32(ww[k]);
              x[8 * q8 + 2 * k] = fmaf(x[8 * q8 + 2 * k], sl2, mid_p) + f.x;
              x[8 * q8 + 2 * k + 1] = fmaf(x[8 * q8 + 2 * k + 1], sl2, mid_p) + f.y;
            }
          }
          __syncwarp();
          // tell the peer this warp has read its partial (a 4-byte token completes
          // the peer's barrier; the loads above have all returned by now)
          if (lane == 0) st_async_b32(r_tok + (uint32_t)gwarp * 4, 1u, r_xe + 8u * xb);
          if (nv < 32) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              if (jj >= nv) x[jj] = -INFINITY;
          }
          // both CTAs' value MMAs of page g-3 are done: P buffer g % 3 is free. (Its
          // previous phase, page g-6, is complete: the value MMAs complete in page
          // order and this group waited for page g-5 at page g-2.)
          const int pb = g % kPBufs;
          if (g >= kPBufs && !wait_phase(bar(PVD0 + pb), ((g / kPBufs) & 1) ^ 1, abort_flag, err_word)) { ok = false; break; }
          const int rows_valid = L - (pg0 + i) * kTile;
          if (rows_valid < kTile) {
            // slack rows past the context may hold any bits: zero this CTA's latent
            // half so 0-weight x NaN cannot reach O. The score MMAs have read the
            // stage (SF); the value MMAs read it after this group's P-ready arrive.
            const int stage = (g + kQSlots * (li + 1)) % kStages;  // ring slot of page g
            const uint32_t sa = sbase + kOffStage + stage * kStageBytes;
            (void)MLA_SMEM_OK(sa, 4 * kCBoxBytes);
            const int nz = (kTile - rows_valid) * 4 * 8;  // 16-byte chunks
            for (int z = gtid; z < nz; z += kGThreads) {
              const int rr = rows_valid + z / 32, cb = (z / 8) & 3, ch = z & 7;
              asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(sa + cb * kCBoxBytes + rr * 128 + ch * 16),
                           "r"(0u)
                           : "memory");
            }
            fence_proxy_async_smem();
          }
          float m = x[0];
#pragma unroll
          for (int jj = 1; jj < 32; ++jj) m = fmaxf(m, x[jj]);
          st_async_b32(r_mx + xb * kVecBytes + vec_off, __float_as_uint(m), r_mxf + 8u * xb);
          if (!wait_phase(bar(MXF0 + xb), (g >> 1) & 1, abort_flag, err_word)) { ok = false; break; }
          if (gtid == 0) mbar_arrive_expect_tx(bar(MXF0 + xb), kVecBytes);
          float m_p;
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(m_p) : "r"(sbase + kOffMX + xb * kVecBytes + vec_off));
          const float mt = fmaxf(m, m_p);
          // the reference maximum: the previous page's decision (the other group's)
          // is raised lazily, only when this page exceeds it by the threshold
          if (g >= 1 && !wait_phase(bar(MRF), (g - 1) & 1, abort_flag, err_word)) { ok = false; break; }
          float m_new = mt, alpha = 1.f;
          bool need = false;
          if (i > 0) {
            float m_prev;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(m_prev) : "r"(sbase + kOffMR + vec_off));
            m_new = m_prev;
            if (mt > m_prev + kRescaleThreshold) {
              alpha = ex2(m_prev - mt);
              m_new = mt;
              need = true;
            }
          }
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(sbase + kOffMR + vec_off), "f"(m_new) : "memory");
          mbar_arrive(bar(MRF));
          if (__any_sync(0xffffffffu, need)) {
#if MLA_DEBUG_CHECKS
            if (lane == 0) atomicAdd(&g_dbg_counters[0], 1ull);
#endif
            // O must hold every earlier page before it is rescaled
            if (!wait_phase(bar(PVD0 + (g - 1) % kPBufs), ((g - 1) / kPBufs) & 1, abort_flag, err_word)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              uint32_t r[32];
              tmem_ld32(tO + 32 * c, r);
              tmem_wait_ld();
#pragma unroll
              for (int v = 0; v < 32; ++v) r[v] = __float_as_uint(__uint_as_float(r[v]) * alpha);
              tmem_st32(tO + 32 * c, r);
            }
          }
          // this group's running sum, on the new reference
          if (fresh) {
            l_g = 0.f;
            m_l = m_new;
            fresh = false;
          } else if (m_l != m_new) {
            if (l_g != 0.f) l_g *= ex2(m_l - m_new);
            m_l = m_new;
          }
          const float mref = m_new == -INFINITY ? 0.f : m_new;  // all masked so far: every p is 0
          // P: into tensor memory for this CTA's value MMAs and into the peer's
          // shared memory (64B-swizzled, K-major) for its own
          const uint32_t pr = r_p + pb * kPPeerBytes + (uint32_t)row * 64;
          const uint32_t pfr = r_pf + 8u * pb;
          (void)MLA_SMEM_OK(sbase + kOffP + pb * kPPeerBytes + (uint32_t)row * 64, 64);
          (void)MLA_TMEM_OK(kTmP + 16 * pb, 16);
          float lsum0 = 0.f, lsum1 = 0.f;
          uint32_t pw[16];
#pragma unroll
          for (int v = 0; v < 16; ++v) {
            const float p0 = ex2(x[2 * v] - mref);
            const float p1 = ex2(x[2 * v + 1] - mref);
            if (kF8) {  // fp16 operands with the FP8 cache
              pw[v] = cvt_f16x2(p0, p1);
              const float2 f = f16x2_to_f32(pw[v]);
              lsum0 += f.x;
              lsum1 += f.y;
            } else {
              pw[v] = cvt_bf16x2(p0, p1);
              lsum0 += bf16_lo(pw[v]);
              lsum1 += bf16_hi(pw[v]);
            }
          }
          tmem_st16(tmem + lane_off + kTmP + 16 * pb, pw);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            st_async_v4(pr + (uint32_t)((c ^ ((row >> 1) & 3)) * 16),
                        make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]), pfr);
          tmem_wait_st();
          l_g += lsum0 + lsum1;
          tc_fence_before();
          mbar_arrive(bar(PF0 + pb));
          if (i == ntiles - 2) {
            // the other group handles the last page of the range: hand over this sum
            const uint32_t lg = sbase + kOffLG + (uint32_t)(lg_n & 1) * 2 * kVecBytes;
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(lg + vec_off), "f"(l_g) : "memory");
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(lg + kVecBytes + vec_off), "f"(m_l) : "memory");
            mbar_arrive(bar(LGF0 + (lg_n & 1)));
          }
          if (i == ntiles - 1) {
            // epilogue: the CTA's sum (both groups), the peer's, the normalised output
            float l_c = l_g;
            if (ntiles >= 2) {
              if (!wait_phase(bar(LGF0 + (lg_n & 1)), (lg_n >> 1) & 1, abort_flag, err_word)) { ok = false; break; }
              const uint32_t lg = sbase + kOffLG + (uint32_t)(lg_n & 1) * 2 * kVecBytes;
              float l_o, m_o;
              asm volatile("ld.shared.f32 %0, [%1];" : "=f"(l_o) : "r"(lg + vec_off));
              asm volatile("ld.shared.f32 %0, [%1];" : "=f"(m_o) : "r"(lg + kVecBytes + vec_off));
              if (l_o != 0.f) l_c += l_o * ex2(m_o - m_new);
            }
            const int lb = li & 1;
            st_async_b32(r_lx + lb * kVecBytes + vec_off, __float_as_uint(l_c), r_lxf + 8u * lb);
            if (!wait_phase(bar(LXF0 + lb), (li >> 1) & 1, abort_flag, err_word)) { ok = false; break; }
            if (gtid == 0) mbar_arrive_expect_tx(bar(LXF0 + lb), kVecBytes);  // arm for range li+2
            float l_p;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(l_p) : "r"(sbase + kOffLX + lb * kVecBytes + vec_off));
            // the same addition in the same order in both CTAs: rank 0's sum first
            const float l_tot = rank == 0 ? l_c + l_p : l_p + l_c;
            const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
            // 1/l for the helper group, which drains the other half of O
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(sbase + kOffIV + vec_off), "f"(inv) : "memory");
            mbar_arrive(bar(IVF0 + (grp ^ 1)));
            if (!wait_phase(bar(PVD0 + pb), (g / kPBufs) & 1, abort_flag, err_word)) { ok = false; break; }
            tc_fence_after();
            const size_t orow = ((size_t)it * n_q + j) * H + row;
            drain_o(it, 0, inv);
            tc_fence_before();
            mbar_arrive(bar(OFREE));
            if (rank == 0 && row < H)
              plan.lse_part[orow] = l_tot > 0.f ? (m_new + log2f(l_tot)) * kLn2 : -INFINITY;
          }
        }
        if (ntiles >= 2) ++lg_n;
      }
    }
  }

  // ------------------------------------------------------------ teardown
  if (warp == 1 && lane == 0) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar(MMAD), 0) && clock64() - t0 < kWaitLimitCycles) {
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer has finished writing into this CTA's shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmCols);
  }
}

}  // namespace

// ---------------------------------------------------------------- host side
int decode_max_workers() {
  if (smem_limit<decode_tc_kernel<false>>(kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return n;
}

namespace {
// The query maps and the launch, shared by the bf16 and FP8 caches (the page
// maps differ: 16-bit swizzled boxes, or unswizzled 8-bit rows).
template <bool kF8>
cudaError_t launch_decode_impl(const CUtensorMap& map_c, const CUtensorMap& map_kr, const uint16_t* q_abs,
                               const float* fp8_scales, const int32_t* block_table, int B, int n_q, int H,
                               int num_pages, int page_size, int max_pages, float scale, int G, const Plan& plan,
                               int32_t* err_word,
                               cudaStream_t s) {
  CUtensorMap map_qkr, map_q;
  const uint64_t q_dims[2] = {kRow, (uint64_t)B * n_q * H};
  const uint64_t row_stride[1] = {kRow * 2};
  const uint32_t box_qkr[2] = {32, 64}, box_q[2] = {64, 128};
  if (!make_tmap(&map_qkr, q_abs, 2, q_dims, row_stride, box_qkr, 64) ||
      !make_tmap(&map_q, q_abs, 2, q_dims, row_stride, box_q, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = smem_limit<decode_tc_kernel<kF8>>(kSmemBytes);
  if (e != cudaSuccess) return e;
  const float sl2 = scale * 1.4426950408889634f;
  dim3 grid(2 * G, n_q, 1);
  return launch_pdl(decode_tc_kernel<kF8>, grid, dim3(kThreads), kSmemBytes, s, map_c, map_kr, map_qkr, map_q,
                    block_table, n_q, H, max_pages, num_pages, page_size == 2 * kTile ? 1 : 0, sl2, plan,
                    fp8_scales, err_word);
}
}  // namespace

cudaError_t launch_decode(const uint16_t* q_abs, const uint16_t* cache, const int32_t* block_table,
                          int B, int n_q, int H, int num_pages, int page_size, int max_pages, float scale, int G,
                          const Plan& plan, int32_t* err_word, cudaStream_t s) {
  CUtensorMap map_c, map_kr;
  const uint64_t cache_dims[2] = {kRow, (uint64_t)num_pages * page_size};
  const uint64_t row_stride[1] = {kRow * 2};
  const uint32_t box_c[2] = {64, 64}, box_kr[2] = {32, 64};
  if (!make_tmap(&map_c, cache, 2, cache_dims, row_stride, box_c, 128) ||
      !make_tmap(&map_kr, cache, 2, cache_dims, row_stride, box_kr, 64))
    return cudaErrorInvalidValue;
  return launch_decode_impl<false>(map_c, map_kr, q_abs, nullptr, block_table, B, n_q, H, num_pages, page_size,
                                   max_pages, scale, G, plan, err_word, s);
}

cudaError_t launch_decode_fp8(const uint16_t* q_abs, const uint8_t* cache8, const float* fp8_scales,
                              const int32_t* block_table, int B, int n_q, int H, int num_pages, int page_size,
                              int max_pages, float scale, int G, const Plan& plan, int32_t* err_word,
                              cudaStream_t s) {
  CUtensorMap map_c, map_kr;
  const uint64_t cache_dims[2] = {kRow, (uint64_t)num_pages * page_size};
  const uint64_t row_stride[1] = {kRow};
  const uint32_t box_c[2] = {64, 64}, box_kr[2] = {32, 16};
  if (!make_tmap(&map_c, cache8, 2, cache_dims, row_stride, box_c, 0, true) ||
      !make_tmap(&map_kr, cache8, 2, cache_dims, row_stride, box_kr, 0, true))
    return cudaErrorInvalidValue;
  return launch_decode_impl<true>(map_c, map_kr, q_abs, fp8_scales, block_table, B, n_q, H, num_pages, page_size,
                                  max_pages, scale, G, plan, err_word, s);
}

}  // namespace mla

#if MLA_DEBUG_CHECKS
// Test-build entry points (declared in include/mla_debug.h). Synchronous
// copies to or from the decode kernel's instrumentation variables on the
// current device; each returns a cudaError_t value (0 = success).
extern "C" {
int mla_debug_read_counters(unsigned long long* out, int n) {
  if (!out || n < 1 || n > 4) return (int)cudaErrorInvalidValue;
  return (int)cudaMemcpyFromSymbol(out, mla::g_dbg_counters, sizeof(unsigned long long) * (size_t)n);
}
int mla_debug_reset(void) {
  const unsigned long long zero[4] = {0, 0, 0, 0};
  const int off = 0;
  const long long nolimit = 0;
  cudaError_t e = cudaMemcpyToSymbol(mla::g_dbg_counters, zero, sizeof(zero));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(mla::g_dbg_skip_producer, &off, sizeof(off));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(mla::sm100::g_wait_limit_override, &nolimit, sizeof(nolimit));
  return (int)e;
}
int mla_debug_set_wait_limit(long long cycles) {
  return (int)cudaMemcpyToSymbol(mla::sm100::g_wait_limit_override, &cycles, sizeof(cycles));
}
int mla_debug_set_skip_producer(int on) {
  return (int)cudaMemcpyToSymbol(mla::g_dbg_skip_producer, &on, sizeof(on));
}
}  // extern "C"
#endif
