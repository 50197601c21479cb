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
// each 64-token page (36 KB), so every cached byte is read from HBM once. The
// 128 heads share every page tile in shared memory (the reuse the absorbed
// formulation creates).
//
// Scores need all 576 columns: each CTA computes a partial score
// S_r[128 heads][64 tokens] (K = 288) with tcgen05 MMAs into tensor memory.
// The softmax of a page is split by tokens: CTA r finishes tokens
// [32r, 32r+32). It sends the partial scores of the other 32 tokens to the
// peer (fp32, 16 KB, st.async into the peer's shared memory), adds the
// peer's partial for its own tokens, and both CTAs exchange their page
// maxima so they share one exact running maximum per head. Each CTA then
// exponentiates its 32 tokens, writes its half of P[128][64] (bf16) into its
// own and the peer's shared memory, and accumulates its 256-column half of
// O[128][512] in tensor memory with the second MMA (P x C[64][256]).
//
// Tensor memory (512 columns x 128 lanes of 32 bits): O [0,256), S double
// buffer [256,384), the CTA's latent half of q_abs as the MMA A operand
// [384,512). Shared memory: 4-stage page ring (147 KB), the positional half of
// q_abs (2 x 8 KB), peer partial scores (2 x 16 KB), P (2 x 16 KB).
//
// Warps: 0 = TMA producer, 1 = MMA issuer (and TMEM owner), 2..5 = softmax
// and epilogue, one thread per head row (TMEM lane). The score MMAs run two
// pages ahead of the value MMAs; the softmax of page g-1 is interleaved with
// the reads of page g so every exchange's latency is covered by other work.
#include "mla_internal.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr uint32_t kCBoxBytes = 64 * 128;   // [64 tokens][64 latent cols] bf16, 128B swizzle
constexpr uint32_t kKrBoxBytes = 64 * 64;   // [64 tokens][32 positional cols] bf16, 64B swizzle
constexpr uint32_t kStageBytes = 4 * kCBoxBytes + kKrBoxBytes;  // 36864
constexpr uint32_t kQkrBytes = 128 * 64;    // [128 heads][32] bf16, 64B swizzle
constexpr uint32_t kXBytes = 8 * 128 * 16;  // peer partial scores: [8 groups of 4 tokens][128 heads] fp32
constexpr uint32_t kPBytes = 128 * 128;     // P [128 heads][64 tokens] bf16, 128B swizzle, K-major
constexpr uint32_t kPHalfBytes = kPBytes / 2;
constexpr uint32_t kVecBytes = 128 * 4;     // one float per head

constexpr uint32_t kOffStage = 0;
constexpr uint32_t kOffQkr = kOffStage + kStages * kStageBytes;
constexpr uint32_t kOffX = kOffQkr + 2 * kQkrBytes;
constexpr uint32_t kOffP = kOffX + 2 * kXBytes;
constexpr uint32_t kOffMX = kOffP + 2 * kPBytes;   // peer page maxima [2][128]
constexpr uint32_t kOffLX = kOffMX + 2 * kVecBytes;  // peer softmax sums [2][128]
constexpr uint32_t kOffTok = kOffLX + 2 * kVecBytes;  // "partial consumed" tokens from the peer [2][4]
constexpr uint32_t kOffBar = kOffTok + 2 * 4 * 4;

// barrier indices
enum {
  FULL0 = 0, EMPTY0 = FULL0 + kStages, QKRF0 = EMPTY0 + kStages, QKRE0 = QKRF0 + 2, QCF = QKRE0 + 2,
  SF0 = QCF + 1, SFREE0 = SF0 + 2, PF0 = SFREE0 + 2, PVD0 = PF0 + 2, XF0 = PVD0 + 2, XE0 = XF0 + 2,
  MXF0 = XE0 + 2, LXF0 = MXF0 + 2, OFREE = LXF0 + 2, MMAD = OFREE + 1, kNumBars = MMAD + 1
};
constexpr uint32_t kOffSlots = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffSlots + 16;  // the base is checked to be 1024-byte aligned
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmO = 0, kTmS = 256, kTmQ = 384, kTmCols = 512;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P values stay <= 256

struct TileInfo {
  int g;       // CTA-local page counter
  int item;    // partial index
  int li;      // range counter within this worker
  int first, last;
  int tok0;    // first token of the page
  int n_att;   // tokens this query attends
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap map_c, const __grid_constant__ CUtensorMap map_kr,
                 const __grid_constant__ CUtensorMap map_qkr, const uint16_t* __restrict__ q_abs,
                 const int32_t* __restrict__ block_table, int n_q, int H, int max_pages, float sl2,
                 Plan plan, int32_t* err_word) {
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
      mbar_init(bar(QKRF0 + i), 1);
      mbar_init(bar(QKRE0 + i), 1);
      mbar_init(bar(SF0 + i), 1);
      mbar_init(bar(SFREE0 + i), 128);
      mbar_init(bar(PF0 + i), 129);  // 128 local halves + the arming arrive for the peer's half
      mbar_init(bar(PVD0 + i), 2);   // the value MMAs of this page done in both CTAs
      mbar_init(bar(XF0 + i), 1);    // armed here, filled by the peer's st.async
      mbar_init(bar(XE0 + i), 1);    // armed here, completed by the peer's four 4-byte tokens
      mbar_init(bar(MXF0 + i), 1);
      mbar_init(bar(LXF0 + i), 1);
    }
    mbar_init(bar(QCF), 128);
    mbar_init(bar(OFREE), 128);
    mbar_init(bar(MMAD), 1);
    *abort_flag = 0;
    fence_mbar_init();
    for (int i = 0; i < 2; ++i) {
      mbar_arrive_expect_tx(bar(XF0 + i), kXBytes);
      mbar_arrive_expect_tx(bar(PF0 + i), kPHalfBytes);
      mbar_arrive_expect_tx(bar(MXF0 + i), kVecBytes);
      mbar_arrive_expect_tx(bar(LXF0 + i), kVecBytes);
      mbar_arrive_expect_tx(bar(XE0 + i), 16);
    }
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map_c);
    prefetch_tmap(&map_kr);
    prefetch_tmap(&map_qkr);
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
  const int it0 = plan.range_item[worker], it1 = plan.range_item[worker + 1];

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    int stage = 0;
    uint32_t ph = 0;
    int last_ph[kStages], last_qph[2] = {-1, -1};
#pragma unroll
    for (int i = 0; i < kStages; ++i) last_ph[i] = -1;
    bool ok = true;
    for (int it = it0; it < it1 && ok; ++it) {
      const int li = it - it0, qb = li & 1;
      const int b = plan.item_seq[it], pg0 = plan.item_page0[it], pg1 = plan.item_page1[it];
      if (!wait_phase(bar(QKRE0 + qb), ((li >> 1) & 1) ^ 1, abort_flag, err_word)) { ok = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(QKRF0 + qb), kQkrBytes);
        tma_load_2d(sbase + kOffQkr + qb * kQkrBytes, &map_qkr, bar(QKRF0 + qb), kDC + 32 * (int)rank,
                    (b * n_q + j) * H, pol_keep);
      }
      last_qph[qb] = (li >> 1) & 1;
      for (int pg = pg0; pg < pg1 && ok; pg += 32) {
        const int mine = pg + lane;
        const int id_l = mine < pg1 ? block_table[(size_t)b * max_pages + mine] : 0;
        const int n = min(32, pg1 - pg);
        for (int t = 0; t < n; ++t) {
          const int pid = __shfl_sync(0xffffffffu, id_l, t);
          if (!wait_phase(bar(EMPTY0 + stage), ph ^ 1u, abort_flag, err_word)) { ok = false; break; }
          if (lane == 0) {
            const uint32_t fb = bar(FULL0 + stage);
            const uint32_t dst = sbase + kOffStage + stage * kStageBytes;
            mbar_arrive_expect_tx(fb, kStageBytes);
            const int y = pid * kPage;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb)
              tma_load_2d(dst + cb * kCBoxBytes, &map_c, fb, 256 * (int)rank + 64 * cb, y, pol_stream);
            tma_load_2d(dst + 4 * kCBoxBytes, &map_kr, fb, kDC + 32 * (int)rank, y, pol_stream);
          }
          last_ph[stage] = (int)ph;
          __syncwarp();
          if (++stage == kStages) { stage = 0; ph ^= 1u; }
        }
      }
    }
    if (!ok) {
      // let every issued copy land before this CTA can exit
#pragma unroll
      for (int i = 0; i < kStages + 2; ++i) {
        const int ph_i = i < kStages ? last_ph[i] : last_qph[i - kStages];
        const uint32_t b_i = i < kStages ? bar(FULL0 + i) : bar(QKRF0 + i - kStages);
        if (ph_i >= 0) {
          const long long t0 = clock64();
          while (!mbar_try_wait(b_i, (uint32_t)ph_i) && clock64() - t0 < kWaitLimitCycles) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Order: QK(g) then PV(g-2). Scores run two pages ahead of the value
    // MMAs, so the tensor pipe has work while the softmax of page g-2 runs.
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16(128, 64, false, false);
      constexpr uint32_t kIdPV = idesc_bf16(128, 256, false, true);
      // descriptor templates; the start address is added per use
      const uint64_t dQK_c = smem_desc(0, 16, 1024, kSwizzle128B);
      const uint64_t dQK_r = smem_desc(0, 16, 512, kSwizzle64B);
      const uint64_t dPV_a = smem_desc(0, 16, 1024, kSwizzle128B);
      const uint64_t dPV_b = smem_desc(0, kCBoxBytes, 1024, kSwizzle128B);
      // start-address field: 14 bits of (shared address >> 4). Shared
      // addresses of the second CTA of a cluster carry high bits that must
      // not spill into the neighbouring descriptor fields.
      auto da = [](uint32_t addr) -> uint64_t { return (uint64_t)((addr >> 4) & 0x3FFFu); };
      int stage = 0;
      uint32_t ph = 0;
      int g = 0;
      bool ok = true;
      // pending value MMAs: (page, stage, first-of-range, range counter)
      int pq_t[3], pq_s[3], pq_f[3], pq_l[3];
      int pq_head = 0, pq_n = 0;

      auto issue_pv = [&](int t, int st, int first, int li) -> bool {
        const int pb = t & 1;
        if (!wait_phase(bar(PF0 + pb), (t >> 1) & 1, abort_flag, err_word)) return false;
        if (first && li > 0 && !wait_phase(bar(OFREE), (li - 1) & 1, abort_flag, err_word)) return false;
        // arm the P buffer for page t+2; its peer half can only come after this
        // page's value MMAs (waited through PVD by the peer)
        mbar_arrive_expect_tx(bar(PF0 + pb), kPHalfBytes);
        fence_proxy_async_smem();  // P written by generic stores, read by the tensor core
        tc_fence_after();
        const uint64_t ad = dPV_a + da(sbase + kOffP + pb * kPBytes);
        const uint64_t bd = dPV_b + da(sbase + kOffStage + st * kStageBytes);
        mma_ss(tmem + kTmO, ad, bd, kIdPV, first ? 0u : 1u);
#pragma unroll
        for (int ks = 1; ks < 4; ++ks) mma_ss(tmem + kTmO, ad + (ks * 32 >> 4), bd + (ks * 2048 >> 4), kIdPV, 1u);
        mma_commit_multicast(bar(PVD0 + pb), 0x3);
        mma_commit(bar(EMPTY0 + st));
        return true;
      };

      for (int it = it0; it < it1 && ok; ++it) {
        const int li = it - it0, qb = li & 1;
        const int ntiles = plan.item_page1[it] - plan.item_page0[it];
        for (int i = 0; i < ntiles; ++i, ++g) {
          if (i == 0) {
            if (!wait_phase(bar(QCF), li & 1, abort_flag, err_word) ||
                !wait_phase(bar(QKRF0 + qb), (li >> 1) & 1, abort_flag, err_word)) { ok = false; break; }
          }
          const int sb = g & 1;
          if (!wait_phase(bar(FULL0 + stage), ph, abort_flag, err_word) ||
              !wait_phase(bar(SFREE0 + sb), ((g >> 1) & 1) ^ 1, abort_flag, err_word)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bc = dQK_c + da(sbase + kOffStage + stage * kStageBytes);
          const uint32_t d = tmem + kTmS + 64 * sb;
          mma_ts(d, tmem + kTmQ, bc, kIdQK, 0u);
#pragma unroll
          for (int ks = 1; ks < 16; ++ks)
            mma_ts(d, tmem + kTmQ + ks * 8, bc + (((ks >> 2) * kCBoxBytes + (ks & 3) * 32) >> 4), kIdQK, 1u);
          const uint64_t ar = dQK_r + da(sbase + kOffQkr + qb * kQkrBytes);
          const uint64_t br = dQK_r + da(sbase + kOffStage + stage * kStageBytes + 4 * kCBoxBytes);
          mma_ss(d, ar, br, kIdQK, 1u);
          mma_ss(d, ar + 2, br + 2, kIdQK, 1u);
          mma_commit(bar(SF0 + sb));
          if (i == ntiles - 1) mma_commit(bar(QKRE0 + qb));
          const int slot = (pq_head + pq_n) % 3;
          pq_t[slot] = g; pq_s[slot] = stage; pq_f[slot] = (i == 0); pq_l[slot] = li;
          ++pq_n;
          if (pq_n == 3) {
            if (!issue_pv(pq_t[pq_head], pq_s[pq_head], pq_f[pq_head], pq_l[pq_head])) { ok = false; break; }
            pq_head = (pq_head + 1) % 3;
            --pq_n;
          }
          if (++stage == kStages) { stage = 0; ph ^= 1u; }
        }
      }
      while (ok && pq_n > 0) {
        ok = issue_pv(pq_t[pq_head], pq_s[pq_head], pq_f[pq_head], pq_l[pq_head]);
        pq_head = (pq_head + 1) % 3;
        --pq_n;
      }
      mma_commit(bar(MMAD));
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // head row == TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + kTmS, tO = tmem + lane_off + kTmO, tQ = tmem + lane_off + kTmQ;
    const int tid128 = threadIdx.x - 64;
    // remote (peer) addresses: its buffers and barriers at the same offsets
    const uint32_t r_x = mapa(sbase + kOffX, peer), r_p = mapa(sbase + kOffP, peer);
    const uint32_t r_mx = mapa(sbase + kOffMX, peer), r_lx = mapa(sbase + kOffLX, peer);
    const uint32_t r_xf = mapa(bar(XF0), peer), r_xe = mapa(bar(XE0), peer), r_pf = mapa(bar(PF0), peer);
    const uint32_t r_tok = mapa(sbase + kOffTok, peer);
    const uint32_t r_mxf = mapa(bar(MXF0), peer), r_lxf = mapa(bar(LXF0), peer);
    // P chunk (8 tokens = 16 bytes) c of this row, 128B swizzle
    const uint32_t prow_off = (uint32_t)row * 128;
    auto pchunk = [&](int c) -> uint32_t { return prow_off + (uint32_t)((c ^ (row & 7)) * 16); };

    auto load_qc = [&](int it) {
      const int b = plan.item_seq[it];
      const size_t qrow = ((size_t)b * n_q + j) * H + row;
      const uint4* src = reinterpret_cast<const uint4*>(q_abs + qrow * kRow + 256 * rank);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint4 w = row < H ? __ldg(src + c * 8 + v) : make_uint4(0, 0, 0, 0);
          r[4 * v] = w.x; r[4 * v + 1] = w.y; r[4 * v + 2] = w.z; r[4 * v + 3] = w.w;
        }
        tmem_st32(tQ + 32 * c, r);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(QCF));
    };

    float s_keep[32];  // this CTA's partial scores of its own 32 tokens, page g
    float x[32];       // full scores (log2 units) of its own tokens, page g-1
    float mt_mine = -INFINITY;
    TileInfo pv{};
    bool have_prev = false, ok = true;
    float m_ref = -INFINITY, l_mine = 0.f;

    // B1(t): add the peer's partial for this CTA's tokens, mask, page maximum,
    // and send that maximum to the peer.
    auto stage_b1 = [&](const TileInfo& t) -> bool {
      const int xb = t.g & 1;
      if (!wait_phase(bar(XF0 + xb), (t.g >> 1) & 1, abort_flag, err_word)) return false;
      if (tid128 == 0) mbar_arrive_expect_tx(bar(XF0 + xb), kXBytes);  // arm for page t+2
      const uint32_t xa = sbase + kOffX + xb * kXBytes + (uint32_t)row * 16;
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        float4 w;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(w.x), "=f"(w.y), "=f"(w.z), "=f"(w.w) : "r"(xa + q8 * 128 * 16));
        x[4 * q8 + 0] = (x[4 * q8 + 0] + w.x) * sl2;
        x[4 * q8 + 1] = (x[4 * q8 + 1] + w.y) * sl2;
        x[4 * q8 + 2] = (x[4 * q8 + 2] + w.z) * sl2;
        x[4 * q8 + 3] = (x[4 * q8 + 3] + w.w) * sl2;
      }
      __syncwarp();
      // tell the peer this warp has read its partial (a 4-byte token completes
      // the peer's barrier; the loads above have all returned by now)
      if (lane == 0) st_async_b32(r_tok + (uint32_t)(xb * 4 + quad) * 4, 1u, r_xe + 8u * xb);
      const int nv = t.n_att - (t.tok0 + 32 * (int)rank);  // valid tokens among this CTA's 32
      if (nv < 32) {
#pragma unroll
        for (int jj = 0; jj < 32; ++jj)
          if (jj >= nv) x[jj] = -INFINITY;
      }
      float m = x[0];
#pragma unroll
      for (int jj = 1; jj < 32; ++jj) m = fmaxf(m, x[jj]);
      mt_mine = m;
      st_async_b32(r_mx + xb * kVecBytes + (uint32_t)row * 4, __float_as_uint(m), r_mxf + 8u * xb);
      return true;
    };

    // B2(t): common page maximum, online-softmax update, this CTA's half of P
    // (to both CTAs), and for the last page of a range the normalised output.
    auto stage_b2 = [&](const TileInfo& t) -> bool {
      const int xb = t.g & 1;
      if (!wait_phase(bar(MXF0 + xb), (t.g >> 1) & 1, abort_flag, err_word)) return false;
      if (tid128 == 0) mbar_arrive_expect_tx(bar(MXF0 + xb), kVecBytes);  // arm for page t+2
      float m_peer;
      asm volatile("ld.shared.f32 %0, [%1];" : "=f"(m_peer) : "r"(sbase + kOffMX + xb * kVecBytes + (uint32_t)row * 4));
      const float mt = fmaxf(mt_mine, m_peer);  // identical in both CTAs
      bool need = false;
      float alpha = 1.f;
      if (t.first) {
        m_ref = mt;
        l_mine = 0.f;
      } else if (mt > m_ref + kRescaleThreshold) {
        alpha = ex2(m_ref - mt);
        l_mine *= alpha;
        m_ref = mt;
        need = true;
      }
      if (__any_sync(0xffffffffu, need)) {
        // O must hold every earlier page before it is rescaled
        if (!wait_phase(bar(PVD0 + ((t.g - 1) & 1)), ((t.g - 1) >> 1) & 1, abort_flag, err_word)) return false;
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
        tmem_wait_st();
      }
      // both CTAs' value MMAs of page t-2 have consumed this P buffer
      if (t.g >= 2 && !wait_phase(bar(PVD0 + xb), ((t.g >> 1) & 1) ^ 1, abort_flag, err_word)) return false;
      const float mref = m_ref == -INFINITY ? 0.f : m_ref;  // all-masked so far: every p is 0
      const uint32_t pl = sbase + kOffP + xb * kPBytes, pr = r_p + xb * kPBytes;
      const uint32_t pfr = r_pf + 8u * xb;
      float lsum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 w;
        uint32_t* pw = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float p0 = ex2(x[8 * c + 2 * v] - mref);
          const float p1 = ex2(x[8 * c + 2 * v + 1] - mref);
          pw[v] = cvt_bf16x2(p0, p1);
          lsum += bf16_lo(pw[v]) + bf16_hi(pw[v]);
        }
        const uint32_t off = pchunk(4 * (int)rank + c);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(pl + off), "r"(w.x), "r"(w.y), "r"(w.z),
                     "r"(w.w)
                     : "memory");
        st_async_v4(pr + off, w, pfr);
      }
      l_mine += lsum;
      tc_fence_before();
      mbar_arrive(bar(PF0 + xb));
      if (t.last) {
        // softmax sum over both token halves, then the normalised output
        const int lb = t.li & 1;
        st_async_b32(r_lx + lb * kVecBytes + (uint32_t)row * 4, __float_as_uint(l_mine), r_lxf + 8u * lb);
        if (!wait_phase(bar(LXF0 + lb), (t.li >> 1) & 1, abort_flag, err_word)) return false;
        if (tid128 == 0) mbar_arrive_expect_tx(bar(LXF0 + lb), kVecBytes);  // arm for range li+2
        float l_peer;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(l_peer) : "r"(sbase + kOffLX + lb * kVecBytes + (uint32_t)row * 4));
        const float l_tot = rank == 0 ? l_mine + l_peer : l_peer + l_mine;
        if (!wait_phase(bar(PVD0 + xb), (t.g >> 1) & 1, abort_flag, err_word)) return false;
        tc_fence_after();
        const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
        const size_t orow = ((size_t)t.item * n_q + j) * H + row;
        float4* dst = reinterpret_cast<float4*>(plan.o_part + orow * kDC + 256 * rank);
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t r[32];
          tmem_ld32(tO + 32 * c, r);
          tmem_wait_ld();
          if (row < H) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[c * 8 + v] = make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                           __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(OFREE));
        if (rank == 0 && row < H)
          plan.lse_part[orow] = l_tot > 0.f ? (m_ref + log2f(l_tot)) * kLn2 : -INFINITY;
      }
      return true;
    };

    if (it0 < it1) load_qc(it0);
    int g = 0;
    int stage = 0;
    for (int it = it0; it < it1 && ok; ++it) {
      const int li = it - it0;
      const int b = plan.item_seq[it], pg0 = plan.item_page0[it], pg1 = plan.item_page1[it];
      const int L = plan.seq_len_eff[b];
      const int n_att = L - n_q + j + 1;
      const int ntiles = pg1 - pg0;
      for (int i = 0; i < ntiles; ++i, ++g) {
        const int sb = g & 1;
        // B1 of the previous page needs only the peer, not this page's scores
        if (have_prev) {
#pragma unroll
          for (int v = 0; v < 32; ++v) x[v] = s_keep[v];
          if (!stage_b1(pv)) { ok = false; break; }
        }
        // A: this CTA's partial scores of page g (its 288 columns)
        if (!wait_phase(bar(SF0 + sb), (g >> 1) & 1, abort_flag, err_word)) { ok = false; break; }
        tc_fence_after();
        {
          uint32_t r[32];
          // the other CTA's tokens first: send them
          tmem_ld32(tS + 64 * sb + 32 * peer, r);
          tmem_wait_ld();
          if (!wait_phase(bar(XE0 + sb), ((g >> 1) & 1) ^ 1, abort_flag, err_word)) { ok = false; break; }
          if (g >= 2 && tid128 == 0) mbar_arrive_expect_tx(bar(XE0 + sb), 16);  // arm for page g+2
          const uint32_t xa = r_x + sb * kXBytes + (uint32_t)row * 16;
          const uint32_t xf = r_xf + 8u * sb;
#pragma unroll
          for (int q8 = 0; q8 < 8; ++q8)
            st_async_v4(xa + q8 * 128 * 16, make_uint4(r[4 * q8], r[4 * q8 + 1], r[4 * q8 + 2], r[4 * q8 + 3]), xf);
          tmem_ld32(tS + 64 * sb + 32 * rank, r);
          tmem_wait_ld();
#pragma unroll
          for (int v = 0; v < 32; ++v) s_keep[v] = __uint_as_float(r[v]);
        }
        tc_fence_before();
        mbar_arrive(bar(SFREE0 + sb));
        const int tok0 = (pg0 + i) * kPage;
        const int rows_valid = L - tok0;
        if (rows_valid < kPage) {
          // slack rows past the context may hold any bits: zero this CTA's latent
          // half so 0-weight x NaN cannot reach O
          const uint32_t sa = sbase + kOffStage + stage * kStageBytes;
          const int nz = (kPage - rows_valid) * 4 * 8;  // 16-byte chunks
          for (int z = tid128; z < nz; z += 128) {
            const int rr = rows_valid + z / 32, cb = (z / 8) & 3, ch = z & 7;
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(sa + cb * kCBoxBytes + rr * 128 + ch * 16),
                         "r"(0u)
                         : "memory");
          }
          fence_proxy_async_smem();
        }
        // every score MMA of this range is done: stage the next range's query
        if (i == ntiles - 1 && it + 1 < it1) load_qc(it + 1);
        if (have_prev && !stage_b2(pv)) { ok = false; break; }
        pv = TileInfo{g, it, li, i == 0, i == ntiles - 1, tok0, n_att};
        have_prev = true;
        if (++stage == kStages) stage = 0;
      }
    }
    if (ok && have_prev) {
#pragma unroll
      for (int v = 0; v < 32; ++v) x[v] = s_keep[v];
      ok = stage_b1(pv) && stage_b2(pv);
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
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
      return -1;
    attr_set = true;
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
  if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return n;
}

cudaError_t launch_decode(const uint16_t* q_abs, const uint16_t* cache, const int32_t* block_table,
                          int B, int n_q, int H, int num_pages, int max_pages, float scale, int G,
                          const Plan& plan, int32_t* err_word, cudaStream_t s) {
  CUtensorMap map_c, map_kr, map_qkr;
  const uint64_t cache_dims[2] = {kRow, (uint64_t)num_pages * kPage};
  const uint64_t q_dims[2] = {kRow, (uint64_t)B * n_q * H};
  const uint64_t row_stride[1] = {kRow * 2};
  const uint32_t box_c[2] = {64, 64}, box_kr[2] = {32, 64}, box_qkr[2] = {32, 128};
  if (!make_tmap(&map_c, cache, 2, cache_dims, row_stride, box_c, 128) ||
      !make_tmap(&map_kr, cache, 2, cache_dims, row_stride, box_kr, 64) ||
      !make_tmap(&map_qkr, q_abs, 2, q_dims, row_stride, box_qkr, 64))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const float sl2 = scale * 1.4426950408889634f;
  dim3 grid(2 * G, n_q, 1);
  decode_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(map_c, map_kr, map_qkr, q_abs, block_table, n_q, H,
                                                      max_pages, sl2, plan, err_word);
  return cudaGetLastError();
}

}  // namespace mla
