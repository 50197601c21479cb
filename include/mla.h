/*
 * mla.h — C ABI of the GB300 (sm_103a) library for Multi-Head Latent
 * Attention (MLA) decode with weight absorption over a paged latent cache.
 *
 * What the four calls compute (notation of Huny's Dev Blog "Multi-Head
 * Latent Attention(MLA) 아키텍처 해부", sections 1-3):
 *   mla_absorb_q      qt = q^C (W^UK)^T per head, the absorbed query      (section 3.1)
 *   mla_decode_paged  z_s = (qt . c_s + q^R . k^R_s) / sqrt(d_nope + d_r)  (section 2.2, 3.1)
 *                     partial softmax over page ranges, partial u = a C^KV (section 3.2)
 *   mla_combine       log-sum-exp merge of the range partials -> u, lse
 *   mla_out_proj      out = u W^UV per head                                (section 3.2)
 * Beside the step: mla_append_kv writes the new tokens' cache rows,
 * mla_merge_w_kq / mla_absorb_q_latent give q_abs from the compressed query
 * latent through the merged query-side weight, and mla_merge_w_comb /
 * mla_out_comb give the layer output from u through the merged value/output
 * weight.
 * One decode step for a batch is: mla_absorb_q -> mla_decode_paged ->
 * mla_combine -> mla_out_proj, all on one stream (or, with the split plan
 * computed ahead: mla_decode_plan -> mla_absorb_q -> mla_decode_paged_planned
 * -> mla_combine -> mla_out_proj).
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers (except where a call says that
 *     pinned host memory is accepted), owned and allocated by the caller; the
 *     library never allocates, frees or synchronises. Every call
 *     only enqueues kernels on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns.
 *   - bf16 tensors are passed as uint16_t* holding IEEE bfloat16 bit patterns.
 *   - Tensors are dense, row-major, in the index order written beside each
 *     argument, and every pointer must be 16-byte aligned.
 *   - Supported shapes: d_nope = d_v = 128, d_r = 64, d_c = 512 (a cache row
 *     holds d_c + d_r = 576 values), page_size 64 or 128 tokens (Huny's
 *     Dev Blog "MLA 아키텍처 해부" section 6 item 2: pages of 64-128 tokens;
 *     the kernels read a page as one or two 64-token tiles), 1 <= H <= 128,
 *     max_pages_per_seq * page_size <= 2^30,
 *     n_q in {1, 2}, 1 <= B <= MLA_MAX_BATCH. Other values return
 *     MLA_ERR_UNSUPPORTED_SHAPE without launching anything.
 *   - Argument errors found on the host return a status before any launch.
 *     A failed launch returns MLA_ERR_CUDA (cudaGetLastError is consumed).
 *   - Kernels start while the kernel enqueued before them on the stream is
 *     still finishing (programmatic dependent launch): mla_absorb_q,
 *     mla_out_proj and mla_append_kv load their weights (w_uk, w_uv, w_dkr)
 *     in that time, so weights must not be written by the kernel enqueued
 *     just before the call. Every other input is read after that kernel has
 *     finished, except seq_lens and the workspace of mla_decode_paged (see
 *     its ordering rule).
 *   - Errors that only the device can see (a context length out of range, a
 *     page id outside [0, num_pages), a wait that timed out) are written as
 *     the first nonzero mla_status into *err_word (a device int32 the caller
 *     zeroes and reads after its own synchronisation). The kernels then clamp
 *     the bad value and finish without faulting; the results are not valid.
 *     The calls without an err_word (the projections, merges and merged-weight
 *     products) read no index from their inputs; their only device-side
 *     failure is a wait that gives up (about 2 s, a GPU fault), after which
 *     the kernel finishes without faulting and leaves its output incomplete.
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_ABI_VERSION 3
#define MLA_MAX_BATCH 4096

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,       /* null/misaligned pointer, negative size, bad count */
    MLA_ERR_UNSUPPORTED_SHAPE = 2, /* dimension outside the supported set */
    MLA_ERR_WORKSPACE_TOO_SMALL = 3,
    MLA_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed */
    MLA_ERR_TIMEOUT = 5,           /* device: a bounded wait gave up */
    MLA_ERR_BOUNDS = 6,            /* device: seq_len or page id out of range */
    MLA_ERR_RANGE = 7              /* device: a split partial outside the fp16 range */
} mla_status;

/* Human-readable name of a status code. Never NULL. */
const char* mla_status_string(int status);

/* MLA_ABI_VERSION of the loaded library. */
int mla_abi_version(void);

/* Bytes one token occupies in one layer's latent cache: (d_c + d_r) * 2.
 * Huny's Dev Blog "MLA 아키텍처 해부", section 2.2: (512 + 64) * 2 = 1152. */
size_t mla_cache_bytes_per_token(int d_c, int d_r);

/* Bytes of one cache page: page_size * (d_c + d_r) * 2 (73,728 at 64 tokens). */
size_t mla_page_bytes(int page_size, int d_c, int d_r);

/* ------------------------------------------------------------------------
 * mla_absorb_q — absorb W_UK into the per-head content query.
 *   q_abs[t][h][c]       = sum_i q_nope[t][h][i] * w_uk[h][i][c]   (c < d_c)
 *   q_abs[t][h][d_c + e] = q_rope[t][h][e]                         (e < d_r)
 * Huny's Dev Blog, section 3.1 (qt = q^C (W_i^UK)^T); tbr8.org "DeepSeek MLA
 * 深度解析", weight-absorption section. The positional query is already
 * rotated by the caller and is copied unchanged. fp32 accumulation, bf16
 * (round-to-nearest-even) output.
 *   q_nope [T][H][d_nope] bf16, q_rope [T][H][d_r] bf16,
 *   w_uk   [H][d_nope][d_c] bf16, q_abs [T][H][d_c + d_r] bf16 (output).
 *   T >= 1 is the number of query rows (B * n_q). */
mla_status mla_absorb_q(const uint16_t* q_nope, const uint16_t* q_rope, const uint16_t* w_uk,
                        uint16_t* q_abs, int T, int H, int d_nope, int d_r, int d_c, void* stream);

/* ------------------------------------------------------------------------
 * Query-side absorption through a merged weight (ingu627.github.io
 * "Multi-Head Latent Attention (MLA)" section 2.2: S = C_KV^T (W_UK^T W_UQ) C_Q,
 * W_KQ = W_UK^T W_UQ, taken per head because the softmax is per head).
 *
 * mla_merge_w_kq — the merge, done once per set of weights:
 *   w_kq[k][h][c] = sum_i w_uq[k][h][i] * w_uk[h][i][c]
 *   w_uq [d_q][H][d_nope] bf16, the query up-projection stored input-major
 *        (w_uq[k][h][i] maps compressed-query column k to head h's no-RoPE
 *        query column i), w_uk [H][d_nope][d_c] bf16,
 *   w_kq [d_q][H][d_c] bf16 (output; fp32 accumulation, round-to-nearest-even).
 *   64 <= d_q <= 16384, d_q % 64 == 0. w_uq and w_uk are read before the kernel
 *   enqueued just before the call has finished.
 *
 * mla_absorb_q_latent — the absorbed query of each row straight from its
 * compressed query latent, in place of mla_absorb_q (no separate W_UQ and
 * W_UK products per step):
 *   q_abs[t][h][c]       = sum_k c_q[t][k] * w_kq[k][h][c]    (c < d_c)
 *   q_abs[t][h][d_c + e] = q_rope[t][h][e]                    (e < d_r)
 *   c_q [T][d_q] bf16, w_kq [d_q][H][d_c] bf16 as written by mla_merge_w_kq,
 *   q_rope [T][H][d_r] bf16 (already rotated), q_abs [T][H][d_c + d_r] bf16
 *   (output). fp32 accumulation, bf16 (round-to-nearest-even) output. w_kq is
 *   read before the kernel enqueued just before the call has finished; c_q and
 *   q_rope after. At decode sizes the merged weight (d_q x H x d_c) is larger
 *   than W_UQ and W_UK together when d_c > d_nope, so this trades bytes read
 *   per step for one product instead of two. */
/* ------------------------------------------------------------------------
 * Merged value/output projection (Huny's Dev Blog "MLA 아키텍처 해부" section 3,
 * item 2: HeadOut_i = (a_i C^KV)(W_i^UV W_i^O), W_i,comb = W_i^UV W_i^O;
 * ikmyungterran.us, W~^O = W^UV W^O). The layer output is the sum of the heads'
 * outputs (the output projection of the concatenated heads).
 *
 * mla_merge_w_comb — the merge, done once per set of weights:
 *   w_comb[n][h][c] = sum_v w_o[n][h][v] * w_uv[h][v][c]
 *   w_uv [H][d_v][d_c] bf16 (as for mla_out_proj), w_o [d_model][H][d_v] bf16,
 *   the output projection with one row per output column, w_comb
 *   [d_model][H][d_c] bf16 (output; fp32 accumulation, round-to-nearest-even).
 *   d_model % 128 == 0, 128 <= d_model <= 65536. w_uv and w_o are read before
 *   the kernel enqueued just before the call has finished.
 *
 * mla_out_comb — the layer output straight from the merged latent outputs u,
 * in place of mla_out_proj followed by the output projection:
 *   out[t][n] = sum_h sum_c u[t][h][c] * w_comb[n][h][c]
 *   u [T][H][d_c] bf16 (mla_combine's output), w_comb as written by
 *   mla_merge_w_comb, out [T][d_model] bf16. The reduction over H * d_c is split
 *   across CTAs into fp32 partials in `workspace` (>= mla_out_comb_workspace_bytes
 *   bytes, no initial contents needed, 16-byte aligned) that a second kernel
 *   adds in a fixed order: results are bit-reproducible. 1 <= T <= 2 *
 *   MLA_MAX_BATCH. w_comb is read before the kernel enqueued just before the
 *   call has finished; u after. The merged weight (d_model x H x d_c) is
 *   d_c / d_v = 4 times the output projection's bytes, so at decode sizes the
 *   merge trades bytes read per step for one product instead of two.
 *
 * mla_out_comb_workspace_bytes: bytes of workspace for these sizes (0 if they
 * are invalid). */
mla_status mla_merge_w_comb(const uint16_t* w_uv, const uint16_t* w_o, uint16_t* w_comb, int H, int d_v, int d_c,
                            int d_model, void* stream);
size_t mla_out_comb_workspace_bytes(int T, int H, int d_model);
mla_status mla_out_comb(const uint16_t* u, const uint16_t* w_comb, uint16_t* out, int T, int H, int d_c,
                        int d_model, void* workspace, size_t workspace_bytes, void* stream);

mla_status mla_merge_w_kq(const uint16_t* w_uq, const uint16_t* w_uk, uint16_t* w_kq, int d_q, int H,
                          int d_nope, int d_c, void* stream);
mla_status mla_absorb_q_latent(const uint16_t* c_q, const uint16_t* q_rope, const uint16_t* w_kq,
                               uint16_t* q_abs, int T, int H, int d_q, int d_r, int d_c, void* stream);

/* ------------------------------------------------------------------------
 * Split-KV decode. The unit of work is a TILE of 64 tokens: a sequence of
 * context L holds ceil(L / 64) tiles, tile t in page block_table[b][t * 64 /
 * page_size] at row offset (t * 64) % page_size. The tiles of all sequences,
 * taken in sequence order, are cut into G = min(num_splits, P) contiguous
 * ranges of near-equal cost (P = total tiles; "page" below means tile). A
 * worker (a pair of CTAs on two SMs) that moves on to another sequence inside
 * its range pays for the switch, so the tiles are laid on a cost line where
 * sequence b (n_b tiles, first global tile P_b)
 * occupies [P_b + a*b, P_b + a*b + n_b) behind a switch stretch of a = 3
 * points (for b >= 1); V = P + a*(B-1), and a = 0 instead when
 * floor((P + 3*(B-1)) / G) < 4. Cut p (0 < p < G) sits at x = floor(p*V/G)
 * and lands on global page P_b + max(0, x - P_b - a*b) of the last sequence
 * b whose stretch starts at or before x (a cut inside a switch lands on the
 * sequence start). Range p covers the pages from cut p to cut p+1 (cut 0 =
 * page 0, cut G = P); ranges p >= G are empty. One worker processes one
 * range for one query index j. Where a range crosses a sequence boundary it
 * yields one partial per sequence it touches, so at most num_splits + B - 1
 * partials exist. The split points depend only on seq_lens and num_splits,
 * so results are bit-reproducible for the same arguments.
 *
 * mla_decode_default_splits: the num_splits that fills the current device
 * (SM count / (2 * n_q)); returns a value >= 1, or -1 if no device.
 *
 * mla_decode_workspace_bytes: bytes of workspace needed by mla_decode_paged
 * and read by mla_combine for these arguments (0 if they are invalid).
 *
 * Workspace layout (int32 unless noted; every block starts at a 256-byte
 * aligned offset; I = num_splits + B):
 *   hdr[64]                 hdr[0] = number of partials, hdr[1] = used splits,
 *                           hdr[2] = total tiles (P)
 *   range_item[num_splits+1] first partial index of each range
 *   seq_item[B+1]           first partial index of each sequence (partials of
 *                           sequence b are seq_item[b] .. seq_item[b+1]-1)
 *   seq_len_eff[B]          the context lengths actually used (clamped)
 *   item_seq[I], item_tile0[I], item_tile1[I]   sequence and tile range
 *                           [tile0, tile1) within the sequence
 *   lse_part[I][n_q][H]     float, natural-log sum-exp of the range's scores
 *   o_part[I][n_q][64][H][8] fp16, the range's softmax-normalised sum of
 *                           latents, head-minor in groups of eight columns:
 *                           o_part[k][j][c / 8][h][c % 8] is column c of head h.
 *                           A normalised partial is a convex combination of
 *                           cached latents, so |value| <= max |c|; values beyond
 *                           the fp16 range (65504) are reported as MLA_ERR_RANGE.
 *   range_desc[num_splits+1][4]  range p's first partial and that partial's
 *                           sequence, first tile and end tile: {range_item[p],
 *                           item_seq, item_tile0, item_tile1} of it, or
 *                           {range_item[p], -1, 0, 0} when the range is empty
 *                           (one 16-byte read for the decode kernel)
 */
int mla_decode_default_splits(int n_q);
size_t mla_decode_workspace_bytes(int B, int n_q, int H, int num_splits);

/* mla_decode_paged — scores of every head against the paged latent cache and
 * softmax-weighted latent sums, one partial per (range piece, query, head).
 * For sequence b with context L = seq_lens[b] (which INCLUDES its n_q new
 * tokens), query j attends logical tokens s = 0 .. L - n_q + j, and
 *   z_s = softmax_scale * sum_{e < 576} q_abs[b][j][h][e] * row_s[e]
 *   row_s = cache[block_table[b][s / page_size]][s % page_size][0:576]
 * (Huny's Dev Blog section 2.2: the cached row is c^KV (512) then the shared
 * rotated k^R (64); section 3.1: scoring in latent space; ikmyungterran.us
 * attention guide section 1.3: softmax(z / sqrt(d_k)); the pages give
 * d_k = d_nope + d_r, so softmax_scale is normally 1/sqrt(192)). The value
 * sum uses only the first 512 columns of each row. Unused block-table
 * entries are never read; slack rows past L in a sequence's last page may
 * hold any bits (NaN included) and never reach the result.
 *   q_abs       [B][n_q][H][576] bf16 (from mla_absorb_q)
 *   cache       [num_pages][page_size][576] bf16
 *   block_table [B][max_pages_per_seq] int32 physical page ids
 *   seq_lens    [B] int32, n_q <= L <= max_pages_per_seq * page_size
 *   workspace   >= mla_decode_workspace_bytes(B, n_q, H, num_splits) bytes
 *   err_word    device int32 or NULL (see the conventions above).
 * Ordering: the split plan is computed while the kernel enqueued just before
 * the call is still finishing (in the step, mla_absorb_q): seq_lens is read
 * and the plan arrays of workspace are written in that time, so that kernel
 * must neither write seq_lens nor use workspace (for example an mla_combine
 * of an earlier call on the same workspace). With programmatic dependent
 * launch that kernel may itself have started before the kernels ahead of it
 * finished, so none of those may still use workspace either: a step that ends
 * with mla_out_proj (or mla_out_comb) lets the next kernel start only once the
 * whole step has finished, so consecutive such steps may share one workspace;
 * after other sequences of calls, alternate two workspaces. q_abs, cache and block_table
 * are read after the kernel before has finished. */
mla_status mla_decode_paged(const uint16_t* q_abs, const uint16_t* cache,
                            const int32_t* block_table, const int32_t* seq_lens,
                            int B, int n_q, int H, int num_pages, int page_size,
                            int max_pages_per_seq, float softmax_scale, int num_splits,
                            void* workspace, size_t workspace_bytes, int32_t* err_word,
                            void* stream);

/* mla_decode_plan + mla_decode_paged_planned — mla_decode_paged in two calls,
 * so that the split plan can be computed earlier in the step: enqueue
 * mla_decode_plan before mla_absorb_q (it then runs beside the kernel before
 * it, under the same ordering rule for seq_lens and workspace), and
 * mla_decode_paged_planned where mla_decode_paged would go. The planned call
 * launches only the decode kernel and reads the plan that mla_decode_plan
 * wrote into workspace for the same B, n_q, H, max_pages_per_seq and
 * num_splits (and the seq_lens it was given); results are bit-identical to
 * mla_decode_paged. Arguments as for mla_decode_paged. */
mla_status mla_decode_plan(const int32_t* seq_lens, int B, int n_q, int H, int num_pages, int page_size,
                           int max_pages_per_seq, int num_splits, void* workspace, size_t workspace_bytes,
                           int32_t* err_word, void* stream);
mla_status mla_decode_paged_planned(const uint16_t* q_abs, const uint16_t* cache, const int32_t* block_table,
                                    int B, int n_q, int H, int num_pages, int page_size, int max_pages_per_seq,
                                    float softmax_scale, int num_splits, void* workspace, size_t workspace_bytes,
                                    int32_t* err_word, void* stream);

/* ------------------------------------------------------------------------
 * FP8 latent cache (Huny's Dev Blog section 6, item 4: FP8 on the latent cache
 * needs fine-grained per-channel or per-block scale factors, not one per
 * tensor, or outliers cost accuracy; ailab.paldyn.com "MQA와 GQA", KV-cache
 * quantisation: 1 byte per value halves the cache, and K's outlier channels are
 * why it is scaled per channel). A cached row is 576 e4m3 codes (1 byte each,
 * 576 bytes per token) with one float32 scale per column, shared by every token
 * of the cache: value = scales[d] * e4m3(code). e4m3: sign bit, 4 exponent bits
 * (bias 7), 3 mantissa bits, subnormals at exponent 0, 0x7F / 0xFF NaN, no
 * infinity, largest finite value 448.
 *
 * mla_quantize_fp8 — codes of bf16 rows with given scales:
 *   codes[r][d] = e4m3(rows[r][d] / scales[d])
 * the quotient one correctly rounded fp32 division, the conversion nearest
 * (ties to even) and saturating at +-448.
 *   rows [n_rows][576] bf16 (a paged cache is rows [num_pages * page_size][576]),
 *   scales [576] float32 (> 0), codes [n_rows][576] uint8 (output).
 *
 * mla_decode_paged_fp8 / mla_decode_paged_planned_fp8 — mla_decode_paged /
 * mla_decode_paged_planned on an FP8 cache: the same partials in the same
 * workspace (merged by mla_combine), computed on the dequantised latents
 *   row_s[d] = scales[d] * e4m3(cache8[block_table[b][s / page_size]][s % page_size][d]).
 * Each code is read from HBM once. The scales are folded into the query (the
 * scores) and into the written partials (the values); the codes are widened to
 * fp16 in shared memory (exactly) and the MMAs take fp16 operands (the scaled
 * query, P and the page), fp32 accumulation.
 *   cache8 [num_pages][page_size][576] uint8, scales [576] float32; the other
 *   arguments, the ordering rule and the error reporting are those of
 *   mla_decode_paged / mla_decode_paged_planned. */
mla_status mla_quantize_fp8(const uint16_t* rows, const float* scales, uint8_t* codes, int64_t n_rows,
                            void* stream);
mla_status mla_decode_paged_fp8(const uint16_t* q_abs, const uint8_t* cache8, const float* scales,
                                const int32_t* block_table, const int32_t* seq_lens, int B, int n_q, int H,
                                int num_pages, int page_size, int max_pages_per_seq, float softmax_scale,
                                int num_splits, void* workspace, size_t workspace_bytes, int32_t* err_word,
                                void* stream);
mla_status mla_decode_paged_planned_fp8(const uint16_t* q_abs, const uint8_t* cache8, const float* scales,
                                        const int32_t* block_table, int B, int n_q, int H, int num_pages,
                                        int page_size, int max_pages_per_seq, float softmax_scale, int num_splits,
                                        void* workspace, size_t workspace_bytes, int32_t* err_word, void* stream);

/* mla_combine — merge the range partials of each (sequence, query, head):
 *   lse = ln sum_k exp(lse_k),  u = sum_k exp(lse_k - lse) * o_k
 * (the flash-decoding merge; Huny's Dev Blog section 4 table names
 * FlashDecoding as the decode technique). A partial with lse_k = -inf has
 * weight 0.
 *   workspace  as filled by mla_decode_paged with the same B, n_q, H, num_splits
 *   u          [B][n_q][H][512] bf16 output (round-to-nearest-even)
 *   lse        [B][n_q][H] float output (natural log), may be NULL; device
 *              memory or pinned (page-locked, mapped) host memory, which the
 *              kernel writes over NVLink-C2C (a serving step's result goes to
 *              the host without a copy of its own). Pageable host memory, or a
 *              pointer the CUDA runtime does not know, returns
 *              MLA_ERR_INVALID_ARG before any launch.
 * Ordering: the plan part of the workspace (seq_item) is read while the kernel
 * before is still finishing, so that kernel must be the decode call that
 * produced the partials (or anything after which the plan is complete); the
 * partials are read after it has finished. The kernel after the merge may
 * start at once (it reads u and lse only after its own dependency wait). */
mla_status mla_combine(const void* workspace, int B, int n_q, int H, int num_splits,
                       uint16_t* u, float* lse, void* stream);

/* ------------------------------------------------------------------------
 * mla_decode_noalloc — mla_decode_paged followed by mla_combine for callers
 * that cannot provide a workspace. No page has a counterpart: this is a
 * deployment convenience of this library, not a step of the method.
 *
 * Who needs it: a serving loop that reserves all device memory for its KV
 * cache at start-up and never allocates afterwards (a cudaMalloc in the step
 * can block on the device and stall every request in flight), or a caller
 * that reaches the GPU through an interface exposing only its own tensors.
 * The plan and partial results live instead in one fixed device array of
 * mla_decode_noalloc_max_bytes() bytes (32 MiB) inside the library, which
 * every device that loads the library holds until the process exits. Calls
 * whose plan and partials would not fit (see mla_decode_workspace_bytes)
 * return MLA_ERR_WORKSPACE_TOO_SMALL without launching.
 *
 * The first call made with a device current looks up the array's device
 * address (cudaGetSymbolAddress); make that first call before any stream
 * capture. The address is kept with the unique id of the context it belongs
 * to; the first call under another context (for example after
 * cudaDeviceReset, which recreates the device's primary context) looks it up
 * again and must also come before any stream capture. All calls share the
 * array: calls whose kernels overlap on the GPU (other streams, other host
 * threads) race on it. Arguments and results
 * are those of mla_decode_paged and mla_combine (u [B][n_q][H][512] bf16,
 * lse [B][n_q][H] float or NULL, both in device memory). Nothing is allocated
 * or freed. */
size_t mla_decode_noalloc_max_bytes(void);
mla_status mla_decode_noalloc(const uint16_t* q_abs, const uint16_t* cache,
                              const int32_t* block_table, const int32_t* seq_lens,
                              int B, int n_q, int H, int num_pages, int page_size,
                              int max_pages_per_seq, float softmax_scale, int num_splits,
                              uint16_t* u, float* lse, int32_t* err_word, void* stream);

/* ------------------------------------------------------------------------
 * mla_out_proj — up-project the latent output through W_UV per head:
 *   out[t][h][v] = sum_c w_uv[h][v][c] * u[t][h][c]
 * Huny's Dev Blog section 3.2 (u_i W_i^UV after aggregation). fp32
 * accumulation, bf16 output.
 *   u [T][H][d_c] bf16, w_uv [H][d_v][d_c] bf16, out [T][H][d_v] bf16.
 * out may also be pinned (page-locked, mapped) host memory: the kernel then
 * writes the rows over NVLink-C2C, so a serving step's output reaches the host
 * without a copy of its own. Pageable host memory, or a pointer the CUDA
 * runtime does not know, returns MLA_ERR_INVALID_ARG before any launch
 * (checked with cudaPointerGetAttributes). The kernel enqueued after this one
 * starts only once every kernel before this one has finished, so the next
 * step's split plan never overlaps this step's decode kernel or merge. */
mla_status mla_out_proj(const uint16_t* u, const uint16_t* w_uv, uint16_t* out,
                        int T, int H, int d_c, int d_v, void* stream);

/* ------------------------------------------------------------------------
 * mla_append_kv — the latent-cache rows of the new tokens, written into their
 * pages (the step before decoding them):
 *   row[i] = sum_k h[t][k] w_dkr[i][k]         i < 576
 *   (row[512 + 2i], row[513 + 2i]) rotated by the angle pos * rope_theta^(-2i/64)
 *   cache[block_table[b][pos / page_size]][pos % page_size][0:576] = row (bf16, nearest even)
 * for new row t = b * n_q + j at position pos = L - n_q + j, L = seq_lens[b]
 * (which already counts the new tokens). Huny's Dev Blog section 1.2: the
 * joint compression c_t^KV = h_t W^DKV; section 2.2: the decoupled positional
 * key k^R_t = RoPE(h_t W^KR), shared by the heads and cached already rotated
 * (consecutive pairs, the convention of the input rows mla_decode_paged reads).
 *   h           [B][n_q][d_model] bf16 hidden states of the new tokens
 *   w_dkr       [576][d_model] bf16: rows 0..511 hold W^DKV transposed
 *               (w_dkr[i][k] = W^DKV[k][i]), rows 512..575 W^KR transposed
 *   cache, block_table, seq_lens, page_size, max_pages_per_seq: as for
 *               mla_decode_paged; only the new rows are written
 *   d_model     a multiple of 64, at most 65536
 *   workspace   >= mla_append_workspace_bytes(B * n_q, d_model) bytes: fp32
 *               partial sums of the d_model reduction (split across CTAs);
 *               no initial contents needed. Calls sharing a workspace must
 *               not overlap on the GPU.
 * The sums over d_model are added in a fixed order, so results are
 * reproducible bit for bit. A context length outside [n_q, max_pages * page_size]
 * is clamped and a page id outside [0, num_pages) skips that row; both are
 * reported in err_word as MLA_ERR_BOUNDS. w_dkr is read while the kernel
 * before it on the stream is still finishing (see the conventions above); h,
 * the cache, block_table and seq_lens only after it has finished (h is usually
 * that kernel's output). */
size_t mla_append_workspace_bytes(int T, int d_model);
mla_status mla_append_kv(const uint16_t* h, const uint16_t* w_dkr, uint16_t* cache,
                         const int32_t* block_table, const int32_t* seq_lens, int B, int n_q,
                         int d_model, int num_pages, int page_size, int max_pages_per_seq,
                         float rope_theta, void* workspace, size_t workspace_bytes,
                         int32_t* err_word, void* stream);

/* ------------------------------------------------------------------------
 * mla_copy16 — bytes copied from src to dst by a kernel on `stream`, for the
 * host I/O of a serving step: each of src and dst is device memory or pinned
 * (page-locked, mapped) host memory, which a GB300 kernel reads and writes
 * over NVLink-C2C; with every SM's accesses in flight a copy of a megabyte or
 * two takes a fraction of a copy-engine transfer's fixed cost.
 *   src, dst   16-byte aligned, not overlapping
 *   bytes      a positive multiple of 16
 * Pageable host memory, or a pointer the CUDA runtime does not know, returns
 * MLA_ERR_INVALID_ARG before any launch (checked with cudaPointerGetAttributes).
 * Unlike the decode calls this is an ordinary launch: it starts after the
 * kernel before it on the stream has finished, and the kernel after it starts
 * after it has finished. */
mla_status mla_copy16(const void* src, void* dst, size_t bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MLA_GB300_H */
