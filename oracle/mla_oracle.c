/*
 * CPU oracle for Multi-Head Latent Attention (MLA) decode over a latent cache.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * statement of what the decode path computes. Only the test suite, the
 * package's smoke check and the benchmark's CPU-baseline leg load it. It shares
 * no code, header or constant with the CUDA library, and reads the LOGICAL
 * (unpaged) per-sequence arrays, so it never sees the block table.
 *
 * Notation (Huny's Dev Blog, "Multi-Head Latent Attention(MLA) 아키텍처 해부",
 * sections 1-3; ikmyungterran.us "attention-mha-gqa-deepseek-mla-guide",
 * sections 1.3-1.4, 5-7):
 *   c_s      latent of cached token s, d_c values        (section 1, eq. c = h W_DKV)
 *   kr_s     shared, already rotated positional key, d_r (section 2, k^R = RoPE(h W_kR))
 *   q^C      per-head content query (no rotation), d_nope
 *   q^R      per-head rotated positional query, d_r
 *   W_UK[h]  stored [d_nope][d_c]; explicit key k_s[i] = sum_c W_UK[h][i][c] c_s[c]
 *   W_UV[h]  stored [d_v][d_c];    explicit value v_s[i] = sum_c W_UV[h][i][c] c_s[c]
 *   score    (q^C . k_s + q^R . kr_s) / sqrt(d_nope + d_r)   (section 2 eq. for q^T k; guide 1.3)
 *
 * Absorbed path (Huny section 3.1 and 3.2; guide section 6):
 *   qt[c]  = sum_i q^C[i] W_UK[h][i][c]                 (query absorbed into latent space)
 *   z_s    = (qt . c_s + q^R . kr_s) * scale
 *   p_s    = exp(z_s - m) / sum exp(z - m),  m = max z,  lse = m + ln(sum exp(z - m))
 *   u[c]   = sum_s p_s c_s[c]                            (u = a C^KV)
 *   out[i] = sum_c W_UV[h][i][c] u[c]                    (u W^UV)
 * Explicit path (Huny section 1.2 up-projection, section 2.2 concatenation):
 *   key_s = [k_s ; kr_s], q = [q^C ; q^R], out = sum_s softmax(q.key*scale)_s v_s
 *
 * Causal reading: sequence b holds L_b cached rows INCLUDING its n_q new
 * tokens; query j (0..n_q-1) attends rows 0 .. L_b - n_q + j.
 *
 * Inputs are bf16 bit patterns (uint16), widened exactly to double (or float
 * for the fp32 variant). Rows are selected by flat index r = (b*n_q + j)*H + h.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* MLA_ORACLE_MUTANT (test-only build flag, default 0) plants one known
 * mistake in the fp64 absorbed path, so the tests can show that the pins
 * catch it: 1 drops the positional term, 2 uses 1/sqrt(d_nope) as the scale,
 * 3 reads W_UK transposed, 4 attends one token too few, 5 aggregates u with
 * unnormalised weights. */
#ifndef MLA_ORACLE_MUTANT
#define MLA_ORACLE_MUTANT 0
#endif

static double bf(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bff(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

int mla_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- absorbed, fp64 */
/* For each selected row: q_abs[d_c + d_r] (absorbed query followed by q^R),
 * u[d_c], lse, out[d_v]. Any output pointer may be NULL. */
int mla_oracle_absorbed_f64(const uint16_t* q_nope, const uint16_t* q_rope,
                            const uint16_t* c, const uint16_t* kr,
                            const int64_t* seq_off, const int32_t* seq_lens,
                            const uint16_t* w_uk, const uint16_t* w_uv,
                            int B, int n_q, int H, int d_nope, int d_r, int d_c, int d_v,
                            double scale, const int64_t* rows, int64_t n_rows,
                            double* q_abs_out, double* u_out, double* lse_out, double* out_out) {
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t ri = 0; ri < n_rows; ++ri) {
        int64_t r = rows[ri];
        int h = (int)(r % H);
        int j = (int)((r / H) % n_q);
        int b = (int)(r / ((int64_t)H * n_q));
        if (b < 0 || b >= B) { bad = 1; continue; }
        int64_t L = seq_lens[b];
        int64_t n_att = L - n_q + j + 1;
#if MLA_ORACLE_MUTANT == 4
        if (n_att > 1) n_att -= 1;
#endif
#if MLA_ORACLE_MUTANT == 2
        scale = 1.0 / sqrt((double)d_nope);
#endif
        if (n_att < 1) { bad = 1; continue; }
        const uint16_t* qn = q_nope + r * d_nope;
        const uint16_t* qr = q_rope + r * d_r;
        const uint16_t* wk = w_uk + (int64_t)h * d_nope * d_c;
        const uint16_t* wv = w_uv + (int64_t)h * d_v * d_c;
        const uint16_t* cb = c + seq_off[b] * d_c;
        const uint16_t* kb = kr + seq_off[b] * d_r;

        double* qt = (double*)calloc((size_t)d_c, sizeof(double));
        double* z = (double*)malloc((size_t)n_att * sizeof(double));
        double* u = (double*)calloc((size_t)d_c, sizeof(double));
        /* absorbed query: qt = q^C W_UK[h] (row vector times [d_nope][d_c]) */
        for (int i = 0; i < d_nope; ++i) {
            double qi = bf(qn[i]);
#if MLA_ORACLE_MUTANT == 3
            for (int cc = 0; cc < d_c; ++cc) qt[cc] += qi * bf(wk[(int64_t)cc * d_nope + i]);
#else
            for (int cc = 0; cc < d_c; ++cc) qt[cc] += qi * bf(wk[(int64_t)i * d_c + cc]);
#endif
        }
        /* scores in latent space plus the positional term */
        double m = -INFINITY;
        for (int64_t s = 0; s < n_att; ++s) {
            double content = 0.0, pos = 0.0;
            for (int cc = 0; cc < d_c; ++cc) content += qt[cc] * bf(cb[s * d_c + cc]);
            for (int e = 0; e < d_r; ++e) pos += bf(qr[e]) * bf(kb[s * d_r + e]);
#if MLA_ORACLE_MUTANT == 1
            pos = 0.0;
#endif
            z[s] = (content + pos) * scale;
            if (z[s] > m) m = z[s];
        }
        double l = 0.0;
        for (int64_t s = 0; s < n_att; ++s) l += exp(z[s] - m);
        /* latent aggregation u = sum_s p_s c_s */
        for (int64_t s = 0; s < n_att; ++s) {
#if MLA_ORACLE_MUTANT == 5
            double p = exp(z[s] - m);
#else
            double p = exp(z[s] - m) / l;
#endif
            for (int cc = 0; cc < d_c; ++cc) u[cc] += p * bf(cb[s * d_c + cc]);
        }
        if (q_abs_out) {
            double* qa = q_abs_out + ri * (d_c + d_r);
            for (int cc = 0; cc < d_c; ++cc) qa[cc] = qt[cc];
            for (int e = 0; e < d_r; ++e) qa[d_c + e] = bf(qr[e]);
        }
        if (u_out) memcpy(u_out + ri * d_c, u, (size_t)d_c * sizeof(double));
        if (lse_out) lse_out[ri] = m + log(l);
        if (out_out) {
            /* up-projection through W_UV after aggregation */
            for (int i = 0; i < d_v; ++i) {
                double acc = 0.0;
                for (int cc = 0; cc < d_c; ++cc) acc += bf(wv[(int64_t)i * d_c + cc]) * u[cc];
                out_out[ri * d_v + i] = acc;
            }
        }
        free(qt);
        free(z);
        free(u);
    }
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------------- explicit, fp64 */
/* Reconstructs k_s = W_UK[h] c_s and v_s = W_UV[h] c_s for every attended
 * token, concatenates the positional parts, and runs textbook softmax
 * attention. logits/probs (optional) are [n_rows][max_tokens], filled up to
 * n_att and zero after. */
int mla_oracle_explicit_f64(const uint16_t* q_nope, const uint16_t* q_rope,
                            const uint16_t* c, const uint16_t* kr,
                            const int64_t* seq_off, const int32_t* seq_lens,
                            const uint16_t* w_uk, const uint16_t* w_uv,
                            int B, int n_q, int H, int d_nope, int d_r, int d_c, int d_v,
                            double scale, const int64_t* rows, int64_t n_rows,
                            double* lse_out, double* out_out,
                            double* logits_out, double* probs_out, int64_t max_tokens) {
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t ri = 0; ri < n_rows; ++ri) {
        int64_t r = rows[ri];
        int h = (int)(r % H);
        int j = (int)((r / H) % n_q);
        int b = (int)(r / ((int64_t)H * n_q));
        if (b < 0 || b >= B) { bad = 1; continue; }
        int64_t L = seq_lens[b];
        int64_t n_att = L - n_q + j + 1;
        if (n_att < 1) { bad = 1; continue; }
        const uint16_t* qn = q_nope + r * d_nope;
        const uint16_t* qr = q_rope + r * d_r;
        const uint16_t* wk = w_uk + (int64_t)h * d_nope * d_c;
        const uint16_t* wv = w_uv + (int64_t)h * d_v * d_c;
        const uint16_t* cb = c + seq_off[b] * d_c;
        const uint16_t* kb = kr + seq_off[b] * d_r;
        int dq = d_nope + d_r;

        double* q = (double*)malloc((size_t)dq * sizeof(double));
        double* key = (double*)malloc((size_t)dq * sizeof(double));
        double* v = (double*)malloc((size_t)d_v * sizeof(double));
        double* z = (double*)malloc((size_t)n_att * sizeof(double));
        double* o = (double*)calloc((size_t)d_v, sizeof(double));
        for (int i = 0; i < d_nope; ++i) q[i] = bf(qn[i]);
        for (int e = 0; e < d_r; ++e) q[d_nope + e] = bf(qr[e]);
        double m = -INFINITY;
        for (int64_t s = 0; s < n_att; ++s) {
            for (int i = 0; i < d_nope; ++i) {
                double acc = 0.0;
                for (int cc = 0; cc < d_c; ++cc) acc += bf(wk[(int64_t)i * d_c + cc]) * bf(cb[s * d_c + cc]);
                key[i] = acc;
            }
            for (int e = 0; e < d_r; ++e) key[d_nope + e] = bf(kb[s * d_r + e]);
            double dot = 0.0;
            for (int i = 0; i < dq; ++i) dot += q[i] * key[i];
            z[s] = dot * scale;
            if (z[s] > m) m = z[s];
        }
        double l = 0.0;
        for (int64_t s = 0; s < n_att; ++s) l += exp(z[s] - m);
        for (int64_t s = 0; s < n_att; ++s) {
            double p = exp(z[s] - m) / l;
            for (int i = 0; i < d_v; ++i) {
                double acc = 0.0;
                for (int cc = 0; cc < d_c; ++cc) acc += bf(wv[(int64_t)i * d_c + cc]) * bf(cb[s * d_c + cc]);
                v[i] = acc;
            }
            for (int i = 0; i < d_v; ++i) o[i] += p * v[i];
            if (probs_out && s < max_tokens) probs_out[ri * max_tokens + s] = p;
            if (logits_out && s < max_tokens) logits_out[ri * max_tokens + s] = z[s];
        }
        if (probs_out)
            for (int64_t s = n_att; s < max_tokens; ++s) probs_out[ri * max_tokens + s] = 0.0;
        if (logits_out)
            for (int64_t s = n_att; s < max_tokens; ++s) logits_out[ri * max_tokens + s] = 0.0;
        if (lse_out) lse_out[ri] = m + log(l);
        if (out_out) memcpy(out_out + ri * d_v, o, (size_t)d_v * sizeof(double));
        free(q); free(key); free(v); free(z); free(o);
    }
    return bad ? -1 : 0;
}

/* Absorbed-path logits and probabilities of one row, for the score and
 * softmax checks (Huny section 5, cases 3 and 4). */
int mla_oracle_absorbed_probs_f64(const uint16_t* q_nope, const uint16_t* q_rope,
                                  const uint16_t* c, const uint16_t* kr,
                                  const int64_t* seq_off, const int32_t* seq_lens,
                                  const uint16_t* w_uk,
                                  int B, int n_q, int H, int d_nope, int d_r, int d_c,
                                  double scale, int64_t row,
                                  double* content_out, double* pos_out,
                                  double* logits_out, double* probs_out) {
    int h = (int)(row % H);
    int j = (int)((row / H) % n_q);
    int b = (int)(row / ((int64_t)H * n_q));
    if (b < 0 || b >= B) return -1;
    int64_t n_att = (int64_t)seq_lens[b] - n_q + j + 1;
    if (n_att < 1) return -1;
    const uint16_t* qn = q_nope + row * d_nope;
    const uint16_t* qr = q_rope + row * d_r;
    const uint16_t* wk = w_uk + (int64_t)h * d_nope * d_c;
    const uint16_t* cb = c + seq_off[b] * d_c;
    const uint16_t* kb = kr + seq_off[b] * d_r;
    double* qt = (double*)calloc((size_t)d_c, sizeof(double));
    for (int i = 0; i < d_nope; ++i) {
        double qi = bf(qn[i]);
        for (int cc = 0; cc < d_c; ++cc) qt[cc] += qi * bf(wk[(int64_t)i * d_c + cc]);
    }
    double m = -INFINITY;
    for (int64_t s = 0; s < n_att; ++s) {
        double content = 0.0, pos = 0.0;
        for (int cc = 0; cc < d_c; ++cc) content += qt[cc] * bf(cb[s * d_c + cc]);
        for (int e = 0; e < d_r; ++e) pos += bf(qr[e]) * bf(kb[s * d_r + e]);
        if (content_out) content_out[s] = content;
        if (pos_out) pos_out[s] = pos;
        logits_out[s] = (content + pos) * scale;
        if (logits_out[s] > m) m = logits_out[s];
    }
    double l = 0.0;
    for (int64_t s = 0; s < n_att; ++s) l += exp(logits_out[s] - m);
    for (int64_t s = 0; s < n_att; ++s) probs_out[s] = exp(logits_out[s] - m) / l;
    free(qt);
    return (int)n_att;
}

/* Explicit keys of one sequence and head: K[s][i] = sum_c W_UK[h][i][c] c_s[c],
 * s < L. (Huny section 5, case 2: the reconstructed keys live in a
 * subspace of dimension at most d_c.) */
int mla_oracle_explicit_keys_f64(const uint16_t* c, const uint16_t* w_uk, int64_t L,
                                 int h, int d_nope, int d_c, double* k_out) {
    const uint16_t* wk = w_uk + (int64_t)h * d_nope * d_c;
    for (int64_t s = 0; s < L; ++s)
        for (int i = 0; i < d_nope; ++i) {
            double acc = 0.0;
            for (int cc = 0; cc < d_c; ++cc) acc += bf(wk[(int64_t)i * d_c + cc]) * bf(c[s * d_c + cc]);
            k_out[s * d_nope + i] = acc;
        }
    return 0;
}

/* ---------------------------------------------------------------- split-KV */
/* Flash-decoding partition (named on the Huny page, section 4 table, as the
 * MHA decode technique): attention restricted to the token range
 * [t0, t1) of the row's attended tokens gives a normalised partial
 * u_k = sum_{s in range} p_s c_s / sum p_s and lse_k = ln sum exp(z_s) over
 * the range. A range with no attended token gives u_k = 0, lse_k = -inf.
 * pieces: [n_pieces][2] token ranges; outputs [n_rows][n_pieces][d_c] and
 * [n_rows][n_pieces]. */
int mla_oracle_split_partials_f64(const uint16_t* q_nope, const uint16_t* q_rope,
                                  const uint16_t* c, const uint16_t* kr,
                                  const int64_t* seq_off, const int32_t* seq_lens,
                                  const uint16_t* w_uk,
                                  int B, int n_q, int H, int d_nope, int d_r, int d_c,
                                  double scale, const int64_t* rows, int64_t n_rows,
                                  const int64_t* pieces, int n_pieces,
                                  double* u_part, double* lse_part) {
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t ri = 0; ri < n_rows; ++ri) {
        int64_t r = rows[ri];
        int h = (int)(r % H);
        int j = (int)((r / H) % n_q);
        int b = (int)(r / ((int64_t)H * n_q));
        if (b < 0 || b >= B) { bad = 1; continue; }
        int64_t n_att = (int64_t)seq_lens[b] - n_q + j + 1;
        const uint16_t* qn = q_nope + r * d_nope;
        const uint16_t* qr = q_rope + r * d_r;
        const uint16_t* wk = w_uk + (int64_t)h * d_nope * d_c;
        const uint16_t* cb = c + seq_off[b] * d_c;
        const uint16_t* kb = kr + seq_off[b] * d_r;
        double* qt = (double*)calloc((size_t)d_c, sizeof(double));
        for (int i = 0; i < d_nope; ++i) {
            double qi = bf(qn[i]);
            for (int cc = 0; cc < d_c; ++cc) qt[cc] += qi * bf(wk[(int64_t)i * d_c + cc]);
        }
        for (int k = 0; k < n_pieces; ++k) {
            int64_t t0 = pieces[2 * k], t1 = pieces[2 * k + 1];
            if (t1 > n_att) t1 = n_att;
            double* uk = u_part + (ri * n_pieces + k) * d_c;
            for (int cc = 0; cc < d_c; ++cc) uk[cc] = 0.0;
            if (t1 <= t0) { lse_part[ri * n_pieces + k] = -INFINITY; continue; }
            double* z = (double*)malloc((size_t)(t1 - t0) * sizeof(double));
            double m = -INFINITY;
            for (int64_t s = t0; s < t1; ++s) {
                double content = 0.0, pos = 0.0;
                for (int cc = 0; cc < d_c; ++cc) content += qt[cc] * bf(cb[s * d_c + cc]);
                for (int e = 0; e < d_r; ++e) pos += bf(qr[e]) * bf(kb[s * d_r + e]);
                z[s - t0] = (content + pos) * scale;
                if (z[s - t0] > m) m = z[s - t0];
            }
            double l = 0.0;
            for (int64_t s = t0; s < t1; ++s) l += exp(z[s - t0] - m);
            for (int64_t s = t0; s < t1; ++s) {
                double p = exp(z[s - t0] - m) / l;
                for (int cc = 0; cc < d_c; ++cc) uk[cc] += p * bf(cb[s * d_c + cc]);
            }
            lse_part[ri * n_pieces + k] = m + log(l);
            free(z);
        }
        free(qt);
    }
    return bad ? -1 : 0;
}

/* Log-sum-exp merge of normalised partials:
 *   lse = ln sum_k exp(lse_k),  u = sum_k exp(lse_k - lse) u_k.
 * Pieces with lse_k = -inf carry weight 0. u_part [n][n_pieces][d_c]. */
int mla_oracle_combine_f64(const double* u_part, const double* lse_part, int64_t n,
                           int n_pieces, int d_c, double* u_out, double* lse_out) {
    for (int64_t i = 0; i < n; ++i) {
        double m = -INFINITY;
        for (int k = 0; k < n_pieces; ++k)
            if (lse_part[i * n_pieces + k] > m) m = lse_part[i * n_pieces + k];
        double sw = 0.0;
        for (int k = 0; k < n_pieces; ++k) {
            double lk = lse_part[i * n_pieces + k];
            if (lk != -INFINITY) sw += exp(lk - m);
        }
        double lse = m + log(sw);
        for (int cc = 0; cc < d_c; ++cc) u_out[i * d_c + cc] = 0.0;
        for (int k = 0; k < n_pieces; ++k) {
            double lk = lse_part[i * n_pieces + k];
            if (lk == -INFINITY) continue;
            double w = exp(lk - lse);
            const double* uk = u_part + (i * n_pieces + k) * d_c;
            for (int cc = 0; cc < d_c; ++cc) u_out[i * d_c + cc] += w * uk[cc];
        }
        lse_out[i] = lse;
    }
    return 0;
}

/* ---------------------------------------------------------------- absorbed, fp32 */
/* The same absorbed loops in float with float accumulation. Timed as the CPU
 * baseline; not used for parity. */
int mla_oracle_absorbed_f32(const uint16_t* q_nope, const uint16_t* q_rope,
                            const uint16_t* c, const uint16_t* kr,
                            const int64_t* seq_off, const int32_t* seq_lens,
                            const uint16_t* w_uk, const uint16_t* w_uv,
                            int B, int n_q, int H, int d_nope, int d_r, int d_c, int d_v,
                            float scale, const int64_t* rows, int64_t n_rows,
                            float* u_out, float* lse_out, float* out_out) {
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t ri = 0; ri < n_rows; ++ri) {
        int64_t r = rows[ri];
        int h = (int)(r % H);
        int j = (int)((r / H) % n_q);
        int b = (int)(r / ((int64_t)H * n_q));
        if (b < 0 || b >= B) { bad = 1; continue; }
        int64_t n_att = (int64_t)seq_lens[b] - n_q + j + 1;
        if (n_att < 1) { bad = 1; continue; }
        const uint16_t* qn = q_nope + r * d_nope;
        const uint16_t* qr = q_rope + r * d_r;
        const uint16_t* wk = w_uk + (int64_t)h * d_nope * d_c;
        const uint16_t* wv = w_uv + (int64_t)h * d_v * d_c;
        const uint16_t* cb = c + seq_off[b] * d_c;
        const uint16_t* kb = kr + seq_off[b] * d_r;
        float* qt = (float*)calloc((size_t)d_c, sizeof(float));
        float* z = (float*)malloc((size_t)n_att * sizeof(float));
        float* u = (float*)calloc((size_t)d_c, sizeof(float));
        for (int i = 0; i < d_nope; ++i) {
            float qi = bff(qn[i]);
            for (int cc = 0; cc < d_c; ++cc) qt[cc] += qi * bff(wk[(int64_t)i * d_c + cc]);
        }
        float m = -INFINITY;
        for (int64_t s = 0; s < n_att; ++s) {
            float content = 0.0f, pos = 0.0f;
            for (int cc = 0; cc < d_c; ++cc) content += qt[cc] * bff(cb[s * d_c + cc]);
            for (int e = 0; e < d_r; ++e) pos += bff(qr[e]) * bff(kb[s * d_r + e]);
            z[s] = (content + pos) * scale;
            if (z[s] > m) m = z[s];
        }
        float l = 0.0f;
        for (int64_t s = 0; s < n_att; ++s) l += expf(z[s] - m);
        for (int64_t s = 0; s < n_att; ++s) {
            float p = expf(z[s] - m) / l;
            for (int cc = 0; cc < d_c; ++cc) u[cc] += p * bff(cb[s * d_c + cc]);
        }
        if (u_out) memcpy(u_out + ri * d_c, u, (size_t)d_c * sizeof(float));
        if (lse_out) lse_out[ri] = m + logf(l);
        if (out_out)
            for (int i = 0; i < d_v; ++i) {
                float acc = 0.0f;
                for (int cc = 0; cc < d_c; ++cc) acc += bff(wv[(int64_t)i * d_c + cc]) * u[cc];
                out_out[ri * d_v + i] = acc;
            }
        free(qt); free(z); free(u);
    }
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------------- single steps */
/* Absorption step alone (Huny section 3.1): q_abs[r][c] = sum_i q^C[r][i] W_UK[h][i][c]
 * for c < d_c, then q^R copied to q_abs[r][d_c + e]. Rows r = t*H + h of a
 * [T][H] query block. */
int mla_oracle_absorb_q_f64(const uint16_t* q_nope, const uint16_t* q_rope, const uint16_t* w_uk,
                            int64_t T, int H, int d_nope, int d_r, int d_c, double* q_abs) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T * H; ++r) {
        int h = (int)(r % H);
        const uint16_t* wk = w_uk + (int64_t)h * d_nope * d_c;
        double* qa = q_abs + r * (d_c + d_r);
        for (int cc = 0; cc < d_c; ++cc) qa[cc] = 0.0;
        for (int i = 0; i < d_nope; ++i) {
            double qi = bf(q_nope[r * d_nope + i]);
            for (int cc = 0; cc < d_c; ++cc) qa[cc] += qi * bf(wk[(int64_t)i * d_c + cc]);
        }
        for (int e = 0; e < d_r; ++e) qa[d_c + e] = bf(q_rope[r * d_r + e]);
    }
    return 0;
}

/* Up-projection step alone (Huny section 3.2): out[r][i] = sum_c W_UV[h][i][c] u[r][c]. */
int mla_oracle_out_proj_f64(const uint16_t* u, const uint16_t* w_uv, int64_t T, int H, int d_c,
                            int d_v, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T * H; ++r) {
        int h = (int)(r % H);
        const uint16_t* wv = w_uv + (int64_t)h * d_v * d_c;
        for (int i = 0; i < d_v; ++i) {
            double acc = 0.0;
            for (int cc = 0; cc < d_c; ++cc) acc += bf(wv[(int64_t)i * d_c + cc]) * bf(u[r * d_c + cc]);
            out[r * d_v + i] = acc;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------- query-side absorption */
/* The merged query weight (ingu627.github.io "Multi-Head Latent Attention (MLA)"
 * section 2.2: S = C_KV^T (W_UK^T W_UQ) C_Q, read per head, since the softmax
 * is taken per head). With the query up-projection stored input-major,
 * w_uq[k][h][i] = weight from compressed-query column k to head h's no-RoPE
 * query column i, and W_UK as w_uk[h][i][c]:
 *   w_kq[k][h][c] = sum_i w_uq[k][h][i] * w_uk[h][i][c]
 * so that sum_k c_q[k] w_kq[k][h][c] = sum_i (sum_k c_q[k] w_uq[k][h][i]) w_uk[h][i][c]. */
int mla_oracle_merge_w_kq_f64(const uint16_t* w_uq, const uint16_t* w_uk, int d_q, int H, int d_nope,
                              int d_c, double* w_kq) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < (int64_t)d_q * H; ++r) {
        const int h = (int)(r % H);
        const uint16_t* wk = w_uk + (int64_t)h * d_nope * d_c;
        double* out = w_kq + r * d_c;
        for (int cc = 0; cc < d_c; ++cc) out[cc] = 0.0;
        for (int i = 0; i < d_nope; ++i) {
            const double a = bf(w_uq[r * d_nope + i]);
            for (int cc = 0; cc < d_c; ++cc) out[cc] += a * bf(wk[(int64_t)i * d_c + cc]);
        }
    }
    return 0;
}

/* The absorbed query straight from the compressed query latent through the
 * merged weight: q_abs[t][h][c] = sum_k c_q[t][k] w_kq[k][h][c] for c < d_c,
 * then the (already rotated) positional query q^R[t][h] copied to columns
 * d_c .. d_c + d_r - 1. w_kq is taken as given (fp64). */
int mla_oracle_absorb_latent_f64(const uint16_t* c_q, const double* w_kq, const uint16_t* q_rope, int64_t T, int H,
                                 int d_q, int d_r, int d_c, double* q_abs) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T * H; ++r) {
        const int64_t t = r / H;
        const int h = (int)(r % H);
        double* qa = q_abs + r * (d_c + d_r);
        for (int cc = 0; cc < d_c; ++cc) qa[cc] = 0.0;
        for (int k = 0; k < d_q; ++k) {
            const double a = bf(c_q[t * d_q + k]);
            const double* w = w_kq + ((int64_t)k * H + h) * d_c;
            for (int cc = 0; cc < d_c; ++cc) qa[cc] += a * w[cc];
        }
        for (int e = 0; e < d_r; ++e) qa[d_c + e] = bf(q_rope[r * d_r + e]);
    }
    return 0;
}

/* ---------------------------------------------------------------- merged output projection */
/* The merged value/output weight (Huny's Dev Blog "MLA 아키텍처 해부" section
 * 3, item 2: HeadOut_i = (a_i C^KV)(W_i^UV W_i^O), W_i,comb = W_i^UV W_i^O of
 * size d_c x d; ikmyungterran.us, the absorbed W~^O = W^UV W^O). With W^UV
 * stored as w_uv[h][v][c] (value column v of head h from latent column c) and
 * the output projection one row per output column, w_o[n][h][v]:
 *   w_comb[n][h][c] = sum_v w_o[n][h][v] * w_uv[h][v][c]. */
int mla_oracle_merge_w_comb_f64(const uint16_t* w_uv, const uint16_t* w_o, int H, int d_v, int d_c, int d_model,
                                double* w_comb) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < (int64_t)d_model * H; ++r) {
        const int h = (int)(r % H);
        const uint16_t* wv = w_uv + (int64_t)h * d_v * d_c;
        double* out = w_comb + r * d_c;
        for (int cc = 0; cc < d_c; ++cc) out[cc] = 0.0;
        for (int v = 0; v < d_v; ++v) {
            const double a = bf(w_o[r * d_v + v]);
            for (int cc = 0; cc < d_c; ++cc) out[cc] += a * bf(wv[(int64_t)v * d_c + cc]);
        }
    }
    return 0;
}

/* The attention layer's output through the merged weight, summed over the
 * heads (the output projection of the concatenated heads):
 *   out[t][n] = sum_h sum_c u[t][h][c] * w_comb[n][h][c]. w_comb is taken as given (fp64). */
int mla_oracle_out_comb_f64(const uint16_t* u, const double* w_comb, int64_t T, int H, int d_c, int d_model,
                            double* out) {
    const int64_t K = (int64_t)H * d_c;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T * d_model; ++r) {
        const int64_t t = r / d_model, n = r % d_model;
        const uint16_t* ut = u + t * K;
        const double* w = w_comb + n * K;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += bf(ut[k]) * w[k];
        out[r] = acc;
    }
    return 0;
}

/* ---------------------------------------------------------------- cache append */
/* Latent-cache row of a new token (Huny section 1.2: c_t^KV = h_t W^DKV, the
 * joint low-rank compression; section 2.2: the decoupled positional key
 * k^R_t = RoPE(h_t W^KR), shared by all heads and cached already rotated).
 * The weights come transposed, one row per output column: w_dkr[i][k] for
 * i < d_c is W^DKV[k][i], for d_c <= i < d_c + d_r it is W^KR[k][i - d_c].
 * For new row t at position pos[t]:
 *   row[t][i]       = sum_k h[t][k] w_dkr[i][k]                 (i < d_c)
 *   k[e]            = sum_k h[t][k] w_dkr[d_c + e][k]           (e < d_r)
 *   (row[t][d_c+2i], row[t][d_c+2i+1]) = (k[2i] cos a - k[2i+1] sin a,
 *                                         k[2i] sin a + k[2i+1] cos a),
 *   a = pos[t] * theta^(-2i / d_r)
 * (the rotation R_t of the pages, applied to consecutive pairs). */
int mla_oracle_append_f64(const uint16_t* h, const uint16_t* w_dkr, const int64_t* pos, int64_t T, int d_model,
                          int d_c, int d_r, double theta, double* row_out) {
    const int D = d_c + d_r;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double* row = row_out + t * D;
        for (int i = 0; i < D; ++i) {
            double acc = 0.0;
            for (int k = 0; k < d_model; ++k) acc += bf(h[t * d_model + k]) * bf(w_dkr[(int64_t)i * d_model + k]);
            row[i] = acc;
        }
        for (int i = 0; i < d_r / 2; ++i) {
            const double a = (double)pos[t] * pow(theta, -2.0 * i / d_r);
            const double x = row[d_c + 2 * i], y = row[d_c + 2 * i + 1];
            row[d_c + 2 * i] = x * cos(a) - y * sin(a);
            row[d_c + 2 * i + 1] = x * sin(a) + y * cos(a);
        }
    }
    return 0;
}


/* ---------------------------------------------------------------- FP8 (e4m3) latents */
/* An FP8 latent cache stores every row as e4m3 codes with one float32 scale per
 * column (the per-channel scaling of Huny's Dev Blog section 6, item 4): the
 * value of code q in column d is scale[d] * e4m3(q). e4m3 (the OCP 8-bit
 * floating-point format): bit 7 sign, bits 6..3 exponent with bias 7, bits 2..0
 * mantissa; exponent field 0 encodes the subnormals (m/8) * 2^-6; the codes with
 * all exponent and mantissa bits set (0x7F, 0xFF) are NaN; there is no infinity. */
static double e4m3_value(uint8_t q) {
    const int sign = (q >> 7) & 1, ex = (q >> 3) & 15, man = q & 7;
    double v;
    if (ex == 15 && man == 7) return NAN;
    if (ex == 0)
        v = ldexp((double)man / 8.0, -6);
    else
        v = ldexp(1.0 + (double)man / 8.0, ex - 7);
    return sign ? -v : v;
}

int mla_oracle_e4m3_decode(const uint8_t* codes, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
    return 0;
}

/* out[r][d] = scale[d] * e4m3(codes[r][d]) for rows r < n_rows, columns d < D. */
int mla_oracle_dequant_fp8_f64(const uint8_t* codes, const float* scale, int64_t n_rows, int D, double* out) {
    for (int64_t r = 0; r < n_rows; ++r)
        for (int d = 0; d < D; ++d) out[r * D + d] = (double)scale[d] * e4m3_value(codes[r * D + d]);
    return 0;
}

/* The absorbed path of mla_oracle_absorbed_f64 on latents given as doubles
 * (c [total][d_c], kr [total][d_r], e.g. dequantised FP8 rows); queries and
 * weights are bf16 bit patterns as there. Same loops, same order. */
int mla_oracle_absorbed_lat_f64(const uint16_t* q_nope, const uint16_t* q_rope,
                                const double* c, const double* kr,
                                const int64_t* seq_off, const int32_t* seq_lens,
                                const uint16_t* w_uk, const uint16_t* w_uv,
                                int B, int n_q, int H, int d_nope, int d_r, int d_c, int d_v,
                                double scale, const int64_t* rows, int64_t n_rows,
                                double* q_abs_out, double* u_out, double* lse_out, double* out_out) {
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t ri = 0; ri < n_rows; ++ri) {
        int64_t r = rows[ri];
        int h = (int)(r % H);
        int j = (int)((r / H) % n_q);
        int b = (int)(r / ((int64_t)H * n_q));
        if (b < 0 || b >= B) { bad = 1; continue; }
        int64_t n_att = (int64_t)seq_lens[b] - n_q + j + 1;
        if (n_att < 1) { bad = 1; continue; }
        const uint16_t* qn = q_nope + r * d_nope;
        const uint16_t* qr = q_rope + r * d_r;
        const uint16_t* wk = w_uk + (int64_t)h * d_nope * d_c;
        const uint16_t* wv = w_uv + (int64_t)h * d_v * d_c;
        const double* cb = c + seq_off[b] * d_c;
        const double* kb = kr + seq_off[b] * d_r;
        double* qt = (double*)calloc((size_t)d_c, sizeof(double));
        double* z = (double*)malloc((size_t)n_att * sizeof(double));
        double* u = (double*)calloc((size_t)d_c, sizeof(double));
        for (int i = 0; i < d_nope; ++i) {
            double qi = bf(qn[i]);
            for (int cc = 0; cc < d_c; ++cc) qt[cc] += qi * bf(wk[(int64_t)i * d_c + cc]);
        }
        double m = -INFINITY;
        for (int64_t s = 0; s < n_att; ++s) {
            double content = 0.0, pos = 0.0;
            for (int cc = 0; cc < d_c; ++cc) content += qt[cc] * cb[s * d_c + cc];
            for (int e = 0; e < d_r; ++e) pos += bf(qr[e]) * kb[s * d_r + e];
            z[s] = (content + pos) * scale;
            if (z[s] > m) m = z[s];
        }
        double l = 0.0;
        for (int64_t s = 0; s < n_att; ++s) l += exp(z[s] - m);
        for (int64_t s = 0; s < n_att; ++s) {
            double p = exp(z[s] - m) / l;
            for (int cc = 0; cc < d_c; ++cc) u[cc] += p * cb[s * d_c + cc];
        }
        if (q_abs_out) {
            double* qa = q_abs_out + ri * (d_c + d_r);
            for (int cc = 0; cc < d_c; ++cc) qa[cc] = qt[cc];
            for (int e = 0; e < d_r; ++e) qa[d_c + e] = bf(qr[e]);
        }
        if (u_out) memcpy(u_out + ri * d_c, u, (size_t)d_c * sizeof(double));
        if (lse_out) lse_out[ri] = m + log(l);
        if (out_out) {
            for (int i = 0; i < d_v; ++i) {
                double acc = 0.0;
                for (int cc = 0; cc < d_c; ++cc) acc += bf(wv[(int64_t)i * d_c + cc]) * u[cc];
                out_out[ri * d_v + i] = acc;
            }
        }
        free(qt);
        free(z);
        free(u);
    }
    return bad ? -1 : 0;
}
