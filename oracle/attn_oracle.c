/*
 * attn_oracle.c -- float64 CPU oracle for the scaled-dot-product attention
 * forward (prefill and seq_len=1 decode over a paged or contiguous KV cache).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA path.
 *
 * What it computes is the plain definition, written out with no blocking,
 * fusion or online rescaling:
 *
 *     s_j  = scale * sum_d q[i,d] * k[j,d]           for every visible key j
 *     m    = max_j s_j
 *     l    = sum_j exp(s_j - m)
 *     o[d] = sum_j exp(s_j - m) * v[j,d] / l
 *     lse  = m + ln(l)
 *
 * Sources followed:
 *   - "attention" / "Prefill attention kernel" (Wave February 2025 Release,
 *     FlashDecoding list; WAVE MLSys 2026 summary, Attention (prefill),
 *     Figures 2-4).  The pages never print the formula; the reading used is
 *     standard scaled-dot-product attention with an optional causal mask.
 *   - BHSD and BSHD are the same computation with the sequence and head
 *     indices swapped (WAVE MLSys 2026 summary, "Assumption 1": BSHD only
 *     swaps the boundary indexing symbols).
 *   - "Flash Decoding Kernel with paged attention" and the fake page table
 *     test fixture (Wave February 2025 Release, FlashDecoding list): decode
 *     is attention of one query per head against a sequence's keys, read
 *     through a page table.
 *
 * Readings where the pages are silent:
 *   - causal visibility is bottom-right aligned: key j is visible to query i
 *     iff j <= i + (S_kv - S_q);
 *   - a row with no visible key gets o = 0 and lse = -inf;
 *   - grouped-query heads: query head h reads kv head h / (H_q / H_kv);
 *   - paged KV: logical key t of sequence b lives in pool page
 *     page_table[b * max_pages + t / page_size], slot t % page_size, with the
 *     pool laid out [num_pages, page_size, H_kv, D]; a NULL page table means
 *     "contiguous", i.e. page b of a pool [B, page_size, H_kv, D].
 *
 * Extend (prefill against a paged KV cache, "Extend Attention", Wave
 * February 2025 Release, De-Prioritized list; the SGLang "extend" mode of
 * the WAVE MLSys 2026 summary, Integration) is the prefill definition applied
 * to each sequence's gathered keys: S_q new queries of sequence b attend to
 * its kv_lens[b] cached keys (which include the new tokens), causal
 * alignment bottom-right per sequence, kv head h / (H_q / H_kv).
 *
 * FP8 prefill ("FAv3 - FP8", Wave February 2025 Release, EvoFormer list)
 * is the same definition on inputs stored as 8-bit E4M3 codes with one
 * descale factor per tensor: x = descale * value(code).  value() follows the
 * OCP 8-bit floating point E4M3 format: sign bit, 4 exponent bits with bias
 * 7, 3 mantissa bits; exponent 0 encodes subnormals m/8 * 2^-6; the all-ones
 * exponent with all-ones mantissa is NaN; there is no infinity (so the
 * largest finite value is 1.75 * 2^8 = 448).
 *
 * Backward ("Backward Flash Attention", Wave February 2025 Release,
 * EvoFormer list; "Functionality & Performance on backward attention",
 * Milestones): the gradients of the same
 * definition, written out from the chain rule with P the exact softmax,
 *     O_i   = sum_j P_ij v_j,          D_i = sum_d dO_i[d] O_i[d]
 *     dV_j  = sum_i P_ij dO_i,         dP_ij = dO_i . v_j
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i
 * over the visible (i, j) pairs.
 *
 * FP8 MQA logits ("[FlyDSL] FP8 MQA logits improvements for gfx950", aiter
 * PR 7412: Summary; Changes/Kernel head_acc, rs_head, lds_scales; Test
 * windows causal/cp/misaligned/empty/past_end; clean_logits).  The page names
 * the pieces but prints no formula; the reading taken: one K row per key
 * shared by all heads (multi-query), a per-head score, a nonlinearity (ReLU)
 * between the per-head products and the weighted head reduction (without it
 * the head sum would collapse into one product), and a per-key scale:
 *     logits[i,j] = sum_h w[i,h] * max(0, kv_scale[j] * (q[i,h] . k[j]))
 * for j in row i's window [start_i, end_i) clamped to [0, S_kv); outside it
 * the entry is -inf when clean_logits is set and left untouched otherwise.
 *
 * Rows are independent; they are spread over POSIX threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BHSD 0
#define ORACLE_BSHD 1

/* Offset of element (b, h, s, d) of a [B,H,S,D] (BHSD) or [B,S,H,D] (BSHD)
 * tensor. */
static size_t offset4(int layout, long b, long h, long s, long d,
                      long H, long S, long D) {
    if (layout == ORACLE_BHSD) return (size_t)(((b * H + h) * S + s) * D + d);
    return (size_t)(((b * S + s) * H + h) * D + d);
}

/* ---------------------------------------------------------------- prefill */

typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    long B, H, S_q, S_kv, D;
    int layout, causal;
    double scale;
    long next_row; /* shared work counter over (b, h, i) */
} prefill_job;

/* One query row (b, h, i): two passes over its visible keys. */
static void prefill_row(const prefill_job *J, long b, long h, long i,
                        double *s_buf) {
    const long D = J->D;
    /* visible keys are 0 .. last (inclusive) */
    long last = J->S_kv - 1;
    if (J->causal) {
        long lim = i + (J->S_kv - J->S_q);
        if (lim < last) last = lim;
    }
    double *o_row = J->o + offset4(J->layout, b, h, i, 0, J->H, J->S_q, D);
    double *lse_out = J->lse + (size_t)((b * J->H + h) * J->S_q + i);
    if (last < 0) {
        for (long d = 0; d < D; ++d) o_row[d] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    const double *q_row = J->q + offset4(J->layout, b, h, i, 0, J->H, J->S_q, D);

    double m = -INFINITY;
    for (long j = 0; j <= last; ++j) {
        const double *k_row = J->k + offset4(J->layout, b, h, j, 0, J->H, J->S_kv, D);
        double dot = 0.0;
        for (long d = 0; d < D; ++d) dot += q_row[d] * k_row[d];
        s_buf[j] = J->scale * dot;
        if (s_buf[j] > m) m = s_buf[j];
    }
    double l = 0.0;
    for (long d = 0; d < D; ++d) o_row[d] = 0.0;
    for (long j = 0; j <= last; ++j) {
        double w = exp(s_buf[j] - m);
        l += w;
        const double *v_row = J->v + offset4(J->layout, b, h, j, 0, J->H, J->S_kv, D);
        for (long d = 0; d < D; ++d) o_row[d] += w * v_row[d];
    }
    for (long d = 0; d < D; ++d) o_row[d] /= l;
    *lse_out = m + log(l);
}

static void *prefill_worker(void *arg) {
    prefill_job *J = (prefill_job *)arg;
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)(J->S_kv > 0 ? J->S_kv : 1));
    if (!s_buf) return (void *)1;
    const long total = J->B * J->H * J->S_q;
    for (;;) {
        long r = __atomic_fetch_add(&J->next_row, 1, __ATOMIC_RELAXED);
        if (r >= total) break;
        long i = r % J->S_q;
        long h = (r / J->S_q) % J->H;
        long b = r / (J->S_q * J->H);
        prefill_row(J, b, h, i, s_buf);
    }
    free(s_buf);
    return NULL;
}

static int run_threads(void *(*fn)(void *), void *job, int n_threads) {
    if (n_threads < 1) n_threads = 1;
    if (n_threads == 1) return fn(job) == NULL ? 0 : -1;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!tid) return -1;
    int started = 0, rc = 0;
    for (; started < n_threads; ++started)
        if (pthread_create(&tid[started], NULL, fn, job) != 0) { rc = -1; break; }
    for (int t = 0; t < started; ++t) {
        void *ret = NULL;
        pthread_join(tid[t], &ret);
        if (ret != NULL) rc = -1;
    }
    free(tid);
    return rc;
}

/* q: [B,H,S_q,D] or [B,S_q,H,D]; k, v: same layout with S_kv; o: as q;
 * lse: [B,H,S_q].  Returns 0 on success, -1 on bad arguments or failure. */
int oracle_prefill_f64(const double *q, const double *k, const double *v,
                       double *o, double *lse, long B, long H, long S_q,
                       long S_kv, long D, int layout, int causal, double scale,
                       int n_threads) {
    if (B < 0 || H < 0 || S_q < 0 || S_kv < 0 || D <= 0) return -1;
    if (layout != ORACLE_BHSD && layout != ORACLE_BSHD) return -1;
    if (B == 0 || H == 0 || S_q == 0) return 0;
    prefill_job J = {q, k, v, o, lse, B, H, S_q, S_kv, D, layout, causal, scale, 0};
    return run_threads(prefill_worker, &J, n_threads);
}

/* ----------------------------------------------------------------- decode */

typedef struct {
    const double *q, *k_pool, *v_pool;
    const int32_t *page_table, *kv_lens;
    double *o, *lse;
    long B, H_q, H_kv, D, page_size, max_pages;
    double scale;
    long next_row; /* shared work counter over (b, h) */
} decode_job;

/* Gather sequence b's keys and values for kv head g into contiguous
 * [kv_len, D] arrays, through the page table (pool [pages, page_size, H_kv,
 * D]; a NULL page table means sequence b owns page b). */
static void gather_sequence(const double *k_pool, const double *v_pool,
                            const int32_t *page_table, long max_pages,
                            long page_size, long H_kv, long D, long b, long g,
                            long kv_len, double *k_seq, double *v_seq) {
    for (long t = 0; t < kv_len; ++t) {
        long page = page_table ? (long)page_table[b * max_pages + t / page_size] : b;
        long slot = t % page_size;
        size_t row = (size_t)(((page * page_size + slot) * H_kv + g) * D);
        memcpy(k_seq + t * D, k_pool + row, sizeof(double) * (size_t)D);
        memcpy(v_seq + t * D, v_pool + row, sizeof(double) * (size_t)D);
    }
}

static void *decode_worker(void *arg) {
    decode_job *J = (decode_job *)arg;
    const long D = J->D;
    const long cap = J->max_pages * J->page_size;
    double *k_seq = (double *)malloc(sizeof(double) * (size_t)(cap * D + 1));
    double *v_seq = (double *)malloc(sizeof(double) * (size_t)(cap * D + 1));
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)(cap + 1));
    if (!k_seq || !v_seq || !s_buf) {
        free(k_seq); free(v_seq); free(s_buf);
        return (void *)1;
    }
    const long group = J->H_q / J->H_kv;
    const long total = J->B * J->H_q;
    long have_b = -1, have_g = -1;
    for (;;) {
        long r = __atomic_fetch_add(&J->next_row, 1, __ATOMIC_RELAXED);
        if (r >= total) break;
        long b = r / J->H_q, h = r % J->H_q, g = h / group;
        long kv_len = J->kv_lens[b];
        if (b != have_b || g != have_g) {
            gather_sequence(J->k_pool, J->v_pool, J->page_table, J->max_pages,
                            J->page_size, J->H_kv, D, b, g, kv_len, k_seq, v_seq);
            have_b = b;
            have_g = g;
        }
        const double *q_row = J->q + (size_t)((b * J->H_q + h) * D);
        double *o_row = J->o + (size_t)((b * J->H_q + h) * D);
        double *lse_out = J->lse + (size_t)(b * J->H_q + h);
        if (kv_len <= 0) {
            for (long d = 0; d < D; ++d) o_row[d] = 0.0;
            *lse_out = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (long t = 0; t < kv_len; ++t) {
            double dot = 0.0;
            for (long d = 0; d < D; ++d) dot += q_row[d] * k_seq[t * D + d];
            s_buf[t] = J->scale * dot;
            if (s_buf[t] > m) m = s_buf[t];
        }
        double l = 0.0;
        for (long d = 0; d < D; ++d) o_row[d] = 0.0;
        for (long t = 0; t < kv_len; ++t) {
            double w = exp(s_buf[t] - m);
            l += w;
            for (long d = 0; d < D; ++d) o_row[d] += w * v_seq[t * D + d];
        }
        for (long d = 0; d < D; ++d) o_row[d] /= l;
        *lse_out = m + log(l);
    }
    free(k_seq);
    free(v_seq);
    free(s_buf);
    return NULL;
}

/* q: [B,H_q,D]; k_pool, v_pool: [num_pages, page_size, H_kv, D] (a NULL
 * page_table means the pool is [B, page_size, H_kv, D] and sequence b owns
 * page b); page_table: [B, max_pages] int32 or NULL; kv_lens: [B] int32;
 * o: [B,H_q,D]; lse: [B,H_q].  Returns 0 on success, -1 on bad arguments. */
int oracle_decode_f64(const double *q, const double *k_pool,
                      const double *v_pool, const int32_t *page_table,
                      const int32_t *kv_lens, double *o, double *lse, long B,
                      long H_q, long H_kv, long D, long page_size,
                      long max_pages, double scale, int n_threads) {
    if (B < 0 || H_q <= 0 || H_kv <= 0 || D <= 0 || page_size <= 0) return -1;
    if (H_q % H_kv != 0) return -1;
    if (page_table == NULL) max_pages = 1;
    if (max_pages <= 0) return -1;
    for (long b = 0; b < B; ++b)
        if (kv_lens[b] < 0 || kv_lens[b] > max_pages * page_size) return -1;
    if (B == 0) return 0;
    decode_job J = {q, k_pool, v_pool, page_table, kv_lens, o, lse,
                    B, H_q, H_kv, D, page_size, max_pages, scale, 0};
    return run_threads(decode_worker, &J, n_threads);
}

/* ----------------------------------------------------------------- extend */

typedef struct {
    const double *q, *k_pool, *v_pool;
    const int32_t *page_table, *kv_lens;
    double *o, *lse;
    long B, S_q, H_q, H_kv, D, page_size, max_pages;
    int causal;
    double scale;
    long next_row; /* shared work counter over (b, h) */
} extend_job;

static void *extend_worker(void *arg) {
    extend_job *J = (extend_job *)arg;
    const long D = J->D;
    const long cap = J->max_pages * J->page_size;
    double *k_seq = (double *)malloc(sizeof(double) * (size_t)(cap * D + 1));
    double *v_seq = (double *)malloc(sizeof(double) * (size_t)(cap * D + 1));
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)(cap + 1));
    if (!k_seq || !v_seq || !s_buf) {
        free(k_seq); free(v_seq); free(s_buf);
        return (void *)1;
    }
    const long group = J->H_q / J->H_kv;
    const long total = J->B * J->H_q;
    for (;;) {
        long r = __atomic_fetch_add(&J->next_row, 1, __ATOMIC_RELAXED);
        if (r >= total) break;
        const long b = r / J->H_q, h = r % J->H_q, kvh = h / group;
        const long kv_len = J->kv_lens[b];
        gather_sequence(J->k_pool, J->v_pool, J->page_table, J->max_pages,
                        J->page_size, J->H_kv, D, b, kvh, kv_len, k_seq, v_seq);
        for (long i = 0; i < J->S_q; ++i) {
            /* q and o are [B, S_q, H_q, D]; lse is [B, H_q, S_q] */
            const double *q_row = J->q + (size_t)(((b * J->S_q + i) * J->H_q + h) * D);
            double *o_row = J->o + (size_t)(((b * J->S_q + i) * J->H_q + h) * D);
            double *lse_out = J->lse + (size_t)((b * J->H_q + h) * J->S_q + i);
            long last = kv_len - 1;
            if (J->causal) {
                long lim = i + (kv_len - J->S_q);
                if (lim < last) last = lim;
            }
            if (last < 0) {
                for (long d = 0; d < D; ++d) o_row[d] = 0.0;
                *lse_out = -INFINITY;
                continue;
            }
            double m = -INFINITY;
            for (long j = 0; j <= last; ++j) {
                double dot = 0.0;
                for (long d = 0; d < D; ++d) dot += q_row[d] * k_seq[j * D + d];
                s_buf[j] = J->scale * dot;
                if (s_buf[j] > m) m = s_buf[j];
            }
            double l = 0.0;
            for (long d = 0; d < D; ++d) o_row[d] = 0.0;
            for (long j = 0; j <= last; ++j) {
                double w = exp(s_buf[j] - m);
                l += w;
                for (long d = 0; d < D; ++d) o_row[d] += w * v_seq[j * D + d];
            }
            for (long d = 0; d < D; ++d) o_row[d] /= l;
            *lse_out = m + log(l);
        }
    }
    free(k_seq);
    free(v_seq);
    free(s_buf);
    return NULL;
}

/* q: [B,S_q,H_q,D]; k_pool, v_pool: [num_pages, page_size, H_kv, D];
 * page_table: [B, max_pages] int32; kv_lens: [B] int32; o: [B,S_q,H_q,D];
 * lse: [B,H_q,S_q].  Returns 0 on success, -1 on bad arguments. */
int oracle_extend_f64(const double *q, const double *k_pool, const double *v_pool,
                      const int32_t *page_table, const int32_t *kv_lens, double *o,
                      double *lse, long B, long S_q, long H_q, long H_kv, long D,
                      long page_size, long max_pages, int causal, double scale,
                      int n_threads) {
    if (B < 0 || S_q < 0 || H_q <= 0 || H_kv <= 0 || D <= 0 || page_size <= 0 || max_pages <= 0)
        return -1;
    if (H_q % H_kv != 0 || page_table == NULL) return -1;
    for (long b = 0; b < B; ++b)
        if (kv_lens[b] < 0 || kv_lens[b] > max_pages * page_size) return -1;
    if (B == 0 || S_q == 0) return 0;
    extend_job J = {q, k_pool, v_pool, page_table, kv_lens, o, lse, B, S_q, H_q, H_kv, D,
                    page_size, max_pages, causal, scale, 0};
    return run_threads(extend_worker, &J, n_threads);
}

/* ------------------------------------------------------------------- e4m3 */

/* Decode n E4M3 codes to float64 (exact: every E4M3 value is a double). */
void oracle_e4m3_decode(const uint8_t *in, double *out, long n) {
    for (long i = 0; i < n; ++i) {
        const unsigned c = in[i];
        const int sign = (c >> 7) & 1;
        const int e = (c >> 3) & 0xF;
        const int m = c & 0x7;
        double v;
        if (e == 0xF && m == 0x7)
            v = NAN;
        else if (e == 0)
            v = ldexp((double)m / 8.0, -6);
        else
            v = ldexp(1.0 + (double)m / 8.0, e - 7);
        out[i] = sign ? -v : v;
    }
}

/* --------------------------------------------------------------- backward */

typedef struct {
    const double *q, *k, *v, *dout;
    double *dq, *dk, *dv;
    long B, H, S_q, S_kv, D;
    int layout, causal;
    double scale;
    long next_head; /* shared work counter over (b, h) */
} bwd_job;

static void *bwd_worker(void *arg) {
    bwd_job *J = (bwd_job *)arg;
    const long D = J->D, S_kv = J->S_kv;
    double *p = (double *)malloc(sizeof(double) * (size_t)(S_kv + 1));
    double *o = (double *)malloc(sizeof(double) * (size_t)(D + 1));
    if (!p || !o) { free(p); free(o); return (void *)1; }
    const long total = J->B * J->H;
    for (;;) {
        long r = __atomic_fetch_add(&J->next_head, 1, __ATOMIC_RELAXED);
        if (r >= total) break;
        const long b = r / J->H, h = r % J->H;
        /* this head's dK and dV start at zero; dQ rows are written whole */
        for (long j = 0; j < S_kv; ++j)
            for (long d = 0; d < D; ++d) {
                J->dk[offset4(J->layout, b, h, j, d, J->H, S_kv, D)] = 0.0;
                J->dv[offset4(J->layout, b, h, j, d, J->H, S_kv, D)] = 0.0;
            }
        for (long i = 0; i < J->S_q; ++i) {
            const double *q_row = J->q + offset4(J->layout, b, h, i, 0, J->H, J->S_q, D);
            const double *do_row = J->dout + offset4(J->layout, b, h, i, 0, J->H, J->S_q, D);
            double *dq_row = J->dq + offset4(J->layout, b, h, i, 0, J->H, J->S_q, D);
            for (long d = 0; d < D; ++d) dq_row[d] = 0.0;
            long last = S_kv - 1;
            if (J->causal) {
                long lim = i + (S_kv - J->S_q);
                if (lim < last) last = lim;
            }
            if (last < 0) continue; /* no visible key: O_i = 0, no gradient */
            /* P_i by the definition */
            double m = -INFINITY;
            for (long j = 0; j <= last; ++j) {
                const double *k_row = J->k + offset4(J->layout, b, h, j, 0, J->H, S_kv, D);
                double dot = 0.0;
                for (long d = 0; d < D; ++d) dot += q_row[d] * k_row[d];
                p[j] = J->scale * dot;
                if (p[j] > m) m = p[j];
            }
            double l = 0.0;
            for (long j = 0; j <= last; ++j) { p[j] = exp(p[j] - m); l += p[j]; }
            for (long j = 0; j <= last; ++j) p[j] /= l;
            /* O_i and D_i */
            for (long d = 0; d < D; ++d) o[d] = 0.0;
            for (long j = 0; j <= last; ++j) {
                const double *v_row = J->v + offset4(J->layout, b, h, j, 0, J->H, S_kv, D);
                for (long d = 0; d < D; ++d) o[d] += p[j] * v_row[d];
            }
            double Di = 0.0;
            for (long d = 0; d < D; ++d) Di += do_row[d] * o[d];
            for (long j = 0; j <= last; ++j) {
                const double *k_row = J->k + offset4(J->layout, b, h, j, 0, J->H, S_kv, D);
                const double *v_row = J->v + offset4(J->layout, b, h, j, 0, J->H, S_kv, D);
                double *dk_row = J->dk + offset4(J->layout, b, h, j, 0, J->H, S_kv, D);
                double *dv_row = J->dv + offset4(J->layout, b, h, j, 0, J->H, S_kv, D);
                double dp = 0.0;
                for (long d = 0; d < D; ++d) dp += do_row[d] * v_row[d];
                const double ds = p[j] * (dp - Di);
                for (long d = 0; d < D; ++d) {
                    dv_row[d] += p[j] * do_row[d];
                    dq_row[d] += J->scale * ds * k_row[d];
                    dk_row[d] += J->scale * ds * q_row[d];
                }
            }
        }
    }
    free(p);
    free(o);
    return NULL;
}

/* Gradients of O = softmax(scale Q K^T + mask) V for the upstream gradient
 * dout (q's shape).  q, dout, dq: [B,H,S_q,D] or [B,S_q,H,D]; k, v, dk, dv:
 * the same layout with S_kv.  Returns 0, or -1 on bad arguments. */
int oracle_prefill_bwd_f64(const double *q, const double *k, const double *v,
                           const double *dout, double *dq, double *dk, double *dv,
                           long B, long H, long S_q, long S_kv, long D, int layout,
                           int causal, double scale, int n_threads) {
    if (B < 0 || H < 0 || S_q < 0 || S_kv < 0 || D <= 0) return -1;
    if (layout != ORACLE_BHSD && layout != ORACLE_BSHD) return -1;
    if (B == 0 || H == 0) return 0;
    bwd_job J = {q, k, v, dout, dq, dk, dv, B, H, S_q, S_kv, D, layout, causal, scale, 0};
    return run_threads(bwd_worker, &J, n_threads);
}

/* ------------------------------------------------------------- MQA logits */

typedef struct {
    const double *q, *kv, *kv_scale, *w;
    const int32_t *start, *end;
    double *logits;
    long S_q, S_kv, H, D, stride;
    int clean;
    long next_row;
} mqa_job;

static void *mqa_worker(void *arg) {
    mqa_job *J = (mqa_job *)arg;
    for (;;) {
        long i = __atomic_fetch_add(&J->next_row, 1, __ATOMIC_RELAXED);
        if (i >= J->S_q) break;
        long lo = J->start[i] < 0 ? 0 : J->start[i];
        long hi = J->end[i] > J->S_kv ? J->S_kv : J->end[i];
        double *row = J->logits + i * J->stride;
        for (long j = 0; j < J->S_kv; ++j) {
            if (j < lo || j >= hi) {
                if (J->clean) row[j] = -INFINITY;
                continue;
            }
            double acc = 0.0;
            for (long h = 0; h < J->H; ++h) {
                const double *q_row = J->q + (i * J->H + h) * J->D;
                double dot = 0.0;
                for (long d = 0; d < J->D; ++d) dot += q_row[d] * J->kv[j * J->D + d];
                const double s = J->kv_scale[j] * dot;
                acc += J->w[i * J->H + h] * (s > 0.0 ? s : 0.0);
            }
            row[j] = acc;
        }
    }
    return NULL;
}

/* q: [S_q, H, D]; kv: [S_kv, D]; kv_scale: [S_kv]; w: [S_q, H]; start, end:
 * [S_q] int32; logits: [S_q, stride] (stride >= S_kv), written as above.
 * Returns 0, or -1 on bad arguments. */
int oracle_mqa_logits_f64(const double *q, const double *kv, const double *kv_scale,
                          const double *w, const int32_t *start, const int32_t *end,
                          double *logits, long S_q, long S_kv, long H, long D, long stride,
                          int clean, int n_threads) {
    if (S_q < 0 || S_kv < 0 || H <= 0 || D <= 0 || stride < S_kv) return -1;
    if (S_q == 0) return 0;
    mqa_job J = {q, kv, kv_scale, w, start, end, logits, S_q, S_kv, H, D, stride, clean, 0};
    return run_threads(mqa_worker, &J, n_threads);
}
