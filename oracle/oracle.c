/*
 * oracle.c -- fp64 CPU oracle for paged, GQA-shared decode attention.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Plain loops, double precision,
 * no blocking, no online softmax, no splitting.  Threads only partition the
 * independent (b, hq) pairs; each pair is computed by one thread in token
 * order.
 *
 * Passages followed (page title, section):
 *  - "FlashDecoding 与 FlashInfer 深度解析", §2.1 step 2 (score = q k^T / sqrt(d),
 *    softmax, weighted sum of V, local max and sum).
 *  - lpnh.cn "FlashDecoding 核心原理", stage one (partial state: unnormalised
 *    output, local max m_i, denominator d_i) and the stage-two formula
 *    (m_global = max m_i, alpha_i = exp(m_i - m_global), d_global =
 *    sum alpha_i d_i, O = sum alpha_i O_i / d_global), evaluated here through
 *    its log-sum-exp: lse = m_global + ln d_global, and the weight of piece i
 *    alpha_i / d_global = exp(m_i - lse).
 *  - "Inference Cookbook" (FlashAttention), §4.2: paged pools
 *    [num_pages, page_size, Hkv, D] and a block table whose unused entries
 *    are -1; §3.5: softmax_lse per (batch, head); §7: FP8 KV with per-head
 *    descale factors (applied here per page and KV head).
 *  - GQA head mapping: query head hq reads KV head hq / (Hq / Hkv)
 *    (contiguous groups; the pages give only the head counts).
 */
#define _GNU_SOURCE
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---------------------------------------------------------------- decoders */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
double orc_f16_to_double(uint16_t bits) {
    int s = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1f;
    int m = bits & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24   */
    else if (e == 31)
        v = (m == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* 1.m * 2^(e-15)         */
    return s ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits. */
double orc_bf16_to_double(uint16_t bits) {
    int s = (bits >> 15) & 1;
    int e = (bits >> 7) & 0xff;
    int m = bits & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133);                /* m/128 * 2^-126         */
    else if (e == 255)
        v = (m == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(128 + m), e - 134);     /* 1.m * 2^(e-127)        */
    return s ? -v : v;
}

/* OCP FP8 E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities;
 * S.1111.111 is NaN; largest finite magnitude 448. */
double orc_e4m3_to_double(uint8_t bits) {
    int s = (bits >> 7) & 1;
    int e = (bits >> 3) & 0xf;
    int m = bits & 0x7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);                  /* m/8 * 2^-6             */
    else
        v = ldexp((double)(8 + m), e - 10);        /* 1.m * 2^(e-7)          */
    return s ? -v : v;
}

/* Nearest finite E4M3 magnitude by exhaustive search over the 127 finite
 * non-negative codes; a tie goes to the code whose mantissa LSB is 0. */
uint8_t orc_e4m3_from_float(float x) {
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return (uint8_t)(sign | 0x7f);
    double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7e);
    int best = 0;
    double best_diff = INFINITY;
    for (int code = 0; code <= 0x7e; ++code) {
        double diff = fabs(a - orc_e4m3_to_double((uint8_t)code));
        if (diff < best_diff || (diff == best_diff && (code & 1) == 0)) {
            best = code;
            best_diff = diff;
        }
    }
    return (uint8_t)(sign | best);
}

static double load_elem(const void *base, int dtype, size_t idx) {
    switch (dtype) {
    case ORC_F16:  return orc_f16_to_double(((const uint16_t *)base)[idx]);
    case ORC_BF16: return orc_bf16_to_double(((const uint16_t *)base)[idx]);
    case ORC_E4M3: return orc_e4m3_to_double(((const uint8_t *)base)[idx]);
    case ORC_F32:  return (double)((const float *)base)[idx];
    default:       return NAN;
    }
}

static int valid_dtype(int t) { return t == ORC_F16 || t == ORC_BF16 || t == ORC_E4M3 || t == ORC_F32; }

static int check_problem(const orc_problem *p) {
    if (!p || p->B < 0 || p->Hq <= 0 || p->Hkv <= 0 || p->D <= 0 || p->page_size <= 0 ||
        p->max_blocks_per_seq < 0 || p->num_pages < 0)
        return ORC_ERR_ARG;
    if (p->Hq % p->Hkv != 0) return ORC_ERR_ARG;
    if (!valid_dtype(p->q_dtype) || !valid_dtype(p->kv_dtype) || p->q_dtype == ORC_E4M3)
        return ORC_ERR_ARG;
    return ORC_OK;
}

/* ------------------------------------------------------------ paged gather */

/* Token t of sequence b lives at page block_table[b][t / page_size], slot
 * t % page_size; its K (or V) row for KV head kvh starts at element
 * ((page * page_size + slot) * Hkv + kvh) * D of the pool.  For E4M3 the
 * decoded value is multiplied by the (page, kvh) scale. */
static int gather_row(const orc_problem *p, const void *pages, const float *scale,
                      const int32_t *block_table, int b, int kvh, int t, double *row) {
    int page = block_table[(size_t)b * p->max_blocks_per_seq + t / p->page_size];
    if (page < 0 || page >= p->num_pages) return ORC_ERR_BAD_PAGE;
    int slot = t % p->page_size;
    size_t base = (((size_t)page * p->page_size + slot) * p->Hkv + kvh) * (size_t)p->D;
    double sc = 1.0;
    if (p->kv_dtype == ORC_E4M3) sc = (double)scale[(size_t)page * p->Hkv + kvh];
    for (int d = 0; d < p->D; ++d) row[d] = load_elem(pages, p->kv_dtype, base + d) * sc;
    return ORC_OK;
}

/* --------------------------------------------------------- one (b, hq) pair */

typedef struct {
    const orc_problem *p;
    const void *q, *k, *v;
    const float *ks, *vs;
    const int32_t *bt;
    /* contiguous layout instead of pages when k_contig != NULL */
    const void *k_contig, *v_contig;
    int max_seqlen;
} orc_inputs;

static int row_of(const orc_inputs *in, int which_v, int b, int kvh, int t, double *row) {
    const orc_problem *p = in->p;
    if (in->k_contig) {
        const void *base = which_v ? in->v_contig : in->k_contig;
        size_t off = (((size_t)b * in->max_seqlen + t) * p->Hkv + kvh) * (size_t)p->D;
        for (int d = 0; d < p->D; ++d) row[d] = load_elem(base, p->kv_dtype, off + d);
        return ORC_OK;
    }
    return gather_row(p, which_v ? in->v : in->k, which_v ? in->vs : in->ks, in->bt, b, kvh, t, row);
}

/* Scores s_t = (q . k_t) / sqrt(D) for t in [t0, t1), written to s[t - t0]. */
static int scores(const orc_inputs *in, int b, int hq, int t0, int t1, double *s, double *qrow,
                  double *krow) {
    const orc_problem *p = in->p;
    int kvh = hq / (p->Hq / p->Hkv);
    size_t qoff = ((size_t)b * p->Hq + hq) * (size_t)p->D;
    for (int d = 0; d < p->D; ++d) qrow[d] = load_elem(in->q, p->q_dtype, qoff + d);
    double inv_sqrt_d = 1.0 / sqrt((double)p->D);
    for (int t = t0; t < t1; ++t) {
        int rc = row_of(in, 0, b, kvh, t, krow);
        if (rc) return rc;
        double dot = 0.0;
        for (int d = 0; d < p->D; ++d) dot += qrow[d] * krow[d];
        s[t - t0] = dot * inv_sqrt_d;
    }
    return ORC_OK;
}

/* Unnormalised partial state over [t0, t1): o, m, d (stage one of the pages). */
static int partial(const orc_inputs *in, int b, int hq, int t0, int t1, double *o, double *m,
                   double *dsum) {
    const orc_problem *p = in->p;
    int D = p->D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    *m = -INFINITY;
    *dsum = 0.0;
    if (t1 <= t0) return ORC_OK;
    int n = t1 - t0;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double *qrow = (double *)malloc(sizeof(double) * (size_t)D);
    double *row = (double *)malloc(sizeof(double) * (size_t)D);
    int rc = ORC_ERR_NOMEM;
    if (s && qrow && row) {
        rc = scores(in, b, hq, t0, t1, s, qrow, row);
        if (rc == ORC_OK) {
            double mx = -INFINITY;
            for (int i = 0; i < n; ++i) if (s[i] > mx) mx = s[i];
            int kvh = hq / (p->Hq / p->Hkv);
            double z = 0.0;
            for (int i = 0; i < n; ++i) {
                double w = exp(s[i] - mx);
                z += w;
                rc = row_of(in, 1, b, kvh, t0 + i, row);
                if (rc) break;
                for (int d = 0; d < D; ++d) o[d] += w * row[d];
            }
            *m = mx;
            *dsum = z;
        }
    }
    free(s);
    free(qrow);
    free(row);
    return rc;
}

/* Normalised output and log-sum-exp over all tokens of sequence b. */
static int attend(const orc_inputs *in, const int32_t *seq_lens, int b, int hq, double *out,
                  double *lse) {
    int D = in->p->D;
    int L = seq_lens[b];
    if (L < 0) return ORC_ERR_ARG;
    double m, z;
    int rc = partial(in, b, hq, 0, L, out, &m, &z);
    if (rc) return rc;
    if (L == 0) {
        *lse = -INFINITY;
        return ORC_OK;
    }
    for (int d = 0; d < D; ++d) out[d] /= z;
    *lse = m + log(z);
    return ORC_OK;
}

/* ----------------------------------------------------------------- threads */

typedef struct {
    const orc_inputs *in;
    const int32_t *seq_lens;
    const int32_t *pairs; /* NULL: all (b, hq) in order */
    int npairs;
    double *out, *lse;
    int tid, nthreads;
    int rc;
} orc_job;

static void *worker(void *arg) {
    orc_job *j = (orc_job *)arg;
    int D = j->in->p->D, Hq = j->in->p->Hq;
    j->rc = ORC_OK;
    for (int i = j->tid; i < j->npairs; i += j->nthreads) {
        int b = j->pairs ? j->pairs[2 * i] : i / Hq;
        int hq = j->pairs ? j->pairs[2 * i + 1] : i % Hq;
        int rc = attend(j->in, j->seq_lens, b, hq, j->out + (size_t)i * D, j->lse + i);
        if (rc && !j->rc) j->rc = rc;
    }
    return NULL;
}

static int run_threads(const orc_inputs *in, const int32_t *seq_lens, const int32_t *pairs,
                       int npairs, double *out, double *lse, int nthreads) {
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > npairs) nthreads = npairs > 0 ? npairs : 1;
    orc_job *jobs = (orc_job *)calloc((size_t)nthreads, sizeof(orc_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return ORC_ERR_NOMEM;
    }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (orc_job){in, seq_lens, pairs, npairs, out, lse, t, nthreads, ORC_OK};
        if (t > 0) pthread_create(&th[t], NULL, worker, &jobs[t]);
    }
    worker(&jobs[0]);
    int rc = jobs[0].rc;
    for (int t = 1; t < nthreads; ++t) {
        pthread_join(th[t], NULL);
        if (jobs[t].rc && !rc) rc = jobs[t].rc;
    }
    free(jobs);
    free(th);
    return rc;
}

/* -------------------------------------------------------------- public API */

int orc_decode_paged(const orc_problem *p, const void *q, const void *k_pages,
                     const void *v_pages, const float *k_scale, const float *v_scale,
                     const int32_t *block_table, const int32_t *seq_lens,
                     double *out, double *lse, int nthreads) {
    if (check_problem(p)) return ORC_ERR_ARG;
    if (p->kv_dtype == ORC_E4M3 && (!k_scale || !v_scale)) return ORC_ERR_ARG;
    orc_inputs in = {p, q, k_pages, v_pages, k_scale, v_scale, block_table, NULL, NULL, 0};
    return run_threads(&in, seq_lens, NULL, p->B * p->Hq, out, lse, nthreads);
}

int orc_decode_paged_pairs(const orc_problem *p, const void *q, const void *k_pages,
                           const void *v_pages, const float *k_scale, const float *v_scale,
                           const int32_t *block_table, const int32_t *seq_lens,
                           const int32_t *pairs, int npairs,
                           double *out, double *lse, int nthreads) {
    if (check_problem(p)) return ORC_ERR_ARG;
    if (p->kv_dtype == ORC_E4M3 && (!k_scale || !v_scale)) return ORC_ERR_ARG;
    for (int i = 0; i < npairs; ++i)
        if (pairs[2 * i] < 0 || pairs[2 * i] >= p->B || pairs[2 * i + 1] < 0 ||
            pairs[2 * i + 1] >= p->Hq)
            return ORC_ERR_ARG;
    orc_inputs in = {p, q, k_pages, v_pages, k_scale, v_scale, block_table, NULL, NULL, 0};
    return run_threads(&in, seq_lens, pairs, npairs, out, lse, nthreads);
}

/* Cookbook §5.2-5.3: indirection to a cache row and a left offset.  The
 * gather of each token is the paged gather above, for the cache row's block
 * table; the softmax is the same definition over the attended range. */
int orc_decode_paged_ex(const orc_problem *p, int cache_rows, const int32_t *cache_batch_idx,
                        const int32_t *cache_leftpad, const void *q, const void *k_pages,
                        const void *v_pages, const float *k_scale, const float *v_scale,
                        const int32_t *block_table, const int32_t *seq_lens,
                        double *out, double *lse) {
    if (check_problem(p) || cache_rows < 1) return ORC_ERR_ARG;
    if (p->kv_dtype == ORC_E4M3 && (!k_scale || !v_scale)) return ORC_ERR_ARG;
    orc_problem pc = *p;
    pc.B = cache_rows;
    for (int b = 0; b < p->B; ++b) {
        int cb = cache_batch_idx ? cache_batch_idx[b] : b;
        if (cb < 0 || cb >= cache_rows) return ORC_ERR_ARG;
        int L = seq_lens[cb];
        int lp = cache_leftpad ? cache_leftpad[cb] : 0;
        if (lp < 0 || lp > L) return ORC_ERR_ARG;
        for (int hq = 0; hq < p->Hq; ++hq) {
            /* q row b of the caller, keys/values of cache row cb */
            const int D = p->D;
            double *o = out + ((size_t)b * p->Hq + hq) * D;
            orc_inputs in = {&pc, NULL, k_pages, v_pages, k_scale, v_scale, block_table, NULL, NULL, 0};
            /* a q buffer view holding only row b at index cb */
            size_t esz = p->q_dtype == ORC_F32 ? 4 : 2;
            void *qv = calloc((size_t)cache_rows * p->Hq * D, esz);
            if (!qv) return ORC_ERR_NOMEM;
            memcpy((char *)qv + ((size_t)cb * p->Hq + hq) * D * esz,
                   (const char *)q + ((size_t)b * p->Hq + hq) * D * esz, D * esz);
            in.q = qv;
            double m, z;
            int rc = partial(&in, cb, hq, lp, L, o, &m, &z);
            free(qv);
            if (rc) return rc;
            if (L - lp == 0) {
                lse[(size_t)b * p->Hq + hq] = -INFINITY;
                continue;
            }
            for (int d = 0; d < D; ++d) o[d] /= z;
            lse[(size_t)b * p->Hq + hq] = m + log(z);
        }
    }
    return ORC_OK;
}

/* Query token i of q_len (causal, aligned to the end of the cache): its
 * scores over the tokens it may see, their maximum, the exponentials, the
 * weighted sum of V and its normalisation -- the definition, written out for
 * one (b, i, hq) with the query row given explicitly. */
static int attend_causal(const orc_inputs *in, int b, int hq, const double *qrow, int t_end, double *out,
                         double *lse) {
    const orc_problem *p = in->p;
    const int D = p->D, kvh = hq / (p->Hq / p->Hkv);
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (t_end <= 0) {
        *lse = -INFINITY;
        return ORC_OK;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)t_end);
    double *row = (double *)malloc(sizeof(double) * (size_t)D);
    int rc = (s && row) ? ORC_OK : ORC_ERR_NOMEM;
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
    for (int t = 0; t < t_end && rc == ORC_OK; ++t) {
        rc = row_of(in, 0, b, kvh, t, row);
        if (rc) break;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qrow[d] * row[d];
        s[t] = dot * inv_sqrt_d;
    }
    if (rc == ORC_OK) {
        double mx = -INFINITY;
        for (int t = 0; t < t_end; ++t) if (s[t] > mx) mx = s[t];
        double z = 0.0;
        for (int t = 0; t < t_end && rc == ORC_OK; ++t) {
            const double w = exp(s[t] - mx);
            z += w;
            rc = row_of(in, 1, b, kvh, t, row);
            if (rc) break;
            for (int d = 0; d < D; ++d) out[d] += w * row[d];
        }
        if (rc == ORC_OK) {
            for (int d = 0; d < D; ++d) out[d] /= z;
            *lse = mx + log(z);
        }
    }
    free(s);
    free(row);
    return rc;
}

int orc_decode_paged_multi(const orc_problem *p, int q_len, const void *q, const void *k_pages,
                           const void *v_pages, const float *k_scale, const float *v_scale,
                           const int32_t *block_table, const int32_t *seq_lens,
                           double *out, double *lse) {
    if (check_problem(p) || q_len < 1) return ORC_ERR_ARG;
    if (p->kv_dtype == ORC_E4M3 && (!k_scale || !v_scale)) return ORC_ERR_ARG;
    const int D = p->D;
    double *qrow = (double *)malloc(sizeof(double) * (size_t)D);
    if (!qrow) return ORC_ERR_NOMEM;
    orc_inputs in = {p, NULL, k_pages, v_pages, k_scale, v_scale, block_table, NULL, NULL, 0};
    int rc = ORC_OK;
    for (int b = 0; b < p->B && rc == ORC_OK; ++b) {
        const int L = seq_lens[b];
        if (L < q_len) { rc = ORC_ERR_ARG; break; }
        for (int i = 0; i < q_len && rc == ORC_OK; ++i) {
            for (int hq = 0; hq < p->Hq && rc == ORC_OK; ++hq) {
                const size_t r = ((size_t)b * q_len + i) * p->Hq + hq;  /* [B, q_len, Hq] */
                for (int d = 0; d < D; ++d) qrow[d] = load_elem(q, p->q_dtype, r * D + d);
                rc = attend_causal(&in, b, hq, qrow, L - q_len + i + 1, out + r * D, lse + r);
            }
        }
    }
    free(qrow);
    return rc;
}

int orc_decode_contiguous(const orc_problem *p, int max_seqlen, const void *q,
                          const void *k_cache, const void *v_cache,
                          const int32_t *seq_lens, double *out, double *lse) {
    if (check_problem(p) || p->kv_dtype == ORC_E4M3) return ORC_ERR_ARG;
    for (int b = 0; b < p->B; ++b)
        if (seq_lens[b] > max_seqlen) return ORC_ERR_ARG;
    orc_inputs in = {p, q, NULL, NULL, NULL, NULL, NULL, k_cache, v_cache, max_seqlen};
    return run_threads(&in, seq_lens, NULL, p->B * p->Hq, out, lse, 1);
}

int orc_partial_state(const orc_problem *p, const void *q, const void *k_pages,
                      const void *v_pages, const float *k_scale, const float *v_scale,
                      const int32_t *block_table, int b, int hq, int t_begin, int t_end,
                      double *o, double *m, double *d) {
    if (check_problem(p) || b < 0 || b >= p->B || hq < 0 || hq >= p->Hq || t_begin < 0)
        return ORC_ERR_ARG;
    if (p->kv_dtype == ORC_E4M3 && (!k_scale || !v_scale)) return ORC_ERR_ARG;
    orc_inputs in = {p, q, k_pages, v_pages, k_scale, v_scale, block_table, NULL, NULL, 0};
    return partial(&in, b, hq, t_begin, t_end, o, m, d);
}

/* Stage two of lpnh.cn "FlashDecoding 核心原理": the merged log-sum-exp is
 * lse = m_g + ln(sum_i exp(m_i - m_g) d_i) with m_g = max_i m_i; each piece
 * then enters the output with the weight exp(m_i - lse) (its alpha_i divided
 * by the merged denominator), out = sum_i exp(m_i - lse) o_i.  Empty pieces
 * (m = -inf) have weight 0; all empty gives out = 0, lse = -inf. */
void orc_merge_states(int n, int D, const double *o, const double *m, const double *d,
                      double *out, double *lse) {
    for (int k = 0; k < D; ++k) out[k] = 0.0;
    double mg = -INFINITY;
    for (int i = 0; i < n; ++i) if (m[i] > mg) mg = m[i];
    if (mg == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double z = 0.0;
    for (int i = 0; i < n; ++i)
        if (m[i] != -INFINITY) z += exp(m[i] - mg) * d[i];
    const double l = mg + log(z);
    for (int i = 0; i < n; ++i) {
        if (m[i] == -INFINITY) continue;
        const double w = exp(m[i] - l);
        for (int k = 0; k < D; ++k) out[k] += w * o[(size_t)i * D + k];
    }
    *lse = l;
}

int orc_append_kv(const orc_problem *p, int new_dtype, const void *k_new, const void *v_new,
                  void *k_pages, void *v_pages, const float *k_scale, const float *v_scale,
                  const int32_t *block_table, const int32_t *seq_lens) {
    if (check_problem(p)) return ORC_ERR_ARG;
    int fp8 = p->kv_dtype == ORC_E4M3;
    if (fp8) {
        if (!k_scale || !v_scale) return ORC_ERR_ARG;
        if (new_dtype != ORC_F16 && new_dtype != ORC_BF16 && new_dtype != ORC_F32) return ORC_ERR_ARG;
    } else if (new_dtype != p->kv_dtype) {
        return ORC_ERR_ARG;
    }
    size_t esz = fp8 ? 1 : (p->kv_dtype == ORC_F32 ? 4 : 2);
    for (int b = 0; b < p->B; ++b) {
        int L = seq_lens[b];
        if (L < 0 || L / p->page_size >= p->max_blocks_per_seq) return ORC_ERR_BAD_PAGE;
        int page = block_table[(size_t)b * p->max_blocks_per_seq + L / p->page_size];
        if (page < 0 || page >= p->num_pages) return ORC_ERR_BAD_PAGE;
        int slot = L % p->page_size;
        for (int kvh = 0; kvh < p->Hkv; ++kvh) {
            size_t src = ((size_t)b * p->Hkv + kvh) * (size_t)p->D;
            size_t dst = (((size_t)page * p->page_size + slot) * p->Hkv + kvh) * (size_t)p->D;
            for (int which = 0; which < 2; ++which) {
                const void *in = which ? v_new : k_new;
                void *pool = which ? v_pages : k_pages;
                if (!fp8) {
                    memcpy((char *)pool + (dst * esz), (const char *)in + (src * esz), esz * (size_t)p->D);
                    continue;
                }
                float sc = (which ? v_scale : k_scale)[(size_t)page * p->Hkv + kvh];
                for (int d = 0; d < p->D; ++d) {
                    float x = (float)load_elem(in, new_dtype, src + d); /* exact */
                    float y = x / sc;                                   /* IEEE fp32 */
                    ((uint8_t *)pool)[dst + d] = orc_e4m3_from_float(y);
                }
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------- rotary */

void orc_rotary_f32(const float *x, int n, int rotary_dim, int interleaved, const float *cos_tab,
                    const float *sin_tab, int pos, float *y) {
    for (int d = 0; d < n; ++d) y[d] = x[d];
    int half = rotary_dim / 2;
    for (int i = 0; i < half; ++i) {
        int a = interleaved ? 2 * i : i;
        int b = interleaved ? 2 * i + 1 : i + half;
        float c = cos_tab[(size_t)pos * half + i];
        float s = sin_tab[(size_t)pos * half + i];
        float x1 = x[a], x2 = x[b];
        float p1 = x1 * c, p2 = x2 * s, p3 = x2 * c, p4 = x1 * s;
        y[a] = p1 - p2;
        y[b] = p3 + p4;
    }
}

/* Round-to-nearest-even of a finite or non-finite float to bfloat16 / f16
 * bits, from the formats' definitions (exhaustive search is not needed:
 * the conversions are exact rounding of the binary32 significand). */
static uint16_t to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40); /* NaN stays NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;                                                      /* ties to even */
    return (uint16_t)(u >> 16);
}

static uint16_t to_f16_bits(float f) {
    /* nearest representable binary16 by search over the neighbours of the
     * double-precision value: decode candidates and pick the closest, ties
     * to the even code. */
    if (isnan(f)) return 0x7e00;
    double v = (double)f;
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    double a = fabs(v);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);  /* rounds to infinity */
    int best = 0;
    double best_diff = INFINITY;
    for (int code = 0; code < 0x7c00; ++code) {
        double diff = fabs(a - orc_f16_to_double((uint16_t)code));
        if (diff < best_diff || (diff == best_diff && (code & 1) == 0)) {
            best = code;
            best_diff = diff;
        }
        if (orc_f16_to_double((uint16_t)code) > a && diff > best_diff) break;
    }
    return (uint16_t)(sign | best);
}

static void store_16(void *base, int dtype, size_t idx, float v) {
    ((uint16_t *)base)[idx] = dtype == ORC_BF16 ? to_bf16_bits(v) : to_f16_bits(v);
}

int orc_append_kv_rotary(const orc_problem *p, int new_dtype, const void *k_new, const void *v_new,
                         void *k_pages, void *v_pages, const float *k_scale, const float *v_scale,
                         const int32_t *block_table, const int32_t *seq_lens,
                         const float *cos_tab, const float *sin_tab, int rotary_dim, int max_pos,
                         int interleaved, void *q_inout) {
    if (check_problem(p) || !cos_tab || !sin_tab || rotary_dim < 2 || rotary_dim % 2 || rotary_dim > p->D ||
        max_pos < 1)
        return ORC_ERR_ARG;
    int fp8 = p->kv_dtype == ORC_E4M3;
    if (!fp8 && new_dtype != p->kv_dtype) return ORC_ERR_ARG;
    if (fp8 && ((!k_scale || !v_scale) || (new_dtype != ORC_F16 && new_dtype != ORC_BF16))) return ORC_ERR_ARG;
    if (new_dtype != ORC_F16 && new_dtype != ORC_BF16) return ORC_ERR_ARG;
    int D = p->D;
    float *x = (float *)malloc(sizeof(float) * D), *y = (float *)malloc(sizeof(float) * D);
    if (!x || !y) { free(x); free(y); return ORC_ERR_NOMEM; }
    int rc = ORC_OK;
    for (int b = 0; b < p->B && rc == ORC_OK; ++b) {
        int L = seq_lens[b];
        if (L < 0 || L >= max_pos || L / p->page_size >= p->max_blocks_per_seq) { rc = ORC_ERR_BAD_PAGE; break; }
        int page = block_table[(size_t)b * p->max_blocks_per_seq + L / p->page_size];
        if (page < 0 || page >= p->num_pages) { rc = ORC_ERR_BAD_PAGE; break; }
        int slot = L % p->page_size;
        for (int kvh = 0; kvh < p->Hkv; ++kvh) {
            size_t src = ((size_t)b * p->Hkv + kvh) * D;
            size_t dst = (((size_t)page * p->page_size + slot) * p->Hkv + kvh) * (size_t)D;
            for (int which = 0; which < 2; ++which) {
                const void *in = which ? v_new : k_new;
                void *pool = which ? v_pages : k_pages;
                for (int d = 0; d < D; ++d) x[d] = (float)load_elem(in, new_dtype, src + d);
                if (which == 0) orc_rotary_f32(x, D, rotary_dim, interleaved, cos_tab, sin_tab, L, y);
                else memcpy(y, x, sizeof(float) * D);
                if (!fp8) {
                    for (int d = 0; d < D; ++d) store_16(pool, p->kv_dtype, dst + d, y[d]);
                } else {
                    float sc = (which ? v_scale : k_scale)[(size_t)page * p->Hkv + kvh];
                    for (int d = 0; d < D; ++d) ((uint8_t *)pool)[dst + d] = orc_e4m3_from_float(y[d] / sc);
                }
            }
        }
        if (q_inout) {
            for (int hq = 0; hq < p->Hq; ++hq) {
                size_t off = ((size_t)b * p->Hq + hq) * D;
                for (int d = 0; d < D; ++d) x[d] = (float)load_elem(q_inout, p->q_dtype, off + d);
                orc_rotary_f32(x, D, rotary_dim, interleaved, cos_tab, sin_tab, L, y);
                for (int d = 0; d < D; ++d) store_16(q_inout, p->q_dtype, off + d, y[d]);
            }
        }
    }
    free(x);
    free(y);
    return rc;
}
