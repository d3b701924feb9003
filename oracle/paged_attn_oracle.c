/*
 * paged_attn_oracle.c -- plain, slow, fp64 CPU restatement of paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled by oracle/__init__.py and
 * called from the test-suite, from the smoke check and from the CPU-baseline
 * leg of the benchmark.  The library (paged_kv_attention_20_gb300) never links,
 * imports or executes it, and it shares no code with the CUDA path.
 *
 * What it computes, and where that is stated:
 *
 *  - ruDNN 0.1.7, src/paged_attention/mod.rs, doc comment of
 *    `DevicePlan::attention`: packed Q is [queries, Hq, D]; the key cache is
 *    [pages, page_size, Hkv, D] and the value cache [pages, page_size, Hkv, Dv];
 *    `causal` uses the absolute positions held by the plan, prefill chunks
 *    included.  The result is [queries, Hq, Dv] (`forward`).
 *  - same page, `execute_attention_into`: Hq must be a multiple of Hkv (query
 *    head h reads key/value head h / (Hq/Hkv): contiguous groups, no per-head
 *    repeat of the cache), scale must be finite and > 0.
 *  - same page, doc of `DevicePlan::mla`: absorbed Q [queries, H, R] and
 *    position Q [queries, H, P] score against one shared latent head
 *    [pages, page_size, 1, R] plus a rotated position cache
 *    [pages, page_size, 1, P]; the latent is both key and value
 *    (`forward(q, latent, latent, Some((qp, kp)), ..)`), so
 *    score_j = scale * (q . c_j + qp . kr_j) and out = sum_j softmax_j c_j.
 *  - same page, doc of `attention_into_split`: the visible history is split
 *    over several planes whose FP32 statistics are merged; the unsplit method
 *    is the reference result.
 *  - same page, `append_with_report`: new rows [queries, heads, d|dv] are
 *    written into the caches at the plan's positions.
 *  - libmir-cuda 0.1.0, src/backend/attention/graph/mod.rs, `Geometry`: a
 *    layer's attention carries a `window` next to its head geometry, and the
 *    split configuration is chosen from the token count and that window.
 *  - boostr 0.1.0, src/inference/decode_graph.rs, `DeviceScalars::update`: a
 *    decode step writes its key/value at position seq_len and then attends
 *    over seq_len + 1 keys, i.e. the query at absolute position p sees keys
 *    0..p inclusive once its own row is stored.
 *
 * Readings taken where the pages are silent (each is also listed in the
 * design notes of the repository):
 *  - logical key j of sequence s lives in physical page block_table[s][j/ps],
 *    row j % ps;
 *  - causal: keys 0..pos inclusive; non-causal: keys 0..seq_len-1;
 *  - split partition: n visible keys, chunk = ceil(n / S) rounded up to a
 *    multiple of page_size, split s covers [s*chunk, min((s+1)*chunk, n));
 *    an empty split has lse = -inf and a zero partial output;
 *  - lse is the natural-log log-sum-exp of the scaled scores;
 *  - sliding window W > 0 (the pages name the field but not its meaning): a
 *    query at position p sees only keys j >= p - W + 1, on top of the causal
 *    or non-causal upper end; W = 0 means no window;
 *  - split partition under a window: the visible keys are [lo, hi); with
 *    base = lo rounded down to a page boundary and chunk = ceil((hi - base) / S)
 *    rounded up to a multiple of page_size, split s covers
 *    [max(lo, base + s*chunk), min(base + (s+1)*chunk, hi)) (W = 0 gives the
 *    rule above, since lo = base = 0).
 *
 * All arithmetic is IEEE binary64 in plain loops, one (query, head) row per
 * OpenMP iteration, in key order.  Inputs are read in their storage type
 * (f32, f16 or bf16), decoded exactly to double.
 *
 * PLANT (compile-time, default 0) deliberately breaks one step so the
 * test-suite can show that its pins catch that kind of mistake:
 *   1 causal range drops the query's own key   2 scale applied twice
 *   3 GQA head map h % Hkv instead of h / G    4 MLA position term dropped
 *   5 page row taken as j / ps instead of j % ps
 *   6 window lower end off by one (p - W instead of p - W + 1)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef PLANT
#define PLANT 0
#endif

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };

/* binary16 -> double, from the IEEE 754 field definition. */
static double half_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24);                 /* zero / subnormal */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(mant + 1024), expo - 25);  /* 1.m * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the top half of a binary32. */
static double bf16_bits_to_double(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double load(const void *base, int64_t idx, int dtype) {
    if (dtype == OR_F32) return (double)((const float *)base)[idx];
    if (dtype == OR_BF16) return bf16_bits_to_double(((const uint16_t *)base)[idx]);
    return half_bits_to_double(((const uint16_t *)base)[idx]);
}

typedef struct {
    const void *q, *qp, *k, *v, *kp;   /* kp/qp NULL unless MLA */
    int dtype;
    int64_t queries, hq, hkv, d, dv, p;
    const int32_t *seq_lens;
    int64_t seqs;
    const int32_t *table;
    int64_t width;
    const int32_t *qseq, *qpos;
    int64_t page_size, pages;
    double scale;
    int causal;
    int64_t window;
} problem;

/* Upper end (exclusive) of the keys that query q may see. */
static int64_t visible(const problem *pb, int64_t q) {
    int64_t s = pb->qseq[q];
    if (pb->causal) {
#if PLANT == 1
        return (int64_t)pb->qpos[q];
#else
        return (int64_t)pb->qpos[q] + 1;
#endif
    }
    return pb->seq_lens[s];
}

/* Lower end (inclusive) of the keys that query q may see. */
static int64_t visible_from(const problem *pb, int64_t q) {
    if (pb->window <= 0) return 0;
#if PLANT == 6
    int64_t lo = (int64_t)pb->qpos[q] - pb->window;
#else
    int64_t lo = (int64_t)pb->qpos[q] - pb->window + 1;
#endif
    return lo > 0 ? lo : 0;
}

/* Physical cache row (page * page_size + row-in-page) of logical key j. */
static int64_t cache_row(const problem *pb, int64_t s, int64_t j) {
    int64_t page = pb->table[s * pb->width + j / pb->page_size];
#if PLANT == 5
    return page * pb->page_size + (j / pb->page_size) % pb->page_size;
#else
    return page * pb->page_size + j % pb->page_size;
#endif
}

static int64_t kv_head_of(const problem *pb, int64_t h) {
#if PLANT == 3
    return h % pb->hkv;
#else
    return h / (pb->hq / pb->hkv);
#endif
}

/* scale * (q . k_j  [+ qp . kr_j]) for row (q, h) and logical key j. */
static double score(const problem *pb, int64_t q, int64_t h, int64_t j) {
    int64_t s = pb->qseq[q];
    int64_t kvh = kv_head_of(pb, h);
    int64_t r = cache_row(pb, s, j);
    double acc = 0.0;
    int64_t qbase = (q * pb->hq + h) * pb->d;
    int64_t kbase = (r * pb->hkv + kvh) * pb->d;
    for (int64_t e = 0; e < pb->d; ++e)
        acc += load(pb->q, qbase + e, pb->dtype) * load(pb->k, kbase + e, pb->dtype);
#if PLANT != 4
    if (pb->qp) {
        int64_t qpbase = (q * pb->hq + h) * pb->p;
        int64_t kpbase = r * pb->p;             /* one shared position head */
        for (int64_t e = 0; e < pb->p; ++e)
            acc += load(pb->qp, qpbase + e, pb->dtype) * load(pb->kp, kpbase + e, pb->dtype);
    }
#endif
#if PLANT == 2
    return pb->scale * pb->scale * acc;
#else
    return pb->scale * acc;
#endif
}

/*
 * Softmax-weighted average of the value rows of keys [j0, j1) for row (q, h):
 * out[e] = sum_j w_j v_j[e] / sum_j w_j with w_j = exp(score_j - max score),
 * lse = max + log(sum_j w_j).  Empty range: out = 0, lse = -inf.
 */
static void attend_range(const problem *pb, int64_t q, int64_t h, int64_t j0, int64_t j1,
                         double *scores, double *out, double *lse) {
    for (int64_t e = 0; e < pb->dv; ++e) out[e] = 0.0;
    if (j1 <= j0) { *lse = -INFINITY; return; }
    int64_t s = pb->qseq[q];
    int64_t kvh = kv_head_of(pb, h);
    double m = -INFINITY;
    for (int64_t j = j0; j < j1; ++j) {
        scores[j - j0] = score(pb, q, h, j);
        if (scores[j - j0] > m) m = scores[j - j0];
    }
    double sum = 0.0;
    for (int64_t j = j0; j < j1; ++j) {
        double w = exp(scores[j - j0] - m);
        sum += w;
        int64_t r = cache_row(pb, s, j);
        /* MLA: the value is the latent row itself (k cache, one head). */
        int64_t vbase = pb->qp ? r * pb->d : (r * pb->hkv + kvh) * pb->dv;
        const void *vsrc = pb->qp ? pb->k : pb->v;
        for (int64_t e = 0; e < pb->dv; ++e) out[e] += w * load(vsrc, vbase + e, pb->dtype);
    }
    for (int64_t e = 0; e < pb->dv; ++e) out[e] /= sum;
    *lse = m + log(sum);
}

/* Split s of S over the visible keys [lo, hi) (see header for the reading). */
static void split_range(int64_t lo, int64_t hi, int64_t splits, int64_t s, int64_t ps, int64_t *j0,
                        int64_t *j1) {
    int64_t base = (lo / ps) * ps;
    int64_t n = hi - base;
    if (n < 0) n = 0;
    int64_t chunk = (n + splits - 1) / splits;
    chunk = ((chunk + ps - 1) / ps) * ps;
    int64_t b = base + s * chunk, e = b + chunk;
    if (b < lo) b = lo;
    if (b > hi) b = hi;
    if (e > hi) e = hi;
    if (e < b) e = b;
    *j0 = b;
    *j1 = e;
}

static int64_t max_visible(const problem *pb, const int64_t *rows, int64_t nrows) {
    int64_t mx = 1;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t q = rows ? rows[i] / pb->hq : i / pb->hq;
        int64_t n = visible(pb, q);
        if (n > mx) mx = n;
    }
    return mx;
}

#define PROBLEM_ARGS                                                                     \
    const void *q, const void *qp, const void *k, const void *v, const void *kp,        \
    int dtype, int64_t queries, int64_t hq, int64_t hkv, int64_t d, int64_t dv,          \
    int64_t p, const int32_t *seq_lens, int64_t seqs, const int32_t *table,              \
    int64_t width, const int32_t *qseq, const int32_t *qpos, int64_t page_size,          \
    int64_t pages, double scale, int causal, int64_t window

#define PROBLEM_INIT                                                                     \
    problem pb = {q, qp, k, v, kp, dtype, queries, hq, hkv, d, dv, p, seq_lens, seqs,    \
                  table, width, qseq, qpos, page_size, pages, scale, causal, window}

/*
 * Unsplit attention.  rows: NULL for every (query, head) in order, else a
 * list of nrows flat indices q*hq + h.  out: [nrows, dv] fp64; lse: [nrows].
 */
int pa_oracle_attention(PROBLEM_ARGS, const int64_t *rows, int64_t nrows,
                        double *out, double *lse, int nthreads) {
    PROBLEM_INIT;
    if (!rows) nrows = queries * hq;
    int64_t nmax = max_visible(&pb, rows, nrows);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int failed = 0;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)nmax);
        if (!scores) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            if (!scores) continue;
            int64_t flat = rows ? rows[i] : i;
            int64_t qi = flat / hq, h = flat % hq;
            attend_range(&pb, qi, h, visible_from(&pb, qi), visible(&pb, qi), scores, out + i * dv, lse + i);
        }
        free(scores);
    }
    return failed ? -1 : 0;
}

/*
 * Per-split partial results: out_part [splits, nrows, dv], lse_part
 * [splits, nrows], each split normalised within its own key range.
 */
int pa_oracle_attention_split(PROBLEM_ARGS, const int64_t *rows, int64_t nrows, int64_t splits,
                              double *out_part, double *lse_part, int nthreads) {
    PROBLEM_INIT;
    if (!rows) nrows = queries * hq;
    int64_t nmax = max_visible(&pb, rows, nrows);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int failed = 0;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)nmax);
        if (!scores) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            if (!scores) continue;
            int64_t flat = rows ? rows[i] : i;
            int64_t qi = flat / hq, h = flat % hq;
            int64_t lo = visible_from(&pb, qi), hi = visible(&pb, qi);
            for (int64_t sp = 0; sp < splits; ++sp) {
                int64_t j0, j1;
                split_range(lo, hi, splits, sp, page_size, &j0, &j1);
                attend_range(&pb, qi, h, j0, j1, scores, out_part + (sp * nrows + i) * dv,
                             lse_part + sp * nrows + i);
            }
        }
        free(scores);
    }
    return failed ? -1 : 0;
}

/*
 * Merge of split partials: M = max_s lse_s, w_s = exp(lse_s - M),
 * out = sum_s w_s o_s / sum_s w_s, lse = M + log(sum_s w_s).
 * Splits with lse = -inf carry weight 0.
 */
void pa_oracle_merge(const double *out_part, const double *lse_part, int64_t splits,
                     int64_t nrows, int64_t dv, double *out, double *lse) {
    for (int64_t i = 0; i < nrows; ++i) {
        double m = -INFINITY;
        for (int64_t sp = 0; sp < splits; ++sp)
            if (lse_part[sp * nrows + i] > m) m = lse_part[sp * nrows + i];
        for (int64_t e = 0; e < dv; ++e) out[i * dv + e] = 0.0;
        if (m == -INFINITY) { lse[i] = -INFINITY; continue; }
        double sum = 0.0;
        for (int64_t sp = 0; sp < splits; ++sp) {
            double l = lse_part[sp * nrows + i];
            if (l == -INFINITY) continue;
            double w = exp(l - m);
            sum += w;
            for (int64_t e = 0; e < dv; ++e) out[i * dv + e] += w * out_part[(sp * nrows + i) * dv + e];
        }
        for (int64_t e = 0; e < dv; ++e) out[i * dv + e] /= sum;
        lse[i] = m + log(sum);
    }
}

/* Split bounds as the oracle partitions them (exposed for the tests). */
void pa_oracle_split_range(int64_t lo, int64_t hi, int64_t splits, int64_t s, int64_t ps, int64_t *j0,
                           int64_t *j1) {
    split_range(lo, hi, splits, s, ps, j0, j1);
}

/*
 * Cache append: new_k[q, h, :] goes to key-cache row
 * block_table[seq][pos / ps] * ps + pos % ps, head h; likewise new_v.
 * Plain byte copies, elem bytes per element.
 */
void pa_oracle_kv_store(const void *new_k, const void *new_v, void *k_cache, void *v_cache,
                        int64_t elem, int64_t queries, int64_t heads, int64_t d, int64_t dv,
                        const int32_t *table, int64_t width, const int32_t *qseq,
                        const int32_t *qpos, int64_t page_size) {
    for (int64_t qi = 0; qi < queries; ++qi) {
        int64_t s = qseq[qi], pos = qpos[qi];
        int64_t row = (int64_t)table[s * width + pos / page_size] * page_size + pos % page_size;
        for (int64_t h = 0; h < heads; ++h) {
            memcpy((char *)k_cache + ((row * heads + h) * d) * elem,
                   (const char *)new_k + ((qi * heads + h) * d) * elem, (size_t)(d * elem));
            memcpy((char *)v_cache + ((row * heads + h) * dv) * elem,
                   (const char *)new_v + ((qi * heads + h) * dv) * elem, (size_t)(dv * elem));
        }
    }
}

int pa_oracle_plant(void) { return PLANT; }

int pa_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
