/*
 * CPU oracle for the indexer -> causal top-k -> sparse MLA layer step.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * definition the CUDA library is checked against. It is built and called only
 * by the tests, by __graft_entry__.smoke() and by bench.py's cpu_baseline /
 * reference legs. It shares no code, header, table or helper with the CUDA
 * path under indexer_top_sparse_score_gb300/csrc.
 *
 * What it computes, for a query row at absolute position `pos` (keys 0..pos):
 *
 *  1. Indexer ("Optimisations de GLM-5.3, partie 2", section "Pourquoi pas TP
 *     ou DP ?": the indexer scores every earlier token to choose what sparse
 *     MLA reads). The formula is the one fixed for this step:
 *        score(t, s) = sum_h w[t,h] * ReLU( q_I[t,h,:] . k_I[s,:] ) * kscale[s]
 *     evaluated in fp32 (dot products accumulated in index order, heads summed
 *     in index order). kscale is the optional per-key indexer-key scale of the
 *     132-byte key row of footnote 3 (128 FP8 values + a 4-byte scale); absent
 *     means 1. "Earlier" includes the query's own position (s <= pos).
 *  2. Causal top-k (same page: the indexer selects the 2,048 tokens sparse MLA
 *     consults): all (score, s) pairs sorted by score descending, ties to the
 *     lower index; the first min(k, pos+1) are kept, reported in ascending
 *     index order, the rest of the row padded with -1.
 *  3. Sparse MLA in MQA form (same page, section "PCP" and footnote 1: each
 *     selected latent row serves all heads; QK over 576 dims, PV over 512):
 *        l_j   = sm_scale * sum_{d<576} q[h,d] * K[s_j,d]
 *        p_j   = exp(l_j - max l) / sum_j exp(l_j - max l)
 *        out_h = sum_j p_j * K[s_j, 0:512]
 *        lse_h = max l + ln sum_j exp(l_j - max l)
 *     in fp64, with K dequantised as float(e4m3) * per-token scale for FP8,
 *     and for the 656-byte tile-scaled FP8 row (footnote 1's fp8_ds_mla size)
 *     as float(e4m3) * the scale of the value's 128-value tile for the 512
 *     latent values and float(bf16) for the 64 rope values.
 *
 * Readings where the pages are silent: the diagonal is included, ties go to
 * the lower index, V is the first 512 values of the same row, lse uses the
 * natural logarithm, rows with fewer than k keys keep them all.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BF16 0
#define ORACLE_FP8 1
#define ORACLE_FP8_DS_MLA 2  /* 656-byte row: 512 e4m3 | 4 fp32 tile scales | 64 bf16 rope */
#define DS_MLA_ROW_BYTES 656

#define D_QK 576
#define D_V 512

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent 0 encodes subnormals m/8 * 2^-6; the
 * all-ones exponent with all-ones mantissa is NaN; there is no infinity. */
float oracle_e4m3_to_float(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    float mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexpf((float)m / 8.0f, -6);
    else mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32. */
float oracle_bf16_to_float(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

typedef struct {
    /* cache (one layer, paged, `page_size` tokens per page) */
    const void *kv;            /* [num_pages][page_size][576] bf16 or e4m3 */
    const float *kv_scale;     /* [num_pages][page_size] (FP8 only) */
    const void *k_idx;         /* [num_pages][page_size][d_idx] bf16 or e4m3 */
    const float *k_idx_scale;  /* [num_pages][page_size] or NULL */
    int32_t kv_dtype, idx_dtype, d_idx, page_size;
    int64_t num_pages;
    /* queries, one row per query token */
    const uint16_t *q;         /* [rows][n_heads][576] bf16 */
    const void *q_idx;         /* [rows][h_idx][d_idx] */
    const float *w;            /* [rows][h_idx] */
    int32_t n_heads, h_idx, topk;
    double sm_scale;
    /* positions and page tables */
    int32_t is_decode;         /* 0: one prefill sequence, 1: decode batch */
    int64_t prefix_len;        /* prefill: row r sits at prefix_len + r */
    const int32_t *seq_lens;   /* decode: [n_seqs] keys incl. new tokens */
    int32_t q_per_seq;         /* decode: rows per sequence */
    const int32_t *page_tables;/* [n_seqs][max_pages] (prefill: n_seqs = 1) */
    int32_t max_pages;
} oracle_problem;

/* Which sequence a row belongs to and its absolute position. */
static void row_place(const oracle_problem *p, int64_t row, int64_t *seq, int64_t *pos) {
    if (!p->is_decode) {
        *seq = 0;
        *pos = p->prefix_len + row;
    } else {
        int64_t b = row / p->q_per_seq;
        int64_t j = row % p->q_per_seq;
        *seq = b;
        *pos = (int64_t)p->seq_lens[b] - p->q_per_seq + j;
    }
}

/* Pool row of logical token s of sequence `seq` (page table lookup). Returns
 * -1 for a page id outside the pool. */
static int64_t pool_row(const oracle_problem *p, int64_t seq, int64_t s) {
    int64_t page = p->page_tables[seq * (int64_t)p->max_pages + s / p->page_size];
    if (page < 0 || page >= p->num_pages) return -1;
    return page * p->page_size + s % p->page_size;
}

/* All 256 e4m3 codes decoded once with oracle_e4m3_to_float, when the
 * library is loaded (before any thread can read the table). */
static float e4m3_table[256];
__attribute__((constructor)) static void init_e4m3_table(void) {
    for (int c = 0; c < 256; ++c) e4m3_table[c] = oracle_e4m3_to_float((uint8_t)c);
}

static float idx_elem(const void *base, int dtype, int64_t i) {
    if (dtype == ORACLE_BF16) return oracle_bf16_to_float(((const uint16_t *)base)[i]);
    return e4m3_table[((const uint8_t *)base)[i]];
}

/* Row `prow` of the latent cache as fp64 values (FP8: e4m3 value * token
 * scale; tile-scaled FP8: byte d < 512 is the e4m3 code of latent value d,
 * bytes 512 + 4t .. 515 + 4t the little-endian fp32 scale of values
 * 128t .. 128t + 127, bytes 528 + 2r, 529 + 2r the bf16 rope value r). */
static void kv_row(const oracle_problem *p, int64_t prow, double *dst) {
    if (p->kv_dtype == ORACLE_FP8_DS_MLA) {
        const uint8_t *row = (const uint8_t *)p->kv + prow * DS_MLA_ROW_BYTES;
        for (int d = 0; d < D_V; ++d) {
            float scale;
            memcpy(&scale, row + D_V + 4 * (d / 128), sizeof scale);
            dst[d] = (double)e4m3_table[row[d]] * (double)scale;
        }
        for (int r = 0; r < D_QK - D_V; ++r) {
            const uint8_t *b = row + D_V + 16 + 2 * r;
            dst[D_V + r] = (double)oracle_bf16_to_float((uint16_t)(b[0] | (b[1] << 8)));
        }
        return;
    }
    for (int d = 0; d < D_QK; ++d) {
        int64_t i = prow * D_QK + d;
        if (p->kv_dtype == ORACLE_BF16) dst[d] = (double)oracle_bf16_to_float(((const uint16_t *)p->kv)[i]);
        else dst[d] = (double)e4m3_table[((const uint8_t *)p->kv)[i]] * (double)p->kv_scale[prow];
    }
}

/* Step 1: indexer scores of query `row` against keys 0..pos (fp32). */
int oracle_scores(const oracle_problem *p, int64_t row, float *scores) {
    int64_t seq, pos;
    row_place(p, row, &seq, &pos);
    const int H = p->h_idx, D = p->d_idx;
    float *qf = (float *)malloc(sizeof(float) * H * D);
    float *kf = (float *)malloc(sizeof(float) * D);
    for (int i = 0; i < H * D; ++i) qf[i] = idx_elem(p->q_idx, p->idx_dtype, row * (int64_t)H * D + i);
    const float *wr = p->w + row * (int64_t)H;
    int bad = 0;
    for (int64_t s = 0; s <= pos; ++s) {
        int64_t pr = pool_row(p, seq, s);
        if (pr < 0) { bad = 1; scores[s] = 0.0f; continue; }
        for (int d = 0; d < D; ++d) kf[d] = idx_elem(p->k_idx, p->idx_dtype, pr * D + d);
        float total = 0.0f;
        for (int h = 0; h < H; ++h) {
            float dot = 0.0f;
            for (int d = 0; d < D; ++d)
                dot += qf[h * D + d] * kf[d];
            float relu = dot > 0.0f ? dot : 0.0f;
            total += wr[h] * relu;
        }
        if (p->k_idx_scale) total *= p->k_idx_scale[pr];
        scores[s] = total;
    }
    free(kf);
    free(qf);
    return bad;
}

typedef struct { float score; int64_t index; } scored;

/* Order: larger score first; equal scores: smaller index first. */
static int by_score_then_index(const void *a, const void *b) {
    const scored *x = (const scored *)a, *y = (const scored *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->index > y->index) - (x->index < y->index);
}

static int by_index(const void *a, const void *b) {
    const scored *x = (const scored *)a, *y = (const scored *)b;
    return (x->index > y->index) - (x->index < y->index);
}

/* Step 2: keep the min(k, n) best of n scores; ascending indices; pad -1. */
void oracle_select_topk(const float *scores, int64_t n, int32_t k, int32_t *idx_out, float *score_out) {
    scored *all = (scored *)malloc(sizeof(scored) * (n > 0 ? n : 1));
    for (int64_t s = 0; s < n; ++s) { all[s].score = scores[s]; all[s].index = s; }
    qsort(all, (size_t)n, sizeof(scored), by_score_then_index);
    int64_t keep = n < k ? n : k;
    qsort(all, (size_t)keep, sizeof(scored), by_index);
    for (int64_t i = 0; i < k; ++i) {
        idx_out[i] = i < keep ? (int32_t)all[i].index : -1;
        if (score_out) score_out[i] = i < keep ? all[i].score : 0.0f;
    }
    free(all);
}

/* Step 3: attention of query `row` over the n_idx tokens listed in `idx`
 * (entries < 0 are skipped). out: [n_heads][512]; lse: [n_heads];
 * probs (optional): [n_heads][n_idx], the softmax weights. */
int oracle_attend(const oracle_problem *p, int64_t row, const int32_t *idx, int32_t n_idx,
                  double *out, double *lse, double *probs) {
    int64_t seq, pos;
    row_place(p, row, &seq, &pos);
    const int H = p->n_heads;
    int64_t *prow = (int64_t *)malloc(sizeof(int64_t) * (n_idx > 0 ? n_idx : 1));
    int bad = 0;
    for (int j = 0; j < n_idx; ++j) {
        prow[j] = -1;
        if (idx[j] < 0) continue;
        if (idx[j] > pos) { bad = 1; continue; }
        prow[j] = pool_row(p, seq, idx[j]);
        if (prow[j] < 0) bad = 1;
    }
    const int64_t n = n_idx > 0 ? n_idx : 1;
    double *logit = (double *)malloc(sizeof(double) * H * n);   /* [H][n_idx] */
    double *qd = (double *)malloc(sizeof(double) * H * D_QK);
    double *kr = (double *)malloc(sizeof(double) * D_QK);
    double *m = (double *)malloc(sizeof(double) * H);
    double *denom = (double *)malloc(sizeof(double) * H);
    for (int h = 0; h < H; ++h) {
        const uint16_t *qr = p->q + (row * (int64_t)H + h) * D_QK;
        for (int d = 0; d < D_QK; ++d) qd[h * D_QK + d] = (double)oracle_bf16_to_float(qr[d]);
        m[h] = -INFINITY;
        denom[h] = 0.0;
    }
    /* logits: l[h][j] = sm_scale * sum_d q[h][d] K[j][d] (d ascending) */
    for (int j = 0; j < n_idx; ++j) {
        if (prow[j] < 0) continue;
        kv_row(p, prow[j], kr);
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            const double *q = qd + h * D_QK;
            for (int d = 0; d < D_QK; ++d) acc += q[d] * kr[d];
            double l = p->sm_scale * acc;
            logit[h * n + j] = l;
            if (l > m[h]) m[h] = l;
        }
    }
    for (int h = 0; h < H; ++h)
        for (int j = 0; j < n_idx; ++j)
            if (prow[j] >= 0) denom[h] += exp(logit[h * n + j] - m[h]);
    for (int h = 0; h < H; ++h) {
        double *o = out + (int64_t)h * D_V;
        for (int d = 0; d < D_V; ++d) o[d] = 0.0;
    }
    /* out[h] = sum_j p[h][j] V[j] (j ascending for every head) */
    for (int j = 0; j < n_idx; ++j) {
        if (prow[j] >= 0) kv_row(p, prow[j], kr);
        for (int h = 0; h < H; ++h) {
            double pj = prow[j] >= 0 ? exp(logit[h * n + j] - m[h]) / denom[h] : 0.0;
            if (probs) probs[(int64_t)h * n_idx + j] = pj;
            if (prow[j] < 0) continue;
            double *o = out + (int64_t)h * D_V;
            for (int d = 0; d < D_V; ++d) o[d] += pj * kr[d];
        }
    }
    for (int h = 0; h < H; ++h) lse[h] = denom[h] > 0.0 ? m[h] + log(denom[h]) : -INFINITY;
    free(kr);
    free(m);
    free(denom);
    free(qd);
    free(logit);
    free(prow);
    return bad;
}

/* Steps 1-3 for one row. idx_out/score_out: [topk]; out: [n_heads][512]; lse: [n_heads].
 * out/lse may be NULL (indexer + top-k only). */
int oracle_row(const oracle_problem *p, int64_t row, int32_t *idx_out, float *score_out,
               double *out, double *lse) {
    int64_t seq, pos;
    row_place(p, row, &seq, &pos);
    float *scores = (float *)malloc(sizeof(float) * (size_t)(pos + 1));
    int bad = oracle_scores(p, row, scores);
    oracle_select_topk(scores, pos + 1, p->topk, idx_out, score_out);
    free(scores);
    if (out && lse) bad |= oracle_attend(p, row, idx_out, p->topk, out, lse, NULL);
    return bad;
}

/* Many rows, OpenMP over rows. Outputs are indexed by position in `rows`.
 * Returns the number of OpenMP threads used. */
int oracle_rows(const oracle_problem *p, const int64_t *rows, int64_t n_rows, int32_t *idx_out,
                float *score_out, double *out, double *lse, int n_threads, int32_t *bad_out) {
    int used = 1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
    {
#pragma omp single
        used = omp_get_num_threads();
    }
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < n_rows; ++i) {
        int32_t *io = idx_out + i * (int64_t)p->topk;
        float *so = score_out ? score_out + i * (int64_t)p->topk : NULL;
        double *oo = out ? out + i * (int64_t)p->n_heads * D_V : NULL;
        double *lo = lse ? lse + i * (int64_t)p->n_heads : NULL;
        int b = oracle_row(p, rows[i], io, so, oo, lo);
        if (bad_out) bad_out[i] = b;
    }
    return used;
}

/* Attention only, for many rows with caller-given index lists [n_rows][n_idx]. */
int oracle_attend_rows(const oracle_problem *p, const int64_t *rows, int64_t n_rows,
                       const int32_t *idx, int32_t n_idx, double *out, double *lse, int n_threads) {
    int used = 1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
    {
#pragma omp single
        used = omp_get_num_threads();
    }
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < n_rows; ++i)
        oracle_attend(p, rows[i], idx + i * (int64_t)n_idx, n_idx,
                      out + i * (int64_t)p->n_heads * D_V, lse + i * (int64_t)p->n_heads, NULL);
    return used;
}
