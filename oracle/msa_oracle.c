/*
 * CPU oracle for MiniMax-M3 block-sparse attention (MSA): plain C, fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the parity reference for the
 * CUDA path.  It shares no code with it (no headers, helpers, tables or
 * kernels) and only tests/, the package smoke check and the benchmark's CPU
 * baseline leg may load or run it.  The product path never calls it.
 *
 * What it computes, per query row r (at absolute position p) and KV head h,
 * written as the plain definition with no blocking or fusion:
 *
 *  1. Lightning-indexer scores (minimax_m3 CUDA backend PR #1388, commit
 *     "MiniMax-M3.1-Flash as a native Metal family": "the index scores and
 *     the top-16 block selection a row and key head"):
 *         s_t = sum_d iq[r,h,d] * ik[t,h,d]      for t = 0 .. p
 *     The pages name the indexer but print no formula; the plain reading is
 *     the dot product of the index query with the index key, no activation,
 *     weight or scale.
 *  2. Block max-pool (MiniMax-M3 on 4x RTX PRO 6000 Blackwell (SM120),
 *     section What this fixes: a block is scored by the largest index score
 *     among its positions):
 *         m_j = max { s_t : t in [jS, jS+S-1], t <= p }   for j = 0 .. J,
 *     J = floor(p / S) the block holding the current position.
 *  3. Top-k block selection per row and GQA group with the forced local
 *     block (same section: each GQA group keeps 16 blocks, one of them always
 *     the block of the current position): the kept set is {J} plus the
 *     (top_k - 1) best blocks
 *     j < J under the order (m_j descending, j ascending).  When J < top_k
 *     every causal block is kept.  The set is returned sorted ascending.
 *  4. Attention of each query head g of group h over the kept keys
 *     (PR #1388: decode rows attend over their kept blocks only; prompt
 *     chunks give the same per-row result, their tiles sharing the rows'
 *     selection):
 *         x_t = scale * (q[r, h*G+g] . k[t, h])  for t in kept blocks, t <= p
 *         o   = sum_t exp(x_t - max x) v[t, h] / sum_t exp(x_t - max x)
 *     Keys, values and index keys are bf16 (PR #1388, the commit that
 *     removes the int8 cache keeps all three caches in bf16); they are
 *     widened exactly to double here.
 *
 * Layouts (contiguous): q [R, H*G, D], iq [R, H, Di], k/v [T, H, D],
 * ik [T, H, Di]; token t of sequence b is cache row cache_starts[b] + t.
 *
 * Shared index key (ik_heads = 1): ik is [T, 1, Di] and every KV head's
 * index query meets the same key, s_t = sum_d iq[r,h,d] * ik[t,0,d].  The
 * pages print no formula for it; their cache arithmetic (MiniMax-M3 PR
 * #1388, commit removing the int8 cache: 135 KiB of cache a token) leaves
 * room for fewer index keys than one per KV head, and this is the plain
 * reading of one key per position for all heads.
 * Rows of sequence b are cu_rows[b] .. cu_rows[b+1]-1; with n rows and cache
 * length L, row i sits at p = L - n + i.
 *
 * int8 key/value cache (kv_int8 = 1): MiniMax-M3 PR #1388, native Metal
 * family commit, caches keys and values as int8 with one scale per position
 * and head (a later commit of the same PR goes back to bf16).  The pages
 * give no formula; the plain reading is dequantisation by that scale:
 *     k[t, h, d] = k_scale[t, h] * k8[t, h, d],  v likewise with v_scale,
 * both factors widened exactly to double (their product is exact), then
 * step 4 unchanged.  k8/v8 are [T, H, D] int8, the scales [T, H] float,
 * indexed by the same cache row as the values.  Index keys stay bf16.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct oracle_problem {
    int32_t num_seqs;
    int32_t H;      /* KV heads */
    int32_t G;      /* query heads per KV head */
    int32_t D;      /* head dim */
    int32_t Di;     /* index dim */
    int32_t S;      /* block size */
    int32_t top_k;  /* kept blocks per row and KV head, local included */
    double scale;   /* softmax scale */
    const int32_t* cu_rows;      /* [num_seqs + 1] */
    const int32_t* cache_lens;   /* [num_seqs] */
    const int64_t* cache_starts; /* [num_seqs] */
    int32_t ik_heads;            /* index keys per position: H, or 1 (shared); 0 means H */
    int32_t kv_int8;             /* 0: k, v bf16; 1: int8 with a scale per (cache row, head) */
    const float* k_scale;        /* [T, H] when kv_int8 */
    const float* v_scale;        /* [T, H] when kv_int8 */
} oracle_problem;

static double widen_bf16(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Element d of the key or value row of cache row `row`, KV head h: a bf16
 * value widened to double, or (kv_int8) the int8 value times its row's scale. */
static double kv_value(const oracle_problem* pr, const void* base, const float* scale, int64_t row, int32_t h,
                       int32_t d) {
    const int64_t i = (row * pr->H + h) * (int64_t)pr->D + d;
    if (pr->kv_int8)
        return (double)scale[row * pr->H + h] * (double)((const int8_t*)base)[i];
    return widen_bf16(((const uint16_t*)base)[i]);
}

/* Sequence index of query row r, and its absolute position p. */
static int locate_row(const oracle_problem* pr, int64_t r, int64_t* p_out) {
    for (int b = 0; b < pr->num_seqs; ++b) {
        if (r >= pr->cu_rows[b] && r < pr->cu_rows[b + 1]) {
            int64_t n = pr->cu_rows[b + 1] - pr->cu_rows[b];
            int64_t i = r - pr->cu_rows[b];
            *p_out = (int64_t)pr->cache_lens[b] - n + i;
            return b;
        }
    }
    return -1;
}

/* Step 1: s[t] for t = 0..p into s (room for cap values).  Returns p + 1,
 * or -1 for a bad row or too small a buffer. */
int oracle_index_scores(const oracle_problem* pr, const uint16_t* iq, const uint16_t* ik,
                        int64_t r, int32_t h, double* s, int64_t cap) {
    int64_t p;
    int b = locate_row(pr, r, &p);
    if (b < 0 || p < 0 || p + 1 > cap) return -1;
    const uint16_t* qi = iq + (r * pr->H + h) * (int64_t)pr->Di;
    for (int64_t t = 0; t <= p; ++t) {
        const int kh = pr->ik_heads == 1 ? 1 : pr->H; /* index-key heads per position */
        const uint16_t* ki = ik + ((pr->cache_starts[b] + t) * kh + (kh == 1 ? 0 : h)) * (int64_t)pr->Di;
        double acc = 0.0;
        for (int d = 0; d < pr->Di; ++d) acc += widen_bf16(qi[d]) * widen_bf16(ki[d]);
        s[t] = acc;
    }
    return (int)(p + 1);
}

/* Step 2: m[j] = max of s over block j, positions < n_pos.  Returns J + 1. */
int oracle_pool(const double* s, int64_t n_pos, int32_t S, double* m) {
    int64_t nblocks = (n_pos + S - 1) / S;
    for (int64_t j = 0; j < nblocks; ++j) {
        double best = -INFINITY;
        for (int64_t t = j * S; t < (j + 1) * S && t < n_pos; ++t)
            if (s[t] > best) best = s[t];
        m[j] = best;
    }
    return (int)nblocks;
}

typedef struct { double m; int32_t j; } scored_block;

/* (m descending, j ascending) */
static int by_score_then_index(const void* a, const void* b) {
    const scored_block* x = (const scored_block*)a;
    const scored_block* y = (const scored_block*)b;
    if (x->m > y->m) return -1;
    if (x->m < y->m) return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

static int ascending_int(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* Step 3: kept blocks from the pooled scores of blocks 0..nblocks-1, where
 * the last block (nblocks-1) holds the current position and is forced.
 * Writes nsel ascending block indices to sel and -1 up to top_k.  Returns
 * nsel. */
int oracle_select(const double* m, int32_t nblocks, int32_t top_k, int32_t* sel) {
    int32_t J = nblocks - 1;
    int32_t others = top_k - 1 < J ? top_k - 1 : J;
    scored_block* cand = (scored_block*)malloc(sizeof(scored_block) * (size_t)(J > 0 ? J : 1));
    for (int32_t j = 0; j < J; ++j) { cand[j].m = m[j]; cand[j].j = j; }
    qsort(cand, (size_t)J, sizeof(scored_block), by_score_then_index);
    int32_t n = 0;
    for (int32_t i = 0; i < others; ++i) sel[n++] = cand[i].j;
    sel[n++] = J;
    free(cand);
    qsort(sel, (size_t)n, sizeof(int32_t), ascending_int);
    for (int32_t i = n; i < top_k; ++i) sel[i] = -1;
    return n;
}

/* Step 4: out[g, d] for the G query heads of KV head h at row r, attending
 * over the keys of the listed blocks that are <= p. */
int oracle_attend(const oracle_problem* pr, const uint16_t* q, const void* k, const void* v,
                  int64_t r, int32_t h, const int32_t* sel, int32_t nsel, double* out) {
    int64_t p;
    int b = locate_row(pr, r, &p);
    if (b < 0 || p < 0) return -1;
    const int D = pr->D, H = pr->H, G = pr->G, S = pr->S;
    int64_t nkeys = 0;
    for (int32_t i = 0; i < nsel; ++i) nkeys += S;
    int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nkeys > 0 ? nkeys : 1));
    double* x = (double*)malloc(sizeof(double) * (size_t)(nkeys > 0 ? nkeys : 1));
    int64_t nk = 0;
    for (int32_t i = 0; i < nsel; ++i)
        for (int64_t t = (int64_t)sel[i] * S; t < (int64_t)(sel[i] + 1) * S; ++t)
            if (t >= 0 && t <= p) keys[nk++] = t;
    for (int g = 0; g < G; ++g) {
        const uint16_t* qg = q + (r * (int64_t)(H * G) + (int64_t)h * G + g) * D;
        double* o = out + (int64_t)g * D;
        double mx = -INFINITY;
        for (int64_t i = 0; i < nk; ++i) {
            const int64_t row = pr->cache_starts[b] + keys[i];
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += widen_bf16(qg[d]) * kv_value(pr, k, pr->k_scale, row, h, d);
            x[i] = pr->scale * acc;
            if (x[i] > mx) mx = x[i];
        }
        double den = 0.0;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int64_t i = 0; i < nk; ++i) {
            double w = exp(x[i] - mx);
            den += w;
            const int64_t row = pr->cache_starts[b] + keys[i];
            for (int d = 0; d < D; ++d) o[d] += w * kv_value(pr, v, pr->v_scale, row, h, d);
        }
        for (int d = 0; d < D; ++d) o[d] = nk > 0 ? o[d] / den : 0.0;
    }
    free(keys);
    free(x);
    return (int)nk;
}

/* Steps 1-4 for the listed rows (all rows when rows == NULL).  Output slot i
 * holds row rows[i]: sel [n, H, top_k], nsel [n, H], pooled (optional)
 * [n, H, max_blocks], out [n, H*G, D].  Returns 0, or -1 on a bad row. */
int oracle_forward(const oracle_problem* pr, const uint16_t* q, const uint16_t* iq,
                   const void* k, const void* v, const uint16_t* ik,
                   const int64_t* rows, int64_t nrows, int32_t* sel, int32_t* nsel,
                   double* out, double* pooled, int64_t max_blocks, int32_t nthreads) {
    const int H = pr->H;
    int64_t total = nrows * H;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
#endif
    for (int64_t w = 0; w < total; ++w) {
        int64_t slot = w / H;
        int32_t h = (int32_t)(w % H);
        int64_t r = rows ? rows[slot] : slot;
        int64_t p;
        if (locate_row(pr, r, &p) < 0 || p < 0) { bad = 1; continue; }
        double* s = (double*)malloc(sizeof(double) * (size_t)(p + 1));
        double* m = (double*)malloc(sizeof(double) * (size_t)(p / pr->S + 1));
        oracle_index_scores(pr, iq, ik, r, h, s, p + 1);
        int32_t nb = oracle_pool(s, p + 1, pr->S, m);
        int32_t* sl = sel + (slot * H + h) * (int64_t)pr->top_k;
        int32_t n = oracle_select(m, nb, pr->top_k, sl);
        nsel[slot * H + h] = n;
        if (pooled) {
            double* pd = pooled + (slot * H + h) * max_blocks;
            for (int64_t j = 0; j < max_blocks; ++j) pd[j] = j < nb ? m[j] : -INFINITY;
        }
        if (out)
            oracle_attend(pr, q, k, v, r, h, sl, n, out + (slot * (int64_t)(H * pr->G) + (int64_t)h * pr->G) * pr->D);
        free(s);
        free(m);
    }
    return bad ? -1 : 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
