/*
 * MiniMax Sparse Attention (MSA) training hot path: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check of the entry module
 * and the CPU-baseline leg of the benchmark may load this library. It shares
 * no code, header, table or helper with the CUDA path, and the CUDA path
 * never calls it.
 *
 * Everything is computed in double precision, in the order the method states
 * it, with no blocking, fusion or reordering:
 *
 *   1. index scores  s[j] = scale_idx * <q_idx[b,t,g,:], k_idx[b,j,:]>, j <= t
 *      (itinai.ru "How to solve the memory problem with MiniMax Sparse
 *      Attention", section "How the indexer works"; dothoosh.com "how
 *      Flash-MSA cuts million-token training cost", "Block-sparsity mechanism")
 *   2. block max-pool pool[c] = max_{j in block c, j <= t} s[j]  (same passages)
 *   3. top-k: the own block t / Bk always, plus the top (k-1) earlier blocks
 *      under (pool descending, block index ascending); stored ascending and
 *      padded with -1  (itinai.ru, "Two-stage process" and "How the indexer
 *      works": k blocks per query, the query's own block always included)
 *   4. selected tokens S(g,t) = { j <= t : block(j) listed in block_idx };
 *      without a block_idx (NULL), every visible token j <= t: the full
 *      causal attention of the indexer warmup (itinai.ru, "Training sparse
 *      attention": the first iterations attend to everything)
 *   5. main branch: exact softmax attention over S, two-pass, with the LSE
 *      (itinai.ru "Two-stage process"; dothoosh.com "how FlashAttention cuts
 *      GPU memory traffic", "Exactness vs approximation")
 *   6. main backward from the closed forms dV += P^T dO, dP = dO V^T,
 *      dS = P (dP - D), D = rowsum(dO * O)  (dothoosh.com FlashAttention page,
 *      "Training and the backward pass")
 *   7. KL alignment: teacher p_main = head-mean of the main softmax, detached;
 *      student p_px = softmax of the index scores over S;
 *      KL = sum p_main (ln p_main - ln p_px); d KL / d s_px = p_px - p_main
 *      (dothoosh.com Flash-MSA page, "Fixing the KL-divergence bottleneck";
 *      itinai.ru "Training sparse attention")
 *
 * Inputs are passed either as bf16 bit patterns (widened exactly to double)
 * or as doubles (used by the finite-difference pins).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t B, T, Hq, G, d, d_idx, Bk, k;
    double scale;      /* main-branch softmax scale (1/sqrt(d) by default)   */
    double scale_idx;  /* index-branch score scale (1/sqrt(d_idx) by default) */
    double kl_weight;  /* weight of the per-row KL terms in the loss          */
} oshape;

enum { DT_BF16 = 0, DT_F64 = 1 };

static inline double ld(const void *p, int dt, size_t i) {
    if (dt == DT_F64) return ((const double *)p)[i];
    uint32_t u = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static inline int imin(int a, int b) { return a < b ? a : b; }

/* ---------------------------------------------------------------- steps 1-3 */
typedef struct {
    double v;
    int c;
} cand_t;

/* order: pool descending, then block index ascending */
static int cand_cmp(const void *pa, const void *pb) {
    const cand_t *a = (const cand_t *)pa, *b = (const cand_t *)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->c > b->c) - (a->c < b->c);
}

static int int_cmp(const void *pa, const void *pb) {
    int a = *(const int *)pa, b = *(const int *)pb;
    return (a > b) - (a < b);
}

/*
 * rows: ids (b*G + g)*T + t; NULL means every row (nrows = B*G*T).
 * block_idx: [nrows, k]; gap: [nrows] (may be NULL): pool of the (k-1)-th
 * selected earlier block minus pool of the best unselected one, +inf when every
 * earlier block fits; pool: [nrows, n_blocks] (may be NULL), -inf past the own block.
 */
int oracle_index_topk(const oshape *s, const void *q_idx, const void *k_idx, int dt,
                      const int64_t *rows, int64_t nrows, int32_t *block_idx, double *gap,
                      double *pool) {
    const int T = s->T, G = s->G, E = s->d_idx, Bk = s->Bk, k = s->k;
    const int nb = (T + Bk - 1) / Bk;
#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)T);
        double *pl = (double *)malloc(sizeof(double) * (size_t)nb);
        cand_t *cd = (cand_t *)malloc(sizeof(cand_t) * (size_t)nb);
        int *sel = (int *)malloc(sizeof(int) * (size_t)(k + 1));
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; r++) {
            const int64_t id = rows ? rows[r] : r;
            const int t = (int)(id % T);
            const int g = (int)((id / T) % G);
            const int b = (int)(id / ((int64_t)T * G));
            const int own = t / Bk;
            /* step 1: dense scores of every causally visible token */
            const size_t qo = (((size_t)b * T + t) * G + g) * E;
            for (int j = 0; j <= t; j++) {
                const size_t ko = ((size_t)b * T + j) * E;
                double acc = 0.0;
                for (int e = 0; e < E; e++) acc += ld(q_idx, dt, qo + e) * ld(k_idx, dt, ko + e);
                sc[j] = s->scale_idx * acc;
            }
            /* step 2: max-pool over each block's visible tokens */
            for (int c = 0; c < nb; c++) {
                pl[c] = -INFINITY;
                if (c > own) continue;
                const int j1 = imin((c + 1) * Bk, t + 1);
                for (int j = c * Bk; j < j1; j++)
                    if (sc[j] > pl[c]) pl[c] = sc[j];
            }
            if (pool)
                for (int c = 0; c < nb; c++) pool[r * nb + c] = pl[c];
            /* step 3: own block + top-(k-1) earlier blocks */
            for (int c = 0; c < own; c++) {
                cd[c].v = pl[c];
                cd[c].c = c;
            }
            qsort(cd, (size_t)own, sizeof(cand_t), cand_cmp);
            const int take = imin(k - 1, own);
            int m = 0;
            for (int i = 0; i < take; i++) sel[m++] = cd[i].c;
            sel[m++] = own;
            qsort(sel, (size_t)m, sizeof(int), int_cmp);
            for (int i = 0; i < k; i++) block_idx[r * k + i] = i < m ? sel[i] : -1;
            if (gap) gap[r] = (k >= 2 && own >= k) ? cd[k - 2].v - cd[k - 1].v : INFINITY;
        }
        free(sc);
        free(pl);
        free(cd);
        free(sel);
    }
    return 0;
}

/* ---------------------------------------------------------------- FP8 index inputs */
/*
 * Low-precision indexer (dothoosh.com "how Flash-MSA cuts million-token
 * training cost", "Current limits and future scaling": training the indexer
 * in low precision, as at inference). Steps 1-3 run on FP8 (E4M3) copies of
 * the index queries and keys. The pages fix no format details; the reading
 * taken here:
 *   - E4M3 "FN" values (1 sign, 4 exponent bits with bias 7, 3 mantissa
 *     bits, subnormals, no infinities, largest finite 448), rounding to
 *     nearest with ties to even, saturating at +-448;
 *   - one scale per q_idx row (b, t, g) and one per 128-key block of k_idx
 *     (b, c): amax = max |x| (fp32), x is multiplied by 448 / amax (fp32
 *     division, then fp32 multiply) and rounded to E4M3; the scale is
 *     amax / 448 (fp32), 1 when amax = 0;
 *   - scores s = scale_idx * (q8 * sq) . (k8 * sk): the quantized values
 *     times their scales, exactly, in double.
 */
double oracle_e4m3(double x) {
    if (isnan(x)) return x;
    const double a = fabs(x);
    if (a >= 448.0) return copysign(448.0, x);
    if (a == 0.0) return x;
    int e;
    frexp(a, &e);                  /* a = m 2^e, m in [1/2, 1): leading bit 2^(e-1) */
    int lead = e - 1;
    if (lead < -6) lead = -6;      /* subnormals: spacing 2^-9 */
    const double ulp = ldexp(1.0, lead - 3);
    const double y = nearbyint(a / ulp) * ulp;  /* round to nearest, ties to even */
    return copysign(y, x);
}

/* amax (fp32) -> (multiplier 448 / amax, scale amax / 448), both fp32 */
static void fp8_scales(float amax, float *mul, float *scale) {
    if (amax > 0.0f) {
        *mul = 448.0f / amax;
        *scale = amax / 448.0f;
    } else {
        *mul = 1.0f;
        *scale = 1.0f;
    }
}

static inline float ldf_bf16(const void *p, size_t i) {
    uint32_t u = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * q_idx [B,T,G,E], k_idx [B,T,E] as bf16 bits. Writes the dequantized values
 * q8 * sq -> q_deq [B,T,G,E] and k8 * sk -> k_deq [B,T,E] (doubles), and the
 * scales sq [B,T,G], sk [B, n_blocks] (fp32).
 */
int oracle_quantize_fp8(const oshape *s, const void *q_idx, const void *k_idx, double *q_deq, double *k_deq,
                        float *sq, float *sk) {
    const int B = s->B, T = s->T, G = s->G, E = s->d_idx, Bk = s->Bk;
    const int nb = (T + Bk - 1) / Bk;
    const int64_t qrows = (int64_t)B * T * G;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < qrows; r++) {
        float amax = 0.0f;
        for (int e = 0; e < E; e++) amax = fmaxf(amax, fabsf(ldf_bf16(q_idx, (size_t)r * E + e)));
        float mul, scale;
        fp8_scales(amax, &mul, &scale);
        sq[r] = scale;
        for (int e = 0; e < E; e++) {
            const float v = ldf_bf16(q_idx, (size_t)r * E + e) * mul;
            q_deq[(size_t)r * E + e] = oracle_e4m3((double)v) * (double)scale;
        }
    }
#pragma omp parallel for schedule(static)
    for (int64_t bc = 0; bc < (int64_t)B * nb; bc++) {
        const int b = (int)(bc / nb), c = (int)(bc % nb);
        const int j0 = c * Bk, j1 = imin((c + 1) * Bk, T);
        float amax = 0.0f;
        for (int j = j0; j < j1; j++)
            for (int e = 0; e < E; e++) amax = fmaxf(amax, fabsf(ldf_bf16(k_idx, ((size_t)b * T + j) * E + e)));
        float mul, scale;
        fp8_scales(amax, &mul, &scale);
        sk[bc] = scale;
        for (int j = j0; j < j1; j++)
            for (int e = 0; e < E; e++) {
                const size_t i = ((size_t)b * T + j) * E + e;
                const float v = ldf_bf16(k_idx, i) * mul;
                k_deq[i] = oracle_e4m3((double)v) * (double)scale;
            }
    }
    return 0;
}

/* ---------------------------------------------------------------- step 4 */
/* Selected, causally visible tokens of (b,g,t), ascending; duplicates in the
 * block list count once. block_idx NULL selects every visible token. Returns
 * |S|. tok must hold k*Bk entries (T without a block_idx). */
static int selected_tokens(const oshape *s, const int32_t *block_idx, int b, int g, int t,
                           int32_t *tok) {
    if (!block_idx) {
        for (int j = 0; j <= t; j++) tok[j] = j;
        return t + 1;
    }
    const int32_t *bl = block_idx + (((size_t)b * s->G + g) * s->T + t) * s->k;
    int cs[256];
    int m = 0;
    for (int i = 0; i < s->k && m < 256; i++) {
        const int c = bl[i];
        if (c < 0) continue;
        int dup = 0;
        for (int q = 0; q < m; q++) dup |= (cs[q] == c);
        if (!dup) cs[m++] = c;
    }
    qsort(cs, (size_t)m, sizeof(int), int_cmp);
    int n = 0;
    for (int i = 0; i < m; i++) {
        const int j0 = cs[i] * s->Bk;
        const int j1 = imin(imin((cs[i] + 1) * s->Bk, t + 1), s->T);
        for (int j = j0; j < j1; j++) tok[n++] = j;
    }
    return n;
}

/* ---------------------------------------------------------------- steps 5-7 */
typedef struct {
    size_t cap;    /* capacity: largest |S|       */
    int n;         /* |S|                         */
    int32_t *tok;  /* [k*Bk]                      */
    double *P;     /* [hg][k*Bk] main softmax     */
    double *dS;    /* [hg][k*Bk]                  */
    double *O;     /* [hg][d]                     */
    double *LSE;   /* [hg]                        */
    double *pmain; /* [k*Bk] head mean of P       */
    double *ppx;   /* [k*Bk] index softmax over S */
    double *gs;    /* [k*Bk] kl_weight*(ppx-pmain)*/
    double *tmp;   /* [k*Bk]                      */
    double KL;
} rowst;

/* Largest |S| of a row: k blocks, or every token without a block_idx. */
static size_t row_capacity(const oshape *s, const int32_t *block_idx) {
    return block_idx ? (size_t)s->k * s->Bk : (size_t)s->T;
}

static void rowst_alloc(const oshape *s, rowst *r, size_t L) {
    const size_t hg = (size_t)(s->Hq / s->G);
    r->cap = L;
    r->tok = (int32_t *)malloc(sizeof(int32_t) * L);
    r->P = (double *)malloc(sizeof(double) * hg * L);
    r->dS = (double *)malloc(sizeof(double) * hg * L);
    r->O = (double *)malloc(sizeof(double) * hg * (size_t)s->d);
    r->LSE = (double *)malloc(sizeof(double) * hg);
    r->pmain = (double *)malloc(sizeof(double) * L);
    r->ppx = (double *)malloc(sizeof(double) * L);
    r->gs = (double *)malloc(sizeof(double) * L);
    r->tmp = (double *)malloc(sizeof(double) * L);
}

static void rowst_free(rowst *r) {
    free(r->tok);
    free(r->P);
    free(r->dS);
    free(r->O);
    free(r->LSE);
    free(r->pmain);
    free(r->ppx);
    free(r->gs);
    free(r->tmp);
}

typedef struct {
    const void *Q, *K, *V, *dO, *q_idx, *k_idx;
    int dt;
    const int32_t *block_idx;
} oinputs;

/* Two-pass softmax of x[0..n): writes exp(x - lse) to p, returns lse. */
static double softmax2(const double *x, int n, double *p) {
    double m = -INFINITY;
    for (int i = 0; i < n; i++)
        if (x[i] > m) m = x[i];
    double z = 0.0;
    for (int i = 0; i < n; i++) z += exp(x[i] - m);
    const double lse = m + log(z);
    for (int i = 0; i < n; i++) p[i] = exp(x[i] - lse);
    return lse;
}

/* Everything one query position (b,g,t) contributes: steps 4-7 for its hg heads.
 * with_bwd = 0 stops after the forward (P, O, LSE). */
static void row_state(const oshape *s, const oinputs *in, int b, int g, int t, int with_bwd,
                      rowst *r) {
    const int T = s->T, Hq = s->Hq, G = s->G, d = s->d, E = s->d_idx;
    const int hg = Hq / G;
    const size_t L = r->cap;
    const int n = selected_tokens(s, in->block_idx, b, g, t, r->tok);
    r->n = n;
    for (int h = 0; h < hg; h++) {
        const int hh = g * hg + h;
        const size_t qo = (((size_t)b * T + t) * Hq + hh) * d;
        double *P = r->P + h * L;
        for (int i = 0; i < n; i++) {
            const size_t ko = (((size_t)b * T + r->tok[i]) * G + g) * d;
            double acc = 0.0;
            for (int e = 0; e < d; e++) acc += ld(in->Q, in->dt, qo + e) * ld(in->K, in->dt, ko + e);
            r->tmp[i] = s->scale * acc;
        }
        r->LSE[h] = softmax2(r->tmp, n, P);
        double *O = r->O + (size_t)h * d;
        for (int e = 0; e < d; e++) O[e] = 0.0;
        for (int i = 0; i < n; i++) {
            const size_t vo = (((size_t)b * T + r->tok[i]) * G + g) * d;
            for (int e = 0; e < d; e++) O[e] += P[i] * ld(in->V, in->dt, vo + e);
        }
    }
    if (!with_bwd) return;
    /* step 6: D = rowsum(dO * O), dP = dO . v_j, dS = P (dP - D) */
    for (int h = 0; h < hg; h++) {
        const int hh = g * hg + h;
        const size_t oo = (((size_t)b * T + t) * Hq + hh) * d;
        const double *O = r->O + (size_t)h * d;
        double D = 0.0;
        for (int e = 0; e < d; e++) D += ld(in->dO, in->dt, oo + e) * O[e];
        const double *P = r->P + h * L;
        double *dS = r->dS + h * L;
        for (int i = 0; i < n; i++) {
            const size_t vo = (((size_t)b * T + r->tok[i]) * G + g) * d;
            double dP = 0.0;
            for (int e = 0; e < d; e++) dP += ld(in->dO, in->dt, oo + e) * ld(in->V, in->dt, vo + e);
            dS[i] = P[i] * (dP - D);
        }
    }
    /* step 7: KL(p_main || p_px) and its closed-form score gradient */
    const size_t qio = (((size_t)b * T + t) * G + g) * E;
    for (int i = 0; i < n; i++) {
        double pm = 0.0;
        for (int h = 0; h < hg; h++) pm += r->P[h * L + i];
        r->pmain[i] = pm / hg;
        const size_t ko = ((size_t)b * T + r->tok[i]) * E;
        double acc = 0.0;
        for (int e = 0; e < E; e++) acc += ld(in->q_idx, in->dt, qio + e) * ld(in->k_idx, in->dt, ko + e);
        r->tmp[i] = s->scale_idx * acc;
    }
    const double lse_px = softmax2(r->tmp, n, r->ppx);
    double kl = 0.0;
    for (int i = 0; i < n; i++) {
        if (r->pmain[i] > 0.0) kl += r->pmain[i] * (log(r->pmain[i]) - (r->tmp[i] - lse_px));
        r->gs[i] = s->kl_weight * (r->ppx[i] - r->pmain[i]);
    }
    r->KL = kl;
}

/*
 * Forward for rows id = (b*T + t)*Hq + h (NULL: all B*T*Hq rows).
 * O: [nrows, d], LSE: [nrows]. block_idx NULL: every visible token (step 4).
 */
int oracle_sparse_fwd(const oshape *s, const void *Q, const void *K, const void *V, int dt,
                      const int32_t *block_idx, const int64_t *rows, int64_t nrows, double *O,
                      double *LSE) {
    const int T = s->T, Hq = s->Hq, G = s->G, d = s->d, hg = Hq / G;
    oinputs in = {Q, K, V, NULL, NULL, NULL, dt, block_idx};
#pragma omp parallel
    {
        rowst r;
        rowst_alloc(s, &r, row_capacity(s, block_idx));
#pragma omp for schedule(dynamic, 8)
        for (int64_t q = 0; q < nrows; q++) {
            const int64_t id = rows ? rows[q] : q;
            const int hh = (int)(id % Hq);
            const int t = (int)((id / Hq) % T);
            const int b = (int)(id / ((int64_t)Hq * T));
            const int g = hh / hg;
            row_state(s, &in, b, g, t, 0, &r);
            memcpy(O + q * d, r.O + (size_t)(hh - g * hg) * d, sizeof(double) * d);
            LSE[q] = r.LSE[hh - g * hg];
        }
        rowst_free(&r);
    }
    return 0;
}

/*
 * Per-query backward outputs for rows id = (b*G + g)*T + t (NULL: all).
 * dQ: [nrows, hg, d]; dq_idx: [nrows, d_idx]; KL: [nrows]. Any may be NULL.
 * block_idx NULL: every visible token (step 4).
 */
int oracle_bwd_rows(const oshape *s, const void *Q, const void *K, const void *V, const void *dO,
                    const void *q_idx, const void *k_idx, int dt, const int32_t *block_idx,
                    const int64_t *rows, int64_t nrows, double *dQ, double *dq_idx, double *KL) {
    const int T = s->T, G = s->G, d = s->d, E = s->d_idx, hg = s->Hq / s->G;
    const size_t L = row_capacity(s, block_idx);
    oinputs in = {Q, K, V, dO, q_idx, k_idx, dt, block_idx};
#pragma omp parallel
    {
        rowst r;
        rowst_alloc(s, &r, row_capacity(s, block_idx));
#pragma omp for schedule(dynamic, 4)
        for (int64_t q = 0; q < nrows; q++) {
            const int64_t id = rows ? rows[q] : q;
            const int t = (int)(id % T);
            const int g = (int)((id / T) % G);
            const int b = (int)(id / ((int64_t)T * G));
            row_state(s, &in, b, g, t, 1, &r);
            if (dQ) {
                for (int h = 0; h < hg; h++) {
                    double *out = dQ + (q * hg + h) * d;
                    for (int e = 0; e < d; e++) out[e] = 0.0;
                    for (int i = 0; i < r.n; i++) {
                        const size_t ko = (((size_t)b * T + r.tok[i]) * G + g) * d;
                        const double w = s->scale * r.dS[h * L + i];
                        for (int e = 0; e < d; e++) out[e] += w * ld(K, dt, ko + e);
                    }
                }
            }
            if (dq_idx) {
                double *out = dq_idx + q * E;
                for (int e = 0; e < E; e++) out[e] = 0.0;
                for (int i = 0; i < r.n; i++) {
                    const size_t ko = ((size_t)b * T + r.tok[i]) * E;
                    const double w = s->scale_idx * r.gs[i];
                    for (int e = 0; e < E; e++) out[e] += w * ld(k_idx, dt, ko + e);
                }
            }
            if (KL) KL[q] = r.KL;
        }
        rowst_free(&r);
    }
    return 0;
}

/*
 * Per-key-block backward outputs for blocks id = b*n_blocks + c (NULL: all).
 * Gathers every query of every group that selected block c (block_idx NULL:
 * every query t >= c*Bk, step 4). group >= 0 restricts the sums to that
 * group's queries (the other groups' dK, dV rows stay zero and dk_idx holds
 * only that group's share); group < 0 takes every group.
 * dK, dV: [nblocks, G, Bk, d]; dk_idx: [nblocks, Bk, d_idx]. Any may be NULL.
 */
int oracle_bwd_blocks(const oshape *s, const void *Q, const void *K, const void *V, const void *dO,
                      const void *q_idx, const void *k_idx, int dt, const int32_t *block_idx,
                      const int64_t *blocks, int64_t nblocks, int group, double *dK, double *dV,
                      double *dk_idx) {
    const int T = s->T, Hq = s->Hq, G = s->G, d = s->d, E = s->d_idx, Bk = s->Bk, k = s->k;
    const int hg = Hq / G, nb = (T + Bk - 1) / Bk;
    const size_t L = row_capacity(s, block_idx);
    oinputs in = {Q, K, V, dO, q_idx, k_idx, dt, block_idx};
#pragma omp parallel
    {
        rowst r;
        rowst_alloc(s, &r, row_capacity(s, block_idx));
#pragma omp for schedule(dynamic, 1)
        for (int64_t q = 0; q < nblocks; q++) {
            const int64_t id = blocks ? blocks[q] : q;
            const int c = (int)(id % nb);
            const int b = (int)(id / nb);
            const int j0 = c * Bk, j1 = imin((c + 1) * Bk, T);
            if (dK) memset(dK + q * (size_t)G * Bk * d, 0, sizeof(double) * (size_t)G * Bk * d);
            if (dV) memset(dV + q * (size_t)G * Bk * d, 0, sizeof(double) * (size_t)G * Bk * d);
            if (dk_idx) memset(dk_idx + q * (size_t)Bk * E, 0, sizeof(double) * (size_t)Bk * E);
            for (int g = 0; g < G; g++) {
                if (group >= 0 && g != group) continue;
                for (int t = j0; t < T; t++) {
                    /* without a block_idx every query t >= j0 sees block c */
                    int hit = !block_idx;
                    if (block_idx) {
                        const int32_t *bl = block_idx + (((size_t)b * G + g) * T + t) * k;
                        for (int i = 0; i < k; i++) hit |= (bl[i] == c);
                    }
                    if (!hit) continue;
                    row_state(s, &in, b, g, t, 1, &r);
                    const size_t qio = (((size_t)b * T + t) * G + g) * E;
                    for (int i = 0; i < r.n; i++) {
                        const int j = r.tok[i];
                        if (j < j0 || j >= j1) continue;
                        const int jj = j - j0;
                        for (int h = 0; h < hg; h++) {
                            const size_t qo = (((size_t)b * T + t) * Hq + g * hg + h) * d;
                            if (dK) {
                                double *out = dK + ((q * G + g) * (size_t)Bk + jj) * d;
                                const double w = s->scale * r.dS[h * L + i];
                                for (int e = 0; e < d; e++) out[e] += w * ld(Q, dt, qo + e);
                            }
                            if (dV) {
                                double *out = dV + ((q * G + g) * (size_t)Bk + jj) * d;
                                const double w = r.P[h * L + i];
                                for (int e = 0; e < d; e++) out[e] += w * ld(dO, dt, qo + e);
                            }
                        }
                        if (dk_idx) {
                            double *out = dk_idx + (q * (size_t)Bk + jj) * E;
                            const double w = s->scale_idx * r.gs[i];
                            for (int e = 0; e < E; e++) out[e] += w * ld(q_idx, dt, qio + e);
                        }
                    }
                }
            }
        }
        rowst_free(&r);
    }
    return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
