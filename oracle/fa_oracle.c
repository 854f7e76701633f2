/*
 * fa_oracle.c -- plain, slow, obviously correct f64 CPU reference for causal
 * prefill attention.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
 * the benchmark's CPU-baseline leg call it; the product path never does.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (the plain definition the tiled kernel reaches up to
 * rounding order), for every batch b, query head hq and query row i:
 *
 *   hk   = hq / (Hq / Hkv)                        contiguous GQA grouping
 *   s_j  = scale * sum_d q[b,i,hq,d] * k[b,j,hk,d]   for all j < Skv
 *   s_j  = -inf  if causal and j > (Skv - Sq) + i  (bottom-right alignment)
 *   m    = max_j s_j ;  if m == -inf the row sees no key and o = 0
 *   p_j  = exp(s_j - m) / sum_j exp(s_j - m)
 *   o[d] = sum_j p_j * v[b,j,hk,d]
 *
 * Sources on the pages:
 *  - the mask: minfer "28 · r23 — f16-path whole-graph wall decomposition +
 *    FA_TKV occupancy raise", section 3.2: a key column is valid when it is at
 *    or before the query's absolute position AND inside the stored KV range.
 *    The query's absolute position is its index among the Skv keys, i.e.
 *    (Skv - Sq) + i: the Sq new rows are the last Sq positions of the cache.
 *  - the fully-masked row: minfer "53 · r50 — FA_TKV 32->16 occupancy
 *    experiment", section 3.2 keeps the running max at -inf when a tile has no
 *    valid column; a row that never sees a key therefore has l = 0, and this
 *    oracle defines its output as 0.
 *  - the GQA head mapping: the same page, section 3.2, passes one KV head
 *    index per query head; the contiguous grouping hq / G is the reading.
 *  - the softmax itself: the exact max-subtracted softmax over the full score
 *    row, which the online softmax of the pages reaches up to f32 regrouping
 *    (same page, section 2, "why byte identity is necessarily lost").
 *
 * Layout: contiguous "BSHD" -- q, o are [B][Sq][Hq][hd]; k, v are
 * [B][Skv][Hkv][hd]; hd fastest.  All arithmetic is IEEE double with libm
 * exp(); inputs are the 16-bit tensors upcast exactly to double by the caller.
 *
 * Every function computes the full score row (all Skv entries) and masks it
 * afterwards, one row at a time, so memory stays O(Skv) per thread.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

/* Planted mistakes, for the pin tests only.  The tests switch one of these on
 * to show that the pins reject a wrong oracle, and switch it back off.  0, the
 * default, is the correct oracle. */
enum {
    PLANT_NONE = 0,
    PLANT_NO_SCALE = 1,        /* scores not multiplied by scale          */
    PLANT_TOP_LEFT = 2,        /* causal mask aligned top-left (off = 0)   */
    PLANT_MASK_OFF_BY_ONE = 3, /* key j = off + i masked as well           */
    PLANT_GQA_MODULO = 4,      /* kv head hq % Hkv instead of hq / G       */
    PLANT_NO_NORMALISE = 5,    /* softmax numerators not divided by the sum */
    PLANT_V_REVERSED = 6,      /* V read with its hd index reversed         */
    PLANT_NO_MAX_SUBTRACT = 7, /* exp(s_j) without subtracting the max      */
    PLANT_EXP2 = 8,            /* base-2 exponential instead of e           */
    PLANT_MASKED_ROW_NAN = 9,  /* no guard for rows that see no key         */
    PLANT_ROUND_TRUNCATE = 10, /* cache append rounds toward zero           */
    PLANT_ROUND_TIES_AWAY = 11,/* cache append breaks ties away from zero   */
    PLANT_APPEND_AT_T = 12,    /* cache append writes row t, not positions[t] */
    PLANT_LSE_LOG2 = 13,       /* log-sum-exp taken in base 2               */
    PLANT_COUNT = 14
};
static int g_plant = PLANT_NONE;

int oracle_plant_mistake(int kind)
{
    if (kind < 0 || kind >= PLANT_COUNT) return ORACLE_BAD_ARG;
    g_plant = kind;
    return ORACLE_OK;
}

typedef struct {
    const double *q, *k, *v;
    int B, Hq, Hkv, Sq, Skv, hd, causal;
    double scale;
} shape_t;

static int check_shape(const shape_t *s)
{
    if (!s->q || !s->k || !s->v) return ORACLE_BAD_ARG;
    if (s->B < 0 || s->Sq < 0 || s->Skv < 0) return ORACLE_BAD_ARG;
    if (s->Hq <= 0 || s->Hkv <= 0 || s->hd <= 0) return ORACLE_BAD_ARG;
    if (s->Hq % s->Hkv != 0) return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

/* Scores of query row (b, hq, i) against every key of its KV head, then the
 * mask.  srow receives Skv entries. Returns the row maximum (-inf if every
 * key is masked). */
static double score_row(const shape_t *s, int b, int hq, int i, double *srow)
{
    const int G = s->Hq / s->Hkv;
    const int hk = (g_plant == PLANT_GQA_MODULO) ? hq % s->Hkv : hq / G;
    const long long off = (g_plant == PLANT_TOP_LEFT) ? 0 : (long long)s->Skv - (long long)s->Sq;
    const double *qr = s->q + (((long long)b * s->Sq + i) * s->Hq + hq) * s->hd;
    double m = -INFINITY;
    for (int j = 0; j < s->Skv; ++j) {
        const double *kr = s->k + (((long long)b * s->Skv + j) * s->Hkv + hk) * s->hd;
        double dot = 0.0;
        for (int d = 0; d < s->hd; ++d) dot += qr[d] * kr[d];
        double sj = (g_plant == PLANT_NO_SCALE) ? dot : s->scale * dot;
        if (s->causal && (long long)j > off + i) sj = -INFINITY;
        if (g_plant == PLANT_MASK_OFF_BY_ONE && s->causal && (long long)j == off + i) sj = -INFINITY;
        srow[j] = sj;
        if (sj > m) m = sj;
    }
    return m;
}

/* Softmax of one score row in place: srow becomes the probabilities.
 * Returns 0 when the row has no visible key (all probabilities 0). */
static int softmax_row(double *srow, int Skv, double m)
{
    if (m == -INFINITY && g_plant != PLANT_MASKED_ROW_NAN) {
        for (int j = 0; j < Skv; ++j) srow[j] = 0.0;
        return 0;
    }
    if (g_plant == PLANT_NO_MAX_SUBTRACT) m = 0.0;
    double sum = 0.0;
    for (int j = 0; j < Skv; ++j) {
        double x = srow[j] - m;
        double e = (g_plant == PLANT_EXP2) ? exp2(x) : exp(x);
        if (srow[j] == -INFINITY && g_plant != PLANT_MASKED_ROW_NAN) e = 0.0;
        srow[j] = e;
        sum += e;
    }
    if (g_plant != PLANT_NO_NORMALISE)
        for (int j = 0; j < Skv; ++j) srow[j] /= sum;
    return 1;
}

/* One output row: o[d] = sum_j p_j v[b,j,hk,d]. */
static void attend_row(const shape_t *s, int b, int hq, int i, double *srow, double *orow)
{
    const int G = s->Hq / s->Hkv;
    const int hk = (g_plant == PLANT_GQA_MODULO) ? hq % s->Hkv : hq / G;
    double m = score_row(s, b, hq, i, srow);
    int any = softmax_row(srow, s->Skv, m);
    for (int d = 0; d < s->hd; ++d) orow[d] = 0.0;
    if (!any) return;
    for (int j = 0; j < s->Skv; ++j) {
        const double pj = srow[j];
        if (pj == 0.0) continue;
        if (pj != pj) { for (int d = 0; d < s->hd; ++d) orow[d] = pj; return; }
        const double *vr = s->v + (((long long)b * s->Skv + j) * s->Hkv + hk) * s->hd;
        for (int d = 0; d < s->hd; ++d)
            orow[d] += pj * vr[(g_plant == PLANT_V_REVERSED) ? s->hd - 1 - d : d];
    }
}

/* ---- threading: a static split of a list of rows over worker threads ---- */

typedef struct {
    const shape_t *s;
    const int32_t *rows;   /* NULL: all rows in (b, i, hq) order */
    long long first, last; /* [first, last) row indices */
    double *out;           /* full o tensor (rows == NULL) or [n][hd] */
    int status;
} work_t;

static void decode_all(const shape_t *s, long long r, int *b, int *hq, int *i)
{
    *hq = (int)(r % s->Hq);
    long long t = r / s->Hq;
    *i = (int)(t % s->Sq);
    *b = (int)(t / s->Sq);
}

static void *worker(void *arg)
{
    work_t *w = (work_t *)arg;
    const shape_t *s = w->s;
    double *srow = (double *)malloc(sizeof(double) * (size_t)(s->Skv > 0 ? s->Skv : 1));
    if (!srow) { w->status = ORACLE_NO_MEMORY; return NULL; }
    for (long long r = w->first; r < w->last; ++r) {
        int b, hq, i;
        double *orow;
        if (w->rows) {
            b = w->rows[3 * r + 0];
            hq = w->rows[3 * r + 1];
            i = w->rows[3 * r + 2];
            orow = w->out + r * s->hd;
        } else {
            decode_all(s, r, &b, &hq, &i);
            orow = w->out + r * s->hd; /* BSHD row (b, i, hq) is row r */
        }
        attend_row(s, b, hq, i, srow, orow);
    }
    free(srow);
    w->status = ORACLE_OK;
    return NULL;
}

static int run_rows(const shape_t *s, const int32_t *rows, long long n, double *out, int nthreads)
{
    if (n <= 0) return ORACLE_OK;
    if (nthreads < 1) nthreads = 1;
    if ((long long)nthreads > n) nthreads = (int)n;
    work_t *w = (work_t *)calloc((size_t)nthreads, sizeof(work_t));
    pthread_t *t = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!w || !t) { free(w); free(t); return ORACLE_NO_MEMORY; }
    int status = ORACLE_OK;
    for (int x = 0; x < nthreads; ++x) {
        w[x].s = s;
        w[x].rows = rows;
        w[x].first = n * x / nthreads;
        w[x].last = n * (x + 1) / nthreads;
        w[x].out = out;
        w[x].status = ORACLE_OK;
    }
    int started = 0;
    for (int x = 1; x < nthreads; ++x) {
        if (pthread_create(&t[x], NULL, worker, &w[x]) != 0) break;
        started = x;
    }
    worker(&w[0]);
    /* rows of threads that failed to start run on this thread */
    for (int x = started + 1; x < nthreads; ++x) worker(&w[x]);
    for (int x = 1; x <= started; ++x) pthread_join(t[x], NULL);
    for (int x = 0; x < nthreads; ++x)
        if (w[x].status != ORACLE_OK) status = w[x].status;
    free(w);
    free(t);
    return status;
}

/* ------------------------------- entry points ---------------------------- */

/* Full output o[B][Sq][Hq][hd]. */
int oracle_attention(const double *q, const double *k, const double *v, double *o,
                     int B, int Hq, int Hkv, int Sq, int Skv, int hd,
                     int causal, double scale, int nthreads)
{
    shape_t s = {q, k, v, B, Hq, Hkv, Sq, Skv, hd, causal, scale};
    if (!o || check_shape(&s) != ORACLE_OK) return ORACLE_BAD_ARG;
    long long n = (long long)B * Sq * Hq;
    return run_rows(&s, NULL, n, o, nthreads);
}

/* Selected output rows: rows is [n][3] = (b, hq, i); out is [n][hd]. */
int oracle_attention_rows(const double *q, const double *k, const double *v,
                          int B, int Hq, int Hkv, int Sq, int Skv, int hd,
                          int causal, double scale,
                          const int32_t *rows, long long n, double *out, int nthreads)
{
    shape_t s = {q, k, v, B, Hq, Hkv, Sq, Skv, hd, causal, scale};
    if (!out || (n > 0 && !rows) || check_shape(&s) != ORACLE_OK) return ORACLE_BAD_ARG;
    for (long long r = 0; r < n; ++r) {
        if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 || rows[3 * r + 1] >= Hq ||
            rows[3 * r + 2] < 0 || rows[3 * r + 2] >= Sq)
            return ORACLE_BAD_ARG;
    }
    return run_rows(&s, rows, n, out, nthreads);
}

/* The probability row P[b, hq, i, :] (Skv entries), exposed so tests can
 * check it on its own (row sums, zeros under the mask). */
int oracle_probs_row(const double *q, const double *k,
                     int B, int Hq, int Hkv, int Sq, int Skv, int hd,
                     int causal, double scale, int b, int hq, int i, double *p)
{
    shape_t s = {q, k, k, B, Hq, Hkv, Sq, Skv, hd, causal, scale};
    if (!p || check_shape(&s) != ORACLE_OK) return ORACLE_BAD_ARG;
    if (b < 0 || b >= B || hq < 0 || hq >= Hq || i < 0 || i >= Sq) return ORACLE_BAD_ARG;
    double m = score_row(&s, b, hq, i, p);
    softmax_row(p, Skv, m);
    return ORACLE_OK;
}


/* ------------------------------------------------------------------------
 * Per-row log-sum-exp (the natural log of the softmax denominator), the
 * quantity split-KV pieces are combined by -- the pages' running max m and
 * sum l of the online softmax (minfer "53 · r50 — FA_TKV 32->16 occupancy
 * experiment", section 2) taken together: lse = m + log(l):
 *
 *   lse = log sum_j exp(s_j)   over the visible keys j (s_j scaled, masked)
 *   lse = -inf                  when the row sees no key
 *
 * computed as m + log(sum_j exp(s_j - m)) from the same score row as the
 * attention.  rows: [n][3] = (b, hq, i).
 */
int oracle_lse_rows(const double *q, const double *k, int B, int Hq, int Hkv, int Sq, int Skv, int hd,
                    int causal, double scale, const int32_t *rows, long long n, double *lse)
{
    shape_t s = {q, k, k, B, Hq, Hkv, Sq, Skv, hd, causal, scale}; /* v is not read */
    if (!lse || (n > 0 && !rows) || check_shape(&s) != ORACLE_OK) return ORACLE_BAD_ARG;
    double *srow = (double *)malloc(sizeof(double) * (size_t)(Skv > 0 ? Skv : 1));
    if (!srow) return ORACLE_NO_MEMORY;
    for (long long r = 0; r < n; ++r) {
        const int b = rows[3 * r], hq = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || hq < 0 || hq >= Hq || i < 0 || i >= Sq) {
            free(srow);
            return ORACLE_BAD_ARG;
        }
        const double m = score_row(&s, b, hq, i, srow);
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int j = 0; j < Skv; ++j)
            if (srow[j] != -INFINITY) sum += exp(srow[j] - m);
        lse[r] = m + ((g_plant == PLANT_LSE_LOG2) ? log2(sum) : log(sum));
    }
    free(srow);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * K/V-cache append (the step before a chunked prefill's attention: the pages'
 * store_kv kernel, minfer "11 · P5 — prefill gap session: TM=128 big tiles +
 * FA rewrite", section 3.2: an f32 token row is written as 16-bit values at
 * cache row positions[t]):
 *
 *   cache[b][positions[b][t]][h][d] = round16(new[b][t][h][d])   for K and V
 *
 * round16 is IEEE 754 round-to-nearest, ties to even, into binary16 or
 * bfloat16 (8 significant bits, binary32's exponent range).  Written from the
 * definition: |f| is exact in double; it is divided by the spacing (ulp) of
 * the target grid in its binade -- a power of two, so exactly -- rounded to an
 * integer with rint() (ties to even in the default rounding mode) and
 * multiplied back; results above the largest finite value become infinity;
 * NaN stays NaN (quiet); the sign is kept, zeros included.
 */

/* mbits: stored significand bits; ebits: exponent bits. */
static uint16_t round16(float f, int mbits, int ebits)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    const uint16_t sign = (uint16_t)((u >> 31) << 15);
    const int bias = (1 << (ebits - 1)) - 1;
    const int emin = 1 - bias, emax = bias;
    const uint16_t exp_ones = (uint16_t)(((1u << ebits) - 1) << mbits);
    if (isnan(f)) return (uint16_t)(sign | exp_ones | (1u << (mbits - 1)));
    if (isinf(f)) return (uint16_t)(sign | exp_ones);
    const double x = fabs((double)f);
    if (x == 0.0) return sign;
    int e;
    frexp(x, &e);               /* x in [2^(e-1), 2^e) */
    int E = e - 1;              /* binade exponent */
    if (E < emin) E = emin;     /* the subnormal range shares the smallest binade's spacing */
    const double ulp = ldexp(1.0, E - mbits);
    const double t = x / ulp;   /* exact */
    double n;
    if (g_plant == PLANT_ROUND_TRUNCATE) {
        n = floor(t);
    } else if (g_plant == PLANT_ROUND_TIES_AWAY) {
        n = floor(t + 0.5);
    } else {
        n = rint(t);            /* nearest, ties to even */
    }
    const double r = n * ulp;
    const double max_finite = ldexp(2.0 - ldexp(1.0, -mbits), emax);
    if (r > max_finite) return (uint16_t)(sign | exp_ones);
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, emin))   /* subnormal: exponent field 0 */
        return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, emin - mbits)));
    int e2;
    frexp(r, &e2);
    const int E2 = e2 - 1;
    const uint16_t mant = (uint16_t)(r / ldexp(1.0, E2 - mbits) - (double)(1u << mbits));
    return (uint16_t)(sign | (uint16_t)((E2 + bias) << mbits) | mant);
}

uint16_t oracle_round_f16(float f) { return round16(f, 10, 5); }
uint16_t oracle_round_bf16(float f) { return round16(f, 7, 8); }

/* new: [B][T][Hkv][hd] f32; positions: [B][T]; cache: [B][cap][Hkv][hd]
 * 16-bit patterns.  Tokens whose position is outside [0, cap) are skipped;
 * returns the number skipped (>= 0), or -ORACLE_BAD_ARG. */
long long oracle_kv_append(const float *k_new, const float *v_new, const int32_t *positions,
                           uint16_t *k_cache, uint16_t *v_cache,
                           int B, int T, int Hkv, int hd, int cap, int bf16)
{
    if (B < 0 || T < 0 || Hkv < 1 || hd < 1 || cap < 1) return -ORACLE_BAD_ARG;
    const long long row = (long long)Hkv * hd;
    long long skipped = 0;
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < T; ++t) {
            const int pos = (g_plant == PLANT_APPEND_AT_T) ? t : positions[(long long)b * T + t];
            if (pos < 0 || pos >= cap) {
                ++skipped;
                continue;
            }
            const float *ks = k_new + ((long long)b * T + t) * row;
            const float *vs = v_new + ((long long)b * T + t) * row;
            uint16_t *kd = k_cache + ((long long)b * cap + pos) * row;
            uint16_t *vd = v_cache + ((long long)b * cap + pos) * row;
            for (long long x = 0; x < row; ++x) {
                kd[x] = bf16 ? oracle_round_bf16(ks[x]) : oracle_round_f16(ks[x]);
                vd[x] = bf16 ? oracle_round_bf16(vs[x]) : oracle_round_f16(vs[x]);
            }
        }
    }
    return skipped;
}
