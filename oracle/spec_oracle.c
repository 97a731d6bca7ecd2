/*
 * CPU oracle for verification attention in long-context speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path calls this code: it is
 * used by the tests, by smoke() and by the benchmark's CPU-baseline leg. It
 * shares no code, header, table or constant with the CUDA library.
 *
 * Everything is the plain definition, in fp64, row by row:
 *
 *   oracle_select   the hybrid verification-set selection of Dustin
 *                   ("Metodologia", section 1 "Aggregazione Ibrida
 *                   dell'Attenzione"): protect an attention-sink prefix and a
 *                   local window of recent tokens, then fill the remaining
 *                   budget in tiers: the top-m tokens by the draft-lookahead
 *                   score, then the most relevant remaining tokens by the
 *                   target-historical score. Done with a full sort per tier.
 *
 *   oracle_attend   softmax attention of each draft-tree query over the
 *                   concatenation [cache keys ; draft keys] with an explicit
 *                   visibility mask. Cache keys are all tokens of the context
 *                   (full-cache verification, Dustin "Definizione del
 *                   Problema") or only the selected index set (Dustin
 *                   "Workflow di Verifica", steps 3-4). Draft key j is visible
 *                   to node i iff j == i or j is an ancestor of i in the
 *                   draft tree (the tree mask of LongSpec section 2.C). The
 *                   softmax is taken over everything at once: no parts, no
 *                   splits, no merge.
 *
 *   oracle_lse_merge  the log-sum-exp combination of two normalised partial
 *                   attentions (LongSpec section 2.C, "Aggregazione").
 *
 *   oracle_attend_paged  oracle_attend over a paged cache (not on the pages: the
 *                   same cache stored in fixed-size blocks of a pool, found through
 *                   a per-sequence block table). A block entry outside the pool
 *                   hides its tokens and is reported as bad input.
 *
 *   oracle_attend_fp8  oracle_attend over a cache stored as 8-bit floats (not on
 *                   the pages): each K (V) element is an E4M3 code of the OCP 8-bit
 *                   floating-point formats (1 sign bit, 4 exponent bits with bias 7,
 *                   3 mantissa bits; subnormals; no infinities; S.1111.111 is NaN),
 *                   and the cache value is that number times a scale per (sequence,
 *                   KV head), one for K and one for V. The draft block stays bf16.
 *
 * Readings where the pages are silent (also listed in the design notes):
 *   - score comparison: larger is better; -0 == +0; NaN ranks below every
 *     number (including -inf) and NaNs tie; ties go to the lower index.
 *   - a context of n <= budget tokens is verified in full: idx = 0..n-1,
 *     then -1 padding.
 *   - sink/window clip to the context: S' = min(S, n), W' = min(W, n - S').
 *   - the top-m and fill tiers draw only from tokens outside sink and window.
 *   - parent[i] == -1: node i hangs off the last cache token. A parent outside
 *     [-1, i) ends the ancestor walk there and is reported as bad input.
 *   - a sparse index entry is used iff 0 <= idx[j] < n and (j == 0 or
 *     idx[j] > idx[j-1]); -1 entries are padding; any other unused entry is
 *     reported as bad input.
 *   - a row that sees no key at all has lse = -inf and o = 0.
 *   - lse is the natural log of sum exp(scale * q.k).
 *
 * Return value of every function: 0 = ok, 1 = invalid argument,
 * 5 = bad input data seen (the masked/clipped result is still written).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_INVALID_ARG 1
#define ORACLE_BAD_INPUT 5

/* bf16 bits -> exact double */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E4M3 code -> exact double (OCP 8-bit floating point, E4M3):
   exponent field 0: (-1)^s * m/8 * 2^(1-7); 1..15: (-1)^s * (1 + m/8) * 2^(e-7);
   exponent 15 with mantissa 7 is NaN (the format has no infinities). */
static double e4m3_to_double(uint8_t x)
{
    int sgn = x >> 7, e = (x >> 3) & 15, m = x & 7;
    if (e == 15 && m == 7) return NAN;
    double v = e == 0 ? ldexp((double)m / 8.0, 1 - 7) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -v : v;
}

/* ------------------------------------------------------------------------ */
/* selection                                                                 */

typedef struct {
    float score;
    int32_t index;
} scored_token;

/* "a ranks before b": larger score first, NaN last, ties by lower index. */
static int ranks_before(const scored_token *a, const scored_token *b)
{
    int an = isnan(a->score), bn = isnan(b->score);
    if (an && bn) return a->index < b->index;
    if (an) return 0;
    if (bn) return 1;
    if (a->score > b->score) return 1;
    if (a->score < b->score) return 0;
    return a->index < b->index; /* equal, including -0 == +0 */
}

static int cmp_rank(const void *pa, const void *pb)
{
    const scored_token *a = (const scored_token *)pa, *b = (const scored_token *)pb;
    if (ranks_before(a, b)) return -1;
    if (ranks_before(b, a)) return 1;
    return 0;
}

int oracle_select(const float *draft_score, const float *target_score, int64_t ld, int B, int L,
                  const int32_t *ctx_lens, int sink, int window, int top_m, int budget,
                  int32_t *idx, int32_t *count)
{
    if (B < 0 || L < 0 || ld < L || sink < 0 || window < 0 || top_m < 0 || budget < 1 ||
        sink + window > budget || !draft_score || !target_score || !idx)
        return ORACLE_INVALID_ARG;
    int status = ORACLE_OK;
    scored_token *pool = (scored_token *)malloc(sizeof(scored_token) * (size_t)(L > 0 ? L : 1));
    unsigned char *chosen = (unsigned char *)malloc((size_t)(L > 0 ? L : 1));
    for (int b = 0; b < B; ++b) {
        int n = ctx_lens ? ctx_lens[b] : L;
        if (n < 0 || n > L) {
            status = ORACLE_BAD_INPUT;
            n = n < 0 ? 0 : L;
        }
        int32_t *out = idx + (int64_t)b * budget;
        if (budget >= n) { /* the whole context fits: verify in full */
            for (int j = 0; j < budget; ++j) out[j] = j < n ? j : -1;
            if (count) count[b] = n;
            continue;
        }
        const float *ds = draft_score + (int64_t)b * ld;
        const float *ts = target_score + (int64_t)b * ld;
        memset(chosen, 0, (size_t)n);
        int s0 = sink < n ? sink : n;
        int w0 = window < n - s0 ? window : n - s0;
        for (int t = 0; t < s0; ++t) chosen[t] = 1;         /* attention sink */
        for (int t = n - w0; t < n; ++t) chosen[t] = 1;     /* local window   */
        int rest_lo = s0, rest_hi = n - w0, nrest = rest_hi - rest_lo;
        int left = budget - s0 - w0;
        /* tier 1: top-m of the remaining tokens by draft-lookahead score */
        int m = top_m;
        if (m > left) m = left;
        if (m > nrest) m = nrest;
        for (int t = rest_lo; t < rest_hi; ++t) {
            pool[t - rest_lo].score = ds[t];
            pool[t - rest_lo].index = t;
        }
        qsort(pool, (size_t)nrest, sizeof(scored_token), cmp_rank);
        for (int j = 0; j < m; ++j) chosen[pool[j].index] = 1;
        left -= m;
        /* tier 2: fill the rest of the budget by target-historical score */
        int np = 0;
        for (int t = rest_lo; t < rest_hi; ++t) {
            if (chosen[t]) continue;
            pool[np].score = ts[t];
            pool[np].index = t;
            ++np;
        }
        qsort(pool, (size_t)np, sizeof(scored_token), cmp_rank);
        for (int j = 0; j < left && j < np; ++j) chosen[pool[j].index] = 1;
        /* emit ascending */
        int c = 0;
        for (int t = 0; t < n; ++t)
            if (chosen[t]) out[c++] = t;
        for (int j = c; j < budget; ++j) out[j] = -1;
        if (count) count[b] = c;
    }
    free(pool);
    free(chosen);
    return status;
}

/* ------------------------------------------------------------------------ */
/* attention                                                                 */

/* Where the cache rows live. Contiguous (table == NULL): element (b, h, t, c) at
   b*sb + h*sh + t*st + c. Paged (a layout the pages do not use; the same cache stored
   in blocks of a pool): token t of sequence b is row t % block_size of pool block
   table[b*table_ld + t / block_size], element (blk, h, o, c) at blk*sb + h*sh + o*st + c. */
typedef struct {
    int64_t sb, sh, st;
    const int32_t *table;
    int64_t table_ld;
    int block_size;
    int64_t num_blocks;
    /* element format: 0 = bf16; 1 = E4M3 codes, value = code * scale[b * Hkv + h] */
    int fp8;
    const float *k_scale, *v_scale;
} cache_layout;

/* Element c of the cache row at element offset off (K or V), as the exact double it stands for. */
static double cache_value(const cache_layout *cl, const void *base, const float *scale_bh, int64_t off, int c)
{
    if (!cl->fp8) return bf16_to_double(((const uint16_t *)base)[off + c]);
    return e4m3_to_double(((const uint8_t *)base)[off + c]) * (double)*scale_bh;
}

/* Element offset of the row of token t (sequence b, KV head hk); 0 when the row does not
   exist (a block entry outside [0, num_blocks)), else 1. */
static int cache_row(const cache_layout *cl, int b, int hk, int64_t t, int64_t *off)
{
    if (!cl->table) {
        *off = b * cl->sb + hk * cl->sh + t * cl->st;
        return 1;
    }
    int64_t blk = cl->table[b * cl->table_ld + t / cl->block_size];
    if (blk < 0 || blk >= cl->num_blocks) return 0;
    *off = blk * cl->sb + hk * cl->sh + (t % cl->block_size) * cl->st;
    return 1;
}

static int attend_core(const uint16_t *q, const void *k_cache, const void *v_cache,
                       const cache_layout *cl, const uint16_t *k_draft, const uint16_t *v_draft,
                       const int32_t *parent, const int32_t *idx, int budget, int B, int N, int Hq,
                       int Hkv, int d, int L, const int32_t *ctx_lens, float scale, int64_t cache_begin,
                       int64_t cache_end, const int64_t *rows, int64_t n_rows, double *out, double *lse)
{
    if (B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || d < 1 || L < 0 || !q || !out ||
        !lse || !rows || (L > 0 && (!k_cache || !v_cache)) || (idx && budget < 0) ||
        (cl->fp8 && L > 0 && (!cl->k_scale || !cl->v_scale)) ||
        ((k_draft == NULL) != (v_draft == NULL)) || (k_draft && !parent))
        return ORACLE_INVALID_ARG;
    const int G = Hq / Hkv;
    const double sc = (double)scale;
    int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1) reduction(max : status)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t row = rows[r];
        int h = (int)(row % Hq);
        int i = (int)((row / Hq) % N);
        int b = (int)(row / ((int64_t)Hq * N));
        int hk = h / G;
        int n = ctx_lens ? ctx_lens[b] : L;
        if (n < 0 || n > L) {
            status = ORACLE_BAD_INPUT;
            n = n < 0 ? 0 : L;
        }
        const uint16_t *qrow = q + (((int64_t)b * N + i) * Hq + h) * d;

        /* cache keys that are candidates at all, in order */
        int64_t ncache_cand = idx ? budget : n;
        int64_t nkeys = ncache_cand + N;
        unsigned char *visible = (unsigned char *)calloc((size_t)(nkeys > 0 ? nkeys : 1), 1);
        int64_t *coff = (int64_t *)malloc(sizeof(int64_t) * (size_t)(ncache_cand > 0 ? ncache_cand : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(nkeys > 0 ? nkeys : 1));

        /* explicit mask, cache part */
        for (int64_t j = 0; j < ncache_cand; ++j) {
            int64_t t;
            if (idx) {
                const int32_t *ib = idx + (int64_t)b * budget;
                t = ib[j];
                int ok = t >= 0 && t < n && (j == 0 || t > ib[j - 1]);
                if (!ok) {
                    if (t != -1) status = ORACLE_BAD_INPUT;
                    continue;
                }
            } else {
                t = j;
            }
            if (t < cache_begin || t >= cache_end) continue;
            if (!cache_row(cl, b, hk, t, &coff[j])) { /* its block is not in the pool */
                status = ORACLE_BAD_INPUT;
                continue;
            }
            visible[j] = 1;
        }
        /* explicit mask, draft part: node i sees itself and its ancestors */
        if (k_draft) {
            const int32_t *pb = parent + (int64_t)b * N;
            visible[ncache_cand + i] = 1;
            int j = i;
            while (1) {
                int p = pb[j];
                if (p == -1) break;
                if (p < -1 || p >= j) {
                    status = ORACLE_BAD_INPUT;
                    break;
                }
                visible[ncache_cand + p] = 1;
                j = p;
            }
        }

        /* scores over all visible keys */
        const float *ks = cl->fp8 ? cl->k_scale + (int64_t)b * Hkv + hk : NULL;
        const float *vs = cl->fp8 ? cl->v_scale + (int64_t)b * Hkv + hk : NULL;
        double mx = -INFINITY;
        for (int64_t j = 0; j < nkeys; ++j) {
            if (!visible[j]) continue;
            double dot = 0.0;
            if (j < ncache_cand) {
                for (int c = 0; c < d; ++c) dot += bf16_to_double(qrow[c]) * cache_value(cl, k_cache, ks, coff[j], c);
            } else {
                const uint16_t *krow = k_draft + (((int64_t)b * N + (j - ncache_cand)) * Hkv + hk) * d;
                for (int c = 0; c < d; ++c) dot += bf16_to_double(qrow[c]) * bf16_to_double(krow[c]);
            }
            s[j] = sc * dot;
            if (s[j] > mx) mx = s[j];
        }
        double *o = out + r * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        if (mx == -INFINITY) { /* nothing visible */
            lse[r] = -INFINITY;
        } else {
            double sum = 0.0;
            for (int64_t j = 0; j < nkeys; ++j)
                if (visible[j]) sum += exp(s[j] - mx);
            double l = mx + log(sum);
            lse[r] = l;
            for (int64_t j = 0; j < nkeys; ++j) {
                if (!visible[j]) continue;
                double p = exp(s[j] - l);
                if (j < ncache_cand) {
                    for (int c = 0; c < d; ++c) o[c] += p * cache_value(cl, v_cache, vs, coff[j], c);
                } else {
                    const uint16_t *vrow = v_draft + (((int64_t)b * N + (j - ncache_cand)) * Hkv + hk) * d;
                    for (int c = 0; c < d; ++c) o[c] += p * bf16_to_double(vrow[c]);
                }
            }
        }
        free(visible);
        free(coff);
        free(s);
    }
    return status;
}

int oracle_attend(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                  int64_t stride_b, int64_t stride_h, int64_t stride_t,
                  const uint16_t *k_draft, const uint16_t *v_draft, const int32_t *parent,
                  const int32_t *idx, int budget, int B, int N, int Hq, int Hkv, int d, int L,
                  const int32_t *ctx_lens, float scale, int64_t cache_begin, int64_t cache_end,
                  const int64_t *rows, int64_t n_rows, double *out, double *lse)
{
    cache_layout cl = {stride_b, stride_h, stride_t, NULL, 0, 0, 0, 0, NULL, NULL};
    return attend_core(q, k_cache, v_cache, &cl, k_draft, v_draft, parent, idx, budget, B, N, Hq, Hkv, d,
                       L, ctx_lens, scale, cache_begin, cache_end, rows, n_rows, out, lse);
}

/* The same attention over a paged cache: pool strides (elements) for block, KV head and
   row, the block table [B, table_ld], the block size and the number of pool blocks. */
int oracle_attend_paged(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                        int64_t stride_blk, int64_t stride_h, int64_t stride_row, const int32_t *table,
                        int64_t table_ld, int block_size, int64_t num_blocks,
                        const uint16_t *k_draft, const uint16_t *v_draft, const int32_t *parent,
                        const int32_t *idx, int budget, int B, int N, int Hq, int Hkv, int d, int L,
                        const int32_t *ctx_lens, float scale, const int64_t *rows, int64_t n_rows,
                        double *out, double *lse)
{
    if (!table || block_size < 1 || num_blocks < 0 || table_ld < (L + block_size - 1) / block_size)
        return ORACLE_INVALID_ARG;
    cache_layout cl = {stride_blk, stride_h, stride_row, table, table_ld, block_size, num_blocks, 0, NULL, NULL};
    return attend_core(q, k_pool, v_pool, &cl, k_draft, v_draft, parent, idx, budget, B, N, Hq, Hkv, d,
                       L, ctx_lens, scale, 0, L, rows, n_rows, out, lse);
}

/* The same attention over a cache of E4M3 codes (element strides, one byte an element) with
   the K and V scales [B * Hkv] (value = code * scale); the queries and the draft block are bf16. */
int oracle_attend_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                      int64_t stride_b, int64_t stride_h, int64_t stride_t, const float *k_scale,
                      const float *v_scale, const uint16_t *k_draft, const uint16_t *v_draft,
                      const int32_t *parent, const int32_t *idx, int budget, int B, int N, int Hq, int Hkv,
                      int d, int L, const int32_t *ctx_lens, float scale, const int64_t *rows,
                      int64_t n_rows, double *out, double *lse)
{
    cache_layout cl = {stride_b, stride_h, stride_t, NULL, 0, 0, 0, 1, k_scale, v_scale};
    return attend_core(q, k_cache, v_cache, &cl, k_draft, v_draft, parent, idx, budget, B, N, Hq, Hkv, d,
                       L, ctx_lens, scale, 0, L, rows, n_rows, out, lse);
}

/* E4M3 code -> double, for the tests that pin the decoding. */
double oracle_e4m3_value(int code) { return e4m3_to_double((uint8_t)code); }

/* ------------------------------------------------------------------------ */
/* log-sum-exp merge of two normalised parts                                 */

int oracle_lse_merge(const float *o_a, const float *lse_a, const float *o_b, const float *lse_b,
                     int64_t rows, int d, double *out, double *lse_out)
{
    if (rows < 0 || d < 1 || !o_a || !lse_a || !o_b || !lse_b || !out || !lse_out)
        return ORACLE_INVALID_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        double la = lse_a[r], lb = lse_b[r];
        double m = la > lb ? la : lb;
        if (isnan(la) || isnan(lb)) m = NAN;
        double *o = out + r * d;
        if (m == -INFINITY) { /* neither part saw a key */
            lse_out[r] = -INFINITY;
            for (int c = 0; c < d; ++c) o[c] = 0.0;
            continue;
        }
        double l = m + log(exp(la - m) + exp(lb - m));
        double wa = exp(la - l), wb = exp(lb - l);
        lse_out[r] = l;
        for (int c = 0; c < d; ++c) o[c] = wa * (double)o_a[r * d + c] + wb * (double)o_b[r * d + c];
    }
    return ORACLE_OK;
}
