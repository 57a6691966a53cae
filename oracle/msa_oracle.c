/*
 * msa_oracle.c -- the CPU oracle for the block-sparse GQA decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, fp64 statement of
 * what the decode step computes.  It exists so that tests, the smoke check and
 * the CPU-baseline leg of the benchmark can check the CUDA path against it.
 * The product path (the CUDA library) never links, loads or calls it, and it
 * shares no source, header, table or constant with that path.
 *
 * Every routine follows its defining passage step by step, with no blocking,
 * fusion or reordering beyond what the definition states.  Sources:
 *
 *   [SA]   vLLM API page "vllm.models.minimax_m3.common.sparse_attention":
 *          MiniMaxM3SparseBackend (head size 128, page == sparse block == 128,
 *          packed K|V cache shape (num_blocks, Hkv, 128, 2*128) in HND order,
 *          fp8 e4m3 dequantised before the dots) and MiniMaxM3SparseTritonImpl
 *          .forward (q and out viewed as [T, Hq, 128], top-k read per token).
 *   [CUT]  vLLM API page "vllm.models.minimax_m3.nvidia.msa_cutlass_sparse_decode":
 *          MSACutlassDecodePlanCache._build_plan (causal, qo_offset =
 *          kv_lens - qo_lens), msa_cutlass_sparse_decode (K = first 128 of the
 *          content dim, V = last 128; sm_scale, k_scale, v_scale; o_scale 1).
 *   [TEST] vLLM test page "test_minimax_m3_msa_cutlass_sparse_decode.py":
 *          _make_topk (visible tokens = seq_len - Q + j + 1, ascending block
 *          ids, -1 padding), the interleaved-cache test (float8_e4m3fn K|V
 *          concatenated on the content dim, block_table [batch, stride]).
 *   [PR]   TensorRT-LLM PR #17171 "Custom decode kernels for MinimaxM3":
 *          the scorer commit (each block's largest q.k under the causal
 *          mask, stored head, token, block; the selector reads any strides)
 *          and the flash-decoding commit (padding rows are written as zeros).
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes): the group of query head h is g = h / G with G = Hq / Hkv; the
 * selector keeps the current block plus the best k-1 earlier blocks ordered by
 * (score descending, block index ascending), outputs them ascending and pads
 * with -1; rows with pos < 0 are padding rows (scores -inf, top-k all -1,
 * output 0); scores are sm_scale * k_scale * q.k8.
 *
 * Status codes: 0 ok, 1 invalid argument, 2 an index out of range or a
 * duplicated top-k entry, 3 a NaN input.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORC_D 128      /* head size            [SA] get_supported_head_sizes */
#define ORC_PAGE 128   /* tokens per page      [SA] get_supported_kernel_block_sizes */
#define ORC_ROW 256    /* bytes per cached token row: K (128) then V (128) [SA] get_kv_cache_shape */

enum { ORC_OK = 0, ORC_EINVAL = 1, ORC_ERANGE = 2, ORC_ENAN = 3 };

/* ------------------------------------------------------------------------ */
/* Number decoding                                                           */
/* ------------------------------------------------------------------------ */

/* OCP fp8 E4M3 ("fn" variant, as torch.float8_e4m3fn): 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent 0 is subnormal; S.1111.111 is
 * NaN; there is no infinity, so the largest magnitude is 448. */
double orc_e4m3_to_f64(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);               /* (m/8) * 2^(1-7) */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* The 256 E4M3 values, filled once from orc_e4m3_to_f64 above. */
static double orc_e4m3_table[256];
static pthread_once_t orc_e4m3_once = PTHREAD_ONCE_INIT;

static void orc_e4m3_fill(void)
{
    for (int c = 0; c < 256; ++c)
        orc_e4m3_table[c] = orc_e4m3_to_f64((uint8_t)c);
}

static double orc_e4m3(uint8_t code)
{
    return orc_e4m3_table[code];
}

/* bfloat16 is the top half of an IEEE binary32 word. */
double orc_bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Problem description shared by the three stages                            */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q;          /* [T, Hq, 128] bf16 bits, T = B*Q, token i = b*Q + j */
    const uint8_t *kv;          /* [NB, Hkv, 128, 256] fp8 e4m3 codes */
    const int32_t *block_table; /* [B, S] */
    const int32_t *seq_lens;    /* [B] */
    int B, Q, Hq, Hkv, S;
    int64_t NB;
    double sm_scale, k_scale, v_scale;
} orc_problem;

/* Causal position of query token j of request b: the query rows are the last
 * Q tokens of the sequence, so the causal offset is seq_len - Q ([CUT]
 * _build_plan qo_offset; [TEST] _make_topk visible tokens). */
static int64_t orc_pos(const orc_problem *p, int b, int j)
{
    return (int64_t)p->seq_lens[b] - p->Q + j;
}

/* K[d] and V[d] of token t of logical block n of request b, KV head g, with
 * the per-tensor scale applied ([CUT] key/value = kv_cache.split(128, -1)). */
static double orc_key(const orc_problem *p, int64_t page, int g, int t, int d)
{
    const uint8_t *row = p->kv + ((page * p->Hkv + g) * ORC_PAGE + t) * (int64_t)ORC_ROW;
    return orc_e4m3(row[d]) * p->k_scale;
}

static double orc_value(const orc_problem *p, int64_t page, int g, int t, int d)
{
    const uint8_t *row = p->kv + ((page * p->Hkv + g) * ORC_PAGE + t) * (int64_t)ORC_ROW;
    return orc_e4m3(row[ORC_D + d]) * p->v_scale;
}

static double orc_query(const orc_problem *p, int i, int h, int d)
{
    return orc_bf16_to_f64(p->q[((int64_t)i * p->Hq + h) * ORC_D + d]);
}

/* Logit of query (i, h) against key t of physical page `page` ([CUT]
 * sm_scale applied to q.k). */
static double orc_logit(const orc_problem *p, int i, int h, int64_t page, int g, int t)
{
    double acc = 0.0;
    for (int d = 0; d < ORC_D; ++d)
        acc += orc_query(p, i, h, d) * orc_key(p, page, g, t, d);
    return p->sm_scale * acc;
}

static int orc_check_problem(const orc_problem *p)
{
    pthread_once(&orc_e4m3_once, orc_e4m3_fill);
    if (!p->q || !p->kv || !p->block_table || !p->seq_lens)
        return ORC_EINVAL;
    if (p->B < 0 || p->Q < 1 || p->Hkv < 1 || p->Hq < 1 || p->Hq % p->Hkv != 0 || p->S < 0 || p->NB < 0)
        return ORC_EINVAL;
    for (int b = 0; b < p->B; ++b) {
        if (p->seq_lens[b] < 0)
            return ORC_EINVAL;
        if (p->seq_lens[b] > 0 && (int64_t)(p->seq_lens[b] - 1) / ORC_PAGE >= p->S)
            return ORC_ERANGE;  /* the block table row cannot hold the sequence */
    }
    return ORC_OK;
}

/* Physical page of logical block n of request b ([TEST] block_table[b, n]). */
static int orc_page(const orc_problem *p, int b, int64_t n, int64_t *page)
{
    int32_t v = p->block_table[(int64_t)b * p->S + n];
    if (v < 0 || v >= p->NB)
        return ORC_ERANGE;
    *page = v;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Thread pool: a plain parallel-for over independent work items              */
/* ------------------------------------------------------------------------ */

typedef int (*orc_item_fn)(void *ctx, int64_t item);

typedef struct {
    orc_item_fn fn;
    void *ctx;
    int64_t n_items;
    int64_t next;
    int status;
    pthread_mutex_t lock;
} orc_pool;

static void *orc_worker(void *arg)
{
    orc_pool *pool = (orc_pool *)arg;
    for (;;) {
        int64_t item;
        pthread_mutex_lock(&pool->lock);
        item = pool->next++;
        pthread_mutex_unlock(&pool->lock);
        if (item >= pool->n_items)
            break;
        int st = pool->fn(pool->ctx, item);
        if (st != ORC_OK) {
            pthread_mutex_lock(&pool->lock);
            if (pool->status == ORC_OK)
                pool->status = st;
            pthread_mutex_unlock(&pool->lock);
        }
    }
    return NULL;
}

int orc_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int orc_parallel_for(orc_item_fn fn, void *ctx, int64_t n_items, int nthreads)
{
    orc_pool pool;
    pool.fn = fn;
    pool.ctx = ctx;
    pool.n_items = n_items;
    pool.next = 0;
    pool.status = ORC_OK;
    pthread_mutex_init(&pool.lock, NULL);
    if (nthreads <= 0)
        nthreads = orc_default_threads();
    if (nthreads > n_items)
        nthreads = (int)(n_items > 0 ? n_items : 1);
    if (nthreads <= 1) {
        orc_worker(&pool);
    } else {
        pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        int started = 0;
        for (int k = 0; k < nthreads; ++k)
            if (pthread_create(&tid[k], NULL, orc_worker, &pool) == 0)
                ++started;
        if (started == 0)
            orc_worker(&pool);
        for (int k = 0; k < started; ++k)
            pthread_join(tid[k], NULL);
        free(tid);
    }
    pthread_mutex_destroy(&pool.lock);
    return pool.status;
}

/* ------------------------------------------------------------------------ */
/* Stage 1: block scores                                                     */
/* ------------------------------------------------------------------------ */
/* [PR] scorer commit: for each KV head g, query token i and KV block n, the
 * causal max of the scaled Q.K over the query heads of g's group and over the
 * keys of block n that token i may see:
 *
 *   s[g, i, n] = max_{h in group g, t : 128 n + t <= pos(i)} sm_scale * q[i,h] . K[n,g,t]
 *
 * with K already multiplied by k_scale.  Blocks past the token's current block
 * (n > floor(pos/128)) and every block of a padding row (pos < 0) get -inf.
 * Output layout [Hkv, T, S] (the scorer's [head, token, block] order). */

typedef struct {
    const orc_problem *p;
    double *scores;
} orc_score_ctx;

static int orc_score_item(void *vctx, int64_t item)
{
    orc_score_ctx *c = (orc_score_ctx *)vctx;
    const orc_problem *p = c->p;
    int G = p->Hq / p->Hkv;
    int b = (int)(item / p->Hkv);
    int g = (int)(item % p->Hkv);
    for (int j = 0; j < p->Q; ++j) {
        int i = b * p->Q + j;
        int64_t pos = orc_pos(p, b, j);
        double *row = c->scores + ((int64_t)g * p->B * p->Q + i) * p->S;
        for (int64_t n = 0; n < p->S; ++n)
            row[n] = -INFINITY;
        if (pos < 0)
            continue;
        int64_t cur = pos / ORC_PAGE;
        for (int64_t n = 0; n <= cur; ++n) {
            int64_t page;
            int st = orc_page(p, b, n, &page);
            if (st != ORC_OK)
                return st;
            double best = -INFINITY;
            for (int hh = 0; hh < G; ++hh) {
                int h = g * G + hh;
                for (int t = 0; t < ORC_PAGE; ++t) {
                    if (n * ORC_PAGE + t > pos)
                        break;
                    double z = orc_logit(p, i, h, page, g, t);
                    if (isnan(z))
                        return ORC_ENAN;
                    if (z > best)
                        best = z;
                }
            }
            row[n] = best;
        }
    }
    return ORC_OK;
}

int orc_score(const uint16_t *q, const uint8_t *kv, const int32_t *block_table,
              const int32_t *seq_lens, double *scores, int B, int Q, int Hq, int Hkv,
              int S, int64_t NB, double sm_scale, double k_scale, int nthreads)
{
    orc_problem p = {q, kv, block_table, seq_lens, B, Q, Hq, Hkv, S, NB, sm_scale, k_scale, 1.0};
    int st = orc_check_problem(&p);
    if (st != ORC_OK)
        return st;
    if (!scores)
        return ORC_EINVAL;
    orc_score_ctx c = {&p, scores};
    return orc_parallel_for(orc_score_item, &c, (int64_t)B * Hkv, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Stage 2: block selection                                                  */
/* ------------------------------------------------------------------------ */
/* For each (token i, KV head g) with pos(i) >= 0 and cur = floor(pos/128):
 *   - if cur + 1 <= k, every block 0..cur is kept ([TEST] _make_topk keeps
 *     every visible page when there are at most TOPK of them);
 *   - otherwise the current block cur is kept, plus the k-1 best blocks of
 *     0..cur-1 in the order (score descending, block index ascending).
 * The kept ids are written ascending, then -1 up to k ([TEST] _make_topk:
 * ascending arange, -1 fill).  Padding rows get k times -1.
 * Scores are read through arbitrary element strides ([PR] the selector takes
 * arbitrary strides).  Output layout [T, Hkv, k] ([CUT] token-major topk). */

typedef struct {
    double score;
    int64_t block;
} orc_cand;

static int orc_cand_better_first(const void *a, const void *b)
{
    const orc_cand *x = (const orc_cand *)a, *y = (const orc_cand *)b;
    if (x->score > y->score)
        return -1;
    if (x->score < y->score)
        return 1;
    return (x->block < y->block) ? -1 : (x->block > y->block) ? 1 : 0;
}

static int orc_int64_ascending(const void *a, const void *b)
{
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return (x < y) ? -1 : (x > y) ? 1 : 0;
}

int orc_topk(const double *scores, int64_t stride_h, int64_t stride_t, int64_t stride_n,
             const int32_t *seq_lens, int32_t *topk, int B, int Q, int Hkv, int S, int k)
{
    if (!scores || !seq_lens || !topk || B < 0 || Q < 1 || Hkv < 1 || S < 0 || k < 1)
        return ORC_EINVAL;
    orc_cand *cand = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)(S > 0 ? S : 1));
    int64_t *kept = (int64_t *)malloc(sizeof(int64_t) * (size_t)k);
    int status = ORC_OK;
    for (int b = 0; b < B && status == ORC_OK; ++b) {
        for (int j = 0; j < Q && status == ORC_OK; ++j) {
            int i = b * Q + j;
            int64_t pos = (int64_t)seq_lens[b] - Q + j;
            for (int g = 0; g < Hkv; ++g) {
                int32_t *out = topk + ((int64_t)i * Hkv + g) * k;
                for (int e = 0; e < k; ++e)
                    out[e] = -1;
                if (pos < 0)
                    continue;
                int64_t cur = pos / ORC_PAGE;
                if (cur >= S) {
                    status = ORC_ERANGE;
                    break;
                }
                int n_kept = 0;
                if (cur + 1 <= k) {
                    for (int64_t n = 0; n <= cur; ++n)
                        kept[n_kept++] = n;
                } else {
                    for (int64_t n = 0; n < cur; ++n) {
                        double s = scores[g * stride_h + (int64_t)i * stride_t + n * stride_n];
                        if (isnan(s)) {
                            status = ORC_ENAN;
                            break;
                        }
                        cand[n].score = s;
                        cand[n].block = n;
                    }
                    if (status != ORC_OK)
                        break;
                    qsort(cand, (size_t)cur, sizeof(orc_cand), orc_cand_better_first);
                    for (int e = 0; e < k - 1; ++e)
                        kept[n_kept++] = cand[e].block;
                    kept[n_kept++] = cur;
                    qsort(kept, (size_t)n_kept, sizeof(int64_t), orc_int64_ascending);
                }
                for (int e = 0; e < n_kept; ++e)
                    out[e] = (int32_t)kept[e];
            }
        }
    }
    free(cand);
    free(kept);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Stage 3: attention over the selected blocks                               */
/* ------------------------------------------------------------------------ */
/* For each query row (i, h), g = h / G: the key set is every token t of every
 * listed block n (entries -1 skipped) with 128 n + t <= pos(i).  The output is
 * the softmax-weighted mean of the values:
 *
 *   z_t = sm_scale * q[i,h] . K_t,   O = sum_t exp(z_t - M) V_t / sum_t exp(z_t - M)
 *
 * with M = max_t z_t (the usual max-subtracted two-pass form), K scaled by
 * k_scale and V by v_scale, no softcap, sink or output scale ([CUT]
 * o_scale = 1.0).  An empty key set or a padding row gives O = 0 ([PR]
 * flash-decoding commit: such rows are written as zeros).  A listed block outside
 * [0, cur] or listed twice is a precondition violation (status 2). */

typedef struct {
    const orc_problem *p;
    const int32_t *topk;
    int k;
    double *out;
} orc_attend_ctx;

/* One query row: item = i * Hq + h, result written to o[0..127]. */
static int orc_attend_row(const orc_attend_ctx *c, int64_t item, double *o)
{
    const orc_problem *p = c->p;
    int G = p->Hq / p->Hkv;
    int i = (int)(item / p->Hq);
    int h = (int)(item % p->Hq);
    int b = i / p->Q, j = i % p->Q;
    int g = h / G;
    int64_t pos = orc_pos(p, b, j);
    for (int d = 0; d < ORC_D; ++d)
        o[d] = 0.0;
    if (pos < 0)
        return ORC_OK;
    int64_t cur = pos / ORC_PAGE;
    const int32_t *list = c->topk + ((int64_t)i * p->Hkv + g) * c->k;

    /* validate the list and resolve its pages */
    int64_t *pages = (int64_t *)malloc(sizeof(int64_t) * (size_t)c->k);
    for (int e = 0; e < c->k; ++e) {
        int32_t n = list[e];
        if (n == -1)
            continue;
        if (n < 0 || n > cur) {
            free(pages);
            return ORC_ERANGE;
        }
        for (int e2 = 0; e2 < e; ++e2)
            if (list[e2] == n) {
                free(pages);
                return ORC_ERANGE;
            }
        int st = orc_page(p, b, n, &pages[e]);
        if (st != ORC_OK) {
            free(pages);
            return st;
        }
    }

    /* pass 1: the maximum logit */
    double M = -INFINITY;
    int64_t n_keys = 0;
    for (int e = 0; e < c->k; ++e) {
        int32_t n = list[e];
        if (n == -1)
            continue;
        for (int t = 0; t < ORC_PAGE && (int64_t)n * ORC_PAGE + t <= pos; ++t) {
            double z = orc_logit(p, i, h, pages[e], g, t);
            if (isnan(z)) {
                free(pages);
                return ORC_ENAN;
            }
            if (z > M)
                M = z;
            ++n_keys;
        }
    }
    if (n_keys == 0) {
        free(pages);
        return ORC_OK;
    }

    /* pass 2: weights, their sum and the weighted sum of values */
    double denom = 0.0;
    for (int e = 0; e < c->k; ++e) {
        int32_t n = list[e];
        if (n == -1)
            continue;
        for (int t = 0; t < ORC_PAGE && (int64_t)n * ORC_PAGE + t <= pos; ++t) {
            double w = exp(orc_logit(p, i, h, pages[e], g, t) - M);
            denom += w;
            for (int d = 0; d < ORC_D; ++d)
                o[d] += w * orc_value(p, pages[e], g, t, d);
        }
    }
    for (int d = 0; d < ORC_D; ++d)
        o[d] /= denom;
    free(pages);
    return ORC_OK;
}

static int orc_attend_item(void *vctx, int64_t item)
{
    orc_attend_ctx *c = (orc_attend_ctx *)vctx;
    return orc_attend_row(c, item, c->out + item * ORC_D);
}

int orc_attend(const uint16_t *q, const uint8_t *kv, const int32_t *block_table,
               const int32_t *seq_lens, const int32_t *topk, double *out, int B, int Q,
               int Hq, int Hkv, int S, int64_t NB, int k, double sm_scale, double k_scale,
               double v_scale, int nthreads)
{
    orc_problem p = {q, kv, block_table, seq_lens, B, Q, Hq, Hkv, S, NB, sm_scale, k_scale, v_scale};
    int st = orc_check_problem(&p);
    if (st != ORC_OK)
        return st;
    if (!topk || !out || k < 1)
        return ORC_EINVAL;
    orc_attend_ctx c = {&p, topk, k, out};
    return orc_parallel_for(orc_attend_item, &c, (int64_t)B * Q * Hq, nthreads);
}

/* Attention of a subset of query rows only: rows[r] = i * Hq + h.  Used for
 * sampled checks at sizes where the full problem is too slow. */
typedef struct {
    orc_attend_ctx base;
    const int64_t *rows;
    double *out_rows;
} orc_attend_rows_ctx;

static int orc_attend_rows_item(void *vctx, int64_t r)
{
    orc_attend_rows_ctx *c = (orc_attend_rows_ctx *)vctx;
    return orc_attend_row(&c->base, c->rows[r], c->out_rows + r * ORC_D);
}

int orc_attend_rows(const uint16_t *q, const uint8_t *kv, const int32_t *block_table,
                    const int32_t *seq_lens, const int32_t *topk, const int64_t *rows,
                    int64_t n_rows, double *out_rows, int B, int Q, int Hq, int Hkv, int S,
                    int64_t NB, int k, double sm_scale, double k_scale, double v_scale,
                    int nthreads)
{
    orc_problem p = {q, kv, block_table, seq_lens, B, Q, Hq, Hkv, S, NB, sm_scale, k_scale, v_scale};
    int st = orc_check_problem(&p);
    if (st != ORC_OK)
        return st;
    if (!topk || !rows || !out_rows || k < 1 || n_rows < 0)
        return ORC_EINVAL;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= (int64_t)B * Q * Hq)
            return ORC_EINVAL;
    orc_attend_rows_ctx c;
    c.base.p = &p;
    c.base.topk = topk;
    c.base.k = k;
    c.base.out = NULL;
    c.rows = rows;
    c.out_rows = out_rows;
    return orc_parallel_for(orc_attend_rows_item, &c, n_rows, nthreads);
}

/* Scores of a subset of (request, KV head) units only: units[u] = b * Hkv + g.
 * Rows of other units are left untouched. */
typedef struct {
    orc_score_ctx base;
    const int64_t *units;
} orc_score_units_ctx;

static int orc_score_units_item(void *vctx, int64_t u)
{
    orc_score_units_ctx *c = (orc_score_units_ctx *)vctx;
    return orc_score_item(&c->base, c->units[u]);
}

int orc_score_units(const uint16_t *q, const uint8_t *kv, const int32_t *block_table,
                    const int32_t *seq_lens, double *scores, const int64_t *units,
                    int64_t n_units, int B, int Q, int Hq, int Hkv, int S, int64_t NB,
                    double sm_scale, double k_scale, int nthreads)
{
    orc_problem p = {q, kv, block_table, seq_lens, B, Q, Hq, Hkv, S, NB, sm_scale, k_scale, 1.0};
    int st = orc_check_problem(&p);
    if (st != ORC_OK)
        return st;
    if (!scores || !units || n_units < 0)
        return ORC_EINVAL;
    for (int64_t u = 0; u < n_units; ++u)
        if (units[u] < 0 || units[u] >= (int64_t)B * Hkv)
            return ORC_EINVAL;
    orc_score_units_ctx c;
    c.base.p = &p;
    c.base.scores = scores;
    c.units = units;
    return orc_parallel_for(orc_score_units_item, &c, n_units, nthreads);
}

/* Scores of listed blocks only: triples[3u..3u+2] = (b, g, n); writes
 * scores[g, b*Q + j, n] for every token j of request b, by the same definition
 * as orc_score.  Used for sampled checks at sizes where whole rows are slow. */
typedef struct {
    const orc_problem *p;
    double *scores;
    const int64_t *triples;
} orc_score_blocks_ctx;

static int orc_score_blocks_item(void *vctx, int64_t u)
{
    orc_score_blocks_ctx *c = (orc_score_blocks_ctx *)vctx;
    const orc_problem *p = c->p;
    int G = p->Hq / p->Hkv;
    int b = (int)c->triples[3 * u], g = (int)c->triples[3 * u + 1];
    int64_t n = c->triples[3 * u + 2];
    for (int j = 0; j < p->Q; ++j) {
        int i = b * p->Q + j;
        int64_t pos = orc_pos(p, b, j);
        double *slot = c->scores + ((int64_t)g * p->B * p->Q + i) * p->S + n;
        *slot = -INFINITY;
        if (pos < 0 || n > pos / ORC_PAGE)
            continue;
        int64_t page;
        int st = orc_page(p, b, n, &page);
        if (st != ORC_OK)
            return st;
        double best = -INFINITY;
        for (int hh = 0; hh < G; ++hh) {
            int h = g * G + hh;
            for (int t = 0; t < ORC_PAGE; ++t) {
                if (n * ORC_PAGE + t > pos)
                    break;
                double z = orc_logit(p, i, h, page, g, t);
                if (isnan(z))
                    return ORC_ENAN;
                if (z > best)
                    best = z;
            }
        }
        *slot = best;
    }
    return ORC_OK;
}

int orc_score_blocks(const uint16_t *q, const uint8_t *kv, const int32_t *block_table,
                     const int32_t *seq_lens, double *scores, const int64_t *triples,
                     int64_t n_triples, int B, int Q, int Hq, int Hkv, int S, int64_t NB,
                     double sm_scale, double k_scale, int nthreads)
{
    orc_problem p = {q, kv, block_table, seq_lens, B, Q, Hq, Hkv, S, NB, sm_scale, k_scale, 1.0};
    int st = orc_check_problem(&p);
    if (st != ORC_OK)
        return st;
    if (!scores || !triples || n_triples < 0)
        return ORC_EINVAL;
    for (int64_t u = 0; u < n_triples; ++u) {
        const int64_t *t = triples + 3 * u;
        if (t[0] < 0 || t[0] >= B || t[1] < 0 || t[1] >= Hkv || t[2] < 0 || t[2] >= S)
            return ORC_EINVAL;
    }
    orc_score_blocks_ctx c = {&p, scores, triples};
    return orc_parallel_for(orc_score_blocks_item, &c, n_triples, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Split-softmax merge                                                       */
/* ------------------------------------------------------------------------ */
/* Merging softmax-weighted sums computed over disjoint key subsets
 * ([PR] flash-decoding commit: fp32 split-K partials).  Part s of row r holds
 * the running maximum m_s (in log2 units, i.e. of z * log2(e)), the weight sum
 * l_s = sum 2^(z log2e - m_s) and the unnormalised value sum
 * o_s = sum 2^(z log2e - m_s) V.  The merged row is
 *
 *   M = max_s m_s,  O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,
 *
 * and 0 when every part is empty (sum of l_s == 0).
 * Layout: o [splits, rows, 128], ml [splits, rows, 2] (m then l). */
int orc_combine(const double *o, const double *ml, double *out, int64_t rows, int splits)
{
    if (!o || !ml || !out || rows < 0 || splits < 1)
        return ORC_EINVAL;
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int s = 0; s < splits; ++s) {
            double l = ml[((int64_t)s * rows + r) * 2 + 1];
            double m = ml[((int64_t)s * rows + r) * 2 + 0];
            if (l > 0.0 && m > M)
                M = m;
        }
        double denom = 0.0;
        double acc[ORC_D];
        for (int d = 0; d < ORC_D; ++d)
            acc[d] = 0.0;
        for (int s = 0; s < splits; ++s) {
            double l = ml[((int64_t)s * rows + r) * 2 + 1];
            double m = ml[((int64_t)s * rows + r) * 2 + 0];
            if (!(l > 0.0))
                continue;
            double w = exp2(m - M);
            denom += w * l;
            for (int d = 0; d < ORC_D; ++d)
                acc[d] += w * o[((int64_t)s * rows + r) * ORC_D + d];
        }
        for (int d = 0; d < ORC_D; ++d)
            out[r * ORC_D + d] = denom > 0.0 ? acc[d] / denom : 0.0;
    }
    return ORC_OK;
}
