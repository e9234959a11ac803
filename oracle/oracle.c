/*
 * oracle.c -- plain, slow, float64 CPU oracle for block-sparse top-k GQA
 * attention.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the product library never does.  It
 * shares no code, header or table with the CUDA path.
 *
 * What it follows (MSA sparse attention pages):
 *   - test_sparse_atten.py, sparse_attention_ref: a query row attends to the
 *     union of the 128-token KV blocks named by its top-k list (entries < 0
 *     are padding), keys past the used KV length are masked, optional
 *     bottom-right causal masking keeps key t iff t <= s + (kv_len - Sq), the
 *     scores are (q * scale) . k, LSE = logsumexp of the visible scores
 *     (natural log) and a row that sees no key gets O = 0, LSE = -inf.
 *   - GQA: query head hq reads KV head hq / (Hq / Hkv) (repeat_interleave).
 *   - test_sparse_atten.py, _decode_paged_kv_chunk / pack_paged_kv: paged
 *     KV, logical block j of sequence b lives in physical page
 *     page_table[b][j]; here the pool layout is [num_pages][page][Hkv][D].
 *   - interface.py module docstring and build_k2q_csr call sites: the k->q
 *     CSR (row_ptr [Hkv][rows+1], q_indices [Hkv][total_q*topk]) and the
 *     scheduler test (test_scheduler_builds_packed_qsplit_metadata): qsplit
 *     packs q | split << 24 and a query's split ids are 0..count-1.
 *   - varlen batches (interface.py sparse_atten_func: cu_seqlens_q/k, q2k
 *     [Hkv][total_q][topK]; test_sparse_atten.py _reference_varlen_forward:
 *     each sequence is its own batch-1 problem), the temperature LSE
 *     (sparse_attention_ref, lse_temperature_scale branch) and the dense
 *     decode selection (sparse_decode_atten_func, q2k_indices = None).
 *   - NVFP4 (interface.py sparse_atten_nvfp4_kv_func docstring; vLLM
 *     sparse-MLA test page, _E2M1_TABLE and unpack_e2m1): e2m1 codes with
 *     magnitudes {0,.5,1,1.5,2,3,4,6}, bit 3 the sign, element 2i in the low
 *     nibble, one e4m3 scale per 16 elements along D, x = value * scale.
 *
 * Readings where the pages are silent (also listed in the design notes):
 *   - a block id >= the number of allocated blocks is padding;
 *   - a block named twice by one query counts once (the golden reference
 *     builds a boolean block mask, so duplicates collapse);
 *   - the CSR lists the queries of a row in ascending global query id, and a
 *     query's split id for a block is the number of earlier distinct valid
 *     slots;
 *   - the NVFP4 group scale is e4m3_rne(amax / 6) and a code is
 *     e2m1_rne_satfinite(x / scale); an all-zero group has scale 0, codes 0.
 *
 * Build: gcc -O2 -shared -fPIC -pthread oracle.c -lm -o liboracle.so
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---------------------------------------------------------------------- */
/* scalar formats                                                          */
/* ---------------------------------------------------------------------- */

/* bf16 bits -> double, exact (bf16 is the top half of an IEEE binary32). */
static double bf16_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_bf16_to_double(uint16_t h) { return bf16_to_double(h); }

/* e4m3 (fn variant: bias 7, no infinities, 0x7f / 0xff are NaN) -> double */
double oracle_e4m3_to_double(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);            /* subnormal: m * 2^-6 / 8 */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* double (finite, >= 0) -> e4m3 with round-to-nearest-even, saturating at 448. */
uint8_t oracle_e4m3_from_double_rne_sat(double x) {
    if (!(x > 0.0)) return 0;
    if (x >= 448.0) return 0x7E;                     /* 1.75 * 2^8 */
    int e;
    frexp(x, &e);                                    /* x = f * 2^e, f in [0.5,1) */
    int unbiased = e - 1;                            /* x in [2^u, 2^(u+1)) */
    double quantum = (unbiased < -6) ? ldexp(1.0, -9) : ldexp(1.0, unbiased - 3);
    double r = nearbyint(x / quantum);               /* ties to even (default mode) */
    double val = r * quantum;
    if (val > 448.0) val = 448.0;
    if (val == 0.0) return 0;
    /* encode val */
    frexp(val, &e);
    unbiased = e - 1;
    if (unbiased < -6) {                             /* subnormal */
        int m = (int)(val / ldexp(1.0, -9));
        return (uint8_t)m;
    }
    int m = (int)(val / ldexp(1.0, unbiased) * 8.0) - 8;
    return (uint8_t)(((unbiased + 7) << 3) | m);
}

/* magnitude grid of e2m1, code & 7 */
static const double kE2m1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_to_double(uint8_t code) {
    double v = kE2m1[code & 7];
    return (code & 8) ? -v : v;
}

/* x -> e2m1 code, round to nearest with ties to the even code, saturating at 6. */
uint8_t oracle_e2m1_from_double_rne_sat(double x) {
    uint8_t sign = 0;
    if (x < 0) { sign = 8; x = -x; }
    if (!(x == x)) return 0;                         /* NaN: not produced by the quantiser */
    int best = 0;
    for (int c = 1; c < 8; ++c) {
        double dc = fabs(kE2m1[c] - x), db = fabs(kE2m1[best] - x);
        if (dc < db || (dc == db && (c & 1) == 0 && (best & 1) == 1)) best = c;
    }
    if (x >= 6.0) best = 7;
    return (uint8_t)(sign | best);
}

/* ---------------------------------------------------------------------- */
/* thread helper                                                           */
/* ---------------------------------------------------------------------- */

int oracle_default_threads(void) {
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof set, &set) == 0) {
        int n = CPU_COUNT(&set);
        if (n > 0) return n;
    }
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

typedef void (*work_fn)(void *ctx, int64_t item);

typedef struct {
    work_fn fn;
    void *ctx;
    int64_t n;
    int tid, nthreads;
} span_t;

static void *run_span(void *p) {
    span_t *s = (span_t *)p;
    for (int64_t i = s->tid; i < s->n; i += s->nthreads) s->fn(s->ctx, i);
    return NULL;
}

/* Run fn(ctx, i) for i in [0, n) on nthreads threads; returns threads used. */
static int parallel_for(int64_t n, int nthreads, work_fn fn, void *ctx) {
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > n) nthreads = n > 0 ? (int)n : 1;
    if (nthreads == 1) {
        for (int64_t i = 0; i < n; ++i) fn(ctx, i);
        return 1;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    span_t *sp = (span_t *)malloc(sizeof(span_t) * nthreads);
    for (int t = 0; t < nthreads; ++t) {
        sp[t].fn = fn; sp[t].ctx = ctx; sp[t].n = n; sp[t].tid = t; sp[t].nthreads = nthreads;
        pthread_create(&th[t], NULL, run_span, &sp[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    free(sp);
    return nthreads;
}

/* ---------------------------------------------------------------------- */
/* sparse attention                                                        */
/* ---------------------------------------------------------------------- */

typedef struct {
    /* query side */
    const uint16_t *q;        /* [B*Sq][Hq][D] (bf16 bits) */
    const int32_t *q2k;       /* [B][Hkv][Sq][topk] */
    int B, Sq, Hq, Hkv, D, blk, topk, causal;
    double scale;
    /* KV side: dense [B][Skv][Hkv][D] when page_table == NULL,
       else pool [num_pages][blk][Hkv][D] addressed through page_table [B][max_pages] */
    const uint16_t *k, *v;
    int Skv;                  /* dense: tokens per sequence; paged: max_pages * blk */
    const int32_t *page_table;
    int max_pages;
    const int32_t *seqused;   /* [B] or NULL -> Skv */
    /* which queries */
    const int64_t *rows;      /* global query ids (b*Sq + s) or NULL -> all */
    int64_t nrows;
    /* outputs, indexed by position in rows */
    double *o;                /* [nrows][Hq][D] */
    double *lse;              /* [nrows][Hq] */
} attn_ctx;

static const uint16_t *kv_row(const attn_ctx *c, const uint16_t *base, int b, int h, int64_t t) {
    if (c->page_table) {
        int64_t page = c->page_table[(int64_t)b * c->max_pages + t / c->blk];
        int64_t off = t % c->blk;
        return base + (((page * c->blk + off) * c->Hkv + h) * (int64_t)c->D);
    }
    return base + ((((int64_t)b * c->Skv + t) * c->Hkv + h) * (int64_t)c->D);
}

/* One (query row, KV head) item: computes the qpk query heads of that group. */
static void attn_item(void *vctx, int64_t item) {
    const attn_ctx *c = (const attn_ctx *)vctx;
    int64_t ri = item / c->Hkv;
    int h = (int)(item % c->Hkv);
    int64_t gq = c->rows ? c->rows[ri] : ri;
    int b = (int)(gq / c->Sq);
    int s = (int)(gq % c->Sq);
    int qpk = c->Hq / c->Hkv;
    int D = c->D;
    int nblk_alloc = (c->Skv + c->blk - 1) / c->blk;
    int64_t kv_len = c->seqused ? c->seqused[b] : c->Skv;

    /* 1. the set J of distinct valid block ids named by this query */
    const int32_t *sel = c->q2k + (((int64_t)b * c->Hkv + h) * c->Sq + s) * c->topk;
    int J[64];
    int nJ = 0;
    for (int t = 0; t < c->topk; ++t) {
        int j = sel[t];
        if (j < 0 || j >= nblk_alloc) continue;      /* padding / out of range */
        int dup = 0;
        for (int u = 0; u < nJ; ++u) dup |= (J[u] == j);
        if (!dup) J[nJ++] = j;
    }

    /* 2. visible tokens: union of the blocks, below kv_len, causal limit */
    int64_t limit = kv_len - 1;
    if (c->causal) {
        int64_t cl = (int64_t)s + (kv_len - c->Sq);
        if (cl < limit) limit = cl;
    }
    int64_t maxtok = (int64_t)nJ * c->blk;
    int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (maxtok > 0 ? maxtok : 1));
    int64_t ntok = 0;
    for (int u = 0; u < nJ; ++u)
        for (int i = 0; i < c->blk; ++i) {
            int64_t t = (int64_t)J[u] * c->blk + i;
            if (t <= limit) tok[ntok++] = t;
        }

    double *sc = (double *)malloc(sizeof(double) * (ntok > 0 ? ntok : 1));
    for (int g = 0; g < qpk; ++g) {
        int hq = h * qpk + g;
        const uint16_t *qr = c->q + ((gq * c->Hq + hq) * (int64_t)D);
        double *orow = c->o + ((ri * c->Hq + hq) * (int64_t)D);
        double *lrow = c->lse + (ri * c->Hq + hq);
        for (int d = 0; d < D; ++d) orow[d] = 0.0;
        if (ntok == 0) {                             /* no visible key: O = 0, LSE = -inf */
            *lrow = -INFINITY;
            continue;
        }
        /* 3. scores, max */
        double m = -INFINITY;
        for (int64_t i = 0; i < ntok; ++i) {
            const uint16_t *kr = kv_row(c, c->k, b, h, tok[i]);
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += bf16_to_double(qr[d]) * bf16_to_double(kr[d]);
            sc[i] = c->scale * acc;
            if (sc[i] > m) m = sc[i];
        }
        /* 4. softmax denominator, LSE, output */
        double l = 0.0;
        for (int64_t i = 0; i < ntok; ++i) {
            double p = exp(sc[i] - m);
            l += p;
            const uint16_t *vr = kv_row(c, c->v, b, h, tok[i]);
            for (int d = 0; d < D; ++d) orow[d] += p * bf16_to_double(vr[d]);
        }
        for (int d = 0; d < D; ++d) orow[d] /= l;
        *lrow = m + log(l);
    }
    free(sc);
    free(tok);
}

/* Dense-KV sparse attention.  Returns the number of threads used. */
int oracle_sparse_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *q2k,
                       int B, int Sq, int Skv, int Hq, int Hkv, int D, int blk, int topk,
                       int causal, double scale, const int32_t *seqused,
                       const int64_t *rows, int64_t nrows, double *o, double *lse, int nthreads) {
    attn_ctx c;
    memset(&c, 0, sizeof c);
    c.q = q; c.q2k = q2k; c.B = B; c.Sq = Sq; c.Hq = Hq; c.Hkv = Hkv; c.D = D; c.blk = blk;
    c.topk = topk; c.causal = causal; c.scale = scale;
    c.k = k; c.v = v; c.Skv = Skv; c.page_table = NULL; c.seqused = seqused;
    c.rows = rows; c.nrows = rows ? nrows : (int64_t)B * Sq;
    c.o = o; c.lse = lse;
    return parallel_for(c.nrows * Hkv, nthreads, attn_item, &c);
}

/* Paged-KV sparse attention (pool [num_pages][page][Hkv][D]). */
int oracle_sparse_attn_paged(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                             const int32_t *page_table, int max_pages, const int32_t *seqused,
                             const int32_t *q2k, int B, int Sq, int Hq, int Hkv, int D, int page,
                             int topk, int causal, double scale,
                             const int64_t *rows, int64_t nrows, double *o, double *lse, int nthreads) {
    attn_ctx c;
    memset(&c, 0, sizeof c);
    c.q = q; c.q2k = q2k; c.B = B; c.Sq = Sq; c.Hq = Hq; c.Hkv = Hkv; c.D = D; c.blk = page;
    c.topk = topk; c.causal = causal; c.scale = scale;
    c.k = k_pool; c.v = v_pool; c.Skv = max_pages * page; c.page_table = page_table;
    c.max_pages = max_pages; c.seqused = seqused;
    c.rows = rows; c.nrows = rows ? nrows : (int64_t)B * Sq;
    c.o = o; c.lse = lse;
    return parallel_for(c.nrows * Hkv, nthreads, attn_item, &c);
}

/* ---------------------------------------------------------------------- */
/* varlen batches, temperature LSE, every-block selection                  */
/* ---------------------------------------------------------------------- */

/*
 * Ragged batches as the interface page's sparse_atten_func takes them
 * (cu_seqlens_q / cu_seqlens_k prefix sums, q [total_q][Hq][D], k and v
 * [total_k][Hkv][D], q2k [Hkv][total_q][topk] with block ids local to each
 * sequence), and as the test page's varlen reference computes them: each
 * sequence is an independent batch-1 problem of sparse_attention_ref on its
 * own slice, so query s of sequence b sees key t (local) iff t lies in one of
 * its blocks, t < kv_len_b and, when causal, t <= s + (kv_len_b - Sq_b).
 *
 * Also, from sparse_attention_ref's lse_temperature_scale branch: a second
 * LSE over the same visible scores divided by the temperature T,
 * lse_T = log sum_t exp(s_t / T), s_t = scale * q . k_t (-inf for an empty row).
 *
 * q2k == NULL selects every block of the sequence (the interface page's
 * dense decode mode, sparse_decode_atten_func with q2k_indices = None).
 * page_table != NULL: k and v are pools [num_pages][blk][Hkv][D] and logical
 * block j of sequence b is page page_table[b][j] (kv_len_b = seqused[b], or
 * max_pages * blk); cu_k is then unused.
 */
typedef struct {
    const uint16_t *q, *k, *v;
    const int32_t *q2k, *cu_q, *cu_k, *page_table, *seqused;
    int B, Hq, Hkv, D, blk, topk, causal, max_pages;
    int64_t total_q;
    double scale, temp;
    const int64_t *rows;
    double *o, *lse, *lse_temp;
} varlen_ctx;

/* Sequence holding global query gq: the largest b with cu_q[b] <= gq. */
static int seq_of(const int32_t *cu_q, int B, int64_t gq) {
    int b = 0;
    while (b + 1 < B && cu_q[b + 1] <= gq) ++b;
    return b;
}

static void attn_item_varlen(void *vctx, int64_t item) {
    const varlen_ctx *c = (const varlen_ctx *)vctx;
    int64_t ri = item / c->Hkv;
    int h = (int)(item % c->Hkv);
    int64_t gq = c->rows ? c->rows[ri] : ri;
    int b = seq_of(c->cu_q, c->B, gq);
    int64_t s = gq - c->cu_q[b];
    int64_t sq_b = c->cu_q[b + 1] - c->cu_q[b];
    int64_t kv_alloc = c->page_table ? (int64_t)c->max_pages * c->blk : (int64_t)(c->cu_k[b + 1] - c->cu_k[b]);
    int64_t kv_len = c->seqused ? c->seqused[b] : kv_alloc;
    int nblk = (int)((kv_alloc + c->blk - 1) / c->blk);
    int qpk = c->Hq / c->Hkv, D = c->D;

    /* 1. the set J of distinct valid block ids (every block when q2k is NULL) */
    int *J = (int *)malloc(sizeof(int) * (size_t)(nblk > 0 ? nblk : 1));
    int nJ = 0;
    if (!c->q2k) {
        for (int j = 0; j < nblk; ++j) J[nJ++] = j;
    } else {
        const int32_t *sel = c->q2k + ((int64_t)h * c->total_q + gq) * c->topk;
        for (int t = 0; t < c->topk; ++t) {
            int j = sel[t];
            if (j < 0 || j >= nblk) continue;
            int dup = 0;
            for (int u = 0; u < nJ; ++u) dup |= (J[u] == j);
            if (!dup) J[nJ++] = j;
        }
    }
    /* 2. visible tokens */
    int64_t limit = kv_len - 1;
    if (c->causal && s + (kv_len - sq_b) < limit) limit = s + (kv_len - sq_b);
    int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)((int64_t)nJ * c->blk + 1));
    int64_t ntok = 0;
    for (int u = 0; u < nJ; ++u)
        for (int i = 0; i < c->blk; ++i) {
            int64_t t = (int64_t)J[u] * c->blk + i;
            if (t <= limit) tok[ntok++] = t;
        }
    double *sc = (double *)malloc(sizeof(double) * (size_t)(ntok > 0 ? ntok : 1));
    for (int g = 0; g < qpk; ++g) {
        int hq = h * qpk + g;
        const uint16_t *qr = c->q + (gq * c->Hq + hq) * (int64_t)D;
        double *orow = c->o + (ri * c->Hq + hq) * (int64_t)D;
        double *lrow = c->lse + ri * c->Hq + hq;
        double *trow = c->lse_temp ? c->lse_temp + ri * c->Hq + hq : NULL;
        for (int d = 0; d < D; ++d) orow[d] = 0.0;
        if (ntok == 0) {
            *lrow = -INFINITY;
            if (trow) *trow = -INFINITY;
            continue;
        }
        /* 3. scores and their max */
        double m = -INFINITY;
        for (int64_t i = 0; i < ntok; ++i) {
            const uint16_t *kr;
            if (c->page_table) {
                int64_t page = c->page_table[(int64_t)b * c->max_pages + tok[i] / c->blk];
                kr = c->k + ((page * c->blk + tok[i] % c->blk) * c->Hkv + h) * (int64_t)D;
            } else {
                kr = c->k + (((int64_t)c->cu_k[b] + tok[i]) * c->Hkv + h) * (int64_t)D;
            }
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += bf16_to_double(qr[d]) * bf16_to_double(kr[d]);
            sc[i] = c->scale * acc;
            if (sc[i] > m) m = sc[i];
        }
        /* 4. softmax, LSE, output; the temperature LSE over s_t / T */
        double l = 0.0, lt = 0.0;
        for (int64_t i = 0; i < ntok; ++i) {
            const uint16_t *vr;
            if (c->page_table) {
                int64_t page = c->page_table[(int64_t)b * c->max_pages + tok[i] / c->blk];
                vr = c->v + ((page * c->blk + tok[i] % c->blk) * c->Hkv + h) * (int64_t)D;
            } else {
                vr = c->v + (((int64_t)c->cu_k[b] + tok[i]) * c->Hkv + h) * (int64_t)D;
            }
            double p = exp(sc[i] - m);
            l += p;
            if (trow) lt += exp((sc[i] - m) / c->temp);
            for (int d = 0; d < D; ++d) orow[d] += p * bf16_to_double(vr[d]);
        }
        for (int d = 0; d < D; ++d) orow[d] /= l;
        *lrow = m + log(l);
        if (trow) *trow = m / c->temp + log(lt);
    }
    free(sc);
    free(tok);
    free(J);
}

/*
 * Varlen (and, with page_table, paged) sparse attention.  temp > 0 and
 * lse_temp != NULL also give the temperature LSE.  Returns the threads used.
 */
int oracle_sparse_attn_varlen(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *q2k,
                              const int32_t *cu_q, const int32_t *cu_k, const int32_t *page_table, int max_pages,
                              const int32_t *seqused, int B, int Hq, int Hkv, int D, int blk, int topk,
                              int causal, double scale, double temp, const int64_t *rows, int64_t nrows,
                              double *o, double *lse, double *lse_temp, int nthreads) {
    varlen_ctx c;
    memset(&c, 0, sizeof c);
    c.q = q; c.k = k; c.v = v; c.q2k = q2k; c.cu_q = cu_q; c.cu_k = cu_k; c.page_table = page_table;
    c.seqused = seqused; c.B = B; c.Hq = Hq; c.Hkv = Hkv; c.D = D; c.blk = blk; c.topk = topk;
    c.causal = causal; c.max_pages = max_pages; c.total_q = cu_q[B]; c.scale = scale;
    c.temp = temp; c.rows = rows; c.o = o; c.lse = lse;
    c.lse_temp = (temp > 0.0) ? lse_temp : NULL;
    int64_t n = rows ? nrows : c.total_q;
    return parallel_for(n * Hkv, nthreads, attn_item_varlen, &c);
}

/* ---------------------------------------------------------------------- */
/* k -> q CSR                                                              */
/* ---------------------------------------------------------------------- */

/*
 * Inverts q2k [B][Hkv][Sq][topk] into, per KV head h:
 *   row r = b * nblk + j (nblk = ceil(Skv / blk)), count = #queries naming j,
 *   row_ptr[h][r] = exclusive prefix of the counts, row_ptr[h][rows] = nnz,
 *   q_indices[h][row_ptr[h][r] ..] = global query ids b*Sq+s, ascending,
 *   q_indices[h][nnz ..] = -1 (tail up to B*Sq*topk),
 *   qsplit = q | (split << 24), split = rank of the slot among the query's
 *   distinct valid slots, qsplit tail = -1,
 *   split_counts[q][h] = number of distinct valid slots.
 * Valid: 0 <= j < ceil(kv_len_b / blk), kv_len_b = seqused[b] or Skv.
 */
int oracle_build_k2q_csr(const int32_t *q2k, int B, int Hkv, int Sq, int Skv, int topk, int blk,
                         const int32_t *seqused,
                         int32_t *row_ptr, int32_t *q_indices, int32_t *qsplit, int32_t *split_counts) {
    int nblk = (Skv + blk - 1) / blk;
    int64_t rows = (int64_t)B * nblk;
    int64_t cap = (int64_t)B * Sq * topk;
    int32_t *rank = (int32_t *)malloc(sizeof(int32_t) * (size_t)(cap > 0 ? cap : 1));
    int64_t *cursor = (int64_t *)malloc(sizeof(int64_t) * (size_t)(rows + 1));
    for (int h = 0; h < Hkv; ++h) {
        int32_t *rp = row_ptr + (int64_t)h * (rows + 1);
        int32_t *qi = q_indices + (int64_t)h * cap;
        int32_t *qs = qsplit + (int64_t)h * cap;
        for (int64_t r = 0; r <= rows; ++r) rp[r] = 0;
        /* pass 1: validity, ranks, counts */
        for (int b = 0; b < B; ++b) {
            int64_t kv_len = seqused ? seqused[b] : Skv;
            int64_t nvalid = (kv_len + blk - 1) / blk;
            if (nvalid > nblk) nvalid = nblk;
            for (int s = 0; s < Sq; ++s) {
                const int32_t *sel = q2k + (((int64_t)b * Hkv + h) * Sq + s) * topk;
                int32_t *rk = rank + ((int64_t)b * Sq + s) * topk;
                int cnt = 0;
                for (int t = 0; t < topk; ++t) {
                    int j = sel[t];
                    int ok = (j >= 0 && j < nvalid);
                    for (int u = 0; ok && u < t; ++u)
                        if (sel[u] == j) ok = 0;
                    rk[t] = ok ? cnt++ : -1;
                    if (ok) rp[(int64_t)b * nblk + j + 1] += 1;
                }
                split_counts[((int64_t)b * Sq + s) * Hkv + h] = cnt;
            }
        }
        for (int64_t r = 0; r < rows; ++r) rp[r + 1] += rp[r];
        /* pass 2: scatter in ascending query order (stable) */
        for (int64_t r = 0; r < rows; ++r) cursor[r] = rp[r];
        for (int64_t i = 0; i < cap; ++i) { qi[i] = -1; qs[i] = -1; }
        for (int b = 0; b < B; ++b)
            for (int s = 0; s < Sq; ++s) {
                const int32_t *sel = q2k + (((int64_t)b * Hkv + h) * Sq + s) * topk;
                const int32_t *rk = rank + ((int64_t)b * Sq + s) * topk;
                int64_t gq = (int64_t)b * Sq + s;
                for (int t = 0; t < topk; ++t) {
                    if (rk[t] < 0) continue;
                    int64_t r = (int64_t)b * nblk + sel[t];
                    int64_t pos = cursor[r]++;
                    qi[pos] = (int32_t)gq;
                    qs[pos] = (int32_t)(gq | ((int64_t)rk[t] << 24));
                }
            }
    }
    free(rank);
    free(cursor);
    return 0;
}

/*
 * Varlen k -> q CSR (interface page, sparse_atten_func: q2k [Hkv][total_q][topK]
 * with sequence-local block ids is inverted into k2q_row_ptr
 * [Hkv][total_rows + 1] and k2q_q_indices [Hkv][total_q * topK]).  Sequence b
 * owns rows row_off[b] .. row_off[b] + nblk_b - 1, nblk_b = ceil(kv_b / blk),
 * kv_b = cu_k[b+1] - cu_k[b]; row_off is the prefix of the nblk_b.  Valid ids:
 * 0 <= j < ceil(kv_len_b / blk), kv_len_b = seqused[b] or kv_b.  Within a
 * row the global query ids are ascending; qsplit, split_counts and the -1
 * tails as in oracle_build_k2q_csr.  total_rows = row_off[B].
 */
int oracle_build_k2q_csr_varlen(const int32_t *q2k, const int32_t *cu_q, const int32_t *cu_k, int B, int Hkv,
                                int topk, int blk, const int32_t *seqused, int32_t *row_ptr, int32_t *q_indices,
                                int32_t *qsplit, int32_t *split_counts) {
    int64_t total_q = cu_q[B];
    int64_t *row_off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(B + 1));
    row_off[0] = 0;
    for (int b = 0; b < B; ++b) row_off[b + 1] = row_off[b] + (cu_k[b + 1] - cu_k[b] + blk - 1) / blk;
    int64_t rows = row_off[B];
    int64_t cap = total_q * topk;
    int32_t *rank = (int32_t *)malloc(sizeof(int32_t) * (size_t)(cap > 0 ? cap : 1));
    int64_t *cursor = (int64_t *)malloc(sizeof(int64_t) * (size_t)(rows + 1));
    for (int h = 0; h < Hkv; ++h) {
        int32_t *rp = row_ptr + (int64_t)h * (rows + 1);
        int32_t *qi = q_indices + (int64_t)h * cap;
        int32_t *qs = qsplit + (int64_t)h * cap;
        for (int64_t r = 0; r <= rows; ++r) rp[r] = 0;
        for (int b = 0; b < B; ++b) {
            int64_t nblk_b = row_off[b + 1] - row_off[b];
            int64_t kv_len = seqused ? seqused[b] : (cu_k[b + 1] - cu_k[b]);
            int64_t nvalid = (kv_len + blk - 1) / blk;
            if (nvalid > nblk_b) nvalid = nblk_b;
            for (int64_t gq = cu_q[b]; gq < cu_q[b + 1]; ++gq) {
                const int32_t *sel = q2k + ((int64_t)h * total_q + gq) * topk;
                int32_t *rk = rank + gq * topk;
                int cnt = 0;
                for (int t = 0; t < topk; ++t) {
                    int j = sel[t];
                    int ok = (j >= 0 && j < nvalid);
                    for (int u = 0; ok && u < t; ++u)
                        if (sel[u] == j) ok = 0;
                    rk[t] = ok ? cnt++ : -1;
                    if (ok) rp[row_off[b] + j + 1] += 1;
                }
                split_counts[gq * Hkv + h] = cnt;
            }
        }
        for (int64_t r = 0; r < rows; ++r) rp[r + 1] += rp[r];
        for (int64_t r = 0; r < rows; ++r) cursor[r] = rp[r];
        for (int64_t i = 0; i < cap; ++i) { qi[i] = -1; qs[i] = -1; }
        for (int b = 0; b < B; ++b)
            for (int64_t gq = cu_q[b]; gq < cu_q[b + 1]; ++gq) {
                const int32_t *sel = q2k + ((int64_t)h * total_q + gq) * topk;
                const int32_t *rk = rank + gq * topk;
                for (int t = 0; t < topk; ++t) {
                    if (rk[t] < 0) continue;
                    int64_t pos = cursor[row_off[b] + sel[t]]++;
                    qi[pos] = (int32_t)gq;
                    qs[pos] = (int32_t)(gq | ((int64_t)rk[t] << 24));
                }
            }
    }
    free(rank);
    free(cursor);
    free(row_off);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* NVFP4 encoding of K/V rows                                               */
/* ---------------------------------------------------------------------- */

/*
 * x: [rows][D] bf16 bits (D % 16 == 0).  packed: [rows][D/2], element 2i in the
 * low nibble.  scales: [rows][D/16] e4m3 bytes.  Per group of 16:
 *   amax = max |x|, s = e4m3_rne_sat(float(amax) / 6.0f)  (binary32 division),
 *   code_i = e2m1_rne_sat(float(x_i) / float(s))          (binary32 division),
 *   s == 0 -> all codes 0.
 */
int oracle_nvfp4_quantize(const uint16_t *x, int64_t rows, int D, uint8_t *packed, uint8_t *scales) {
    for (int64_t r = 0; r < rows; ++r) {
        for (int g = 0; g < D / 16; ++g) {
            const uint16_t *xg = x + r * D + g * 16;
            float amax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float a = fabsf((float)bf16_to_double(xg[i]));
                if (a > amax) amax = a;
            }
            float q6 = amax / 6.0f;
            uint8_t sb = oracle_e4m3_from_double_rne_sat((double)q6);
            scales[r * (D / 16) + g] = sb;
            float sf = (float)oracle_e4m3_to_double(sb);
            for (int i = 0; i < 16; i += 2) {
                uint8_t c0 = 0, c1 = 0;
                if (sf > 0.0f) {
                    float y0 = (float)bf16_to_double(xg[i]) / sf;
                    float y1 = (float)bf16_to_double(xg[i + 1]) / sf;
                    c0 = oracle_e2m1_from_double_rne_sat((double)y0);
                    c1 = oracle_e2m1_from_double_rne_sat((double)y1);
                }
                packed[r * (D / 2) + (g * 16 + i) / 2] = (uint8_t)(c0 | (c1 << 4));
            }
        }
    }
    return 0;
}

/* Dequantise to bf16 bits: value * scale is exact in bf16 (<= 2 + 4 significant bits). */
int oracle_nvfp4_dequantize(const uint8_t *packed, const uint8_t *scales, int64_t rows, int D, uint16_t *x) {
    for (int64_t r = 0; r < rows; ++r)
        for (int e = 0; e < D; ++e) {
            uint8_t byte = packed[r * (D / 2) + e / 2];
            uint8_t code = (e & 1) ? (byte >> 4) : (byte & 0xF);
            double val = oracle_e2m1_to_double(code) * oracle_e4m3_to_double(scales[r * (D / 16) + e / 16]);
            float f = (float)val;
            uint32_t u;
            memcpy(&u, &f, sizeof u);
            x[r * D + e] = (uint16_t)(u >> 16);      /* exact: low 16 bits are zero */
        }
    return 0;
}
