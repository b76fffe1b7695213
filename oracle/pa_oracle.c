/*
 * pa_oracle.c -- plain CPU statement of paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA library is
 * checked against.  Only the tests, the smoke check and the benchmark's CPU
 * baseline leg may load it.  It shares no source, header, table or helper with
 * the CUDA path, and the CUDA path never calls it.
 *
 * Everything here is written for a reader to check by eye against the pages:
 *   - "Paged attention" (k4i.top), section "block table": token t of a sequence
 *     lives in physical_block = block_table[t // block_size] at offset
 *     t % block_size; the 38-token example maps logical blocks 0, 1, 2 to
 *     physical blocks 1, 5, 3 with 6 tokens in the last one.
 *   - "PagedAttention 在 vLLM 中的实现分析" (blog.chen3feng.top), section 3.2
 *     "Slot Mapping": slot = block_number * block_size + block_offset, and a
 *     negative slot is a padding token that is ignored; section 3.3 "KV Cache
 *     布局": the pool is [2, num_blocks, block_size, num_kv_heads, head_size]
 *     with key at index 0 and value at index 1; section 7.4: the cache-write
 *     kernel writes key[token] and value[token] to the slot when slot >= 0.
 *   - "Paged attention" (k4i.top), section "对非连续 blocks 做 attention": the
 *     block-wise online softmax is mathematically the same as standard softmax
 *     attention over the concatenated sequence.  The oracle therefore states
 *     the standard definition (gather, scores, max, exp, sum, weighted sum of
 *     values) in two plain passes, in fp64.  The online block merge is stated
 *     separately (or_online_softmax) only to check that identity.
 *
 * Floating point: all attention arithmetic is double precision.  fp16/bf16
 * inputs are decoded from their bit patterns by the IEEE 754 binary16 and the
 * bfloat16 (upper half of binary32) definitions; outputs are encoded back with
 * round-to-nearest, ties-to-even.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - query head h uses kv head h / (num_heads / num_kv_heads) (contiguous
 *     grouped-query groups);
 *   - seq_lens[s] counts every cached token of sequence s, the newest included;
 *   - seq_lens[s] == 0 gives an all-zero output row;
 *   - scale is an explicit argument (the configs use 1/sqrt(head_size));
 *   - the prefill readings are listed above or_prefill.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_FP16 0
#define OR_BF16 1

#define OR_OK 0
#define OR_ERR_ARG (-1)
#define OR_ERR_BLOCK_ID (-2)
#define OR_ERR_SEQ_LEN (-3)
#define OR_ERR_SLOT (-4)
#define OR_ERR_NOMEM (-5)

/* ------------------------------------------------------------------------ */
/* Number formats.                                                           */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16: sign, 5 exponent bits (bias 15), 10 fraction bits. */
double or_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^-14 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of a binary32 -- 8 exponent bits (bias 127),
 * 7 fraction bits. */
double or_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133); /* subnormal: f * 2^-7 * 2^-126 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134); /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

/* Encode x in a binary format with `ebits` exponent bits and `fbits` fraction
 * bits (IEEE-style: bias 2^(ebits-1)-1, subnormals, infinities), rounding to
 * nearest with ties to even. */
static uint16_t or_encode(double x, int ebits, int fbits)
{
    int bias = (1 << (ebits - 1)) - 1;
    int emin = 1 - bias;          /* exponent of the smallest normal */
    int emax_field = (1 << ebits) - 1;
    uint16_t sbit = (uint16_t)(signbit(x) ? 0x8000 : 0);
    if (isnan(x))
        return (uint16_t)(0x7fff & ((emax_field << fbits) | (1 << (fbits - 1))));
    double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sbit | (emax_field << fbits));
    if (a == 0.0)
        return sbit;
    int E;
    frexp(a, &E);
    E -= 1; /* a lies in [2^E, 2^(E+1)) */
    if (E < emin)
        E = emin; /* below the normal range the spacing stays 2^(emin-fbits) */
    double quantum = ldexp(1.0, E - fbits);
    double n = nearbyint(a / quantum); /* default mode: nearest, ties to even */
    double r = n * quantum;
    if (r >= ldexp(1.0, bias + 1)) /* above the largest finite value */
        return (uint16_t)(sbit | (emax_field << fbits));
    if (r < ldexp(1.0, emin)) /* subnormal (or rounded to zero) */
        return (uint16_t)(sbit | (uint16_t)(r / ldexp(1.0, emin - fbits)));
    int E2;
    frexp(r, &E2);
    E2 -= 1;
    uint16_t field = (uint16_t)(E2 + bias);
    uint16_t frac = (uint16_t)(r / ldexp(1.0, E2 - fbits) - (double)(1 << fbits));
    return (uint16_t)(sbit | (field << fbits) | frac);
}

uint16_t or_double_to_half(double x) { return or_encode(x, 5, 10); }
uint16_t or_double_to_bf16(double x) { return or_encode(x, 8, 7); }

static double or_load(const uint16_t *p, size_t i, int dtype)
{
    return dtype == OR_BF16 ? or_bf16_to_double(p[i]) : or_half_to_double(p[i]);
}

void or_round(const double *x, uint16_t *bits, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; i++)
        bits[i] = dtype == OR_BF16 ? or_double_to_bf16(x[i]) : or_double_to_half(x[i]);
}

void or_widen(const uint16_t *bits, double *x, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; i++)
        x[i] = or_load(bits, (size_t)i, dtype);
}

/* ------------------------------------------------------------------------ */
/* Address translation and slot mapping.                                     */
/* ------------------------------------------------------------------------ */

/* k4i.top "Paged attention", section "block table":
 * physical_block = block_table[t // block_size], offset = t % block_size. */
void or_translate(const int32_t *block_table_row, int t, int block_size,
                  int32_t *physical_block, int32_t *offset)
{
    *physical_block = block_table_row[t / block_size];
    *offset = t % block_size;
}

/* chen3feng vLLM analysis, section 3.2 "Slot Mapping":
 * slot = block_number * block_size + block_offset. */
int64_t or_slot_of_token(const int32_t *block_table_row, int t, int block_size)
{
    int32_t phys, off;
    or_translate(block_table_row, t, block_size, &phys, &off);
    return (int64_t)phys * block_size + off;
}

/* Element index of (plane, physical block, offset, kv head, dim) in the pool
 * [2, num_blocks, block_size, num_kv_heads, head_size] (section 3.3). */
static size_t or_pool_index(int plane, int64_t phys, int64_t off, int kvh, int d,
                            int num_blocks, int block_size, int num_kv_heads,
                            int head_size)
{
    return ((((size_t)plane * num_blocks + phys) * block_size + off) * num_kv_heads + kvh) *
               head_size + d;
}

/* ------------------------------------------------------------------------ */
/* Cache write (chen3feng vLLM analysis, sections 3.2 and 7.4).              */
/* ------------------------------------------------------------------------ */

/* For every token i with slot_mapping[i] >= 0 copy key[i] and value[i]
 * (num_kv_heads x head_size elements each, rows key_stride/value_stride
 * elements apart) into the pool at block slot / block_size, offset
 * slot % block_size.  Negative slots are padding and write nothing.  The copy
 * moves bit patterns; there is no arithmetic on the values. */
int or_reshape_and_cache(const uint16_t *key, const uint16_t *value, uint16_t *cache,
                         const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                         int head_size, int block_size, int num_blocks,
                         int64_t key_stride, int64_t value_stride)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 ||
        num_blocks <= 0)
        return OR_ERR_ARG;
    for (int i = 0; i < num_tokens; i++) {
        int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        if (slot >= (int64_t)num_blocks * block_size)
            return OR_ERR_SLOT;
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; h++) {
            for (int d = 0; d < head_size; d++) {
                cache[or_pool_index(0, blk, off, h, d, num_blocks, block_size, num_kv_heads,
                                    head_size)] = key[(size_t)i * key_stride + (size_t)h * head_size + d];
                cache[or_pool_index(1, blk, off, h, d, num_blocks, block_size, num_kv_heads,
                                    head_size)] = value[(size_t)i * value_stride + (size_t)h * head_size + d];
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Decode attention: the standard definition over the gathered sequence.    */
/* ------------------------------------------------------------------------ */

typedef struct {
    double *out;                 /* [num_seqs, num_heads, head_size] */
    const uint16_t *q;           /* [num_seqs, num_heads, head_size] */
    const uint16_t *cache;       /* [2, num_blocks, block_size, num_kv_heads, head_size] */
    const int32_t *block_tables; /* [num_seqs, max_blocks_per_seq] */
    const int32_t *seq_lens;     /* [num_seqs] */
    int num_seqs, num_heads, num_kv_heads, head_size, block_size, num_blocks,
        max_blocks_per_seq;
    double scale;
    int dtype;
    const int32_t *items; /* (seq * num_heads + head) indices, or NULL for all */
    int64_t num_items;
} or_decode_args;

/* One output row: sequence s, query head h.  Kc/Vc/a are scratch of at least
 * L*head_size, L*head_size and L doubles. */
static int or_attend_one(const or_decode_args *A, int s, int h, double *Kc, double *Vc,
                         double *a)
{
    const int D = A->head_size;
    const int G = A->num_heads / A->num_kv_heads;
    const int kvh = h / G;
    double *o = A->out + ((size_t)s * A->num_heads + h) * D;
    int L = A->seq_lens[s];
    if (L < 0 || L > A->max_blocks_per_seq * A->block_size)
        return OR_ERR_SEQ_LEN;
    if (L == 0) {
        for (int d = 0; d < D; d++)
            o[d] = 0.0;
        return OR_OK;
    }
    const int32_t *bt = A->block_tables + (size_t)s * A->max_blocks_per_seq;

    /* 1. Gather the sequence's keys and values into contiguous rows. */
    for (int t = 0; t < L; t++) {
        int32_t phys, off;
        or_translate(bt, t, A->block_size, &phys, &off);
        if (phys < 0 || phys >= A->num_blocks)
            return OR_ERR_BLOCK_ID;
        for (int d = 0; d < D; d++) {
            Kc[(size_t)t * D + d] = or_load(
                A->cache, or_pool_index(0, phys, off, kvh, d, A->num_blocks, A->block_size,
                                        A->num_kv_heads, D), A->dtype);
            Vc[(size_t)t * D + d] = or_load(
                A->cache, or_pool_index(1, phys, off, kvh, d, A->num_blocks, A->block_size,
                                        A->num_kv_heads, D), A->dtype);
        }
    }

    /* 2. Scores a_t = scale * sum_d q[d] * K[t][d]. */
    const size_t qrow = ((size_t)s * A->num_heads + h) * D;
    for (int t = 0; t < L; t++) {
        double acc = 0.0;
        for (int d = 0; d < D; d++)
            acc += or_load(A->q, qrow + d, A->dtype) * Kc[(size_t)t * D + d];
        a[t] = A->scale * acc;
    }

    /* 3. softmax(a) = exp(a_t - max) / sum_u exp(a_u - max). */
    double m = a[0];
    for (int t = 1; t < L; t++)
        if (a[t] > m)
            m = a[t];
    double l = 0.0;
    for (int t = 0; t < L; t++) {
        a[t] = exp(a[t] - m);
        l += a[t];
    }

    /* 4. Output o[d] = sum_t softmax_t * V[t][d]. */
    for (int d = 0; d < D; d++) {
        double acc = 0.0;
        for (int t = 0; t < L; t++)
            acc += a[t] * Vc[(size_t)t * D + d];
        o[d] = acc / l;
    }
    return OR_OK;
}

typedef struct {
    const or_decode_args *A;
    int tid, nthreads;
    int status;
} or_worker;

static void *or_decode_worker(void *p)
{
    or_worker *w = (or_worker *)p;
    const or_decode_args *A = w->A;
    int64_t n = A->items ? A->num_items : (int64_t)A->num_seqs * A->num_heads;
    size_t cap = (size_t)A->max_blocks_per_seq * A->block_size;
    if (cap == 0)
        cap = 1;
    double *Kc = (double *)malloc(cap * A->head_size * sizeof(double));
    double *Vc = (double *)malloc(cap * A->head_size * sizeof(double));
    double *a = (double *)malloc(cap * sizeof(double));
    w->status = OR_OK;
    if (!Kc || !Vc || !a) {
        w->status = OR_ERR_NOMEM;
    } else {
        for (int64_t i = w->tid; i < n; i += w->nthreads) {
            int64_t item = A->items ? A->items[i] : i;
            int s = (int)(item / A->num_heads);
            int h = (int)(item % A->num_heads);
            int rc = or_attend_one(A, s, h, Kc, Vc, a);
            if (rc != OR_OK) {
                w->status = rc;
                break;
            }
        }
    }
    free(Kc);
    free(Vc);
    free(a);
    return NULL;
}

/* Decode attention for every (sequence, query head), or only for the listed
 * items (seq * num_heads + head) when items != NULL.  Results go to out
 * [num_seqs, num_heads, head_size] in double precision; rows not listed are
 * left untouched.  Work items are dealt round-robin to nthreads threads. */
int or_decode(double *out, const uint16_t *q, const uint16_t *cache,
              const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
              int num_heads, int num_kv_heads, int head_size, int block_size,
              int num_blocks, int max_blocks_per_seq, double scale, int dtype,
              const int32_t *items, int64_t num_items, int nthreads)
{
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads != 0 || head_size <= 0 || block_size <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0 || (dtype != OR_FP16 && dtype != OR_BF16))
        return OR_ERR_ARG;
    if (nthreads < 1)
        nthreads = 1;
    or_decode_args A = {out, q, cache, block_tables, seq_lens, num_seqs, num_heads,
                        num_kv_heads, head_size, block_size, num_blocks,
                        max_blocks_per_seq, scale, dtype, items, num_items};
    or_worker *w = (or_worker *)calloc((size_t)nthreads, sizeof(or_worker));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!w || !th) {
        free(w);
        free(th);
        return OR_ERR_NOMEM;
    }
    for (int i = 0; i < nthreads; i++) {
        w[i].A = &A;
        w[i].tid = i;
        w[i].nthreads = nthreads;
    }
    int started = 0;
    for (int i = 1; i < nthreads; i++) {
        if (pthread_create(&th[i], NULL, or_decode_worker, &w[i]) != 0)
            break;
        started = i;
    }
    /* Threads that failed to start leave their items to this thread. */
    if (started < nthreads - 1) {
        for (int i = 0; i < nthreads; i++)
            w[i].nthreads = 1;
        for (int i = 1; i <= started; i++)
            pthread_join(th[i], NULL);
        w[0].tid = 0;
        or_decode_worker(&w[0]);
        int st = w[0].status;
        free(w);
        free(th);
        return st;
    }
    or_decode_worker(&w[0]);
    for (int i = 1; i < nthreads; i++)
        pthread_join(th[i], NULL);
    int st = OR_OK;
    for (int i = 0; i < nthreads; i++)
        if (w[i].status != OR_OK)
            st = w[i].status;
    free(w);
    free(th);
    return st;
}

/* ------------------------------------------------------------------------ */
/* The block-wise online softmax, as k4i.top "Paged attention" states it in */
/* section "对非连续 blocks 做 attention".                                   */
/* ------------------------------------------------------------------------ */

/* Scores a[0..n) (already scaled) and value rows V[n][D] are cut into blocks
 * of `block` entries.  Each block j gives m_j = max a, l_j = sum exp(a - m_j),
 * o_j = sum exp(a - m_j) V; the running (m, l, o) absorbs it with
 * m_new = max(m, m_j), l = e^(m-m_new) l + e^(m_j-m_new) l_j,
 * o = e^(m-m_new) o + e^(m_j-m_new) o_j.  The result o / l goes to out[D].
 * Also returns the final (m, l) so a caller can merge further. */
int or_online_softmax(double *out, double *m_out, double *l_out, const double *a,
                      const double *V, int n, int D, int block)
{
    if (n <= 0 || D <= 0 || block <= 0)
        return OR_ERR_ARG;
    double *o = (double *)calloc((size_t)D, sizeof(double));
    double *oj = (double *)malloc((size_t)D * sizeof(double));
    if (!o || !oj) {
        free(o);
        free(oj);
        return OR_ERR_NOMEM;
    }
    double m = -INFINITY, l = 0.0;
    for (int j0 = 0; j0 < n; j0 += block) {
        int j1 = j0 + block < n ? j0 + block : n;
        double mj = a[j0];
        for (int t = j0 + 1; t < j1; t++)
            if (a[t] > mj)
                mj = a[t];
        double lj = 0.0;
        for (int d = 0; d < D; d++)
            oj[d] = 0.0;
        for (int t = j0; t < j1; t++) {
            double p = exp(a[t] - mj);
            lj += p;
            for (int d = 0; d < D; d++)
                oj[d] += p * V[(size_t)t * D + d];
        }
        double m_new = m > mj ? m : mj;
        double c_old = exp(m - m_new); /* exp(-inf) = 0 on the first block */
        double c_new = exp(mj - m_new);
        l = c_old * l + c_new * lj;
        for (int d = 0; d < D; d++)
            o[d] = c_old * o[d] + c_new * oj[d];
        m = m_new;
    }
    for (int d = 0; d < D; d++)
        out[d] = o[d] / l;
    if (m_out)
        *m_out = m;
    if (l_out)
        *l_out = l;
    free(o);
    free(oj);
    return OR_OK;
}

/* Merge of independently computed partial states (m_p, l_p, o_p), with o_p
 * the unnormalised weighted value sum of part p (chen3feng vLLM analysis,
 * section 7.3: the partitioned kernel's parts are combined by rescaling with
 * the online-softmax correction).  out[d] = sum_p e^(m_p - M) o_p[d] /
 * sum_p e^(m_p - M) l_p with M = max_p m_p. */
int or_merge_partials(double *out, const double *m, const double *l, const double *o,
                      int parts, int D)
{
    if (parts <= 0 || D <= 0)
        return OR_ERR_ARG;
    double M = m[0];
    for (int p = 1; p < parts; p++)
        if (m[p] > M)
            M = m[p];
    double denom = 0.0;
    for (int p = 0; p < parts; p++)
        denom += exp(m[p] - M) * l[p];
    for (int d = 0; d < D; d++) {
        double num = 0.0;
        for (int p = 0; p < parts; p++)
            num += exp(m[p] - M) * o[(size_t)p * D + d];
        out[d] = num / denom;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Copy-on-write block copy ("Paged attention", k4i.top, section            */
/* "并行采样中的 copy-on-write": a new block receives a copy of the shared  */
/* block before the writer's token goes into it).                           */
/* ------------------------------------------------------------------------ */

/* For each pair i, copy every key and value row of physical block
 * mapping[2i] into physical block mapping[2i+1] of the pool
 * [2, num_blocks, block_size, num_kv_heads, head_size].  Pairs are applied in
 * order.  Ids outside [0, num_blocks) are an error. */
int or_copy_blocks(uint16_t *cache, const int64_t *mapping, int num_pairs, int num_blocks,
                   int block_size, int num_kv_heads, int head_size)
{
    const size_t block_elems = (size_t)block_size * num_kv_heads * head_size;
    for (int i = 0; i < num_pairs; i++) {
        int64_t src = mapping[2 * i], dst = mapping[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks)
            return OR_ERR_BLOCK_ID;
        for (int plane = 0; plane < 2; plane++) {
            const size_t base = (size_t)plane * num_blocks * block_elems;
            memmove(cache + base + (size_t)dst * block_elems,
                    cache + base + (size_t)src * block_elems, block_elems * sizeof(uint16_t));
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Prefill and chunked prefill over the paged cache (chen3feng vLLM          */
/* analysis, section 6.2: the FlashAttention backend attends the batch's     */
/* new query tokens, packed by query_start_loc, to the paged keys of each    */
/* request with seqlen_k = seq_lens, the block table and causal masking;     */
/* section 5.4 lists query_start_loc as each request's first query row).     */
/* ------------------------------------------------------------------------ */

/* Readings where the section is silent:
 *   - the q_len = query_start_loc[r+1] - query_start_loc[r] query rows of
 *     request r are its LAST q_len tokens: seq_lens[r] counts them and the
 *     cache write has already put them in the pool, so query row i of the
 *     request sits at position p = seq_lens[r] - q_len + i;
 *   - causal: position p attends keys 0..p; not causal (the shared-prefix
 *     pass of section 6.4): every key 0..seq_lens[r]-1;
 *   - lse is the natural log of the softmax denominator,
 *     log sum_t exp(scale * q . k_t). */
typedef struct {
    double *out;                   /* [num_tokens, num_heads, head_size] */
    double *lse;                   /* [num_tokens, num_heads] or NULL */
    const uint16_t *q;             /* [num_tokens, num_heads, head_size] */
    const uint16_t *cache;         /* [2, num_blocks, block_size, num_kv_heads, head_size] */
    const int32_t *block_tables;   /* row r at block_tables + r * block_table_stride */
    int64_t block_table_stride;
    const int32_t *seq_lens;       /* [num_reqs] */
    const int32_t *query_start_loc; /* [num_reqs + 1] */
    int num_reqs, num_heads, num_kv_heads, head_size, block_size, num_blocks,
        max_blocks_per_seq, causal;
    double scale;
    int dtype;
    const int64_t *items; /* (token * num_heads + head) indices, or NULL for all */
    int64_t num_items;
} or_prefill_args;

/* One output row: query token tok, query head h. */
static int or_prefill_row(const or_prefill_args *A, int64_t tok, int h, double *Kc,
                          double *Vc, double *a)
{
    const int D = A->head_size;
    const int kvh = h / (A->num_heads / A->num_kv_heads);
    int r = -1;
    for (int i = 0; i < A->num_reqs; i++)
        if (A->query_start_loc[i] <= tok && tok < A->query_start_loc[i + 1]) {
            r = i;
            break;
        }
    if (r < 0)
        return OR_ERR_ARG;
    const int L = A->seq_lens[r];
    const int q_len = A->query_start_loc[r + 1] - A->query_start_loc[r];
    if (L < q_len || L > A->max_blocks_per_seq * A->block_size)
        return OR_ERR_SEQ_LEN;
    const int pos = L - q_len + (int)(tok - A->query_start_loc[r]);
    const int n_keys = A->causal ? pos + 1 : L;
    const int32_t *bt = A->block_tables + (size_t)r * A->block_table_stride;

    /* 1. Gather keys and values 0..n_keys-1 into contiguous rows. */
    for (int t = 0; t < n_keys; t++) {
        int32_t phys, off;
        or_translate(bt, t, A->block_size, &phys, &off);
        if (phys < 0 || phys >= A->num_blocks)
            return OR_ERR_BLOCK_ID;
        for (int d = 0; d < D; d++) {
            Kc[(size_t)t * D + d] = or_load(
                A->cache, or_pool_index(0, phys, off, kvh, d, A->num_blocks, A->block_size,
                                        A->num_kv_heads, D), A->dtype);
            Vc[(size_t)t * D + d] = or_load(
                A->cache, or_pool_index(1, phys, off, kvh, d, A->num_blocks, A->block_size,
                                        A->num_kv_heads, D), A->dtype);
        }
    }

    /* 2. Scores a_t = scale * q . k_t. */
    const size_t qrow = ((size_t)tok * A->num_heads + h) * D;
    for (int t = 0; t < n_keys; t++) {
        double acc = 0.0;
        for (int d = 0; d < D; d++)
            acc += or_load(A->q, qrow + d, A->dtype) * Kc[(size_t)t * D + d];
        a[t] = A->scale * acc;
    }

    /* 3. Softmax with its maximum m and denominator l. */
    double m = a[0];
    for (int t = 1; t < n_keys; t++)
        if (a[t] > m)
            m = a[t];
    double l = 0.0;
    for (int t = 0; t < n_keys; t++) {
        a[t] = exp(a[t] - m);
        l += a[t];
    }

    /* 4. out[d] = sum_t softmax_t v_t[d]; lse = m + log l. */
    double *o = A->out + ((size_t)tok * A->num_heads + h) * D;
    for (int d = 0; d < D; d++) {
        double acc = 0.0;
        for (int t = 0; t < n_keys; t++)
            acc += a[t] * Vc[(size_t)t * D + d];
        o[d] = acc / l;
    }
    if (A->lse)
        A->lse[(size_t)tok * A->num_heads + h] = m + log(l);
    return OR_OK;
}

typedef struct {
    const or_prefill_args *A;
    int tid, nthreads;
    int status;
} or_prefill_worker_t;

static void *or_prefill_worker(void *p)
{
    or_prefill_worker_t *w = (or_prefill_worker_t *)p;
    const or_prefill_args *A = w->A;
    const int64_t num_tokens = A->query_start_loc[A->num_reqs];
    const int64_t n = A->items ? A->num_items : num_tokens * A->num_heads;
    size_t cap = (size_t)A->max_blocks_per_seq * A->block_size;
    if (cap == 0)
        cap = 1;
    double *Kc = (double *)malloc(cap * A->head_size * sizeof(double));
    double *Vc = (double *)malloc(cap * A->head_size * sizeof(double));
    double *a = (double *)malloc(cap * sizeof(double));
    w->status = OR_OK;
    if (!Kc || !Vc || !a) {
        w->status = OR_ERR_NOMEM;
    } else {
        for (int64_t i = w->tid; i < n; i += w->nthreads) {
            int64_t item = A->items ? A->items[i] : i;
            if (item < 0 || item >= num_tokens * A->num_heads) {
                w->status = OR_ERR_ARG;
                break;
            }
            int rc = or_prefill_row(A, item / A->num_heads, (int)(item % A->num_heads), Kc,
                                    Vc, a);
            if (rc != OR_OK) {
                w->status = rc;
                break;
            }
        }
    }
    free(Kc);
    free(Vc);
    free(a);
    return NULL;
}

/* Attention of every packed query row (or only the listed items) to its
 * request's paged keys.  out [num_tokens, num_heads, head_size] and lse
 * [num_tokens, num_heads] (may be NULL) are double precision; rows not listed
 * are left untouched.  num_tokens = query_start_loc[num_reqs]. */
int or_prefill(double *out, double *lse, const uint16_t *q, const uint16_t *cache,
               const int32_t *block_tables, int64_t block_table_stride,
               const int32_t *seq_lens, const int32_t *query_start_loc, int num_reqs,
               int num_heads, int num_kv_heads, int head_size, int block_size, int num_blocks,
               int max_blocks_per_seq, double scale, int causal, int dtype,
               const int64_t *items, int64_t num_items, int nthreads)
{
    if (num_reqs < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads != 0 || head_size <= 0 || block_size <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0 || block_table_stride < max_blocks_per_seq ||
        (dtype != OR_FP16 && dtype != OR_BF16))
        return OR_ERR_ARG;
    if (query_start_loc[0] != 0)
        return OR_ERR_ARG;
    for (int r = 0; r < num_reqs; r++)
        if (query_start_loc[r + 1] < query_start_loc[r])
            return OR_ERR_ARG;
    if (nthreads < 1)
        nthreads = 1;
    or_prefill_args A = {out, lse, q, cache, block_tables, block_table_stride, seq_lens,
                         query_start_loc, num_reqs, num_heads, num_kv_heads, head_size,
                         block_size, num_blocks, max_blocks_per_seq, causal ? 1 : 0, scale,
                         dtype, items, num_items};
    or_prefill_worker_t *w =
        (or_prefill_worker_t *)calloc((size_t)nthreads, sizeof(or_prefill_worker_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!w || !th) {
        free(w);
        free(th);
        return OR_ERR_NOMEM;
    }
    int started = 1;
    for (int i = 0; i < nthreads; i++) {
        w[i].A = &A;
        w[i].tid = i;
        w[i].nthreads = nthreads;
    }
    for (int i = 1; i < nthreads; i++) {
        if (pthread_create(&th[i], NULL, or_prefill_worker, &w[i]) != 0)
            break;
        started = i + 1;
    }
    or_prefill_worker(&w[0]);
    for (int i = 1; i < started; i++)
        pthread_join(th[i], NULL);
    /* Items of threads that never started are done here, one by one. */
    for (int i = started; i < nthreads; i++)
        or_prefill_worker(&w[i]);
    int st = OR_OK;
    for (int i = 0; i < nthreads; i++)
        if (w[i].status != OR_OK)
            st = w[i].status;
    free(w);
    free(th);
    return st;
}

/* Merge of two attention results over disjoint key sets, each given with its
 * log-sum-exp (chen3feng vLLM analysis, section 6.4: the shared-prefix pass
 * and the per-request suffix pass are combined with the online-softmax
 * correction).  With M = max(lse_a, lse_b), w_x = exp(lse_x - M):
 *   out = (w_a o_a + w_b o_b) / (w_a + w_b),  lse = M + log(w_a + w_b).
 * A part with lse = -inf is empty; two empty parts give out = 0,
 * lse = -inf.  lse_out may be NULL. */
int or_merge_attn_states(double *out, double *lse_out, const double *o_a,
                         const double *lse_a, const double *o_b, const double *lse_b,
                         int64_t rows, int D)
{
    if (rows < 0 || D <= 0)
        return OR_ERR_ARG;
    for (int64_t i = 0; i < rows; i++) {
        const double la = lse_a[i], lb = lse_b[i];
        double *o = out + (size_t)i * D;
        if (isinf(la) && la < 0 && isinf(lb) && lb < 0) {
            for (int d = 0; d < D; d++)
                o[d] = 0.0;
            if (lse_out)
                lse_out[i] = -INFINITY;
            continue;
        }
        const double M = la > lb ? la : lb;
        const double wa = exp(la - M), wb = exp(lb - M);
        for (int d = 0; d < D; d++)
            o[d] = (wa * o_a[(size_t)i * D + d] + wb * o_b[(size_t)i * D + d]) / (wa + wb);
        if (lse_out)
            lse_out[i] = M + log(wa + wb);
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* FP8 KV cache ("PagedAttention 在 vLLM 中的实现分析", section 6.3: the    */
/* cache write converts K/V to FP8 with k_scale / v_scale when the cache    */
/* dtype is FP8; section 8 lists FP8 KV-cache quantisation).                */
/* ------------------------------------------------------------------------ */

/* Readings where the pages are silent:
 *   - the FP8 format is e4m3 (1 sign, 4 exponent bits with bias 7, 3 fraction
 *     bits, no infinities; exponent 15 with fraction 7 is NaN, so the largest
 *     finite magnitude is 1.75 * 2^8 = 448);
 *   - k_scale and v_scale are one float each: the cache stores x / scale and
 *     a read gives stored * scale;
 *   - the quotient x / scale is a float32 division (the precision the CUDA
 *     kernel decides the code in), then rounded to e4m3, nearest with ties to
 *     even, magnitudes above 448 saturating to 448, NaN staying NaN. */

double or_fp8e4m3_to_double(uint8_t b)
{
    const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);           /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp(8.0 + m, e - 10);         /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

uint8_t or_double_to_fp8e4m3(double x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0)
        return sign | 0x7E;                 /* saturate to 448 */
    /* quantum of the binade holding a: 2^(e-3) for a in [2^e, 2^(e+1)),
     * e >= -6; the subnormal range [0, 2^-6) has quantum 2^-9 */
    int e;
    frexp(a, &e);                           /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                                 /* a in [2^e, 2^(e+1)) */
    if (a == 0.0 || e < -6)
        e = -6;
    const double quantum = ldexp(1.0, e - 3);
    double n = nearbyint(a / quantum);      /* ties to even (default mode) */
    double r = n * quantum;
    if (r > 448.0)
        r = 448.0;
    /* encode r exactly */
    if (r < ldexp(1.0, -6))
        return sign | (uint8_t)(r / ldexp(1.0, -9));
    int er;
    double f = frexp(r, &er);               /* r = f * 2^er, f in [0.5, 1) */
    const int exp_field = er - 1 + 7;
    const int frac = (int)((f * 2.0 - 1.0) * 8.0);
    return sign | (uint8_t)(exp_field << 3) | (uint8_t)frac;
}

void or_fp8_widen(const uint8_t *bits, double *x, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        x[i] = or_fp8e4m3_to_double(bits[i]);
}

/* Quantise float32 values: code = e4m3(fp32(x / scale)). */
void or_fp8_quantize(const float *x, uint8_t *bits, int64_t n, float scale)
{
    for (int64_t i = 0; i < n; i++) {
        const float qv = x[i] / scale;
        bits[i] = or_double_to_fp8e4m3((double)qv);
    }
}

/* The cache write with an FP8 pool: token i with slot_mapping[i] >= 0 gets
 * key[i] / k_scale and value[i] / v_scale, each quantised as above, at
 * (slot / block_size, slot % block_size) of the pool
 * [2, num_blocks, block_size, num_kv_heads, head_size] (uint8 codes). */
int or_reshape_and_cache_fp8(const uint16_t *key, const uint16_t *value, uint8_t *cache,
                             const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                             int head_size, int block_size, int num_blocks, int64_t key_stride,
                             int64_t value_stride, int src_dtype, float k_scale, float v_scale)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 ||
        num_blocks <= 0 || !(k_scale > 0.f) || !(v_scale > 0.f))
        return OR_ERR_ARG;
    for (int i = 0; i < num_tokens; i++) {
        const int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        if (slot >= (int64_t)num_blocks * block_size)
            return OR_ERR_SLOT;
        const int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; h++)
            for (int d = 0; d < head_size; d++) {
                const size_t src = (size_t)h * head_size + d;
                const float kx = (float)or_load(key, (size_t)i * key_stride + src, src_dtype);
                const float vx = (float)or_load(value, (size_t)i * value_stride + src, src_dtype);
                cache[or_pool_index(0, blk, off, h, d, num_blocks, block_size, num_kv_heads,
                                    head_size)] = or_double_to_fp8e4m3((double)(kx / k_scale));
                cache[or_pool_index(1, blk, off, h, d, num_blocks, block_size, num_kv_heads,
                                    head_size)] = or_double_to_fp8e4m3((double)(vx / v_scale));
            }
    }
    return OR_OK;
}

/* Decode attention over an FP8 pool: keys k_scale * e4m3(K), values
 * v_scale * e4m3(V); otherwise the definition of or_decode (two passes in
 * fp64).  One output row per (sequence, query head), or only the items. */
int or_decode_fp8(double *out, const uint16_t *q, const uint8_t *cache,
                  const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                  int num_heads, int num_kv_heads, int head_size, int block_size,
                  int num_blocks, int max_blocks_per_seq, double scale, int q_dtype,
                  double k_scale, double v_scale, const int32_t *items, int64_t num_items)
{
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads != 0 || head_size <= 0 || block_size <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0)
        return OR_ERR_ARG;
    const int D = head_size, G = num_heads / num_kv_heads;
    const size_t cap = (size_t)max_blocks_per_seq * block_size;
    double *Kc = (double *)malloc((cap ? cap : 1) * D * sizeof(double));
    double *Vc = (double *)malloc((cap ? cap : 1) * D * sizeof(double));
    double *a = (double *)malloc((cap ? cap : 1) * sizeof(double));
    int status = OR_OK;
    if (!Kc || !Vc || !a) {
        status = OR_ERR_NOMEM;
        goto done;
    }
    const int64_t n = items ? num_items : (int64_t)num_seqs * num_heads;
    for (int64_t it = 0; it < n; it++) {
        const int64_t item = items ? items[it] : it;
        const int s = (int)(item / num_heads), h = (int)(item % num_heads);
        const int kvh = h / G;
        double *o = out + ((size_t)s * num_heads + h) * D;
        const int L = seq_lens[s];
        if (L < 0 || (size_t)L > cap) {
            status = OR_ERR_SEQ_LEN;
            goto done;
        }
        if (L == 0) {
            for (int d = 0; d < D; d++)
                o[d] = 0.0;
            continue;
        }
        const int32_t *bt = block_tables + (size_t)s * max_blocks_per_seq;
        for (int t = 0; t < L; t++) {
            int32_t phys, off;
            or_translate(bt, t, block_size, &phys, &off);
            if (phys < 0 || phys >= num_blocks) {
                status = OR_ERR_BLOCK_ID;
                goto done;
            }
            for (int d = 0; d < D; d++) {
                Kc[(size_t)t * D + d] = k_scale * or_fp8e4m3_to_double(cache[or_pool_index(
                                            0, phys, off, kvh, d, num_blocks, block_size,
                                            num_kv_heads, D)]);
                Vc[(size_t)t * D + d] = v_scale * or_fp8e4m3_to_double(cache[or_pool_index(
                                            1, phys, off, kvh, d, num_blocks, block_size,
                                            num_kv_heads, D)]);
            }
        }
        const size_t qrow = ((size_t)s * num_heads + h) * D;
        for (int t = 0; t < L; t++) {
            double acc = 0.0;
            for (int d = 0; d < D; d++)
                acc += or_load(q, qrow + d, q_dtype) * Kc[(size_t)t * D + d];
            a[t] = scale * acc;
        }
        double m = a[0];
        for (int t = 1; t < L; t++)
            if (a[t] > m)
                m = a[t];
        double l = 0.0;
        for (int t = 0; t < L; t++) {
            a[t] = exp(a[t] - m);
            l += a[t];
        }
        for (int d = 0; d < D; d++) {
            double acc = 0.0;
            for (int t = 0; t < L; t++)
                acc += a[t] * Vc[(size_t)t * D + d];
            o[d] = acc / l;
        }
    }
done:
    free(Kc);
    free(Vc);
    free(a);
    return status;
}

/* Host check of the caller preconditions the CUDA library documents:
 * 0 <= seq_lens[s] <= max_blocks_per_seq * block_size and every block id a
 * sequence uses lies in [0, num_blocks).  Returns OR_OK or an error code. */
int or_check_tables(const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                    int max_blocks_per_seq, int block_size, int num_blocks)
{
    for (int s = 0; s < num_seqs; s++) {
        int L = seq_lens[s];
        if (L < 0 || L > max_blocks_per_seq * block_size)
            return OR_ERR_SEQ_LEN;
        int nb = (L + block_size - 1) / block_size;
        for (int j = 0; j < nb; j++) {
            int32_t b = block_tables[(size_t)s * max_blocks_per_seq + j];
            if (b < 0 || b >= num_blocks)
                return OR_ERR_BLOCK_ID;
        }
    }
    return OR_OK;
}
