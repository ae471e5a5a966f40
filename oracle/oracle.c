/*
 * Paged-KV oracle: plain, slow, obviously correct CPU restatement of the
 * PagedAttention decode path, in double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or helper with
 * the CUDA path.
 *
 * Sources (web pages on "Efficient Memory Management for Large Language
 * Model Serving with PagedAttention", Kwon et al. 2023):
 *  - aiplusplus "PagedAttention: OS virtual memory for LLM inference",
 *    section "core idea", items 1-4: the KV cache is cut into fixed-size
 *    blocks of B tokens, each sequence keeps a block table mapping its i-th
 *    logical block to a physical block, and blocks need not be contiguous.
 *  - same page, "key techniques" 1: the attention kernel follows the block
 *    table to assemble the scattered K and V blocks.
 *  - auturnal "paged-attention serving guide", section 1: paging changes how
 *    storage is allocated and indexed, not what attention has to read; the
 *    verification protocol asks for a check against a contiguous-KV baseline.
 *  Hence the decode result is ordinary softmax attention of one query per
 *  sequence over that sequence's logical K/V, and this oracle computes it by
 *  (1) walking the block table to copy the sequence's K and V into
 *  contiguous double arrays and (2) evaluating softmax(scale * q K^T) V.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - cache layout [num_blocks][num_kv_heads][block_size][head_dim];
 *  - query head h reads KV head h / (num_heads / num_kv_heads);
 *  - token i of a sequence lives in logical block i / B at offset i % B;
 *  - context_len counts the tokens attended (including the one written this
 *    step); positions >= context_len and blocks not in the table are never
 *    read; context_len == 0 gives an all-zero output row;
 *  - slot < 0 in a slot mapping marks padding and is skipped.
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

enum {
    ORC_OK = 0,
    ORC_BAD_ARG = -1,
    ORC_BAD_BLOCK = -2,
    ORC_BAD_LEN = -3,
    ORC_BAD_SLOT = -4,
    ORC_NO_MEM = -5
};

/* ---- widening of stored scalars to double (IEEE 754 definitions) ------- */

static double widen_f16(uint16_t h)
{
    /* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static double widen_bf16(uint16_t b)
{
    /* bfloat16 is the upper half of a binary32 word. */
    uint32_t w = (uint32_t)b << 16;
    float x;
    memcpy(&x, &w, sizeof x);
    return (double)x;
}

static double load_elem(const void* base, int dtype, size_t idx)
{
    if (dtype == ORC_F32) {
        float x;
        memcpy(&x, (const char*)base + 4 * idx, 4);
        return (double)x;
    }
    uint16_t h;
    memcpy(&h, (const char*)base + 2 * idx, 2);
    return dtype == ORC_F16 ? widen_f16(h) : widen_bf16(h);
}

static int elem_bytes(int dtype)
{
    return dtype == ORC_F32 ? 4 : (dtype == ORC_F16 || dtype == ORC_BF16) ? 2 : 0;
}

int orc_widen(const void* src, int dtype, int64_t n, double* dst)
{
    if (!elem_bytes(dtype)) return ORC_BAD_ARG;
    for (int64_t i = 0; i < n; ++i) dst[i] = load_elem(src, dtype, (size_t)i);
    return ORC_OK;
}

/* ---- cache write: store each new token's K and V in its slot ----------- */
/* key/value: [num_tokens][num_kv_heads][head_dim]; slot = block*B + offset. */
int orc_kv_write(void* k_cache, void* v_cache, const void* key, const void* value,
                 const int64_t* slot_mapping, int num_tokens, int num_blocks,
                 int num_kv_heads, int head_dim, int block_size, int dtype)
{
    int eb = elem_bytes(dtype);
    if (!eb || num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0)
        return ORC_BAD_ARG;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue; /* padding */
        if (slot >= (int64_t)num_blocks * block_size) return ORC_BAD_SLOT;
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t dst = (size_t)(((blk * num_kv_heads + h) * block_size + off) * head_dim);
            size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
            memcpy((char*)k_cache + dst * eb, (const char*)key + src * eb, (size_t)head_dim * eb);
            memcpy((char*)v_cache + dst * eb, (const char*)value + src * eb, (size_t)head_dim * eb);
        }
    }
    return ORC_OK;
}

/* ---- copy-on-write copy: whole physical block src -> dst, in pair order - */
int orc_kv_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs, int num_pairs,
                       int num_blocks, int num_kv_heads, int head_dim, int block_size, int dtype)
{
    int eb = elem_bytes(dtype);
    if (!eb || num_pairs < 0) return ORC_BAD_ARG;
    size_t blk_bytes = (size_t)num_kv_heads * block_size * head_dim * eb;
    for (int i = 0; i < num_pairs; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return ORC_BAD_BLOCK;
        memcpy((char*)k_cache + dst * blk_bytes, (const char*)k_cache + src * blk_bytes, blk_bytes);
        memcpy((char*)v_cache + dst * blk_bytes, (const char*)v_cache + src * blk_bytes, blk_bytes);
    }
    return ORC_OK;
}

/* ---- swap: whole blocks from one pool to another (preemption by swapping:
 *      a preempted sequence's blocks move to CPU memory and back) --------- */
int orc_kv_swap_blocks(void* dst_k, void* dst_v, const void* src_k, const void* src_v,
                       const int64_t* pairs, int num_pairs, int num_src_blocks,
                       int num_dst_blocks, int num_kv_heads, int head_dim, int block_size,
                       int dtype)
{
    int eb = elem_bytes(dtype);
    if (!eb || num_pairs < 0) return ORC_BAD_ARG;
    size_t blk_bytes = (size_t)num_kv_heads * block_size * head_dim * eb;
    for (int i = 0; i < num_pairs; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_src_blocks || dst < 0 || dst >= num_dst_blocks)
            return ORC_BAD_BLOCK;
        memcpy((char*)dst_k + dst * blk_bytes, (const char*)src_k + src * blk_bytes, blk_bytes);
        memcpy((char*)dst_v + dst * blk_bytes, (const char*)src_v + src * blk_bytes, blk_bytes);
    }
    return ORC_OK;
}

/* ---- decode attention: gather through the block table, then softmax ---- */

typedef struct {
    double* out;            /* [S][Hq][D] */
    const void* q;          /* [S][Hq][D], stored dtype */
    const void* k_cache;
    const void* v_cache;
    int dtype;
    const int32_t* block_tables; /* [S][max_blocks] */
    const int32_t* context_lens; /* [S] */
    double scale;
    int B, Hkv, S, Hq, D, max_blocks, NB;
    int nthreads, tid;
    int status;
} attn_job;

static int attend_one_sequence(const attn_job* j, int s)
{
    const int B = j->B, Hkv = j->Hkv, Hq = j->Hq, D = j->D;
    const int G = Hq / Hkv;
    const int L = j->context_lens[s];
    double* out_s = j->out + (size_t)s * Hq * D;
    if (L < 0 || (int64_t)L > (int64_t)j->max_blocks * B) return ORC_BAD_LEN;
    if (L == 0) {
        memset(out_s, 0, sizeof(double) * (size_t)Hq * D);
        return ORC_OK;
    }

    /* Step 1: logical, contiguous K and V of this sequence: [L][Hkv][D]. */
    double* K = malloc(sizeof(double) * (size_t)L * Hkv * D);
    double* V = malloc(sizeof(double) * (size_t)L * Hkv * D);
    double* z = malloc(sizeof(double) * (size_t)L);
    double* qd = malloc(sizeof(double) * (size_t)D);
    if (!K || !V || !z || !qd) {
        free(K); free(V); free(z); free(qd);
        return ORC_NO_MEM;
    }
    const int32_t* table = j->block_tables + (size_t)s * j->max_blocks;
    for (int i = 0; i < L; ++i) {
        int32_t phys = table[i / B];
        if (phys < 0 || phys >= j->NB) {
            free(K); free(V); free(z); free(qd);
            return ORC_BAD_BLOCK;
        }
        int off = i % B;
        for (int g = 0; g < Hkv; ++g) {
            size_t src = (((size_t)phys * Hkv + g) * B + off) * D;
            size_t dst = ((size_t)i * Hkv + g) * D;
            for (int d = 0; d < D; ++d) {
                K[dst + d] = load_elem(j->k_cache, j->dtype, src + d);
                V[dst + d] = load_elem(j->v_cache, j->dtype, src + d);
            }
        }
    }

    /* Step 2: per query head, softmax(scale * q . k_i) weighted sum of v_i. */
    for (int h = 0; h < Hq; ++h) {
        int g = h / G;
        size_t qoff = ((size_t)s * Hq + h) * D;
        for (int d = 0; d < D; ++d) qd[d] = load_elem(j->q, j->dtype, qoff + d);
        double m = -INFINITY;
        for (int i = 0; i < L; ++i) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qd[d] * K[((size_t)i * Hkv + g) * D + d];
            z[i] = j->scale * dot;
            if (z[i] > m) m = z[i];
        }
        double den = 0.0;
        for (int i = 0; i < L; ++i) {
            z[i] = exp(z[i] - m); /* now p_i */
            den += z[i];
        }
        for (int d = 0; d < D; ++d) {
            double num = 0.0;
            for (int i = 0; i < L; ++i) num += z[i] * V[((size_t)i * Hkv + g) * D + d];
            out_s[(size_t)h * D + d] = num / den;
        }
    }
    free(K); free(V); free(z); free(qd);
    return ORC_OK;
}

/* Multi-token (prefill) form: the query rows query_start[s] ..
 * query_start[s+1]-1 are the last qn tokens of sequence s; row t sits at
 * position L - qn + t and attends causally to tokens 0 .. L - qn + t. */
typedef struct {
    attn_job base;
    const int32_t* query_start;
} prefill_job;

static int prefill_one_sequence(const prefill_job* pj, int s)
{
    const attn_job* j = &pj->base;
    const int B = j->B, Hkv = j->Hkv, Hq = j->Hq, D = j->D;
    const int G = Hq / Hkv;
    const int L = j->context_lens[s];
    const int r0 = pj->query_start[s], qn = pj->query_start[s + 1] - r0;
    if (L < 0 || (int64_t)L > (int64_t)j->max_blocks * B || qn < 0 || qn > L) return ORC_BAD_LEN;
    if (qn == 0) return ORC_OK;
    double* K = malloc(sizeof(double) * (size_t)L * Hkv * D);
    double* V = malloc(sizeof(double) * (size_t)L * Hkv * D);
    double* z = malloc(sizeof(double) * (size_t)L);
    double* qd = malloc(sizeof(double) * (size_t)D);
    if (!K || !V || !z || !qd) {
        free(K); free(V); free(z); free(qd);
        return ORC_NO_MEM;
    }
    const int32_t* table = j->block_tables + (size_t)s * j->max_blocks;
    for (int i = 0; i < L; ++i) {
        int32_t phys = table[i / B];
        if (phys < 0 || phys >= j->NB) {
            free(K); free(V); free(z); free(qd);
            return ORC_BAD_BLOCK;
        }
        for (int g = 0; g < Hkv; ++g)
            for (int d = 0; d < D; ++d) {
                size_t src = (((size_t)phys * Hkv + g) * B + i % B) * D + d;
                K[((size_t)i * Hkv + g) * D + d] = load_elem(j->k_cache, j->dtype, src);
                V[((size_t)i * Hkv + g) * D + d] = load_elem(j->v_cache, j->dtype, src);
            }
    }
    for (int t = 0; t < qn; ++t) {
        const int last = L - qn + t;  /* newest key this row may see */
        for (int h = 0; h < Hq; ++h) {
            const int g = h / G;
            const size_t row = ((size_t)(r0 + t) * Hq + h) * D;
            for (int d = 0; d < D; ++d) qd[d] = load_elem(j->q, j->dtype, row + d);
            double m = -INFINITY;
            for (int i = 0; i <= last; ++i) {
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += qd[d] * K[((size_t)i * Hkv + g) * D + d];
                z[i] = j->scale * dot;
                if (z[i] > m) m = z[i];
            }
            double den = 0.0;
            for (int i = 0; i <= last; ++i) {
                z[i] = exp(z[i] - m);
                den += z[i];
            }
            for (int d = 0; d < D; ++d) {
                double num = 0.0;
                for (int i = 0; i <= last; ++i) num += z[i] * V[((size_t)i * Hkv + g) * D + d];
                j->out[row + d] = num / den;
            }
        }
    }
    free(K); free(V); free(z); free(qd);
    return ORC_OK;
}

static void* prefill_worker(void* arg)
{
    prefill_job* pj = (prefill_job*)arg;
    for (int s = pj->base.tid; s < pj->base.S; s += pj->base.nthreads) {
        int rc = prefill_one_sequence(pj, s);
        if (rc != ORC_OK) {
            pj->base.status = rc;
            break;
        }
    }
    return NULL;
}

static void* attn_worker(void* arg)
{
    attn_job* j = (attn_job*)arg;
    for (int s = j->tid; s < j->S; s += j->nthreads) {
        int rc = attend_one_sequence(j, s);
        if (rc != ORC_OK) {
            j->status = rc;
            break;
        }
    }
    return NULL;
}

/* Sequences are independent, so they are spread over nthreads host threads. */
int orc_paged_decode_attention(double* out, const void* q, const void* k_cache,
                               const void* v_cache, int dtype, const int32_t* block_tables,
                               const int32_t* context_lens, double scale, int block_size,
                               int num_kv_heads, int num_seqs, int num_heads, int head_dim,
                               int max_blocks_per_seq, int num_blocks, int nthreads)
{
    if (!elem_bytes(dtype) || block_size <= 0 || num_kv_heads <= 0 || num_heads <= 0 ||
        head_dim <= 0 || num_seqs < 0 || num_heads % num_kv_heads != 0)
        return ORC_BAD_ARG;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > num_seqs) nthreads = num_seqs > 0 ? num_seqs : 1;

    attn_job* jobs = calloc((size_t)nthreads, sizeof(attn_job));
    pthread_t* th = calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs); free(th);
        return ORC_NO_MEM;
    }
    for (int t = 0; t < nthreads; ++t) {
        attn_job j = {out, q, k_cache, v_cache, dtype, block_tables, context_lens, scale,
                      block_size, num_kv_heads, num_seqs, num_heads, head_dim,
                      max_blocks_per_seq, num_blocks, nthreads, t, ORC_OK};
        jobs[t] = j;
    }
    int rc = ORC_OK;
    if (nthreads == 1) {
        attn_worker(&jobs[0]);
    } else {
        int started = 0;
        for (int t = 0; t < nthreads; ++t) {
            if (pthread_create(&th[t], NULL, attn_worker, &jobs[t]) != 0) break;
            ++started;
        }
        for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
        if (started != nthreads) {
            /* finish the strides of threads that could not be started */
            for (int t = started; t < nthreads; ++t) attn_worker(&jobs[t]);
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != ORC_OK) rc = jobs[t].status;
    free(jobs);
    free(th);
    return rc;
}

/* out: [total rows][num_heads][head_dim] doubles, rows as query_start says. */
int orc_paged_prefill_attention(double* out, const void* q, const void* k_cache,
                                const void* v_cache, int dtype, const int32_t* block_tables,
                                const int32_t* context_lens, const int32_t* query_start,
                                double scale, int block_size, int num_kv_heads, int num_seqs,
                                int num_heads, int head_dim, int max_blocks_per_seq,
                                int num_blocks, int nthreads)
{
    if (!elem_bytes(dtype) || block_size <= 0 || num_kv_heads <= 0 || num_heads <= 0 ||
        head_dim <= 0 || num_seqs < 0 || num_heads % num_kv_heads != 0)
        return ORC_BAD_ARG;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > num_seqs) nthreads = num_seqs > 0 ? num_seqs : 1;
    prefill_job* jobs = calloc((size_t)nthreads, sizeof(prefill_job));
    pthread_t* th = calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs); free(th);
        return ORC_NO_MEM;
    }
    for (int t = 0; t < nthreads; ++t) {
        attn_job j = {out, q, k_cache, v_cache, dtype, block_tables, context_lens, scale,
                      block_size, num_kv_heads, num_seqs, num_heads, head_dim,
                      max_blocks_per_seq, num_blocks, nthreads, t, ORC_OK};
        jobs[t].base = j;
        jobs[t].query_start = query_start;
    }
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, prefill_worker, &jobs[t]) != 0) break;
        ++started;
    }
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    for (int t = started; t < nthreads; ++t) prefill_worker(&jobs[t]);
    int rc = ORC_OK;
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].base.status != ORC_OK) rc = jobs[t].base.status;
    free(jobs);
    free(th);
    return rc;
}
