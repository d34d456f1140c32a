/*
 * pkv_oracle.c -- plain CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may call,
 * link or load this file; only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no source, header, helper or
 * table with the CUDA library.
 *
 * What it computes, and where the pages define it:
 *
 *  - The KV cache is cut into fixed blocks of 16 tokens that may sit anywhere
 *    in the pool; each request keeps a block table mapping its logical block
 *    i to a physical block ("PagedAttention: splitting KV into blocks",
 *    section 2, subsection "Blocks and block tables", of the serving-engine KV
 *    blog).  Token p of a sequence is therefore row p % 16 of physical block
 *    block_table[p / 16].  Pool layout: [num_blocks][num_kv_heads][16][d].
 *
 *  - The attention kernel walks the block table and reads K/V from the
 *    scattered blocks, and the result is the same as with one contiguous
 *    array (same subsection).  So the oracle first gathers each sequence's
 *    rows into contiguous arrays and then evaluates the plain definition
 *        out = softmax(scale * q K^T) V
 *    over them, in double precision, in the order the definition is written
 *    (scores, their maximum, exponentials, their sum, weighted V sum).
 *
 *  - Decode computes only the new token's column and reads every past column
 *    from the cache ("KV Cache" section of the inference-engine talk
 *    write-up); this step's K/V are written to the cache before attention,
 *    so a decode row attends to context_lens[s] keys including itself.
 *
 *  - Chunked prefill splits a long prompt into consecutive slices that share
 *    a step with single decode tokens ("Chunked Prefill" section of the same
 *    write-up).  A query row at absolute position pos attends keys 0..pos
 *    (causal).  Query row i of sequence s sits at position
 *    context_lens[s] - query_len[s] + i; a decode row is query_len = 1.
 *
 *  - Copy-on-write: a block shared by several requests (reference counted)
 *    is copied only when someone has to append to it ("Sharing blocks"
 *    subsection).  copy_blocks copies whole blocks, all 16 slots of every kv
 *    head, K and V.
 *
 *  - cache_write stores this step's new K/V rows into their slots
 *    (block = slot / 16, row = slot % 16); a negative slot means "skip".
 *
 * Readings where the pages are silent (the library takes the same ones):
 *  - scale is passed in (1/sqrt(d) in every workload);
 *  - q head h reads kv head h / (Hq / Hkv) (contiguous GQA groups);
 *  - a sequence with context 0 produces a zero output row;
 *  - bf16 inputs are widened exactly (bf16 is the top half of binary32).
 *
 * Threads: sequences are dealt to pthreads round-robin; each thread's
 * arithmetic is the same sequential loop a single thread would run.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_RANGE (-2)
#define ORACLE_ERR_NOMEM (-3)

/* bf16 bit pattern -> double: place the 16 bits in the top half of a binary32. */
static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Exposed for the tests: widen n bf16 values to double. */
void oracle_bf16_to_f64(const uint16_t* src, double* dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i) dst[i] = bf16_to_double(src[i]);
}

/* ------------------------------------------------------------------------ */
/* cache_write: one row per (token, kv head), K and V.                       */
/* ------------------------------------------------------------------------ */
int oracle_cache_write(uint16_t* k_pool, uint16_t* v_pool, int64_t num_blocks, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, const uint16_t* k_new, const uint16_t* v_new,
                       const int32_t* slot_mapping, int64_t num_tokens) {
    if (num_blocks < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_tokens < 0)
        return ORACLE_ERR_ARG;
    const int64_t row = head_dim;
    const int64_t block_elems = (int64_t)num_kv_heads * block_size * head_dim;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;                         /* skipped token */
        if (slot >= num_blocks * block_size) return ORACLE_ERR_RANGE;
        int64_t block = slot / block_size;
        int64_t off = slot % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            int64_t dst = block * block_elems + ((int64_t)h * block_size + off) * head_dim;
            int64_t src = (t * num_kv_heads + h) * row;
            memcpy(k_pool + dst, k_new + src, (size_t)row * sizeof(uint16_t));
            memcpy(v_pool + dst, v_new + src, (size_t)row * sizeof(uint16_t));
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* copy_blocks: pool[dst[i]] <- pool[src[i]], whole blocks, K and V; a pair  */
/* with a negative src is skipped.                                           */
/* ------------------------------------------------------------------------ */
int oracle_copy_blocks(uint16_t* k_pool, uint16_t* v_pool, int64_t num_blocks, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, const int32_t* src, const int32_t* dst, int64_t n) {
    if (num_blocks < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || n < 0) return ORACLE_ERR_ARG;
    const int64_t block_elems = (int64_t)num_kv_heads * block_size * head_dim;
    for (int64_t i = 0; i < n; ++i) {
        if (src[i] < 0) continue;                       /* unused pair entry: skipped */
        if (src[i] >= num_blocks || dst[i] < 0 || dst[i] >= num_blocks) return ORACLE_ERR_RANGE;
        memmove(k_pool + (int64_t)dst[i] * block_elems, k_pool + (int64_t)src[i] * block_elems,
                (size_t)block_elems * sizeof(uint16_t));
        memmove(v_pool + (int64_t)dst[i] * block_elems, v_pool + (int64_t)src[i] * block_elems,
                (size_t)block_elems * sizeof(uint16_t));
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Paged causal attention (decode rows are the query_len == 1 case).         */
/* ------------------------------------------------------------------------ */
typedef struct {
    const uint16_t* k_pool;
    const uint16_t* v_pool;
    int64_t num_blocks;
    int32_t hkv, d, bs;
    const uint16_t* q;
    int32_t hq;
    const int32_t* qsl;
    const int32_t* ctx;
    int32_t num_seqs;
    const int32_t* tables;
    int32_t max_blocks;
    double scale;
    double* out;
    int32_t tid, nthreads;
    int status;
} attn_job;

/* Gather rows 0..n-1 of kv head h of sequence s into contiguous [n][d] arrays. */
static int gather_contiguous(const attn_job* J, int32_t s, int32_t h, int64_t n, double* Kc, double* Vc) {
    const int64_t block_elems = (int64_t)J->hkv * J->bs * J->d;
    for (int64_t j = 0; j < n; ++j) {
        int64_t logical = j / J->bs;
        int64_t off = j % J->bs;
        if (logical >= J->max_blocks) return ORACLE_ERR_RANGE;
        int64_t phys = J->tables[(int64_t)s * J->max_blocks + logical];
        if (phys < 0 || phys >= J->num_blocks) return ORACLE_ERR_RANGE;
        int64_t base = phys * block_elems + ((int64_t)h * J->bs + off) * J->d;
        for (int32_t c = 0; c < J->d; ++c) {
            Kc[j * J->d + c] = bf16_to_double(J->k_pool[base + c]);
            Vc[j * J->d + c] = bf16_to_double(J->v_pool[base + c]);
        }
    }
    return ORACLE_OK;
}

static void* attn_worker(void* arg) {
    attn_job* J = (attn_job*)arg;
    const int32_t group = J->hq / J->hkv;
    int64_t max_n = 0;
    for (int32_t s = 0; s < J->num_seqs; ++s)
        if (J->ctx[s] > max_n) max_n = J->ctx[s];
    double* Kc = (double*)malloc((size_t)(max_n > 0 ? max_n : 1) * J->d * sizeof(double));
    double* Vc = (double*)malloc((size_t)(max_n > 0 ? max_n : 1) * J->d * sizeof(double));
    double* x = (double*)malloc((size_t)(max_n > 0 ? max_n : 1) * sizeof(double));
    double* qd = (double*)malloc((size_t)J->d * sizeof(double));
    double* acc = (double*)malloc((size_t)J->d * sizeof(double));
    if (!Kc || !Vc || !x || !qd || !acc) {
        J->status = ORACLE_ERR_NOMEM;
        goto done;
    }
    for (int32_t s = J->tid; s < J->num_seqs; s += J->nthreads) {
        const int64_t n = J->ctx[s];
        const int64_t row0 = J->qsl[s];
        const int64_t qlen = (int64_t)J->qsl[s + 1] - J->qsl[s];
        if (qlen <= 0) continue;
        if (n <= 0) { /* empty context: zero output rows */
            memset(J->out + row0 * J->hq * J->d, 0, (size_t)(qlen * J->hq * J->d) * sizeof(double));
            continue;
        }
        for (int32_t g = 0; g < J->hkv; ++g) {
            int rc = gather_contiguous(J, s, g, n, Kc, Vc);
            if (rc != ORACLE_OK) { J->status = rc; goto done; }
            for (int32_t h = g * group; h < (g + 1) * group; ++h) {
                for (int64_t i = 0; i < qlen; ++i) {
                    const int64_t pos = n - qlen + i;       /* keys 0..pos are visible */
                    const uint16_t* qrow = J->q + ((row0 + i) * J->hq + h) * J->d;
                    double* orow = J->out + ((row0 + i) * J->hq + h) * J->d;
                    for (int32_t c = 0; c < J->d; ++c) qd[c] = bf16_to_double(qrow[c]);
                    /* scores */
                    for (int64_t j = 0; j <= pos; ++j) {
                        double dot = 0.0;
                        for (int32_t c = 0; c < J->d; ++c) dot += qd[c] * Kc[j * J->d + c];
                        x[j] = J->scale * dot;
                    }
                    /* softmax: max, exponentials, sum */
                    double m = x[0];
                    for (int64_t j = 1; j <= pos; ++j)
                        if (x[j] > m) m = x[j];
                    double L = 0.0;
                    for (int64_t j = 0; j <= pos; ++j) {
                        x[j] = exp(x[j] - m);
                        L += x[j];
                    }
                    /* weighted sum of V rows, normalised */
                    for (int32_t c = 0; c < J->d; ++c) acc[c] = 0.0;
                    for (int64_t j = 0; j <= pos; ++j)
                        for (int32_t c = 0; c < J->d; ++c) acc[c] += x[j] * Vc[j * J->d + c];
                    for (int32_t c = 0; c < J->d; ++c) orow[c] = acc[c] / L;
                }
            }
        }
    }
done:
    free(Kc);
    free(Vc);
    free(x);
    free(qd);
    free(acc);
    return NULL;
}

/*
 * q       : bf16 bits [num_tokens][hq][d], rows of sequence s are
 *           query_start_loc[s] .. query_start_loc[s+1]-1
 * out     : double    [num_tokens][hq][d]
 * returns : 0, or a negative error (bad argument / block id out of range /
 *           out of memory).
 */
int oracle_paged_attention(const uint16_t* k_pool, const uint16_t* v_pool, int64_t num_blocks, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, const uint16_t* q, int32_t num_q_heads,
                           const int32_t* query_start_loc, const int32_t* context_lens, int32_t num_seqs,
                           const int32_t* block_tables, int32_t max_blocks_per_seq, double scale, double* out,
                           int32_t num_threads) {
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || num_seqs < 0 || max_blocks_per_seq < 0)
        return ORACLE_ERR_ARG;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t qlen = query_start_loc[s + 1] - query_start_loc[s];
        if (qlen < 0) return ORACLE_ERR_ARG;
        if (context_lens[s] > 0 && qlen > context_lens[s]) return ORACLE_ERR_ARG;
        if ((int64_t)context_lens[s] > (int64_t)max_blocks_per_seq * block_size) return ORACLE_ERR_RANGE;
    }
    if (num_threads < 1) num_threads = 1;
    if (num_threads > num_seqs && num_seqs > 0) num_threads = num_seqs;
    attn_job* jobs = (attn_job*)calloc((size_t)num_threads, sizeof(attn_job));
    pthread_t* th = (pthread_t*)calloc((size_t)num_threads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return ORACLE_ERR_NOMEM;
    }
    for (int32_t t = 0; t < num_threads; ++t) {
        attn_job* J = &jobs[t];
        J->k_pool = k_pool; J->v_pool = v_pool; J->num_blocks = num_blocks;
        J->hkv = num_kv_heads; J->d = head_dim; J->bs = block_size;
        J->q = q; J->hq = num_q_heads; J->qsl = query_start_loc; J->ctx = context_lens;
        J->num_seqs = num_seqs; J->tables = block_tables; J->max_blocks = max_blocks_per_seq;
        J->scale = scale; J->out = out; J->tid = t; J->nthreads = num_threads; J->status = ORACLE_OK;
    }
    int started = 0;
    for (int32_t t = 1; t < num_threads; ++t) {
        if (pthread_create(&th[t], NULL, attn_worker, &jobs[t]) != 0) break;
        started = t;
    }
    attn_worker(&jobs[0]);
    for (int32_t t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    int rc = ORACLE_OK;
    for (int32_t t = 0; t < num_threads; ++t)
        if (jobs[t].status != ORACLE_OK) rc = jobs[t].status;
    /* threads that failed to start: run their share here */
    for (int32_t t = started + 1; t < num_threads && rc == ORACLE_OK; ++t) {
        attn_worker(&jobs[t]);
        if (jobs[t].status != ORACLE_OK) rc = jobs[t].status;
    }
    free(jobs);
    free(th);
    return rc;
}
