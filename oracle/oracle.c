/*
 * oracle.c -- float64 CPU oracle for paged decode attention and the
 * cache write that precedes it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline arm use it.  It shares no code, header, table or constant with
 * the CUDA library: it is written from the plain definitions below.
 *
 * What it computes
 * ----------------
 * Paged KV cache (Qualiteg, "About PagedAttention for LLM serving": the
 * section on logical blocks, physical blocks and the block table, and point
 * 1-2 under "[Regarding Problem 1]" on splitting the cache into blocks): the keys and
 * values of a sequence live in fixed-size blocks of a shared pool; logical
 * block i of sequence s is physical block block_tables[s][i].  Storage order
 * inside the pool (our choice, stated with the library): separate K and V
 * pools, each [num_blocks][num_kv_heads][block_size][head_dim].
 *
 * Attention (vAttention, section 3.1 "Requires re-writing the attention
 * kernel", which names the attention operator over K and V but does not
 * print it): the standard scaled dot-product form.  For sequence s and query
 * head h with kv head g = h / (num_heads / num_kv_heads) (contiguous GQA
 * grouping), gather K[j], V[j] for logical positions j < ctx[s] into
 * contiguous arrays, then
 *     z_j = scale * <q[s][h], K[j]>
 *     p_j = exp(z_j - max z) / sum_i exp(z_i - max z)
 *     out[s][h] = sum_j p_j V[j]
 * all in float64 on the exact input values (bf16 and fp16 widened exactly).
 * ctx = 0 yields a zero row (softmax over an empty set is undefined).
 *
 * Cache write: each new token t with slot = slot_mapping[t] >= 0 copies its
 * [num_kv_heads][head_dim] key and value rows into
 * pool[slot / block_size][h][slot % block_size][:]; slots < 0 are padding and
 * skipped; slots past the pool are counted as faults and skipped.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2 };

static int elem_size(int dtype) { return dtype == ORACLE_F32 ? 4 : 2; }

/* Exact value of an IEEE binary16 bit pattern: sign, 5-bit exponent (bias
 * 15), 10-bit fraction; exponent 0 holds the subnormals frac * 2^-24. */
static double half_value(uint16_t h) {
    const int sign = h >> 15, ex = (h >> 10) & 31, frac = h & 1023;
    double v;
    if (ex == 0)
        v = ldexp((double)frac, -24);
    else if (ex == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), ex - 25);
    return sign ? -v : v;
}

/* Exact widening of one stored element to float64.  bf16 is the top half of
 * an IEEE binary32, so shifting its 16 bits up gives the same value. */
static double load_elem(const void *base, int dtype, size_t idx) {
    if (dtype == ORACLE_F16) {
        uint16_t h;
        memcpy(&h, (const char *)base + idx * 2, 2);
        return half_value(h);
    }
    if (dtype == ORACLE_BF16) {
        uint16_t h;
        memcpy(&h, (const char *)base + idx * 2, 2);
        uint32_t w = (uint32_t)h << 16;
        float f;
        memcpy(&f, &w, 4);
        return (double)f;
    }
    float f;
    memcpy(&f, (const char *)base + idx * 4, 4);
    return (double)f;
}

/* Plain attention of one query row over contiguous K[ctx][D], V[ctx][D]. */
int oracle_attention_contiguous(double *out, const double *q, const double *K,
                                const double *V, int ctx, int head_dim, double scale) {
    if (ctx < 0 || head_dim <= 0) return -1;
    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    if (ctx == 0) return 0;
    double *z = (double *)malloc(sizeof(double) * (size_t)ctx);
    if (!z) return -2;
    double zmax = -INFINITY;
    for (int j = 0; j < ctx; ++j) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d) dot += q[d] * K[(size_t)j * head_dim + d];
        z[j] = scale * dot;
        if (z[j] > zmax) zmax = z[j];
    }
    double denom = 0.0;
    for (int j = 0; j < ctx; ++j) {
        z[j] = exp(z[j] - zmax);
        denom += z[j];
    }
    for (int j = 0; j < ctx; ++j) {
        double p = z[j] / denom;
        for (int d = 0; d < head_dim; ++d) out[d] += p * V[(size_t)j * head_dim + d];
    }
    free(z);
    return 0;
}

typedef struct {
    double *out;
    const void *query, *k_pool, *v_pool;
    int dtype, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    const int32_t *context_lens;
    double scale;
    int next;              /* next (s, h) work item, taken atomically */
    int status;
    pthread_mutex_t lock;
} decode_job;

static int take(decode_job *job) {
    return __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
}

static void *decode_worker(void *arg) {
    decode_job *job = (decode_job *)arg;
    const int D = job->head_dim, BS = job->block_size, Hkv = job->num_kv_heads;
    const int group = job->num_heads / job->num_kv_heads;
    double *K = NULL, *V = NULL, *q = (double *)malloc(sizeof(double) * (size_t)D);
    size_t cap = 0;
    for (;;) {
        int item = take(job);
        if (item >= job->num_seqs * job->num_heads) break;
        int s = item / job->num_heads, h = item % job->num_heads, g = h / group;
        int ctx = job->context_lens[s];
        double *o = job->out + ((size_t)s * job->num_heads + h) * D;
        for (int d = 0; d < D; ++d)
            q[d] = load_elem(job->query, job->dtype, ((size_t)s * job->num_heads + h) * D + d);
        if (ctx > cap) {
            free(K);
            free(V);
            cap = (size_t)ctx;
            K = (double *)malloc(sizeof(double) * cap * D);
            V = (double *)malloc(sizeof(double) * cap * D);
        }
        int bad = 0;
        /* gather: logical position j -> block_tables[s][j / BS], row j % BS */
        for (int j = 0; j < ctx && !bad; ++j) {
            int lb = j / BS;
            int pb = lb < job->max_blocks_per_seq
                         ? job->block_tables[(size_t)s * job->max_blocks_per_seq + lb] : -1;
            if (pb < 0 || pb >= job->num_blocks) { bad = 1; break; }
            size_t row = (((size_t)pb * Hkv + g) * BS + (size_t)(j % BS)) * D;
            for (int d = 0; d < D; ++d) {
                K[(size_t)j * D + d] = load_elem(job->k_pool, job->dtype, row + d);
                V[(size_t)j * D + d] = load_elem(job->v_pool, job->dtype, row + d);
            }
        }
        if (bad) {
            pthread_mutex_lock(&job->lock);
            job->status = -3;
            pthread_mutex_unlock(&job->lock);
            for (int d = 0; d < D; ++d) o[d] = NAN;
            continue;
        }
        if (oracle_attention_contiguous(o, q, K, V, ctx, D, job->scale) != 0) {
            pthread_mutex_lock(&job->lock);
            job->status = -2;
            pthread_mutex_unlock(&job->lock);
        }
    }
    free(K);
    free(V);
    free(q);
    return NULL;
}

/*
 * out: float64 [num_seqs][num_heads][head_dim].  query: [num_seqs][num_heads]
 * [head_dim] in `dtype`.  Pools: [num_blocks][num_kv_heads][block_size]
 * [head_dim] in `dtype`.  Returns 0, -1 on bad shapes, -3 if a block-table
 * entry a context position needs is out of range (that row is NaN).
 */
int oracle_paged_decode(double *out, const void *query, const void *k_pool, const void *v_pool,
                        int dtype, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                        int block_size, int num_blocks, const int32_t *block_tables,
                        int max_blocks_per_seq, const int32_t *context_lens, double scale,
                        int num_threads) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_heads % num_kv_heads != 0)
        return -1;
    for (int s = 0; s < num_seqs; ++s)
        if (context_lens[s] < 0) return -1;
    decode_job job;
    memset(&job, 0, sizeof(job));
    job.out = out; job.query = query; job.k_pool = k_pool; job.v_pool = v_pool;
    job.dtype = dtype; job.num_seqs = num_seqs; job.num_heads = num_heads;
    job.num_kv_heads = num_kv_heads; job.head_dim = head_dim; job.block_size = block_size;
    job.num_blocks = num_blocks; job.block_tables = block_tables;
    job.max_blocks_per_seq = max_blocks_per_seq; job.context_lens = context_lens;
    job.scale = scale;
    pthread_mutex_init(&job.lock, NULL);
    if (num_threads < 1) num_threads = 1;
    if (num_threads > 256) num_threads = 256;
    pthread_t th[256];
    int started = 0;
    for (int t = 1; t < num_threads; ++t)
        if (pthread_create(&th[started], NULL, decode_worker, &job) == 0) ++started;
    decode_worker(&job);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&job.lock);
    return job.status;
}

/*
 * Scatter each new token's key/value rows into its pool slot.  key/value:
 * [num_tokens][num_kv_heads][head_dim] in the pool's element type (copied as
 * bytes).  Returns the number of slots past the pool (each skipped).
 */
int oracle_reshape_and_cache(void *k_pool, void *v_pool, int dtype, int num_blocks,
                             int block_size, int num_kv_heads, int head_dim, const void *key,
                             const void *value, const int64_t *slot_mapping, int num_tokens) {
    const size_t es = (size_t)elem_size(dtype);
    const size_t row_bytes = (size_t)head_dim * es;
    int faults = 0;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) { ++faults; continue; }
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t dst = ((((size_t)blk * num_kv_heads + h) * block_size) + (size_t)off) * row_bytes;
            size_t src = ((size_t)t * num_kv_heads + h) * row_bytes;
            memcpy((char *)k_pool + dst, (const char *)key + src, row_bytes);
            memcpy((char *)v_pool + dst, (const char *)value + src, row_bytes);
        }
    }
    return faults;
}
