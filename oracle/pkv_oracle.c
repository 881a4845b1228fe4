/*
 * pkv_oracle.c -- plain fp64 CPU oracle for PagedAttention decode.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline / reference arm of bench.py may load or call this library.
 * The product path (the CUDA library and its Python binding) never does,
 * and this file shares no code, header or table with it.
 *
 * What it computes
 * ----------------
 * "PagedAttention: gestionar la KV cache como memoria de un sistema
 * operativo" (josueisai.com), section "Cómo funciona por dentro": the
 * attention for one query walks the sequence's block table in logical order,
 * reads each physical block's keys and values, scores the query against the
 * keys and returns the softmax-weighted sum of the values.  The page leaves
 * the normalisation helper undefined; this oracle takes the textbook
 * definition: x_t = scale * <q, K_t>, p = exp(x - max x) / sum exp(x - max x),
 * out = sum_t p_t V_t.
 *
 * "Batching Continuo y PagedAttention" (cruxr.ai), section "PagedAttention:
 * Memoria virtual para la KV cache": blocks hold a fixed P = 16 tokens;
 * logical block i holds tokens 16i .. 16i+15 and maps to a physical block id
 * through the per-sequence table.
 *
 * Everything is done in double precision after an exact widening of the
 * stored elements (fp32 values, or bf16 bit patterns shifted into the top 16
 * bits of an fp32).  Each (sequence, kv head) is gathered into contiguous
 * arrays first, so the arithmetic is the unpaged definition, with no
 * blocking, partitioning or online rescaling.
 *
 * Layout of the caches (the library's chosen layout; the pages state a block
 * holds 2*P*d_h elements per layer and head but fix no order):
 *   cache[num_blocks][num_kv_heads][16][head_dim]
 * Query heads map to kv heads by consecutive grouping:
 *   kv_head = q_head / (num_q_heads / num_kv_heads).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PKV_ORACLE_BLOCK 16

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* error codes */
#define ORACLE_OK 0
#define ORACLE_EARG -1        /* bad scalar argument */
#define ORACLE_EINDEX -3      /* block id out of range, or length beyond the table */
#define ORACLE_ENOMEM -6

static double widen(const void *base, size_t idx, int dtype) {
    if (dtype == ORACLE_F32) {
        return (double)((const float *)base)[idx];
    }
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

typedef struct {
    double *out;
    const void *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens, *seq_ids;
    double scale;
    int num_kv_heads, num_q_heads, head_dim, max_blocks_per_seq, num_blocks, dtype;
    int num_out_seqs;
    int nthreads;
    int thread_index;
    int status;
} job_t;

/* One (sequence, kv head): gather, then textbook softmax attention for each
 * query head of the group. */
static int one_unit(const job_t *j, int out_row, int s, int hkv, double *K, double *V, double *x) {
    const int d = j->head_dim;
    const int g = j->num_q_heads / j->num_kv_heads;
    const int len = j->context_lens[s];
    double *out_base = j->out + ((size_t)out_row * j->num_q_heads) * d;

    if (len < 0) return ORACLE_EINDEX;
    if (len == 0) {
        /* Empty context: the library defines the output as zeros. */
        for (int n = 0; n < g; ++n)
            for (int i = 0; i < d; ++i) out_base[(size_t)(hkv * g + n) * d + i] = 0.0;
        return ORACLE_OK;
    }
    if (len > j->max_blocks_per_seq * PKV_ORACLE_BLOCK) return ORACLE_EINDEX;

    /* Gather: token t lives in logical block t/16, slot t%16. */
    for (int t = 0; t < len; ++t) {
        int32_t blk = j->block_tables[(size_t)s * j->max_blocks_per_seq + t / PKV_ORACLE_BLOCK];
        if (blk < 0 || blk >= j->num_blocks) return ORACLE_EINDEX;
        size_t row = (((size_t)blk * j->num_kv_heads + hkv) * PKV_ORACLE_BLOCK + t % PKV_ORACLE_BLOCK) * d;
        for (int i = 0; i < d; ++i) {
            K[(size_t)t * d + i] = widen(j->k_cache, row + i, j->dtype);
            V[(size_t)t * d + i] = widen(j->v_cache, row + i, j->dtype);
        }
    }

    for (int n = 0; n < g; ++n) {
        const int hq = hkv * g + n;
        const size_t qrow = ((size_t)s * j->num_q_heads + hq) * d;
        double mx = -INFINITY;
        for (int t = 0; t < len; ++t) {
            double dot = 0.0;
            for (int i = 0; i < d; ++i) dot += widen(j->q, qrow + i, j->dtype) * K[(size_t)t * d + i];
            x[t] = j->scale * dot;
            if (x[t] > mx) mx = x[t];
        }
        double z = 0.0;
        for (int t = 0; t < len; ++t) {
            x[t] = exp(x[t] - mx);
            z += x[t];
        }
        double *o = out_base + (size_t)hq * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        for (int t = 0; t < len; ++t) {
            const double p = x[t] / z;
            for (int i = 0; i < d; ++i) o[i] += p * V[(size_t)t * d + i];
        }
    }
    return ORACLE_OK;
}

static void *worker(void *arg) {
    job_t *j = (job_t *)arg;
    const int d = j->head_dim;
    int maxlen = j->max_blocks_per_seq * PKV_ORACLE_BLOCK;
    double *K = (double *)malloc((size_t)maxlen * d * sizeof(double));
    double *V = (double *)malloc((size_t)maxlen * d * sizeof(double));
    double *x = (double *)malloc((size_t)maxlen * sizeof(double));
    j->status = ORACLE_OK;
    if (!K || !V || !x) {
        j->status = ORACLE_ENOMEM;
    } else {
        const long units = (long)j->num_out_seqs * j->num_kv_heads;
        for (long u = j->thread_index; u < units; u += j->nthreads) {
            int row = (int)(u / j->num_kv_heads);
            int hkv = (int)(u % j->num_kv_heads);
            int s = j->seq_ids ? j->seq_ids[row] : row;
            int rc = one_unit(j, row, s, hkv, K, V, x);
            if (rc != ORACLE_OK) {
                j->status = rc;
                break;
            }
        }
    }
    free(K);
    free(V);
    free(x);
    return NULL;
}

/*
 * out[num_out_seqs][num_q_heads][head_dim] (double) receives the attention of
 * sequence seq_ids[i] (or i when seq_ids is NULL, with num_out_seqs equal to
 * the batch size) for every query head.
 * q[num_seqs][num_q_heads][head_dim], caches as in the header comment; both
 * fp32 or both bf16 bit patterns (dtype).
 * Returns 0, or a negative code; the output is then unspecified.
 */
int oracle_paged_decode_attention(double *out, const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_tables, const int32_t *context_lens, double scale,
                                  int num_kv_heads, int num_q_heads, int head_dim, int max_blocks_per_seq,
                                  int num_blocks, int dtype, const int32_t *seq_ids, int num_out_seqs,
                                  int nthreads) {
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0) return ORACLE_EARG;
    if (head_dim <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || num_out_seqs < 0) return ORACLE_EARG;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return ORACLE_EARG;
    if (num_out_seqs == 0) return ORACLE_OK;
    if (nthreads < 1) nthreads = 1;
    long units = (long)num_out_seqs * num_kv_heads;
    if (nthreads > units) nthreads = (int)units;

    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return ORACLE_ENOMEM;
    }
    for (int t = 0; t < nthreads; ++t) {
        job_t *j = &jobs[t];
        j->out = out;
        j->q = q;
        j->k_cache = k_cache;
        j->v_cache = v_cache;
        j->block_tables = block_tables;
        j->context_lens = context_lens;
        j->seq_ids = seq_ids;
        j->scale = scale;
        j->num_kv_heads = num_kv_heads;
        j->num_q_heads = num_q_heads;
        j->head_dim = head_dim;
        j->max_blocks_per_seq = max_blocks_per_seq;
        j->num_blocks = num_blocks;
        j->dtype = dtype;
        j->num_out_seqs = num_out_seqs;
        j->nthreads = nthreads;
        j->thread_index = t;
    }
    int status = ORACLE_OK;
    if (nthreads == 1) {
        worker(&jobs[0]);
        status = jobs[0].status;
    } else {
        int started = 0;
        for (int t = 0; t < nthreads; ++t) {
            if (pthread_create(&tid[t], NULL, worker, &jobs[t]) != 0) break;
            ++started;
        }
        for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
        if (started < nthreads) status = ORACLE_ENOMEM;
        for (int t = 0; t < started; ++t)
            if (jobs[t].status != ORACLE_OK) status = jobs[t].status;
    }
    free(jobs);
    free(tid);
    return status;
}

/*
 * Causal attention for the prefill of several new tokens per sequence
 * ("Batching Continuo y PagedAttention" (cruxr.ai), section "Juntándolo todo:
 * Arquitectura de vLLM": the prefill processes the whole prompt in one
 * forward pass to fill the KV cache; "Continuous Batching" (ultralytics.com
 * glossary), section "Cómo funciona la planificación a nivel de iteración":
 * long prompts are prefilled in chunks).
 *
 * Sequence s has context_lens[s] tokens in the cache, the last n_s of which
 * are its new tokens, n_s = query_start[s+1] - query_start[s]; query row
 * query_start[s] + i is the token at position context_lens[s] - n_s + i and
 * attends, causally, to positions 0 .. context_lens[s] - n_s + i. The textbook
 * definition per query: x_t = scale <q, K_t> over those positions, softmax,
 * weighted sum of V_t.
 * q, out: [total queries][num_q_heads][head_dim]; out in double.
 */
typedef struct {
    double *out;
    const void *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens, *query_start;
    double scale;
    int num_kv_heads, num_q_heads, head_dim, max_blocks_per_seq, num_blocks, dtype, num_seqs;
    int nthreads, thread_index, status;
} prefill_job_t;

static void *prefill_worker(void *arg) {
    prefill_job_t *j = (prefill_job_t *)arg;
    const int d = j->head_dim, g = j->num_q_heads / j->num_kv_heads;
    const int maxlen = j->max_blocks_per_seq * PKV_ORACLE_BLOCK;
    double *K = (double *)malloc((size_t)maxlen * d * sizeof(double));
    double *V = (double *)malloc((size_t)maxlen * d * sizeof(double));
    double *x = (double *)malloc((size_t)maxlen * sizeof(double));
    j->status = ORACLE_OK;
    if (!K || !V || !x) j->status = ORACLE_ENOMEM;
    const long units = (long)j->num_seqs * j->num_kv_heads;
    for (long u = j->thread_index; u < units && j->status == ORACLE_OK; u += j->nthreads) {
        const int s = (int)(u / j->num_kv_heads), hkv = (int)(u % j->num_kv_heads);
        const int len = j->context_lens[s];
        const int q0 = j->query_start[s], n = j->query_start[s + 1] - q0;
        if (len < 0 || len > maxlen || n < 0 || n > len) {
            j->status = ORACLE_EINDEX;
            break;
        }
        for (int t = 0; t < len; ++t) {
            int32_t blk = j->block_tables[(size_t)s * j->max_blocks_per_seq + t / PKV_ORACLE_BLOCK];
            if (blk < 0 || blk >= j->num_blocks) {
                j->status = ORACLE_EINDEX;
                break;
            }
            size_t row = (((size_t)blk * j->num_kv_heads + hkv) * PKV_ORACLE_BLOCK + t % PKV_ORACLE_BLOCK) * d;
            for (int i = 0; i < d; ++i) {
                K[(size_t)t * d + i] = widen(j->k_cache, row + i, j->dtype);
                V[(size_t)t * d + i] = widen(j->v_cache, row + i, j->dtype);
            }
        }
        if (j->status != ORACLE_OK) break;
        for (int qi = 0; qi < n; ++qi) {
            const int pos = len - n + qi;  /* this query's position: it sees keys 0 .. pos */
            for (int m = 0; m < g; ++m) {
                const int hq = hkv * g + m;
                const size_t qrow = ((size_t)(q0 + qi) * j->num_q_heads + hq) * d;
                double mx = -INFINITY;
                for (int t = 0; t <= pos; ++t) {
                    double dot = 0.0;
                    for (int i = 0; i < d; ++i) dot += widen(j->q, qrow + i, j->dtype) * K[(size_t)t * d + i];
                    x[t] = j->scale * dot;
                    if (x[t] > mx) mx = x[t];
                }
                double z = 0.0;
                for (int t = 0; t <= pos; ++t) {
                    x[t] = exp(x[t] - mx);
                    z += x[t];
                }
                double *o = j->out + qrow;
                for (int i = 0; i < d; ++i) o[i] = 0.0;
                for (int t = 0; t <= pos; ++t) {
                    const double p = x[t] / z;
                    for (int i = 0; i < d; ++i) o[i] += p * V[(size_t)t * d + i];
                }
            }
        }
    }
    free(K);
    free(V);
    free(x);
    return NULL;
}

int oracle_paged_prefill_attention(double *out, const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, const int32_t *context_lens,
                                   const int32_t *query_start, double scale, int num_kv_heads, int num_q_heads,
                                   int head_dim, int max_blocks_per_seq, int num_blocks, int dtype, int num_seqs,
                                   int nthreads) {
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0) return ORACLE_EARG;
    if (head_dim <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || num_seqs < 0) return ORACLE_EARG;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return ORACLE_EARG;
    if (num_seqs == 0) return ORACLE_OK;
    if (nthreads < 1) nthreads = 1;
    long units = (long)num_seqs * num_kv_heads;
    if (nthreads > units) nthreads = (int)units;
    prefill_job_t *jobs = (prefill_job_t *)calloc((size_t)nthreads, sizeof(prefill_job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return ORACLE_ENOMEM;
    }
    int status = ORACLE_OK, started = 0;
    for (int t = 0; t < nthreads; ++t) {
        prefill_job_t *j = &jobs[t];
        j->out = out;
        j->q = q;
        j->k_cache = k_cache;
        j->v_cache = v_cache;
        j->block_tables = block_tables;
        j->context_lens = context_lens;
        j->query_start = query_start;
        j->scale = scale;
        j->num_kv_heads = num_kv_heads;
        j->num_q_heads = num_q_heads;
        j->head_dim = head_dim;
        j->max_blocks_per_seq = max_blocks_per_seq;
        j->num_blocks = num_blocks;
        j->dtype = dtype;
        j->num_seqs = num_seqs;
        j->nthreads = nthreads;
        j->thread_index = t;
        if (pthread_create(&tid[t], NULL, prefill_worker, j) != 0) break;
        ++started;
    }
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    if (started < nthreads) status = ORACLE_ENOMEM;
    for (int t = 0; t < started; ++t)
        if (jobs[t].status != ORACLE_OK) status = jobs[t].status;
    free(jobs);
    free(tid);
    return status;
}
