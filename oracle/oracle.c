/*
 * fp64 CPU oracle for paged-KV attention.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library. The product path (the
 * CUDA library and its Python binding) never calls it and shares no code,
 * header, table or constant with it.
 *
 * What it computes, and where the pages say so ("Inside vLLM: Anatomy of a
 * High-Throughput LLM Inference System", page 1 unless noted):
 *
 *  - Block size in bytes (page 2, "LLM Engine 构造函数", the KV-cache-manager
 *    note): 2 (key and value) * block_size * num_kv_heads * head_size *
 *    dtype_num_bytes.
 *  - Blocks of 16 tokens handed to a request, ceil(new_tokens / 16) of them
 *    ("Scheduler", allocate_slots step 1), kept per request in an ordered list
 *    ("Scheduler", allocate_slots step 3) that the model runner uses to index
 *    the paged KV memory ("Run forward pass", steps 1-2, where slot_mapping
 *    is built).
 *  - The forward pass populates the KVs of the new tokens in the paged memory
 *    ("Prefix Caching", the populate-KV figure caption and text).
 *  - Attention over one flattened "super sequence": each sequence only
 *    attends to its own tokens under position indices and masks ("Run
 *    forward pass", step 3). Chunked prefill only changes how many new tokens
 *    a step carries; the indexing does the rest ("Chunked prefill").
 *
 * Readings where the pages are silent (their concrete example figure was
 * lost in extraction):
 *  - slot = block_table[r][pos / B] * B + pos % B, with pos the absolute
 *    position of the token in its request; a negative slot means "skip".
 *  - KV-cache layout [num_blocks][2][num_kv_heads][B][head_size]: one block
 *    is one contiguous unit of exactly the formula's byte count.
 *  - A request r with L = seq_lens[r] (this step's tokens included) and
 *    n = query_start_loc[r+1] - query_start_loc[r] new tokens: its query i
 *    sits at position p = L - n + i and sees keys 0..p (causal).
 *  - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *
 * Arithmetic: inputs are bf16 bit patterns, widened exactly to double; the
 * softmax is the two-pass max-subtracted form, summed in logical key order,
 * so the result does not depend on which physical blocks hold the keys.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_E_ARG (-1)
#define ORC_E_QSL (-2)
#define ORC_E_LEN (-3)
#define ORC_E_BLOCK (-4)
#define ORC_E_SLOT (-5)
#define ORC_E_MEM (-6)

static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Page 2, the block-size note: 2 * block_size * num_kv_heads * head_size *
 * dtype_num_bytes bytes per block per layer. */
int64_t orc_block_bytes(int block_size, int num_kv_heads, int head_size, int dtype_bytes) {
    return (int64_t)2 * block_size * num_kv_heads * head_size * dtype_bytes;
}

/* Number of blocks a request needs for `tokens` tokens ("Scheduler",
 * allocate_slots step 1: ceil(17/16) = 2). */
int64_t orc_blocks_needed(int64_t tokens, int block_size) {
    return (tokens + block_size - 1) / block_size;
}

/* Checks the ragged batch description shared by the functions below. */
static int check_batch(int num_reqs, const int32_t *seq_lens, const int32_t *qsl,
                       int num_tokens, int max_blocks_per_req, int block_size) {
    if (num_reqs < 0 || num_tokens < 0) return ORC_E_ARG;
    if (qsl[0] != 0 || qsl[num_reqs] != num_tokens) return ORC_E_QSL;
    for (int r = 0; r < num_reqs; ++r) {
        int n = qsl[r + 1] - qsl[r];
        if (n < 0) return ORC_E_QSL;
        if (n > seq_lens[r]) return ORC_E_LEN;
        if ((int64_t)seq_lens[r] > (int64_t)max_blocks_per_req * block_size) return ORC_E_LEN;
    }
    return ORC_OK;
}

/* slot_mapping for the new tokens of a flattened batch ("Run forward pass",
 * step 2), under the slot reading stated in the file header. */
int orc_slot_mapping(const int32_t *block_table, int num_reqs, int max_blocks_per_req,
                     const int32_t *seq_lens, const int32_t *qsl, int num_tokens,
                     int block_size, int num_blocks, int32_t *slot_mapping) {
    int rc = check_batch(num_reqs, seq_lens, qsl, num_tokens, max_blocks_per_req, block_size);
    if (rc) return rc;
    for (int r = 0; r < num_reqs; ++r) {
        int n = qsl[r + 1] - qsl[r];
        int L = seq_lens[r];
        for (int i = 0; i < n; ++i) {
            int pos = L - n + i;
            int32_t block = block_table[(int64_t)r * max_blocks_per_req + pos / block_size];
            if (block < 0 || block >= num_blocks) return ORC_E_BLOCK;
            slot_mapping[qsl[r] + i] = block * block_size + pos % block_size;
        }
    }
    return ORC_OK;
}

/* Byte offset, in bf16 elements, of row `offset` of (block, kv, head) in the
 * [num_blocks][2][num_kv_heads][B][head_size] layout. */
static int64_t cache_row(int64_t block, int kv, int head, int offset,
                         int num_kv_heads, int block_size, int head_size) {
    return (((block * 2 + kv) * num_kv_heads + head) * block_size + offset) * (int64_t)head_size;
}

/* Writes the new tokens' K and V into their slots ("Prefix Caching": the
 * forward pass populates the KVs in paged memory). k, v: [T][Hkv][D]. A
 * negative slot is skipped; every other cache element is left as it was. */
int orc_kv_write(const uint16_t *k, const uint16_t *v, const int32_t *slot_mapping,
                 int num_tokens, uint16_t *kv_cache, int num_blocks, int block_size,
                 int num_kv_heads, int head_size) {
    for (int t = 0; t < num_tokens; ++t) {
        int32_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if ((int64_t)slot >= (int64_t)num_blocks * block_size) return ORC_E_SLOT;
        int64_t block = slot / block_size;
        int offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const uint16_t *ks = k + ((int64_t)t * num_kv_heads + h) * head_size;
            const uint16_t *vs = v + ((int64_t)t * num_kv_heads + h) * head_size;
            uint16_t *kd = kv_cache + cache_row(block, 0, h, offset, num_kv_heads, block_size, head_size);
            uint16_t *vd = kv_cache + cache_row(block, 1, h, offset, num_kv_heads, block_size, head_size);
            for (int d = 0; d < head_size; ++d) {
                kd[d] = ks[d];
                vd[d] = vs[d];
            }
        }
    }
    return ORC_OK;
}

/* Block-granular KV transfer for disaggregated prefill/decode (page 1,
 * "Disaggregated P/D": the decode instance loads the KV the prefill instance
 * computed and injects it into paged memory). staging is [num_ids][block]
 * with block = 2 * B * Hkv * D elements, the whole unit of one physical
 * block; gather copies pool blocks out, scatter copies them in. An id
 * outside the pool is an error. */
int orc_kv_gather_blocks(const uint16_t *kv_cache, int num_blocks, int block_size, int num_kv_heads,
                         int head_size, const int32_t *block_ids, int num_ids, uint16_t *staging) {
    const int64_t per_block = (int64_t)2 * block_size * num_kv_heads * head_size;
    for (int i = 0; i < num_ids; ++i) {
        if (block_ids[i] < 0 || block_ids[i] >= num_blocks) return ORC_E_BLOCK;
        for (int kv = 0; kv < 2; ++kv)
            for (int h = 0; h < num_kv_heads; ++h)
                for (int row = 0; row < block_size; ++row) {
                    const uint16_t *src = kv_cache + cache_row(block_ids[i], kv, h, row, num_kv_heads, block_size, head_size);
                    uint16_t *dst = staging + (int64_t)i * per_block +
                                    (((int64_t)kv * num_kv_heads + h) * block_size + row) * head_size;
                    for (int d = 0; d < head_size; ++d) dst[d] = src[d];
                }
    }
    return ORC_OK;
}

int orc_kv_scatter_blocks(const uint16_t *staging, const int32_t *block_ids, int num_ids, uint16_t *kv_cache,
                          int num_blocks, int block_size, int num_kv_heads, int head_size) {
    const int64_t per_block = (int64_t)2 * block_size * num_kv_heads * head_size;
    for (int i = 0; i < num_ids; ++i) {
        if (block_ids[i] < 0 || block_ids[i] >= num_blocks) return ORC_E_BLOCK;
        for (int kv = 0; kv < 2; ++kv)
            for (int h = 0; h < num_kv_heads; ++h)
                for (int row = 0; row < block_size; ++row) {
                    uint16_t *dst = kv_cache + cache_row(block_ids[i], kv, h, row, num_kv_heads, block_size, head_size);
                    const uint16_t *src = staging + (int64_t)i * per_block +
                                          (((int64_t)kv * num_kv_heads + h) * block_size + row) * head_size;
                    for (int d = 0; d < head_size; ++d) dst[d] = src[d];
                }
    }
    return ORC_OK;
}

typedef struct {
    const uint16_t *q;
    const uint16_t *kv_cache;
    const int32_t *block_table;
    const int32_t *seq_lens;
    const int32_t *qsl;
    const int32_t *row_token;
    const int32_t *row_head;
    double *out;
    int num_reqs, max_blocks_per_req, num_q_heads, num_kv_heads, head_size, block_size;
    int64_t num_rows;
    double scale;
    int thread_index, num_threads, max_seq_len;
    int status;
} attn_job;

/* out[row] = sum_j softmax_j(scale * q . K[j]) V[j] over the visible keys of
 * the row's request (the file header gives the masking reading). */
static void *attention_worker(void *arg) {
    attn_job *job = (attn_job *)arg;
    const int D = job->head_size, B = job->block_size, Hkv = job->num_kv_heads;
    const int group = job->num_q_heads / Hkv;
    double *score = (double *)malloc(sizeof(double) * (size_t)(job->max_seq_len > 0 ? job->max_seq_len : 1));
    double *qrow = (double *)malloc(sizeof(double) * (size_t)D);
    if (!score || !qrow) {
        job->status = ORC_E_MEM;
        free(score);
        free(qrow);
        return NULL;
    }
    for (int64_t row = job->thread_index; row < job->num_rows; row += job->num_threads) {
        int t = job->row_token[row];
        int hq = job->row_head[row];
        /* The request that owns token t in the flattened batch. */
        int r = 0;
        while (r < job->num_reqs && !(job->qsl[r] <= t && t < job->qsl[r + 1])) ++r;
        if (r == job->num_reqs) { job->status = ORC_E_QSL; break; }
        int n = job->qsl[r + 1] - job->qsl[r];
        int L = job->seq_lens[r];
        int i = t - job->qsl[r];
        int p = L - n + i;              /* absolute position of this query */
        int hk = hq / group;            /* kv head shared by this query head */
        const int32_t *blocks = job->block_table + (int64_t)r * job->max_blocks_per_req;

        for (int d = 0; d < D; ++d)
            qrow[d] = bf16_bits_to_double(job->q[((int64_t)t * job->num_q_heads + hq) * D + d]);

        double m = -INFINITY;
        for (int j = 0; j <= p; ++j) {
            const uint16_t *krow = job->kv_cache + cache_row(blocks[j / B], 0, hk, j % B, Hkv, B, D);
            double s = 0.0;
            for (int d = 0; d < D; ++d) s += qrow[d] * bf16_bits_to_double(krow[d]);
            s *= job->scale;
            score[j] = s;
            if (s > m) m = s;
        }
        double z = 0.0;
        for (int j = 0; j <= p; ++j) {
            score[j] = exp(score[j] - m);
            z += score[j];
        }
        double *o = job->out + row * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int j = 0; j <= p; ++j) {
            const uint16_t *vrow = job->kv_cache + cache_row(blocks[j / B], 1, hk, j % B, Hkv, B, D);
            double w = score[j] / z;
            for (int d = 0; d < D; ++d) o[d] += w * bf16_bits_to_double(vrow[d]);
        }
    }
    free(score);
    free(qrow);
    return NULL;
}

/* Attention for a list of output rows (row_token[i], row_head[i]); out is
 * [num_rows][head_size] fp64. Work is split over `num_threads` POSIX
 * threads by row; each row is computed start to finish by one thread. */
int orc_paged_attention_rows(const uint16_t *q, int num_tokens, int num_q_heads,
                             const uint16_t *kv_cache, int num_blocks, int block_size,
                             int num_kv_heads, int head_size,
                             const int32_t *block_table, int num_reqs, int max_blocks_per_req,
                             const int32_t *seq_lens, const int32_t *qsl, double scale,
                             const int32_t *row_token, const int32_t *row_head, int64_t num_rows,
                             double *out, int num_threads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_size <= 0 || block_size <= 0)
        return ORC_E_ARG;
    int rc = check_batch(num_reqs, seq_lens, qsl, num_tokens, max_blocks_per_req, block_size);
    if (rc) return rc;
    int max_seq_len = 0;
    for (int r = 0; r < num_reqs; ++r) {
        if (seq_lens[r] > max_seq_len) max_seq_len = seq_lens[r];
        int nb = (int)orc_blocks_needed(seq_lens[r], block_size);
        for (int j = 0; j < nb; ++j) {
            int32_t b = block_table[(int64_t)r * max_blocks_per_req + j];
            if (b < 0 || b >= num_blocks) return ORC_E_BLOCK;
        }
    }
    for (int64_t i = 0; i < num_rows; ++i)
        if (row_token[i] < 0 || row_token[i] >= num_tokens || row_head[i] < 0 || row_head[i] >= num_q_heads)
            return ORC_E_ARG;
    if (num_threads < 1) num_threads = 1;
    attn_job *jobs = (attn_job *)calloc((size_t)num_threads, sizeof(attn_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)num_threads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return ORC_E_MEM; }
    for (int i = 0; i < num_threads; ++i) {
        attn_job *j = &jobs[i];
        j->q = q; j->kv_cache = kv_cache; j->block_table = block_table;
        j->seq_lens = seq_lens; j->qsl = qsl; j->row_token = row_token; j->row_head = row_head;
        j->out = out; j->num_reqs = num_reqs; j->max_blocks_per_req = max_blocks_per_req;
        j->num_q_heads = num_q_heads; j->num_kv_heads = num_kv_heads; j->head_size = head_size;
        j->block_size = block_size; j->num_rows = num_rows; j->scale = scale;
        j->thread_index = i; j->num_threads = num_threads; j->max_seq_len = max_seq_len;
        j->status = ORC_OK;
    }
    /* A job whose thread could not be created runs on this thread instead. */
    char *running = (char *)calloc((size_t)num_threads, 1);
    if (!running) { free(jobs); free(tids); return ORC_E_MEM; }
    for (int i = 1; i < num_threads; ++i)
        running[i] = pthread_create(&tids[i], NULL, attention_worker, &jobs[i]) == 0;
    attention_worker(&jobs[0]);
    for (int i = 1; i < num_threads; ++i) {
        if (running[i]) pthread_join(tids[i], NULL);
        else attention_worker(&jobs[i]);
    }
    free(running);
    rc = ORC_OK;
    for (int i = 0; i < num_threads; ++i)
        if (jobs[i].status != ORC_OK) rc = jobs[i].status;
    free(jobs);
    free(tids);
    return rc;
}
