/*
 * pagedkv.h - C ABI of the GB300 (sm_103a) paged-KV attention library.
 *
 * The library implements the attention layer's hot path of a vLLM-style
 * engine as described in "Inside vLLM: Anatomy of a High-Throughput LLM
 * Inference System" (page 1 unless noted):
 *
 *   paged_slot_mapping  - the slot_mapping built in "prepare inputs"
 *                         ("Run forward pass", step 2);
 *   paged_kv_write      - the forward pass populating the new tokens' KVs in
 *                         paged KV memory ("Prefix Caching", populate-KV
 *                         figure text);
 *   paged_attention     - attention of every sequence over only its own
 *                         tokens in one flattened "super sequence", reading
 *                         K/V through per-request block tables ("Run forward
 *                         pass", step 3), for decode tokens and chunked-
 *                         prefill chunks in the same batch ("Scheduler": V1
 *                         mixes prefill and decode in one step; "Chunked
 *                         prefill"), with prefix-cached requests sharing
 *                         physical blocks ("Prefix Caching").
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All array arguments are DEVICE pointers owned by the caller. The
 *    library allocates no device memory and keeps no per-call state; the
 *    caller provides the attention workspace.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Every call only enqueues work on that stream and returns; the
 *    outputs are ready when the stream reaches that point.
 *  - bf16 tensors are row-major with the innermost dimension contiguous and
 *    must start on a 16-byte boundary. int32 arrays need 4-byte alignment.
 *  - The return value is PKV_OK or a negative PKV_E_* code. Argument errors
 *    are detected on the host before anything is enqueued. Bad METADATA
 *    (values inside device arrays, which the host never reads) is detected
 *    by the kernels: they skip the offending entry, never access memory out
 *    of bounds, and OR a PKV_DEV_* bit into a device status word that
 *    pkv_read_status() fetches.
 *  - Block size is fixed at 16 tokens ("Scheduler", allocate_slots: each
 *    block stores 16 tokens by default).
 *
 * KV-cache layout
 * ---------------
 *  One bf16 tensor per layer, [num_blocks][2][num_kv_heads][16][head_size]:
 *  index 0 of the second dimension holds K, index 1 holds V. One block is
 *  one contiguous run of 2 * 16 * num_kv_heads * head_size * 2 bytes, the
 *  per-block size the pages give (page 2, "LLM Engine 构造函数", KV-cache
 *  manager note). Token slot s lives in block s / 16, row s % 16.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_BLOCK_SIZE 16

/* Return codes. */
#define PKV_OK 0
#define PKV_E_NULL (-1)        /* a required pointer is NULL */
#define PKV_E_DIMS (-2)        /* a size or count is out of range */
#define PKV_E_GQA (-3)         /* num_q_heads is not a positive multiple of num_kv_heads */
#define PKV_E_BLOCK_SIZE (-4)  /* block_size != 16 */
#define PKV_E_HEAD_SIZE (-5)   /* head_size unsupported (attention: 64 or 128; KV write: multiple of 8) */
#define PKV_E_WORKSPACE (-6)   /* workspace smaller than paged_attention_workspace_bytes() requires */
#define PKV_E_ALIGN (-7)       /* a pointer is not aligned as required */
#define PKV_E_CUDA (-8)        /* a CUDA runtime call or kernel launch failed */
#define PKV_E_DEVICE (-9)      /* the device status word holds PKV_DEV_* bits */

/* Bits of the device status word (OR-ed in by the kernels). */
#define PKV_DEV_BAD_QSL 0x1      /* query_start_loc not ragged offsets 0 = qsl[0] <= ... <= qsl[R] = T */
#define PKV_DEV_BAD_LEN 0x2      /* a request has new tokens > seq_len, or seq_len > 16 * max_blocks_per_req */
#define PKV_DEV_BAD_BLOCK 0x4    /* a block_table entry that is read lies outside [0, num_blocks) */
#define PKV_DEV_BAD_SLOT 0x8     /* a slot_mapping entry lies at or beyond 16 * num_blocks */
#define PKV_DEV_TIMEOUT 0x10     /* an internal pipeline wait gave up (never expected) */
#define PKV_DEV_OVERFLOW 0x20    /* internal work list overflow (never expected) */

typedef struct {
    int32_t num_blocks;    /* blocks in the pool */
    int32_t block_size;    /* must be 16 */
    int32_t num_kv_heads;
    int32_t head_size;
} pkv_cache_desc;

/*
 * Bytes of the whole KV pool of one layer: num_blocks * 2 * 16 *
 * num_kv_heads * head_size * 2 (page 2 block-size note, bf16). Host only.
 */
int pkv_kv_cache_bytes(const pkv_cache_desc *desc, size_t *bytes);

/*
 * slot_mapping[t] for every new token t of a flattened batch ("Run forward
 * pass", step 2). Request r owns tokens query_start_loc[r] ..
 * query_start_loc[r+1]-1; with L = seq_lens[r] (context length including
 * this step's tokens) and n its new-token count, token i of the request sits
 * at position p = L - n + i and goes to slot
 *     block_table[r][p / 16] * 16 + p % 16.
 *
 *  block_table      int32 [num_reqs][max_blocks_per_req]
 *  seq_lens         int32 [num_reqs]
 *  query_start_loc  int32 [num_reqs + 1]
 *  slot_mapping     int32 [num_tokens] (output). A token whose request has
 *                   bad metadata, or whose block id is outside the pool,
 *                   gets -1 (which paged_kv_write skips) and raises a
 *                   status bit.
 *  status           optional device int32 (may be NULL); PKV_DEV_* bits are
 *                   OR-ed in, never cleared.
 */
int paged_slot_mapping(const int32_t *block_table, int32_t num_reqs, int32_t max_blocks_per_req,
                       const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_tokens,
                       int32_t num_blocks, int32_t *slot_mapping, int32_t *status, void *stream);

/*
 * Scatters this step's K and V into the pool ("Prefix Caching": the forward
 * pass populates the KVs in paged memory). For token t with slot s >= 0 and
 * every kv head h:
 *     kv_cache[s/16][0][h][s%16][:] = k[t][h][:]
 *     kv_cache[s/16][1][h][s%16][:] = v[t][h][:]
 * A negative slot is skipped (padding). A slot >= 16 * num_blocks is skipped
 * and raises PKV_DEV_BAD_SLOT. Slots must be distinct within one call, and
 * no block shared by several requests (a prefix-cache hit) may be a target.
 *
 *  k, v       bf16 [num_tokens][num_kv_heads][head_size]
 *  kv_cache   bf16 pool, layout above; head_size a multiple of 8
 */
int paged_kv_write(const void *k, const void *v, const int32_t *slot_mapping, int32_t num_tokens,
                   void *kv_cache, const pkv_cache_desc *desc, int32_t *status, void *stream);

/*
 * paged_slot_mapping and paged_kv_write in one launch: each new token's slot
 * is resolved from the tables (same rule, same status bits), stored in
 * slot_mapping (device int32 [num_tokens], written) and used for that
 * token's K/V at once. Same results as the two calls in sequence; one kernel
 * launch fewer per step. Arguments as for those two calls.
 *
 * Ordering: block_table, seq_lens and query_start_loc must hold this call's
 * values when the call is enqueued (written by host copies, or by kernels
 * that complete before their dependents launch): the slots are looked up
 * while the stream's previous kernel may still be running. k, v and the
 * pool are read, and slot_mapping, status and the pool written, only after
 * every earlier kernel on the stream has completed.
 */
int paged_kv_write_slots(const void *k, const void *v, const int32_t *block_table, int32_t num_reqs,
                         int32_t max_blocks_per_req, const int32_t *seq_lens, const int32_t *query_start_loc,
                         int32_t num_tokens, void *kv_cache, const pkv_cache_desc *desc, int32_t *slot_mapping,
                         int32_t *status, void *stream);

/*
 * Block-granular KV transfer for disaggregated prefill/decode (page 1,
 * "Disaggregated P/D": the prefill instance uploads the KV it computed, and
 * before decoding, start_load_kv loads it and injects it into paged memory;
 * the transfer may run per layer). One block of one layer is one
 * contiguous run of block_bytes = 2 * 16 * num_kv_heads * head_size * 2
 * bytes in the pool layout.
 *
 * paged_kv_gather_blocks:  staging[i] = pool block block_ids[i]
 * paged_kv_scatter_blocks: pool block block_ids[i] = staging[i]
 *
 *  staging    bytes [num_ids][block_bytes], device, 16-byte aligned
 *  block_ids  int32 [num_ids], device. An id outside [0, num_blocks) is
 *             skipped (its staging slot, or nothing, is left as it was) and
 *             raises PKV_DEV_BAD_BLOCK. Scatter ids must be distinct.
 *  status     optional device int32, PKV_DEV_* bits OR-ed in.
 */
int paged_kv_gather_blocks(const void *kv_cache, const pkv_cache_desc *desc, const int32_t *block_ids,
                           int32_t num_ids, void *staging, int32_t *status, void *stream);
int paged_kv_scatter_blocks(const void *staging, const int32_t *block_ids, int32_t num_ids, void *kv_cache,
                            const pkv_cache_desc *desc, int32_t *status, void *stream);

/*
 * Workspace bytes paged_attention needs for batches of at most
 * max_num_reqs requests and max_num_tokens new tokens on the current
 * device. It includes split-KV partial rows for the persistent grid and,
 * up to 2^20 rows, two per query row (room for the shared-prefix pass). A
 * smaller workspace (down to the size for max_num_reqs and max_num_tokens
 * with no room for split-KV partials) still works: the library then splits
 * long contexts less, or not at all, and skips the shared-prefix pass when
 * its partial rows do not fit.
 */
int paged_attention_workspace_bytes(int32_t max_num_reqs, int32_t max_num_tokens, int32_t num_q_heads,
                                    const pkv_cache_desc *desc, size_t *bytes);

/*
 * The smallest workspace paged_attention accepts for those bounds: room for
 * the work list but none for split-KV partials, so every (request, kv head,
 * 16-row tile) is processed by one CTA over its whole context. Host only.
 */
int paged_attention_min_workspace_bytes(int32_t max_num_reqs, int32_t max_num_tokens, int32_t num_q_heads,
                                        const pkv_cache_desc *desc, size_t *bytes);

/*
 * Causal GQA attention of a flattened ragged batch over the paged pool
 * ("Run forward pass", step 3). For new token t of request r (token i of
 * the request, position p = L - n + i) and query head hq:
 *
 *   out[t][hq][:] = sum_{j=0..p} softmax_j(scale * q[t][hq] . K_r[j]) V_r[j]
 *
 * where K_r[j] / V_r[j] are row j % 16 of kv head hq / (num_q_heads /
 * num_kv_heads) in block block_table[r][j / 16]. Decode tokens (n = 1),
 * speculative/multi-token queries and chunked-prefill chunks (any n <= L)
 * mix freely in one call. Call it after paged_kv_write of the same step, on
 * the same stream. Long contexts are split across CTAs (split-KV) and
 * merged with a log-sum-exp weighted reduction.
 *
 * Ordering: block_table, seq_lens and query_start_loc must hold this call's
 * values when the call is enqueued (written by host copies, or by kernels
 * that complete before their dependents launch): the work-list kernel may
 * start reading them while the stream's previous kernel is still running.
 * q and kv_cache are read only after every earlier kernel on the stream
 * has completed. The workspace is written only after that point too.
 *
 *  q          bf16 [num_tokens][num_q_heads][head_size], head_size 64 or 128
 *  kv_cache   bf16 pool (read only)
 *  out        bf16 [num_tokens][num_q_heads][head_size]; rows of requests
 *             with bad metadata are left unwritten
 *  workspace  device scratch of workspace_bytes bytes, 256-byte aligned;
 *             its first 4 bytes are this call's device status word (cleared
 *             at the start of the call). Calls that run concurrently need
 *             separate workspaces.
 */
int paged_attention(const void *q, int32_t num_tokens, int32_t num_q_heads,
                    const void *kv_cache, const pkv_cache_desc *desc,
                    const int32_t *block_table, int32_t num_reqs, int32_t max_blocks_per_req,
                    const int32_t *seq_lens, const int32_t *query_start_loc,
                    float scale, void *out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * paged_attention, plus CUDA events recorded on `stream` between its
 * launches, for measuring each kernel on the stream it runs on: events[0]
 * before the work-list kernel, events[1] after it, events[2] after the
 * chunk-tile kernel (requests with >= 128 query rows; equal to events[1]
 * when it is not launched), events[3] after the split-KV kernel (all other
 * rows; it also merges split partials).
 * `events` holds four cudaEvent_t handles created by the caller (a NULL
 * entry is skipped). Same arguments, results and errors as paged_attention.
 */
int paged_attention_timed(const void *q, int32_t num_tokens, int32_t num_q_heads,
                          const void *kv_cache, const pkv_cache_desc *desc,
                          const int32_t *block_table, int32_t num_reqs, int32_t max_blocks_per_req,
                          const int32_t *seq_lens, const int32_t *query_start_loc,
                          float scale, void *out, void *workspace, size_t workspace_bytes, void *stream,
                          void *const *events);

/*
 * paged_attention with a caller bound on new tokens per request, as an
 * engine's scheduler knows it for each step (the pages' attention metadata
 * carries the longest query of the batch): max_query_len >= every request's
 * query_start_loc[r + 1] - query_start_loc[r], or 0 for no bound. When
 * max_query_len x (num_q_heads / num_kv_heads) < 128 no request can fill a
 * 128-row chunk tile, and the chunk-tile kernel is not launched at all (a
 * decode-only step saves that launch). A bound that is too small is not
 * detected and stays correct: every row then takes the split-KV path.
 * events: NULL, or four cudaEvent_t handles as for paged_attention_timed.
 * Other arguments, results and errors as paged_attention.
 */
int paged_attention_bounded(const void *q, int32_t num_tokens, int32_t num_q_heads,
                            const void *kv_cache, const pkv_cache_desc *desc,
                            const int32_t *block_table, int32_t num_reqs, int32_t max_blocks_per_req,
                            const int32_t *seq_lens, const int32_t *query_start_loc, int32_t max_query_len,
                            float scale, void *out, void *workspace, size_t workspace_bytes, void *stream,
                            void *const *events);

/*
 * paged_attention without a workspace argument, for callers that cannot
 * allocate device memory at the point where they run attention: an engine
 * that has already given nearly all free device memory to its KV pool (the
 * pages size the pool to fill what a profiling pass leaves), a plugin whose
 * host framework owns all device memory, or a latency-critical loop that
 * cannot take cudaMalloc's implicit synchronisation. The paper has no
 * counterpart to this entry point; it exists for those callers.
 *
 * The work list and split-KV partials live in one fixed 16 MiB device
 * array inside this library, which every GPU that loads the library keeps
 * until the process exits; the call allocates nothing. A batch whose work
 * list does not fit in 16 MiB (about 150k new tokens at 32 query heads) is
 * rejected with PKV_E_WORKSPACE; a large batch that fits gets fewer
 * split-KV partitions than paged_attention would give it.
 *
 * The first call on each device looks up the array's device address and
 * sets up the kernels (with that device current); make that first call
 * before any stream capture. All calls on a device share the one array and
 * it keeps the previous call's contents (each call rebuilds what it reads),
 * so calls whose work overlaps on the GPU race with each other: issue them
 * on one stream, or order them. The device status word of this variant
 * stays inside the array and cannot be read back; bad metadata is still
 * skipped safely. Arguments, layouts and results are otherwise those of
 * paged_attention.
 *
 * Lifetime: the array's device address and the kernels' attributes are
 * looked up once per device and kept for the life of the process. The
 * library does not survive cudaDeviceReset (or any other teardown of a
 * device's primary context): after one, the cached address may name memory
 * of the old context, so no entry point of this library may be called again
 * in that process.
 */
int paged_attention_static(const void *q, int32_t num_tokens, int32_t num_q_heads,
                           const void *kv_cache, const pkv_cache_desc *desc,
                           const int32_t *block_table, int32_t num_reqs, int32_t max_blocks_per_req,
                           const int32_t *seq_lens, const int32_t *query_start_loc,
                           float scale, void *out, void *stream);

/*
 * Host-buffer step pipeline: steps whose inputs come from, and whose output
 * goes to, pinned host memory, with the copies overlapped across steps
 * (the engine loop's per-step transfer of the batch's tensors and metadata,
 * "Run forward pass"). The caller owns every buffer; the pipeline owns only
 * CUDA events. Each step:
 *   h2d stream:     one copy of slot s's packed inputs (host_in[s] ->
 *                   dev_in[s]), after the step that last used slot s has
 *                   finished its kernels;
 *   compute stream: paged_kv_write_slots and paged_attention_bounded on
 *                   slot s's device arrays,
 *                   after that copy and after slot s's previous output has
 *                   left the device;
 *   d2h stream:     one copy of slot s's output to the caller's host
 *                   buffer.
 * Slots are used in turn (step i uses slot i % depth). Packed inputs of a
 * slot: q [num_tokens][num_q_heads][head_size] bf16, k and v
 * [num_tokens][num_kv_heads][head_size] bf16, block_table
 * [max_num_reqs][max_blocks_per_req] int32, seq_lens [max_num_reqs] int32,
 * query_start_loc [max_num_reqs + 1] int32, at the given byte offsets.
 */
#define PKV_PIPELINE_MAX_DEPTH 4
typedef struct {
    int32_t depth;                     /* slots, 1 .. PKV_PIPELINE_MAX_DEPTH */
    void *host_in[PKV_PIPELINE_MAX_DEPTH];  /* pinned host packed inputs, in_bytes each */
    void *dev_in[PKV_PIPELINE_MAX_DEPTH];   /* device packed inputs, same layout */
    size_t in_bytes;
    size_t off_q, off_k, off_v, off_block_table, off_seq_lens, off_query_start_loc;  /* 16-byte aligned */
    int32_t num_tokens, num_q_heads, max_num_reqs, max_blocks_per_req;
    pkv_cache_desc cache;              /* every pool the steps use has this shape */
    int32_t *slot_mapping[PKV_PIPELINE_MAX_DEPTH];  /* device int32 [num_tokens] */
    void *out[PKV_PIPELINE_MAX_DEPTH];              /* device bf16 [num_tokens][num_q_heads][head_size] */
    int32_t *status;                   /* device status word of slot mapping and KV write */
    void *workspace;                   /* attention workspace, workspace_bytes */
    size_t workspace_bytes;
    float scale;
    void *h2d_stream, *compute_stream, *d2h_stream;  /* cudaStream_t (NULL: the legacy default stream);
                                                        distinct streams overlap the copies with the
                                                        neighbouring steps' kernels, equal ones serialise */
} pkv_pipeline_desc;
typedef struct pkv_pipeline pkv_pipeline;

/* Checks the description and creates the pipeline's events. The pointers
 * in `desc` must stay valid until pkv_pipeline_destroy. */
int pkv_pipeline_create(const pkv_pipeline_desc *desc, pkv_pipeline **pipeline);

/* The slot the next submit uses; waits (host) until that slot's previous
 * input copy has been read, so its host_in may be rewritten. */
int pkv_pipeline_next(pkv_pipeline *pipeline, int32_t *slot);

/* Enqueues the next step: num_reqs requests (1 .. max_num_reqs) of the
 * slot's inputs against kv_cache (a pool of desc.cache's shape), output to
 * out_host (pinned, num_tokens * num_q_heads * head_size bf16).
 * max_query_len as for paged_attention_bounded; a negative value takes it
 * from the slot's host query_start_loc. Does not wait. */
int pkv_pipeline_submit(pkv_pipeline *pipeline, int32_t num_reqs, void *kv_cache, void *out_host,
                        int32_t max_query_len);

/* Waits until every submitted step's output is in host memory. */
int pkv_pipeline_sync(pkv_pipeline *pipeline);

/* Waits for the submitted steps, then frees the pipeline's events. */
int pkv_pipeline_destroy(pkv_pipeline *pipeline);

/*
 * Failure-detection self-test: runs one thread that waits, with the bounded
 * wait every pipeline stage of the attention kernels uses, on an mbarrier
 * that nothing arrives on. After timeout_us (1 .. 1000000) the wait gives
 * up, PKV_DEV_TIMEOUT is ORed into *status (device, 4-byte aligned, not
 * cleared by the call) and the kernel returns; the CUDA context stays
 * usable. A stuck stage in a real launch is reported the same way, after
 * 2 s. Returns PKV_E_* for bad arguments or a launch error.
 */
int pkv_selftest_bounded_wait(int32_t *status, uint32_t timeout_us, void *stream);

/*
 * Copies a device status word to *host_status after the work queued on
 * `stream` so far has finished (synchronises the stream). Returns PKV_OK if
 * the word is 0, PKV_E_DEVICE if bits are set, PKV_E_CUDA on a CUDA error.
 * For paged_attention, pass the workspace pointer (its status word).
 */
int pkv_read_status(const int32_t *status, void *stream, int32_t *host_status);

/* A static English description of a return code. */
const char *pkv_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
