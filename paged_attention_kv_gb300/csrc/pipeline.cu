// Host-buffer step pipeline: the engine loop's per-step transfer of the
// batch ("Inside vLLM", page 1, "Run forward pass": the step's tensors and
// attention metadata go to the device, the output comes back) overlapped
// across steps, in one C call per step. Step i uses slot i % depth:
//   h2d stream      [wait: slot's previous kernels]  copy host_in -> dev_in,
//                   record loaded
//   compute stream  [wait: loaded, slot's previous output copy]  slot
//                   mapping with the KV write (one launch), attention;
//                   record computed
//   d2h stream      [wait: computed]  copy out -> out_host, record returned
// All buffers belong to the caller; the pipeline owns its events only.
#include <cuda_runtime.h>

#include <cstdint>
#include <new>

#include "pagedkv.h"
#include "pkv_host.h"

struct pkv_pipeline {
    pkv_pipeline_desc d;
    cudaEvent_t loaded[PKV_PIPELINE_MAX_DEPTH], computed[PKV_PIPELINE_MAX_DEPTH], returned[PKV_PIPELINE_MAX_DEPTH];
    bool used[PKV_PIPELINE_MAX_DEPTH];
    long long step;
    size_t out_bytes;
};

namespace pkv {
namespace {

bool fits(size_t off, size_t bytes, size_t total) { return off % 16 == 0 && off <= total && bytes <= total - off; }

int check_pipeline_desc(const pkv_pipeline_desc &d, size_t *out_bytes) {
    if (d.depth < 1 || d.depth > PKV_PIPELINE_MAX_DEPTH) return PKV_E_DIMS;
    int rc = check_cache_desc(d.cache, /*attention=*/true);
    if (rc) return rc;
    if (d.num_tokens <= 0 || d.num_q_heads <= 0 || d.max_num_reqs <= 0 || d.max_blocks_per_req <= 0)
        return PKV_E_DIMS;
    if (d.num_q_heads % d.cache.num_kv_heads != 0) return PKV_E_GQA;
    for (int s = 0; s < d.depth; ++s)
        if (!d.host_in[s] || !d.dev_in[s] || !d.slot_mapping[s] || !d.out[s]) return PKV_E_NULL;
    if (!d.status || !d.workspace) return PKV_E_NULL;
    const size_t T = (size_t)d.num_tokens, Hq = (size_t)d.num_q_heads, Hkv = (size_t)d.cache.num_kv_heads;
    const size_t D = (size_t)d.cache.head_size, R = (size_t)d.max_num_reqs, M = (size_t)d.max_blocks_per_req;
    if (!fits(d.off_q, T * Hq * D * 2, d.in_bytes) || !fits(d.off_k, T * Hkv * D * 2, d.in_bytes) ||
        !fits(d.off_v, T * Hkv * D * 2, d.in_bytes) || !fits(d.off_block_table, R * M * 4, d.in_bytes) ||
        !fits(d.off_seq_lens, R * 4, d.in_bytes) || !fits(d.off_query_start_loc, (R + 1) * 4, d.in_bytes))
        return PKV_E_DIMS;
    *out_bytes = T * Hq * D * 2;
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" PKV_API int pkv_pipeline_create(const pkv_pipeline_desc *desc, pkv_pipeline **pipeline) {
    if (!desc || !pipeline) return PKV_E_NULL;
    *pipeline = nullptr;
    size_t out_bytes = 0;
    const int rc = pkv::check_pipeline_desc(*desc, &out_bytes);
    if (rc) return rc;
    pkv_pipeline *p = new (std::nothrow) pkv_pipeline();
    if (!p) return PKV_E_CUDA;
    p->d = *desc;
    p->out_bytes = out_bytes;
    p->step = 0;
    int made = 0;
    for (; made < desc->depth; ++made) {
        p->used[made] = false;
        if (cudaEventCreateWithFlags(&p->loaded[made], cudaEventDisableTiming) != cudaSuccess) break;
        if (cudaEventCreateWithFlags(&p->computed[made], cudaEventDisableTiming) != cudaSuccess) {
            cudaEventDestroy(p->loaded[made]);
            break;
        }
        if (cudaEventCreateWithFlags(&p->returned[made], cudaEventDisableTiming) != cudaSuccess) {
            cudaEventDestroy(p->loaded[made]);
            cudaEventDestroy(p->computed[made]);
            break;
        }
    }
    if (made < desc->depth) {
        for (int s = 0; s < made; ++s) {
            cudaEventDestroy(p->loaded[s]);
            cudaEventDestroy(p->computed[s]);
            cudaEventDestroy(p->returned[s]);
        }
        delete p;
        return PKV_E_CUDA;
    }
    *pipeline = p;
    return PKV_OK;
}

extern "C" PKV_API int pkv_pipeline_next(pkv_pipeline *p, int32_t *slot) {
    if (!p || !slot) return PKV_E_NULL;
    const int s = (int)(p->step % p->d.depth);
    if (p->used[s] && cudaEventSynchronize(p->loaded[s]) != cudaSuccess) return PKV_E_CUDA;
    *slot = s;
    return PKV_OK;
}

extern "C" PKV_API int pkv_pipeline_submit(pkv_pipeline *p, int32_t num_reqs, void *kv_cache, void *out_host,
                                           int32_t max_query_len) {
    if (!p || !kv_cache || !out_host) return PKV_E_NULL;
    const pkv_pipeline_desc &d = p->d;
    if (num_reqs < 1 || num_reqs > d.max_num_reqs) return PKV_E_DIMS;
    const int s = (int)(p->step % d.depth);
    cudaStream_t h2d = static_cast<cudaStream_t>(d.h2d_stream);
    cudaStream_t comp = static_cast<cudaStream_t>(d.compute_stream);
    cudaStream_t d2h = static_cast<cudaStream_t>(d.d2h_stream);
    const uint8_t *hin = static_cast<const uint8_t *>(d.host_in[s]);
    uint8_t *din = static_cast<uint8_t *>(d.dev_in[s]);

    // inputs: once the step that last used this slot has run its kernels
    if (p->used[s] && cudaStreamWaitEvent(h2d, p->computed[s], 0) != cudaSuccess) return PKV_E_CUDA;
    if (cudaMemcpyAsync(din, hin, d.in_bytes, cudaMemcpyHostToDevice, h2d) != cudaSuccess) return PKV_E_CUDA;
    if (cudaEventRecord(p->loaded[s], h2d) != cudaSuccess) return PKV_E_CUDA;
    // kernels: after the inputs landed and the slot's previous output left
    if (cudaStreamWaitEvent(comp, p->loaded[s], 0) != cudaSuccess) return PKV_E_CUDA;
    if (p->used[s] && cudaStreamWaitEvent(comp, p->returned[s], 0) != cudaSuccess) return PKV_E_CUDA;

    if (max_query_len < 0) {  // the longest request, from the host copy of query_start_loc
        const int32_t *qsl = reinterpret_cast<const int32_t *>(hin + d.off_query_start_loc);
        max_query_len = 0;
        for (int r = 0; r < num_reqs; ++r) {
            const int32_t n = qsl[r + 1] - qsl[r];
            if (n > max_query_len) max_query_len = n;
        }
    }
    const int32_t *bt = reinterpret_cast<const int32_t *>(din + d.off_block_table);
    const int32_t *sl = reinterpret_cast<const int32_t *>(din + d.off_seq_lens);
    const int32_t *qsl = reinterpret_cast<const int32_t *>(din + d.off_query_start_loc);
    int rc = paged_kv_write_slots(din + d.off_k, din + d.off_v, bt, num_reqs, d.max_blocks_per_req, sl, qsl,
                                  d.num_tokens, kv_cache, &d.cache, d.slot_mapping[s], d.status, comp);
    if (!rc)
        rc = paged_attention_bounded(din + d.off_q, d.num_tokens, d.num_q_heads, kv_cache, &d.cache, bt, num_reqs,
                                     d.max_blocks_per_req, sl, qsl, max_query_len, d.scale, d.out[s], d.workspace,
                                     d.workspace_bytes, comp, nullptr);
    if (rc) return rc;
    if (cudaEventRecord(p->computed[s], comp) != cudaSuccess) return PKV_E_CUDA;
    // output
    if (cudaStreamWaitEvent(d2h, p->computed[s], 0) != cudaSuccess) return PKV_E_CUDA;
    if (cudaMemcpyAsync(out_host, d.out[s], p->out_bytes, cudaMemcpyDeviceToHost, d2h) != cudaSuccess)
        return PKV_E_CUDA;
    if (cudaEventRecord(p->returned[s], d2h) != cudaSuccess) return PKV_E_CUDA;
    p->used[s] = true;
    ++p->step;
    return PKV_OK;
}

extern "C" PKV_API int pkv_pipeline_sync(pkv_pipeline *p) {
    if (!p) return PKV_E_NULL;
    const void *streams[3] = {p->d.h2d_stream, p->d.compute_stream, p->d.d2h_stream};
    for (const void *st : streams)
        if (cudaStreamSynchronize(static_cast<cudaStream_t>(const_cast<void *>(st))) != cudaSuccess) return PKV_E_CUDA;
    return PKV_OK;
}

extern "C" PKV_API int pkv_pipeline_destroy(pkv_pipeline *p) {
    if (!p) return PKV_OK;
    const int rc = pkv_pipeline_sync(p);
    for (int s = 0; s < p->d.depth; ++s) {
        cudaEventDestroy(p->loaded[s]);
        cudaEventDestroy(p->computed[s]);
        cudaEventDestroy(p->returned[s]);
    }
    delete p;
    return rc;
}
