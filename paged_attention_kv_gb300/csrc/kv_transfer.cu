// Block-granular KV transfer between the paged pool and a contiguous staging
// buffer, the device side of disaggregated prefill/decode ("Inside vLLM",
// page 1, "Disaggregated P/D": the prefill instance uploads the KV it
// computed; before decoding, the connector's start_load_kv loads it and
// injects it into paged memory; the transfer can also run per layer, page 2
// note on the same section). In the pool layout [NB][2][Hkv][16][D] one
// block of one layer is one contiguous run of 2 * 16 * Hkv * D * 2 bytes, so
// both directions are streams of 16-byte vector copies.
#include <cuda_runtime.h>

#include <cstdint>

#include "pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

// dst[i] = src[i] over `num_ids` blocks of `vecs` uint4 each; the pool side
// of block i is block_ids[i]. gather: pool -> staging; scatter: staging ->
// pool. An id outside [0, num_blocks) is skipped and flagged.
template <bool kGather>
__global__ void __launch_bounds__(256) block_copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                          const int32_t *__restrict__ block_ids, int num_ids,
                                                          long long vecs, int num_blocks, int32_t *status) {
    // A CTA copies whole blocks (each one contiguous run of vecs 16-byte
    // chunks), every thread with four loads in flight before its stores.
    pdl_launch_dependents();
    pdl_wait();
    constexpr int kUnroll = 4;
    for (int i = blockIdx.x; i < num_ids; i += gridDim.x) {
        const int32_t b = __ldg(block_ids + i);
        if (b < 0 || b >= num_blocks) {
            if (threadIdx.x == 0) raise_status(status, PKV_DEV_BAD_BLOCK);
            continue;
        }
        const uint4 *s = src + (kGather ? (long long)b : (long long)i) * vecs;
        uint4 *d = dst + (kGather ? (long long)i : (long long)b) * vecs;
        for (long long base = threadIdx.x; base < vecs; base += (long long)blockDim.x * kUnroll) {
            uint4 val[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const long long v = base + (long long)u * blockDim.x;
                if (v < vecs) val[u] = __ldcs(s + v);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const long long v = base + (long long)u * blockDim.x;
                if (v < vecs) d[v] = val[u];
            }
        }
    }
}

template <bool kGather>
int block_copy(const void *src, void *dst, const int32_t *block_ids, int32_t num_ids, const pkv_cache_desc *desc,
               int32_t *status, void *stream) {
    if (!desc) return PKV_E_NULL;
    const int rc = check_cache_desc(*desc, /*attention=*/false);
    if (rc) return rc;
    if (num_ids < 0) return PKV_E_DIMS;
    if (num_ids == 0) return PKV_OK;
    if (!src || !dst || !block_ids) return PKV_E_NULL;
    if (!aligned(src, 16) || !aligned(dst, 16) || !aligned(block_ids, 4) || !aligned(status, 4)) return PKV_E_ALIGN;
    const long long vecs = 2LL * PKV_BLOCK_SIZE * desc->num_kv_heads * desc->head_size * 2 / 16;
    const int grid = num_ids < (1 << 20) ? num_ids : (1 << 20);  // a CTA per block
    const cudaError_t err = launch_pdl(block_copy_kernel<kGather>, dim3(grid), dim3(256), 0,
                                       static_cast<cudaStream_t>(stream), static_cast<const uint4 *>(src),
                                       static_cast<uint4 *>(dst), block_ids, (int)num_ids, vecs,
                                       (int)desc->num_blocks, status);
    return err == cudaSuccess ? PKV_OK : PKV_E_CUDA;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" PKV_API int paged_kv_gather_blocks(const void *kv_cache, const pkv_cache_desc *desc, const int32_t *block_ids,
                                              int32_t num_ids, void *staging, int32_t *status, void *stream) {
    return block_copy<true>(kv_cache, staging, block_ids, num_ids, desc, status, stream);
}

extern "C" PKV_API int paged_kv_scatter_blocks(const void *staging, const int32_t *block_ids, int32_t num_ids,
                                               void *kv_cache, const pkv_cache_desc *desc, int32_t *status,
                                               void *stream) {
    return block_copy<false>(staging, kv_cache, block_ids, num_ids, desc, status, stream);
}
