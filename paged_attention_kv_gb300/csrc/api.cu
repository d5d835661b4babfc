// Entry points of the C ABI outside the attention path: pool sizing,
// status read-back, status strings, and the bounded-wait self-test.
#include <cuda_runtime.h>

#include <cstdint>

#include "pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

using namespace pkv;

namespace {

// One thread waits on an mbarrier that nothing arrives on, with the same
// bounded wait every pipeline stage uses, so the give-up path (status bit,
// abort flag, kernel returns) runs without a stuck pipeline.
__global__ void selftest_wait_kernel(int32_t *status, unsigned long long timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    mbar_init(&bar, 1);
    mbar_fence_init();
    volatile int *abort = &abort_flag;
    if (mbar_wait(&bar, 0, status, abort, timeout_ns)) raise_status(status, PKV_DEV_OVERFLOW);  // cannot complete
    mbar_arrive(&bar);  // complete the phase before the CTA exits
}

}  // namespace

extern "C" PKV_API int pkv_selftest_bounded_wait(int32_t *status, uint32_t timeout_us, void *stream) {
    if (!status) return PKV_E_NULL;
    if (!aligned(status, 4)) return PKV_E_ALIGN;
    if (timeout_us == 0 || timeout_us > 1000000) return PKV_E_DIMS;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, 1000ull * timeout_us);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_E_CUDA;
}

// Page 2 ("LLM Engine 构造函数", KV-cache-manager note) gives the bytes of one
// block of one layer as 2 * block_size * num_kv_heads * head_size *
// dtype_num_bytes; the pool is num_blocks of those.
extern "C" PKV_API int pkv_kv_cache_bytes(const pkv_cache_desc *desc, size_t *bytes) {
    if (!desc || !bytes) return PKV_E_NULL;
    const int rc = check_cache_desc(*desc, /*attention=*/false);
    if (rc) return rc;
    *bytes = (size_t)desc->num_blocks * 2 * desc->block_size * desc->num_kv_heads * desc->head_size * 2;
    return PKV_OK;
}

extern "C" PKV_API int pkv_read_status(const int32_t *status, void *stream, int32_t *host_status) {
    if (!status || !host_status) return PKV_E_NULL;
    if (!aligned(status, 4)) return PKV_E_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, status, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess) return PKV_E_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return PKV_E_CUDA;
    *host_status = v;
    return v == 0 ? PKV_OK : PKV_E_DEVICE;
}

extern "C" PKV_API const char *pkv_status_string(int code) {
    switch (code) {
        case PKV_OK: return "ok";
        case PKV_E_NULL: return "a required pointer is NULL";
        case PKV_E_DIMS: return "a size or count is out of range";
        case PKV_E_GQA: return "num_q_heads is not a positive multiple of num_kv_heads";
        case PKV_E_BLOCK_SIZE: return "block_size must be 16";
        case PKV_E_HEAD_SIZE: return "unsupported head_size";
        case PKV_E_WORKSPACE: return "workspace too small";
        case PKV_E_ALIGN: return "a pointer is misaligned";
        case PKV_E_CUDA: return "a CUDA call or kernel launch failed";
        case PKV_E_DEVICE: return "the device status word reports bad metadata";
        default: return "unknown status code";
    }
}
