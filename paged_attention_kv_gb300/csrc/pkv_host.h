// Host-side helpers shared by the C-ABI translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

#include "pagedkv.h"

#define PKV_API __attribute__((visibility("default")))

namespace pkv {

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Validates a cache descriptor. Attention supports head sizes 64 and 128;
// the KV write any multiple of 8 (16-byte rows).
inline int check_cache_desc(const pkv_cache_desc &d, bool attention) {
    if (d.block_size != PKV_BLOCK_SIZE) return PKV_E_BLOCK_SIZE;
    if (d.num_blocks <= 0 || d.num_kv_heads <= 0 || d.head_size <= 0) return PKV_E_DIMS;
    if (attention) {
        if (d.head_size != 64 && d.head_size != 128) return PKV_E_HEAD_SIZE;
    } else if (d.head_size % 8 != 0) {
        return PKV_E_HEAD_SIZE;
    }
    if (d.num_blocks > INT32_MAX / PKV_BLOCK_SIZE) return PKV_E_DIMS;
    if (d.num_kv_heads > 4096 || d.head_size > 4096) return PKV_E_DIMS;
    return PKV_OK;
}

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel on the stream is still running; it calls pdl_wait()
// before touching global memory, so it still sees all of that kernel's
// writes, and it cannot complete before its predecessor has.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pkv
