// Host-side helpers shared by the C-ABI translation units.
#pragma once

#include <cstddef>
#include <cstdint>

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

}  // namespace pkv
