// Slot mapping and KV write: the two bandwidth kernels in front of the
// attention call ("Inside vLLM", page 1: "Run forward pass" step 2 builds
// slot_mapping; the forward pass then populates the new tokens' KVs in paged
// memory, "Prefix Caching").
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

// Last r in [0, num_reqs) with qsl[r] <= t (qsl sorted ascending).
__device__ __forceinline__ int find_request(const int32_t *__restrict__ qsl, int num_reqs, int t) {
    int lo = 0, hi = num_reqs;  // answer in [lo, hi)
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (__ldg(qsl + mid) <= t) lo = mid; else hi = mid;
    }
    return lo;
}

// Slot of new token t (-1 when its metadata is bad, which is reported).
__device__ __forceinline__ int32_t token_slot(const int32_t *__restrict__ block_table, int num_reqs,
                                              int max_blocks_per_req, const int32_t *__restrict__ seq_lens,
                                              const int32_t *__restrict__ qsl, int num_blocks, int t,
                                              int32_t *status) {
    const int r = find_request(qsl, num_reqs, t);
    const int q0 = __ldg(qsl + r), q1 = __ldg(qsl + r + 1);
    int32_t slot = -1;
    if (!(q0 <= t && t < q1)) {
        raise_status(status, PKV_DEV_BAD_QSL);
    } else {
        const int n = q1 - q0;
        const int L = __ldg(seq_lens + r);
        const int pos = L - n + (t - q0);
        if (n > L || (long long)L > (long long)max_blocks_per_req * PKV_BLOCK_SIZE || pos < 0) {
            raise_status(status, PKV_DEV_BAD_LEN);
        } else {
            const int32_t blk = __ldg(block_table + (long long)r * max_blocks_per_req + pos / PKV_BLOCK_SIZE);
            if (blk < 0 || blk >= num_blocks) raise_status(status, PKV_DEV_BAD_BLOCK);
            else slot = blk * PKV_BLOCK_SIZE + pos % PKV_BLOCK_SIZE;
        }
    }
    return slot;
}

// One thread per new token.
__global__ void slot_mapping_kernel(const int32_t *__restrict__ block_table, int num_reqs, int max_blocks_per_req,
                                    const int32_t *__restrict__ seq_lens, const int32_t *__restrict__ qsl,
                                    int num_tokens, int num_blocks, int32_t *__restrict__ slot_mapping,
                                    int32_t *status) {
    pdl_launch_dependents();
    pdl_wait();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t == 0 && (__ldg(qsl) != 0 || __ldg(qsl + num_reqs) != num_tokens)) raise_status(status, PKV_DEV_BAD_QSL);
    if (t >= num_tokens) return;
    slot_mapping[t] = token_slot(block_table, num_reqs, max_blocks_per_req, seq_lens, qsl, num_blocks, t, status);
}

// Where the KV write takes its slots from: the slot mapping (plain), or the
// tables, resolving each token's slot on the way and storing it (fused).
struct SlotSource {
    const int32_t *block_table, *seq_lens, *qsl;
    int num_reqs, max_blocks_per_req, num_blocks;
    int32_t *slot_out;
};

// Each warp takes R adjacent (token, K or V) rows per pass: a row (the
// token's K or V for all kv heads) is contiguous in k / v, and each head's D
// columns go to one row of a 16-row block tile. Slots and destinations are
// worked out once per row; each lane then has R x (4 / R) = 4 16-byte loads
// in flight before its stores (R = 1 for rows of >= 128 chunks, 4 for rows
// of 32 or fewer).
template <int R, bool kFused>
__global__ void kv_write_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                const int32_t *__restrict__ slot_mapping, long long num_tokens,
                                uint4 *__restrict__ kv_cache, long long num_slots, int num_kv_heads,
                                int chunks_per_row, int32_t *status, const SlotSource src_tables) {
    pdl_launch_dependents();
    constexpr int C = 4 / R;  // chunks per lane per row and pass
    const int lane = threadIdx.x & 31;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const int per_kv = num_kv_heads * chunks_per_row;  // 16-byte chunks of one token's K (or V) row
    const long long tile = (long long)PKV_BLOCK_SIZE * chunks_per_row;  // chunks of one (block, K|V, head) tile
    const long long units = 2 * num_tokens;
    const long long g0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    // Fused: the tables hold this call's values when it is enqueued, so the
    // slots of the warp's first pass (every pass, for any grid this library
    // launches) are resolved before waiting on the previous kernel; that
    // kernel (in a step, the previous attention) then no longer waits on the
    // lookups. Nothing is written before the wait: bad metadata is reported
    // after it, by resolving the slot again with the status word.
    int32_t first_slot[R];
    bool qsl_bad = false;
    if (kFused) {
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const long long u = g0 * R + j;
            int32_t s0 = -1;
            if (u < units && lane == 0)
                s0 = token_slot(src_tables.block_table, src_tables.num_reqs, src_tables.max_blocks_per_req,
                                src_tables.seq_lens, src_tables.qsl, src_tables.num_blocks, (int)(u >> 1), nullptr);
            first_slot[j] = __shfl_sync(0xffffffffu, s0, 0);
        }
        qsl_bad = blockIdx.x == 0 && threadIdx.x == 0 &&
                  (__ldg(src_tables.qsl) != 0 || __ldg(src_tables.qsl + src_tables.num_reqs) != num_tokens);
    }
    pdl_wait();
    if (qsl_bad) raise_status(status, PKV_DEV_BAD_QSL);
    for (long long g = g0; g * R < units; g += nwarps) {
        const uint4 *src[R];
        uint4 *dst[R];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const long long u = g * R + j;
            src[j] = nullptr;
            dst[j] = nullptr;
            if (u >= units) continue;
            const long long t = u >> 1;
            const int kv = (int)(u & 1);
            int32_t slot;
            if (kFused) {
                // lane 0 resolves the slot (reporting bad metadata once, on the
                // token's K row) and stores it; the warp shares it. The first
                // pass has it already; a failed lookup is redone here to
                // report it.
                int32_t s0 = 0;
                const bool have = g == g0;
                if (lane == 0 && (!have || first_slot[j] < 0))
                    s0 = token_slot(src_tables.block_table, src_tables.num_reqs, src_tables.max_blocks_per_req,
                                    src_tables.seq_lens, src_tables.qsl, src_tables.num_blocks, (int)t,
                                    kv == 0 ? status : nullptr);
                slot = have && first_slot[j] >= 0 ? first_slot[j] : __shfl_sync(0xffffffffu, s0, 0);
                if (lane == 0 && kv == 0) src_tables.slot_out[t] = slot;
            } else {
                slot = __ldg(slot_mapping + t);
            }
            if (slot < 0) continue;
            if ((long long)slot >= num_slots) {
                if (lane == 0 && kv == 0) raise_status(status, PKV_DEV_BAD_SLOT);
                continue;
            }
            src[j] = (kv ? v : k) + t * per_kv;
            dst[j] = kv_cache + ((long long)slot / PKV_BLOCK_SIZE * 2 + kv) * num_kv_heads * tile +
                     (long long)(slot % PKV_BLOCK_SIZE) * chunks_per_row;
        }
        for (int base = 0; base < per_kv; base += 32 * C) {
            uint4 val[R][C];
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    const int hc = base + c * 32 + lane;
                    if (src[j] && hc < per_kv) val[j][c] = __ldg(src[j] + hc);
                }
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const int hc = base + c * 32 + lane;
                if (hc >= per_kv) continue;
                const int h = hc / chunks_per_row;
                const long long off = h * tile + (hc - h * chunks_per_row);
#pragma unroll
                for (int j = 0; j < R; ++j)
                    if (dst[j]) dst[j][off] = val[j][c];
            }
        }
    }
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" PKV_API int paged_slot_mapping(const int32_t *block_table, int32_t num_reqs, int32_t max_blocks_per_req,
                                          const int32_t *seq_lens, const int32_t *query_start_loc,
                                          int32_t num_tokens, int32_t num_blocks, int32_t *slot_mapping,
                                          int32_t *status, void *stream) {
    if (num_reqs < 0 || num_tokens < 0 || max_blocks_per_req < 0 || num_blocks <= 0) return PKV_E_DIMS;
    if (num_blocks > INT32_MAX / PKV_BLOCK_SIZE) return PKV_E_DIMS;
    if (num_tokens == 0) return PKV_OK;
    if (num_reqs == 0) return PKV_E_DIMS;
    if (!block_table || !seq_lens || !query_start_loc || !slot_mapping) return PKV_E_NULL;
    if (!aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(query_start_loc, 4) ||
        !aligned(slot_mapping, 4) || !aligned(status, 4))
        return PKV_E_ALIGN;
    const int threads = 256;
    const int blocks = (num_tokens + threads - 1) / threads;
    const cudaError_t err = launch_pdl(slot_mapping_kernel, dim3(blocks), dim3(threads), 0,
                                       static_cast<cudaStream_t>(stream), block_table, num_reqs, max_blocks_per_req,
                                       seq_lens, query_start_loc, num_tokens, num_blocks, slot_mapping, status);
    return err == cudaSuccess ? PKV_OK : PKV_E_CUDA;
}

namespace pkv {
namespace {

int kv_write_launch(const void *k, const void *v, const int32_t *slot_mapping, int32_t num_tokens, void *kv_cache,
                    const pkv_cache_desc &desc, int32_t *status, void *stream, const SlotSource *fused) {
    const int chunks_per_row = desc.head_size / 8;
    const int threads = 256;  // 8 warps
    const int per_kv = desc.num_kv_heads * chunks_per_row;
    const int rows = per_kv >= 128 ? 1 : per_kv >= 64 ? 2 : 4;  // rows per warp and pass
    const long long want = ((long long)num_tokens * 2 + 8 * rows - 1) / (8 * rows);
    const int blocks = (int)(want < (1 << 20) ? want : (1 << 20));
    const SlotSource none{};
    auto kernel = fused ? (rows == 1 ? kv_write_kernel<1, true> : rows == 2 ? kv_write_kernel<2, true>
                                                                            : kv_write_kernel<4, true>)
                        : (rows == 1 ? kv_write_kernel<1, false> : rows == 2 ? kv_write_kernel<2, false>
                                                                             : kv_write_kernel<4, false>);
    const cudaError_t err = launch_pdl(
        kernel, dim3(blocks), dim3(threads), 0, static_cast<cudaStream_t>(stream), static_cast<const uint4 *>(k),
        static_cast<const uint4 *>(v), slot_mapping, (long long)num_tokens, static_cast<uint4 *>(kv_cache),
        (long long)desc.num_blocks * PKV_BLOCK_SIZE, (int)desc.num_kv_heads, chunks_per_row, status,
        fused ? *fused : none);
    return err == cudaSuccess ? PKV_OK : PKV_E_CUDA;
}

int check_kv_write_args(const void *k, const void *v, void *kv_cache, const pkv_cache_desc *desc, int32_t num_tokens,
                        int32_t *status) {
    if (!desc) return PKV_E_NULL;
    int rc = check_cache_desc(*desc, /*attention=*/false);
    if (rc) return rc;
    if (num_tokens < 0) return PKV_E_DIMS;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !kv_cache) return PKV_E_NULL;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(kv_cache, 16) || !aligned(status, 4)) return PKV_E_ALIGN;
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" PKV_API int paged_kv_write(const void *k, const void *v, const int32_t *slot_mapping, int32_t num_tokens,
                                      void *kv_cache, const pkv_cache_desc *desc, int32_t *status, void *stream) {
    int rc = check_kv_write_args(k, v, kv_cache, desc, num_tokens, status);
    if (rc || num_tokens == 0) return rc;
    if (!slot_mapping) return PKV_E_NULL;
    if (!aligned(slot_mapping, 4)) return PKV_E_ALIGN;
    return kv_write_launch(k, v, slot_mapping, num_tokens, kv_cache, *desc, status, stream, nullptr);
}

extern "C" PKV_API int paged_kv_write_slots(const void *k, const void *v, const int32_t *block_table, int32_t num_reqs,
                                            int32_t max_blocks_per_req, const int32_t *seq_lens,
                                            const int32_t *query_start_loc, int32_t num_tokens, void *kv_cache,
                                            const pkv_cache_desc *desc, int32_t *slot_mapping, int32_t *status,
                                            void *stream) {
    int rc = check_kv_write_args(k, v, kv_cache, desc, num_tokens, status);
    if (rc || num_tokens == 0) return rc;
    if (num_reqs <= 0 || max_blocks_per_req < 0) return PKV_E_DIMS;
    if (!block_table || !seq_lens || !query_start_loc || !slot_mapping) return PKV_E_NULL;
    if (!aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(query_start_loc, 4) ||
        !aligned(slot_mapping, 4))
        return PKV_E_ALIGN;
    SlotSource src{block_table, seq_lens, query_start_loc, num_reqs, max_blocks_per_req, desc->num_blocks,
                   slot_mapping};
    return kv_write_launch(k, v, nullptr, num_tokens, kv_cache, *desc, status, stream, &src);
}
