// Chunk-tile attention on tcgen05 tensor cores, for requests that bring many
// new tokens in one step (chunked prefill, "Inside vLLM", page 1, "Chunked
// prefill"; V1 mixes such chunks with decode tokens, "Scheduler").
//
// A work item is 128 query rows (tokens x the q heads of one GQA group,
// token-major) of one request and kv head, over all keys the rows may see.
// Per 128-key tile:
//   S = Q K^T   tcgen05.mma (M=128, N=128, K=16 steps), bf16 operands from
//               128B-swizzled shared memory, fp32 accumulator in TMEM
//               (two S buffers, so S of the next tile overlaps softmax);
//   softmax     one thread per row (its TMEM lane): causal mask, exp2 with
//               a running reference max that only moves (and rescales O)
//               when a row max grows by more than 2^8;
//   O += P V    tcgen05.mma (M=128, N=D), P from shared memory (K-major),
//               V MN-major straight from its TMA tile, O resident in TMEM.
// Warps: 0 TMA producer (Q tile; K and V tiles of 8 blocks, one box per 64
// columns of each block), 1 MMA issuer (one thread) and TMEM owner, 2-5
// softmax and output. Every wait is bounded; on a timeout the CTA raises
// PKV_DEV_TIMEOUT, stops, lets its in-flight copies and MMAs finish and
// frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attention_chunk.h"
#include "attention_plan.cuh"
#include "pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kChunkThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.f;  // log2 units: P stays <= 2^8

// mbarrier slots: the Q tile handoff, the K/V ring and S buffers (two each,
// by tile parity), P ready, PV done, and the final drain.
enum ChunkBar {
    kBarQFull = 0,
    kBarQEmpty,
    kBarQTaken,
    kBarKFull,                    // [2]
    kBarVFull = kBarKFull + 2,    // [2]
    kBarKvEmpty = kBarVFull + 2,  // [2]
    kBarSFull = kBarKvEmpty + 2,  // [2]
    kBarSFree = kBarSFull + 2,    // [2]
    kBarPFull = kBarSFree + 2,
    kBarODone,
    kBarDrain,
    kNumBars
};

struct ChunkDesc {
    int item, r, mt, h, kv_end, q0, n, L, nv, nt, pad[6];
};

template <int D>
struct ChunkSmem {
    static constexpr int kHalf = 16384;             // 128 rows x 128 B (64 bf16 columns)
    static constexpr int kTile = (D / 64) * kHalf;  // 128 rows x D bf16
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTile;     // 2 stages
    static constexpr int kOffV = kOffK + 2 * kTile; // 2 stages
    static constexpr int kOffP = kOffV + 2 * kTile; // 128 rows x 128 keys bf16, two 64-key halves
    static constexpr int kOffDesc = kOffP + 2 * kHalf;
    static constexpr int kOffBar = kOffDesc + (int)sizeof(ChunkDesc);
    static constexpr int kBars = kNumBars;
    static constexpr int kOffTmem = kOffBar + kBars * 8;
    static constexpr int kBytes = kOffTmem + 16;
    static constexpr int kAlloc = kBytes + 1024;
};

template <int D>
__global__ void __launch_bounds__(kChunkThreads, 1)
chunk_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
             const ChunkArgs a) {
    using S = ChunkSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_abort;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::kOffBar);
    uint64_t *q_full = bar + kBarQFull, *q_empty = bar + kBarQEmpty, *q_taken = bar + kBarQTaken;
    uint64_t *k_full = bar + kBarKFull, *v_full = bar + kBarVFull, *kv_empty = bar + kBarKvEmpty;
    uint64_t *s_full = bar + kBarSFull, *s_free = bar + kBarSFree, *p_full = bar + kBarPFull;
    uint64_t *o_done = bar + kBarODone, *drain = bar + kBarDrain;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::kOffTmem);
    ChunkDesc *desc = reinterpret_cast<ChunkDesc *>(smem + S::kOffDesc);
    volatile int *abort = &s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *status = &a.header->status;
    int32_t *diag = &a.header->diag;
    const int g = a.group;

    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(q_taken, 5);  // four softmax warps and the MMA thread
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&kv_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 4);
        }
        mbar_init(p_full, 4);
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tm = *tmem_slot;
    // The prologue above overlaps the previous kernel; the work list it
    // wrote is read only after this.
    pdl_wait();
    pdl_launch_dependents();
    const int n_items = a.header->n_chunk_items;

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            tma_prefetch_desc(&kv_map);
            tma_prefetch_desc(&q_map);
        }
        const int Hkv = a.num_kv_heads;
        uint32_t jt = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            int it = 0;
            if (lane == 0) it = atomicAdd(&a.header->next_chunk_item, 1);
            it = __shfl_sync(0xffffffffu, it, 0);
            if (!mbar_wait(q_taken, (k & 1) ^ 1, status, abort) || !mbar_wait(q_empty, (k & 1) ^ 1, status, abort)) {
                ok = false;
                break;
            }
            if (it >= n_items) {
                if (lane == 0) {
                    desc->item = -1;
                    mbar_arrive(q_full);
                }
                break;
            }
            const ChunkItem w = a.items[it];
            const int r = w.a.x, mt = w.a.y, h = w.a.z, kv_end = w.a.w;
            const int q0 = w.b.x, n = w.b.y, L = w.b.z, nv = w.b.w;
            const int nt = (kv_end + kChunkKeys - 1) / kChunkKeys;
            const int kvb = (kv_end + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE;
            if (lane == 0) {
                ChunkDesc d;
                d.item = it; d.r = r; d.mt = mt; d.h = h; d.kv_end = kv_end; d.q0 = q0; d.n = n; d.L = L;
                d.nv = nv; d.nt = nt;
                *desc = d;
                mbar_arrive_expect_tx(q_full, kChunkRows * D * 2);
#pragma unroll
                for (int bx = 0; bx < D / 64; ++bx)
                    tma_load_3d(smem + S::kOffQ + bx * S::kHalf, &q_map, bx * 64, h * g, q0 + mt * (kChunkRows / g),
                                q_full);
            }
            __syncwarp();
            const int32_t *bt = a.block_table + (long long)r * a.max_blocks_per_req;
            for (int j = 0; j < nt; ++j, ++jt) {
                const int st = jt & 1;
                if (!mbar_wait(&kv_empty[st], ((jt >> 1) & 1) ^ 1, status, abort)) { ok = false; break; }
                int blk = a.num_blocks;  // past the map: TMA fills zeros
                const int kb = j * (kChunkKeys / PKV_BLOCK_SIZE) + lane;
                if (lane < kChunkKeys / PKV_BLOCK_SIZE && kb < kvb) {
                    blk = __ldg(bt + kb);
                    if (blk < 0 || blk >= a.num_blocks) {
                        raise_status(status, PKV_DEV_BAD_BLOCK);
                        blk = a.num_blocks;
                    }
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&k_full[st], kChunkKeys * D * 2);
                    mbar_arrive_expect_tx(&v_full[st], kChunkKeys * D * 2);
                }
                __syncwarp();
                if (lane < kChunkKeys / PKV_BLOCK_SIZE) {
                    uint8_t *ks = smem + S::kOffK + st * S::kTile + lane * 2048;
                    uint8_t *vs = smem + S::kOffV + st * S::kTile + lane * 2048;
#pragma unroll
                    for (int bx = 0; bx < D / 64; ++bx) {
                        tma_load_3d(ks + bx * S::kHalf, &kv_map, bx * 64, h * PKV_BLOCK_SIZE, blk, &k_full[st]);
                        tma_load_3d(vs + bx * S::kHalf, &kv_map, bx * 64, (Hkv + h) * PKV_BLOCK_SIZE, blk, &v_full[st]);
                    }
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) {
            // let copies already issued land before the CTA can leave
            for (uint32_t x = jt > 2 ? jt - 2 : 0; x < jt; ++x) {
                mbar_drain(&k_full[x & 1], (x >> 1) & 1, status, diag, 0x2);
                mbar_drain(&v_full[x & 1], (x >> 1) & 1, status, diag, 0x2);
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer -----------------------------
        if (lane == 0) {
            constexpr uint32_t kIdS = umma_idesc_bf16(128, kChunkKeys, 0, 0);
            constexpr uint32_t kIdPV = umma_idesc_bf16(128, D, 0, 1);
            const uint32_t q_s = smem_u32(smem + S::kOffQ), p_s = smem_u32(smem + S::kOffP);
            const uint32_t k_s = smem_u32(smem + S::kOffK), v_s = smem_u32(smem + S::kOffV);
            uint32_t jt = 0;
            bool ok = true;
            auto pv = [&](uint32_t x, bool first) {
                const int st = x & 1;
                if (!mbar_wait(p_full, x & 1, status, abort) || !mbar_wait(&v_full[st], (x >> 1) & 1, status, abort))
                    return false;
                tmem_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kChunkKeys / 16; ++kk) {
                    const uint64_t ad = umma_desc_sw128(p_s + (kk / 4) * S::kHalf + (kk % 4) * 32, 16, 1024);
                    const uint64_t bd = umma_desc_sw128(v_s + st * S::kTile + kk * 2048, S::kHalf, 1024);
                    umma_bf16(tm + 256, ad, bd, kIdPV, (!first || kk > 0) ? 1u : 0u);
                }
                umma_commit(o_done);
                umma_commit(&kv_empty[st]);
                return true;
            };
            for (int k = 0; ok; ++k) {
                if (!mbar_wait(q_full, k & 1, status, abort)) { ok = false; break; }
                const ChunkDesc d = *desc;
                mbar_arrive(q_taken);
                if (d.item < 0) break;
                for (int j = 0; j < d.nt && ok; ++j) {
                    const uint32_t x = jt + j;
                    const int st = x & 1;
                    if (!mbar_wait(&k_full[st], (x >> 1) & 1, status, abort) ||
                        !mbar_wait(&s_free[st], ((x >> 1) & 1) ^ 1, status, abort)) {
                        ok = false;
                        break;
                    }
                    tmem_fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk / 4) * S::kHalf + (kk % 4) * 32;
                        umma_bf16(tm + st * kChunkKeys, umma_desc_sw128(q_s + off, 16, 1024),
                                  umma_desc_sw128(k_s + st * S::kTile + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&s_full[st]);
                    if (j == d.nt - 1) umma_commit(q_empty);
                    if (j > 0 && !pv(x - 1, j == 1)) { ok = false; break; }
                }
                if (ok && !pv(jt + d.nt - 1, d.nt == 1)) ok = false;
                jt += d.nt;
            }
            // make sure no MMA is still writing TMEM before it is freed
            umma_commit(drain);
            mbar_drain(drain, 0, status, diag, 0x4);
        }
        __syncwarp();
    } else {
        // --------------------------- softmax and output ---------------------------
        const int q4 = warp & 3;                 // TMEM lane quadrant this warp may access
        const int row = q4 * 32 + lane;          // query row of the tile = TMEM lane
        const uint32_t lane_base = tm + ((uint32_t)(q4 * 32) << 16);
        uint8_t *p_s = smem + S::kOffP;
        uint32_t jt = 0;
        for (int k = 0;; ++k) {
            if (!mbar_wait(q_full, k & 1, status, abort)) break;
            const ChunkDesc d = *desc;
            __syncwarp();
            if (lane == 0) mbar_arrive(q_taken);
            if (d.item < 0) break;
            const int rho = d.mt * kChunkRows + row;
            const bool valid = row < d.nv;
            const int i = valid ? rho / g : 0;
            const int limit = valid ? d.L - d.n + i : d.kv_end - 1;
            float m_run = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < d.nt; ++j) {
                const uint32_t x = jt + j;
                const int st = x & 1;
                if (!mbar_wait(&s_full[st], (x >> 1) & 1, status, abort)) { ok = false; break; }
                tmem_fence_after_sync();
                float s[kChunkKeys];
#pragma unroll
                for (int c = 0; c < kChunkKeys / 32; ++c)
                    tmem_ld32(lane_base + st * kChunkKeys + c * 32, *reinterpret_cast<float(*)[32]>(&s[c * 32]));
                tmem_wait_ld();
                tmem_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[st]);

                const int key0 = j * kChunkKeys;
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < kChunkKeys; ++c) {
                    s[c] = key0 + c <= limit ? s[c] * a.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, s[c]);
                }
                if (j > 0 && !mbar_wait(o_done, (x - 1) & 1, status, abort)) { ok = false; break; }
                if (j == 0) {
                    m_run = mx;  // key 0 is visible to every row, so this is finite
                } else {
                    const bool resc = mx > m_run + kRescaleThreshold;
                    if (__any_sync(0xffffffffu, resc)) {
                        const float alpha = resc ? fast_exp2(m_run - mx) : 1.f;
                        tmem_fence_after_sync();
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            float o[32];
                            tmem_ld32(lane_base + 256 + c * 32, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] *= alpha;
                            tmem_st32(lane_base + 256 + c * 32, o);
                        }
                        tmem_wait_st();
                        l *= alpha;
                        if (resc) m_run = mx;
                    }
                }
                // P = 2^(s - m_run) as bf16, row `row` of the K-major P tile.
#pragma unroll
                for (int c = 0; c < kChunkKeys / 8; ++c) {
                    float p[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        p[e] = fast_exp2(s[c * 8 + e] - m_run);
                        l += p[e];
                    }
                    uint4 pk;
                    pk.x = pack_bf16x2(p[0], p[1]);
                    pk.y = pack_bf16x2(p[2], p[3]);
                    pk.z = pack_bf16x2(p[4], p[5]);
                    pk.w = pack_bf16x2(p[6], p[7]);
                    *reinterpret_cast<uint4 *>(p_s + (c / 8) * S::kHalf + swz128(row, c % 8)) = pk;
                }
                // V rows past the last visible key hold other data (maybe
                // NaN); their P is 0 but 0 * NaN is not, so clear them.
                if (j == d.nt - 1) {
                    const int first = d.kv_end - key0;
                    const int stop = min(kChunkKeys, ((d.kv_end + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE) * PKV_BLOCK_SIZE - key0);
                    if (first < stop) {
                        if (!mbar_wait(&v_full[st], (x >> 1) & 1, status, abort)) { ok = false; break; }
                        uint8_t *vt = smem + S::kOffV + st * S::kTile;
                        const int per_row = (D / 64) * 8;  // 16-byte chunks per V row
                        for (int c = (warp - 2) * 32 + lane; c < (stop - first) * per_row; c += 128) {
                            const int vr = first + c / per_row, rem = c % per_row;
                            *reinterpret_cast<uint4 *>(vt + (rem / 8) * S::kHalf + vr * 128 + (rem % 8) * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                fence_proxy_async_smem();
                tmem_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
            }
            if (!ok) break;
            // Output: O / l for the valid rows.
            const uint32_t x_last = jt + d.nt - 1;
            if (!mbar_wait(o_done, x_last & 1, status, abort)) break;
            tmem_fence_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const long long t = (long long)d.q0 + d.mt * (kChunkRows / g) + row / g;
            const int hq = d.h * g + row % g;
            __nv_bfloat16 *dst = a.out + (t * a.num_q_heads + hq) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                tmem_ld32(lane_base + 256 + c * 32, o);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 pk;
                        pk.x = pack_bf16x2(o[e] * inv, o[e + 1] * inv);
                        pk.y = pack_bf16x2(o[e + 2] * inv, o[e + 3] * inv);
                        pk.z = pack_bf16x2(o[e + 4] * inv, o[e + 5] * inv);
                        pk.w = pack_bf16x2(o[e + 6] * inv, o[e + 7] * inv);
                        *reinterpret_cast<uint4 *>(dst + c * 32 + e) = pk;
                    }
                }
            }
            tmem_fence_before_sync();
            jt += d.nt;
        }
    }

    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (warp == 1) tmem_dealloc(tm, kTmemCols);
}

}  // namespace

int chunk_smem_bytes(int head_size) {
    return head_size == 128 ? ChunkSmem<128>::kAlloc : ChunkSmem<64>::kAlloc;
}

int chunk_configure() {
    if (cudaFuncSetAttribute(chunk_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, ChunkSmem<128>::kAlloc) !=
            cudaSuccess ||
        cudaFuncSetAttribute(chunk_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, ChunkSmem<64>::kAlloc) !=
            cudaSuccess)
        return PKV_E_CUDA;
    return PKV_OK;
}

cudaError_t chunk_launch(int head_size, int grid, const CUtensorMap &kv_map, const CUtensorMap &q_map,
                         const ChunkArgs &args, cudaStream_t stream) {
    if (head_size == 128)
        return launch_pdl(chunk_kernel<128>, dim3(grid), dim3(kChunkThreads), ChunkSmem<128>::kAlloc, stream, kv_map,
                          q_map, args);
    return launch_pdl(chunk_kernel<64>, dim3(grid), dim3(kChunkThreads), ChunkSmem<64>::kAlloc, stream, kv_map, q_map,
                      args);
}

}  // namespace pkv
