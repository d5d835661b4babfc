// Chunk-tile attention on tcgen05 tensor cores, for requests that bring many
// new tokens in one step (chunked prefill, "Inside vLLM", page 1, "Chunked
// prefill"; V1 mixes such chunks with decode tokens, "Scheduler").
//
// A work item is a pair of 128-row query tiles A and B (rows = tokens x the
// q heads of one GQA group, token-major; B is the next 128 rows of the same
// request and may be empty) of one request and kv head. Both tiles run over
// one stream of 128-key K/V tiles (B, later in the chunk, sees as many keys
// as A or more), and take turns on the tensor core:
//   S_t = Q_t K^T   tcgen05.mma (M=128, N=128, K=16 steps), bf16 operands in
//                   128B-swizzled shared memory, fp32 accumulator in TMEM;
//   softmax         four warps per tile, one thread per row (its TMEM lane):
//                   causal mask, exp2 against a running reference max that
//                   only moves (and rescales O_t) when a row max grows by
//                   more than 2^8; P_t goes back into the TMEM columns of S_t
//                   as bf16 pairs;
//   O_t += P_t V    tcgen05.mma (M=128, N=D) with A = P_t read from TMEM and
//                   B = V MN-major straight from its TMA tile; O_t stays in
//                   TMEM.
// The MMA warp issues S_A(0), S_B(0), then PV_A(j), S_A(j+1), PV_B(j),
// S_B(j+1), ...: while the softmax warps of one tile work, the tensor core
// can run the other tile's products. Warps: 0 TMA producer (Q tiles; K and V tiles of 8 blocks, one
// box per 64 columns of each block), 1 MMA issuer (one elected lane) and
// TMEM owner, 2-5 softmax and output of tile A, 6-9 of tile B. Every wait is
// bounded; on a timeout the CTA raises PKV_DEV_TIMEOUT, stops, lets its
// in-flight copies and MMAs finish and frees its TMEM.
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

// Warps 0-3 softmax of tile A, 4-7 of tile B (one warpgroup each), 8 TMA
// producer, 9 MMA issuer, 10-11 idle (they only give their registers to
// the softmax warpgroups).
constexpr int kChunkThreads = 384;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
// Register budget per thread after the split (launch allocation: 168 per
// thread at 384 threads). 256 softmax threads x 192 + 128 x 120 = 64512 =
// 384 x 168: the decreases return exactly what the increases take; per
// sub-partition 192 + 192 + 120 = 504 <= 512.
constexpr uint32_t kRegsSoftmax = 192, kRegsOther = 120;
constexpr uint32_t kTmemCols = 512;       // S_A | S_B | O_A | O_B
constexpr float kRescaleThreshold = 8.f;  // log2 units: P stays <= 2^8
constexpr int kSoftmaxArrivals = 4;       // warps per tile

// mbarrier slots. Per tile t (0 = A, 1 = B): S ready, P stored, the item's
// last PV done, O read out. K and V have rings of kStages slots each; a K
// slot is released once the last S product reading it is done, a V slot
// after the last PV, so K runs a tile ahead of V.
template <int kStages>
struct ChunkBars {
    static constexpr int kQFull = 0, kQTaken = 1, kQEmpty = 2;
    static constexpr int kKFull = 3;
    static constexpr int kVFull = kKFull + kStages;
    static constexpr int kKEmpty = kVFull + kStages;
    static constexpr int kVEmpty = kKEmpty + kStages;
    static constexpr int kSFull = kVEmpty + kStages;  // [2]
    static constexpr int kPFull = kSFull + 2;          // [2]
    static constexpr int kODone = kPFull + 2;          // [2]
    static constexpr int kOFree = kODone + 2;          // [2]
    static constexpr int kDrain = kOFree + 2;
    static constexpr int kCount = kDrain + 1;
};

// Item as the producer hands it to the other roles.
struct ChunkDesc {
    int item, r, pair, h, q0, n, L, nv_a, nv_b, kv_end_a, kv_end_b, nt_a, nt_b, pad[3];
};

template <int D>
struct ChunkSmem {
    static constexpr int kStages = D == 128 ? 2 : 4;
    using Bars = ChunkBars<kStages>;
    static constexpr int kHalf = 16384;             // 128 rows x 128 B (64 bf16 columns)
    static constexpr int kTile = (D / 64) * kHalf;  // 128 rows x D bf16
    static constexpr int kOffQ = 0;                 // Q_A, Q_B
    static constexpr int kOffK = kOffQ + 2 * kTile;
    static constexpr int kOffV = kOffK + kStages * kTile;
    static constexpr int kOffDesc = kOffV + kStages * kTile;
    static constexpr int kOffBar = kOffDesc + (int)sizeof(ChunkDesc);
    static constexpr int kOffTmem = kOffBar + Bars::kCount * 8;
    static constexpr int kBytes = kOffTmem + 16;
    static constexpr int kAlloc = kBytes + 1024;
};
static_assert(ChunkSmem<128>::kAlloc <= 232448, "chunk kernel shared memory");
static_assert(ChunkSmem<64>::kAlloc <= 232448, "chunk kernel shared memory");

// Keys visible to the last valid row of a tile that starts at row `row0` of
// a request (n new tokens, context L, GQA group g) and holds nv rows.
__device__ __forceinline__ int chunk_tile_kv_end(int n, int L, int g, int row0, int nv) {
    return L - n + (row0 + nv - 1) / g + 1;
}

// A bounded wait that the whole warp leaves with one answer (the warp runs
// warp-collective TMEM instructions afterwards).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int32_t *status, volatile int *abort) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, abort));
}

template <int D>
__global__ void __launch_bounds__(kChunkThreads, 1)
chunk_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
             const ChunkArgs a) {
    using S = ChunkSmem<D>;
    using B = typename S::Bars;
    constexpr int kStages = S::kStages;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_abort;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::kOffBar);
    uint64_t *q_full = bar + B::kQFull, *q_taken = bar + B::kQTaken, *q_empty = bar + B::kQEmpty;
    uint64_t *k_full = bar + B::kKFull, *v_full = bar + B::kVFull;
    uint64_t *k_empty = bar + B::kKEmpty, *v_empty = bar + B::kVEmpty;
    uint64_t *s_full = bar + B::kSFull, *p_full = bar + B::kPFull;
    uint64_t *o_done = bar + B::kODone, *o_free = bar + B::kOFree, *drain = bar + B::kDrain;
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
        mbar_init(q_taken, 1 + 2 * kSoftmaxArrivals);  // the MMA thread and eight softmax warps
        mbar_init(q_empty, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], kSoftmaxArrivals);
            mbar_init(&o_done[t], 1);
            mbar_init(&o_free[t], kSoftmaxArrivals);
        }
        mbar_init(drain, 1);
        mbar_fence_init();
    }
    // The barrier setup above overlaps the previous kernel; the work list it
    // wrote is read only after this. A batch without chunk tiles ends here,
    // before any TMEM is allocated.
    pdl_wait();
    pdl_launch_dependents();
    const int n_items = a.header->n_chunk_items;
    if (n_items == 0) return;
    if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tm = *tmem_slot;

    if (warp >= 2 * kSoftmaxArrivals) {
        setmaxnreg_dec<kRegsOther>();
        if (warp == kProducerWarp) {
            // ------------------------------ producer ------------------------------
            if (lane == 0) {
                tma_prefetch_desc(&kv_map);
                tma_prefetch_desc(&q_map);
            }
            const int Hkv = a.num_kv_heads;
            uint32_t jt = 0;                   // K/V tiles of the items so far
            uint32_t k_issued = 0, v_issued = 0;
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
                const int r = w.a.x, pair = w.a.y, h = w.a.z;
                const int q0 = w.b.x, n = w.b.y, L = w.b.z, nv = w.b.w;  // nv: valid rows of the pair
                const int nv_a = min(kChunkRows, nv), nv_b = nv - nv_a;
                const int row0 = pair * kChunkPairRows;
                const int kv_end_a = chunk_tile_kv_end(n, L, g, row0, nv_a);
                const int kv_end_b = nv_b > 0 ? chunk_tile_kv_end(n, L, g, row0 + kChunkRows, nv_b) : 0;
                const int nt_a = (kv_end_a + kChunkKeys - 1) / kChunkKeys;
                const int nt_b = (kv_end_b + kChunkKeys - 1) / kChunkKeys;
                const int nt = max(nt_a, nt_b);
                const int kvb = (max(kv_end_a, kv_end_b) + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE;
                if (lane == 0) {
                    ChunkDesc d;
                    d.item = it; d.r = r; d.pair = pair; d.h = h; d.q0 = q0; d.n = n; d.L = L;
                    d.nv_a = nv_a; d.nv_b = nv_b; d.kv_end_a = kv_end_a; d.kv_end_b = kv_end_b;
                    d.nt_a = nt_a; d.nt_b = nt_b;
                    *desc = d;
                    const int tiles = nv_b > 0 ? 2 : 1;
                    mbar_arrive_expect_tx(q_full, (uint32_t)tiles * kChunkRows * D * 2);
                    for (int t = 0; t < tiles; ++t) {
                        const int tok = q0 + (row0 + t * kChunkRows) / g;
    #pragma unroll
                        for (int bx = 0; bx < D / 64; ++bx)
                            tma_load_3d(smem + S::kOffQ + t * S::kTile + bx * S::kHalf, &q_map, bx * 64, h * g, tok,
                                        q_full);
                    }
                }
                __syncwarp();
                const int32_t *bt = a.block_table + (long long)r * a.max_blocks_per_req;
                // K or V of key tile j into its ring slot: eight blocks, one box
                // per 64 columns of each.
                auto load = [&](bool is_v, int j) {
                    const uint32_t x = jt + j;
                    const int st = x % kStages;
                    uint64_t *full = is_v ? &v_full[st] : &k_full[st];
                    if (!mbar_wait(is_v ? &v_empty[st] : &k_empty[st], ((x / kStages) & 1) ^ 1, status, abort))
                        return false;
                    int blk = a.num_blocks;  // past the map: TMA fills zeros
                    const int kb = j * (kChunkKeys / PKV_BLOCK_SIZE) + lane;
                    if (lane < kChunkKeys / PKV_BLOCK_SIZE && kb < kvb) {
                        blk = __ldg(bt + kb);
                        if (blk < 0 || blk >= a.num_blocks) {
                            raise_status(status, PKV_DEV_BAD_BLOCK);
                            blk = a.num_blocks;
                        }
                    }
                    if (lane == 0) mbar_arrive_expect_tx(full, kChunkKeys * D * 2);
                    __syncwarp();
                    if (lane < kChunkKeys / PKV_BLOCK_SIZE) {
                        uint8_t *dst = smem + (is_v ? S::kOffV : S::kOffK) + st * S::kTile + lane * 2048;
                        const int row = (is_v ? Hkv + h : h) * PKV_BLOCK_SIZE;
    #pragma unroll
                        for (int bx = 0; bx < D / 64; ++bx) tma_load_3d(dst + bx * S::kHalf, &kv_map, bx * 64, row, blk, full);
                    }
                    __syncwarp();
                    if (is_v) ++v_issued; else ++k_issued;
                    return true;
                };
                // K runs one tile ahead of V.
                ok = load(false, 0);
                for (int j = 0; j < nt && ok; ++j) {
                    if (j + 1 < nt) ok = load(false, j + 1);
                    if (ok) ok = load(true, j);
                }
                jt += nt;
            }
            if (!ok && lane == 0) {
                // let copies already issued land before the CTA can leave
                for (uint32_t x = k_issued > (uint32_t)kStages ? k_issued - kStages : 0; x < k_issued; ++x)
                    mbar_drain(&k_full[x % kStages], (x / kStages) & 1, status, diag, 0x2);
                for (uint32_t x = v_issued > (uint32_t)kStages ? v_issued - kStages : 0; x < v_issued; ++x)
                    mbar_drain(&v_full[x % kStages], (x / kStages) & 1, status, diag, 0x2);
            }
        } else if (warp == kMmaWarp) {
            // ------------------------------ MMA issuer -----------------------------
            // The whole warp runs this loop with the same values (so descriptors
            // and TMEM addresses stay warp-uniform); one elected lane issues
            // every tcgen05.mma and commit.
            {
                constexpr uint32_t kIdS = umma_idesc_bf16(128, kChunkKeys, 0, 0);
                constexpr uint32_t kIdPV = umma_idesc_bf16(128, D, 0, 1);
                const uint32_t q_s = smem_u32(smem + S::kOffQ);
                const uint32_t k_s = smem_u32(smem + S::kOffK), v_s = smem_u32(smem + S::kOffV);
                uint32_t jt = 0;                 // K/V tiles consumed so far
                uint32_t n_p[2] = {0, 0};        // P handoffs taken per tile
                uint32_t n_items_t[2] = {0, 0};  // items finished per tile
                bool ok = true;
                // S_t(x) = Q_t K(x)^T into TMEM columns t * 128
                auto issue_s = [&](int t, uint32_t x) {
                    const int st = x % kStages;
    #pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk / 4) * S::kHalf + (kk % 4) * 32;
                        umma_bf16_warp(tm + t * kChunkKeys, umma_desc_sw128(q_s + t * S::kTile + off, 16, 1024),
                                       umma_desc_sw128(k_s + st * S::kTile + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
                    }
                    umma_commit_warp(&s_full[t]);
                };
                for (int k = 0; ok; ++k) {
                    if (!warp_wait(q_full, k & 1, status, abort)) { ok = false; break; }
                    const ChunkDesc d = *desc;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(q_taken);
                    if (d.item < 0) break;
                    const int nt_t[2] = {d.nt_a, d.nt_b};
                    const int nt = max(d.nt_a, d.nt_b);
                    int s_left = d.nt_a + d.nt_b;  // S products of this item still to issue
                    // S of the first key tile, for both tiles
                    if (!warp_wait(&k_full[jt % kStages], (jt / kStages) & 1, status, abort)) { ok = false; break; }
                    tmem_fence_after_sync();
    #pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (nt_t[t] > 0) {
                            issue_s(t, jt);
                            if (--s_left == 0) umma_commit_warp(q_empty);
                        }
                    }
                    umma_commit_warp(&k_empty[jt % kStages]);  // both S products of key tile 0 are issued
                    for (int j = 0; j < nt && ok; ++j) {
                        const uint32_t x = jt + j;
                        const int st = x % kStages;
                        bool v_ready = false, k_next_ready = false;
    #pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            if (j >= nt_t[t]) continue;
                            if (!warp_wait(&p_full[t], n_p[t] & 1, status, abort)) { ok = false; break; }
                            ++n_p[t];
                            if (j == 0 && n_items_t[t] > 0 &&
                                !warp_wait(&o_free[t], (n_items_t[t] - 1) & 1, status, abort)) {
                                ok = false;
                                break;
                            }
                            if (!v_ready) {
                                if (!warp_wait(&v_full[st], (x / kStages) & 1, status, abort)) { ok = false; break; }
                                v_ready = true;
                            }
                            tmem_fence_after_sync();
                            // O_t += P_t V: P_t from TMEM (64 columns of bf16 pairs), V MN-major.
    #pragma unroll
                            for (int kk = 0; kk < kChunkKeys / 16; ++kk) {
                                const uint64_t bd = umma_desc_sw128(v_s + st * S::kTile + kk * 2048, S::kHalf, 1024);
                                umma_bf16_tmem_a_warp(tm + 256 + t * D, tm + t * kChunkKeys + kk * 8, bd, kIdPV,
                                                      (j > 0 || kk > 0) ? 1u : 0u);
                            }
                            if (j == nt_t[t] - 1) {
                                umma_commit_warp(&o_done[t]);
                                ++n_items_t[t];
                            }
                            if (t == 1 || nt_t[1] <= j) umma_commit_warp(&v_empty[st]);  // last PV on this V tile
                            if (j + 1 < nt_t[t]) {
                                // S_t(j+1) follows PV_t(j), which read P_t from the same columns
                                if (!k_next_ready) {
                                    const uint32_t y = x + 1;
                                    if (!warp_wait(&k_full[y % kStages], (y / kStages) & 1, status, abort)) {
                                        ok = false;
                                        break;
                                    }
                                    k_next_ready = true;
                                }
                                issue_s(t, x + 1);
                                if (--s_left == 0) umma_commit_warp(q_empty);
                                if (t == 1 || nt_t[1] <= j + 1) umma_commit_warp(&k_empty[(x + 1) % kStages]);
                            }
                        }
                    }
                    jt += nt;
                }
                // make sure no MMA is still writing TMEM before it is freed
                umma_commit_warp(drain);
                if (lane == 0) mbar_drain(drain, 0, status, diag, 0x4);
            }
            __syncwarp();
        }
    } else {
        setmaxnreg_inc<kRegsSoftmax>();
        // --------------------------- softmax and output ---------------------------
        const int t = warp >> 2;         // 0: tile A (warps 0-3), 1: tile B (warps 4-7)
        const int q4 = warp & 3;        // TMEM lane quadrant this warp may access
        const int row = q4 * 32 + lane; // query row of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const uint32_t s_col = tm + lane_off + t * kChunkKeys;
        const uint32_t o_col = tm + lane_off + 256 + t * D;
        uint32_t n_s = 0;     // S handoffs taken
        uint32_t n_done = 0;  // items finished
        uint32_t jt = 0;      // K/V tiles of the items seen so far
        for (int k = 0;; ++k) {
            if (!warp_wait(q_full, k & 1, status, abort)) break;
            const int item = desc->item;
            const int nt_a = desc->nt_a, nt_b = desc->nt_b;
            const int nv = t ? desc->nv_b : desc->nv_a;
            const int kv_end = t ? desc->kv_end_b : desc->kv_end_a;
            const int kv_end_pair = max(desc->kv_end_a, desc->kv_end_b);
            const int rho = desc->pair * kChunkPairRows + t * kChunkRows + row;
            const int ctx0 = desc->L - desc->n;  // keys before the chunk's first token
            const long long out_row0 = (long long)desc->q0 * a.num_q_heads + desc->h * g;
            __syncwarp();
            if (lane == 0) mbar_arrive(q_taken);
            if (item < 0) break;
            const int nt_mine = t ? nt_b : nt_a;
            const int nt = max(nt_a, nt_b);
            // The tile whose PV comes first on the last K/V tile clears
            // that tile's V rows past the pair's last visible key.
            const bool zeroes = t ? (nt_a < nt) : (nt_a == nt);
            const bool valid = row < nv;
            const int i = valid ? rho / g : 0;
            const int limit = valid ? ctx0 + i : kv_end - 1;
            float m_run = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < nt_mine; ++j) {
                if (!warp_wait(&s_full[t], n_s & 1, status, abort)) { ok = false; break; }
                ++n_s;
                tmem_fence_after_sync();
                const int key0 = j * kChunkKeys;
                // Tiles the whole warp sees unmasked (all but the diagonal
                // ones) take a path without per-key tests; with a positive
                // scale the max can be taken on the raw scores.
                const bool fast = __all_sync(0xffffffffu, key0 + kChunkKeys - 1 <= limit) && a.scale_log2 > 0.f;
                // The row's 128 scores of this key tile: one TMEM round trip.
                float sv[kChunkKeys / 32][32];
#pragma unroll
                for (int c = 0; c < kChunkKeys / 32; ++c) tmem_ld32(s_col + c * 32, sv[c]);
#pragma unroll
                for (int c = 0; c < kChunkKeys / 32; ++c) tmem_wait_ld_regs(sv[c]);
                // Row max (scaled, masked), eight independent maxima.
                float mx = -INFINITY;
                {
                    float mxa[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) mxa[e] = -INFINITY;
                    if (fast) {
#pragma unroll
                        for (int c = 0; c < kChunkKeys / 32; ++c)
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                mxa[(c * 16 + e) & 7] = fmax3(mxa[(c * 16 + e) & 7], sv[c][2 * e], sv[c][2 * e + 1]);
                    } else {
#pragma unroll
                        for (int c = 0; c < kChunkKeys / 32; ++c)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                mxa[e & 7] = fmaxf(mxa[e & 7], key0 + c * 32 + e <= limit ? sv[c][e] * a.scale_log2
                                                                                         : -INFINITY);
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx = fmaxf(mx, mxa[e]);
                    if (fast) mx *= a.scale_log2;
                }
                if (j == 0) {
                    m_run = mx;  // key 0 is visible to every row, so this is finite
                } else {
                    // PV_t(j-1) completed before S_t(j) was reported, so O_t
                    // may be rescaled in place.
                    const bool resc = mx > m_run + kRescaleThreshold;
                    if (__any_sync(0xffffffffu, resc)) {
                        const float alpha = resc ? fast_exp2(m_run - mx) : 1.f;
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            float o[32];
                            tmem_ld32(o_col + c * 32, o);
                            tmem_wait_ld_regs(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] *= alpha;
                            tmem_st32(o_col + c * 32, o);
                        }
                        l *= alpha;
                        if (resc) m_run = mx;
                    }
                }
                // P = 2^(s * scale - m_run) as bf16 pairs over the first 64
                // columns of S_t (32 keys -> 16 columns per store).
                {
                    const float neg_m = -m_run;
                    float la[4] = {0.f, 0.f, 0.f, 0.f};
                    float2 la2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                    for (int c = 0; c < kChunkKeys / 32; ++c) {
                        uint32_t pk[16];
                        if (fast) {
                            const float2 sc2 = make_float2(a.scale_log2, a.scale_log2), nm2 = make_float2(neg_m, neg_m);
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const float2 x = ffma2(make_float2(sv[c][2 * e], sv[c][2 * e + 1]), sc2, nm2);
                                const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                                la2[e & 1] = fadd2(la2[e & 1], p);
                                pk[e] = pack_bf16x2(p.x, p.y);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const int kk = key0 + c * 32 + 2 * e;
                                const float p0 = kk <= limit ? fast_exp2(fmaf(sv[c][2 * e], a.scale_log2, neg_m)) : 0.f;
                                const float p1 =
                                    kk + 1 <= limit ? fast_exp2(fmaf(sv[c][2 * e + 1], a.scale_log2, neg_m)) : 0.f;
                                la[e & 3] += p0 + p1;
                                pk[e] = pack_bf16x2(p0, p1);
                            }
                        }
                        tmem_st16u(s_col + c * 16, pk);
                    }
                    l += ((la[0] + la[1]) + (la[2] + la[3])) + ((la2[0].x + la2[0].y) + (la2[1].x + la2[1].y));
                }
                // V rows past the pair's last visible key hold other data
                // (maybe NaN); their P is 0 but 0 * NaN is not, so clear them.
                if (zeroes && j == nt - 1) {
                    const int first = kv_end_pair - key0;
                    const int stop =
                        min(kChunkKeys, ((kv_end_pair + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE) * PKV_BLOCK_SIZE - key0);
                    if (first < stop) {
                        const uint32_t x = jt + j;
                        const int st = x % kStages;
                        if (!warp_wait(&v_full[st], (x / kStages) & 1, status, abort)) { ok = false; break; }
                        uint8_t *vt = smem + S::kOffV + st * S::kTile;
                        const int per_row = (D / 64) * 8;  // 16-byte chunks per V row
                        for (int c = q4 * 32 + lane; c < (stop - first) * per_row; c += 128) {
                            const int vr = first + c / per_row, rem = c % per_row;
                            *reinterpret_cast<uint4 *>(vt + (rem / 8) * S::kHalf + vr * 128 + (rem % 8) * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                    }
                }
                tmem_wait_st();
                tmem_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[t]);
            }
            jt += nt;
            if (!ok) break;
            if (nt_mine == 0) continue;
            // Output: O_t / l for the valid rows.
            if (!warp_wait(&o_done[t], n_done & 1, status, abort)) break;
            ++n_done;
            tmem_fence_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *dst = a.out + (out_row0 + (long long)i * a.num_q_heads + rho % g) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                tmem_ld32(o_col + c * 32, o);
                tmem_wait_ld_regs(o);
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
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[t]);
        }
    }

    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (warp == kMmaWarp) tmem_dealloc(tm, kTmemCols);
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
