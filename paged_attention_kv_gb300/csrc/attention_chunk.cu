// Chunk-tile attention on tcgen05 tensor cores, for requests that bring many
// new tokens in one step (chunked prefill, "Inside vLLM", page 1, "Chunked
// prefill"; V1 mixes such chunks with decode tokens, "Scheduler").
//
// A work item is one 128-row query tile (rows = tokens x the q heads of one
// GQA group, token-major) of one request and kv head, over all keys its rows
// may see, in 128-key tiles. Per key tile x:
//   S(x) = Q K(x)^T   tcgen05.mma (M=128, N=128, K=16 steps), bf16 operands
//                     in 128B-swizzled shared memory, fp32 accumulator in
//                     TMEM; two S buffers, so S(x+1) is ready while the
//                     softmax works on S(x);
//   softmax           sixteen warps, four per TMEM lane quadrant: a row is
//                     one lane, its 128 keys split into four 32-key parts,
//                     one per warp; the four partial row maxima meet in
//                     shared memory (published before P is computed against
//                     the current reference, collected after). Causal mask,
//                     exp2 against a running reference max that only moves
//                     (P redone, O rescaled) when a row max grows by more
//                     than 2^8; P(x) goes to one of two P buffers in TMEM as
//                     bf16 pairs;
//   O += P(x) V(x)    tcgen05.mma (M=128, N=D) with A = P(x) read from TMEM
//                     and B = V MN-major straight from its TMA tile; O stays
//                     in TMEM.
// K and V tiles arrive one copy per block (16 keys x D; the copy engine
// spends a fixed cost per box, so one box per block rather than per 64
// columns), laid out [token half][D / 64][8 tokens][128 B]: the tile's 16
// groups of 8 keys are evenly spaced, so S is one N=128 product per K step
// and the PV product's K steps are single blocks.
// The softmax of tile x waits only for S(x) and for the P buffer of tile x-2
// to be consumed; the tensor core runs PV(x-1) and S(x+1) meanwhile. One
// warp per row would leave each SM sub-partition a single long dependency
// chain per tile; four shorter ones interleave. Warps: 0-15 softmax and
// output (warp w: lane quadrant w % 4, key part w / 4), 16 copies (item
// claims, Q tile, K tiles of 8 blocks), 17 MMA issuer (one elected lane) and
// TMEM owner, 18 copies of the V tiles (two warps issuing bulk copies get
// more into one SM than one warp issuing them all). Every wait is bounded;
// on a timeout the CTA raises PKV_DEV_TIMEOUT, stops, lets its in-flight
// copies and MMAs finish and frees its TMEM.
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


constexpr int kParts = 4;                          // softmax warps per TMEM lane quadrant
constexpr int kSoftmaxWarps = 4 * kParts;
constexpr int kPartKeys = kChunkKeys / kParts;     // keys of one warp's part
// Two copy warps, one for K and one for V: one SM takes in more when two
// warps issue its bulk copies than when one issues them all.
constexpr int kProducerWarp = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + 1, kVWarp = kSoftmaxWarps + 2;
constexpr int kChunkThreads = 32 * (kSoftmaxWarps + 3);
// TMEM columns: S0 | S1 (fp32, 128 each) | P0 | P1 (bf16 pairs, 64 each) | O (D).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColP = 256, kColO = 384;
constexpr float kRescaleThreshold = 8.f;  // log2 units: P stays <= 2^8

// mbarrier slots. S, P and PV-done by buffer (tile parity); a K ring of
// kK slots and a V ring of kV; a K slot is released once its S product is
// done, a V slot after its PV product. XBar: per lane quadrant and exchange
// parity, the four part warps' partial values are in shared memory.
template <int kK, int kV>
struct ChunkBars {
    static constexpr int kQFull = 0, kQTaken = 1, kQEmpty = 2;
    static constexpr int kKFull = 3;
    static constexpr int kKEmpty = kKFull + kK;
    static constexpr int kVFull = kKEmpty + kK;
    static constexpr int kVEmpty = kVFull + kV;
    static constexpr int kSFull = kVEmpty + kV;  // [2]
    static constexpr int kPFull = kSFull + 2;     // [2]
    static constexpr int kPvDone = kPFull + 2;    // [2]
    static constexpr int kODone = kPvDone + 2;
    static constexpr int kOFree = kODone + 1;
    static constexpr int kDrain = kOFree + 1;
    static constexpr int kXBar = kDrain + 1;      // [4 quadrants][2 parities]
    static constexpr int kDFull = kXBar + 8;      // the item is in desc (for the V copy warp)
    static constexpr int kCount = kDFull + 1;
};

// Item as the producer hands it to the other roles.
struct ChunkDesc {
    int item, r, mt, h, q0, n, L, nv, kv_end, nt, pad[6];
};

template <int D>
struct ChunkSmem {
    // K ring three deep at D = 128 (the S products wait on K more than the
    // PV products wait on V); that is what fits next to Q and the V ring.
    static constexpr int kKStages = D == 128 ? 3 : 4;
    static constexpr int kVStages = D == 128 ? 2 : 4;
    using Bars = ChunkBars<kKStages, kVStages>;
    static constexpr int kHalf = 16384;             // Q: 128 rows x 128 B (64 bf16 columns)
    static constexpr int kTile = (D / 64) * kHalf;  // 128 rows x D bf16
    static constexpr int kGrp = (D / 64) * 1024;    // K / V: 8 keys of one block [D / 64][8][128 B]
    static constexpr int kBlk = 2 * kGrp;           // one block: two 8-key groups
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTile;
    static constexpr int kOffV = kOffK + kKStages * kTile;
    static constexpr int kOffX = kOffV + kVStages * kTile;  // float [2][kParts][128]: partial maxima / sums
    static constexpr int kOffDesc = kOffX + 2 * kParts * kChunkRows * 4;
    static constexpr int kOffBar = kOffDesc + (int)sizeof(ChunkDesc);
    static constexpr int kOffTmem = kOffBar + Bars::kCount * 8;
    static constexpr int kBytes = kOffTmem + 16;
    static constexpr int kAlloc = kBytes + 1024;
};
static_assert(ChunkSmem<128>::kAlloc <= 232448, "chunk kernel shared memory");
static_assert(ChunkSmem<64>::kAlloc <= 232448, "chunk kernel shared memory");

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
    constexpr int kKStages = S::kKStages, kVStages = S::kVStages;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_abort;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::kOffBar);
    uint64_t *q_full = bar + B::kQFull, *q_taken = bar + B::kQTaken, *q_empty = bar + B::kQEmpty;
    uint64_t *k_full = bar + B::kKFull, *v_full = bar + B::kVFull;
    uint64_t *k_empty = bar + B::kKEmpty, *v_empty = bar + B::kVEmpty;
    uint64_t *s_full = bar + B::kSFull, *p_full = bar + B::kPFull, *pv_done = bar + B::kPvDone;
    uint64_t *o_done = bar + B::kODone, *o_free = bar + B::kOFree, *drain = bar + B::kDrain;
    uint64_t *xbar = bar + B::kXBar;
    uint64_t *d_full = bar + B::kDFull;
    float *xbuf = reinterpret_cast<float *>(smem + S::kOffX);
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
        mbar_init(q_taken, 2 + kSoftmaxWarps);  // the MMA warp, the V copy warp and the softmax warps
        mbar_init(q_empty, 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], kSoftmaxWarps);
            mbar_init(&pv_done[b], 1);
        }
        mbar_init(o_done, 1);
        mbar_init(o_free, kSoftmaxWarps);
        mbar_init(drain, 1);
        mbar_init(d_full, 1);
        for (int i = 0; i < 8; ++i) mbar_init(&xbar[i], kParts);
        mbar_fence_init();
    }
    // The barrier setup above overlaps the previous kernel; the work list it
    // wrote is read only after this. A batch without chunk tiles ends here,
    // before any TMEM is allocated.
    pdl_wait();
    pdl_launch_dependents();
    const int n_items = a.header->n_chunk_items;
    // Beside the split-KV kernel, CTAs past the work list's share leave
    // their SMs to it at once.
    if (n_items == 0 || (a.beside && (int)blockIdx.x >= a.header->chunk_ctas)) return;
    if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tm = *tmem_slot;

    if (warp == kProducerWarp) {
        // ---------------------- item, Q and K copy warp ----------------------
        if (lane == 0) {
            tma_prefetch_desc(&kv_map);
            tma_prefetch_desc(&q_map);
        }
        constexpr int kTileBlocks = kChunkKeys / PKV_BLOCK_SIZE;  // 8 blocks per key tile
        uint32_t jt = 0;  // K tiles of the items so far
        uint32_t k_issued = 0;
        bool ok = true;
        // Global reads that a load depends on are issued ahead of it: the
        // next item is claimed while the current one issues its last K tile,
        // and each key tile's block ids are read three tiles ahead (lane b <
        // 8 holds block b of the tile), so no copy waits on a round trip to
        // memory once the slot is free.
        int it_raw = 0;
        if (lane == 0) it_raw = atomicAdd(&a.header->next_chunk_item, 1);
        int it = __shfl_sync(0xffffffffu, it_raw, 0);
        ChunkItem w{};
        if (it < n_items) w = a.items[it];
        for (int k = 0; ok; ++k) {
            const int r = w.a.x, mt = w.a.y, h = w.a.z, kv_end = w.a.w;
            const int q0 = w.b.x, n = w.b.y, L = w.b.z, nv = w.b.w;
            const int nt = it < n_items ? (kv_end + kChunkKeys - 1) / kChunkKeys : 0;
            const int kvb = (kv_end + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE;
            const int32_t *bt = a.block_table + (long long)r * a.max_blocks_per_req;
            // Block id of lane `lane` in key tile t; past the request's
            // blocks it is a.num_blocks, past the map: TMA fills zeros.
            auto fetch = [&](int t) {
                const int kb = t * kTileBlocks + lane;
                return (lane < kTileBlocks && t < nt && kb < kvb) ? __ldg(bt + kb) : a.num_blocks;
            };
            int id0 = fetch(0), id1 = fetch(1), id2 = fetch(2);
            if (!mbar_wait(q_taken, (k & 1) ^ 1, status, abort) || !mbar_wait(q_empty, (k & 1) ^ 1, status, abort)) {
                ok = false;
                break;
            }
            if (it >= n_items) {
                if (lane == 0) {
                    desc->item = -1;
                    mbar_arrive(d_full);
                    mbar_arrive(q_full);
                }
                break;
            }
            if (lane == 0) {
                ChunkDesc d;
                d.item = it; d.r = r; d.mt = mt; d.h = h; d.q0 = q0; d.n = n; d.L = L; d.nv = nv;
                d.kv_end = kv_end; d.nt = nt;
                *desc = d;
                mbar_arrive(d_full);
                mbar_arrive_expect_tx(q_full, kChunkRows * D * 2);
#pragma unroll
                for (int bx = 0; bx < D / 64; ++bx)
                    tma_load_3d(smem + S::kOffQ + bx * S::kHalf, &q_map, bx * 64, h * g, q0 + mt * (kChunkRows / g),
                                q_full);
            }
            __syncwarp();
            // K of key tile j into its ring slot: eight blocks, one box each.
            auto load = [&](int j, int blk) {
                const uint32_t x = jt + j;
                const int st = x % kKStages;
                uint64_t *full = &k_full[st];
                if (!mbar_wait(&k_empty[st], ((x / kKStages) & 1) ^ 1, status, abort)) return false;
                if (blk < 0 || blk > a.num_blocks || (blk == a.num_blocks && j * kTileBlocks + lane < kvb)) {
                    if (lane < kTileBlocks) raise_status(status, PKV_DEV_BAD_BLOCK);
                    blk = a.num_blocks;
                }
                if (lane == 0) mbar_arrive_expect_tx(full, kChunkKeys * D * 2);
                __syncwarp();
                if (lane < kTileBlocks)
                    tma_load_5d(smem + S::kOffK + st * S::kTile + lane * S::kBlk, &kv_map, 0, 0, 0, h * 2, blk, full);
                __syncwarp();
                ++k_issued;
                return true;
            };
            auto claim_next = [&]() {
                if (lane == 0) it_raw = atomicAdd(&a.header->next_chunk_item, 1);
            };
            for (int j = 0; j < nt && ok; ++j) {
                ok = load(j, id0);
                if (j + 1 == nt) claim_next();
                id0 = id1;
                id1 = id2;
                id2 = fetch(j + 3);
            }
            jt += nt;
            it = __shfl_sync(0xffffffffu, it_raw, 0);
            if (it < n_items) w = a.items[it];
        }
        if (!ok && lane == 0) {
            // let copies already issued land before the CTA can leave
            for (uint32_t x = k_issued > (uint32_t)kKStages ? k_issued - kKStages : 0; x < k_issued; ++x)
                mbar_drain(&k_full[x % kKStages], (x / kKStages) & 1, status, diag, 0x2);
        }
    } else if (warp == kVWarp) {
        // ---------------------------- V copy warp ----------------------------
        // Takes each item from desc (d_full) and copies its V tiles, one box
        // per block, into the V ring; block ids read three tiles ahead.
        const int Hkv = a.num_kv_heads;
        constexpr int kTileBlocks = kChunkKeys / PKV_BLOCK_SIZE;
        uint32_t jt = 0, v_issued = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            if (!warp_wait(d_full, k & 1, status, abort)) { ok = false; break; }
            const ChunkDesc d = *desc;
            __syncwarp();
            if (lane == 0) mbar_arrive(q_taken);
            if (d.item < 0) break;
            const int nt = d.nt;
            const int kvb = (d.kv_end + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE;
            const int32_t *bt = a.block_table + (long long)d.r * a.max_blocks_per_req;
            auto fetch = [&](int t) {
                const int kb = t * kTileBlocks + lane;
                return (lane < kTileBlocks && t < nt && kb < kvb) ? __ldg(bt + kb) : a.num_blocks;
            };
            int id0 = fetch(0), id1 = fetch(1), id2 = fetch(2);
            for (int j = 0; j < nt && ok; ++j) {
                const uint32_t x = jt + j;
                const int st = x % kVStages;
                if (!warp_wait(&v_empty[st], ((x / kVStages) & 1) ^ 1, status, abort)) { ok = false; break; }
                int blk = id0;  // a bad id was reported by the K copy warp; TMA fills zeros for it here
                if (blk < 0 || blk > a.num_blocks || (blk == a.num_blocks && j * kTileBlocks + lane < kvb))
                    blk = a.num_blocks;
                if (lane == 0) mbar_arrive_expect_tx(&v_full[st], kChunkKeys * D * 2);
                __syncwarp();
                if (lane < kTileBlocks)
                    tma_load_5d(smem + S::kOffV + st * S::kTile + lane * S::kBlk, &kv_map, 0, 0, 0, (Hkv + d.h) * 2,
                                blk, &v_full[st]);
                __syncwarp();
                ++v_issued;
                id0 = id1;
                id1 = id2;
                id2 = fetch(j + 3);
            }
            jt += nt;
        }
        if (!ok && lane == 0) {
            // let copies already issued land before the CTA can leave
            for (uint32_t x = v_issued > (uint32_t)kVStages ? v_issued - kVStages : 0; x < v_issued; ++x)
                mbar_drain(&v_full[x % kVStages], (x / kVStages) & 1, status, diag, 0x2);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------ MMA issuer -----------------------------
        // The whole warp walks the schedule with the same values (so
        // descriptors and TMEM addresses stay warp-uniform); one elected lane
        // issues every tcgen05.mma and commit.
        constexpr uint32_t kIdS = umma_idesc_bf16(128, kChunkKeys, 0, 0);
        constexpr uint32_t kIdPV = umma_idesc_bf16(128, D, 0, 1);
        const uint32_t q_s = smem_u32(smem + S::kOffQ);
        const uint32_t k_s = smem_u32(smem + S::kOffK), v_s = smem_u32(smem + S::kOffV);
        uint32_t jt = 0;  // key tiles of the items so far (global tile index base)
        uint32_t n_items_done = 0;
        bool ok = true;
        // S(x) = Q K(x)^T into S buffer x & 1 (the key tile's 8-key groups
        // kGrp bytes apart). Its K slot is released when the product is done
        // (it is the slot's only reader).
        auto issue_s = [&](uint32_t x) {
            const int st = x % kKStages;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma_bf16_warp(tm + (x & 1) * kChunkKeys,
                               umma_desc_sw128(q_s + (kk / 4) * S::kHalf + (kk % 4) * 32, 16, 1024),
                               umma_desc_sw128(k_s + st * S::kTile + (kk / 4) * 1024 + (kk % 4) * 32, 16, S::kGrp),
                               kIdS, kk > 0 ? 1u : 0u);
            umma_commit_warp(&s_full[x & 1]);
            umma_commit_warp(&k_empty[st]);
        };
        for (int k = 0; ok; ++k) {
            if (!warp_wait(q_full, k & 1, status, abort)) { ok = false; break; }
            const ChunkDesc d = *desc;
            __syncwarp();
            if (lane == 0) mbar_arrive(q_taken);
            if (d.item < 0) break;
            const int nt = d.nt;
            // S of the first two key tiles
            for (int j = 0; j < min(nt, 2) && ok; ++j) {
                const uint32_t x = jt + j;
                if (!warp_wait(&k_full[x % kKStages], (x / kKStages) & 1, status, abort)) { ok = false; break; }
                tmem_fence_after_sync();
                issue_s(x);
            }
            if (!ok) break;
            if (nt <= 2) umma_commit_warp(q_empty);  // every S of the item is issued
            for (int j = 0; j < nt && ok; ++j) {
                const uint32_t x = jt + j;
                const int st = x % kVStages;
                if (!warp_wait(&p_full[x & 1], (x >> 1) & 1, status, abort)) { ok = false; break; }
                if (j == 0 && n_items_done > 0 && !warp_wait(o_free, (n_items_done - 1) & 1, status, abort)) {
                    ok = false;
                    break;
                }
                if (!warp_wait(&v_full[st], (x / kVStages) & 1, status, abort)) { ok = false; break; }
                tmem_fence_after_sync();
                // O += P(x) V(x): P from TMEM (64 columns of bf16 pairs), V
                // MN-major; K step kk is block kk (its two 8-key groups kGrp
                // apart, its 64-column halves 1 KiB apart).
#pragma unroll
                for (int kk = 0; kk < kChunkKeys / 16; ++kk) {
                    const uint64_t bd = umma_desc_sw128(v_s + st * S::kTile + kk * S::kBlk, 1024, S::kGrp);
                    umma_bf16_tmem_a_warp(tm + kColO, tm + kColP + (x & 1) * 64 + kk * 8, bd, kIdPV,
                                          (j > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit_warp(&pv_done[x & 1]);
                umma_commit_warp(&v_empty[st]);
                if (j == nt - 1) umma_commit_warp(o_done);
                if (j + 2 < nt) {
                    // S(x+2) reuses the S buffer of x, which the softmax read
                    // before it stored P(x).
                    const uint32_t y = x + 2;
                    if (!warp_wait(&k_full[y % kKStages], (y / kKStages) & 1, status, abort)) { ok = false; break; }
                    tmem_fence_after_sync();
                    issue_s(y);
                    if (j + 3 == nt) umma_commit_warp(q_empty);  // that was the item's last S
                }
            }
            jt += nt;
            ++n_items_done;
        }
        // make sure no MMA is still writing TMEM before it is freed
        umma_commit_warp(drain);
        if (lane == 0) mbar_drain(drain, 0, status, diag, 0x4);
        __syncwarp();
    } else {
        // --------------------------- softmax and output ---------------------------
        constexpr int kOCols = D / kParts;  // O columns this warp rescales and writes
        const int q4 = warp & 3;            // TMEM lane quadrant of this warp
        const int part = warp >> 2;         // which 32 keys of each key tile
        const int row = q4 * 32 + lane;     // query row of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const uint32_t o_col = tm + lane_off + kColO + part * kOCols;
        uint32_t jt = 0;      // key tiles of the items so far (global tile index base)
        uint32_t n_done = 0;  // items finished
        uint32_t n_x = 0;     // exchanges so far (the same sequence in the quadrant's four warps)
        // The four part warps of this quadrant pool one float per row:
        // publish, then (maybe after other work) collect; the result is the
        // same in all four (same values, same order). A warp publishes
        // exchange n + 2 into the slot of n only after collecting n + 1,
        // which every warp published after collecting n.
        auto publish = [&](float v) {
            xbuf[(n_x & 1) * (kParts * kChunkRows) + part * kChunkRows + row] = v;
            __syncwarp();
            if (lane == 0) mbar_arrive(&xbar[q4 * 2 + (n_x & 1)]);
        };
        auto collect = [&](bool is_max, float &res) -> bool {
            const int par = n_x & 1;
            if (!warp_wait(&xbar[q4 * 2 + par], (n_x >> 1) & 1, status, abort)) return false;
            const float *xb = xbuf + par * (kParts * kChunkRows);
            float r = xb[row];
#pragma unroll
            for (int p = 1; p < kParts; ++p) r = is_max ? fmaxf(r, xb[p * kChunkRows + row]) : r + xb[p * kChunkRows + row];
            res = r;
            ++n_x;
            return true;
        };
        for (int k = 0;; ++k) {
            if (!warp_wait(q_full, k & 1, status, abort)) break;
            const ChunkDesc d = *desc;
            __syncwarp();
            if (lane == 0) mbar_arrive(q_taken);
            if (d.item < 0) break;
            const int nt = d.nt;
            const int rho = d.mt * kChunkRows + row;
            const bool valid = row < d.nv;
            const int i = valid ? rho / g : 0;
            const int limit = valid ? d.L - d.n + i : d.kv_end - 1;
            float m_run = -INFINITY, l = 0.f;  // l: this part's keys only
            bool ok = true;
            for (int j = 0; j < nt; ++j) {
                const uint32_t x = jt + j;
                const uint32_t s_col = tm + lane_off + (x & 1) * kChunkKeys + part * kPartKeys;
                const uint32_t p_col = tm + lane_off + kColP + (x & 1) * 64 + part * (kPartKeys / 2);
                if (!warp_wait(&s_full[x & 1], (x >> 1) & 1, status, abort)) { ok = false; break; }
                tmem_fence_after_sync();
                const int key0 = j * kChunkKeys + part * kPartKeys;  // first key of this part
                // Parts the whole warp sees unmasked take a path without
                // per-key tests; with a positive scale the max can be taken
                // on the raw scores.
                const bool fast = __all_sync(0xffffffffu, key0 + kPartKeys - 1 <= limit) && a.scale_log2 > 0.f;
                float sv[kPartKeys];
                tmem_ld32(s_col, sv);
                tmem_wait_ld_regs(sv);
                // This part's P = 2^(s * scale - m) as bf16 pairs (32 keys ->
                // 16 columns); returns the sum of the unrounded values.
                auto compute_p = [&](const float (&sv)[kPartKeys], float neg_m, uint32_t (&pk)[kPartKeys / 2]) {
                    if (fast) {
                        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2), nm2 = make_float2(neg_m, neg_m);
                        float2 la2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                        for (int e = 0; e < kPartKeys / 2; ++e) {
                            const float2 xv = ffma2(make_float2(sv[2 * e], sv[2 * e + 1]), sc2, nm2);
                            const float2 p = make_float2(fast_exp2(xv.x), fast_exp2(xv.y));
                            la2[e & 1] = fadd2(la2[e & 1], p);
                            pk[e] = pack_bf16x2(p.x, p.y);
                        }
                        return (la2[0].x + la2[0].y) + (la2[1].x + la2[1].y);
                    }
                    float la[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int e = 0; e < kPartKeys / 2; ++e) {
                        const int kk = key0 + 2 * e;
                        const float p0 = kk <= limit ? fast_exp2(fmaf(sv[2 * e], a.scale_log2, neg_m)) : 0.f;
                        const float p1 = kk + 1 <= limit ? fast_exp2(fmaf(sv[2 * e + 1], a.scale_log2, neg_m)) : 0.f;
                        la[e & 3] += p0 + p1;
                        pk[e] = pack_bf16x2(p0, p1);
                    }
                    return (la[0] + la[1]) + (la[2] + la[3]);
                };
                // Partial row max (scaled, masked), published to the other
                // three parts of the row.
                {
                    float mxa[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                    if (fast) {
#pragma unroll
                        for (int e = 0; e < kPartKeys / 2; ++e)
                            mxa[e & 3] = fmax3(mxa[e & 3], sv[2 * e], sv[2 * e + 1]);
                    } else {
#pragma unroll
                        for (int e = 0; e < kPartKeys; ++e)
                            mxa[e & 3] = fmaxf(mxa[e & 3], key0 + e <= limit ? sv[e] * a.scale_log2 : -INFINITY);
                    }
                    float pm = fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3]));
                    if (fast) pm *= a.scale_log2;
                    publish(pm);
                }
                // The reference max moves only when the row max outgrows it by
                // more than 2^8. The first tile sets it (key 0 is visible to
                // every row, so the row max is finite there); later tiles
                // compute P against the current reference while the partial
                // maxima meet, and redo it in the rare case the row max
                // moved the reference.
                float mx;
                if (j == 0) {
                    if (!collect(true, mx)) { ok = false; break; }
                    m_run = mx;
                }
                uint32_t pk[kPartKeys / 2];
                float sum = compute_p(sv, -m_run, pk);
                float alpha = 1.f;
                bool any_resc = false;
                if (j > 0) {
                    if (!collect(true, mx)) { ok = false; break; }
                    const bool resc = mx > m_run + kRescaleThreshold;
                    any_resc = __any_sync(0xffffffffu, resc);
                    if (any_resc) {
                        if (resc) {
                            alpha = fast_exp2(m_run - mx);
                            m_run = mx;
                        }
                        // S(x) is still in TMEM: its buffer is rewritten only
                        // after PV(x), which waits for this P.
                        float sv2[kPartKeys];
                        tmem_ld32(s_col, sv2);
                        tmem_wait_ld_regs(sv2);
                        sum = compute_p(sv2, -m_run, pk);
                    }
                }
                // The P buffer of x was last read by PV(x-2).
                if (x >= 2) {
                    const uint32_t y = x - 2;
                    if (!warp_wait(&pv_done[y & 1], (y >> 1) & 1, status, abort)) { ok = false; break; }
                    tmem_fence_after_sync();
                }
                tmem_st16u(p_col, pk);
                l = fmaf(l, alpha, sum);
                // O (this warp's columns) follows a moved reference once
                // PV(x-1) is done, before PV(x) is issued.
                if (any_resc) {
                    const uint32_t y = x - 1;
                    if (!warp_wait(&pv_done[y & 1], (y >> 1) & 1, status, abort)) { ok = false; break; }
                    tmem_fence_after_sync();
                    float o[kOCols];
                    tmem_ld_cols(o_col, o);
                    tmem_wait_ld_regs(o);
#pragma unroll
                    for (int e = 0; e < kOCols; ++e) o[e] *= alpha;
                    tmem_st_cols(o_col, o);
                }
                // V rows past the tile's last visible key hold other data
                // (maybe NaN); their P is 0 but 0 * NaN is not, so clear them.
                if (j == nt - 1) {
                    const int tile0 = j * kChunkKeys;
                    const int first = d.kv_end - tile0;
                    const int stop =
                        min(kChunkKeys, ((d.kv_end + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE) * PKV_BLOCK_SIZE - tile0);
                    if (first < stop) {
                        const int st = x % kVStages;
                        if (!warp_wait(&v_full[st], (x / kVStages) & 1, status, abort)) { ok = false; break; }
                        uint8_t *vt = smem + S::kOffV + st * S::kTile;
                        const int per_row = (D / 64) * 8;  // 16-byte chunks per V row
                        for (int c = warp * 32 + lane; c < (stop - first) * per_row; c += kSoftmaxWarps * 32) {
                            const int vr = first + c / per_row, rem = c % per_row;
                            *reinterpret_cast<uint4 *>(vt + (vr / 8) * S::kGrp + (rem / 8) * 1024 + (vr % 8) * 128 +
                                                       (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                    }
                }
                tmem_wait_st();
                tmem_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[x & 1]);
            }
            jt += nt;
            if (!ok) break;
            // Output: O / l for the valid rows, this warp's D / 4 columns.
            float l_row;
            publish(l);
            if (!collect(false, l_row)) break;
            if (!warp_wait(o_done, n_done & 1, status, abort)) break;
            ++n_done;
            tmem_fence_after_sync();
            const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
            __nv_bfloat16 *dst =
                a.out + (((long long)d.q0 + i) * a.num_q_heads + d.h * g + rho % g) * D + part * kOCols;
            {
                float o[kOCols];
                tmem_ld_cols(o_col, o);
                tmem_wait_ld_regs(o);
                if (valid) {
#pragma unroll
                    for (int e = 0; e < kOCols; e += 8) {
                        uint4 pk;
                        pk.x = pack_bf16x2(o[e] * inv, o[e + 1] * inv);
                        pk.y = pack_bf16x2(o[e + 2] * inv, o[e + 3] * inv);
                        pk.z = pack_bf16x2(o[e + 4] * inv, o[e + 5] * inv);
                        pk.w = pack_bf16x2(o[e + 6] * inv, o[e + 7] * inv);
                        *reinterpret_cast<uint4 *>(dst + e) = pk;
                    }
                }
            }
            tmem_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
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
