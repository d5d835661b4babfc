// Paged attention over a flattened ragged batch ("Inside vLLM", page 1, "Run
// forward pass" step 3: one super sequence, each sequence attending only to
// its own tokens; decode and chunked-prefill requests mixed in one step).
//
// Three launches on the caller's stream:
//   plan_kernel    one CTA turns query_start_loc / seq_lens into a work list
//                  (attention_plan.cuh), choosing the split-KV length so the
//                  persistent grid gets ~kItemsPerCta items per CTA;
//   decode_kernel  persistent, warp-specialised: one producer warp gathers
//                  each K/V block tile (16 rows x D, contiguous in the pool)
//                  with TMA into a shared-memory ring; four consumer warps run
//                  S = Q K^T and O += P V on bf16 mma.sync tensor-core tiles
//                  with an fp32 online softmax (exp2 domain), then combine
//                  their partial states in shared memory;
//   merge_kernel   combines the split partials of tiles with several splits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attention_plan.cuh"
#include "pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kPlanThreads = 1024;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// plan
// ---------------------------------------------------------------------------

struct PlanArgs {
    const int32_t *qsl;
    const int32_t *seq_lens;
    int num_reqs, num_tokens, max_blocks_per_req, group, num_kv_heads;
    long long target_items, parts_cap, groups_cap, items_cap;
    WsHeader *header;
    int32_t *req_group_base;
    int32_t *group_kvb;
    int2 *tile_info;
    WorkItem *items;
};

// Exclusive scan over the 1024 threads of the block; *total gets the sum.
template <typename T>
__device__ T block_exclusive_scan(T v, T *total, T *smem32) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) smem32[warp] = x;
    __syncthreads();
    if (warp == 0) {
        T w = (lane < (int)(blockDim.x >> 5)) ? smem32[lane] : T(0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            T y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        smem32[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    const T warp_prefix = warp ? smem32[warp - 1] : T(0);
    *total = smem32[(blockDim.x >> 5) - 1];
    __syncthreads();
    return warp_prefix + x - v;
}

template <typename T>
__device__ T block_sum(T v, T *smem32) {
    T total;
    block_exclusive_scan<T>(v, &total, smem32);
    return total;
}

// Keys visible to the last valid row of tile mt of a request (n new tokens,
// context L, GQA group g): rows are ordered by token, so that row sees the
// most keys.
__device__ __forceinline__ int tile_kv_end(int n, int L, int g, int mt) {
    const long long last_row = min((long long)n * g - 1, (long long)mt * kRowsPerTile + kRowsPerTile - 1);
    return L - n + (int)(last_row / g) + 1;
}

__device__ __forceinline__ int find_group_request(const int32_t *req_group_base, int num_reqs, int gi) {
    int lo = 0, hi = num_reqs;  // last r with base[r] <= gi, requests with no tiles skipped
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (req_group_base[mid] <= gi) lo = mid; else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
    __shared__ long long s_ll[32];
    __shared__ int s_i[32];
    __shared__ int s_split;
    const int tid = threadIdx.x;
    int32_t *status = &a.header->status;
    if (tid == 0) {
        a.header->status = 0;
        if (a.qsl[0] != 0 || a.qsl[a.num_reqs] != a.num_tokens) atomicOr(status, PKV_DEV_BAD_QSL);
    }
    __syncthreads();

    // 1. tiles per request -> req_group_base (exclusive scan, chunked).
    int carry = 0;
    for (int base = 0; base < a.num_reqs; base += kPlanThreads) {
        const int r = base + tid;
        int mtiles = 0;
        if (r < a.num_reqs) {
            const int q0 = a.qsl[r], q1 = a.qsl[r + 1], L = a.seq_lens[r];
            const int n = q1 - q0;
            if (n < 0 || q0 < 0 || q1 > a.num_tokens) {
                atomicOr(status, PKV_DEV_BAD_QSL);
            } else if (n > L || (long long)L > (long long)a.max_blocks_per_req * PKV_BLOCK_SIZE) {
                atomicOr(status, PKV_DEV_BAD_LEN);
            } else {
                mtiles = (int)(((long long)n * a.group + kRowsPerTile - 1) / kRowsPerTile);
            }
        }
        int chunk_total;
        const int ex = block_exclusive_scan<int>(mtiles, &chunk_total, s_i);
        if (r < a.num_reqs) a.req_group_base[r] = carry + ex;
        carry += chunk_total;
    }
    int n_groups = carry;
    if (n_groups > a.groups_cap) {
        // Only overlapping (invalid) query_start_loc ranges get here: keep
        // every table index in bounds.
        if (tid == 0) atomicOr(status, PKV_DEV_OVERFLOW);
        n_groups = (int)a.groups_cap;
        __syncthreads();
        for (int r = tid; r < a.num_reqs; r += kPlanThreads)
            a.req_group_base[r] = min(a.req_group_base[r], n_groups);
    }
    if (tid == 0) a.req_group_base[a.num_reqs] = n_groups;
    __syncthreads();

    // 2. keys per group, total work in block loads.
    long long work = 0;
    for (int gi = tid; gi < n_groups; gi += kPlanThreads) {
        const int r = find_group_request(a.req_group_base, a.num_reqs, gi);
        const int mt = gi - a.req_group_base[r];
        const int n = a.qsl[r + 1] - a.qsl[r], L = a.seq_lens[r];
        const int kvb = (tile_kv_end(n, L, a.group, mt) + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE;
        a.group_kvb[gi] = kvb;
        work += (long long)kvb * a.num_kv_heads;
    }
    work = block_sum<long long>(work, s_ll);

    // 3. split length: about target_items items, partials within capacity.
    if (tid == 0) {
        long long s = (work + a.target_items - 1) / max(1LL, a.target_items);
        s = max(s, (long long)kMinSplitBlocks);
        if (a.parts_cap <= 0) s = INT_MAX / 2;
        s_split = (int)min(s, (long long)(INT_MAX / 2));
    }
    __syncthreads();
    while (true) {
        const int split = s_split;
        long long parts = 0;
        for (int gi = tid; gi < n_groups; gi += kPlanThreads) {
            const int ns = (a.group_kvb[gi] + split - 1) / split;
            if (ns > 1) parts += (long long)ns * a.num_kv_heads;
        }
        parts = block_sum<long long>(parts, s_ll);
        if (parts <= a.parts_cap) break;
        if (tid == 0) s_split = split * 2;
        __syncthreads();
    }
    const int split = s_split;

    // 4. items and tile info, chunked scans over groups.
    int item_carry = 0, part_carry = 0;
    for (int base = 0; base < n_groups; base += kPlanThreads) {
        const int gi = base + tid;
        int ns = 0, r = 0, mt = 0, kvb = 0;
        if (gi < n_groups) {
            r = find_group_request(a.req_group_base, a.num_reqs, gi);
            mt = gi - a.req_group_base[r];
            kvb = a.group_kvb[gi];
            ns = max(1, (kvb + split - 1) / split);
        }
        const int n_it = gi < n_groups ? ns * a.num_kv_heads : 0;
        const int n_pt = (gi < n_groups && ns > 1) ? ns * a.num_kv_heads : 0;
        int tot_it, tot_pt;
        const int it0 = item_carry + block_exclusive_scan<int>(n_it, &tot_it, s_i);
        const int pt0 = part_carry + block_exclusive_scan<int>(n_pt, &tot_pt, s_i);
        if (gi < n_groups) {
            const int q0 = a.qsl[r], n = a.qsl[r + 1] - q0, L = a.seq_lens[r];
            const int kv_end = tile_kv_end(n, L, a.group, mt);
            for (int h = 0; h < a.num_kv_heads; ++h) {
                const long long tile = (long long)gi * a.num_kv_heads + h;
                const int pbase = ns > 1 ? pt0 + h * ns : -1;
                a.tile_info[tile] = make_int2(ns, pbase);
                for (int s = 0; s < ns; ++s) {
                    const long long idx = (long long)it0 + (long long)h * ns + s;
                    if (idx >= a.items_cap) { atomicOr(status, PKV_DEV_OVERFLOW); continue; }
                    const int kb0 = s * split;
                    const int kb1 = min(kvb, kb0 + split);
                    WorkItem w;
                    w.a = make_int4(r, mt, h, s);
                    w.b = make_int4(kb0, kb1, ns > 1 ? pbase + s : -1, q0);
                    w.c = make_int4(n, L, kv_end, 0);
                    a.items[idx] = w;
                }
            }
        }
        item_carry += tot_it;
        part_carry += tot_pt;
    }
    if (tid == 0) {
        a.header->n_items = (int)min((long long)item_carry, a.items_cap);
        a.header->split_blocks = split;
        a.header->n_groups = n_groups;
        a.header->n_partials = part_carry;
    }
}

// ---------------------------------------------------------------------------
// decode (split-KV) kernel
// ---------------------------------------------------------------------------

struct DecodeArgs {
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
    const int32_t *block_table;
    int max_blocks_per_req, num_blocks, num_q_heads, num_kv_heads, group;
    float scale_log2;
    const WorkItem *items;
    WsHeader *header;
    float2 *part_ml;
    float *part_o;
};

// Per-item description handed from the producer to the consumers through
// shared memory, next to the item's Q rows.
struct ItemDesc {
    int kb0, kb1, part, n_valid, kv_end, h, pad0, pad1;
    int row_t[kRowsPerTile];
    int row_hq[kRowsPerTile];
    int row_limit[kRowsPerTile];
};

template <int D>
struct DecodeSmem {
    static constexpr int kBoxes = D / 64;                   // 64-column TMA boxes per tile
    static constexpr int kTileBytes = kBoxes * 2048;        // 16 rows x D bf16
    static constexpr int kStageBytes = 2 * kTileBytes;      // K tile + V tile
    static constexpr int kStages = D == 128 ? 8 : 12;
    static constexpr int kQStride = 2 * D + 16;             // padded row: conflict-free ldmatrix
    static constexpr int kQBytes = kRowsPerTile * kQStride;
    static constexpr int kScrStride = D + 8;                // floats per scratch row
    static constexpr int kScrBytes = kConsumerWarps * kRowsPerTile * kScrStride * 4;
    static constexpr int kOffStages = 0;
    static constexpr int kOffQ = kOffStages + kStages * kStageBytes;
    static constexpr int kOffDesc = kOffQ + 2 * kQBytes;
    static constexpr int kOffScr = kOffDesc + 2 * (int)sizeof(ItemDesc);
    static constexpr int kOffML = kOffScr + kScrBytes;
    static constexpr int kOffBar = kOffML + kConsumerWarps * kRowsPerTile * 8;
    static constexpr int kBars = 2 * kStages + 4;
    static constexpr int kBytes = kOffBar + kBars * 8;
    static constexpr int kAlloc = kBytes + 1024;            // slack for 1024-byte alignment
};

template <int D>
__global__ void __launch_bounds__(kDecodeThreads, D == 128 ? 2 : 3)
decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeArgs a) {
    using S = DecodeSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_abort;  // set by any wait that gives up; every later wait returns at once
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::kOffBar);
    uint64_t *full = bar, *empty = bar + S::kStages, *qfull = bar + 2 * S::kStages, *qempty = qfull + 2;
    ItemDesc *desc = reinterpret_cast<ItemDesc *>(smem + S::kOffDesc);
    volatile int *abort = &s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *status = &a.header->status;
    const int n_items = a.header->n_items;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int i = 0; i < S::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 32);
            mbar_init(&qempty[i], kConsumerWarps);
        }
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) tma_prefetch_desc(&kv_map);
        const int Hkv = a.num_kv_heads;
        uint32_t e = 0;  // ring element counter
        int k = 0;       // item counter
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++k) {
            const WorkItem w = a.items[it];
            const int r = w.a.x, mt = w.a.y, h = w.a.z;
            const int kb0 = w.b.x, kb1 = w.b.y, part = w.b.z, q0 = w.b.w;
            const int n = w.c.x, L = w.c.y, kv_end = w.c.z;
            const int qb = k & 1;
            if (!mbar_wait(&qempty[qb], ((k >> 1) & 1) ^ 1, status, abort)) { ok = false; break; }
            // Item description and Q rows for the consumers.
            ItemDesc &d = desc[qb];
            const long long rows = (long long)n * a.group;
            if (lane < kRowsPerTile) {
                const long long rho = (long long)mt * kRowsPerTile + lane;
                const bool valid = rho < rows;
                const int i = valid ? (int)(rho / a.group) : 0;
                const int j = valid ? (int)(rho % a.group) : 0;
                d.row_t[lane] = q0 + i;
                d.row_hq[lane] = h * a.group + j;
                d.row_limit[lane] = valid ? L - n + i : kv_end - 1;
            }
            if (lane == 0) {
                const long long nv = rows - (long long)mt * kRowsPerTile;
                d.kb0 = kb0; d.kb1 = kb1; d.part = part;
                d.n_valid = (int)min(nv, (long long)kRowsPerTile);
                d.kv_end = kv_end; d.h = h;
            }
            uint8_t *qs = smem + S::kOffQ + qb * S::kQBytes;
            constexpr int kChunks = D / 8;
#pragma unroll
            for (int c = lane; c < kRowsPerTile * kChunks; c += 32) {
                const int row = c / kChunks, ch = c % kChunks;
                const long long rho = (long long)mt * kRowsPerTile + row;
                uint4 val = make_uint4(0, 0, 0, 0);
                if (rho < rows) {
                    const int i = (int)(rho / a.group), j = (int)(rho % a.group);
                    const long long t = (long long)q0 + i;
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        a.q + (t * a.num_q_heads + (long long)h * a.group + j) * D);
                    val = __ldg(src + ch);
                }
                *reinterpret_cast<uint4 *>(qs + row * S::kQStride + ch * 16) = val;
            }
            mbar_arrive(&qfull[qb]);

            // K/V block tiles through the ring.
            const int32_t *bt = a.block_table + (long long)r * a.max_blocks_per_req;
            for (int base = kb0; base < kb1 && ok; base += 32) {
                int my_blk = 0;
                if (base + lane < kb1) {
                    my_blk = __ldg(bt + base + lane);
                    if (my_blk < 0 || my_blk >= a.num_blocks) {
                        raise_status(status, PKV_DEV_BAD_BLOCK);
                        my_blk = a.num_blocks;  // outside the tensor map: TMA fills zeros
                    }
                }
                const int cnt = min(32, kb1 - base);
                for (int j = 0; j < cnt; ++j) {
                    const int blk = __shfl_sync(0xffffffffu, my_blk, j);
                    const int stage = e % S::kStages;
                    if (!mbar_wait(&empty[stage], ((e / S::kStages) & 1) ^ 1, status, abort)) { ok = false; break; }
                    if (lane == 0) {
                        uint8_t *st = smem + S::kOffStages + stage * S::kStageBytes;
                        mbar_arrive_expect_tx(&full[stage], S::kStageBytes);
#pragma unroll
                        for (int bx = 0; bx < S::kBoxes; ++bx) {
                            tma_load_3d(st + bx * 2048, &kv_map, bx * 64, h * PKV_BLOCK_SIZE, blk, &full[stage]);
                            tma_load_3d(st + S::kTileBytes + bx * 2048, &kv_map, bx * 64,
                                        (Hkv + h) * PKV_BLOCK_SIZE, blk, &full[stage]);
                        }
                    }
                    __syncwarp();
                    ++e;
                }
            }
        }
        // After a failure, do not leave while copies into this CTA's shared
        // memory are still in flight: wait (bounded) for the last issue of
        // every stage.
        if (!ok && lane == 0) {
            for (uint32_t x = e > (uint32_t)S::kStages ? e - S::kStages : 0; x < e; ++x) {
                const uint32_t stage = x % S::kStages, parity = (x / S::kStages) & 1;
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(&full[stage], parity) && global_timer_ns() - t0 < kWaitTimeoutNs) {
                }
            }
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    const int tid = threadIdx.x;  // 0..127
    const int qrow = lane >> 2;   // fragment rows qrow and qrow + 8
    const int qcol = (lane & 3) * 2;
    float *scr = reinterpret_cast<float *>(smem + S::kOffScr);
    float2 *sml = reinterpret_cast<float2 *>(smem + S::kOffML);
    uint32_t e = 0;
    int k = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++k) {
        const int qb = k & 1;
        // Any failed wait below sets *abort; the warps still meet at both
        // named barriers of this item and then leave together.
        const bool have_q = mbar_wait(&qfull[qb], (k >> 1) & 1, status, abort);
        const ItemDesc &d = desc[qb];
        float o[D / 8][4];
#pragma unroll
        for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

        if (have_q) {
            const int kb0 = d.kb0, kb1 = d.kb1, kv_end = d.kv_end;
            const int lim0 = d.row_limit[qrow], lim1 = d.row_limit[qrow + 8];

            // Q fragments (A operand, 16 rows x D) for the whole item.
            uint32_t qa[D / 16][4];
            {
                const uint32_t qs = smem_u32(smem + S::kOffQ + qb * S::kQBytes);
                const int mi = lane >> 3;
                const int row = ((mi & 1) << 3) + (lane & 7);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int chunk = 2 * kk + (mi >> 1);
                    ldmatrix_x4(qs + row * S::kQStride + chunk * 16, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
                }
            }

            for (int kb = kb0; kb < kb1; ++kb, ++e) {
                if (((kb - kb0) & (kConsumerWarps - 1)) != warp) continue;
                const int stage = e % S::kStages;
                if (!mbar_wait(&full[stage], (e / S::kStages) & 1, status, abort)) break;
                uint8_t *st = smem + S::kOffStages + stage * S::kStageBytes;
                const uint32_t kbase = smem_u32(st), vbase = kbase + S::kTileBytes;
                const int key0 = kb * PKV_BLOCK_SIZE;

                // Rows of V past the tile's last visible key may hold anything
                // (other requests' stale data, NaN); their P is 0, but 0 * NaN
                // is not, so clear them.
                const bool tail = key0 + PKV_BLOCK_SIZE > kv_end;
                if (tail) {
                    const int first = kv_end - key0;  // 1..15
                    for (int c = lane; c < (PKV_BLOCK_SIZE - first) * S::kBoxes * 8; c += 32) {
                        const int row = first + c / (S::kBoxes * 8);
                        const int rem = c % (S::kBoxes * 8);
                        *reinterpret_cast<uint4 *>(st + S::kTileBytes + (rem >> 3) * 2048 + row * 128 +
                                                   (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
                    }
                    __syncwarp();
                }

                // S = Q K^T for 16 keys: two n-tiles of 8 keys.
                float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                {
                    const int mi = lane >> 3;
                    const int key = ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int chunk = 2 * kk + (mi & 1);
                        uint32_t b0, b1, b2, b3;
                        ldmatrix_x4(kbase + (chunk >> 3) * 2048 + swz128(key, chunk & 7), b0, b1, b2, b3);
                        mma_bf16_16816(sc[0], qa[kk], b0, b1);
                        mma_bf16_16816(sc[1], qa[kk], b2, b3);
                    }
                }

                // Scale into the log2 domain, causal mask, online softmax.
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int key = key0 + nt * 8 + qcol + c;
                        const float s0 = key <= lim0 ? sc[nt][c] * a.scale_log2 : -INFINITY;
                        const float s1 = key <= lim1 ? sc[nt][2 + c] * a.scale_log2 : -INFINITY;
                        sc[nt][c] = s0;
                        sc[nt][2 + c] = s1;
                        mx0 = fmaxf(mx0, s0);
                        mx1 = fmaxf(mx1, s1);
                    }
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float base0 = mn0 == -INFINITY ? 0.f : mn0;
                const float base1 = mn1 == -INFINITY ? 0.f : mn1;
                const float al0 = fast_exp2(m0 - base0), al1 = fast_exp2(m1 - base1);
                m0 = mn0;
                m1 = mn1;
                float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        sc[nt][c] = fast_exp2(sc[nt][c] - base0);
                        sc[nt][2 + c] = fast_exp2(sc[nt][2 + c] - base1);
                        ps0 += sc[nt][c];
                        ps1 += sc[nt][2 + c];
                    }
                }
                l0 = l0 * al0 + ps0;
                l1 = l1 * al1 + ps1;
                if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                    for (int i = 0; i < D / 8; ++i) {
                        o[i][0] *= al0; o[i][1] *= al0;
                        o[i][2] *= al1; o[i][3] *= al1;
                    }
                }

                // O += P V: P (16 rows x 16 keys) as the A operand.
                uint32_t pa[4];
                pa[0] = pack_bf16x2(sc[0][0], sc[0][1]);
                pa[1] = pack_bf16x2(sc[0][2], sc[0][3]);
                pa[2] = pack_bf16x2(sc[1][0], sc[1][1]);
                pa[3] = pack_bf16x2(sc[1][2], sc[1][3]);
                {
                    const int mi = lane >> 3;
                    const int key = ((mi & 1) << 3) + (lane & 7);
#pragma unroll
                    for (int dp = 0; dp < D / 16; ++dp) {
                        const int chunk = 2 * dp + (mi >> 1);
                        uint32_t b0, b1, b2, b3;
                        ldmatrix_x4_trans(vbase + (chunk >> 3) * 2048 + swz128(key, chunk & 7), b0, b1, b2, b3);
                        mma_bf16_16816(o[2 * dp], pa, b0, b1);
                        mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    if (tail) fence_proxy_async_smem();
                    mbar_arrive(&empty[stage]);
                }
            }
            // Keep the ring counter in step with the producer if the loop
            // above stopped early (the CTA is aborting then anyway).
        }

        // Combine the four warps' states: each warp's rows -> scratch.
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        {
            float *ws = scr + warp * kRowsPerTile * S::kScrStride;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                const int col = i * 8 + qcol;
                *reinterpret_cast<float2 *>(ws + qrow * S::kScrStride + col) = make_float2(o[i][0], o[i][1]);
                *reinterpret_cast<float2 *>(ws + (qrow + 8) * S::kScrStride + col) = make_float2(o[i][2], o[i][3]);
            }
            if ((lane & 3) == 0) {
                sml[warp * kRowsPerTile + qrow] = make_float2(m0, l0);
                sml[warp * kRowsPerTile + qrow + 8] = make_float2(m1, l1);
            }
        }
        named_barrier_sync(1, kConsumerWarps * 32);
        // No wait happens between the two barriers, so every warp reads the
        // same abort value here.
        const bool aborted = *abort != 0;
        if (!aborted) {
            const int n_valid = d.n_valid, part = d.part;
            constexpr int kC4 = D / 4;
            for (int idx = tid; idx < kRowsPerTile * kC4; idx += kConsumerWarps * 32) {
                const int row = idx / kC4, c4 = idx % kC4;
                if (row >= n_valid) break;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sml[w * kRowsPerTile + row].x);
                float lsum = 0.f;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                if (M != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        const float2 ml = sml[w * kRowsPerTile + row];
                        const float f = fast_exp2(ml.x - M);
                        lsum += ml.y * f;
                        const float4 v = *reinterpret_cast<const float4 *>(
                            scr + (w * kRowsPerTile + row) * S::kScrStride + c4 * 4);
                        acc.x += v.x * f; acc.y += v.y * f; acc.z += v.z * f; acc.w += v.w * f;
                    }
                }
                if (part < 0) {
                    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
                    const long long off = ((long long)d.row_t[row] * a.num_q_heads + d.row_hq[row]) * D + c4 * 4;
                    uint2 pk;
                    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
                    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
                    *reinterpret_cast<uint2 *>(a.out + off) = pk;
                } else {
                    const long long prow = (long long)part * kRowsPerTile + row;
                    *reinterpret_cast<float4 *>(a.part_o + prow * D + c4 * 4) = acc;
                    if (c4 == 0) a.part_ml[prow] = make_float2(M, lsum);
                }
            }
        }
        named_barrier_sync(1, kConsumerWarps * 32);
        if (aborted) return;
        if (lane == 0) mbar_arrive(&qempty[qb]);
    }
}

// ---------------------------------------------------------------------------
// merge of split partials
// ---------------------------------------------------------------------------

struct MergeArgs {
    __nv_bfloat16 *out;
    const int32_t *qsl;
    int num_reqs, num_tokens, num_q_heads, num_kv_heads, group;
    const int32_t *req_group_base;
    const int2 *tile_info;
    const float2 *part_ml;
    const float *part_o;
};

template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const MergeArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row_id = (long long)blockIdx.x * 8 + warp;
    if (row_id >= (long long)a.num_tokens * a.num_q_heads) return;
    const int t = (int)(row_id / a.num_q_heads), hq = (int)(row_id % a.num_q_heads);
    int lo = 0, hi = a.num_reqs;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a.qsl[mid] <= t) lo = mid; else hi = mid;
    }
    const int r = lo, q0 = a.qsl[r];
    if (!(q0 <= t && t < a.qsl[r + 1])) return;
    const long long rho = (long long)(t - q0) * a.group + hq % a.group;
    const int mt = (int)(rho / kRowsPerTile), row = (int)(rho % kRowsPerTile);
    const int g0 = a.req_group_base[r];
    if (mt >= a.req_group_base[r + 1] - g0) return;
    const int2 info = a.tile_info[(long long)(g0 + mt) * a.num_kv_heads + hq / a.group];
    const int ns = info.x, pb = info.y;
    if (ns <= 1) return;
    float M = -INFINITY;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, a.part_ml[(long long)(pb + s) * kRowsPerTile + row].x);
    constexpr int kPer = D / 32;
    float acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
    float lsum = 0.f;
    for (int s = 0; s < ns; ++s) {
        const long long prow = (long long)(pb + s) * kRowsPerTile + row;
        const float2 ml = a.part_ml[prow];
        const float f = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - M);
        lsum += ml.y * f;
        const float *src = a.part_o + prow * D + lane * kPer;
        if constexpr (kPer == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(src);
            acc[0] += v.x * f; acc[1] += v.y * f; acc[2] += v.z * f; acc[3] += v.w * f;
        } else {
            const float2 v = *reinterpret_cast<const float2 *>(src);
            acc[0] += v.x * f; acc[1] += v.y * f;
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    __nv_bfloat16 *dst = a.out + ((long long)t * a.num_q_heads + hq) * D + lane * kPer;
    if constexpr (kPer == 4) {
        uint2 pk;
        pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2 *>(dst) = pk;
    } else {
        *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

struct DeviceInfo {
    int sm_count = 0;
    int ctas_per_sm[2] = {0, 0};  // decode kernel, D = 64 / 128
    bool ready = false;
};

std::mutex g_mu;
DeviceInfo g_dev[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

template <int D>
int decode_occupancy() {
    using S = DecodeSmem<D>;
    if (cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc) !=
        cudaSuccess)
        return -1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<D>, kDecodeThreads, S::kAlloc) !=
        cudaSuccess)
        return -1;
    return n;
}

int device_info(DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_E_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &di = g_dev[dev];
    if (!di.ready) {
        if (cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PKV_E_CUDA;
        di.ctas_per_sm[0] = decode_occupancy<64>();
        di.ctas_per_sm[1] = decode_occupancy<128>();
        if (di.ctas_per_sm[0] <= 0 || di.ctas_per_sm[1] <= 0) return PKV_E_CUDA;
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return PKV_E_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        di.ready = true;
    }
    *out = &di;
    return PKV_OK;
}

// Default split-KV partial capacity: enough records for kItemsPerCta items
// per CTA of a full persistent grid.
long long default_parts_cap(int sm_count) { return (long long)sm_count * 4 * kItemsPerCta; }

int encode_kv_map(CUtensorMap *map, const void *kv_cache, const pkv_cache_desc &d) {
    const cuuint64_t rows_per_block = 2ull * d.num_kv_heads * PKV_BLOCK_SIZE;
    cuuint64_t dims[3] = {(cuuint64_t)d.head_size, rows_per_block, (cuuint64_t)d.num_blocks};
    cuuint64_t strides[2] = {(cuuint64_t)d.head_size * 2, rows_per_block * d.head_size * 2};
    cuuint32_t box[3] = {64, PKV_BLOCK_SIZE, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult res = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(kv_cache), dims, strides,
                            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? PKV_OK : PKV_E_CUDA;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" PKV_API int paged_attention_workspace_bytes(int32_t max_num_reqs, int32_t max_num_tokens,
                                                       int32_t num_q_heads, const pkv_cache_desc *desc,
                                                       size_t *bytes) {
    if (!desc || !bytes) return PKV_E_NULL;
    int rc = check_cache_desc(*desc, /*attention=*/true);
    if (rc) return rc;
    if (max_num_reqs < 0 || max_num_tokens < 0) return PKV_E_DIMS;
    if (num_q_heads <= 0 || num_q_heads % desc->num_kv_heads != 0) return PKV_E_GQA;
    DeviceInfo *di = nullptr;
    rc = device_info(&di);
    if (rc) return rc;
    const WsLayout L = ws_layout(max_num_reqs, max_num_tokens, num_q_heads, desc->num_kv_heads, desc->head_size,
                                 default_parts_cap(di->sm_count));
    *bytes = L.total;
    return PKV_OK;
}

extern "C" PKV_API int paged_attention_min_workspace_bytes(int32_t max_num_reqs, int32_t max_num_tokens,
                                                           int32_t num_q_heads, const pkv_cache_desc *desc,
                                                           size_t *bytes) {
    if (!desc || !bytes) return PKV_E_NULL;
    int rc = check_cache_desc(*desc, /*attention=*/true);
    if (rc) return rc;
    if (max_num_reqs < 0 || max_num_tokens < 0) return PKV_E_DIMS;
    if (num_q_heads <= 0 || num_q_heads % desc->num_kv_heads != 0) return PKV_E_GQA;
    *bytes = ws_layout(max_num_reqs, max_num_tokens, num_q_heads, desc->num_kv_heads, desc->head_size, 0).total;
    return PKV_OK;
}

namespace pkv {
namespace {

void record(void *const *events, int i, cudaStream_t st) {
    if (events && events[i]) cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st);
}

int attention_impl(const void *q, int32_t num_tokens, int32_t num_q_heads, const void *kv_cache,
                   const pkv_cache_desc *desc, const int32_t *block_table, int32_t num_reqs,
                   int32_t max_blocks_per_req, const int32_t *seq_lens, const int32_t *query_start_loc, float scale,
                   void *out, void *workspace, size_t workspace_bytes, void *stream, void *const *events) {
    if (!desc) return PKV_E_NULL;
    int rc = check_cache_desc(*desc, /*attention=*/true);
    if (rc) return rc;
    if (num_tokens < 0 || num_reqs < 0 || max_blocks_per_req < 0) return PKV_E_DIMS;
    if (num_q_heads <= 0 || num_q_heads % desc->num_kv_heads != 0) return PKV_E_GQA;
    if (num_tokens == 0) return PKV_OK;
    if (num_reqs == 0 || max_blocks_per_req == 0) return PKV_E_DIMS;
    if (!q || !kv_cache || !block_table || !seq_lens || !query_start_loc || !out || !workspace) return PKV_E_NULL;
    if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(workspace, 256) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(query_start_loc, 4))
        return PKV_E_ALIGN;
    if (!(scale == scale)) return PKV_E_DIMS;

    const int D = desc->head_size, Hkv = desc->num_kv_heads;
    const WsLayout base = ws_layout(num_reqs, num_tokens, num_q_heads, Hkv, D, 0);
    if (workspace_bytes < base.total) return PKV_E_WORKSPACE;

    DeviceInfo *di = nullptr;
    rc = device_info(&di);
    if (rc) return rc;
    // Largest partial capacity (up to the default) that fits the workspace.
    long long parts_cap = default_parts_cap(di->sm_count);
    const size_t per_part = sizeof(WorkItem) + kRowsPerTile * (sizeof(float2) + sizeof(float) * D);
    const size_t spare = workspace_bytes - base.total;
    const long long fit = spare > 1024 ? (long long)((spare - 1024) / per_part) : 0;
    if (fit < parts_cap) parts_cap = fit;
    const WsLayout L = ws_layout(num_reqs, num_tokens, num_q_heads, Hkv, D, parts_cap);
    if (L.total > workspace_bytes) return PKV_E_WORKSPACE;

    CUtensorMap kv_map;
    rc = encode_kv_map(&kv_map, kv_cache, *desc);
    if (rc) return rc;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    WsHeader *header = reinterpret_cast<WsHeader *>(ws);
    const int ctas = di->sm_count * di->ctas_per_sm[D == 128 ? 1 : 0];

    PlanArgs pa;
    pa.qsl = query_start_loc;
    pa.seq_lens = seq_lens;
    pa.num_reqs = num_reqs;
    pa.num_tokens = num_tokens;
    pa.max_blocks_per_req = max_blocks_per_req;
    pa.group = num_q_heads / Hkv;
    pa.num_kv_heads = Hkv;
    pa.target_items = (long long)ctas * kItemsPerCta;
    pa.parts_cap = L.parts_cap;
    pa.groups_cap = L.groups_cap;
    pa.items_cap = L.items_cap;
    pa.header = header;
    pa.req_group_base = reinterpret_cast<int32_t *>(ws + L.req_group_base);
    pa.group_kvb = reinterpret_cast<int32_t *>(ws + L.group_kvb);
    pa.tile_info = reinterpret_cast<int2 *>(ws + L.tile_info);
    pa.items = reinterpret_cast<WorkItem *>(ws + L.items);
    record(events, 0, st);
    plan_kernel<<<1, kPlanThreads, 0, st>>>(pa);

    DecodeArgs da;
    da.q = static_cast<const __nv_bfloat16 *>(q);
    da.out = static_cast<__nv_bfloat16 *>(out);
    da.block_table = block_table;
    da.max_blocks_per_req = max_blocks_per_req;
    da.num_blocks = desc->num_blocks;
    da.num_q_heads = num_q_heads;
    da.num_kv_heads = Hkv;
    da.group = num_q_heads / Hkv;
    da.scale_log2 = scale * kLog2e;
    da.items = pa.items;
    da.header = header;
    da.part_ml = reinterpret_cast<float2 *>(ws + L.part_ml);
    da.part_o = reinterpret_cast<float *>(ws + L.part_o);

    MergeArgs ma;
    ma.out = da.out;
    ma.qsl = query_start_loc;
    ma.num_reqs = num_reqs;
    ma.num_tokens = num_tokens;
    ma.num_q_heads = num_q_heads;
    ma.num_kv_heads = Hkv;
    ma.group = da.group;
    ma.req_group_base = pa.req_group_base;
    ma.tile_info = pa.tile_info;
    ma.part_ml = da.part_ml;
    ma.part_o = da.part_o;
    const long long rows = (long long)num_tokens * num_q_heads;
    const unsigned merge_blocks = (unsigned)((rows + 7) / 8);

    record(events, 1, st);
    if (D == 128) decode_kernel<128><<<ctas, kDecodeThreads, DecodeSmem<128>::kAlloc, st>>>(kv_map, da);
    else decode_kernel<64><<<ctas, kDecodeThreads, DecodeSmem<64>::kAlloc, st>>>(kv_map, da);
    record(events, 2, st);
    if (D == 128) merge_kernel<128><<<merge_blocks, 256, 0, st>>>(ma);
    else merge_kernel<64><<<merge_blocks, 256, 0, st>>>(ma);
    record(events, 3, st);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_E_CUDA;
}

}  // namespace
}  // namespace pkv

extern "C" PKV_API int paged_attention(const void *q, int32_t num_tokens, int32_t num_q_heads, const void *kv_cache,
                                       const pkv_cache_desc *desc, const int32_t *block_table, int32_t num_reqs,
                                       int32_t max_blocks_per_req, const int32_t *seq_lens,
                                       const int32_t *query_start_loc, float scale, void *out, void *workspace,
                                       size_t workspace_bytes, void *stream) {
    return attention_impl(q, num_tokens, num_q_heads, kv_cache, desc, block_table, num_reqs, max_blocks_per_req,
                          seq_lens, query_start_loc, scale, out, workspace, workspace_bytes, stream, nullptr);
}

extern "C" PKV_API int paged_attention_timed(const void *q, int32_t num_tokens, int32_t num_q_heads,
                                             const void *kv_cache, const pkv_cache_desc *desc,
                                             const int32_t *block_table, int32_t num_reqs,
                                             int32_t max_blocks_per_req, const int32_t *seq_lens,
                                             const int32_t *query_start_loc, float scale, void *out, void *workspace,
                                             size_t workspace_bytes, void *stream, void *const *events) {
    return attention_impl(q, num_tokens, num_q_heads, kv_cache, desc, block_table, num_reqs, max_blocks_per_req,
                          seq_lens, query_start_loc, scale, out, workspace, workspace_bytes, stream, events);
}

// ---------------------------------------------------------------------------
// Allocation-free variant
// ---------------------------------------------------------------------------
// Some callers cannot allocate device memory when they call attention: an
// engine that, after its profiling pass, has handed almost all free device
// memory to the KV pool; a plugin whose host framework owns the device
// memory and offers it no allocator; a latency-critical loop where
// cudaMalloc's implicit synchronisation is not acceptable. For them the
// work list and split partials live in this fixed array instead of a
// caller-provided workspace. Every GPU that loads this library holds the
// array until the process exits.

static constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

namespace pkv {
namespace {

std::mutex g_scratch_mu;
void *g_scratch_addr[64] = {};

// Device address of g_static_scratch on the current device. In host code the
// symbol itself is only a host-side stand-in, so the address is looked up
// once per device with that device current.
int static_scratch_address(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_E_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return PKV_E_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" PKV_API int paged_attention_static(const void *q, int32_t num_tokens, int32_t num_q_heads,
                                              const void *kv_cache, const pkv_cache_desc *desc,
                                              const int32_t *block_table, int32_t num_reqs,
                                              int32_t max_blocks_per_req, const int32_t *seq_lens,
                                              const int32_t *query_start_loc, float scale, void *out, void *stream) {
    if (!desc) return PKV_E_NULL;
    void *scratch = nullptr;
    const int rc = static_scratch_address(&scratch);
    if (rc) return rc;
    return attention_impl(q, num_tokens, num_q_heads, kv_cache, desc, block_table, num_reqs, max_blocks_per_req,
                          seq_lens, query_start_loc, scale, out, scratch, kStaticScratchBytes, stream, nullptr);
}
