// Paged attention over a flattened ragged batch ("Inside vLLM", page 1, "Run
// forward pass" step 3: one super sequence, each sequence attending only to
// its own tokens; decode and chunked-prefill requests mixed in one step).
//
// Up to three launches on the caller's stream:
//   plan_kernel    one CTA turns query_start_loc / seq_lens into a work list
//                  (attention_plan.cuh): it picks the split-KV length so the
//                  persistent grid gets ~kItemsPerCta items per CTA and lists
//                  the items longest first;
//   chunk_kernel   (attention_chunk.cu) the 128-row tensor-core tiles of
//                  requests with many new tokens, on a share of the SMs
//                  beside the next kernel; skipped when no request can fill
//                  a tile;
//   decode_kernel  persistent, warp-specialised. One producer warp takes
//                  items from an atomic counter, bulk-copies each item's Q
//                  rows and gathers each (block, kv head)'s K and V rows (16
//                  x D each, contiguous in the pool) with one TMA box into a
//                  shared-memory ring; four consumer warps run S = Q K^T and
//                  O += P V on
//                  bf16 mma.sync tensor-core tiles with an fp32 online
//                  softmax (exp2 domain), combine their states in shared
//                  memory, and either write the output or a split partial;
//                  the CTA finishing a tile's last split merges its partials.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attention_chunk.h"
#include "attention_plan.cuh"
#include "pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
// One CTA builds the work list. 512 threads: its phases are short and
// separated by block-wide barriers and scans, which cost less with fewer
// warps (same-box steps: 2 requests 10.3 -> 10.0 us, 64 TinyLlama requests
// 30.4 -> 30.1 us against 1024 threads; 256 threads slowed the 256-request
// Llama-3-8B step by 0.3 %).
constexpr int kPlanThreads = 512;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// plan
// ---------------------------------------------------------------------------

struct PlanArgs {
    const int32_t *qsl;
    const int32_t *seq_lens;
    int num_reqs, num_tokens, max_blocks_per_req, group, num_kv_heads;
    int block_bytes_kv;  // K + V bytes of one (block, kv head): 2 * 16 * D * 2
    int chunk_ok;        // the tcgen05 chunk kernel can take this shape (128 % g == 0)
    int sm_count;
    float chunk_sm_us_per_tile;  // SM-microseconds one 128 x 128 chunk tile step costs
    float decode_bytes_per_us;   // split-KV streaming rate of the whole GPU
    long long target_items, part_rows_cap, groups_cap, items_cap, chunk_items_cap;
    WsHeader *header;
    int32_t *req_cache;  // kReqCacheArrays * (num_reqs + 1) ints, when the batch has too many requests for shared memory
    int32_t *group_req;
    int32_t *group_kvb;
    int32_t *tile_counter;
    WorkItem *items;
    GroupRec *group_rec;
    ChunkItem *chunk_items;
    const int32_t *block_table;
    int4 *prefix_map;  // per global row T_r * g + j: {slot-0 partial row at kv head 0, row stride per kv head, group, arrivals}
};

// Exclusive scan over the threads of the block; *total gets the sum.
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

// Device-scope atomic add with acquire-release ordering; returns the old value.
__device__ __forceinline__ int atom_add_acq_rel(int32_t *p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ int tile_rows(int n, int g, int mt) {
    return (int)min((long long)kRowsPerTile, (long long)n * g - (long long)mt * kRowsPerTile);
}

// Last r in [0, num_reqs) with base[r] <= gi (requests without tiles are skipped).
__device__ __forceinline__ int find_group_request(const int32_t *base, int num_reqs, int gi) {
    int lo = 0, hi = num_reqs;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (base[mid] <= gi) lo = mid; else hi = mid;
    }
    return lo;
}

// Size bucket of an item of `size` blocks: 0 for a full split, then 1..8
// from longest to shortest.
__device__ __forceinline__ int size_bucket(int size, int split) {
    if (size >= split) return 0;
    return kSizeBuckets - 1 - min(kSizeBuckets - 2, (int)((long long)size * (kSizeBuckets - 1) / split));
}

// All 32 lanes call this together; each lane with key >= 0 claims `per`
// consecutive slots of counters[key] and gets the first one. Lanes of the
// warp with the same key share one shared-memory atomic.
__device__ __forceinline__ int warp_claim(int key, int per, int *counters) {
    const int lane = threadIdx.x & 31;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int leader = __ffs(peers) - 1;
    int base = 0;
    if (lane == leader && key >= 0) base = atomicAdd(&counters[key], per * __popc(peers));
    base = __shfl_sync(0xffffffffu, base, leader);
    return base + per * __popc(peers & ((1u << lane) - 1u));
}

// Smallest j < pcap with table[r][j] != table[0][j] over this thread's
// share of the pairs (r >= 1, j), INT_MAX if none; eight independent loads
// per pass.
template <typename I>
__device__ __forceinline__ int first_table_diff(const int32_t *bt0, long long mbr, I total, int pcap) {
    int first = INT_MAX;
    for (I e0 = threadIdx.x; e0 < total; e0 += (I)8 * blockDim.x) {
        int x[8], y[8], jj[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const I e = e0 + (I)k * blockDim.x;
            x[k] = y[k] = 0;
            jj[k] = INT_MAX;
            if (e < total) {
                const I rr = e / pcap;
                const int j = (int)(e - rr * pcap);
                x[k] = __ldg(bt0 + (long long)(rr + 1) * mbr + j);
                y[k] = __ldg(bt0 + j);
                jj[k] = j;
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (x[k] != y[k]) first = min(first, jj[k]);
    }
    return first;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
    // Dynamic shared memory: the per-request tables when the batch has at
    // most kPlanSmemReqs requests, then the per-group tables when there are
    // at most kPlanSmemGroups decode groups; else those live in the workspace.
    extern __shared__ int32_t s_dyn[];
    __shared__ long long s_ll[32];
    __shared__ unsigned long long s_ull[32];
    __shared__ int s_split, s_kvmax, s_full_total, s_full_count, s_n_items, s_n_chunk_items;
    __shared__ int s_pcap, s_pfx, s_cas_ok;  // shared-prefix pass: cap, blocks found, still possible
    __shared__ int4 s_place[kPlanThreads];  // per group of a chunk: first full-split item, first tail item, splits
    __shared__ int s_bucket_count[kSizeBuckets], s_bucket_base[kSizeBuckets], s_bucket_cursor[kSizeBuckets];
    __shared__ int s_cbucket_count[kSizeBuckets], s_cbucket_base[kSizeBuckets], s_cbucket_cursor[kSizeBuckets];
    __shared__ int s_status;  // status bits found before the workspace may be written
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    const int R = a.num_reqs, Hkv = a.num_kv_heads, g = a.group;
    const int stride = R + 1;
    const bool req_smem = R <= kPlanSmemReqs;
    int32_t *cache = req_smem ? s_dyn : a.req_cache;
    int32_t *req_n = cache, *req_L = cache + stride, *req_q0 = cache + 2 * stride, *req_g = cache + 3 * stride;
    int32_t *req_c = cache + 4 * stride;  // first chunk tile of each request
    int32_t *grp_req = a.group_req, *grp_kvb = a.group_kvb;
    // With every per-request and per-group table in shared memory, steps 1-3
    // only read this call's metadata (query_start_loc, seq_lens,
    // block_table, complete before the call is enqueued) and write shared
    // memory, so they overlap the previous kernel; the workspace (still read
    // by the previous call's attention kernels) is written only after
    // pdl_wait.
    const bool early = req_smem && a.groups_cap <= kPlanSmemGroups;
    if (early) {
        grp_req = s_dyn + kReqCacheArrays * stride;
        grp_kvb = grp_req + a.groups_cap;
    } else {
        pdl_wait();
    }
    int32_t *status = early ? &s_status : &a.header->status;

    if (tid == 0) {
        s_status = 0;
        if (!early) {
            a.header->status = 0;
            a.header->next_item = 0;
            a.header->next_chunk_item = 0;
            a.header->diag = 0;
        }
        s_kvmax = 0;
        s_pcap = kCascadeMaxBlocks;
        s_cas_ok = R >= kCascadeMinReqs ? 1 : 0;
    }
    if (tid < kSizeBuckets) {
        s_cbucket_count[tid] = 0;
        s_cbucket_cursor[tid] = 0;
        s_bucket_cursor[tid] = 0;
    }
    __syncthreads();

    // 1. validate requests, cache (n, L, q0), tiles per request. Requests
    // with at least kChunkRows query rows go to the chunk kernel. One scan
    // carries both tile counts (decode tiles low, chunk tiles high).
    long long carry = 0;
    for (int base = 0; base < R; base += kPlanThreads) {
        const int r = base + tid;
        unsigned long long tiles = 0;
        if (r < R) {
            const int q0 = a.qsl[r], q1 = a.qsl[r + 1], L = a.seq_lens[r];
            // block 0 of every table against request 0's (the shared-prefix test)
            if (r > 0 && __ldg(a.block_table + (long long)r * a.max_blocks_per_req) != __ldg(a.block_table))
                s_cas_ok = 0;
            if ((r == 0 && q0 != 0) || (r == R - 1 && q1 != a.num_tokens)) {
                atomicOr(status, PKV_DEV_BAD_QSL);
                s_cas_ok = 0;  // some token would belong to no request
            }
            const int n = q1 - q0;
            bool ok = false;
            if (n < 0 || q0 < 0 || q1 > a.num_tokens) {
                atomicOr(status, PKV_DEV_BAD_QSL);
            } else if (n > L || (long long)L > (long long)a.max_blocks_per_req * PKV_BLOCK_SIZE) {
                atomicOr(status, PKV_DEV_BAD_LEN);
            } else {
                ok = true;
                const long long rows = (long long)n * g;
                if (a.chunk_ok && rows >= kChunkRows) {
                    tiles = (unsigned long long)((rows + kChunkRows - 1) / kChunkRows) << 32;
                    atomicMax(&s_kvmax, L);
                    s_cas_ok = 0;  // the shared-prefix pass covers split-KV rows only
                } else {
                    tiles = (unsigned long long)((rows + kRowsPerTile - 1) / kRowsPerTile);
                }
                // shared blocks must hold only keys every query row sees
                atomicMin(&s_pcap, (L - n) / PKV_BLOCK_SIZE);
            }
            if (!ok) s_cas_ok = 0;
            req_n[r] = ok ? n : 0;
            req_L[r] = L;
            req_q0[r] = q0;
        }
        unsigned long long total;
        const unsigned long long ex = block_exclusive_scan<unsigned long long>(tiles, &total, s_ull);
        const unsigned long long c = (unsigned long long)carry + ex;
        if (r < R) {
            req_g[r] = (int)(c & 0xffffffffu);
            req_c[r] = (int)(c >> 32);
        }
        carry += (long long)total;
    }
    int n_groups = (int)(carry & 0xffffffff), n_cgroups = (int)((unsigned long long)carry >> 32);
    if (n_groups > a.groups_cap || (long long)n_cgroups * Hkv > a.chunk_items_cap) {
        // Only overlapping (invalid) query_start_loc ranges get here: keep
        // every table index in bounds.
        if (tid == 0) atomicOr(status, PKV_DEV_OVERFLOW);
        n_groups = (int)min((long long)n_groups, a.groups_cap);
        n_cgroups = (int)min((long long)n_cgroups, a.chunk_items_cap / Hkv);
        __syncthreads();
        for (int r = tid; r < R; r += kPlanThreads) {
            req_g[r] = min(req_g[r], n_groups);
            req_c[r] = min(req_c[r], n_cgroups);
        }
    }
    if (tid == 0) {
        req_g[R] = n_groups;
        req_c[R] = n_cgroups;
        s_pfx = (s_cas_ok && s_pcap >= kCascadeMinBlocks) ? s_pcap : 0;
    }
    __syncthreads();

    // 1b. shared prefix: the leading block ids every table has in common.
    if (s_pfx > 0) {
        const int pcap = s_pfx;
        const int32_t *bt0 = a.block_table;
        const long long mbr = a.max_blocks_per_req;
        __syncthreads();  // every thread has read pcap before any lowers s_pfx
        const long long total = (long long)(R - 1) * pcap;
        const bool small = total <= (long long)INT_MAX - 16LL * kPlanThreads;  // int indexes cannot wrap
        const int first_diff = small ? first_table_diff<int>(bt0, mbr, (int)total, pcap)
                                     : first_table_diff<long long>(bt0, mbr, total, pcap);
        if (first_diff != INT_MAX) atomicMin(&s_pfx, first_diff);
        __syncthreads();
        if (tid == 0 && s_pfx < kCascadeMinBlocks) s_pfx = 0;
        __syncthreads();
    }
    const int P0 = s_pfx;

    // 2. keys per decode group, total work in block loads; chunk buckets.
    long long work = 0;
    for (int gi = tid; gi < n_groups; gi += kPlanThreads) {
        const int r = find_group_request(req_g, R, gi);
        const int mt = gi - req_g[r];
        const int kvb = (tile_kv_end(req_n[r], req_L[r], g, mt) + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE;
        grp_req[gi] = r;
        grp_kvb[gi] = kvb;
        work += (long long)(kvb - P0) * Hkv;
    }
    if (tid == 0 && P0 > 0)  // the prefix tiles
        work += ((long long)a.num_tokens * g + kRowsPerTile - 1) / kRowsPerTile * Hkv * P0;
    const int kvmax = s_kvmax;
    auto chunk_kv_end = [&](int r, int mt) {  // keys seen by the tile's last row
        const long long last_row = min((long long)req_n[r] * g - 1, (long long)mt * kChunkRows + kChunkRows - 1);
        return req_L[r] - req_n[r] + (int)(last_row / g) + 1;
    };
    auto chunk_bucket = [&](int kv_end) {  // longest first
        return min(kSizeBuckets - 1, (int)((long long)(kvmax - kv_end) * (kSizeBuckets - 1) / (kvmax + 1)));
    };
    for (int base = 0; base < n_cgroups; base += kPlanThreads) {
        const int gi = base + tid;
        int key = -1;
        if (gi < n_cgroups) {
            const int r = find_group_request(req_c, R, gi);
            key = chunk_bucket(chunk_kv_end(r, gi - req_c[r]));
        }
        warp_claim(key, Hkv, s_cbucket_count);
    }
    work = block_sum<long long>(work, s_ll);  // (its barriers also publish the group tables)

    // 3. split length: about target_items items, partial rows within
    // capacity; the same pass counts items per size bucket.
    if (tid == 0) {
        long long sp = (work + a.target_items - 1) / max(1LL, a.target_items);
        sp = max(sp, (long long)kMinSplitBlocks);
        sp = max(sp, (long long)(kMinItemBytes / a.block_bytes_kv));
        if (a.part_rows_cap <= 0) sp = INT_MAX / 2;
        s_split = (int)min(sp, (long long)(INT_MAX / 2));
    }
    // With a shared prefix every tile also gets partial slot 0 for the
    // prefix pass, so it always takes the partial path; its splits cover
    // only the blocks after the prefix. If the partial rows cannot fit even
    // unsplit, the prefix pass is dropped.
    while (true) {
        if (tid < kSizeBuckets) s_bucket_count[tid] = 0;
        if (tid == 0) s_full_count = 0;
        __syncthreads();
        const int split = s_split, Pl = s_pfx;
        long long rows = 0;
        for (int base = 0; base < n_groups; base += kPlanThreads) {
            const int gi = base + tid;
            int full = 0, tail_key = -1;
            if (gi < n_groups) {
                const int sb = grp_kvb[gi] - Pl;
                const int ns = max(1, (sb + split - 1) / split);
                const int slots = ns + (Pl > 0 ? 1 : 0);
                if (slots > 1) {
                    const int r = grp_req[gi];
                    rows += (long long)slots * Hkv * tile_rows(req_n[r], g, gi - req_g[r]);
                }
                full = (ns - 1) * Hkv;
                tail_key = size_bucket(sb - (ns - 1) * split, split);
            }
            const int full_warp = __reduce_add_sync(0xffffffffu, full);
            if ((tid & 31) == 0 && full_warp) {
                atomicAdd(&s_bucket_count[0], full_warp);
                atomicAdd(&s_full_count, full_warp);
            }
            warp_claim(tail_key, Hkv, s_bucket_count);
        }
        rows = block_sum<long long>(rows, s_ll);
        if (rows <= a.part_rows_cap) break;
        if (tid == 0) {
            if (split < INT_MAX / 2) s_split = split > INT_MAX / 4 ? INT_MAX / 2 : split * 2;
            else s_pfx = 0;  // cannot happen without a prefix: unsplit tiles need no partial rows
        }
    }
    const int split = s_split;
    const int P = s_pfx;
    if (tid == 0) {
        s_full_total = s_full_count;
        s_bucket_cursor[0] = 0;
        int acc = 0, cacc = 0;
        for (int b = 0; b < kSizeBuckets; ++b) {
            s_bucket_base[b] = acc;
            acc += s_bucket_count[b];
            s_cbucket_base[b] = cacc;
            cacc += s_cbucket_count[b];
        }
        s_n_items = acc;
        s_n_chunk_items = cacc;
    }
    __syncthreads();

    // 4. partial-row bases (chunked scan over groups) and the decode items.
    // Per chunk of kPlanThreads groups (thread tid = group base + tid): the
    // scan, the items' places and the group record, in registers and shared
    // memory only (compute4); then the workspace writes (write4). When every
    // group fits in one chunk and the tables live in shared memory, compute4
    // runs before pdl_wait, so that after the previous kernel only the
    // writes stand between it and the attention kernel.
    struct Step4 {
        GroupRec rec;
        long long grow0;
        int row0, tot_rows, valid;
    };
    int row_carry = 0, full_carry = 0;
    auto compute4 = [&](int base) {
        Step4 c;
        const int gi = base + tid;
        int ns = 0, r = 0, mt = 0, kvb = 0, nv = 0;
        int slots = 0;
        if (gi < n_groups) {
            r = grp_req[gi];
            mt = gi - req_g[r];
            kvb = grp_kvb[gi];
            ns = max(1, (kvb - P + split - 1) / split);
            slots = ns + (P > 0 ? 1 : 0);
            nv = tile_rows(req_n[r], g, mt);
        }
        const int n_rows = (gi < n_groups && slots > 1) ? slots * Hkv * nv : 0;
        const int full_cnt = gi < n_groups ? (ns - 1) * Hkv : 0;
        // One scan carries the partial rows (low half) and the full-size
        // split items (high half); both totals are within int range once the
        // split length fits the capacities.
        unsigned long long tot;
        const unsigned long long ex = block_exclusive_scan<unsigned long long>(
            ((unsigned long long)full_cnt << 32) | (unsigned)n_rows, &tot, s_ull);
        c.row0 = row_carry + (int)(ex & 0xffffffffu);
        c.tot_rows = (int)(tot & 0xffffffffu);
        const int full0 = s_bucket_base[0] + full_carry + (int)(ex >> 32);
        full_carry += (int)(tot >> 32);
        const int tail_b = gi < n_groups ? size_bucket(kvb - P - (ns - 1) * split, split) : -1;
        // tail items of bucket 0 come after every full-size split
        const int tail0 = (tail_b > 0 ? s_bucket_base[tail_b] : s_bucket_base[0] + s_full_total) +
                          warp_claim(tail_b, Hkv, s_bucket_cursor);
        c.valid = gi < n_groups;
        c.grow0 = 0;
        if (c.valid) {
            const int n = req_n[r], L = req_L[r], q0 = req_q0[r];
            c.rec.a = make_int4(r, mt, q0, n);
            c.rec.b = make_int4(L, tile_kv_end(n, L, g, mt), kvb, nv);
            // arrivals: the splits, plus the prefix tiles over its rows
            c.grow0 = (long long)q0 * g + (long long)mt * kRowsPerTile;
            const int arrivals =
                ns + (P > 0 ? (int)((c.grow0 + nv - 1) / kRowsPerTile - c.grow0 / kRowsPerTile) + 1 : 0);
            c.rec.c = make_int4(ns, slots > 1 ? c.row0 : -1, slots, arrivals);
            s_place[tid] = make_int4(full0, tail0, ns, slots);
        }
        return c;
    };
    // Needs every thread's s_place of this chunk published (a barrier after
    // compute4).
    auto write4 = [&](int base, const Step4 &c) {
        const int gi = base + tid;
        if (c.valid) {
            a.group_rec[gi] = c.rec;
            if (P > 0) {  // the prefix-tile view of this group's rows
                int4 *m = a.prefix_map + c.grow0;
                const int nv = c.rec.b.w, slots = c.rec.c.z, arrivals = c.rec.c.w;
                for (int row = 0; row < nv; ++row) m[row] = make_int4(c.row0 + row, slots * nv, gi, arrivals);
            }
        }
        // Items of this chunk of groups, one (group, kv head) pair per thread.
        const int chunk_groups = min(kPlanThreads, n_groups - base);
        for (int p = tid; p < chunk_groups * Hkv; p += kPlanThreads) {
            const int lg = p / Hkv, h = p - lg * Hkv;
            const int4 pl = s_place[lg];
            const int gq = base + lg, ns_g = pl.z;
            if (pl.w > 1) a.tile_counter[gq * Hkv + h] = 0;
            for (int s = 0; s < ns_g; ++s) {
                const long long idx = s < ns_g - 1 ? (long long)pl.x + h * (ns_g - 1) + s : (long long)pl.y + h;
                if (idx < a.items_cap) a.items[idx].v = make_int4(gq, h, s, grp_req[gq]);
            }
        }
    };
    const bool early4 = early && n_groups <= kPlanThreads;
    Step4 c4{};
    if (early4) {
        c4 = compute4(0);
        __syncthreads();
    }
    if (early) {
        pdl_wait();
        if (tid == 0) {
            a.header->status = s_status;
            a.header->next_item = 0;
            a.header->next_chunk_item = 0;
            a.header->diag = 0;
        }
        status = &a.header->status;
    }
    if (tid == 0) {
        const int acc = s_n_items, cacc = s_n_chunk_items;
        a.header->n_items = (int)min((long long)acc, a.items_cap);
        if (acc > a.items_cap) atomicOr(status, PKV_DEV_OVERFLOW);
        a.header->n_chunk_items = cacc;
        a.header->split_blocks = split;
        a.header->n_groups = n_groups;
        a.header->cascade_blocks = P;
        a.header->n_prefix_items =
            P > 0 ? (int)(((long long)a.num_tokens * g + kRowsPerTile - 1) / kRowsPerTile) * Hkv : 0;
    }
    if (early4) {
        write4(0, c4);
        row_carry = c4.tot_rows;
    } else {
        __syncthreads();
        for (int base = 0; base < n_groups; base += kPlanThreads) {
            const Step4 c = compute4(base);
            __syncthreads();
            write4(base, c);
            __syncthreads();
            row_carry += c.tot_rows;
        }
    }
    if (tid == 0) a.header->n_partial_rows = row_carry;

    // 5. chunk items, longest first.
    long long csteps = 0;  // (item, 128-key tile) steps of the chunk kernel
    for (int base = 0; base < n_cgroups; base += kPlanThreads) {
        const int gi = base + tid;
        int r = 0, mt = 0, kv_end = 0, b = -1;
        if (gi < n_cgroups) {
            r = find_group_request(req_c, R, gi);
            mt = gi - req_c[r];
            kv_end = chunk_kv_end(r, mt);
            b = chunk_bucket(kv_end);
        }
        const int first = (b >= 0 ? s_cbucket_base[b] : 0) + warp_claim(b, Hkv, s_cbucket_cursor);
        if (gi >= n_cgroups) continue;
        csteps += (long long)((kv_end + kChunkKeys - 1) / kChunkKeys) * Hkv;
        const int n = req_n[r];
        const long long rows = (long long)n * g;
        const int nv = (int)min((long long)kChunkRows, rows - (long long)mt * kChunkRows);
        for (int h = 0; h < Hkv; ++h) {
            const int idx = first + h;
            ChunkItem c;
            c.a = make_int4(r, mt, h, kv_end);
            c.b = make_int4(req_q0[r], n, req_L[r], nv);
            a.chunk_items[idx] = c;
        }
    }
    // 6. The chunk kernel's share of the SMs when it runs beside the
    // split-KV kernel: about what makes its tiles take as long as the split-KV
    // stream, capped so the stream keeps the SMs it needs to saturate HBM.
    if (n_cgroups > 0) csteps = block_sum<long long>(csteps, s_ll);  // n_cgroups is the same in every thread
    if (tid == 0) {
        int ctas = 0;
        if (csteps > 0) {
            const double chunk_sm_us = (double)csteps * a.chunk_sm_us_per_tile;
            const double decode_us = (double)work * a.block_bytes_kv / a.decode_bytes_per_us;
            if (decode_us < 1.0) {
                ctas = a.sm_count;
            } else {
                ctas = (int)ceil(chunk_sm_us / decode_us);
                ctas = max(1, min(ctas, a.sm_count * 9 / 20));
            }
        }
        a.header->chunk_ctas = ctas;
    }
}

// ---------------------------------------------------------------------------
// split-KV attention kernel
// ---------------------------------------------------------------------------

struct DecodeArgs {
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
    const int32_t *block_table;
    int max_blocks_per_req, num_blocks, num_q_heads, num_kv_heads, group;
    float scale_log2;
    const WorkItem *items;
    const GroupRec *group_rec;
    const int4 *prefix_map;
    int num_tokens;
    WsHeader *header;
    int32_t *tile_counter;
    float2 *part_ml;
    float *part_o;
    int beside_chunk;  // launched after the chunk kernel, running beside it (see attention_impl)
    int static_first;  // CTA b starts on item b (not beside the chunk kernel)
};

// Per-item description handed from the producer to the consumers through
// shared memory, next to the item's Q rows. item < 0 ends the CTA's loop.
// A split item's rows all belong to one decode tile; a prefix-tile item's
// rows may belong to up to 16 (row_tile: the tile's counter, -1 past
// n_valid).
struct ItemDesc {
    int item, kb0, kb1, n_valid, kv_end, partial, prefix, slots, part_row0, pad[7];
    int row_t[kRowsPerTile];
    int row_hq[kRowsPerTile];
    int row_limit[kRowsPerTile];
    int row_prow[kRowsPerTile];  // partial row this item writes for the row (when partial)
    int row_tile[kRowsPerTile];  // the row's tile counter (-1 past n_valid)
    int row_arr[kRowsPerTile];   // arrivals that tile waits for
};

// Blocks before an item's last copy at which the producer claims its CTA's
// next item. Same-box sweep on GB300 (Llama-3-8B decode step): claimed at the
// item's start 340.2 us; 8 blocks ahead 339.1; 16: 337.6; 32: 336.3; 64: 338.7.
#ifndef PKV_CLAIM_AHEAD
#define PKV_CLAIM_AHEAD 32
#endif

template <int D>
struct DecodeSmem {
    static constexpr int kBoxes = D / 64;                   // 64-column TMA boxes per tile
    static constexpr int kTileBytes = kBoxes * 2048;        // 16 rows x D bf16
    static constexpr int kStageBytes = 2 * kTileBytes;      // K tile + V tile
    static constexpr int kStages = D == 128 ? 8 : 12;
    static constexpr int kQStride = 2 * D;                  // Q rows as bulk-copied from q
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

__device__ __forceinline__ void bulk_copy_g2s(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// One work item on the producer warp: its description (rows, key range,
// where the result goes), its Q rows and its K/V block tiles through the
// ring. Prefix tiles and split items get separate copies of the streaming
// loop. Returns false when a wait gave up.
template <int D, bool kPrefix>
__device__ __forceinline__ bool produce_item(const CUtensorMap *kv_map, const DecodeArgs &a, uint8_t *smem, ItemDesc &d,
                                             int qb, int cur, int n_prefix, int split, int P, uint64_t *bar,
                                             uint32_t &e, int32_t *status, volatile int *abort, int claim_base,
                                             int &nxt) {
    using S = DecodeSmem<D>;
    uint64_t *full = bar, *empty = bar + S::kStages, *qfull = bar + 2 * S::kStages;
    const int lane = threadIdx.x & 31;
    const int Hkv = a.num_kv_heads, g = a.group;
    bool ok = true;
    int r, mt, q0, nv, kb0, kb1, kv_end, h;
    const int32_t *early_bt = nullptr;  // split items: block table row and first entries read early
    int early_raw = 0;
    if constexpr (kPrefix) {
        // Prefix tile: global rows [pt * 16, +16) over the shared
        // blocks [0, P), which every row sees whole.
        const int pt = cur / Hkv;
        h = cur - pt * Hkv;
        r = 0; mt = pt; q0 = 0;
        nv = (int)min((long long)kRowsPerTile, (long long)a.num_tokens * g - (long long)pt * kRowsPerTile);
        kb0 = 0; kb1 = P; kv_end = P * PKV_BLOCK_SIZE;
        if (lane < kRowsPerTile) {
            const int rho = pt * kRowsPerTile + lane;
            const bool valid = lane < nv;
            d.row_t[lane] = valid ? rho / g : 0;
            d.row_hq[lane] = h * g + (valid ? rho % g : 0);
            d.row_limit[lane] = kv_end - 1;
            const int4 m = valid ? a.prefix_map[rho] : make_int4(0, 0, -1, 0);
            d.row_prow[lane] = m.x + h * m.y;
            d.row_tile[lane] = valid ? m.z * Hkv + h : -1;
            d.row_arr[lane] = m.w;
        }
        if (lane == 0) { d.partial = 1; d.prefix = 1; }
    } else {
        const int4 w = a.items[cur - n_prefix].v;
        const int gi = w.x, s = w.z;
        h = w.y;
        // The item names its request, so the first 32 block-table entries
        // are requested together with the group record, not after it; they
        // are checked against the item's block range below.
        kb0 = P + s * split;
        early_bt = a.block_table + (long long)w.w * a.max_blocks_per_req;
        early_raw = kb0 + lane < a.max_blocks_per_req ? __ldg(early_bt + kb0 + lane) : 0;
        const GroupRec G = a.group_rec[gi];
        r = G.a.x; mt = G.a.y; q0 = G.a.z;
        const int n = G.a.w, L = G.b.x, kvb = G.b.z, slots = G.c.z;
        nv = G.b.w;
        kv_end = G.b.y;
        kb1 = min(kvb, kb0 + split);
        // Rows: token, q head, last visible key, partial row.
        if (lane < kRowsPerTile) {
            const int rho = mt * kRowsPerTile + lane;
            const bool valid = lane < nv;
            const int i = valid ? rho / g : 0;
            d.row_t[lane] = q0 + i;
            d.row_hq[lane] = h * g + (valid ? rho % g : 0);
            d.row_limit[lane] = valid ? L - n + i : kv_end - 1;
            d.row_prow[lane] = G.c.y + (h * slots + s + slots - G.c.x) * nv + lane;
            d.row_tile[lane] = valid ? gi * Hkv + h : -1;
            d.row_arr[lane] = G.c.w;
        }
        if (lane == 0) {
            d.partial = slots > 1; d.prefix = 0; d.slots = slots; d.part_row0 = G.c.y + h * slots * nv;
        }
    }
    if (lane == 0) {
        d.item = cur; d.kb0 = kb0; d.kb1 = kb1; d.n_valid = nv; d.kv_end = kv_end;
    }
    __syncwarp();
    // Q rows: one bulk copy per run of rows that belong to one token
    // (consecutive q heads, contiguous in q).
    uint8_t *qs = smem + S::kOffQ + qb * S::kQBytes;
    if (lane == 0) mbar_arrive_expect_tx(&qfull[qb], (uint32_t)nv * D * 2);
    __syncwarp();
    if (lane < nv) {
        const int rho = mt * kRowsPerTile + lane;
        const int i = rho / g;
        const bool run_start = lane == 0 || (rho - 1) / g != i;
        if (run_start) {
            int len = 1;
            while (lane + len < nv && (rho + len) / g == i) ++len;
            const __nv_bfloat16 *src = a.q + ((long long)(q0 + i) * a.num_q_heads + h * g + rho % g) * D;
            bulk_copy_g2s(qs + lane * S::kQStride, src, (uint32_t)len * D * 2, &qfull[qb]);
        }
    }
    if (lane != 0) mbar_arrive(&qfull[qb]);

    // K/V block tiles through the ring; block-table entries are
    // fetched 32 at a time, one batch ahead.
    const int32_t *bt = a.block_table + (long long)r * a.max_blocks_per_req;
    auto fetch = [&](int base) {
        int b = 0;
        if (base + lane < kb1) {
            b = __ldg(bt + base + lane);
            if (b < 0 || b >= a.num_blocks) {
                raise_status(status, PKV_DEV_BAD_BLOCK);
                b = a.num_blocks;  // outside the tensor map: TMA fills zeros
            }
        }
        return b;
    };
    // The CTA's next item is claimed PKV_CLAIM_AHEAD blocks before this
    // one's last copy is issued: late enough that a CTA never holds a whole
    // item in reserve while others run dry at the end of the list, early
    // enough that the claim's round trip is hidden.
    bool claimed = false;
    int my_blk;
    if (!kPrefix && early_bt == bt) {
        my_blk = 0;
        if (kb0 + lane < kb1) {
            my_blk = early_raw;
            if (my_blk < 0 || my_blk >= a.num_blocks) {
                raise_status(status, PKV_DEV_BAD_BLOCK);
                my_blk = a.num_blocks;
            }
        }
    } else {
        my_blk = fetch(kb0);
    }
    for (int base = kb0; base < kb1 && ok; base += 32) {
        const int nxt_blk = fetch(base + 32);
        const int cnt = min(32, kb1 - base);
        for (int j = 0; j < cnt; ++j) {
            if (!claimed && kb1 - (base + j) <= PKV_CLAIM_AHEAD) {
                if (lane == 0) nxt = claim_base + atomicAdd(&a.header->next_item, 1);
                claimed = true;
            }
            const int blk = __shfl_sync(0xffffffffu, my_blk, j);
            const int stage = e % S::kStages;
            if (!mbar_wait(&empty[stage], ((e / S::kStages) & 1) ^ 1, status, abort)) { ok = false; break; }
            if (lane == 0) {
                uint8_t *st = smem + S::kOffStages + stage * S::kStageBytes;
                mbar_arrive_expect_tx(&full[stage], S::kStageBytes);
                tma_load_5d(st, kv_map, 0, h * PKV_BLOCK_SIZE, 0, 0, blk, &full[stage]);
            }
            __syncwarp();
            ++e;
        }
        my_blk = nxt_blk;
    }
    if (!claimed && lane == 0) nxt = claim_base + atomicAdd(&a.header->next_item, 1);
    return ok;
}

// One consumer warp's share of an item: its blocks (every kConsumerWarps-th
// of [kb0, kb1)) against the item's NT * 8 query rows, then its unnormalised
// O, running max and sum per row into the CTA's scratch for the combine.
//
// The products run transposed, with the query rows as the mma's N = 8
// dimension: S^T (16 keys x 8 rows) = K Q^T and O^T (D x 8 rows) += V^T P^T.
// One 8-row n-tile (NT = 1) costs half the mma instructions of a 16-row
// tile, half or more of whose rows are padding for a decode token's GQA
// group of 4 or 8; the legacy mma path's rate per SM is what bounds a
// consumer warp's per-block time. P^T goes from the accumulator layout to the B
// operand layout with two 8x8 register transposes (movmatrix).
template <int D, int NT>
__device__ __forceinline__ void consume_item(const DecodeArgs &a, uint8_t *smem, const ItemDesc &d, int qb,
                                             uint64_t *full, uint64_t *empty, uint32_t &e, int32_t *status,
                                             volatile int *abort, int warp, int lane, float *scr, float2 *sml) {
    using S = DecodeSmem<D>;
    const int gid = lane >> 2, tig = lane & 3;  // fragment row group and column pair
    const int mi = lane >> 3;                   // ldmatrix: which 8x8 matrix this lane addresses
    // Per thread: rows r = nt * 8 + 2 tig + i (i = 0, 1) of each n-tile;
    // O^T accumulators ot[dc][nt]: {d = 16 dc + gid, 16 dc + gid + 8} x
    // {row 2 tig, 2 tig + 1}.
    float ot[D / 16][NT][4];
#pragma unroll
    for (int dc = 0; dc < D / 16; ++dc)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) ot[dc][nt][0] = ot[dc][nt][1] = ot[dc][nt][2] = ot[dc][nt][3] = 0.f;
    float m[NT][2], l[NT][2];
    int lim[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            m[nt][i] = -INFINITY;
            l[nt][i] = 0.f;
            lim[nt][i] = d.row_limit[nt * 8 + 2 * tig + i];
        }

    const int kb0 = d.kb0, kb1 = d.kb1, kv_end = d.kv_end;
    // Q^T as the B operand of S^T, for the whole item: qf[kk][nt] = rows
    // nt * 8 + gid, columns 16 kk + 2 tig (+ 8). Rows past n_valid hold stale
    // data; they only affect their own rows, which are never written.
    uint32_t qf[D / 16][NT][2];
    {
        const uint32_t qs = smem_u32(smem + S::kOffQ + qb * S::kQBytes);
        const int row = (lane & 7) + ((mi >> 1) & 1) * 8;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t r0, r1, r2, r3;
            ldmatrix_x4(qs + row * S::kQStride + (16 * kk + (mi & 1) * 8) * 2, r0, r1, r2, r3);
            qf[kk][0][0] = r0;
            qf[kk][0][1] = r1;
            if constexpr (NT == 2) {
                qf[kk][NT - 1][0] = r2;
                qf[kk][NT - 1][1] = r3;
            }
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
        // (other requests' stale data, NaN); their P is 0, but 0 * NaN is
        // not, so clear them.
        const bool tail = key0 + PKV_BLOCK_SIZE > kv_end;
        if (tail) {
            const int first = kv_end - key0;  // 1..15
            for (int c = lane; c < (PKV_BLOCK_SIZE - first) * S::kBoxes * 8; c += 32) {
                const int row = first + c / (S::kBoxes * 8);
                const int rem = c % (S::kBoxes * 8);
                *reinterpret_cast<uint4 *>(st + S::kTileBytes + (rem >> 3) * 2048 + row * 128 + (rem & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
        }

        // S^T = K Q^T: A = the block's 16 keys x 16 columns per K step; even
        // and odd K steps accumulate apart (two dependency chains of half
        // the length), then add.
        float sc[NT][4], sc2[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
            sc2[nt][0] = sc2[nt][1] = sc2[nt][2] = sc2[nt][3] = 0.f;
        }
        {
            const int key = (mi & 1) * 8 + (lane & 7);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int chunk = 2 * kk + (mi >> 1);
                uint32_t ka[4];
                ldmatrix_x4(kbase + (chunk >> 3) * 2048 + swz128(key, chunk & 7), ka[0], ka[1], ka[2], ka[3]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_bf16_16816((kk & 1) ? sc2[nt] : sc[nt], ka, qf[kk][nt][0], qf[kk][nt][1]);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c) sc[nt][c] += sc2[nt][c];
        }


        // Scale into the log2 domain, causal mask, online softmax per row
        // (a column of S^T: keys gid and gid + 8 here, the rest across the
        // lanes of equal tig).
        uint32_t pb[NT][2];
        float al[NT][2];
        bool moved = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float mx[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float s0 = key0 + gid <= lim[nt][i] ? sc[nt][i] * a.scale_log2 : -INFINITY;
                const float s1 = key0 + gid + 8 <= lim[nt][i] ? sc[nt][2 + i] * a.scale_log2 : -INFINITY;
                sc[nt][i] = s0;
                sc[nt][2 + i] = s1;
                mx[i] = fmaxf(s0, s1);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 4));
                mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 8));
                mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 16));
            }
            float p[4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float mn = fmaxf(m[nt][i], mx[i]);
                const float base = mn == -INFINITY ? 0.f : mn;
                al[nt][i] = fast_exp2(m[nt][i] - base);
                moved |= al[nt][i] != 1.f;
                m[nt][i] = mn;
                p[i] = fast_exp2(sc[nt][i] - base);
                p[2 + i] = fast_exp2(sc[nt][2 + i] - base);
                l[nt][i] = l[nt][i] * al[nt][i] + (p[i] + p[2 + i]);
            }
            // P^T (keys x rows) in the accumulator layout, as bf16 pairs,
            // transposed into the B operand of O^T += V^T P^T.
            pb[nt][0] = movmatrix_trans(pack_bf16x2(p[0], p[1]));  // keys 0-7
            pb[nt][1] = movmatrix_trans(pack_bf16x2(p[2], p[3]));  // keys 8-15
        }
        if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
            for (int dc = 0; dc < D / 16; ++dc)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    ot[dc][nt][0] *= al[nt][0];
                    ot[dc][nt][1] *= al[nt][1];
                    ot[dc][nt][2] *= al[nt][0];
                    ot[dc][nt][3] *= al[nt][1];
                }
        }

        // O^T += V^T P^T: A = V^T, 16 columns x the block's 16 keys per step.
        {
            const int key = (mi >> 1) * 8 + (lane & 7);
#pragma unroll
            for (int dc = 0; dc < D / 16; ++dc) {
                const int chunk = 2 * dc + (mi & 1);
                uint32_t va[4];
                ldmatrix_x4_trans(vbase + (chunk >> 3) * 2048 + swz128(key, chunk & 7), va[0], va[1], va[2], va[3]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(ot[dc][nt], va, pb[nt][0], pb[nt][1]);
            }
        }
        __syncwarp();
        if (lane == 0) {
            if (tail) fence_proxy_async_smem();
            mbar_arrive(&empty[stage]);
        }
    }

    // This warp's state per row -> scratch: sums over the lanes of equal
    // tig, O^T transposed back into rows.
    float *ws = scr + warp * kRowsPerTile * S::kScrStride;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float s = l[nt][i];
            s += __shfl_xor_sync(0xffffffffu, s, 4);
            s += __shfl_xor_sync(0xffffffffu, s, 8);
            s += __shfl_xor_sync(0xffffffffu, s, 16);
            const int row = nt * 8 + 2 * tig + i;
            if (gid == 0) sml[warp * kRowsPerTile + row] = make_float2(m[nt][i], s);
#pragma unroll
            for (int dc = 0; dc < D / 16; ++dc) {
                ws[row * S::kScrStride + 16 * dc + gid] = ot[dc][nt][i];
                ws[row * S::kScrStride + 16 * dc + gid + 8] = ot[dc][nt][2 + i];
            }
        }
    }
}

// One consumer warp's share of an item with more than 8 valid rows: its
// blocks against all 16 rows of the tile (S = Q K^T, O += P V with the rows
// as M = 16), then its unnormalised O, running max and sum per row into the
// CTA's scratch.
template <int D>
__device__ __forceinline__ void consume_item16(const DecodeArgs &a, uint8_t *smem, const ItemDesc &d, int qb,
                                               uint64_t *full, uint64_t *empty, uint32_t &e, int32_t *status,
                                               volatile int *abort, int warp, int lane, float *scr, float2 *sml) {
    using S = DecodeSmem<D>;
    const int qrow = lane >> 2;  // fragment rows qrow and qrow + 8
    const int qcol = (lane & 3) * 2;
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    {
        const int kb0 = d.kb0, kb1 = d.kb1, kv_end = d.kv_end;
        const int lim0 = d.row_limit[qrow], lim1 = d.row_limit[qrow + 8];

        // Q fragments (A operand, 16 rows x D) for the whole item. Rows
        // past n_valid hold stale data; they only affect their own rows,
        // which are never written.
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
}

template <int D>
__global__ void __launch_bounds__(kDecodeThreads, D == 128 ? 2 : 3)
decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeArgs a) {
    using S = DecodeSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_abort;  // set by any wait that gives up; every later wait returns at once
    __shared__ int s_stop;   // consumers' uniform loop decision, written by consumer thread 0
    __shared__ int s_last;   // rows of this item whose tile it finished (bit per row)
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::kOffBar);
    uint64_t *full = bar, *empty = bar + S::kStages, *qfull = bar + 2 * S::kStages, *qempty = qfull + 2;
    ItemDesc *desc = reinterpret_cast<ItemDesc *>(smem + S::kOffDesc);
    volatile int *abort = &s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *status = &a.header->status;

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
    // The prologue above overlaps the previous kernel; the work list it
    // wrote is read only after this. Beside the chunk kernel, the previous
    // kernel is the chunk kernel, which launched this one only after the
    // work list was complete; this kernel waits for it at its end instead.
    if (!a.beside_chunk) pdl_wait();
    pdl_launch_dependents();
    const int n_prefix = a.header->n_prefix_items;
    const int n_items = n_prefix + a.header->n_items;
    const int split = a.header->split_blocks;
    const int P = a.header->cascade_blocks;

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) tma_prefetch_desc(&kv_map);
        uint32_t e = 0;  // ring element counter
        bool ok = true;
        // CTA b starts on item b (the list is longest first, so the longest
        // items spread over the SMs) and later items come from the counter,
        // past the grid's first items (a CTA whose b is past the list just
        // leaves). Beside the chunk kernel (where some CTAs start only when
        // chunk CTAs leave), every item is claimed from the counter.
        const int claim_base = a.static_first ? (int)gridDim.x : 0;
        int cur = (int)blockIdx.x;
        if (!a.static_first) {
            if (lane == 0) cur = atomicAdd(&a.header->next_item, 1);
            cur = __shfl_sync(0xffffffffu, cur, 0);
        }
        for (int k = 0;; ++k) {
            const int qb = k & 1;
            if (!mbar_wait(&qempty[qb], ((k >> 1) & 1) ^ 1, status, abort)) { ok = false; break; }
            ItemDesc &d = desc[qb];
            if (cur >= n_items) {
                if (lane == 0) d.item = -1;
                mbar_arrive(&qfull[qb]);
                break;
            }
            int nxt = 0;  // lane 0: the next item, claimed inside produce_item
            ok = cur < n_prefix
                     ? produce_item<D, true>(&kv_map, a, smem, desc[qb], qb, cur, n_prefix, split, P, bar, e, status,
                                             abort, claim_base, nxt)
                     : produce_item<D, false>(&kv_map, a, smem, desc[qb], qb, cur, n_prefix, split, P, bar, e, status,
                                              abort, claim_base, nxt);
            if (!ok) break;
            cur = __shfl_sync(0xffffffffu, nxt, 0);
        }
        // After a failure, do not leave while copies into this CTA's shared
        // memory are still in flight: wait (bounded) for the last issue of
        // every stage.
        if (!ok && lane == 0) {
            for (uint32_t x = e > (uint32_t)S::kStages ? e - S::kStages : 0; x < e; ++x)
                mbar_drain(&full[x % S::kStages], (x / S::kStages) & 1, status, &a.header->diag, 0x1);
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    const int tid = threadIdx.x;  // 0..127
    float *scr = reinterpret_cast<float *>(smem + S::kOffScr);
    float2 *sml = reinterpret_cast<float2 *>(smem + S::kOffML);
    uint32_t e = 0;
    for (int k = 0;; ++k) {
        const int qb = k & 1;
        const bool have_q = mbar_wait(&qfull[qb], (k >> 1) & 1, status, abort);
        const ItemDesc &d = desc[qb];
        // One thread decides for all four warps whether to go on, so that
        // they leave together and never strand each other at a barrier.
        if (tid == 0) s_stop = (!have_q || *abort || d.item < 0) ? 1 : 0;
        named_barrier_sync(1, kConsumerWarps * 32);
        if (s_stop) {
            // beside the chunk kernel: end only after it (one thread holds the CTA)
            if (a.beside_chunk && tid == 0) pdl_wait();
            return;
        }

        // Up to 8 rows (a decode token's GQA group of 8 or fewer): the
        // transposed 8-row products, half the mma instructions of 16-row
        // ones; more: 16-row products.
        if (d.n_valid <= 8)
            consume_item<D, 1>(a, smem, d, qb, full, empty, e, status, abort, warp, lane, scr, sml);
        else
            consume_item16<D>(a, smem, d, qb, full, empty, e, status, abort, warp, lane, scr, sml);
        named_barrier_sync(1, kConsumerWarps * 32);
        const int n_valid = d.n_valid;
        const bool partial = d.partial != 0;
        constexpr int kC4 = D / 4;
        for (int idx = tid; idx < n_valid * kC4; idx += kConsumerWarps * 32) {
            const int row = idx / kC4, c4 = idx % kC4;
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
                    const float4 v =
                        *reinterpret_cast<const float4 *>(scr + (w * kRowsPerTile + row) * S::kScrStride + c4 * 4);
                    acc.x += v.x * f; acc.y += v.y * f; acc.z += v.z * f; acc.w += v.w * f;
                }
            }
            if (!partial) {
                const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
                const long long off = ((long long)d.row_t[row] * a.num_q_heads + d.row_hq[row]) * D + c4 * 4;
                uint2 pk;
                pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
                pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
                *reinterpret_cast<uint2 *>(a.out + off) = pk;
            } else {
                const long long prow = d.row_prow[row];
                *reinterpret_cast<float4 *>(a.part_o + prow * D + c4 * 4) = acc;
                if (c4 == 0) a.part_ml[prow] = make_float2(M, lsum);
            }
        }
        if (partial) {
            // Publish the partial rows, then count one arrival at each tile
            // they belong to (the first row of each run of equal tiles
            // counts); the CTA that brings a tile's count to its arrivals
            // merges the tile (no waiting). The count is an acquire-release
            // atomic after the consumers' barrier: it releases every
            // consumer thread's partial rows, and for the last arriver it
            // acquires the other CTAs' rows, which its threads read after
            // the next barrier.
            named_barrier_sync(1, kConsumerWarps * 32);
            if (warp == 0) {
                bool last = false;
                if (lane < n_valid) {
                    const int tile = d.row_tile[lane];
                    if (lane == 0 || d.row_tile[lane - 1] != tile)
                        last = atom_add_acq_rel(&a.tile_counter[tile], 1) == d.row_arr[lane] - 1;
                }
                const unsigned mask = __ballot_sync(0xffffffffu, last);
                if (lane == 0) s_last = (int)mask;
            }
            named_barrier_sync(1, kConsumerWarps * 32);
            unsigned todo = (unsigned)s_last;
            while (todo) {
                const int tile = d.row_tile[__ffs(todo) - 1];
                todo &= todo - 1;
                // A split item merges its own tile (all in the description);
                // a prefix tile looks up the tile it completed.
                const int g = a.group;
                int h, mt = 0, q0 = 0, nv = n_valid, slots = d.slots;
                long long prow0 = d.part_row0;
                const bool pfx = d.prefix != 0;
                if (pfx) {
                    const int gi = tile / a.num_kv_heads;
                    h = tile - gi * a.num_kv_heads;
                    const GroupRec G = a.group_rec[gi];
                    mt = G.a.y; q0 = G.a.z; nv = G.b.w; slots = G.c.z;
                    prow0 = G.c.y + (long long)h * slots * nv;
                } else {
                    h = tile % a.num_kv_heads;
                }
                for (int idx = tid; idx < nv * kC4; idx += kConsumerWarps * 32) {
                    const int row = idx / kC4, c4 = idx % kC4;
                    float M = -INFINITY;
                    for (int sp = 0; sp < slots; ++sp)
                        M = fmaxf(M, __ldcg(&a.part_ml[prow0 + (long long)sp * nv + row]).x);
                    float lsum = 0.f;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int sp = 0; sp < slots; ++sp) {
                        const long long prow = prow0 + (long long)sp * nv + row;
                        const float2 ml = __ldcg(&a.part_ml[prow]);
                        const float f = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - M);
                        lsum += ml.y * f;
                        const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.part_o + prow * D + c4 * 4));
                        acc.x += v.x * f; acc.y += v.y * f; acc.z += v.z * f; acc.w += v.w * f;
                    }
                    long long orow;
                    if (pfx) {
                        const int rho = mt * kRowsPerTile + row;
                        orow = (long long)(q0 + rho / g) * a.num_q_heads + h * g + rho % g;
                    } else {
                        orow = (long long)d.row_t[row] * a.num_q_heads + d.row_hq[row];
                    }
                    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
                    uint2 pk;
                    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
                    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
                    *reinterpret_cast<uint2 *>(a.out + orow * D + c4 * 4) = pk;
                }
            }
        }
        named_barrier_sync(1, kConsumerWarps * 32);
        if (lane == 0) mbar_arrive(&qempty[qb]);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// SM-microseconds one 128 x 128 chunk tile step is costed at when the work
// list shares the SMs between the chunk and split-KV kernels. Measured on
// GB300: ~1.8 at head 128 (the mixed batch's 4352 steps in ~52 us on 152
// SMs); the mixed step was flat from 1.8 to 3.6 (the split-KV stream was the
// longer side) and 35 % slower at 1.2, so the value sits inside that range.
// Head 64 is scaled the same way, not measured.
#ifndef PKV_CHUNK_SM_US_128
#define PKV_CHUNK_SM_US_128 2.8f
#endif
#ifndef PKV_CHUNK_SM_US_64
#define PKV_CHUNK_SM_US_64 1.9f
#endif

struct DeviceInfo {
    int sm_count = 0;
    int ctas_per_sm[2] = {0, 0};  // attention kernel, D = 64 / 128
    bool ready = false;
};

std::mutex g_mu;
DeviceInfo g_dev[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

constexpr int kPlanSmemBytes = (kReqCacheArrays * (kPlanSmemReqs + 1) + 2 * kPlanSmemGroups) * 4;

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
        if (cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPlanSmemBytes) !=
            cudaSuccess)
            return PKV_E_CUDA;
        if (chunk_configure() != PKV_OK) return PKV_E_CUDA;
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

// Default split-KV partial capacity in rows: twice a full persistent grid's
// worth of split items (up to 3 CTAs per SM), each with a full 16-row tile.
// Partial-row capacity a full workspace gets: enough for the split-KV
// schedule of a persistent grid, and for two slots per query row (a shared-
// prefix slot and one split) up to 2^20 rows.
long long default_part_rows_cap(int sm_count, long long num_tokens, int num_q_heads) {
    const long long grid_rows = (long long)sm_count * 3 * kItemsPerCta * kRowsPerTile * 2;
    const long long prefix_rows = min(2 * num_tokens * num_q_heads, 1LL << 20);
    return max(grid_rows, prefix_rows);
}

// The pool [NB][2][Hkv][16][D] as a 5-D map {64 columns, row of the head
// (head * 16 + token), 64-column half, K or V, block}; one box is a whole
// (block, head): its 16 K rows and 16 V rows x D columns, landing in shared
// memory as [K / V][D / 64][16 rows][128 B] (128-byte swizzle). One copy per
// block and head instead of one per 64 columns of K and of V: the copy
// engine spends a fixed cost per box.
int encode_kv_map(CUtensorMap *map, const void *kv_cache, const pkv_cache_desc &d) {
    const cuuint64_t rows_per_kv = (cuuint64_t)d.num_kv_heads * PKV_BLOCK_SIZE;
    const cuuint64_t row = (cuuint64_t)d.head_size * 2;
    cuuint64_t dims[5] = {64, rows_per_kv, (cuuint64_t)d.head_size / 64, 2, (cuuint64_t)d.num_blocks};
    cuuint64_t strides[4] = {row, 128, rows_per_kv * row, 2 * rows_per_kv * row};
    cuuint32_t box[5] = {64, PKV_BLOCK_SIZE, (cuuint32_t)d.head_size / 64, 2, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult res = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(kv_cache), dims, strides,
                            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? PKV_OK : PKV_E_CUDA;
}

// The pool as the chunk kernel stages it: a 5-D map {64 columns, token
// within an 8-token half, 64-column half, 8-token group of the block's rows
// ((kv * Hkv + head) * 2 + token half), block}; one box is a whole (block, K
// or V, head), landing as [token half][D / 64][8 tokens][128 B] (128-byte
// swizzle). The 8-token groups of consecutive blocks are then evenly spaced,
// so one N=128 tensor-core product covers a 128-key tile.
int encode_kv_map_chunk(CUtensorMap *map, const void *kv_cache, const pkv_cache_desc &d) {
    const cuuint64_t groups_per_block = 2ull * d.num_kv_heads * 2;
    const cuuint64_t row = (cuuint64_t)d.head_size * 2;
    cuuint64_t dims[5] = {64, 8, (cuuint64_t)d.head_size / 64, groups_per_block, (cuuint64_t)d.num_blocks};
    cuuint64_t strides[4] = {row, 128, 8 * row, groups_per_block * 8 * row};
    cuuint32_t box[5] = {64, 8, (cuuint32_t)d.head_size / 64, 2, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult res = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(kv_cache), dims, strides,
                            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? PKV_OK : PKV_E_CUDA;
}

// q [T][Hq][D] as a 3-D map; one box is the 128 rows of a chunk tile: 128/g
// tokens x the g q heads of one kv head x 64 columns.
int encode_q_map(CUtensorMap *map, const void *q, int num_tokens, int num_q_heads, int head_size, int group) {
    cuuint64_t dims[3] = {(cuuint64_t)head_size, (cuuint64_t)num_q_heads, (cuuint64_t)num_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)head_size * 2, (cuuint64_t)num_q_heads * head_size * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)(kChunkRows / group)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult res = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? PKV_OK : PKV_E_CUDA;
}

void record(void *const *events, int i, cudaStream_t st) {
    if (events && events[i]) cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st);
}

int attention_impl(const void *q, int32_t num_tokens, int32_t num_q_heads, const void *kv_cache,
                   const pkv_cache_desc *desc, const int32_t *block_table, int32_t num_reqs,
                   int32_t max_blocks_per_req, const int32_t *seq_lens, const int32_t *query_start_loc, float scale,
                   void *out, void *workspace, size_t workspace_bytes, void *stream, void *const *events,
                   int32_t max_query_len) {
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
    long long part_rows = default_part_rows_cap(di->sm_count, num_tokens, num_q_heads);
    WsLayout L = ws_layout(num_reqs, num_tokens, num_q_heads, Hkv, D, part_rows);
    if (L.total > workspace_bytes) {
        const size_t spare = workspace_bytes - base.total;
        const long long fit = spare > 1024 ? (long long)((spare - 1024) / part_row_bytes(D)) : 0;
        if (fit < part_rows) part_rows = fit;
        L = ws_layout(num_reqs, num_tokens, num_q_heads, Hkv, D, part_rows);
        if (L.total > workspace_bytes) return PKV_E_WORKSPACE;
    }

    CUtensorMap kv_map;
    rc = encode_kv_map(&kv_map, kv_cache, *desc);
    if (rc) return rc;
    const int group = num_q_heads / Hkv;
    // The chunk kernel takes requests with >= 128 query rows when a 128-row
    // tile holds whole tokens.
    // A caller bound on new tokens per request (0: none) that keeps every
    // request below 128 rows means no chunk tiles: the chunk kernel is not
    // launched and the work list puts every row on the split-KV path (so a
    // bound that is too small costs speed, never correctness).
    const bool chunk_ok = kChunkRows % group == 0 && (long long)num_tokens * group >= kChunkRows &&
                          (max_query_len <= 0 || (long long)max_query_len * group >= kChunkRows);
    CUtensorMap q_map, kv_map_chunk;
    if (chunk_ok) {
        rc = encode_q_map(&q_map, q, num_tokens, num_q_heads, D, group);
        if (!rc) rc = encode_kv_map_chunk(&kv_map_chunk, kv_cache, *desc);
        if (rc) return rc;
    }

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
    pa.block_bytes_kv = 2 * PKV_BLOCK_SIZE * D * 2;
    pa.chunk_ok = chunk_ok ? 1 : 0;
    pa.sm_count = di->sm_count;
    pa.chunk_sm_us_per_tile = D == 128 ? PKV_CHUNK_SM_US_128 : PKV_CHUNK_SM_US_64;  // the split-KV stream: ~6.8 TB/s
    pa.decode_bytes_per_us = 6.8e6f;
    pa.chunk_items_cap = L.chunk_items_cap;
    pa.chunk_items = reinterpret_cast<ChunkItem *>(ws + L.chunk_items);
    pa.target_items = (long long)ctas * kItemsPerCta;
    pa.part_rows_cap = L.part_rows_cap;
    pa.groups_cap = L.groups_cap;
    pa.items_cap = L.items_cap;
    pa.header = header;
    pa.req_cache = reinterpret_cast<int32_t *>(ws + L.req_cache);
    pa.group_req = reinterpret_cast<int32_t *>(ws + L.group_req);
    pa.group_kvb = reinterpret_cast<int32_t *>(ws + L.group_kvb);
    pa.tile_counter = reinterpret_cast<int32_t *>(ws + L.tile_counter);
    pa.items = reinterpret_cast<WorkItem *>(ws + L.items);
    pa.group_rec = reinterpret_cast<GroupRec *>(ws + L.group_rec);
    pa.block_table = block_table;
    pa.prefix_map = reinterpret_cast<int4 *>(ws + L.prefix_map);
    int plan_smem = 0;
    if (num_reqs <= kPlanSmemReqs) {
        plan_smem = kReqCacheArrays * (num_reqs + 1) * 4;
        if (L.groups_cap <= kPlanSmemGroups) plan_smem += 2 * (int)L.groups_cap * 4;
    }
    record(events, 0, st);
    cudaError_t err = launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), plan_smem, st, pa);
    if (err != cudaSuccess) return PKV_E_CUDA;
    record(events, 1, st);

    DecodeArgs da{};
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
    da.group_rec = pa.group_rec;
    da.prefix_map = pa.prefix_map;
    da.num_tokens = num_tokens;
    da.header = header;
    da.tile_counter = pa.tile_counter;
    da.part_ml = reinterpret_cast<float2 *>(ws + L.part_ml);
    da.part_o = reinterpret_cast<float *>(ws + L.part_o);

    auto launch_decode = [&]() {
        return D == 128 ? launch_pdl(decode_kernel<128>, dim3(ctas), dim3(kDecodeThreads), DecodeSmem<128>::kAlloc,
                                     st, kv_map, da)
                        : launch_pdl(decode_kernel<64>, dim3(ctas), dim3(kDecodeThreads), DecodeSmem<64>::kAlloc,
                                     st, kv_map, da);
    };
    ChunkArgs ca{};
    if (chunk_ok) {
        ca.block_table = block_table;
        ca.max_blocks_per_req = max_blocks_per_req;
        ca.num_blocks = desc->num_blocks;
        ca.num_q_heads = num_q_heads;
        ca.num_kv_heads = Hkv;
        ca.group = group;
        ca.scale_log2 = scale * kLog2e;
        ca.items = pa.chunk_items;
        ca.header = header;
        ca.out = static_cast<__nv_bfloat16 *>(out);
    }
    // With chunk tiles (and no per-kernel timing), the chunk kernel runs
    // beside the split-KV kernel: its CTAs past the work list's share leave
    // at once, and the split-KV kernel (which may launch only once every
    // chunk CTA has started or left) fills the SMs they free. The split-KV
    // kernel then reads the work list without waiting for the chunk kernel
    // and waits for it only at its end, so later work on `st` still starts
    // after both.
    if (chunk_ok && !events) {
        ca.beside = 1;
        da.beside_chunk = 1;
    }
    // CTA b starts on item b without a claim (a CTA whose b is past the
    // list leaves, as it would after a claim past it): one atomic round
    // trip less before the first copies, which is most of a small batch's
    // start-up. Beside the chunk kernel some CTAs start only when chunk
    // CTAs leave, so there every item is claimed from the counter.
    da.static_first = !da.beside_chunk ? 1 : 0;
    if (chunk_ok && chunk_launch(D, di->sm_count, kv_map_chunk, q_map, ca, st) != cudaSuccess) return PKV_E_CUDA;
    record(events, 2, st);
    err = launch_decode();
    record(events, 3, st);
    return err == cudaSuccess && cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_E_CUDA;
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
                                 default_part_rows_cap(di->sm_count, max_num_tokens, num_q_heads));
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

extern "C" PKV_API int paged_attention(const void *q, int32_t num_tokens, int32_t num_q_heads, const void *kv_cache,
                                       const pkv_cache_desc *desc, const int32_t *block_table, int32_t num_reqs,
                                       int32_t max_blocks_per_req, const int32_t *seq_lens,
                                       const int32_t *query_start_loc, float scale, void *out, void *workspace,
                                       size_t workspace_bytes, void *stream) {
    return attention_impl(q, num_tokens, num_q_heads, kv_cache, desc, block_table, num_reqs, max_blocks_per_req,
                          seq_lens, query_start_loc, scale, out, workspace, workspace_bytes, stream, nullptr, 0);
}

extern "C" PKV_API int paged_attention_bounded(const void *q, int32_t num_tokens, int32_t num_q_heads,
                                               const void *kv_cache, const pkv_cache_desc *desc,
                                               const int32_t *block_table, int32_t num_reqs,
                                               int32_t max_blocks_per_req, const int32_t *seq_lens,
                                               const int32_t *query_start_loc, int32_t max_query_len, float scale,
                                               void *out, void *workspace, size_t workspace_bytes, void *stream,
                                               void *const *events) {
    return attention_impl(q, num_tokens, num_q_heads, kv_cache, desc, block_table, num_reqs, max_blocks_per_req,
                          seq_lens, query_start_loc, scale, out, workspace, workspace_bytes, stream, events,
                          max_query_len);
}

extern "C" PKV_API int paged_attention_timed(const void *q, int32_t num_tokens, int32_t num_q_heads,
                                             const void *kv_cache, const pkv_cache_desc *desc,
                                             const int32_t *block_table, int32_t num_reqs,
                                             int32_t max_blocks_per_req, const int32_t *seq_lens,
                                             const int32_t *query_start_loc, float scale, void *out, void *workspace,
                                             size_t workspace_bytes, void *stream, void *const *events) {
    return attention_impl(q, num_tokens, num_q_heads, kv_cache, desc, block_table, num_reqs, max_blocks_per_req,
                          seq_lens, query_start_loc, scale, out, workspace, workspace_bytes, stream, events, 0);
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
                          seq_lens, query_start_loc, scale, out, scratch, kStaticScratchBytes, stream, nullptr, 0);
}
