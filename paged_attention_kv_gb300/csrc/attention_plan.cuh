// Work decomposition shared by the attention kernels.
//
// Rows. Request r with n new tokens and GQA group g = Hq / Hkv owns, per kv
// head h, n * g query rows; row rho is token i = rho / g of the request and
// query head h * g + rho % g. Rows are cut into tiles of 16 (mma M).
//
// Groups and tiles. A group is one (request, row tile mt); it expands into
// Hkv tiles (one per kv head).
//
// Items. A tile's keys [0, kv_end) are cut into splits of split_blocks
// blocks; each (tile, split) is one work item for one CTA. A tile with one
// split writes `out` directly. A tile with ns > 1 splits writes, per split,
// its n_valid rows of (unnormalised O, running max m in log2 units, sum l)
// to the partial rows [part_row0 + s * n_valid, ...); the CTA that finishes
// the tile's last split (a per-tile arrival counter) merges them with
// weights 2^(m_s - max_s m_s). Items are listed longest first (full-size
// splits, then the shorter ones in size buckets) and handed out through an
// atomic counter.
#pragma once

#include <cstddef>
#include <cstdint>

namespace pkv {

constexpr int kRowsPerTile = 16;
#ifndef PKV_MIN_ITEM_KB
#define PKV_MIN_ITEM_KB 256
#endif
#ifndef PKV_ITEMS_PER_CTA
#define PKV_ITEMS_PER_CTA 4
#endif
constexpr int kMinSplitBlocks = 4;   // at least one block per consumer warp
// Split target. Each item ends with a CTA-wide combine whose latency idles
// the CTA's HBM stream, so fewer, longer items win as long as the longest-
// first order still balances the grid (a sweep on GB300 put the best at ~4
// items per CTA and >= 256 KiB of K+V per item).
constexpr int kMinItemBytes = PKV_MIN_ITEM_KB << 10;  // at least this much K+V per item
constexpr int kItemsPerCta = PKV_ITEMS_PER_CTA;      // items per persistent CTA
constexpr int kPlanSmemReqs = 4096;    // per-request tables kept in shared memory up to this many requests
constexpr int kPlanSmemGroups = 8192;  // per-group tables likewise, up to this many decode groups
constexpr int kSizeBuckets = 9;      // 0 = full-size split, 1..8 = shorter, longest first

// Shared prefix. When every request's block table starts with the same
// P >= kCascadeMinBlocks blocks (a prefix-cache hit shared by the whole
// batch) and those keys are visible to every query row, the batch's rows
// are also cut, across request boundaries, into "prefix tiles" of 16 rows
// (global row T_r * g + rho for token T_r of the flattened batch) that run
// against those P blocks only: the shared blocks are read once per 16 rows
// instead of once per request. Every decode tile then has ns + 1 partial
// slots: slot 0 is written by the prefix tiles covering its rows, slots
// 1..ns by its splits over the blocks [P, kv blocks); its arrival count is
// ns plus the number of prefix tiles overlapping it.
constexpr int kCascadeMinBlocks = 4;
constexpr int kCascadeMinReqs = 4;
constexpr int kCascadeMaxBlocks = 4096;

// Chunk tiles (tcgen05 path): requests with at least kChunkRows query rows
// (n * g) are cut into 128-row tiles that run over 128-key tiles; a work
// item is one tile of one request and kv head.
constexpr int kChunkRows = 128;
constexpr int kChunkKeys = 128;

struct WsHeader {
    int32_t status;        // device status word (first 4 bytes of the workspace)
    int32_t n_items;
    int32_t split_blocks;
    int32_t n_groups;
    int32_t n_partial_rows;
    int32_t next_item;     // dynamic scheduling counter
    int32_t n_chunk_items;
    int32_t next_chunk_item;
    int32_t diag;          // bits naming the pipeline waits that timed out (PKV_DEV_TIMEOUT)
    int32_t n_prefix_items; // prefix-tile items (listed before the split items; 0 without a shared prefix)
    int32_t cascade_blocks; // P: leading blocks shared by every request (0: none)
    int32_t chunk_ctas;     // chunk-kernel CTAs that stay when it runs beside the split-KV kernel
    int32_t pad[52];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte line");

// One split-KV work item: {group, kv head h, split s, request}. The rest
// lives in the group's record, written once per group; the request is here
// too so that the attention kernel can read its block-table row while the
// group record is on its way.
struct WorkItem {
    int4 v;
};

// a = {r, mt, qstart, n}, b = {L, kv_end, kv blocks, valid rows},
// c = {splits ns over the blocks after the shared prefix, first partial row
// of kv head 0 (or -1), partial slots (ns, or ns + 1 with a shared prefix),
// arrivals before the merge}. Kv head h's slot s holds rows
// [c.y + (h * slots + s) * valid rows, ...).
struct GroupRec {
    int4 a, b, c;
};

struct WsLayout {
    size_t req_cache, group_req, group_kvb, group_rec, tile_counter, items, chunk_items, prefix_map, part_ml, part_o,
        total;
    long long groups_cap, tiles_cap, items_cap, chunk_items_cap, part_rows_cap;
};

constexpr int kReqCacheArrays = 5;  // n, L, q0, decode-tile base, chunk-tile base

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(long long num_reqs, long long num_tokens, int num_q_heads, int num_kv_heads,
                          int head_size, long long part_rows_cap) {
    WsLayout L{};
    const long long g = num_q_heads / num_kv_heads;
    L.groups_cap = (num_tokens * g + kRowsPerTile - 1) / kRowsPerTile + num_reqs;
    L.tiles_cap = L.groups_cap * num_kv_heads;
    L.part_rows_cap = part_rows_cap;
    L.items_cap = L.tiles_cap + part_rows_cap;
    L.chunk_items_cap = ((num_tokens * g + kChunkRows - 1) / kChunkRows + num_reqs) * num_kv_heads;
    size_t off = sizeof(WsHeader);
    L.req_cache = off;    off = align256(off + sizeof(int32_t) * kReqCacheArrays * (num_reqs + 1));
    L.group_req = off;    off = align256(off + sizeof(int32_t) * L.groups_cap);
    L.group_kvb = off;    off = align256(off + sizeof(int32_t) * L.groups_cap);
    L.group_rec = off;    off = align256(off + sizeof(GroupRec) * L.groups_cap);
    L.tile_counter = off; off = align256(off + sizeof(int32_t) * L.tiles_cap);
    L.items = off;        off = align256(off + sizeof(WorkItem) * L.items_cap);
    L.chunk_items = off;  off = align256(off + 32 * L.chunk_items_cap);
    L.prefix_map = off;   off = align256(off + sizeof(int4) * num_tokens * g);
    L.part_ml = off;      off = align256(off + sizeof(float2) * part_rows_cap);
    L.part_o = off;       off = align256(off + sizeof(float) * head_size * part_rows_cap);
    L.total = off;
    return L;
}

// Bytes per partial row (item slot, m/l pair, O row) used to size capacity.
inline size_t part_row_bytes(int head_size) {
    return sizeof(WorkItem) + sizeof(float2) + sizeof(float) * head_size;
}

}  // namespace pkv
