// Work decomposition shared by the attention kernels.
//
// Rows. Request r with n new tokens and GQA group g = Hq / Hkv owns, per kv
// head h, n * g query rows; row rho is token i = rho / g of the request and
// query head h * g + rho % g. Rows are cut into tiles of 16 (mma M).
//
// Groups and tiles. A group is one (request, row tile mt); it expands into
// Hkv tiles (one per kv head). req_group_base[r] is the first group of
// request r (an exclusive prefix sum of the per-request tile counts).
//
// Items. A tile's keys [0, kv_end) are cut into splits of split_blocks
// blocks; each (tile, split) is one work item for one CTA. A tile with one
// split writes `out` directly; a tile with several writes one partial
// (unnormalised O, running max m in log2 units, sum l) per split, merged by
// the merge kernel with weights 2^(m_s - max_s m_s).
#pragma once

#include <cstddef>
#include <cstdint>

namespace pkv {

constexpr int kRowsPerTile = 16;
constexpr int kMinSplitBlocks = 4;   // at least one block per consumer warp
constexpr int kItemsPerCta = 16;     // split target: items per persistent CTA

struct WsHeader {
    int32_t status;        // device status word (first 4 bytes of the workspace)
    int32_t n_items;
    int32_t split_blocks;
    int32_t n_groups;
    int32_t n_partials;
    int32_t pad[59];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte line");

// One work item: a = {r, mt, h, s}, b = {kb0, kb1, partial or -1, qstart},
// c = {n, L, kv_end, 0}. kv_end is the tile's last visible key + 1.
struct WorkItem {
    int4 a, b, c;
};

struct WsLayout {
    size_t req_group_base, group_kvb, tile_info, items, part_ml, part_o, total;
    long long groups_cap, tiles_cap, items_cap, parts_cap;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(long long num_reqs, long long num_tokens, int num_q_heads, int num_kv_heads,
                          int head_size, long long parts_cap) {
    WsLayout L{};
    const long long g = num_q_heads / num_kv_heads;
    L.groups_cap = (num_tokens * g + kRowsPerTile - 1) / kRowsPerTile + num_reqs;
    L.tiles_cap = L.groups_cap * num_kv_heads;
    L.parts_cap = parts_cap;
    L.items_cap = L.tiles_cap + parts_cap;
    size_t off = sizeof(WsHeader);
    L.req_group_base = off; off = align256(off + sizeof(int32_t) * (num_reqs + 1));
    L.group_kvb = off;      off = align256(off + sizeof(int32_t) * L.groups_cap);
    L.tile_info = off;      off = align256(off + sizeof(int2) * L.tiles_cap);
    L.items = off;          off = align256(off + sizeof(WorkItem) * L.items_cap);
    L.part_ml = off;        off = align256(off + sizeof(float2) * kRowsPerTile * parts_cap);
    L.part_o = off;         off = align256(off + sizeof(float) * kRowsPerTile * head_size * parts_cap);
    L.total = off;
    return L;
}

}  // namespace pkv
