// Interface between the attention host code and the tcgen05 chunk kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attention_plan.cuh"

namespace pkv {

// a = {r, 128-row tile mt, kv head h, keys seen by the tile's last row},
// b = {qstart, n, L, valid rows of the tile}.
struct ChunkItem {
    int4 a, b;
};

struct ChunkArgs {
    const int32_t *block_table;
    int max_blocks_per_req, num_blocks, num_q_heads, num_kv_heads, group;
    float scale_log2;
    const ChunkItem *items;
    WsHeader *header;
    __nv_bfloat16 *out;
    int beside;  // running beside the split-KV kernel: only the first header->chunk_ctas CTAs work
};

int chunk_smem_bytes(int head_size);
int chunk_configure();  // kernel attributes; once per device
cudaError_t chunk_launch(int head_size, int grid, const CUtensorMap &kv_map, const CUtensorMap &q_map,
                         const ChunkArgs &args, cudaStream_t stream);

}  // namespace pkv
