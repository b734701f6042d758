// Causal attention of a prefill chunk (ql_chunk_attn.cu): the internal launch interface.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace ql {

struct ChunkAttnArgs {
    const __half* q;              // [T][n_heads][head_dim], normalised and rotated
    const __half* k_pool;         // this layer's pools [num_blocks][n_kv_heads][16][head_dim]
    const __half* v_pool;
    const int32_t* block_table;   // the sequence's row [max_blocks_per_seq]
    const int32_t* position;      // device: position of the chunk's first token
    int T, n_heads, n_kv_heads, head_dim, max_blocks_per_seq, num_blocks;
    float scale;
    __half* out;                  // [T][n_heads * head_dim]
    void* workspace;              // chunk_attn_workspace_bytes
    size_t workspace_bytes;
};

size_t chunk_attn_workspace_bytes(int T, int n_heads, int n_kv_heads, int head_dim);
int chunk_attn_launch(const ChunkAttnArgs& a, cudaStream_t s, bool pdl);

}  // namespace ql
