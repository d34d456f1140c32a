// pkv_internal.h -- host-side declarations shared by the libpagedkv
// translation units (kernel launchers and the C-ABI layer).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace pkv {

// Split-KV decode launch description (everything already validated).
struct DecodeArgs {
    const void* k_pool;
    const void* v_pool;
    const void* q;                 // bf16 rows of [rows][Hq][d]
    const int32_t* block_tables;   // [S][max_blocks]
    const int32_t* context_lens;   // [S]
    const int32_t* query_start_loc;// [S+1] or null: row of sequence s is s
    float* out;                    // fp32 [rows][Hq][d]
    void* workspace;               // zeroed-on-entry scratch (see decode_ws_layout)
    unsigned long long* err;       // device error word
    int32_t num_blocks, num_kv_heads, num_q_heads, head_dim;
    int32_t num_seqs, max_blocks_per_seq, max_context_len;
    int32_t part_blocks;           // blocks per split-KV partition (>= 1)
    int32_t max_parts;             // ceil(ceil(max_context_len/16) / part_blocks), >= 1
    float scale;
    int32_t grid;                  // persistent CTAs
};

struct DecodeWsLayout {
    size_t header;      // offset of the 256-byte header (work / done counters)
    size_t counters;    // uint32 [S][Hkv]
    size_t part_ml;     // float2 [S][Hq][max_parts]
    size_t part_o;      // float [S][Hq][max_parts][d]
    size_t total;
};

DecodeWsLayout decode_ws_layout(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t max_parts);

// Blocks per partition chosen for a launch (req > 0 forces it).
int32_t plan_part_blocks(int32_t num_seqs, int32_t num_kv_heads, int32_t max_context_len, int32_t num_sms,
                         int32_t req);

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

cudaError_t launch_cache_write(const void* k_new, const void* v_new, const int32_t* slot_mapping, int32_t num_tokens,
                               void* k_pool, void* v_pool, int32_t num_blocks, int32_t num_kv_heads,
                               int32_t head_dim, unsigned long long* err, cudaStream_t stream);

cudaError_t launch_copy_blocks(const int32_t* src, const int32_t* dst, int32_t num_pairs, void* k_pool,
                               void* v_pool, int32_t num_blocks, int32_t num_kv_heads, int32_t head_dim,
                               unsigned long long* err, cudaStream_t stream);

// Chunked prefill (tcgen05) launch description.
struct PrefillArgs {
    const void* k_pool;
    const void* v_pool;
    const void* q;                    // bf16 [num_tokens][Hq][d]
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* query_start_loc;   // device [S+1]
    float* out;
    unsigned long long* err;
    int32_t num_blocks, num_kv_heads, num_q_heads, head_dim;
    int32_t num_seqs, num_tokens, max_blocks_per_seq, max_context_len;
    int32_t num_tiles;                // query tiles of the prefill sequences
    float scale;
};

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);

}  // namespace pkv
