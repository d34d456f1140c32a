// pkv_internal.h -- host-side declarations shared by the libpagedkv
// translation units (kernel launchers and the C-ABI layer).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pkv {

// How a decode launch cuts its work: the units (sequence, kv head, 16-token
// block) are split into ranges of range_units consecutive units (0 = one
// range per CTA, computed on the device from context_lens).
struct DecodePlan {
    int32_t range_units;
    int32_t max_ranges;  // ranges the workspace must hold
    int32_t grid;        // persistent CTAs
};

DecodePlan plan_decode_ranges(int32_t num_seqs, int32_t num_kv_heads, int32_t max_context_len, int32_t num_sms,
                              int32_t req_range_units);

// Split-KV decode launch description (everything already validated).
struct DecodeArgs {
    void* k_pool;                  // written only by a fused step (its new rows)
    void* v_pool;
    const void* q;                 // bf16 rows of [rows][Hq][d]
    const int32_t* block_tables;   // [S][max_blocks]
    const int32_t* context_lens;   // [S]
    const int32_t* query_start_loc;// [S+1] or null: row of sequence s is s
    float* out;                    // fp32 [rows][Hq][d]
    void* workspace;               // zeroed-on-entry scratch (see decode_ws_layout)
    unsigned long long* err;       // device error word
    int32_t num_blocks, num_kv_heads, num_q_heads, head_dim;
    int32_t num_seqs, max_blocks_per_seq, max_context_len;
    DecodePlan plan;
    float scale;
    bool kv_e4m3;                  // pools hold e4m3 codes (else bf16)
    float k_scale, v_scale;        // e4m3 pools: element = code value * scale
    // Fused step: each sequence's new row (bf16 [S][Hkv][d]) and its slot,
    // stored and used in the same launch; all null for plain decode.
    const void* k_new = nullptr;
    const void* v_new = nullptr;
    const int32_t* slot_mapping = nullptr;
    // Shared prefix: every sequence's first skip_blocks blocks are attended
    // by launch_shared_prefix (prefix_chunks CTAs per kv head and query
    // tile, one cluster), which leaves one state per (sequence, q head) in
    // the workspace; decode attends the rest and merges.  0 for plain decode.
    int32_t skip_blocks = 0;
    int32_t prefix_chunks = 0;
};

struct DecodeWsLayout {
    size_t header;      // 256 reserved bytes
    size_t counters;    // uint32 [S][Hkv] arrival tickets
    size_t part_ml;     // float2 [max_ranges][2][G]
    size_t part_o;      // float [max_ranges][2][G][d]
    size_t pre_ml;      // shared prefix: float2 [S][Hq] (m, l) of the shared blocks
    size_t pre_o;       //                float [S][Hq][d] their unnormalised o
    size_t total;
};

DecodeWsLayout decode_ws_layout(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t max_ranges, bool prefix = false);

// Shared-prefix decode: CTAs (one cluster) that split the shared blocks of
// one kv head and query tile (0 when shared_blocks is 0).
int32_t shared_prefix_chunks(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t shared_blocks);

// The shared blocks' state per (sequence, q head) for a decode launch `a`
// (a.skip_blocks shared blocks in a.prefix_chunks chunks, bf16 pools);
// launch it right before launch_decode(a) on the same stream.
cudaError_t launch_shared_prefix(const DecodeArgs& a, cudaStream_t stream);

// A tiled tensor map with the 128-byte swizzle (element type dtype, or bf16).
bool make_tile_map(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, cuuint32_t rank,
                   const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box);
bool make_bf16_map(CUtensorMap* map, const void* base, cuuint32_t rank, const cuuint64_t* dims,
                   const cuuint64_t* strides_bytes, const cuuint32_t* box);

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
// The fused step's variant (a.k_new set), called by launch_decode.
cudaError_t launch_decode_fused(const DecodeArgs& a, bool stall, cudaStream_t stream);

// Test hook: the next `launches` decode launches run with a producer warp
// that issues nothing, so their other warps time out (PKV_ERR_TIMEOUT).
void arm_decode_stall(int32_t launches);

cudaError_t launch_cache_write(const void* k_new, const void* v_new, const int32_t* slot_mapping, int32_t num_tokens,
                               void* k_pool, void* v_pool, int32_t num_blocks, int32_t num_kv_heads,
                               int32_t head_dim, unsigned long long* err, cudaStream_t stream);

// e4m3 pools: code(bf16 value * inv_scale), the product in fp32, nearest
// even, saturating to +-448.
cudaError_t launch_cache_write_e4m3(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                                    int32_t num_tokens, void* k_pool, void* v_pool, int32_t num_blocks,
                                    int32_t num_kv_heads, int32_t head_dim, float k_inv_scale, float v_inv_scale,
                                    unsigned long long* err, cudaStream_t stream);

// elem_bytes: 2 for bf16 pools, 1 for e4m3 pools.
cudaError_t launch_copy_blocks(const int32_t* src, const int32_t* dst, int32_t num_pairs, void* k_pool,
                               void* v_pool, int32_t num_blocks, int32_t num_kv_heads, int32_t head_dim,
                               int32_t elem_bytes, unsigned long long* err, cudaStream_t stream);

// Copy `chunks` 16-byte chunks from src to dst (device addresses) with a
// kernel.
cudaError_t launch_copy16(void* dst, const void* src, int64_t chunks, int num_sms, cudaStream_t stream);

cudaError_t launch_swap_blocks(int32_t direction, const int32_t* blocks, const int32_t* slots, int32_t n,
                               void* host, int64_t num_slots, void* k_pool, void* v_pool, int32_t num_blocks,
                               int32_t num_kv_heads, int32_t head_dim, int32_t elem_bytes, unsigned long long* err,
                               cudaStream_t stream);

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
    int32_t split_last;               // last row tiles of each sequence split by head (two-head CTAs only)
    int32_t split_tiles;              // tiles so split over all sequences (extra CTAs per head pair)
    float scale;
};

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);

// Block bookkeeping state (pkv_blocks_t), all device memory.
struct BlocksArgs {
    int32_t* tables;      // [max_seqs][max_blocks]
    int32_t* lens;        // [max_seqs]
    int32_t* refs;        // [num_blocks]
    int32_t* free_ring;   // [2 * num_blocks] ring of free block ids (LRU order; stale entries skipped)
    int32_t* ring_pos;    // [num_blocks] ring index of a free block's live entry, -1 when held
    int32_t* free_state;  // [3] {head, entries, free blocks}
    int32_t* scratch;     // [3 * num_blocks]; the first 2 * num_blocks zero between calls
    uint8_t* block_keys;  // [num_blocks][32] prefix-cache keys, or null (no prefix cache)
    int32_t* key_table;   // [table_size] block ids by key (linear probing, -1 empty), or null
    int32_t* cached;      // [num_blocks] 1 if the block's key is in the table, or null
    int32_t num_blocks, max_seqs, max_blocks, table_size;
};

// Rows per fork or release call (the kernels keep per-row offsets on chip).
constexpr int32_t kBlocksMaxRows = 4096;

cudaError_t launch_blocks_reset(const BlocksArgs& st, cudaStream_t stream);
cudaError_t launch_blocks_append(const BlocksArgs& st, const int32_t* query_start_loc, int32_t num_seqs,
                                 int32_t num_tokens, int32_t* slot_mapping, int32_t* cow_src, int32_t* cow_dst,
                                 int32_t* cow_count, unsigned long long* err, cudaStream_t stream);
cudaError_t launch_blocks_fork(const BlocksArgs& st, const int32_t* parents, const int32_t* children, int32_t n,
                               unsigned long long* err, cudaStream_t stream);
cudaError_t launch_prefix_keys(const int32_t* token_ids, const int32_t* token_start_loc, const int64_t* extra,
                               const uint8_t* parent_keys, int32_t num_seqs, int32_t max_blocks, uint8_t* keys,
                               unsigned long long* err, cudaStream_t stream);
cudaError_t launch_blocks_match(const BlocksArgs& st, const uint8_t* keys, int32_t key_stride,
                                const int32_t* num_keys, int32_t num_seqs, int32_t* matched,
                                unsigned long long* err, cudaStream_t stream);
cudaError_t launch_blocks_register(const BlocksArgs& st, const uint8_t* keys, int32_t key_stride,
                                   const int32_t* num_keys, int32_t num_seqs, unsigned long long* err,
                                   cudaStream_t stream);
cudaError_t launch_blocks_release(const BlocksArgs& st, const int32_t* rows, int32_t n, unsigned long long* err,
                                  cudaStream_t stream);

}  // namespace pkv
