/*
 * pkv.h -- libpagedkv: attention over a paged KV cache on one GB300 (sm_103a).
 *
 * The problem these calls implement is stated on the pages this library
 * follows:
 *   [KV2] "LLM KV cache part 2: KV management in serving engines"
 *         (ttlab.hopto.org), section 2 "PagedAttention: splitting KV into
 *         blocks" (subsections "Blocks and block tables", "Sharing blocks"),
 *         section 3 (continuous batching, chunked prefill).
 *   [ENG] "How LLM inference engines work: from one token to agent caches"
 *         (xiaohu-jiedu.pages.dev), sections "KV Cache", "PagedAttention",
 *         "Chunked Prefill".
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every array argument is a DEVICE pointer unless its name ends in
 *    `_host`.  The caller owns every buffer; the library allocates no device
 *    memory and keeps no state besides a per-device error word and cached
 *    device properties.
 *  - `stream` is a cudaStream_t passed as `void*` (NULL = legacy default
 *    stream).  Every call only enqueues work: PKV_OK means the arguments
 *    passed the host checks and the kernels were launched.  Errors found on
 *    the device (an out-of-range block id, slot or length; a bounded wait
 *    that expired) are recorded in the error word and read with
 *    pkv_get_error().  No kernel traps, asserts or waits without a limit;
 *    an invalid id is never dereferenced.
 *  - bf16 is IEEE bfloat16; out is fp32.
 *  - Device pointers must be 16-byte aligned.
 *  - Kernels are launched with programmatic stream serialization: one may
 *    start while the previous kernel on the stream finishes, but it reads and
 *    writes nothing in global memory (other than L2 prefetches) before that
 *    kernel has completed, so results are those of serialised launches.  The
 *    environment variable PKV_OVERLAP=0 turns this off.
 *
 * Cache layout ([KV2] section 2, "Blocks and block tables")
 * ----------------------------------------------------------
 * KV is cut into fixed blocks of 16 tokens that may sit anywhere in the pool;
 * each sequence's block table maps its logical block i to a physical block.
 * K and V are separate pools, each
 *     elem [num_blocks][num_kv_heads][16][head_dim]
 * with elem bf16 (2 bytes) or an 8-bit e4m3 code (pkv_cache_t.kv_dtype), so
 * the 16 rows of one (block, kv head) are one contiguous run of
 * 16*head_dim*sizeof(elem) bytes.  Token p of a sequence is row p % 16 of physical block
 * block_table[p / 16].  A slot id is block * 16 + row.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_NULL = 1,        /* a required pointer is NULL                                  */
    PKV_ERR_SHAPE = 2,       /* a count or size is negative or inconsistent                 */
    PKV_ERR_HEADS = 3,       /* num_q_heads / num_kv_heads is not one of 1, 2, 4, 8         */
    PKV_ERR_HEADDIM = 4,     /* head_dim is not 64 or 128                                   */
    PKV_ERR_BLOCKSIZE = 5,   /* block_size is not 16                                        */
    PKV_ERR_ALIAS = 6,       /* copy_blocks: a dst repeats, or a dst is also a src          */
    PKV_ERR_WORKSPACE = 7,   /* workspace NULL, too small or not 256-byte aligned           */
    PKV_ERR_ALIGN = 8,       /* a device pointer is not 16-byte aligned                     */
    PKV_ERR_RANGE = 9,       /* (device) block id, slot, length or V value out of range     */
    PKV_ERR_TIMEOUT = 10,    /* (device) a bounded wait inside a kernel expired             */
    PKV_ERR_CUDA = 11,       /* a CUDA runtime call failed (see pkv_last_cuda_error)        */
    PKV_ERR_UNSUPPORTED = 12, /* the current device is not compute capability 10.3          */
    PKV_ERR_SCRATCH_LIMIT = 13, /* the problem needs more than the built-in scratch buffer  */
    PKV_ERR_NO_BLOCKS = 14,  /* (device) the free queue cannot supply the blocks an append needs */
    PKV_ERR_HOST_MEMORY = 15, /* a host buffer is not page-locked memory mapped for the device   */
    PKV_ERR_DTYPE = 16       /* kv_dtype unknown, e4m3 scales not finite and > 0, or the call
                                does not take an e4m3 pool                                     */
} pkv_status;

/*
 * Element type of the pools.  PKV_KV_E4M3 halves the bytes decode reads:
 * each element is an 8-bit code of the OCP e4m3 format (sign, 4 exponent
 * bits with bias 7, 3 mantissa bits; subnormals; largest finite 448; S.1111.111
 * is NaN, no infinities), and stands for value(code) * scale, one scale per
 * pool.  The pages have no fp8 pool: it is the bandwidth-halving variant of
 * the write and the gather, chosen because decode reads the whole cache every
 * step ([ENG] "Prefill/Decode").
 */
enum { PKV_KV_BF16 = 0, PKV_KV_E4M3 = 1 };

typedef struct pkv_cache {
    void* k_pool;         /* elem [num_blocks][num_kv_heads][16][head_dim], device        */
    void* v_pool;         /* same layout                                                  */
    int32_t num_blocks;   /* physical blocks in each pool, >= 0                           */
    int32_t num_kv_heads; /* >= 1                                                         */
    int32_t head_dim;     /* 64 or 128                                                    */
    int32_t block_size;   /* tokens per block; must be 16 ([KV2] section 2 default)       */
    int32_t kv_dtype;     /* PKV_KV_BF16 (0, also what zero-initialisation gives) or
                             PKV_KV_E4M3                                                   */
    float k_scale;        /* e4m3 pools: K element = value(code) * k_scale; finite, > 0    */
    float v_scale;        /* e4m3 pools: V element = value(code) * v_scale; ignored for bf16 */
} pkv_cache_t;

/*
 * pkv_cache_write -- store this step's new K/V rows in their slots.
 * [ENG] "KV Cache": each step computes only the new token's K/V column and
 * keeps it, reading every past column from the cache; [KV2] section 2: the
 * token lands in its sequence's current block.
 *
 *   k_new, v_new  bf16 [num_tokens][num_kv_heads][head_dim]
 *   slot_mapping  int32 [num_tokens]; row t goes to slot slot_mapping[t]
 *                 (block slot/16, row slot%16) for every kv head; a negative
 *                 slot skips the row.  Slots within one call must be distinct.
 *   A slot >= num_blocks*16 is not written and raises PKV_ERR_RANGE on the
 *   device.  The copy is bit-exact.  num_tokens == 0 is a no-op.
 *   e4m3 pools: each element x is stored as the code nearest to
 *   x * (1/scale), where 1/scale is the fp32 reciprocal of the pool's scale
 *   and the product is rounded to fp32 first; ties go to the even code and
 *   values beyond 448 saturate to +-448 (a NaN gives a NaN code).
 */
pkv_status pkv_cache_write(const pkv_cache_t* cache, const void* k_new, const void* v_new,
                           const int32_t* slot_mapping, int32_t num_tokens, void* stream);

/*
 * pkv_copy_blocks -- copy-on-write of shared blocks.
 * [KV2] section 2, "Sharing blocks": requests may point at the same physical
 * block under a reference count; a block is copied only when someone must
 * append to it.  For every i: K[dst[i]] <- K[src[i]] and V[dst[i]] <- V[src[i]],
 * whole blocks (all kv heads, all 16 rows), bit-exact.
 *
 *   src, dst              int32 [num_pairs], device.  A pair whose src is
 *                         negative is skipped without error (the unused
 *                         entries pkv_blocks_append leaves are -1).
 *   src_host, dst_host    optional host copies of src/dst; when both are given
 *                         the call checks that the dst ids are distinct and
 *                         that no dst is also a src (PKV_ERR_ALIAS), and that
 *                         ids are in range (PKV_ERR_RANGE) before launching.
 *                         The same src may appear many times.
 *   Other ids out of range found on the device are skipped and raise
 *   PKV_ERR_RANGE.
 */
pkv_status pkv_copy_blocks(const pkv_cache_t* cache, const int32_t* src, const int32_t* dst, int32_t num_pairs,
                           const int32_t* src_host, const int32_t* dst_host, void* stream);

/*
 * pkv_swap_blocks -- move whole blocks between the pool and host memory (KV
 * offloading).  [ENG] "traffic characteristics and system control": a
 * request idle for seconds or minutes (an agent waiting on a tool) has its KV
 * cache swapped out to cheaper, larger CPU memory and swapped back in when
 * the next turn starts, instead of holding GPU memory; [KV2] section 5: a
 * request that loses its KV is otherwise prefilled again from the start.
 *
 *   direction      0 = out (pool -> host), 1 = in (host -> pool)
 *   blocks, slots  int32 [n], device: pair i moves pool block blocks[i] and
 *                  host slab slots[i]; a negative block id skips the pair
 *   host           page-locked host memory mapped for the device
 *                  (cudaHostAlloc, or cudaHostRegister with the mapped flag),
 *                  16-byte aligned, holding num_host_slots slabs of
 *                  [2][num_kv_heads][16][head_dim] pool elements (the K block, then the
 *                  V block); the kernel reads and writes it directly, over the
 *                  host link, bit-exact
 *   Returns PKV_ERR_HOST_MEMORY, launching nothing, when `host` is not such
 *   memory.  Block ids or slots out of range found on the device are skipped
 *   and raise PKV_ERR_RANGE.  n <= 65535 pairs per call.
 */
pkv_status pkv_swap_blocks(const pkv_cache_t* cache, int32_t direction, const int32_t* blocks, const int32_t* slots,
                           int32_t n, void* host, int64_t num_host_slots, void* stream);

/*
 * pkv_copy -- copy `bytes` bytes from src to dst with a kernel, for moving a
 * step's inputs in from host memory and its output back without the copy
 * engine: on a Grace system the GPU reads and writes page-locked host memory
 * directly over the host link, and a kernel chains with the launches around
 * it (programmatic serialization) where a copy-engine transfer cannot.
 * Not on the pages: the transfer helper of the end-to-end step.
 *
 *   dst, src   each device memory or page-locked host memory mapped for the
 *              device (cudaHostAlloc, or cudaHostRegister with the mapped
 *              flag); 16-byte aligned; they must not overlap
 *   bytes      a multiple of 16 (else PKV_ERR_SHAPE); 0 does nothing
 *   Returns PKV_ERR_HOST_MEMORY, launching nothing, for any other memory
 *   (pageable host memory).  Asynchronous on `stream`, like every call.
 */
pkv_status pkv_copy(void* dst, const void* src, size_t bytes, void* stream);

/*
 * pkv_decode_workspace_size -- bytes of workspace pkv_decode_attention needs
 * (a 256-byte header, one arrival counter per (sequence, kv head) and the
 * split-KV partial results).  Depends on the current device's SM count.
 * partition_blocks: 0 = automatic, else the number of (sequence, kv head,
 * 16-token block) units per work range (see pkv_decode_attention).
 * Returns 0 for invalid arguments.
 */
size_t pkv_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t max_context_len, int32_t partition_blocks);

/*
 * pkv_decode_attention -- one query token per sequence over its paged context.
 * [KV2] section 2, "Blocks and block tables": the kernel follows the block
 * table and reads K/V from scattered blocks; the result equals attention over
 * one contiguous array.  [ENG] "Prefill/Decode": decode reads the whole
 * context cache every step and is memory-bandwidth bound.
 *
 *   For sequence s with n = context_lens[s] (this step's token already
 *   written, so it attends to itself) and q head h (kv head h / (Hq/Hkv)):
 *       out[s][h] = softmax_j(scale * q[s][h] . K_j) V_j,   j = 0 .. n-1
 *   with K_j, V_j row j % 16 of block block_tables[s][j / 16].
 *
 *   q              bf16 [num_seqs][num_q_heads][head_dim]
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]
 *   context_lens   int32 [num_seqs]; 0 gives a zero output row; a value above
 *                  max_blocks_per_seq*16 or max_context_len is clamped and
 *                  raises PKV_ERR_RANGE
 *   max_context_len host-side upper bound of context_lens (sizes the split)
 *   out            fp32 [num_seqs][num_q_heads][head_dim]: device memory,
 *                  or page-locked host memory mapped for the device (the
 *                  kernel then writes the rows there directly, with no copy
 *                  after it); other host memory gives PKV_ERR_HOST_MEMORY
 *   workspace      device buffer of >= pkv_decode_workspace_size() bytes,
 *                  256-byte aligned, ZERO-FILLED BEFORE ITS FIRST USE.  Its
 *                  first part (a 256-byte header and one arrival counter per
 *                  (sequence, kv head)) must be zero when a call starts, and
 *                  every call that completes without PKV_ERR_TIMEOUT leaves
 *                  it zero again, so the same workspace serves the next call
 *                  as is; the rest holds split-KV partial results and is
 *                  scratch.  After a call that reported PKV_ERR_TIMEOUT,
 *                  zero-fill the workspace again before reusing it (a part
 *                  that gave up may leave its pair's counter raised).  Calls
 *                  that run concurrently need separate workspaces.
 *   partition_blocks 0 = automatic; > 0 forces the size of a work range in
 *                  units (the workspace must be sized with the same value).
 *   Work is the sequence of units (sequence, kv head, 16-token block) cut
 *   into equal ranges, one per SM by default; a (sequence, kv head) whose
 *   blocks straddle ranges is computed as split-KV partitions whose partial
 *   results are merged with the log-sum-exp rule inside the same launch, in
 *   a fixed order (results are bitwise reproducible).
 *   e4m3 pools: K_j and V_j are value(code) * k_scale and value(code) *
 *   v_scale, exactly as pkv_cache_write defines them (a NaN code, which that
 *   call never stores for finite input, reads as NaN).
 */
pkv_status pkv_decode_attention(const pkv_cache_t* cache, const void* q, int32_t num_q_heads,
                                const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
                                int32_t num_seqs, int32_t max_context_len, float scale, float* out, void* workspace,
                                size_t workspace_bytes, int32_t partition_blocks, void* stream);

/*
 * pkv_decode_step -- one decode step in one launch: the store of each
 * sequence's new K/V row (pkv_cache_write) and decode attention over the
 * context that includes it (pkv_decode_attention).  [ENG] "KV Cache": a
 * step computes only the new token's column, keeps it, and attends over all
 * the columns; [KV2] section 2: the new token lands in its sequence's
 * current (last) block.
 *
 *   k_new, v_new   bf16 [num_seqs][num_kv_heads][head_dim]: row s is the new
 *                  token of sequence s, at position context_lens[s] - 1
 *   slot_mapping   int32 [num_seqs]: the slot of that position, i.e.
 *                  block_tables[s][(n-1)/16] * 16 + (n-1) % 16 with
 *                  n = context_lens[s]; a negative slot skips the store (the
 *                  pool's row at that position is then used as it is)
 *   All other arguments, the workspace rules and the result are those of
 *   pkv_decode_attention; the pools end as pkv_cache_write leaves them.
 *   The result equals pkv_cache_write(cache, k_new, v_new, slot_mapping,
 *   num_seqs) followed by pkv_decode_attention(...).  A non-negative slot
 *   that is not the slot of position n - 1 is not written and raises
 *   PKV_ERR_RANGE (detail: the sequence); that sequence then attends over
 *   the pool's row as it is.  The new rows' blocks must not be read by other
 *   sequences of the batch (they are the sequences' own last blocks, as
 *   copy-on-write guarantees).  e4m3 pools store code(x * (1/scale)) as
 *   pkv_cache_write does and attend over those codes.
 */
pkv_status pkv_decode_step(const pkv_cache_t* cache, const void* k_new, const void* v_new,
                           const int32_t* slot_mapping, const void* q, int32_t num_q_heads,
                           const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t num_seqs, int32_t max_context_len, float scale, float* out, void* workspace,
                           size_t workspace_bytes, int32_t partition_blocks, void* stream);

/*
 * pkv_decode_attention_shared_prefix -- pkv_decode_attention for a batch
 * whose sequences all begin with the same blocks.  [KV2] section 2,
 * "Sharing blocks": several requests may point at one physical block (a
 * prompt shared by parallel samples or beams, a system prompt the prefix
 * cache maps to the same blocks).  The first shared_blocks entries of every
 * block table are read once per kv head and attended by the queries of all
 * sequences together on tensor cores; each sequence's remaining blocks are
 * attended by the decode kernel, which merges both parts (log-sum-exp).
 *
 *   shared_blocks  host int32: block_tables[s][j] is the same id for every
 *                  s and every j < shared_blocks, and each context holds
 *                  those blocks in full (context_lens[s] >= 16 *
 *                  shared_blocks).  0 <= shared_blocks <= max_blocks_per_seq
 *                  and 16 * shared_blocks <= max_context_len, else
 *                  PKV_ERR_SHAPE.  pkv_common_prefix_blocks computes the
 *                  largest such value from host copies of the tables.
 *   workspace      device buffer of >= pkv_decode_shared_prefix_workspace_size()
 *                  bytes, 256-byte aligned, under the rules of
 *                  pkv_decode_attention (zero on first use; left zeroed).
 *   All other arguments and the result are those of pkv_decode_attention
 *   (automatic partitioning).  The result equals pkv_decode_attention's up
 *   to fp32 rounding (the shared part's P is carried as a bf16 hi + lo pair,
 *   2^-17 relative).
 *   The promise is checked on the device: a sequence whose table differs in
 *   the shared part, or whose context is shorter than it, raises
 *   PKV_ERR_RANGE (detail: the sequence), and the call's results are then
 *   not valid.  e4m3 pools, pools of more than 2^31 rows of 16 tokens x kv
 *   heads, and devices that refuse the kernel's 8-CTA clusters attend the
 *   shared blocks per sequence, as pkv_decode_attention does; the promise is
 *   then not checked.
 */
size_t pkv_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                               int32_t head_dim, int32_t max_context_len, int32_t shared_blocks);
pkv_status pkv_decode_attention_shared_prefix(const pkv_cache_t* cache, const void* q, int32_t num_q_heads,
                                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                                              const int32_t* context_lens, int32_t num_seqs,
                                              int32_t max_context_len, int32_t shared_blocks, float scale,
                                              float* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pkv_common_prefix_blocks -- host-only: the largest J such that the first J
 * entries of every row of block_tables_host ([num_seqs][max_blocks_per_seq])
 * equal row 0's and every context_lens_host[s] >= 16 J.  Reads host memory
 * only; 0 when num_seqs <= 0, a pointer is NULL or max_blocks_per_seq <= 0.
 */
int32_t pkv_common_prefix_blocks(const int32_t* block_tables_host, int32_t max_blocks_per_seq,
                                 const int32_t* context_lens_host, int32_t num_seqs);

/*
 * pkv_prefill_workspace_size -- bytes of workspace
 * pkv_chunked_prefill_attention needs.  Returns 0 for invalid arguments.
 */
size_t pkv_prefill_workspace_size(int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_context_len);

/*
 * pkv_chunked_prefill_attention -- attention of a mixed batch.
 * [ENG] "Chunked Prefill": a long prompt is split into slices under a
 * per-step token budget, and each slice shares its forward pass with the
 * single decode tokens of the active users; [KV2] section 3 (chunks mixed
 * with decode tokens).
 *
 *   Sequence s owns query rows query_start_loc[s] .. query_start_loc[s+1]-1
 *   (query_len = their count).  Row i sits at absolute position
 *   pos = context_lens[s] - query_len + i and attends keys 0..pos (causal),
 *   read through the block table; the chunk's own K/V must already be in the
 *   cache (pkv_cache_write first).  query_len == 1 rows are decode rows.
 *
 *   q                     bf16 [num_tokens][num_q_heads][head_dim]
 *   query_start_loc       int32 [num_seqs+1], device
 *   query_start_loc_host  the same values on the host (plans the launch)
 *   context_lens          int32 [num_seqs], device, including this step's rows
 *   out                   fp32 [num_tokens][num_q_heads][head_dim], device
 *                         memory or page-locked host memory mapped for the
 *                         device (as for pkv_decode_attention)
 *   workspace             >= pkv_prefill_workspace_size() bytes, 256-byte
 *                         aligned, zero-filled before first use; used as the
 *                         decode workspace for the decode rows (its counters
 *                         are left zero, so it is reused as is)
 *   Query rows are computed on tcgen05 tensor cores: Q.K^T in bf16, P.V in
 *   fp16 (P rounded to fp16, V converted from bf16, exact for 2^-14 <= |v|
 *   <= 65504); decode rows take the decode kernel.  A tile of 128 query rows
 *   (of one or two q heads) whose visible V values leave that range (some
 *   |v| > 65504, or every |v| < 2^-12) is recomputed in the same launch in
 *   fp32 on CUDA cores, so every finite bf16 V is accepted (|v| up to about
 *   1e36, where fp32 sums of weighted rows overflow), at a lower speed for
 *   such tiles.  head_dim 64 or 128.  Takes bf16 pools only (an e4m3 pool:
 *   PKV_ERR_DTYPE).
 */
pkv_status pkv_chunked_prefill_attention(const pkv_cache_t* cache, const void* q, int32_t num_q_heads,
                                         int32_t num_tokens, const int32_t* query_start_loc,
                                         const int32_t* query_start_loc_host, const int32_t* context_lens,
                                         int32_t num_seqs, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         int32_t max_context_len, float scale, float* out, void* workspace,
                                         size_t workspace_bytes, void* stream);

/*
 * pkv_decode_attention_static -- pkv_decode_attention for callers that
 * cannot allocate device memory.  The pages have no counterpart of this
 * call; it exists for code that may not call cudaMalloc at the point where
 * it decodes (host callbacks and other paths where allocation is forbidden,
 * plug-ins that do not own the process's memory pool, runtimes that freeze
 * device allocation after start-up).  It allocates nothing: its workspace is
 * a fixed buffer of pkv_decode_static_scratch_bytes() bytes (4 MiB) that the
 * library keeps on every GPU that loads it, until the process exits.  The
 * caller still passes every input and the output, with the meaning they have
 * in pkv_decode_attention (automatic partitioning).
 *
 *   - Returns PKV_ERR_SCRATCH_LIMIT, launching nothing, when the batch needs
 *     more workspace than the buffer holds (pkv_decode_workspace_size with
 *     partition_blocks = 0 tells the need).
 *   - The first call on a device looks up the buffer's device address with
 *     that device current; make that first call before any stream capture.
 *   - Each call clears the buffer's counters on `stream` before launching.
 *   - All calls on a device share the one buffer: calls whose work overlaps
 *     on the GPU (different streams, no ordering between them) race on it
 *     and give wrong results.  Order them on one stream, or use
 *     pkv_decode_attention with separate workspaces.
 */
pkv_status pkv_decode_attention_static(const pkv_cache_t* cache, const void* q, int32_t num_q_heads,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, int32_t num_seqs, int32_t max_context_len,
                                       float scale, float* out, void* stream);

/* Size in bytes of the built-in scratch buffer pkv_decode_attention_static uses. */
size_t pkv_decode_static_scratch_bytes(void);

/*
 * Block bookkeeping on the device.
 * [KV2] section 2, "Blocks and block tables": a request's KV is cut into
 * 16-token blocks that may sit anywhere in free memory; its block table maps
 * logical to physical blocks, and a block is allocated at the moment the
 * tokens fill the last one (nothing is reserved ahead).  "Sharing blocks":
 * requests may point at one block under a reference count, and a shared block
 * is copied only when a holder must append to it (copy-on-write).  [KV2]
 * section 4: a finished request's blocks return to the free queue tail block
 * first.
 *
 * The state is caller-owned device memory; rows of the tables are sequences.
 * block_tables and context_lens are the arrays the attention calls read, so
 * a step is: pkv_blocks_append -> pkv_copy_blocks (its pairs) ->
 * pkv_cache_write (its slot mapping) -> attention, with no host round trip.
 * Every call is one launch on `stream`; device-side failures are recorded in
 * the error word (pkv_get_error) and leave the state unchanged.
 *
 * Prefix cache ([KV2] section 4), when block_keys/key_table/cached are given:
 * a block registered with its key (pkv_blocks_register) keeps its content and
 * key after its last holder releases it ("empty but content kept"), waiting
 * in the free queue in least-recently-freed order; a new row whose leading
 * keys are cached takes those blocks (pkv_blocks_match), taking a free one
 * back out of the queue; an append that takes a cached block from the queue
 * drops its key.  The free queue is a ring of 2 * num_blocks entries: a block
 * taken back by a match leaves a stale entry (ring_pos no longer points at
 * it), which pops skip and a release compacts away when the ring would
 * overflow.  Keys come from pkv_prefix_keys.
 */
typedef struct pkv_blocks {
    int32_t* block_tables;   /* int32 [max_seqs][max_blocks_per_seq]; -1 = no block          */
    int32_t* context_lens;   /* int32 [max_seqs]: tokens each row holds                      */
    int32_t* ref_counts;     /* int32 [num_blocks]: rows holding each block                  */
    int32_t* free_ring;      /* int32 [2 * num_blocks]: the free queue, least recently freed
                                first (a ring that may hold stale entries, see below)         */
    int32_t* ring_pos;       /* int32 [num_blocks]: ring index of a free block, -1 if held    */
    int32_t* free_state;     /* int32 [3]: {head, ring entries, free blocks}                  */
    int32_t* scratch;        /* int32 [3 * num_blocks]; the first 2 * num_blocks are zero
                                between calls (pkv_blocks_reset zeroes them)                  */
    uint8_t* block_keys;     /* uint8 [num_blocks][32] prefix-cache keys, 16-byte aligned,
                                or NULL: no prefix cache                                      */
    int32_t* key_table;      /* int32 [table_size]: cached blocks by key, or NULL             */
    int32_t* cached;         /* int32 [num_blocks]: 1 = the block's key is in key_table, or NULL */
    int32_t num_blocks;      /* >= 0                                                          */
    int32_t max_seqs;        /* rows, >= 0                                                    */
    int32_t max_blocks_per_seq; /* >= 1                                                       */
    int32_t table_size;      /* power of two >= 2 * num_blocks, or 0 without a prefix cache  */
} pkv_blocks_t;

/*
 * pkv_blocks_reset -- every row empty (tables -1, lengths 0), every count 0,
 * the free queue holding blocks 0, 1, ..., num_blocks-1 in that order,
 * scratch 0, the prefix cache empty.
 */
pkv_status pkv_blocks_reset(const pkv_blocks_t* blocks, void* stream);

/*
 * pkv_blocks_append -- row s (0 <= s < num_seqs) gains
 * query_start_loc[s+1] - query_start_loc[s] tokens (0 = untouched).
 *
 *   query_start_loc  int32 [num_seqs+1], device; [0] must be 0 and
 *                    [num_seqs] == num_tokens (host value), non-decreasing
 *   slot_mapping     int32 [num_tokens] out: slot (block*16 + row) of each new
 *                    token, the input of pkv_cache_write
 *   cow_src, cow_dst int32 [num_seqs] out: copy-on-write pairs in sequence
 *                    order, then -1 (pkv_copy_blocks with num_pairs = num_seqs
 *                    copies exactly these)
 *   cow_count        int32 [1] out: number of pairs
 *
 *   Sequences are processed as if one after another in index order:
 *   - a row whose last block is partly filled and held by others copies it
 *     into a new block (the pair is emitted and the old block loses a
 *     holder); when every holder appends in the same call, the last one
 *     writes in place;
 *   - new blocks (one per 16 tokens crossing a block boundary) and the
 *     copy-on-write blocks come from the free queue's head in that order; a
 *     cached block taken this way loses its key.
 *   Errors, found on the device, change no state; slot_mapping is then all
 *   -1 and the pairs all -1 (so the cache write and copies that follow do
 *   nothing):
 *   - PKV_ERR_RANGE: query_start_loc malformed, a length beyond
 *     max_blocks_per_seq*16, a partly filled last block not held, or more
 *     appenders than holders;
 *   - PKV_ERR_NO_BLOCKS: the free queue holds fewer blocks than the call needs.
 *   num_seqs <= max_seqs (else PKV_ERR_SHAPE).
 */
pkv_status pkv_blocks_append(const pkv_blocks_t* blocks, const int32_t* query_start_loc, int32_t num_seqs,
                             int32_t num_tokens, int32_t* slot_mapping, int32_t* cow_src, int32_t* cow_dst,
                             int32_t* cow_count, void* stream);

/*
 * pkv_blocks_fork -- row children[i] takes row parents[i]'s blocks and
 * length (parallel sampling, beam search: [KV2] "Sharing blocks"); each
 * shared block gains a holder.  n <= 4096 (else PKV_ERR_SHAPE).  Device
 * errors: PKV_ERR_RANGE (a row out of range, a child not empty, a parent's
 * block not held), PKV_ERR_ALIAS (children repeat, or a child is a parent).
 */
pkv_status pkv_blocks_fork(const pkv_blocks_t* blocks, const int32_t* parents, const int32_t* children, int32_t n,
                           void* stream);

/*
 * pkv_blocks_match -- prefix-cache hits.  Rows s < num_seqs with
 * num_keys[s] > 0 (each must be empty) take the cached blocks of their
 * leading keys keys[s][0 .. matched[s]), stopping at the first key not
 * cached; a block nobody holds leaves the free queue; the row's length
 * becomes 16 * matched[s].  Rows with num_keys[s] == 0 are untouched.
 *
 *   keys       uint8 [num_seqs][key_stride][32], device, 16-byte aligned
 *              (the layout pkv_prefix_keys writes, key_stride = its max_blocks)
 *   num_keys   int32 [num_seqs], device
 *   matched    int32 [num_seqs] out
 *   num_seqs <= min(max_seqs, 4096).  Device errors (PKV_ERR_RANGE): a row with
 *   keys that is not empty, or num_keys beyond key_stride or the table width.
 */
pkv_status pkv_blocks_match(const pkv_blocks_t* blocks, const void* keys, int32_t key_stride,
                            const int32_t* num_keys, int32_t num_seqs, int32_t* matched, void* stream);

/*
 * pkv_blocks_register -- rows s < num_seqs give their first num_keys[s]
 * blocks (full ones) the keys keys[s][0 .. num_keys[s]), in (row, block)
 * order: a block that already has a key keeps it, and a key already cached
 * (or given to an earlier row or block of the call) keeps its block.
 * num_seqs <= min(max_seqs, 4096).  Device errors (PKV_ERR_RANGE):
 * num_keys beyond the row's full blocks or key_stride, a block not held.
 */
pkv_status pkv_blocks_register(const pkv_blocks_t* blocks, const void* keys, int32_t key_stride,
                               const int32_t* num_keys, int32_t num_seqs, void* stream);

/*
 * pkv_blocks_release -- rows[i] (in order) drop their blocks, each row's
 * last block first; a block whose count reaches 0 joins the free queue's
 * tail, keeping its content and (if registered) its key.
 * The rows end empty.  n <= 4096 (else PKV_ERR_SHAPE).  Device errors:
 * PKV_ERR_RANGE (a row out of range, a block not held, more releases than
 * holders), PKV_ERR_ALIAS (a row repeats).
 */
pkv_status pkv_blocks_release(const pkv_blocks_t* blocks, const int32_t* rows, int32_t n, void* stream);

/*
 * pkv_prefix_keys -- prefix-cache keys of the full blocks of a batch of
 * token lists.  [KV2] section 4, "Prefix cache": a block's key hashes the
 * previous block's key, the block's token ids and extra information (adapter,
 * multimodal hashes, a per-user cache salt), so a key stands for the whole
 * prefix up to its block; only full blocks are keyed; SHA-256 by default.
 *
 *   key_i = SHA-256(key_{i-1} || the block's 16 token ids as little-endian
 *           int32 || extra[s] as little-endian int64)   (104-byte message)
 *   key_{-1} = parent_keys[s] (continuing a chain), or 32 zero bytes.
 *
 *   token_ids        int32 [T], device
 *   token_start_loc  int32 [num_seqs+1], device: sequence s owns
 *                    token_ids[token_start_loc[s] .. token_start_loc[s+1])
 *   extra            int64 [num_seqs], device, or NULL (all 0)
 *   parent_keys      uint8 [num_seqs][32], device, or NULL; 16-byte aligned
 *   keys             uint8 [num_seqs][max_blocks][32] out, 16-byte aligned:
 *                    the key of full block i of sequence s at [s][i] (the
 *                    32-byte digest); entries past its full blocks untouched
 *   A sequence with a decreasing range or more than max_blocks full blocks
 *   writes no key and raises PKV_ERR_RANGE (detail: the sequence).  Keys
 *   depend on each other along a sequence: one thread hashes one sequence.
 */
pkv_status pkv_prefix_keys(const int32_t* token_ids, const int32_t* token_start_loc, const int64_t* extra,
                           const void* parent_keys, int32_t num_seqs, int32_t max_blocks, void* keys, void* stream);

/*
 * pkv_test_arm_decode_stall -- test hook for the bounded waits; no page
 * describes it.  The next `launches` decode launches of this process (those
 * of pkv_decode_attention, pkv_decode_attention_static and the decode rows of
 * pkv_chunked_prefill_attention, on any device) run with a producer warp that
 * issues no work: their other warps wait for work descriptors that never
 * arrive, give up after the bounded wait (2 s), and the launch records
 * PKV_ERR_TIMEOUT (detail: the wait site).  Nothing is copied or in flight
 * when they leave; the output is not written and the workspace is left as it
 * was.  0 disarms.  Returns PKV_ERR_SHAPE for a negative count.
 */
pkv_status pkv_test_arm_decode_stall(int32_t launches);

/*
 * pkv_get_error -- synchronise `stream`, then return (and clear) the first
 * error a kernel recorded on the current device since the last call:
 * PKV_OK, PKV_ERR_RANGE, PKV_ERR_ALIAS, PKV_ERR_NO_BLOCKS or PKV_ERR_TIMEOUT.
 * `detail` (optional) receives
 * the offending index (a token, pair or sequence number) or wait site.
 */
pkv_status pkv_get_error(void* stream, int32_t* detail);

/* Human-readable name of a status code (static storage). */
const char* pkv_status_string(pkv_status status);

/* Text of the last CUDA runtime error seen by this thread (static storage). */
const char* pkv_last_cuda_error(void);

/* Library version, "major.minor.patch". */
const char* pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
