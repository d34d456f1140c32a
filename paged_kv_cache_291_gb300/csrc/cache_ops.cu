// cache_ops.cu -- the two cache-maintenance kernels of libpagedkv.
//
//  cache_write: each step computes only the new token's K/V column and keeps
//  it ("KV Cache" section of the inference-engine talk write-up); the row
//  lands in slot (block = slot / 16, row = slot % 16) of the paged pool
//  ("Blocks and block tables", section 2 of the serving-engine KV blog).
//
//  copy_blocks: copy-on-write of a shared, reference-counted block, done
//  only when someone must append to it ("Sharing blocks", same section).
//
// Both are pure byte movement: 16-byte vector loads and stores, coalesced
// along head_dim, bit-exact.  Both wait for the previous kernel on the
// stream before their first access (overlapped launch, pkv_device.cuh).
//
//  cache_write_e4m3: the write into a pool of 8-bit e4m3 codes (the OCP
//  format: 4 exponent bits with bias 7, 3 mantissa bits, largest finite
//  448).  Each bf16 element is multiplied by the pool's fp32 inverse scale
//  (one rounding) and converted to the nearest code, ties to even, values
//  beyond 448 saturating to +-448 (cvt.rn.satfinite).
#include <cuda_runtime.h>

#include <cstdint>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// One thread per 16-byte chunk of one (token, kv head) row; the same chunk
// of K and of V.  Rows of k_new/v_new are [T][Hkv][d].
__global__ void __launch_bounds__(256) cache_write_kernel(const uint4* __restrict__ k_new,
                                                          const uint4* __restrict__ v_new,
                                                          const int32_t* __restrict__ slot_mapping, int64_t total,
                                                          int32_t chunks_per_row, int32_t num_kv_heads,
                                                          int64_t num_slots, uint4* __restrict__ k_pool,
                                                          uint4* __restrict__ v_pool, unsigned long long* err) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int64_t row = i / chunks_per_row;          // (token, head)
    const int32_t c = static_cast<int32_t>(i - row * chunks_per_row);
    const int64_t t = row / num_kv_heads;
    const int32_t h = static_cast<int32_t>(row - t * num_kv_heads);
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (h == 0 && c == 0) record_error(err, kErrRange, static_cast<uint32_t>(t));
        return;
    }
    const int64_t block = slot / kBlockSize;
    const int64_t off = slot - block * kBlockSize;
    // pool row index: ((block * Hkv + h) * 16 + off), each row chunks_per_row chunks
    const int64_t dst = ((block * num_kv_heads + h) * kBlockSize + off) * chunks_per_row + c;
    const uint4 kv = __ldg(k_new + i);
    const uint4 vv = __ldg(v_new + i);
    k_pool[dst] = kv;
    v_pool[dst] = vv;
}

// One thread per 8 elements of one (token, kv head) row, K and V.
__global__ void __launch_bounds__(256) cache_write_e4m3_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, const int32_t* __restrict__ slot_mapping,
    int64_t total, int32_t chunks_per_row, int32_t num_kv_heads, int64_t num_slots, float k_inv, float v_inv,
    uint2* __restrict__ k_pool, uint2* __restrict__ v_pool, unsigned long long* err) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int64_t row = i / chunks_per_row;
    const int32_t c = static_cast<int32_t>(i - row * chunks_per_row);
    const int64_t t = row / num_kv_heads;
    const int32_t h = static_cast<int32_t>(row - t * num_kv_heads);
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (h == 0 && c == 0) record_error(err, kErrRange, static_cast<uint32_t>(t));
        return;
    }
    const int64_t block = slot / kBlockSize;
    const int64_t off = slot - block * kBlockSize;
    const int64_t dst = ((block * num_kv_heads + h) * kBlockSize + off) * chunks_per_row + c;
    k_pool[dst] = quantise8(__ldg(k_new + i), k_inv);
    v_pool[dst] = quantise8(__ldg(v_new + i), v_inv);
}

// Grid: x = chunk groups, y = pair.  Each pair copies the K slab then the V
// slab of one block ([Hkv][16][d] elements each).
__global__ void __launch_bounds__(256) copy_blocks_kernel(const int32_t* __restrict__ src,
                                                          const int32_t* __restrict__ dst, int64_t block_chunks,
                                                          int32_t num_blocks, uint4* __restrict__ k_pool,
                                                          uint4* __restrict__ v_pool, unsigned long long* err) {
    griddep_launch_dependents();
    griddep_wait();
    const int32_t pair = blockIdx.y;
    const int32_t s = __ldg(src + pair);
    const int32_t d = __ldg(dst + pair);
    if (s < 0) return;  // unused pair entry
    if (s >= num_blocks || d < 0 || d >= num_blocks) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(err, kErrRange, static_cast<uint32_t>(pair));
        return;
    }
    const uint4* ks = k_pool + static_cast<int64_t>(s) * block_chunks;
    const uint4* vs = v_pool + static_cast<int64_t>(s) * block_chunks;
    uint4* kd = k_pool + static_cast<int64_t>(d) * block_chunks;
    uint4* vd = v_pool + static_cast<int64_t>(d) * block_chunks;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < 2 * block_chunks;
         i += stride) {
        if (i < block_chunks) {
            kd[i] = ks[i];
        } else {
            vd[i - block_chunks] = vs[i - block_chunks];
        }
    }
}

// Grid: x = chunk groups, y = pair.  Pair i moves block blocks[i] of the
// pool and slab slots[i] of the host buffer ([slots][2][Hkv][16][d] pool
// elements: the K block, then the V block) in the given direction.
__global__ void __launch_bounds__(256) swap_blocks_kernel(int32_t direction, const int32_t* __restrict__ blocks,
                                                          const int32_t* __restrict__ slots, int64_t block_chunks,
                                                          int32_t num_blocks, int64_t num_slots,
                                                          uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                                          uint4* __restrict__ host, unsigned long long* err) {
    griddep_launch_dependents();
    griddep_wait();
    const int32_t pair = blockIdx.y;
    const int32_t b = __ldg(blocks + pair);
    const int32_t h = __ldg(slots + pair);
    if (b < 0) return;  // unused pair entry
    if (b >= num_blocks || h < 0 || h >= num_slots) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(err, kErrRange, static_cast<uint32_t>(pair));
        return;
    }
    uint4* kb = k_pool + static_cast<int64_t>(b) * block_chunks;
    uint4* vb = v_pool + static_cast<int64_t>(b) * block_chunks;
    uint4* slab = host + static_cast<int64_t>(h) * 2 * block_chunks;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < 2 * block_chunks;
         i += stride) {
        uint4* dev = i < block_chunks ? kb + i : vb + (i - block_chunks);
        if (direction == 0) slab[i] = *dev;
        else *dev = slab[i];
    }
}

// A plain copy of n 16-byte chunks by the SMs: either side may be device
// memory or page-locked host memory that the device reaches directly (the
// host link of a Grace system), so a transfer needs no copy engine and
// chains with the kernels around it like any other launch.
__global__ void __launch_bounds__(256) copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                     int64_t n) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy16(void* dst, const void* src, int64_t chunks, int num_sms, cudaStream_t stream) {
    const int threads = 256;
    int64_t blocks = (chunks + threads - 1) / threads;
    blocks = blocks < 1 ? 1 : (blocks > 4 * num_sms ? 4 * num_sms : blocks);
    return launch_overlapped(copy16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                             static_cast<const uint4*>(src), static_cast<uint4*>(dst), chunks);
}

cudaError_t launch_swap_blocks(int32_t direction, const int32_t* blocks, const int32_t* slots, int32_t n,
                               void* host, int64_t num_slots, void* k_pool, void* v_pool, int32_t num_blocks,
                               int32_t num_kv_heads, int32_t head_dim, int32_t elem_bytes, unsigned long long* err,
                               cudaStream_t stream) {
    const int64_t block_chunks = static_cast<int64_t>(num_kv_heads) * kBlockSize * head_dim * elem_bytes / 16;
    const int threads = 256;
    int64_t gx = (2 * block_chunks + threads - 1) / threads;
    if (gx > 64) gx = 64;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(n));
    return launch_overlapped(swap_blocks_kernel, grid, dim3(threads), 0, stream, direction, blocks, slots,
                             block_chunks, num_blocks, num_slots, static_cast<uint4*>(k_pool),
                             static_cast<uint4*>(v_pool), static_cast<uint4*>(host), err);
}

cudaError_t launch_cache_write(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                               int32_t num_tokens, void* k_pool, void* v_pool, int32_t num_blocks,
                               int32_t num_kv_heads, int32_t head_dim, unsigned long long* err,
                               cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int32_t chunks = head_dim * 2 / 16;
    const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * chunks;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    return launch_overlapped(cache_write_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                             static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping, total,
                             chunks, num_kv_heads, static_cast<int64_t>(num_blocks) * kBlockSize,
                             static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), err);
}

cudaError_t launch_cache_write_e4m3(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                                    int32_t num_tokens, void* k_pool, void* v_pool, int32_t num_blocks,
                                    int32_t num_kv_heads, int32_t head_dim, float k_inv_scale, float v_inv_scale,
                                    unsigned long long* err, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int32_t chunks = head_dim / 8;
    const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * chunks;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    return launch_overlapped(cache_write_e4m3_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                             static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping, total,
                             chunks, num_kv_heads, static_cast<int64_t>(num_blocks) * kBlockSize, k_inv_scale,
                             v_inv_scale, static_cast<uint2*>(k_pool), static_cast<uint2*>(v_pool), err);
}

cudaError_t launch_copy_blocks(const int32_t* src, const int32_t* dst, int32_t num_pairs, void* k_pool,
                               void* v_pool, int32_t num_blocks, int32_t num_kv_heads, int32_t head_dim,
                               int32_t elem_bytes, unsigned long long* err, cudaStream_t stream) {
    if (num_pairs == 0) return cudaSuccess;
    const int64_t block_chunks = static_cast<int64_t>(num_kv_heads) * kBlockSize * head_dim * elem_bytes / 16;
    const int threads = 256;
    int64_t gx = (2 * block_chunks + threads - 1) / threads;
    if (gx > 64) gx = 64;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(num_pairs));
    return launch_overlapped(copy_blocks_kernel, grid, dim3(threads), 0, stream, src, dst, block_chunks, num_blocks,
                             static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), err);
}

}  // namespace pkv
