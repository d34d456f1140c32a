// api.cu -- the C-ABI of libpagedkv: argument checks, per-device state, the
// device error word, workspace sizing and dispatch to the kernels.
//
// The calls and their contracts are declared (with the passages of the
// pages that define each operation) in include/pkv.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_set>

#include "pkv.h"
#include "pkv_internal.h"

#define PKV_API extern "C" __attribute__((visibility("default")))

// First device-side error since the last pkv_get_error: (code << 32) | detail.
__device__ unsigned long long g_pkv_error_word;

namespace pkv {
// Overlapped launches are on unless PKV_OVERLAP=0 (read once per process).
bool overlap_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("PKV_OVERLAP");
        return !(v != nullptr && v[0] == '0' && v[1] == '\0');
    }();
    return on;
}
}  // namespace pkv

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    unsigned long long* err = nullptr;
};

DeviceState g_devices[kMaxDevices];
std::mutex g_mutex;
thread_local char g_cuda_error[256] = "no error";

pkv_status cuda_fail(cudaError_t e) {
    std::snprintf(g_cuda_error, sizeof g_cuda_error, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return PKV_ERR_CUDA;
}

// Properties and the error-word address of the current device, looked up
// once per device with that device current.
pkv_status current_device(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& d = g_devices[dev];
    if (!d.ready) {
        if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(e);
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_pkv_error_word)) != cudaSuccess) return cuda_fail(e);
        d.err = static_cast<unsigned long long*>(p);
        d.ready = true;
    }
    if (d.cc_major != 10 || d.cc_minor != 3) return PKV_ERR_UNSUPPORTED;
    *out = &d;
    return PKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pkv_status check_cache(const pkv_cache_t* c) {
    if (c == nullptr || c->k_pool == nullptr || c->v_pool == nullptr) return PKV_ERR_NULL;
    if (c->block_size != 16) return PKV_ERR_BLOCKSIZE;
    if (c->num_blocks < 0 || c->num_kv_heads < 1) return PKV_ERR_SHAPE;
    if (c->head_dim != 64 && c->head_dim != 128) return PKV_ERR_HEADDIM;
    if (!aligned16(c->k_pool) || !aligned16(c->v_pool)) return PKV_ERR_ALIGN;
    if (c->kv_dtype != PKV_KV_BF16 && c->kv_dtype != PKV_KV_E4M3) return PKV_ERR_DTYPE;
    if (c->kv_dtype == PKV_KV_E4M3) {
        // 1/scale must be a finite fp32 too.
        for (float x : {c->k_scale, c->v_scale})
            if (!(std::isfinite(x) && x > 0.f && std::isfinite(1.f / x))) return PKV_ERR_DTYPE;
    }
    return PKV_OK;
}

int32_t elem_bytes(const pkv_cache_t* c) { return c->kv_dtype == PKV_KV_E4M3 ? 1 : 2; }

// The address a kernel uses for p: device memory as it is, page-locked host
// memory mapped for the device through the pointer the runtime reports for
// it; anything else (pageable host memory) is refused.
pkv_status device_address(const void* p, const void** out) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_HOST_MEMORY;
    }
    if (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged) {
        *out = p;
        return PKV_OK;
    }
    if (attr.type == cudaMemoryTypeHost && attr.devicePointer != nullptr) {
        *out = attr.devicePointer;
        return PKV_OK;
    }
    return PKV_ERR_HOST_MEMORY;
}

pkv_status check_heads(int32_t hq, int32_t hkv) {
    if (hq < 1 || hkv < 1 || hq % hkv != 0) return PKV_ERR_HEADS;
    const int32_t g = hq / hkv;
    if (g != 1 && g != 2 && g != 4 && g != 8) return PKV_ERR_HEADS;
    return PKV_OK;
}

// Shared by the decode call and the decode rows of the mixed batch.
// prefix: the workspace also holds the shared-prefix state of every
// (sequence, q head).
pkv_status plan_decode(int32_t num_seqs, int32_t hq, int32_t hkv, int32_t head_dim, int32_t max_context_len,
                       int32_t req_range_units, int num_sms, pkv::DecodePlan* plan, size_t* ws_bytes,
                       bool prefix = false) {
    if (num_seqs < 0 || max_context_len < 0 || req_range_units < 0) return PKV_ERR_SHAPE;
    *plan = pkv::plan_decode_ranges(num_seqs, hkv, max_context_len, num_sms, req_range_units);
    *ws_bytes = pkv::decode_ws_layout(num_seqs, hq, hkv, head_dim, plan->max_ranges, prefix).total;
    return PKV_OK;
}

// Shared blocks are checked against max_context_len (every context holds
// them in full) and the table width.
pkv_status check_shared_blocks(int32_t shared_blocks, int32_t max_blocks_per_seq, int32_t max_context_len) {
    if (shared_blocks < 0 || shared_blocks > max_blocks_per_seq ||
        static_cast<int64_t>(shared_blocks) * 16 > max_context_len)
        return PKV_ERR_SHAPE;
    return PKV_OK;
}

}  // namespace

PKV_API const char* pkv_version(void) { return "0.1.0"; }

PKV_API const char* pkv_last_cuda_error(void) { return g_cuda_error; }

PKV_API const char* pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_NULL: return "PKV_ERR_NULL: a required pointer is NULL";
        case PKV_ERR_SHAPE: return "PKV_ERR_SHAPE: a count or size is negative or inconsistent";
        case PKV_ERR_HEADS: return "PKV_ERR_HEADS: num_q_heads / num_kv_heads must be 1, 2, 4 or 8";
        case PKV_ERR_HEADDIM: return "PKV_ERR_HEADDIM: head_dim must be 64 or 128";
        case PKV_ERR_BLOCKSIZE: return "PKV_ERR_BLOCKSIZE: block_size must be 16";
        case PKV_ERR_ALIAS: return "PKV_ERR_ALIAS: copy_blocks destinations repeat or overlap sources";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE: workspace missing, too small or misaligned";
        case PKV_ERR_ALIGN: return "PKV_ERR_ALIGN: a device pointer is not 16-byte aligned";
        case PKV_ERR_RANGE: return "PKV_ERR_RANGE: a block id, slot or context length was out of range";
        case PKV_ERR_TIMEOUT: return "PKV_ERR_TIMEOUT: a bounded wait inside a kernel expired";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA: a CUDA runtime call failed";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED: the current device is not compute capability 10.3";
        case PKV_ERR_SCRATCH_LIMIT:
            return "PKV_ERR_SCRATCH_LIMIT: the batch needs more workspace than the built-in 4 MiB scratch buffer";
        case PKV_ERR_NO_BLOCKS: return "PKV_ERR_NO_BLOCKS: the free queue holds fewer blocks than the append needs";
        case PKV_ERR_HOST_MEMORY: return "PKV_ERR_HOST_MEMORY: the host buffer is not page-locked memory mapped for the device";
        case PKV_ERR_DTYPE:
            return "PKV_ERR_DTYPE: unknown kv_dtype, e4m3 scales not finite and positive, or a call without e4m3 support";
    }
    return "unknown pkv_status";
}

PKV_API pkv_status pkv_cache_write(const pkv_cache_t* cache, const void* k_new, const void* v_new,
                                   const int32_t* slot_mapping, int32_t num_tokens, void* stream) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return PKV_ERR_SHAPE;
    if (num_tokens == 0) return PKV_OK;
    if (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr) return PKV_ERR_NULL;
    if (!aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_ALIGN;
    DeviceState* dev = nullptr;
    if ((st = current_device(&dev)) != PKV_OK) return st;
    cudaError_t e =
        cache->kv_dtype == PKV_KV_E4M3
            ? pkv::launch_cache_write_e4m3(k_new, v_new, slot_mapping, num_tokens, cache->k_pool, cache->v_pool,
                                           cache->num_blocks, cache->num_kv_heads, cache->head_dim,
                                           1.f / cache->k_scale, 1.f / cache->v_scale, dev->err,
                                           static_cast<cudaStream_t>(stream))
            : pkv::launch_cache_write(k_new, v_new, slot_mapping, num_tokens, cache->k_pool, cache->v_pool,
                                      cache->num_blocks, cache->num_kv_heads, cache->head_dim, dev->err,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

PKV_API pkv_status pkv_copy_blocks(const pkv_cache_t* cache, const int32_t* src, const int32_t* dst,
                                   int32_t num_pairs, const int32_t* src_host, const int32_t* dst_host,
                                   void* stream) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (num_pairs < 0) return PKV_ERR_SHAPE;
    if (num_pairs == 0) return PKV_OK;
    if (src == nullptr || dst == nullptr) return PKV_ERR_NULL;
    if ((src_host == nullptr) != (dst_host == nullptr)) return PKV_ERR_NULL;
    if (src_host != nullptr) {
        std::unordered_set<int32_t> dsts, srcs;
        for (int32_t i = 0; i < num_pairs; ++i) {
            if (src_host[i] < 0) continue;  // skipped pair
            if (src_host[i] >= cache->num_blocks || dst_host[i] < 0 ||
                dst_host[i] >= cache->num_blocks)
                return PKV_ERR_RANGE;
            if (!dsts.insert(dst_host[i]).second) return PKV_ERR_ALIAS;
            srcs.insert(src_host[i]);
        }
        for (int32_t d : dsts)
            if (srcs.count(d)) return PKV_ERR_ALIAS;
    }
    DeviceState* dev = nullptr;
    if ((st = current_device(&dev)) != PKV_OK) return st;
    // grid.y is limited to 65,535 pairs per launch.
    for (int32_t base = 0; base < num_pairs; base += 65535) {
        const int32_t n = std::min<int32_t>(65535, num_pairs - base);
        cudaError_t e = pkv::launch_copy_blocks(src + base, dst + base, n, cache->k_pool, cache->v_pool,
                                                cache->num_blocks, cache->num_kv_heads, cache->head_dim,
                                                elem_bytes(cache), dev->err, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return PKV_OK;
}

namespace {

pkv_status check_blocks(const pkv_blocks_t* b, pkv::BlocksArgs* a) {
    if (b == nullptr || b->block_tables == nullptr || b->context_lens == nullptr || b->ref_counts == nullptr ||
        b->free_ring == nullptr || b->ring_pos == nullptr || b->free_state == nullptr || b->scratch == nullptr)
        return PKV_ERR_NULL;
    if (b->num_blocks < 0 || b->max_seqs < 0 || b->max_blocks_per_seq < 1) return PKV_ERR_SHAPE;
    if (static_cast<int64_t>(b->max_blocks_per_seq) * 16 > INT32_MAX || b->num_blocks > INT32_MAX / 3)
        return PKV_ERR_SHAPE;
    const int n_cache = (b->block_keys != nullptr) + (b->key_table != nullptr) + (b->cached != nullptr);
    if (n_cache != 0 && n_cache != 3) return PKV_ERR_NULL;
    if (n_cache == 3) {
        const int64_t t = b->table_size;
        if (t < 2 * static_cast<int64_t>(b->num_blocks) || t < 1 || (t & (t - 1)) != 0) return PKV_ERR_SHAPE;
        if (!aligned16(b->block_keys)) return PKV_ERR_ALIGN;
    }
    *a = pkv::BlocksArgs{b->block_tables, b->context_lens, b->ref_counts, b->free_ring, b->ring_pos,
                         b->free_state,   b->scratch,      b->block_keys, b->key_table, b->cached,
                         b->num_blocks,   b->max_seqs,     b->max_blocks_per_seq,
                         n_cache == 3 ? b->table_size : 0};
    return PKV_OK;
}

}  // namespace

PKV_API pkv_status pkv_blocks_reset(const pkv_blocks_t* blocks, void* stream) {
    pkv::BlocksArgs a;
    pkv_status st = check_blocks(blocks, &a);
    if (st != PKV_OK) return st;
    DeviceState* dev = nullptr;
    if ((st = current_device(&dev)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_blocks_reset(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

PKV_API pkv_status pkv_blocks_append(const pkv_blocks_t* blocks, const int32_t* query_start_loc, int32_t num_seqs,
                                     int32_t num_tokens, int32_t* slot_mapping, int32_t* cow_src, int32_t* cow_dst,
                                     int32_t* cow_count, void* stream) {
    pkv::BlocksArgs a;
    pkv_status st = check_blocks(blocks, &a);
    if (st != PKV_OK) return st;
    if (num_seqs < 0 || num_tokens < 0 || num_seqs > blocks->max_seqs) return PKV_ERR_SHAPE;
    if (num_seqs == 0) return num_tokens == 0 ? PKV_OK : PKV_ERR_SHAPE;
    if (query_start_loc == nullptr || cow_src == nullptr || cow_dst == nullptr || cow_count == nullptr)
        return PKV_ERR_NULL;
    if (num_tokens > 0 && slot_mapping == nullptr) return PKV_ERR_NULL;
    DeviceState* dev = nullptr;
    if ((st = current_device(&dev)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_blocks_append(a, query_start_loc, num_seqs, num_tokens, slot_mapping, cow_src,
                                              cow_dst, cow_count, dev->err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

PKV_API pkv_status pkv_blocks_fork(const pkv_blocks_t* blocks, const int32_t* parents, const int32_t* children,
                                   int32_t n, void* stream) {
    pkv::BlocksArgs a;
    pkv_status st = check_blocks(blocks, &a);
    if (st != PKV_OK) return st;
    if (n < 0 || n > pkv::kBlocksMaxRows) return PKV_ERR_SHAPE;
    if (n == 0) return PKV_OK;
    if (parents == nullptr || children == nullptr) return PKV_ERR_NULL;
    DeviceState* dev = nullptr;
    if ((st = current_device(&dev)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_blocks_fork(a, parents, children, n, dev->err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

PKV_API pkv_status pkv_blocks_match(const pkv_blocks_t* blocks, const void* keys, int32_t key_stride,
                                    const int32_t* num_keys, int32_t num_seqs, int32_t* matched, void* stream) {
    pkv::BlocksArgs a;
    pkv_status st = check_blocks(blocks, &a);
    if (st != PKV_OK) return st;
    if (a.key_table == nullptr) return PKV_ERR_NULL;
    if (num_seqs < 0 || num_seqs > blocks->max_seqs || num_seqs > pkv::kBlocksMaxRows || key_stride < 0)
        return PKV_ERR_SHAPE;
    if (num_seqs == 0) return PKV_OK;
    if (keys == nullptr || num_keys == nullptr || matched == nullptr) return PKV_ERR_NULL;
    if (!aligned16(keys)) return PKV_ERR_ALIGN;
    DeviceState* dev = nullptr;
    if ((st = current_device(&dev)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_blocks_match(a, static_cast<const uint8_t*>(keys), key_stride, num_keys, num_seqs,
                                             matched, dev->err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

PKV_API pkv_status pkv_blocks_register(const pkv_blocks_t* blocks, const void* keys, int32_t key_stride,
                                       const int32_t* num_keys, int32_t num_seqs, void* stream) {
    pkv::BlocksArgs a;
    pkv_status st = check_blocks(blocks, &a);
    if (st != PKV_OK) return st;
    if (a.key_table == nullptr) return PKV_ERR_NULL;
    if (num_seqs < 0 || num_seqs > blocks->max_seqs || num_seqs > pkv::kBlocksMaxRows || key_stride < 0)
        return PKV_ERR_SHAPE;
    if (num_seqs == 0) return PKV_OK;
    if (keys == nullptr || num_keys == nullptr) return PKV_ERR_NULL;
    if (!aligned16(keys)) return PKV_ERR_ALIGN;
    DeviceState* dev = nullptr;
    if ((st = current_device(&dev)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_blocks_register(a, static_cast<const uint8_t*>(keys), key_stride, num_keys,
                                                num_seqs, dev->err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

PKV_API pkv_status pkv_blocks_release(const pkv_blocks_t* blocks, const int32_t* rows, int32_t n, void* stream) {
    pkv::BlocksArgs a;
    pkv_status st = check_blocks(blocks, &a);
    if (st != PKV_OK) return st;
    if (n < 0 || n > pkv::kBlocksMaxRows) return PKV_ERR_SHAPE;
    if (n == 0) return PKV_OK;
    if (rows == nullptr) return PKV_ERR_NULL;
    DeviceState* dev = nullptr;
    if ((st = current_device(&dev)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_blocks_release(a, rows, n, dev->err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

PKV_API pkv_status pkv_prefix_keys(const int32_t* token_ids, const int32_t* token_start_loc, const int64_t* extra,
                                   const void* parent_keys, int32_t num_seqs, int32_t max_blocks, void* keys,
                                   void* stream) {
    if (num_seqs < 0 || max_blocks < 0) return PKV_ERR_SHAPE;
    if (num_seqs == 0) return PKV_OK;
    if (token_ids == nullptr || token_start_loc == nullptr || keys == nullptr) return PKV_ERR_NULL;
    if (!aligned16(keys) || (parent_keys != nullptr && !aligned16(parent_keys))) return PKV_ERR_ALIGN;
    pkv_status st;
    DeviceState* dev = nullptr;
    if ((st = current_device(&dev)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_prefix_keys(token_ids, token_start_loc, extra,
                                            static_cast<const uint8_t*>(parent_keys), num_seqs, max_blocks,
                                            static_cast<uint8_t*>(keys), dev->err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

PKV_API pkv_status pkv_swap_blocks(const pkv_cache_t* cache, int32_t direction, const int32_t* blocks,
                                   const int32_t* slots, int32_t n, void* host, int64_t num_host_slots, void* stream) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (direction != 0 && direction != 1) return PKV_ERR_SHAPE;
    if (n < 0 || n > 65535 || num_host_slots < 0) return PKV_ERR_SHAPE;
    if (n == 0) return PKV_OK;
    if (blocks == nullptr || slots == nullptr || host == nullptr) return PKV_ERR_NULL;
    if (!aligned16(host)) return PKV_ERR_ALIGN;
    DeviceState* dev = nullptr;
    if ((st = current_device(&dev)) != PKV_OK) return st;
    // Only page-locked host memory mapped for this device is handed to the
    // kernel, through the device pointer the runtime reports for it.
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, host) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_HOST_MEMORY;
    }
    if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return PKV_ERR_HOST_MEMORY;
    cudaError_t e = pkv::launch_swap_blocks(direction, blocks, slots, n, attr.devicePointer, num_host_slots,
                                            cache->k_pool, cache->v_pool, cache->num_blocks, cache->num_kv_heads,
                                            cache->head_dim, elem_bytes(cache), dev->err,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

PKV_API pkv_status pkv_copy(void* dst, const void* src, size_t bytes, void* stream) {
    if (bytes == 0) return PKV_OK;
    if (dst == nullptr || src == nullptr) return PKV_ERR_NULL;
    if (bytes % 16 != 0 || bytes > (static_cast<size_t>(1) << 40)) return PKV_ERR_SHAPE;
    if (!aligned16(dst) || !aligned16(src)) return PKV_ERR_ALIGN;
    DeviceState* dev = nullptr;
    pkv_status st = current_device(&dev);
    if (st != PKV_OK) return st;
    const void *d = nullptr, *s = nullptr;
    if ((st = device_address(dst, &d)) != PKV_OK) return st;
    if ((st = device_address(src, &s)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_copy16(const_cast<void*>(d), s, static_cast<int64_t>(bytes / 16), dev->num_sms,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

PKV_API size_t pkv_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t max_context_len, int32_t partition_blocks) {
    if (check_heads(num_q_heads, num_kv_heads) != PKV_OK) return 0;
    if (head_dim != 64 && head_dim != 128) return 0;
    DeviceState* dev = nullptr;
    if (current_device(&dev) != PKV_OK) return 0;
    pkv::DecodePlan plan;
    size_t bytes = 0;
    if (plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len, partition_blocks,
                    dev->num_sms, &plan, &bytes) != PKV_OK)
        return 0;
    return bytes;
}

namespace {

pkv_status decode_common(const pkv_cache_t* cache, const void* q, int32_t num_q_heads,
                         const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
                         const int32_t* query_start_loc, int32_t num_seqs, int32_t max_context_len, float scale,
                         float* out, void* workspace, size_t workspace_bytes, int32_t partition_blocks,
                         void* stream, const void* k_new = nullptr, const void* v_new = nullptr,
                         const int32_t* slot_mapping = nullptr, int32_t shared_blocks = 0) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if ((st = check_heads(num_q_heads, cache->num_kv_heads)) != PKV_OK) return st;
    if (num_seqs < 0 || max_blocks_per_seq < 0 || max_context_len < 0 || partition_blocks < 0)
        return PKV_ERR_SHAPE;
    if (num_seqs == 0) return PKV_OK;
    if (q == nullptr || block_tables == nullptr || context_lens == nullptr || out == nullptr) return PKV_ERR_NULL;
    if (!aligned16(q) || !aligned16(out)) return PKV_ERR_ALIGN;
    DeviceState* dev = nullptr;
    if ((st = current_device(&dev)) != PKV_OK) return st;
    // out may be page-locked host memory: the kernel then writes the rows
    // there directly.
    const void* out_dev = nullptr;
    if ((st = device_address(out, &out_dev)) != PKV_OK) return st;
    out = static_cast<float*>(const_cast<void*>(out_dev));
    // A shared prefix is read once for all sequences on bf16 pools whose rows
    // a tensor map can address; otherwise every sequence reads it (the same
    // result).  The workspace is sized for the shared-prefix states either way.
    const int32_t chunks = pkv::shared_prefix_chunks(num_seqs, num_q_heads, cache->num_kv_heads, shared_blocks);
    const bool share = chunks > 0 && cache->kv_dtype == PKV_KV_BF16 &&
                       static_cast<int64_t>(cache->num_blocks) * cache->num_kv_heads * 16 <= INT32_MAX;
    pkv::DecodePlan plan;
    size_t need = 0;
    if ((st = plan_decode(num_seqs, num_q_heads, cache->num_kv_heads, cache->head_dim, max_context_len,
                          partition_blocks, dev->num_sms, &plan, &need, chunks > 0)) != PKV_OK)
        return st;
    if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return PKV_ERR_WORKSPACE;
    pkv::DecodeArgs a;
    a.k_pool = cache->k_pool;
    a.v_pool = cache->v_pool;
    a.q = q;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start_loc = query_start_loc;
    a.out = out;
    a.workspace = workspace;
    a.err = dev->err;
    a.num_blocks = cache->num_blocks;
    a.num_kv_heads = cache->num_kv_heads;
    a.num_q_heads = num_q_heads;
    a.head_dim = cache->head_dim;
    a.num_seqs = num_seqs;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.max_context_len = max_context_len;
    a.plan = plan;
    a.scale = scale;
    a.kv_e4m3 = cache->kv_dtype == PKV_KV_E4M3;
    a.k_scale = cache->k_scale;
    a.v_scale = cache->v_scale;
    a.k_new = k_new;
    a.v_new = v_new;
    a.slot_mapping = slot_mapping;
    if (share) {
        a.skip_blocks = shared_blocks;
        a.prefix_chunks = chunks;
        cudaError_t e = pkv::launch_shared_prefix(a, static_cast<cudaStream_t>(stream));
        if (e == cudaErrorInvalidClusterSize) {
            // A device that cannot place the kernel's clusters: every
            // sequence attends the shared blocks itself (the same result).
            cudaGetLastError();
            a.skip_blocks = 0;
            a.prefix_chunks = 0;
        } else if (e != cudaSuccess) {
            return cuda_fail(e);
        }
    }
    cudaError_t e = pkv::launch_decode(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

}  // namespace

PKV_API pkv_status pkv_decode_attention(const pkv_cache_t* cache, const void* q, int32_t num_q_heads,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* context_lens, int32_t num_seqs, int32_t max_context_len,
                                        float scale, float* out, void* workspace, size_t workspace_bytes,
                                        int32_t partition_blocks, void* stream) {
    return decode_common(cache, q, num_q_heads, block_tables, max_blocks_per_seq, context_lens, nullptr, num_seqs,
                         max_context_len, scale, out, workspace, workspace_bytes, partition_blocks, stream);
}

PKV_API size_t pkv_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                                       int32_t num_kv_heads, int32_t head_dim,
                                                       int32_t max_context_len, int32_t shared_blocks) {
    if (check_heads(num_q_heads, num_kv_heads) != PKV_OK) return 0;
    if (head_dim != 64 && head_dim != 128) return 0;
    if (shared_blocks < 0 || static_cast<int64_t>(shared_blocks) * 16 > max_context_len) return 0;
    DeviceState* dev = nullptr;
    if (current_device(&dev) != PKV_OK) return 0;
    pkv::DecodePlan plan;
    size_t bytes = 0;
    const bool prefix = pkv::shared_prefix_chunks(num_seqs, num_q_heads, num_kv_heads, shared_blocks) > 0;
    if (plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len, 0, dev->num_sms, &plan, &bytes,
                    prefix) != PKV_OK)
        return 0;
    return bytes;
}

PKV_API pkv_status pkv_decode_attention_shared_prefix(const pkv_cache_t* cache, const void* q, int32_t num_q_heads,
                                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                      const int32_t* context_lens, int32_t num_seqs,
                                                      int32_t max_context_len, int32_t shared_blocks, float scale,
                                                      float* out, void* workspace, size_t workspace_bytes,
                                                      void* stream) {
    pkv_status st = check_shared_blocks(shared_blocks, max_blocks_per_seq, max_context_len);
    if (st != PKV_OK) return st;
    return decode_common(cache, q, num_q_heads, block_tables, max_blocks_per_seq, context_lens, nullptr, num_seqs,
                         max_context_len, scale, out, workspace, workspace_bytes, 0, stream, nullptr, nullptr,
                         nullptr, shared_blocks);
}

PKV_API int32_t pkv_common_prefix_blocks(const int32_t* block_tables_host, int32_t max_blocks_per_seq,
                                         const int32_t* context_lens_host, int32_t num_seqs) {
    if (block_tables_host == nullptr || context_lens_host == nullptr || num_seqs <= 0 || max_blocks_per_seq <= 0)
        return 0;
    int32_t j = max_blocks_per_seq;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int32_t n = context_lens_host[s];
        j = std::min(j, n > 0 ? n / 16 : 0);
    }
    for (int32_t s = 1; s < num_seqs && j > 0; ++s) {
        const int32_t* row = block_tables_host + static_cast<size_t>(s) * max_blocks_per_seq;
        int32_t k = 0;
        while (k < j && row[k] == block_tables_host[k]) ++k;
        j = k;
    }
    return j;
}

PKV_API pkv_status pkv_decode_step(const pkv_cache_t* cache, const void* k_new, const void* v_new,
                                   const int32_t* slot_mapping, const void* q, int32_t num_q_heads,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, int32_t num_seqs, int32_t max_context_len,
                                   float scale, float* out, void* workspace, size_t workspace_bytes,
                                   int32_t partition_blocks, void* stream) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (num_seqs > 0) {
        if (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr) return PKV_ERR_NULL;
        if (!aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_ALIGN;
    }
    return decode_common(cache, q, num_q_heads, block_tables, max_blocks_per_seq, context_lens, nullptr, num_seqs,
                         max_context_len, scale, out, workspace, workspace_bytes, partition_blocks, stream, k_new,
                         v_new, slot_mapping);
}

PKV_API size_t pkv_prefill_workspace_size(int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_dim, int32_t max_context_len) {
    if (num_tokens < 0) return 0;
    return pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len, 0);
}

PKV_API pkv_status pkv_chunked_prefill_attention(const pkv_cache_t* cache, const void* q, int32_t num_q_heads,
                                                 int32_t num_tokens, const int32_t* query_start_loc,
                                                 const int32_t* query_start_loc_host, const int32_t* context_lens,
                                                 int32_t num_seqs, const int32_t* block_tables,
                                                 int32_t max_blocks_per_seq, int32_t max_context_len, float scale,
                                                 float* out, void* workspace, size_t workspace_bytes,
                                                 void* stream) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (cache->kv_dtype != PKV_KV_BF16) return PKV_ERR_DTYPE;  // the tcgen05 tiles read bf16 K/V
    if ((st = check_heads(num_q_heads, cache->num_kv_heads)) != PKV_OK) return st;
    if (num_seqs < 0 || num_tokens < 0 || max_blocks_per_seq < 0 || max_context_len < 0) return PKV_ERR_SHAPE;
    if (num_seqs == 0 || num_tokens == 0) return PKV_OK;
    if (q == nullptr || query_start_loc == nullptr || query_start_loc_host == nullptr || context_lens == nullptr ||
        block_tables == nullptr || out == nullptr)
        return PKV_ERR_NULL;
    if (!aligned16(q) || !aligned16(out)) return PKV_ERR_ALIGN;
    if (query_start_loc_host[0] != 0 || query_start_loc_host[num_seqs] != num_tokens) return PKV_ERR_SHAPE;
    int32_t tiles = 0, decode_rows = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int32_t ql = query_start_loc_host[s + 1] - query_start_loc_host[s];
        if (ql < 0) return PKV_ERR_SHAPE;
        if (ql == 1) ++decode_rows;
        if (ql > 1) tiles += (ql + 127) / 128;
    }
    DeviceState* dev = nullptr;
    if ((st = current_device(&dev)) != PKV_OK) return st;
    const void* out_dev = nullptr;
    if ((st = device_address(out, &out_dev)) != PKV_OK) return st;
    out = static_cast<float*>(const_cast<void*>(out_dev));
    if (decode_rows > 0) {
        st = decode_common(cache, q, num_q_heads, block_tables, max_blocks_per_seq, context_lens, query_start_loc,
                           num_seqs, max_context_len, scale, out, workspace, workspace_bytes, 0, stream);
        if (st != PKV_OK) return st;
    }
    if (tiles > 0) {
        pkv::PrefillArgs a;
        a.k_pool = cache->k_pool;
        a.v_pool = cache->v_pool;
        a.q = q;
        a.block_tables = block_tables;
        a.context_lens = context_lens;
        a.query_start_loc = query_start_loc;
        a.out = out;
        a.err = dev->err;
        a.num_blocks = cache->num_blocks;
        a.num_kv_heads = cache->num_kv_heads;
        a.num_q_heads = num_q_heads;
        a.head_dim = cache->head_dim;
        a.num_seqs = num_seqs;
        a.num_tokens = num_tokens;
        a.max_blocks_per_seq = max_blocks_per_seq;
        a.max_context_len = max_context_len;
        a.num_tiles = tiles;
        // The longest row tiles of each sequence (its last ones: they hold
        // the most keys) go to two one-head CTAs each, as many of them as
        // keep the whole grid within one CTA per SM.
        a.split_last = 0;
        a.split_tiles = 0;
        const int64_t pairs = (num_q_heads / cache->num_kv_heads) % 2 == 0 ? num_q_heads / 2 : 0;
        for (int32_t k = 1; pairs > 0; ++k) {
            int64_t extra = 0, longest = 0;
            for (int32_t s = 0; s < num_seqs; ++s) {
                const int32_t ql = query_start_loc_host[s + 1] - query_start_loc_host[s];
                const int64_t nt = ql > 1 ? (ql + 127) / 128 : 0;
                extra += std::min<int64_t>(k, nt);
                longest = std::max(longest, nt);
            }
            if (k > longest || (tiles + extra) * pairs > dev->num_sms) break;
            a.split_last = k;
            a.split_tiles = static_cast<int32_t>(extra);
        }
        a.scale = scale;
        cudaError_t e = pkv::launch_prefill(a, static_cast<cudaStream_t>(stream));
        if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return PKV_OK;
}

PKV_API pkv_status pkv_test_arm_decode_stall(int32_t launches) {
    if (launches < 0) return PKV_ERR_SHAPE;
    pkv::arm_decode_stall(launches);
    return PKV_OK;
}

PKV_API pkv_status pkv_get_error(void* stream, int32_t* detail) {
    DeviceState* dev = nullptr;
    pkv_status st = current_device(&dev);
    if (st != PKV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned long long word = 0;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMemcpyAsync(&word, dev->err, sizeof word, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return cuda_fail(e);
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e);
    if (word == 0) {
        if (detail) *detail = 0;
        return PKV_OK;
    }
    if ((e = cudaMemsetAsync(dev->err, 0, sizeof word, s)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e);
    if (detail) *detail = static_cast<int32_t>(word & 0xffffffffu);
    return static_cast<pkv_status>(word >> 32);
}
