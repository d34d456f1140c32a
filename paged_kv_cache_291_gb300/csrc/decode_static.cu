// decode_static.cu -- decode attention for callers that cannot allocate
// device memory.
//
// pkv_decode_attention needs a caller-provided, zero-initialised workspace.
// Some callers cannot provide one: code that runs inside a host callback or
// a signal-safe path where cudaMalloc must not be called, plug-ins loaded
// into a host process whose memory pool they do not own, or embedded
// runtimes that forbid device allocation after start-up.  For them this
// file keeps one fixed scratch buffer in the library itself (a file-scope
// __device__ array, present on every GPU that loads the library until the
// process exits) and runs the same decode path on it.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

#define PKV_API extern "C" __attribute__((visibility("default")))

namespace {

// Largest workspace the built-in scratch can stand in for.
constexpr size_t kScratchBytes = 4u << 20;  // 4 MiB

// In host code this name is only a stand-in for the device array; its
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device, looked up once
// per device with that device current; also returns the device index.
pkv_status scratch_address(void** out, int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return PKV_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    *dev_out = dev;
    return PKV_OK;
}

}  // namespace

PKV_API size_t pkv_decode_static_scratch_bytes(void) { return kScratchBytes; }

PKV_API pkv_status pkv_decode_attention_static(const pkv_cache_t* cache, const void* q, int32_t num_q_heads,
                                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                                               const int32_t* context_lens, int32_t num_seqs,
                                               int32_t max_context_len, float scale, float* out, void* stream) {
    if (cache == nullptr) return PKV_ERR_NULL;
    if (num_seqs == 0) {
        // Nothing to launch, but the arguments are checked exactly as the
        // regular call checks them (it returns PKV_OK for an empty batch
        // before it looks at the workspace).
        return pkv_decode_attention(cache, q, num_q_heads, block_tables, max_blocks_per_seq, context_lens, 0,
                                    max_context_len, scale, out, nullptr, 0, 0, stream);
    }
    const size_t need = pkv_decode_workspace_size(num_seqs, num_q_heads, cache->num_kv_heads, cache->head_dim,
                                                  max_context_len, 0);
    if (need == 0) {
        // Bad shape or heads: let the regular call report the exact reason.
        return pkv_decode_attention(cache, q, num_q_heads, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                    max_context_len, scale, out, nullptr, 0, 0, stream);
    }
    if (need > kScratchBytes) return PKV_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    int dev = 0;
    pkv_status st = scratch_address(&scratch, &dev);
    if (st != PKV_OK) return st;
    // Every call shares the array and finds the previous call's contents:
    // clear the counters that must start at zero (the partial results are
    // always written before they are read).
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PKV_ERR_CUDA;
    const pkv::DecodePlan plan = pkv::plan_decode_ranges(num_seqs, cache->num_kv_heads, max_context_len, sms, 0);
    const pkv::DecodeWsLayout L =
        pkv::decode_ws_layout(num_seqs, num_q_heads, cache->num_kv_heads, cache->head_dim, plan.max_ranges);
    if (cudaMemsetAsync(scratch, 0, L.part_ml, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKV_ERR_CUDA;
    return pkv_decode_attention(cache, q, num_q_heads, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                max_context_len, scale, out, scratch, kScratchBytes, 0, stream);
}
