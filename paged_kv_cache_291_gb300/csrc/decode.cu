// decode.cu -- paged decode attention: host side (workspace layout, work
// plan, the launch of the plain decode variant, the test hook).  The kernel
// is in decode_kernel.cuh; the fused decode step's variant is instantiated in
// decode_fused.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "decode_kernel.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

// Decode launches still to be made with a stalled producer (test hook).
std::atomic<int> g_stall_launches{0};

// Takes one armed stall, if any.
bool take_stall() {
    int n = g_stall_launches.load();
    while (n > 0 && !g_stall_launches.compare_exchange_weak(n, n - 1)) {
    }
    return n > 0;
}

}  // namespace

void arm_decode_stall(int32_t launches) { g_stall_launches.store(launches > 0 ? launches : 0); }

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

DecodeWsLayout decode_ws_layout(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t max_ranges, bool prefix) {
    const size_t G = static_cast<size_t>(num_q_heads / num_kv_heads);
    DecodeWsLayout L;
    L.header = 0;
    L.counters = 256;
    L.part_ml = L.counters + align256(static_cast<size_t>(num_seqs) * num_kv_heads * 4);
    const size_t slots = static_cast<size_t>(max_ranges) * 2 * G;
    L.part_o = L.part_ml + align256(slots * 8);
    L.pre_ml = L.part_o + align256(slots * head_dim * 4);
    const size_t pre = prefix ? static_cast<size_t>(num_seqs) * num_q_heads : 0;
    L.pre_o = L.pre_ml + align256(pre * 8);
    L.total = L.pre_o + align256(pre * head_dim * 4);
    return L;
}

DecodePlan plan_decode_ranges(int32_t num_seqs, int32_t num_kv_heads, int32_t max_context_len, int32_t num_sms,
                              int32_t req_range_units) {
    DecodePlan pl;
    const int64_t units_max = std::max<int64_t>(1, (static_cast<int64_t>(max_context_len) + kBlockSize - 1) / kBlockSize);
    const int64_t total_max = std::max<int64_t>(1, static_cast<int64_t>(num_seqs) * num_kv_heads * units_max);
    if (req_range_units > 0) {
        // Fixed ranges: CTAs loop over them; the workspace holds them all.
        pl.range_units = req_range_units;
        pl.max_ranges = static_cast<int32_t>((total_max + req_range_units - 1) / req_range_units);
        pl.grid = num_sms;
    } else {
        // One range per CTA, at least kMinRangeUnits blocks each.
        pl.range_units = 0;
        pl.grid = static_cast<int32_t>(
            std::max<int64_t>(1, std::min<int64_t>(num_sms, (total_max + kMinRangeUnits - 1) / kMinRangeUnits)));
        pl.max_ranges = pl.grid;
    }
    return pl;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    if (a.num_seqs == 0) return cudaSuccess;
    const bool stall = take_stall();
    if (a.k_new != nullptr) return launch_decode_fused(a, stall, stream);
    return launch_decode_t<false>(a, stall, stream);
}

}  // namespace pkv
