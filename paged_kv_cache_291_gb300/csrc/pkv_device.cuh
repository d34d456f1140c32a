// pkv_device.cuh -- device-side helpers shared by the libpagedkv kernels
// (sm_103a): mbarriers with bounded waits, 1-D bulk (TMA) copies, error
// recording, bf16 unpacking.  Inline PTX only; no library code.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace pkv {

constexpr int kBlockSize = 16;  // tokens per KV block

// Error word layout: (code << 32) | detail; the first error wins.
constexpr uint32_t kErrRange = 9;    // PKV_ERR_RANGE
constexpr uint32_t kErrTimeout = 10; // PKV_ERR_TIMEOUT
constexpr uint32_t kErrAlias = 6;    // PKV_ERR_ALIAS
constexpr uint32_t kErrNoBlocks = 14; // PKV_ERR_NO_BLOCKS

// Upper bound on any wait inside a kernel (nanoseconds of %globaltimer).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void record_error(unsigned long long* err, uint32_t code, uint32_t detail) {
    if (err != nullptr) atomicCAS(err, 0ull, (static_cast<unsigned long long>(code) << 32) | detail);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- launch overlap
// Every libpagedkv kernel is launched with programmatic stream
// serialization (launch_overlapped below): it may start while the kernel
// before it on the stream is still running.  Before griddep_wait() returns,
// a kernel touches global memory only through L2 prefetches (which cannot
// make it read stale data: L2 is where every write lands); griddep_wait()
// returns once the previous kernel has completed and its writes are
// visible.  launch_dependents lets the next overlapped launch start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// Load that bypasses L1 (cached in L2 only): for values read before
// griddep_wait() that must not leave a stale copy in L1.
__device__ __forceinline__ int32_t ld_l2_only(const int32_t* p) {
    int32_t v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Prefetch [p, p + bytes) into L2 with one bulk request (p and bytes
// multiples of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Item k of the 128-byte lines that overlap [base, base + bytes): returns
// an address inside the range on that line, or nullptr past the end.
__device__ __forceinline__ const void* range_line(const void* base, long long bytes, long long k) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(base);
    const uintptr_t line = (a & ~static_cast<uintptr_t>(127)) + static_cast<uintptr_t>(k) * 128u;
    if (line >= a + static_cast<uintptr_t>(bytes)) return nullptr;
    return reinterpret_cast<const void*>(line < a ? a : line);
}

// Upper bound on the 128-byte lines that overlap a range of `bytes` bytes.
__host__ __device__ __forceinline__ long long range_lines(long long bytes) { return bytes > 0 ? bytes / 128 + 2 : 0; }

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most
// kWaitLimitNs.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Warp-uniform bounded wait: every lane polls, then the warp agrees, so
// that a timeout can never split a warp before a collective operation.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return __all_sync(0xffffffffu, ok);
}

// Generic-proxy shared-memory writes ordered before later async-proxy
// (bulk copy) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------ bulk (TMA) copies
// 1-D bulk copy global -> shared, completion signalled on `bar` as tx bytes.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_g2s_hint(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------- bf16
// Two packed bf16 (low half = element 0) -> two floats, exactly.
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ uint2 lds64(const void* p) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_addr(p)));
    return v;
}

// ---------------------------------------------------------------- e4m3
// Two fp32 -> two e4m3 codes (nearest, ties to even, saturating to +-448),
// lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Eight bf16 (one uint4) times inv (one fp32 rounding each) -> eight codes
// (one uint2), element 0 in the lowest byte.
__device__ __forceinline__ uint2 quantise8(uint4 x, float inv) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = __fmul_rn(__uint_as_float(w[i] << 16), inv);
        const float hi = __fmul_rn(__uint_as_float(w[i] & 0xffff0000u), inv);
        c[i] = e4m3x2(lo, hi);
    }
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Maximum over the full warp in one instruction (sm_100 family); inputs are
// finite or -inf.
__device__ __forceinline__ float warp_max_redux(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Host: launch `kernel` with programmatic stream serialization unless the
// PKV_OVERLAP environment variable is "0" (then a plain launch).
bool overlap_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace pkv
