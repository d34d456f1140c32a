// decode_kernel.cuh -- paged decode attention with split-KV and log-sum-exp
// merge: the kernel, shared by decode.cu (plain decode) and decode_fused.cu
// (the decode step with its new rows), each of which instantiates one
// variant in its own translation unit.
//
// What it computes ("Blocks and block tables", section 2 of the
// serving-engine KV blog): for each sequence s and q head h, attention of
// one query over context_lens[s] keys that live in 16-token blocks scattered
// through the pool; the kernel follows the block table and the result equals
// attention over one contiguous array.  Decode reads the whole context every
// step and is memory-bandwidth bound ("Prefill/Decode" section of the
// inference-engine talk write-up), so the design is about keeping HBM busy:
//
//  * Work is measured in units = (sequence, kv head, 16-token block), all
//    G = Hq/Hkv query heads of a kv head served together so that every K/V
//    byte is read from HBM once.  The unit sequence is cut into equal
//    contiguous ranges, one per CTA of a persistent grid (a stream-K style
//    split: every CTA gets the same number of blocks whatever the mix of
//    context lengths).  The part of a (sequence, kv head) pair inside one
//    range is an item; a pair that straddles ranges is split-KV.
//  * Warp 8 (producer) walks the block table and streams each (block, kv
//    head) K slab and V slab -- 16 rows x d bf16, one contiguous 2-4 KB run
//    each -- with 1-D bulk (TMA) copies that complete on mbarriers,
//    evict-first in L2, into a shared-memory ring split into one sub-ring
//    per consumer warp (each warp consumes its stages strictly in order).
//  * Warps 0..7 (consumers) take an item's blocks round-robin, starting at
//    a warp given by the item's global index.  A lane owns 8 dims of a row
//    (one 16-byte shared load); q.K partial dots are summed across the
//    lanes of a row by a transpose-reduce, leaving one token score per lane
//    pair.  Online
//    softmax in the log2 domain, P.V on CUDA cores in fp32.  Rows past the
//    context are never loaded, so whatever the unused tail of a block holds
//    (NaN included) cannot reach the result.
//  * Warp 9 (merger) combines the 8 warps' (m, l, o) states of an item with
//    the log-sum-exp rule, off the consumers' critical path.  For a split
//    pair it stores the part's (m, l, o) in a per-range workspace slot; the
//    last part to arrive (atomic ticket) merges all of them in part order
//    and writes the output: one launch, no inter-CTA waiting, and results
//    that do not depend on timing.
//  * Every wait is an mbarrier wait bounded by %globaltimer; on expiry the
//    CTA records PKV_ERR_TIMEOUT and unwinds.
//  * Start-up: the launch may overlap the previous kernel on the stream.
//    Until that kernel has finished, the CTA only prefetches context_lens,
//    the block tables and q into L2, so its first reads after the wait hit
//    L2.
//  * e4m3 pools (one byte per element, the same layout and the same
//    kernel with half the bytes per slab): a lane loads its 8 dims with one
//    8-byte shared load and widens them with cvt.rn.f16x2.e4m3x2 (two codes
//    per instruction, exact: every e4m3 value is an fp16 value) and
//    cvt.f32.f16.  The K scale folds into q and the V scale into the final
//    1/l, so no per-element multiply is added.  The extra conversion work
//    per block makes the consumers the limit, so e4m3 pools with head
//    groups of 1 and 2 run 16 consumer warps; at d = 128 with G >= 2 the
//    block math runs on tensor cores instead (run_consumer_mma).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

// e4m3 pools with d = 128 and head groups of 2 or more take the consumers'
// block math on tensor cores (see run_consumer_mma); their slabs arrive as
// swizzled TMA tiles.  With one q head per kv head, 7 of the MMA's 8
// columns would be empty and the CUDA-core math is faster (LLaMA-13B MHA:
// 389 against 418 us).  A build can turn it off with PKV_DECODE_NO_MMA.
template <int D, int G, int EB>
constexpr bool use_mma() {
#ifdef PKV_DECODE_NO_MMA
    return false;
#else
    return D == 128 && EB == 1 && G >= 2;
#endif
}

// Consumer warps per CTA: 12 for head groups of 1, 11 for bf16 groups of 2
// (their per-lane state is small, and a third or fourth warp per scheduler
// hides more of the latency of the dependent shuffle and FMA chains; for
// groups of 2, timed at 9-12 and 16 warps, 11 ran the Qwen3-1.7B step in
// 20.5 us against 20.9 with 12, 20.7 with 10), 8 for groups of 4 (which need more than
// the 128 registers a thread that 14 warps leave), 6 for groups of 8 (about
// 220 registers a thread, no spills).  e4m3 pools
// (EB = 1) with groups of 1 or 2 on CUDA cores take 16: their blocks cost
// more issue (the widening) and half the ring bytes, so the same ring still
// gives each warp 3 stages.  The tensor-core block math (e4m3, d = 128,
// groups of 2) takes 10: 15.0 us on Qwen3-1.7B against 15.2 with 12, 8 or
// 11 and 15.5 with 14.  A build can force one count for every group with
// PKV_DECODE_CONSUMER_WARPS.
template <int D, int G, int EB>
constexpr int consumer_warps() {
#ifdef PKV_DECODE_CONSUMER_WARPS
    return PKV_DECODE_CONSUMER_WARPS;
#else
    return use_mma<D, G, EB>() ? (G <= 2 ? 10 : 8)
                               : (G <= 2 ? (EB == 1 ? 16 : (G == 2 ? 11 : 12)) : (G == 4 ? 8 : 6));
#endif
}
constexpr int kItemRing = 8;
// Smallest automatic range (blocks per CTA).  It sets the grid of small
// batches: Llama-3.2-1B (4 sequences, 336 units) ran in 12.2 us with 4,
// 12.6 with 6, 14.6 with 8 and 16.9 with 2 or 3 (split pairs' merges then
// cost more than the extra CTAs bring).
constexpr int kMinRangeUnits = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// One item = the part of one (sequence, kv head) pair that falls in one
// range of units.  When the pair spans several ranges (nparts > 1) each part
// leaves a partial result in slot `slot` of its range `r`: the pair's first
// part, in range r0, ends its range and uses slot slot0 = 1; every later
// part starts its range and uses slot 0.
struct __align__(16) ItemDesc {
    int32_t s, g, r, nparts;
    int32_t n, b0, b1, row;
    int32_t rot, slot, r0, slot0;  // rot: warp that takes the item's first block
};

struct DecodeParams {
    uint8_t* k_pool;  // written only by a fused step (its new rows)
    uint8_t* v_pool;
    const uint8_t* q;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* qsl;
    float* out;
    float2* part_ml;    // [max_ranges][2][G]      (m, l) of a partial result, log2 domain
    float* part_o;      // [max_ranges][2][G][D]   its unnormalised o
    uint32_t* counters; // [S][Hkv] arrival tickets of split pairs
    unsigned long long* err;
    int32_t num_blocks, hkv, hq, num_seqs, max_blocks, ctx_cap;
    int32_t range_units;  // units per range, 0 = automatic
    int32_t max_ranges;   // ranges the workspace holds
    float scale_log2;     // softmax scale * log2(e); e4m3 pools: also * k_scale
    float v_scale;        // e4m3 pools: the V pool's scale
    int32_t stall;        // test hook: the producer issues nothing (see arm_decode_stall)
    // Fused step (pkv_decode_step): this step's new rows, stored into the
    // pool by the warp that takes the pair's last block and used from
    // registers in that block.  k_new == nullptr: plain decode.
    const uint8_t* k_new;         // bf16 [S][Hkv][D]
    const uint8_t* v_new;
    const int32_t* slot_mapping;  // [S]
    float k_inv, v_inv;           // e4m3 pools: 1 / scale (fp32)
    // Shared prefix: the first skip_blocks blocks of every sequence were
    // attended by the shared-prefix kernel, which left one state per
    // (sequence, q head) in pre_ml ([S][Hq] (m, l), log2 domain) and pre_o
    // ([S][Hq][D], unnormalised).  The item holding a pair's first block
    // merges it into its own state.  null: no shared prefix.
    int32_t skip_blocks;
    const float2* pre_ml;
    const float* pre_o;
};

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int D, int G, int EB>
struct Cfg {
    static constexpr bool MMA = use_mma<D, G, EB>();
    static constexpr int ALIGN_PAD = MMA ? 1024 : 0;  // swizzled tiles need a 1024-byte aligned ring
    static constexpr int W = consumer_warps<D, G, EB>();  // consumer warps
    static_assert(W >= 1 && W <= 16, "consumer warps");
    // Lanes per q head in the merger's weight reduction: W rounded up to a
    // power of two (the extra lanes carry empty states).
    static constexpr int MERGE_LANES = W <= 1 ? 1 : W <= 2 ? 2 : W <= 4 ? 4 : W <= 8 ? 8 : 16;
    static constexpr int MERGE_BUFS = W > 8 ? 1 : 2;  // consumer states the merger can lag by
    static constexpr int PRODUCER_WARP = W;
    static constexpr int MERGER_WARP = W + 1;
    static constexpr int THREADS = 32 * (W + 2);
    static constexpr int LPR = D / 8;                  // lanes per K/V row, 8 dims (16 B) each
    static constexpr int RPP = 32 / LPR;               // rows per warp pass
    static constexpr int NV = kBlockSize / RPP;        // rows per lane per block
    static constexpr int SLAB = kBlockSize * D * EB;   // bytes of one (block, kv head); EB = 2 (bf16) or 1 (e4m3)
    static constexpr int STAGE_BYTES = 2 * SLAB;       // K slab then V slab
    static constexpr int QBYTES = G * D * 2;
    static constexpr int HG = G < 4 ? G : 4;           // heads per pass over K
    // Everything but the ring (offsets relative to the end of the ring).
    static constexpr int R_ITEMQ = 0;
    static constexpr int R_DESC = R_ITEMQ + kItemRing * QBYTES;
    static constexpr int R_P = R_DESC + kItemRing * (int)sizeof(ItemDesc);
    static constexpr int R_MO = R_P + W * G * kBlockSize * 8;  // p stored as (p, p)
    static constexpr int R_ML = R_MO + MERGE_BUFS * W * G * D * 4;
    static constexpr int R_WT = R_ML + MERGE_BUFS * W * G * 8;  // merger: [G][W] weights, then [G] prefix weights
    static constexpr int R_MSM = align_up(R_WT + G * (W + 1) * 4, 8);  // merger: [G] (M, L), float2-aligned
    static constexpr int R_BAR = align_up(R_MSM + G * 8, 8);
    static constexpr int STAGES_FIT = (220 * 1024 - R_BAR - 64 * 8 - 16 - ALIGN_PAD) / STAGE_BYTES;
    // Each consumer warp owns SW consecutive stages that it consumes in
    // order (an mbarrier parity wait is only exact when the waiter is at
    // most one phase ahead of the barrier).
    static constexpr int SW_FIT = STAGES_FIT / W;
    static constexpr int SW_CAP = EB == 2 ? 6 : 12;    // the same bytes in flight for either element
    static constexpr int SW = SW_FIT < SW_CAP ? SW_FIT : SW_CAP;
    static constexpr int STAGES = SW * W;
    static constexpr int NBAR = 2 * STAGES + 2 * kItemRing + 2 * MERGE_BUFS;
    static constexpr int OFF_REST = STAGES * STAGE_BYTES;
    static constexpr int OFF_ITEMQ = OFF_REST + R_ITEMQ;
    static constexpr int OFF_DESC = OFF_REST + R_DESC;
    static constexpr int OFF_P = OFF_REST + R_P;
    static constexpr int OFF_MO = OFF_REST + R_MO;
    static constexpr int OFF_ML = OFF_REST + R_ML;
    static constexpr int OFF_WT = OFF_REST + R_WT;
    static constexpr int OFF_MSM = OFF_REST + R_MSM;
    static constexpr int OFF_BAR = OFF_REST + R_BAR;
    static constexpr int OFF_FLAG = OFF_BAR + NBAR * 8;
    static constexpr int OFF_NEW = OFF_FLAG + 16;  // [STAGES] fused step: slot of a stage's new row, or -1
    static constexpr int SMEM = OFF_NEW + STAGES * 4 + ALIGN_PAD;
    static_assert(SW >= 1, "ring too shallow");
    static_assert(OFF_ITEMQ % 16 == 0 && OFF_DESC % 16 == 0 && OFF_P % 16 == 0 && OFF_MO % 16 == 0 &&
                      OFF_ML % 8 == 0 && OFF_MSM % 8 == 0 && OFF_BAR % 8 == 0 && OFF_NEW % 4 == 0 &&
                      STAGE_BYTES % 16 == 0 && (!MMA || STAGE_BYTES % 1024 == 0),
                  "shared-memory regions aligned for their widest access");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(NV * RPP == kBlockSize, "rows");
};

struct Bars {
    uint64_t* full;    // [STAGES]   producer -> consumer (tx bytes)
    uint64_t* empty;   // [STAGES]   consumer -> producer
    uint64_t* ifull;   // [ITEMS]    item descriptor + q landed
    uint64_t* iempty;  // [ITEMS]    consumers and merger read the descriptor
    uint64_t* mfull;   // [MERGE]    8 consumer states published
    uint64_t* mempty;  // [MERGE]    merger done with the buffer
};

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Sum NV per-lane values over the LPR lanes that share a row group; on
// return lane l holds the total of value index (l >> 1) & (NV - 1).
template <int NV, int LPR>
__device__ __forceinline__ float transpose_reduce(float (&v)[NV], int lane) {
    int off = LPR / 2;
#pragma unroll
    for (int n = NV; n > 1; n >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (; off >= 1; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    return v[0];
}

// A fused step stores a sequence's new row only at the slot of its last
// position n - 1: row srow = (n - 1) % 16 of the pair's last block, whose id
// must lie inside the pool.
__device__ __forceinline__ bool new_row_fits(int slot, int phys, int srow, int num_blocks) {
    return slot >= 0 && phys >= 0 && phys < num_blocks && slot == phys * kBlockSize + srow;
}

// e4m3 pools, fused step: quantise this lane's 8 elements of the new K and V
// rows (bytes `off` of k_new/v_new), store the codes to the pool (byte `at`)
// and over the stage's row (kr, V at kr + slab).  Out of line: it runs once
// per pair and keeps its registers out of the consumers' block loop.
__device__ __noinline__ void store_new_row_e4m3(const DecodeParams& P, size_t off, size_t at, uint8_t* kr,
                                                int slab) {
    const uint2 kc = quantise8(__ldg(reinterpret_cast<const uint4*>(P.k_new + off)), P.k_inv);
    const uint2 vc = quantise8(__ldg(reinterpret_cast<const uint4*>(P.v_new + off)), P.v_inv);
    *reinterpret_cast<uint2*>(P.k_pool + at) = kc;
    *reinterpret_cast<uint2*>(P.v_pool + at) = vc;
    *reinterpret_cast<uint2*>(kr) = kc;
    *reinterpret_cast<uint2*>(kr + slab) = vc;
    // The stage is refilled by bulk copies (async proxy) once the warp
    // releases it.
    fence_proxy_async_shared();
}

// Units per range when the caller lets the kernel choose: the total over
// the grid, at least kMinRangeUnits.  When every pair has the same number
// of units u (a batch of equal contexts), a range of whole pairs -- u times
// the pairs it then holds -- is taken instead if it costs at most 15% more
// units: no pair is split, so no part waits for another's partial result
// (Qwen3-1.7B, 34 x 640: 80 units on 136 CTAs beat 72 on 152).
__device__ __forceinline__ long long auto_range_units(long long T, unsigned grid, int umin, int umax) {
    long long RU = max(static_cast<long long>(kMinRangeUnits), (T + grid - 1) / grid);
    if (umin == umax && umin > 0) {
        const long long whole = static_cast<long long>(umin) * ((RU + umin - 1) / umin);
        if (whole * 20 <= RU * 23) RU = whole;
    }
    return RU;
}

// Units of work of one kv head of sequence s: one per 16-token block of its
// context past the shared prefix (at least one, so that an empty context
// still yields its output row), 0 for rows that are not decode rows.  The
// context length is clamped to what the block table can address.
__device__ __forceinline__ int seq_units(const DecodeParams& P, int s, int& n_out, bool report) {
    const int qlen = P.qsl ? (__ldg(P.qsl + s + 1) - __ldg(P.qsl + s)) : 1;
    if (qlen != 1) {
        n_out = 0;
        return 0;
    }
    int n = __ldg(P.context_lens + s);
    if (n < 0 || n > P.ctx_cap) {
        if (report) record_error(P.err, kErrRange, static_cast<uint32_t>(s));
        n = n < 0 ? 0 : P.ctx_cap;
    }
    n_out = n;
    return max(1, (n + kBlockSize - 1) / kBlockSize - P.skip_blocks);
}

__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) { return make_float2(bf16lo(u), bf16hi(u)); }

// Tiled 2-D TMA load of a box at (x, y) of `map` into shared memory,
// completed on `bar` as tx bytes, with an L2 cache policy.
__device__ __forceinline__ void tma_tile_g2s(void* smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                             uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Byte offset of 16-byte chunk c of row r in a slab stored as 128-byte
// swizzled panels of 16 rows (a tiled TMA copy with the 128-byte swizzle:
// within a row's 128 bytes the chunk index is XORed with r mod 8).
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>((c >> 3) * (kBlockSize * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}


__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h) {
    float2 r;
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(h));
    return r;
}

// Four e4m3 codes (bytes of w, lowest first) -> their values as fp32, in
// order: a = (code 0, code 1), b = (code 2, code 3).  e4m3 -> fp16 is exact
// (every e4m3 value, subnormals included, is a normal fp16 or zero), and so
// is fp16 -> fp32; a NaN code gives NaN.
__device__ __forceinline__ void e4m3x4_to_float(uint32_t w, float2& a, float2& b) {
    uint32_t h01, h23;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h01), "=r"(h23)
        : "r"(w));
    a = f16x2_to_float2(h01);
    b = f16x2_to_float2(h23);
}

// o / l of one output chunk; an e4m3 pool's o is in code units, so its V
// scale is applied here (o / l is a weighted mean of codes, at most 448).
template <int EB>
__device__ __forceinline__ float4 normalise(float4 a, float l, float v_scale) {
    if constexpr (EB == 2) {
        return make_float4(a.x / l, a.y / l, a.z / l, a.w / l);
    } else {
        const float f = v_scale / l;
        return make_float4(a.x * f, a.y * f, a.z * f, a.w * f);
    }
}

// One 16-row block for one warp.  Lane (sub, cl) owns dims 8cl..8cl+7 of
// rows i*RPP + sub.  q.K partial dots use packed fp32x2 FMAs; the row sums
// come from a transpose-reduce over the LPR lanes of a row; P.V accumulates
// with packed fp32x2 FMAs.  Rows >= valid are never loaded.
template <int D, int G, int EB>
__device__ __forceinline__ void compute_block(const uint8_t* kst, const uint8_t* vst, int valid,
                                              const float2 (&q2)[G][4], float (&m)[G], float (&lsum)[G],
                                              float2 (&o2)[G][4], float2* psm, int lane) {
    using C = Cfg<D, G, EB>;
    const int sub = lane / C::LPR;
    const int cl = lane % C::LPR;
    const int myrow = ((lane >> 1) & (C::NV - 1)) * C::RPP + sub;
#pragma unroll
    for (int g0 = 0; g0 < G; g0 += C::HG) {
        float acc[C::HG][C::NV];
#pragma unroll
        for (int i = 0; i < C::NV; ++i) {
            const int row = i * C::RPP + sub;
            float2 k0, k1, k2, k3;
            if constexpr (EB == 2) {
                uint4 u = make_uint4(0u, 0u, 0u, 0u);
                if (row < valid) u = lds128(kst + row * D * 2 + cl * 16);
                k0 = bf16x2_to_float2(u.x), k1 = bf16x2_to_float2(u.y);
                k2 = bf16x2_to_float2(u.z), k3 = bf16x2_to_float2(u.w);
            } else {  // e4m3 codes; q carries k_scale
                uint2 u = make_uint2(0u, 0u);
                if (row < valid) u = lds64(kst + row * D + cl * 8);
                e4m3x4_to_float(u.x, k0, k1);
                e4m3x4_to_float(u.y, k2, k3);
            }
#pragma unroll
            for (int g = 0; g < C::HG; ++g) {
                float2 a = __fmul2_rn(q2[g0 + g][0], k0);
                a = __ffma2_rn(q2[g0 + g][1], k1, a);
                a = __ffma2_rn(q2[g0 + g][2], k2, a);
                a = __ffma2_rn(q2[g0 + g][3], k3, a);
                acc[g][i] = a.x + a.y;
            }
        }
#pragma unroll
        for (int g = 0; g < C::HG; ++g) {
            float sc = transpose_reduce<C::NV, C::LPR>(acc[g], lane);
            sc = (myrow < valid) ? sc : -INFINITY;
            const float mb = warp_max_redux(sc);
            // The reference m moves only when a block's maximum exceeds it by
            // more than 2^8 (log2 units; the condition is warp-uniform): p
            // stays below 256 and O and l are rescaled on few blocks.  The
            // merge divides by l taken against the same reference.
            if (mb > m[g0 + g] + kRescaleThreshold) {
                const float alpha = fast_exp2(m[g0 + g] - mb);
                lsum[g0 + g] *= alpha;
                const float2 al = make_float2(alpha, alpha);
#pragma unroll
                for (int j = 0; j < 4; ++j) o2[g0 + g][j] = __fmul2_rn(o2[g0 + g][j], al);
                m[g0 + g] = mb;
            }
            const float p = fast_exp2(sc - m[g0 + g]);
            lsum[g0 + g] += (lane & 1) ? 0.f : p;
            if (!(lane & 1)) psm[myrow * G + g0 + g] = make_float2(p, p);
        }
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < C::NV; ++i) {
        const int row = i * C::RPP + sub;
        if (row < valid) {
            float2 v0, v1, v2, v3;
            if constexpr (EB == 2) {
                const uint4 u = lds128(vst + row * D * 2 + cl * 16);
                v0 = bf16x2_to_float2(u.x), v1 = bf16x2_to_float2(u.y);
                v2 = bf16x2_to_float2(u.z), v3 = bf16x2_to_float2(u.w);
            } else {  // e4m3 codes: v_scale is applied with 1/l at the end
                const uint2 u = lds64(vst + row * D + cl * 8);
                e4m3x4_to_float(u.x, v0, v1);
                e4m3x4_to_float(u.y, v2, v3);
            }
            // p of this row for every head: psm is [row][head] (p, p) pairs,
            // read two heads per 16-byte load.
            float2 pr[G];
            if constexpr (G % 2 == 0) {
#pragma unroll
                for (int g = 0; g < G; g += 2) {
                    const float4 q4 = *reinterpret_cast<const float4*>(&psm[row * G + g]);
                    pr[g] = make_float2(q4.x, q4.y);
                    pr[g + 1] = make_float2(q4.z, q4.w);
                }
            } else {
#pragma unroll
                for (int g = 0; g < G; ++g) pr[g] = psm[row * G + g];
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                o2[g][0] = __ffma2_rn(pr[g], v0, o2[g][0]);
                o2[g][1] = __ffma2_rn(pr[g], v1, o2[g][1]);
                o2[g][2] = __ffma2_rn(pr[g], v2, o2[g][2]);
                o2[g][3] = __ffma2_rn(pr[g], v3, o2[g][3]);
            }
        }
    }
    __syncwarp();
}

template <int D, int G, int EB, bool FUSED>
__device__ void run_producer(const DecodeParams& P, const CUtensorMap* tmk, const CUtensorMap* tmv, uint8_t* smem,
                             const Bars& B, volatile int* abort_flag, int lane) {
    using C = Cfg<D, G, EB>;
    ItemDesc* descs = reinterpret_cast<ItemDesc*>(smem + C::OFF_DESC);
    int* stage_new = reinterpret_cast<int*>(smem + C::OFF_NEW);
    const unsigned FULL = 0xffffffffu;
    // Work is the sequence of units (s, kv head, block), sequences in order,
    // kv heads in order within a sequence, blocks in order within a head.
    // It is cut into ranges of RU consecutive units; range r goes to CTA
    // r % grid.  Every CTA derives the same cut from context_lens.
    //
    // Window of 32 sequences: lane j describes sequence s0 + j with its units
    // per kv head (u), context (n) and the inclusive prefix of u over the
    // window (incl); base = units per kv head before the window.
    struct Win {
        int s0, base, u, n, incl;
    };
    auto load_window = [&](Win& W, bool report) {
        const int s = W.s0 + lane;
        W.u = 0;
        W.n = 0;
        if (s < P.num_seqs) W.u = seq_units(P, s, W.n, report);
        W.incl = W.u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(FULL, W.incl, o);
            if (lane >= o) W.incl += t;
        }
    };
    // Move W forward to the sequence holding unit x; returns its lane or -1.
    auto locate = [&](Win& W, long long x) -> int {
        while (true) {
            const unsigned hit = __ballot_sync(FULL, static_cast<long long>(W.base + W.incl) * P.hkv > x);
            if (hit) return __ffs(hit) - 1;
            if (W.s0 + 32 >= P.num_seqs) return -1;  // cannot happen for consistent inputs
            W.base += __shfl_sync(FULL, W.incl, 31);
            W.s0 += 32;
            load_window(W, false);
        }
    };
    Win win{0, 0, 0, 0, 0};
    load_window(win, blockIdx.x == 0);
    long long per_head = __shfl_sync(FULL, win.incl, 31);
    // Smallest and largest units of a decode row's pair (rows with none
    // excluded): equal for a batch whose contexts span the same blocks.
    int umin = win.u > 0 ? win.u : INT32_MAX, umax = win.u;
    for (int s0 = 32; s0 < P.num_seqs; s0 += 32) {
        int n, u = 0;
        if (s0 + lane < P.num_seqs) u = seq_units(P, s0 + lane, n, blockIdx.x == 0);
        umin = min(umin, u > 0 ? u : INT32_MAX);
        umax = max(umax, u);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) u += __shfl_xor_sync(FULL, u, o);
        per_head += u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        umin = min(umin, __shfl_xor_sync(FULL, umin, o));
        umax = max(umax, __shfl_xor_sync(FULL, umax, o));
    }
    const long long T = per_head * P.hkv;
    long long RU = P.range_units;
    if (RU <= 0) RU = auto_range_units(T, gridDim.x, umin, umax);
    const long long shift_max = max(8LL, RU / 8);  // largest move of a range boundary (see snap)
    long long R = (T + RU - 1) / RU;
    if (R > P.max_ranges) {  // cannot happen with a workspace sized by the library
        record_error(P.err, kErrRange, 0xFFFFFFFEu);
        R = P.max_ranges;
    }

    const uint64_t policy = l2_policy_evict_first();
    uint32_t given = 0;  // lane w < W: blocks handed to consumer warp w so far
    uint32_t item_seq = 0;
    bool aborted = false;

    // Emit the item of the pair holding unit `pos` (located in W), clipped to
    // [pos, hi); returns the unit after it.
    auto emit_item = [&](Win& W, long long pos, long long hi, long long lo, long long r) -> long long {
        const int j = locate(W, pos);
        if (j < 0) {
            record_error(P.err, kErrRange, 0xFFFFFFFFu);
            return hi;
        }
        const int win_s0 = W.s0, win_base = W.base, w_u = W.u, w_n = W.n, w_incl = W.incl;
        const long long end = hi;
        const int s = win_s0 + j;
        const int u = __shfl_sync(FULL, w_u, j);
        const int n = __shfl_sync(FULL, w_n, j);
        const long long seq0 = static_cast<long long>(win_base + __shfl_sync(FULL, w_incl, j) - u) * P.hkv;
        const int g = static_cast<int>((pos - seq0) / u);
        const long long P0 = seq0 + static_cast<long long>(g) * u;  // the pair's units: [P0, P0 + u)
        const long long u1 = min(P0 + u, end);
        // Block indices in the sequence's table: the pair's units start at
        // its first block past the shared prefix.
        const int nblk = (n + kBlockSize - 1) / kBlockSize;
        const int b0 = P.skip_blocks + static_cast<int>(pos - P0);
        const int b1 = min(P.skip_blocks + static_cast<int>(u1 - P0), nblk);
        const long long r0 = P0 / RU;
        // A pair is split by every boundary strictly inside it: for a pair
        // longer than a range these are the multiples of RU; a shorter pair
        // holds at most one, which stays only when it did not snap to an
        // edge.  The parts are ranges r0, r0 + 1, ... (r0 = P0 / RU).
        int nparts;
        if (u > RU) {
            nparts = static_cast<int>((P0 + u - 1) / RU - r0 + 1);
        } else {
            const long long b = (r0 + 1) * RU;  // the only nominal boundary that can fall inside
            const long long down = b - P0, up = P0 + u - b;
            nparts = (b > P0 && b < P0 + u && min(down, up) > shift_max) ? 2 : 1;
        }
        const int rot = static_cast<int>(pos % C::W);
        const int row = P.qsl ? __ldg(P.qsl + s) : s;
        const int32_t* trow = P.block_tables + static_cast<size_t>(s) * P.max_blocks;
        // First batch of table entries, requested before the descriptor work.
        int e = 0;
        if (lane < b1 - b0) e = __ldg(trow + b0 + lane);
        // Fused step (bf16 pools): the item holds the pair's last block, whose
        // row srow is the new token; its slot is read now, used when that
        // block is issued.
        const bool has_new = FUSED && n > 0 && b1 == nblk && b1 > b0;
        const int srow = (n - 1) % kBlockSize;
        int new_slot = -1;
        if (has_new && lane == 0) new_slot = __ldg(P.slot_mapping + s);
        const uint32_t slot = item_seq % kItemRing;
        if (!mbar_wait_warp(&B.iempty[slot], ((item_seq / kItemRing) & 1) ^ 1)) {
            aborted = true;
            return hi;
        }
        if (lane == 0) {
            ItemDesc d;
            d.s = s; d.g = g; d.r = static_cast<int>(r); d.nparts = nparts;
            d.n = n; d.b0 = b0; d.b1 = max(b0, b1); d.row = row;
            d.rot = rot;
            // A split pair's first part ends its range (slot 1); every later
            // part starts its range (slot 0).
            d.slot = (nparts > 1 && P0 >= lo) ? 1 : 0;
            d.r0 = static_cast<int>(r0);
            d.slot0 = 1;
            descs[slot] = d;
            mbar_arrive_expect_tx(&B.ifull[slot], C::QBYTES);
            const uint8_t* qsrc = P.q + (static_cast<size_t>(row) * P.hq + static_cast<size_t>(g) * G) * D * 2;
            bulk_g2s(smem + C::OFF_ITEMQ + slot * C::QBYTES, qsrc, C::QBYTES, &B.ifull[slot]);
        }
        __syncwarp();
        ++item_seq;
        // Stream the item's blocks.  Block b goes to consumer warp
        // w = (b + rot) % W, into stage j % SW of w's sub-ring, where j
        // counts the blocks w has been given so far (lane w keeps that
        // count in `given`).  Blocks go out in batches of up to min(32,
        // STAGES): lane k of a batch waits for its own stage and issues
        // that block's two copies.  A batch holds at most SW blocks of any
        // warp, so a lane's stage was last used by a block of an earlier
        // batch and no lane waits on its own batch.  The next batch's
        // table entries are requested before this batch's copies.
        constexpr int kBatch = C::STAGES < 32 ? C::STAGES : 32;
        for (int base = b0; base < b1; base += kBatch) {
            const int cnt = min(kBatch, b1 - base);
            int e_next = 0;
            if (lane < kBatch && base + kBatch + lane < b1) e_next = __ldg(trow + base + kBatch + lane);
            const int bl = base - b0 + lane;  // block index within the item
            const int w = (bl + rot) % C::W;
            const int first_w = (w - rot + C::W) % C::W;
            const uint32_t jw = static_cast<uint32_t>(__shfl_sync(FULL, static_cast<int>(given), w)) +
                                static_cast<uint32_t>((bl - first_w) / C::W);
            const uint32_t st = static_cast<uint32_t>(w * C::SW) + jw % C::SW;
            // The lane of this batch (if any) that issues the pair's last block.
            const int last_lane = has_new ? b1 - 1 - base : -1;
            int ns = -1;
            if (last_lane >= 0 && last_lane < cnt) ns = __shfl_sync(FULL, new_slot, 0);
            int bad = 0;
            if (lane < cnt) {
                int phys = e;
                if (phys < 0 || phys >= P.num_blocks) {
                    record_error(P.err, kErrRange, static_cast<uint32_t>(s));
                    phys = 0;  // never dereference an invalid id
                }
                if (!mbar_wait(&B.empty[st], ((jw / C::SW) & 1) ^ 1)) {
                    bad = 1;
                } else {
                    const size_t slab = (static_cast<size_t>(phys) * P.hkv + g) * C::SLAB;
                    uint8_t* dst = smem + st * C::STAGE_BYTES;
                    // Tell the consumer whether this stage carries a new row
                    // (visible to it through the arrive below).
                    const bool fresh = lane == last_lane && new_row_fits(ns, e, srow, P.num_blocks);
                    if constexpr (FUSED) stage_new[st] = fresh ? ns : -1;
                    if (lane == last_lane && ns >= 0 && !fresh) {
                        // A slot other than position n - 1's: reported, not
                        // written (the pool's row is used as it is).
                        record_error(P.err, kErrRange, static_cast<uint32_t>(s));
                    }
                    if (FUSED && EB == 2 && fresh && !C::MMA) {
                        // Rows before the new token from the pool, the new
                        // row from k_new/v_new (rows past it are never read).
                        constexpr uint32_t kRow = D * EB;
                        const size_t nr = (static_cast<size_t>(s) * P.hkv + g) * kRow;
                        mbar_arrive_expect_tx(&B.full[st], 2 * (srow + 1) * kRow);
                        if (srow > 0) {
                            bulk_g2s_hint(dst, P.k_pool + slab, srow * kRow, &B.full[st], policy);
                            bulk_g2s_hint(dst + C::SLAB, P.v_pool + slab, srow * kRow, &B.full[st], policy);
                        }
                        bulk_g2s(dst + srow * kRow, P.k_new + nr, kRow, &B.full[st]);
                        bulk_g2s(dst + C::SLAB + srow * kRow, P.v_new + nr, kRow, &B.full[st]);
                    } else if constexpr (C::MMA) {
                        // One swizzled 16-row tile per slab (rows of 128
                        // bytes); its first row in the pool's row space.
                        static_assert(D * EB == 128, "one 128-byte panel per row");
                        const int y = (phys * P.hkv + g) * kBlockSize;
                        mbar_arrive_expect_tx(&B.full[st], 2 * C::SLAB);
                        tma_tile_g2s(dst, tmk, 0, y, &B.full[st], policy);
                        tma_tile_g2s(dst + C::SLAB, tmv, 0, y, &B.full[st], policy);
                    } else {
                        mbar_arrive_expect_tx(&B.full[st], 2 * C::SLAB);
                        bulk_g2s_hint(dst, P.k_pool + slab, C::SLAB, &B.full[st], policy);
                        bulk_g2s_hint(dst + C::SLAB, P.v_pool + slab, C::SLAB, &B.full[st], policy);
                    }
                }
            }
            if (__any_sync(FULL, bad)) {
                // Let this batch's issued copies land before unwinding.
                if (lane < cnt && !bad) mbar_wait(&B.full[st], (jw / C::SW) & 1);
                aborted = true;
                break;
            }
            e = e_next;
        }
        // Blocks each warp received from this item.
        if (lane < C::W && !aborted) {
            const int first_w = (lane - rot + C::W) % C::W;
            const int nb = b1 - b0;
            if (first_w < nb)
                given += static_cast<uint32_t>((nb - first_w + C::W - 1) / C::W);
        }
        return u1;
    };

    // Range boundaries: nominally r * RU.  A boundary that falls within
    // `shift_max` units of an edge of the pair it cuts moves to that edge
    // (the pair is not split and the range sizes change by little); other
    // boundaries split their pair.  Only pairs no longer than a range move:
    // boundaries inside longer pairs stay at multiples of RU.
    auto snap = [&](Win& W, long long b) -> long long {
        if (b <= 0) return 0;
        if (b >= T) return T;
        const int j = locate(W, b);
        if (j < 0) return b;
        const int u = __shfl_sync(FULL, W.u, j);
        const long long seq0 = static_cast<long long>(W.base + __shfl_sync(FULL, W.incl, j) - u) * P.hkv;
        const long long P0 = seq0 + (b - seq0) / u * u;
        if (b == P0 || u > RU) return b;
        const long long down = b - P0, up = P0 + u - b;
        if (min(down, up) > shift_max) return b;
        return (down <= up) ? P0 : P0 + u;
    };
    for (long long r = blockIdx.x; r < R && !aborted; r += gridDim.x) {
        const long long lo = snap(win, r * RU);
        long long hi;
        {
            Win tw = win;
            hi = snap(tw, (r + 1) * RU);
        }
        if (lo >= hi) continue;
        // When the range's last item is the first part of a pair that goes
        // on into the next range, stream it first: both parts of every split
        // pair then run at the start of their CTAs, and their merge overlaps
        // the rest of the work instead of trailing it.
        long long stop = hi;
        {
            Win tw = win;
            const int j = locate(tw, hi - 1);
            if (j >= 0) {
                const int u = __shfl_sync(FULL, tw.u, j);
                const long long seq0 = static_cast<long long>(tw.base + __shfl_sync(FULL, tw.incl, j) - u) * P.hkv;
                const long long P0 = seq0 + (hi - 1 - seq0) / u * u;
                if (P0 > lo && P0 + u > hi) {
                    emit_item(tw, P0, hi, lo, r);
                    stop = P0;
                }
            }
        }
        long long pos = lo;
        while (pos < stop && !aborted) pos = emit_item(win, pos, stop, lo, r);
    }
    if (!aborted) {  // end marker
        const uint32_t slot = item_seq % kItemRing;
        if (mbar_wait_warp(&B.iempty[slot], ((item_seq / kItemRing) & 1) ^ 1)) {
            if (lane == 0) {
                descs[slot].s = -1;
                mbar_arrive(&B.ifull[slot]);
            }
            __syncwarp();
            ++item_seq;
        } else {
            aborted = true;
        }
    }
    if (aborted) {
        *abort_flag = 1;
        record_error(P.err, kErrTimeout, 1u);
        // Never leave with bulk copies still in flight.
        if (lane < C::W) {
            for (uint32_t k = 0; k < C::SW; ++k) {
                if (k < given) {
                    const uint32_t jl = given - 1 - ((given - 1 - k) % C::SW);  // last use of stage k
                    mbar_wait(&B.full[lane * C::SW + k], (jl / C::SW) & 1);
                }
            }
        }
        if (lane == 0) {
            for (uint32_t sl = 0; sl < kItemRing; ++sl)
                if (sl < item_seq) mbar_wait(&B.ifull[sl], ((item_seq - 1 - sl) / kItemRing) & 1);
        }
    }
}

// Fused step: if the producer noted a new row (slot ns >= 0) for this stage,
// row srow = ns % 16 of the block is the new token: store it to the pool.
// bf16 pools: the producer placed it in the stage.  e4m3 pools: quantise it
// here and write the codes over the stage's row too.  Lane (sub, cl) moves
// 8 elements (the lane layout of a K/V row in compute_block).
template <int D, int G, int EB>
__device__ __forceinline__ void store_stage_new_row(const DecodeParams& P, const ItemDesc& d, uint8_t* kst, int ns,
                                                    int lane) {
    using C = Cfg<D, G, EB>;
    if (ns < 0) return;
    const int sub = lane / C::LPR;
    const int cl = lane % C::LPR;
    const int srow = ns % kBlockSize;
    if (sub == srow % C::RPP) {
        const size_t at = (static_cast<size_t>(ns / kBlockSize) * P.hkv + d.g) * C::SLAB +
                          static_cast<size_t>(srow) * D * EB + cl * 8 * EB;
        // The stage holds the row at its place in the slab, or (MMA
        // configurations) in the swizzled tile layout.
        const int byte = cl * 8 * EB;
        uint8_t* kr = kst + (C::MMA ? static_cast<int>(swz(srow, byte >> 4)) + (byte & 15) : srow * D * EB + byte);
        if constexpr (EB == 2) {
            *reinterpret_cast<uint4*>(P.k_pool + at) = lds128(kr);
            *reinterpret_cast<uint4*>(P.v_pool + at) = lds128(kr + C::SLAB);
        } else {
            const size_t off = (static_cast<size_t>(d.s) * P.hkv + d.g) * D * 2 + cl * 16;
            store_new_row_e4m3(P, off, at, kr, C::SLAB);
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------- MMA consumers
// e4m3 pools with d = 128 and G >= 2 run the consumers' block math on
// warp-level tensor cores (mma.sync m16n8k16, f16 operands, fp32
// accumulators); their slabs arrive as tiled TMA copies with the 128-byte
// swizzle (one 16-row box of 128 codes per slab), so no fragment load waits
// on a bank conflict.  Per
// 16-row block, S = K q^T (16 keys x 8 columns: the group's G heads, the
// rest zero) and O^T += V^T P^T (16 dims x 8 heads per MMA).  Lane (g, t) =
// (lane / 4, lane % 4) holds the MMA fragments; the contractions are sums,
// so their order is permuted:
//  * q.K^T: lane (g, t) reads 16-byte chunks 2t and 2t+1 of key rows g and
//    g+8 (32 codes); q of head g over the same dims is its B fragment;
//  * P.V: lane (g, t) reads chunk g (16 codes) of key rows 2t, 2t+1, 2t+8,
//    2t+9; MMA 2i's rows g and g+8 are dims 16g + 4i and 16g + 4i + 1, MMA
//    2i+1's dims 16g + 4i + 2 and + 3.
// With the swizzle (chunk c of row r at 16 (c xor (r mod 8))), the 8 lanes
// of every 16-byte load phase hit 8 different bank groups.  S lands as keys
// {g, g+8} x heads {2t, 2t+1}, the heads of the lane's O columns, so the
// online softmax moves no data; P goes to the B layout (head g, keys 2t,
// 2t+1, 2t+8, 2t+9) by shuffles.  P is split into an f16 hi and lo part
// (P.V runs twice), P to 2^-22 relative.  e4m3 codes widen to f16 exactly;
// q is scaled per head by a power of two into [1, 2) (exact) for f16, the
// factor given back to the scores.  Rows past the context are masked in S
// and zeroed in V (0 x NaN would poison the sum).
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two e4m3 codes (low 16 bits of w) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t w) {
    uint32_t h;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(h) : "r"(w));
    return h;
}

// Two floats -> f16x2 (nearest even), lo in the low half.
__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// A pair of probabilities (below 256) as two f16 MMA operands: hi is p
// rounded, lo the rounded rest, so hi + lo = p to 2^-22 relative.
__device__ __forceinline__ void split_pair_f16(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = f16x2_rn(a, b);
    const float2 h = f16x2_to_float2(hi);
    lo = f16x2_rn(a - h.x, b - h.y);
}

template <int D, int G>
__device__ __forceinline__ void compute_block_mma(const uint8_t* kst, const uint8_t* vst, int valid,
                                                  const uint32_t (&qb)[D / 8], float f0, float f1, float& m0,
                                                  float& m1, float& l0, float& l1, float (&o)[D / 16][4],
                                                  int lane) {
    const unsigned FULL = 0xffffffffu;
    const int g = lane >> 2, t = lane & 3;
    // ---- S = K q^T: chunk 2t + c of key rows g and g + 8, 16 codes =
    // k-steps 4c .. 4c + 3.
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
        const uint4 r0 = lds128(kst + swz(g, 2 * t + c)), r8 = lds128(kst + swz(g + 8, 2 * t + c));
        const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w}, w8[4] = {r8.x, r8.y, r8.z, r8.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const int kk = 4 * c + w;
            mma_f16(s, e4m3x2_f16x2(w0[w]), e4m3x2_f16x2(w8[w]), e4m3x2_f16x2(w0[w] >> 16),
                    e4m3x2_f16x2(w8[w] >> 16), qb[2 * kk], qb[2 * kk + 1]);
        }
    }
    // ---- online softmax (log2 domain) on keys {g, g+8} x heads {2t, 2t+1}
    const bool vg = g < valid, vg8 = g + 8 < valid;
    const float x00 = vg ? s[0] * f0 : -INFINITY, x01 = vg ? s[1] * f1 : -INFINITY;
    const float x10 = vg8 ? s[2] * f0 : -INFINITY, x11 = vg8 ? s[3] * f1 : -INFINITY;
    float mb0 = fmaxf(x00, x10), mb1 = fmaxf(x01, x11);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mb0 = fmaxf(mb0, __shfl_xor_sync(FULL, mb0, off));
        mb1 = fmaxf(mb1, __shfl_xor_sync(FULL, mb1, off));
    }
    // The reference moves only when the block's maximum exceeds it by more
    // than 2^8, so P stays below 256 and O is rescaled on few blocks.
    if (mb0 > m0 + kRescaleThreshold) {
        const float a = fast_exp2(m0 - mb0);
        l0 *= a;
#pragma unroll
        for (int mm = 0; mm < D / 16; ++mm) o[mm][0] *= a, o[mm][2] *= a;
        m0 = mb0;
    }
    if (mb1 > m1 + kRescaleThreshold) {
        const float a = fast_exp2(m1 - mb1);
        l1 *= a;
#pragma unroll
        for (int mm = 0; mm < D / 16; ++mm) o[mm][1] *= a, o[mm][3] *= a;
        m1 = mb1;
    }
    const float p00 = fast_exp2(x00 - m0), p01 = fast_exp2(x01 - m1);
    const float p10 = fast_exp2(x10 - m0), p11 = fast_exp2(x11 - m1);
    l0 += p00 + p10;
    l1 += p01 + p11;
    // ---- P^T in the B layout: head g, keys (2t, 2t+1) and (2t+8, 2t+9).
    // Key 2t of head g sits in lane 8t + g/2 (key 2t+1: + 4), as element
    // g % 2 of its (key, key+8) pair.
    uint32_t x0h, x0l, x1h, x1l;  // (key g, key g+8) of heads 2t and 2t+1
    split_pair_f16(p00, p10, x0h, x0l);
    split_pair_f16(p01, p11, x1h, x1l);
    const int la = 8 * t + (g >> 1), lb = la + 4;
    const bool odd = g & 1;
    uint32_t ah = __shfl_sync(FULL, x0h, la), ah1 = __shfl_sync(FULL, x1h, la);
    uint32_t bh = __shfl_sync(FULL, x0h, lb), bh1 = __shfl_sync(FULL, x1h, lb);
    uint32_t al = __shfl_sync(FULL, x0l, la), al1 = __shfl_sync(FULL, x1l, la);
    uint32_t bl = __shfl_sync(FULL, x0l, lb), bl1 = __shfl_sync(FULL, x1l, lb);
    if (odd) ah = ah1, bh = bh1, al = al1, bl = bl1;
    const uint32_t ph0 = __byte_perm(ah, bh, 0x5410), ph1 = __byte_perm(ah, bh, 0x7632);
    const uint32_t pl0 = __byte_perm(al, bl, 0x5410), pl1 = __byte_perm(al, bl, 0x7632);
    // ---- O^T += V^T P^T over this lane's dims 16g .. 16g + 15: chunk g of
    // rows 2t, 2t+1, 2t+8, 2t+9; word i holds dims 16g + 4i .. + 3 (MMAs
    // 2i, 2i+1).  Rows past the context are zero.
    const int key0 = 2 * t, key2 = 2 * t + 8;
    uint4 ra = lds128(vst + swz(key0, g)), rb = lds128(vst + swz(key0 + 1, g));
    uint4 rc = lds128(vst + swz(key2, g)), rd = lds128(vst + swz(key2 + 1, g));
    if (key0 >= valid) ra = make_uint4(0u, 0u, 0u, 0u);
    if (key0 + 1 >= valid) rb = make_uint4(0u, 0u, 0u, 0u);
    if (key2 >= valid) rc = make_uint4(0u, 0u, 0u, 0u);
    if (key2 + 1 >= valid) rd = make_uint4(0u, 0u, 0u, 0u);
    const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
    const uint32_t wc[4] = {rc.x, rc.y, rc.z, rc.w}, wd[4] = {rd.x, rd.y, rd.z, rd.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t ab0 = __byte_perm(wa[i], wb[i], 0x5140), ab1 = __byte_perm(wa[i], wb[i], 0x7362);
        const uint32_t cd0 = __byte_perm(wc[i], wd[i], 0x5140), cd1 = __byte_perm(wc[i], wd[i], 0x7362);
        const uint32_t a0 = e4m3x2_f16x2(ab0), a1 = e4m3x2_f16x2(ab0 >> 16);
        const uint32_t a2 = e4m3x2_f16x2(cd0), a3 = e4m3x2_f16x2(cd0 >> 16);
        mma_f16(o[2 * i], a0, a1, a2, a3, ph0, ph1);
        mma_f16(o[2 * i], a0, a1, a2, a3, pl0, pl1);
        const uint32_t b0 = e4m3x2_f16x2(ab1), b1 = e4m3x2_f16x2(ab1 >> 16);
        const uint32_t b2 = e4m3x2_f16x2(cd1), b3 = e4m3x2_f16x2(cd1 >> 16);
        mma_f16(o[2 * i + 1], b0, b1, b2, b3, ph0, ph1);
        mma_f16(o[2 * i + 1], b0, b1, b2, b3, pl0, pl1);
    }
}

// Consumer warps with MMA block math (e4m3 pools, d = 128): the item loop
// of run_consumer, with q, the softmax state and O in the MMA layouts.
template <int D, int G, int EB, bool FUSED>
__device__ void run_consumer_mma(const DecodeParams& P, uint8_t* smem, const Bars& B, volatile int* abort_flag,
                                 int warp, int lane) {
    using C = Cfg<D, G, EB>;
    constexpr int QW = D / 8;  // q words (two elements each) of a lane: its D/4 dims
    const unsigned FULL = 0xffffffffu;
    const ItemDesc* descs = reinterpret_cast<const ItemDesc*>(smem + C::OFF_DESC);
    const volatile int* stage_new = reinterpret_cast<const volatile int*>(smem + C::OFF_NEW);
    float* mo = reinterpret_cast<float*>(smem + C::OFF_MO);
    float2* ml = reinterpret_cast<float2*>(smem + C::OFF_ML);
    const int g = lane >> 2, t = lane & 3;
    uint32_t taken = 0, item_seq = 0;
    bool ok = true;
    while (ok) {
        const uint32_t slot = item_seq % kItemRing;
        if (*abort_flag || !mbar_wait_warp(&B.ifull[slot], (item_seq / kItemRing) & 1)) {
            ok = false;
            break;
        }
        const ItemDesc d = descs[slot];
        if (d.s < 0) break;
        // q of head g, dims 32t .. 32t + 31, as B fragments (zero for
        // g >= G), scaled by 2^-e into [1, 2) for f16 (exact); the scores
        // of heads 2t and 2t + 1 get the factor 2^e back.
        uint32_t qb[QW];
        float f0, f1;
        {
            const uint8_t* qs = smem + C::OFF_ITEMQ + slot * C::QBYTES + (g * D + t * (D / 4)) * 2;
#pragma unroll
            for (int c = 0; c < QW / 4; ++c) {
                uint4 u = make_uint4(0u, 0u, 0u, 0u);
                if (g < G) u = lds128(qs + 16 * c);
                qb[4 * c] = u.x, qb[4 * c + 1] = u.y, qb[4 * c + 2] = u.z, qb[4 * c + 3] = u.w;
            }
            float mx = 0.f;
#pragma unroll
            for (int i = 0; i < QW; ++i) mx = fmaxf(mx, fmaxf(fabsf(bf16lo(qb[i])), fabsf(bf16hi(qb[i]))));
            mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 2));
            int e = (mx >= 0x1p-100f && mx < INFINITY) ? static_cast<int>((__float_as_uint(mx) >> 23) & 0xFF) - 127
                                                         : 0;
            e = min(e, 100);  // |q| up to 2^101 (f16 would overflow beyond)
            const float down = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
            const float up = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);    // 2^e
#pragma unroll
            for (int i = 0; i < QW; ++i) qb[i] = f16x2_rn(bf16lo(qb[i]) * down, bf16hi(qb[i]) * down);
            f0 = P.scale_log2 * __shfl_sync(FULL, up, (8 * t) & 31);
            f1 = P.scale_log2 * __shfl_sync(FULL, up, (8 * t + 4) & 31);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.iempty[slot]);
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        float o[D / 16][4];
#pragma unroll
        for (int mm = 0; mm < D / 16; ++mm) o[mm][0] = o[mm][1] = o[mm][2] = o[mm][3] = 0.f;
        const int nb = d.b1 - d.b0;
        const int first = (warp - d.rot + C::W) % C::W;  // see run_consumer
        const bool may_have_new = FUSED && d.b1 == (d.n + kBlockSize - 1) / kBlockSize;
        for (int b = first; b < nb; b += C::W) {
            const uint32_t st = static_cast<uint32_t>(warp * C::SW) + taken % C::SW;
            if (*abort_flag || !mbar_wait_warp(&B.full[st], (taken / C::SW) & 1)) {
                ok = false;
                break;
            }
            const int blk = d.b0 + b;
            const int valid = min(kBlockSize, d.n - blk * kBlockSize);
            uint8_t* kst = smem + st * C::STAGE_BYTES;
            if (may_have_new && b == nb - 1) store_stage_new_row<D, G, EB>(P, d, kst, stage_new[st], lane);
            compute_block_mma<D, G>(kst, kst + C::SLAB, valid, qb, f0, f1, m0, m1, l0, l1, o, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.empty[st]);
            ++taken;
        }
        if (!ok) break;
        // Publish this warp's state for the merger: (m, l) and O of heads
        // 2t and 2t+1 (those below G), each lane its dims 16g .. 16g + 15.
        const int buf = item_seq % C::MERGE_BUFS;
        if (!mbar_wait_warp(&B.mempty[buf], ((item_seq / C::MERGE_BUFS) & 1) ^ 1)) {
            ok = false;
            break;
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(FULL, l0, off);
            l1 += __shfl_xor_sync(FULL, l1, off);
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = 2 * t + e;
            if (h < G) {
                const size_t base = static_cast<size_t>((buf * C::W + warp) * G + h);
                if (g == 0) ml[base] = make_float2(e ? m1 : m0, e ? l1 : l0);
                float2* dst = reinterpret_cast<float2*>(mo + base * D + g * (D / 8));
#pragma unroll
                for (int mm = 0; mm < D / 16; ++mm) dst[mm] = make_float2(o[mm][e], o[mm][2 + e]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.mfull[buf]);
        ++item_seq;
    }
    if (!ok) {
        *abort_flag = 1;
        record_error(P.err, kErrTimeout, 2u);
    }
}

template <int D, int G, int EB, bool FUSED>
__device__ void run_consumer(const DecodeParams& P, uint8_t* smem, const Bars& B, volatile int* abort_flag,
                             int warp, int lane) {
    using C = Cfg<D, G, EB>;
    const ItemDesc* descs = reinterpret_cast<const ItemDesc*>(smem + C::OFF_DESC);
    const volatile int* stage_new = reinterpret_cast<const volatile int*>(smem + C::OFF_NEW);
    float2* psm = reinterpret_cast<float2*>(smem + C::OFF_P) + warp * G * kBlockSize;
    float* mo = reinterpret_cast<float*>(smem + C::OFF_MO);
    float2* ml = reinterpret_cast<float2*>(smem + C::OFF_ML);
    const int sub = lane / C::LPR;
    const int cl = lane % C::LPR;
    uint32_t taken = 0, item_seq = 0;  // taken: blocks this warp consumed so far
    bool ok = true;
    while (ok) {
        const uint32_t slot = item_seq % kItemRing;
        if (*abort_flag || !mbar_wait_warp(&B.ifull[slot], (item_seq / kItemRing) & 1)) {
            ok = false;
            break;
        }
        const ItemDesc d = descs[slot];
        if (d.s < 0) break;
        float2 q2[G][4];
        const float2 sc2 = make_float2(P.scale_log2, P.scale_log2);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const uint4 u = lds128(smem + C::OFF_ITEMQ + slot * C::QBYTES + (g * D + cl * 8) * 2);
            q2[g][0] = __fmul2_rn(bf16x2_to_float2(u.x), sc2);
            q2[g][1] = __fmul2_rn(bf16x2_to_float2(u.y), sc2);
            q2[g][2] = __fmul2_rn(bf16x2_to_float2(u.z), sc2);
            q2[g][3] = __fmul2_rn(bf16x2_to_float2(u.w), sc2);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.iempty[slot]);
        float m[G], lsum[G];
        float2 o2[G][4];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m[g] = -INFINITY;
            lsum[g] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) o2[g][j] = make_float2(0.f, 0.f);
        }
        const int nb = d.b1 - d.b0;
        // Block b of the item goes to warp (b + rot) % 8: the rotation comes
        // from the item's global index, so the extra blocks of items whose
        // length is not a multiple of 8 spread over the warps while every
        // item is summed in an order that does not depend on which CTA took
        // it (results are bitwise reproducible).
        const int first = (warp - d.rot + C::W) % C::W;
        // Fused step: the pair's last block may carry the new token's row
        // (the producer checked its slot and noted it for the stage).
        const bool may_have_new = FUSED && d.b1 == (d.n + kBlockSize - 1) / kBlockSize;
        for (int b = first; b < nb; b += C::W) {
            const uint32_t st = static_cast<uint32_t>(warp * C::SW) + taken % C::SW;
            if (*abort_flag || !mbar_wait_warp(&B.full[st], (taken / C::SW) & 1)) {
                ok = false;
                break;
            }
            const int blk = d.b0 + b;
            const int valid = min(kBlockSize, d.n - blk * kBlockSize);
            uint8_t* kst = smem + st * C::STAGE_BYTES;
            if (may_have_new && b == nb - 1) store_stage_new_row<D, G, EB>(P, d, kst, stage_new[st], lane);
            compute_block<D, G, EB>(kst, kst + C::SLAB, valid, q2, m, lsum, o2, psm, lane);
            if (lane == 0) mbar_arrive(&B.empty[st]);
            ++taken;
        }
        if (!ok) break;
        // Publish this warp's state for the merger.
        const int buf = item_seq % C::MERGE_BUFS;
        if (!mbar_wait_warp(&B.mempty[buf], ((item_seq / C::MERGE_BUFS) & 1) ^ 1)) {
            ok = false;
            break;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float lt = warp_sum(lsum[g]);
            // Lanes with the same dims but different rows hold partial o.
#pragma unroll
            for (int off = C::LPR; off < 32; off <<= 1) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    o2[g][j].x += __shfl_xor_sync(0xffffffffu, o2[g][j].x, off);
                    o2[g][j].y += __shfl_xor_sync(0xffffffffu, o2[g][j].y, off);
                }
            }
            if (lane == 0) ml[(buf * C::W + warp) * G + g] = make_float2(m[g], lt);
            if (sub == 0) {
                float4* dst = reinterpret_cast<float4*>(mo + ((buf * C::W + warp) * G + g) * D + cl * 8);
                dst[0] = make_float4(o2[g][0].x, o2[g][0].y, o2[g][1].x, o2[g][1].y);
                dst[1] = make_float4(o2[g][2].x, o2[g][2].y, o2[g][3].x, o2[g][3].y);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.mfull[buf]);
        ++item_seq;
    }
    if (!ok) {
        *abort_flag = 1;
        record_error(P.err, kErrTimeout, 2u);
    }
}

template <int D, int G, int EB>
__device__ void run_merger(const DecodeParams& P, uint8_t* smem, const Bars& B, volatile int* abort_flag, int lane) {
    using C = Cfg<D, G, EB>;
    const ItemDesc* descs = reinterpret_cast<const ItemDesc*>(smem + C::OFF_DESC);
    const float* mo = reinterpret_cast<const float*>(smem + C::OFF_MO);
    const float2* ml = reinterpret_cast<const float2*>(smem + C::OFF_ML);
    float* wsm = reinterpret_cast<float*>(smem + C::OFF_WT);
    float2* msm = reinterpret_cast<float2*>(smem + C::OFF_MSM);
    uint32_t item_seq = 0;
    bool ok = true;
    while (true) {
        const uint32_t slot = item_seq % kItemRing;
        if (*abort_flag || !mbar_wait_warp(&B.ifull[slot], (item_seq / kItemRing) & 1)) {
            ok = false;
            break;
        }
        const ItemDesc d = descs[slot];
        if (d.s < 0) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.iempty[slot]);
        const unsigned FULL = 0xffffffffu;
        constexpr int W = C::W;
        constexpr int CH = G * D / 4;
        constexpr int WL = C::MERGE_LANES;
        constexpr int NJ = (CH + 31) / 32;
        const int h0 = d.g * G;
        // Shared prefix: the item holding the pair's first block (the only
        // part, or the first of a split pair) merges the prefix state of
        // the pair's G heads into its own.  It is read now, while the
        // consumers still work on the item: (m, l) of head `lane` and this
        // lane's float4 chunks of the o rows.
        const bool fold = P.pre_ml != nullptr && (d.nparts == 1 || d.slot == 1);
        float2 pml = make_float2(-INFINITY, 0.f);
        float4 po[NJ];
        if (fold) {
            const size_t hrow = static_cast<size_t>(d.s) * P.hq + h0;
            if (lane < G) pml = __ldcg(P.pre_ml + hrow + lane);
            const float4* src = reinterpret_cast<const float4*>(P.pre_o + hrow * D);
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int k = lane + 32 * j;
                po[j] = (k < CH) ? __ldcg(src + k) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        const int buf = item_seq % C::MERGE_BUFS;
        if (!mbar_wait_warp(&B.mfull[buf], (item_seq / C::MERGE_BUFS) & 1)) {
            ok = false;
            break;
        }
        // Combine the consumer warps' states (log-sum-exp).  First the
        // weights of all (q head g, warp w) pairs at once: lane g * W + w,
        // W lanes per head; then each lane combines whole float4 chunks of
        // the item's G output rows (contiguous in out and in part_o), with
        // the W chunk loads issued together.  With a prefix state (m_p,
        // l_p, o_p) the reference becomes max(M, m_p): the warps' weights
        // take the factor 2^(M - max) and o_p the weight 2^(m_p - max).
#pragma unroll
        for (int i0 = 0; i0 < G * WL; i0 += 32) {
            const int i = i0 + lane;
            const int w = i % WL, gi = i / WL;
            const bool live = gi < G && w < W;
            const float2 e = live ? ml[(buf * W + w) * G + gi] : make_float2(-INFINITY, 0.f);
            float M = e.x;
#pragma unroll
            for (int o = 1; o < WL; o <<= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
            float wt = (e.x == -INFINITY) ? 0.f : fast_exp2(e.x - M);
            float L = e.y * wt;
#pragma unroll
            for (int o = 1; o < WL; o <<= 1) L += __shfl_xor_sync(FULL, L, o);
            float wp = 0.f;  // weight of the prefix state
            if (fold) {
                const float2 pe = make_float2(__shfl_sync(FULL, pml.x, gi & 31), __shfl_sync(FULL, pml.y, gi & 31));
                const float Mx = fmaxf(M, pe.x);
                const float fl = (M == -INFINITY) ? 0.f : fast_exp2(M - Mx);
                wp = (pe.x == -INFINITY) ? 0.f : fast_exp2(pe.x - Mx);
                wt *= fl;
                L = L * fl + pe.y * wp;
                M = Mx;
            }
            if (live) {
                wsm[gi * W + w] = wt;
                if (w == 0) msm[gi] = make_float2(M, L);
                if (w == 0 && fold) wsm[G * W + gi] = wp;
            }
        }
        __syncwarp();
        const size_t pi0 = (static_cast<size_t>(d.r) * 2 + d.slot) * G;  // this part's partial slots, one per head
        const float4* mo4 = reinterpret_cast<const float4*>(mo) + static_cast<size_t>(buf) * W * CH;
        float4* dst = (d.nparts == 1)
                          ? reinterpret_cast<float4*>(P.out + (static_cast<size_t>(d.row) * P.hq + h0) * D)
                          : reinterpret_cast<float4*>(P.part_o + pi0 * D);
#pragma unroll
        for (int j = 0; j < (CH + 31) / 32; ++j) {
            const int k = lane + 32 * j;
            if (k < CH) {
                const int g = k / (D / 4);
                float4 v[W];
#pragma unroll
                for (int w = 0; w < W; ++w) v[w] = mo4[w * CH + k];
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                if (fold) {
                    const float wp = wsm[G * W + g];
                    a = make_float4(po[j].x * wp, po[j].y * wp, po[j].z * wp, po[j].w * wp);
                }
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    const float wt = wsm[g * W + w];
                    a.x = fmaf(v[w].x, wt, a.x);
                    a.y = fmaf(v[w].y, wt, a.y);
                    a.z = fmaf(v[w].z, wt, a.z);
                    a.w = fmaf(v[w].w, wt, a.w);
                }
                if (d.nparts == 1) {
                    const float L = msm[g].y;
                    a = (L > 0.f) ? normalise<EB>(a, L, P.v_scale) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                dst[k] = a;
            }
        }
        if (d.nparts > 1 && lane < G) P.part_ml[pi0 + lane] = msm[lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.mempty[buf]);
        if (d.nparts > 1) {
            __threadfence();
            __syncwarp();
            uint32_t ticket = 0;
            uint32_t* ctr = P.counters + static_cast<size_t>(d.s) * P.hkv + d.g;
            if (lane == 0) ticket = atomicAdd(ctr, 1u);
            ticket = __shfl_sync(FULL, ticket, 0);
            if (ticket == static_cast<uint32_t>(d.nparts - 1)) {
                // Last part in: merge all parts of (s, kv head), in part
                // order.  Part k of the pair lives in range r0 + k, in slot
                // slot0 for k = 0 and slot 0 after that; its G heads' (m, l)
                // and o rows are contiguous.  Lanes hold the parts' weights
                // for every head, 32 parts at a time.
                __threadfence();
                auto part_base = [&](int k) -> size_t {
                    return (static_cast<size_t>(d.r0 + k) * 2 + (k == 0 ? d.slot0 : 0)) * G;
                };
                auto pick = [](const float (&x)[G], int g) {
                    float r = x[0];
#pragma unroll
                    for (int i = 1; i < G; ++i) r = (g == i) ? x[i] : r;
                    return r;
                };
                float M[G], L[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    M[g] = -INFINITY;
                    L[g] = 0.f;
                }
                for (int p0 = 0; p0 < d.nparts; p0 += 32) {
                    if (p0 + lane < d.nparts) {
                        const float2* pm = P.part_ml + part_base(p0 + lane);
#pragma unroll
                        for (int g = 0; g < G; ++g) M[g] = fmaxf(M[g], __ldcg(pm + g).x);
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) M[g] = warp_max(M[g]);
                float4 acc[NJ];
#pragma unroll
                for (int j = 0; j < NJ; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int p0 = 0; p0 < d.nparts; p0 += 32) {
                    const int pp = p0 + lane;
                    float wt[G];
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float2 e = (pp < d.nparts) ? __ldcg(P.part_ml + part_base(pp) + g)
                                                         : make_float2(-INFINITY, 0.f);
                        wt[g] = (e.x == -INFINITY) ? 0.f : fast_exp2(e.x - M[g]);
                        L[g] = fmaf(e.y, wt[g], L[g]);
                    }
                    const int cnt = min(32, d.nparts - p0);
#pragma unroll 2
                    for (int k = 0; k < cnt; ++k) {
                        float wk[G];
#pragma unroll
                        for (int g = 0; g < G; ++g) wk[g] = __shfl_sync(FULL, wt[g], k);
                        const float4* orow = reinterpret_cast<const float4*>(P.part_o + part_base(p0 + k) * D);
#pragma unroll
                        for (int j = 0; j < NJ; ++j) {
                            const int c = lane + 32 * j;
                            if (c < CH) {
                                const float4 o = __ldcg(orow + c);
                                const float w = pick(wk, c / (D / 4));
                                acc[j].x = fmaf(o.x, w, acc[j].x);
                                acc[j].y = fmaf(o.y, w, acc[j].y);
                                acc[j].z = fmaf(o.z, w, acc[j].z);
                                acc[j].w = fmaf(o.w, w, acc[j].w);
                            }
                        }
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) L[g] = warp_sum(L[g]);
                float4* out4 = reinterpret_cast<float4*>(P.out + (static_cast<size_t>(d.row) * P.hq + h0) * D);
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int c = lane + 32 * j;
                    if (c < CH) {
                        const float Lg = pick(L, c / (D / 4));
                        out4[c] = (Lg > 0.f) ? normalise<EB>(acc[j], Lg, P.v_scale) : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                if (lane == 0) atomicExch(ctr, 0u);
            }
        }
        ++item_seq;
    }
    if (!ok) {
        *abort_flag = 1;
        record_error(P.err, kErrTimeout, 3u);
    }
}

// Warm L2 with what every CTA reads first: context_lens (and
// query_start_loc), the used part of every block-table row and, for a pure
// decode batch, the query rows.  Runs before griddep_wait(), so the chain
// context_lens -> table -> K/V that opens each CTA starts from L2 rather than
// from DRAM.  Thread t of CTA c takes lines c * nthr + t + k * gridDim.x * nthr.
// A region past kPrefetchCap bytes is left to the regular loads.
template <int D, bool FUSED>
__device__ void prefetch_inputs(const DecodeParams& P, int t, int nthr) {
    constexpr long long kPrefetchCap = 16ll << 20;
    const long long S = P.num_seqs;
    const long long nb = min(static_cast<long long>(P.max_blocks),
                             static_cast<long long>(P.ctx_cap + kBlockSize - 1) / kBlockSize);
    const long long n_ctx = range_lines(S * 4);
    const long long n_qsl = P.qsl ? range_lines((S + 1) * 4) : 0;
    const long long lpr = range_lines(nb * 4);
    const long long n_tab = (S * nb * 4 <= kPrefetchCap) ? S * lpr : 0;
    const long long q_bytes = S * P.hq * D * 2;
    const long long n_q = (P.qsl == nullptr && q_bytes <= kPrefetchCap) ? range_lines(q_bytes) : 0;
    // Fused step: the new rows and their slots.
    const long long kn_bytes = S * P.hkv * D * 2;
    const long long n_kn = (FUSED && kn_bytes <= kPrefetchCap) ? range_lines(kn_bytes) : 0;
    const long long n_sl = FUSED ? range_lines(S * 4) : 0;
    const long long base_new = n_ctx + n_qsl + n_tab + n_q;
    const long long total = base_new + 2 * n_kn + n_sl;
    const long long step = static_cast<long long>(gridDim.x) * nthr;
    for (long long k = static_cast<long long>(blockIdx.x) * nthr + t; k < total; k += step) {
        const void* a;
        if (k < n_ctx) {
            a = range_line(P.context_lens, S * 4, k);
        } else if (k < n_ctx + n_qsl) {
            a = range_line(P.qsl, (S + 1) * 4, k - n_ctx);
        } else if (k < n_ctx + n_qsl + n_tab) {
            const long long j = k - n_ctx - n_qsl;
            a = range_line(P.block_tables + (j / lpr) * P.max_blocks, nb * 4, j % lpr);
        } else if (k < base_new) {
            a = range_line(P.q, q_bytes, k - n_ctx - n_qsl - n_tab);
        } else if (k < base_new + n_kn) {
            a = range_line(P.k_new, kn_bytes, k - base_new);
        } else if (k < base_new + 2 * n_kn) {
            a = range_line(P.v_new, kn_bytes, k - base_new - n_kn);
        } else {
            a = range_line(P.slot_mapping, S * 4, k - base_new - 2 * n_kn);
        }
        if (a != nullptr) prefetch_l2(a);
    }
}

// Guess this CTA's first blocks and prefetch their K and V slabs into L2,
// before the previous kernel on the stream has finished.  The reads here
// may see values that kernel is still writing (they bypass L1, so no stale
// copy outlives the wait); they only choose what to prefetch, and every
// address is checked against the pool first.  The guess is the nominal
// range start (no boundary snapping); the producer recomputes everything
// after the wait.  Up to kSpecWindows * 32 sequences; larger batches skip
// the guess.
constexpr int kSpecWindows = 8;

template <int D, int G, int EB>
__device__ void prefetch_first_blocks(const DecodeParams& P, int lane, int max_units) {
    using C = Cfg<D, G, EB>;
    const unsigned FULL = 0xffffffffu;
    if (P.num_seqs > kSpecWindows * 32) return;
    int u[kSpecWindows], incl[kSpecWindows];
#pragma unroll
    for (int w = 0; w < kSpecWindows; ++w) {
        const int s = w * 32 + lane;
        u[w] = 0;
        if (s < P.num_seqs) {
            const bool dec = P.qsl == nullptr || ld_l2_only(P.qsl + s + 1) - ld_l2_only(P.qsl + s) == 1;
            const int n = min(max(ld_l2_only(P.context_lens + s), 0), P.ctx_cap);
            u[w] = dec ? max(1, (n + kBlockSize - 1) / kBlockSize - P.skip_blocks) : 0;
        }
    }
    long long per_head = 0;
#pragma unroll
    for (int w = 0; w < kSpecWindows; ++w) {
        incl[w] = u[w];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(FULL, incl[w], o);
            if (lane >= o) incl[w] += t;
        }
        per_head += __shfl_sync(FULL, incl[w], 31);
    }
    int umin = INT32_MAX, umax = 0;
#pragma unroll
    for (int w = 0; w < kSpecWindows; ++w) {
        umin = min(umin, u[w] > 0 ? u[w] : INT32_MAX);
        umax = max(umax, u[w]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        umin = min(umin, __shfl_xor_sync(FULL, umin, o));
        umax = max(umax, __shfl_xor_sync(FULL, umax, o));
    }
    const long long T = per_head * P.hkv;
    long long RU = P.range_units;
    if (RU <= 0) RU = auto_range_units(T, gridDim.x, umin, umax);
    long long x = static_cast<long long>(blockIdx.x) * RU;
    const long long hi = min(T, x + min(RU, static_cast<long long>(max_units)));
    // Walk the pairs from x: find the sequence (window w, lane j) holding x.
    long long base = 0;  // units per kv head before window w
#pragma unroll
    for (int w = 0; w < kSpecWindows; ++w) {
        while (x < hi) {
            const unsigned hit = __ballot_sync(FULL, (base + incl[w]) * P.hkv > x);
            if (!hit) break;
            const int j = __ffs(hit) - 1;
            const int us = __shfl_sync(FULL, u[w], j);
            const long long seq0 = (base + __shfl_sync(FULL, incl[w], j) - us) * P.hkv;
            const int g = static_cast<int>((x - seq0) / us);
            const int b0 = static_cast<int>(x - seq0 - static_cast<long long>(g) * us);
            const int cnt = static_cast<int>(min(static_cast<long long>(us - b0), hi - x));
            const int32_t* trow = P.block_tables + static_cast<size_t>(w * 32 + j) * P.max_blocks + P.skip_blocks;
            for (int b = lane; b < cnt && P.skip_blocks + b0 + b < P.max_blocks; b += 32) {
                const int phys = ld_l2_only(trow + b0 + b);
                if (phys >= 0 && phys < P.num_blocks) {
                    const size_t slab = (static_cast<size_t>(phys) * P.hkv + g) * C::SLAB;
                    bulk_prefetch_l2(P.k_pool + slab, C::SLAB);
                    bulk_prefetch_l2(P.v_pool + slab, C::SLAB);
                }
            }
            x += cnt;
        }
        base += __shfl_sync(FULL, incl[w], 31);
    }
}

template <int D, int G, int EB, bool FUSED>
__global__ void __launch_bounds__(Cfg<D, G, EB>::THREADS, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DecodeParams P) {
    using C = Cfg<D, G, EB>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // MMA configurations: the ring starts on a 1024-byte boundary (the
    // swizzle pattern of a tile follows its shared-memory address).
    uint8_t* smem = smem_raw + (C::MMA ? ((1024 - (smem_addr(smem_raw) & 1023)) & 1023) : 0);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    Bars B;
    B.full = bars;
    B.empty = bars + C::STAGES;
    B.ifull = bars + 2 * C::STAGES;
    B.iempty = B.ifull + kItemRing;
    B.mfull = B.iempty + kItemRing;
    B.mempty = B.mfull + C::MERGE_BUFS;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&B.full[i], 1);
            mbar_init(&B.empty[i], 1);
        }
        for (int i = 0; i < kItemRing; ++i) {
            mbar_init(&B.ifull[i], 1);
            mbar_init(&B.iempty[i], C::W + 1);
        }
        for (int i = 0; i < C::MERGE_BUFS; ++i) {
            mbar_init(&B.mfull[i], C::W);
            mbar_init(&B.mempty[i], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    griddep_launch_dependents();
    __syncthreads();
    // Until griddep_wait() returns, only L2 prefetches touch global memory.
    // Consumer warps read shared memory only and need no wait.
    if (warp == C::PRODUCER_WARP) {
        griddep_wait();
        // Test hook: no descriptor is ever published, so the other warps
        // leave through their bounded waits; nothing is in flight.
        if (!P.stall) run_producer<D, G, EB, FUSED>(P, &tm_k, &tm_v, smem, B, abort_flag, lane);
    } else if (warp == C::MERGER_WARP) {
        prefetch_first_blocks<D, G, EB>(P, lane, C::STAGES);
        griddep_wait();
        run_merger<D, G, EB>(P, smem, B, abort_flag, lane);
    } else {
        prefetch_inputs<D, FUSED>(P, threadIdx.x, C::W * 32);
        if constexpr (C::MMA) {
            run_consumer_mma<D, G, EB, FUSED>(P, smem, B, abort_flag, warp, lane);
        } else {
            run_consumer<D, G, EB, FUSED>(P, smem, B, abort_flag, warp, lane);
        }
    }
}

template <int D, int G, int EB, bool FUSED>
cudaError_t launch_one(const DecodeParams& P, int grid, cudaStream_t stream) {
    using C = Cfg<D, G, EB>;
    // MMA configurations read the pools through tiled tensor maps (rows of
    // D * EB = 128 bytes, 16-row boxes, 128-byte swizzle); the others get
    // unused zero maps.
    CUtensorMap tk, tv;
    std::memset(&tk, 0, sizeof(tk));
    std::memset(&tv, 0, sizeof(tv));
    if constexpr (C::MMA) {
        const cuuint64_t rows = static_cast<cuuint64_t>(P.num_blocks) * P.hkv * kBlockSize;
        if (rows > static_cast<cuuint64_t>(INT32_MAX)) return cudaErrorInvalidValue;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), rows > 0 ? rows : 1};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * EB};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / EB), kBlockSize};
        const CUtensorMapDataType dt = EB == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        if (!make_tile_map(&tk, dt, P.k_pool, 2, dims, strides, box)) return cudaErrorInvalidValue;
        if (!make_tile_map(&tv, dt, P.v_pool, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G, EB, FUSED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    return launch_overlapped(decode_kernel<D, G, EB, FUSED>, dim3(grid), dim3(C::THREADS), C::SMEM, stream, tk, tv,
                             P);
}

template <int D, int EB, bool FUSED>
cudaError_t dispatch_g(const DecodeParams& P, int G, int grid, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_one<D, 1, EB, FUSED>(P, grid, stream);
        case 2: return launch_one<D, 2, EB, FUSED>(P, grid, stream);
        case 4: return launch_one<D, 4, EB, FUSED>(P, grid, stream);
        case 8: return launch_one<D, 8, EB, FUSED>(P, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

// One decode launch (FUSED: with each sequence's new row) from the checked
// arguments; a.stall set arms the test hook for this launch.
template <bool FUSED>
cudaError_t launch_decode_t(const DecodeArgs& a, bool stall, cudaStream_t stream) {
    const DecodeWsLayout L =
        decode_ws_layout(a.num_seqs, a.num_q_heads, a.num_kv_heads, a.head_dim, a.plan.max_ranges,
                         a.prefix_chunks > 0);
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    DecodeParams P;
    P.k_pool = static_cast<uint8_t*>(a.k_pool);
    P.v_pool = static_cast<uint8_t*>(a.v_pool);
    P.q = static_cast<const uint8_t*>(a.q);
    P.block_tables = a.block_tables;
    P.context_lens = a.context_lens;
    P.qsl = a.query_start_loc;
    P.out = a.out;
    P.part_ml = reinterpret_cast<float2*>(ws + L.part_ml);
    P.part_o = reinterpret_cast<float*>(ws + L.part_o);
    P.counters = reinterpret_cast<uint32_t*>(ws + L.counters);
    P.err = a.err;
    P.num_blocks = a.num_blocks;
    P.hkv = a.num_kv_heads;
    P.hq = a.num_q_heads;
    P.num_seqs = a.num_seqs;
    P.max_blocks = a.max_blocks_per_seq;
    P.ctx_cap = static_cast<int32_t>(
        std::min<int64_t>(a.max_context_len, static_cast<int64_t>(a.max_blocks_per_seq) * kBlockSize));
    P.range_units = a.plan.range_units;
    P.max_ranges = a.plan.max_ranges;
    P.scale_log2 = a.scale * kLog2e;
    P.v_scale = 1.f;
    P.stall = stall ? 1 : 0;
    P.k_new = static_cast<const uint8_t*>(a.k_new);
    P.v_new = static_cast<const uint8_t*>(a.v_new);
    P.slot_mapping = a.slot_mapping;
    P.k_inv = a.kv_e4m3 ? 1.f / a.k_scale : 1.f;
    P.v_inv = a.kv_e4m3 ? 1.f / a.v_scale : 1.f;
    P.skip_blocks = a.skip_blocks;
    P.pre_ml = a.prefix_chunks > 0 ? reinterpret_cast<const float2*>(ws + L.pre_ml) : nullptr;
    P.pre_o = a.prefix_chunks > 0 ? reinterpret_cast<const float*>(ws + L.pre_o) : nullptr;
    const int G = a.num_q_heads / a.num_kv_heads;
    if (a.kv_e4m3) {
        // q' = q * scale*log2(e) * k_scale against the K codes.
        P.scale_log2 = a.scale * kLog2e * a.k_scale;
        P.v_scale = a.v_scale;
        if (a.head_dim == 128) return dispatch_g<128, 1, FUSED>(P, G, a.plan.grid, stream);
        if (a.head_dim == 64) return dispatch_g<64, 1, FUSED>(P, G, a.plan.grid, stream);
        return cudaErrorInvalidValue;
    }
    if (a.head_dim == 128) return dispatch_g<128, 2, FUSED>(P, G, a.plan.grid, stream);
    if (a.head_dim == 64) return dispatch_g<64, 2, FUSED>(P, G, a.plan.grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace pkv
