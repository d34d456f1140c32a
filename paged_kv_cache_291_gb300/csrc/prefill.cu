// prefill.cu -- causal chunked-prefill attention tiles on tcgen05 tensor cores.
//
// What it computes ("Chunked Prefill" section of the inference-engine talk
// write-up; section 3 of the serving-engine KV blog): a long prompt is split
// into slices that share a step with decode tokens.  Query row i of a
// sequence with query_len rows and context_len keys (the chunk's own K/V are
// already in the paged cache) sits at position context_len - query_len + i
// and attends keys 0..pos, read through the sequence's block table
// ("Blocks and block tables", section 2 of the blog).  The prefill part of
// a step is a dense contraction ("Prefill/Decode" section of the talk
// write-up), so these tiles run on the tensor cores:
//
//  * A CTA owns 128 query rows of the two q heads of a GQA group ("units";
//    one unit when Hq/Hkv is odd).  Both units read the same K/V tiles, so a
//    tile is loaded once for two heads.  Warp 16 loads the two Q tiles and
//    the K/V key tiles (128 keys = 8 paged blocks, each block a 16-row TMA
//    box with 128-byte swizzle) into rings of 2 (K) and 3 (V) stages.
//    Warp 17 issues tcgen05.mma.  Warps 0-7 and 8-15 run the softmax of
//    units 0 and 1 (TMEM lane = query row; two warps per lane quarter, 16
//    rows each), so one unit's softmax overlaps the other unit's MMAs.
//  * Per unit, TMEM holds S (128 fp32 columns) and O (128 columns).  S =
//    Q K^T is written there; the softmax reads it, then writes P into the
//    first 64 of the same columns as fp16 pairs, and O += P V takes P
//    straight from TMEM (the A operand of the MMA) with V from shared
//    memory (MN-major operand).
//  * P V runs in fp16: P (in [0, 256]) is rounded to fp16, 2^-11 relative,
//    where a bf16 P (2^-9) can miss a 2e-3 absolute bound when a few keys
//    carry all the weight.  The MMA needs V in the same type, so warps 0-15
//    rewrite each V tile in shared memory from bf16 to fp16 in place, a
//    sixteenth each, between their softmax passes (exact for 2^-14 <= |v| <=
//    65504, absolute error at most 2^-25 below).  l sums P in fp32.
//  * A CTA whose visible V values leave that range (some |v| above 65504,
//    which became inf, or every |v| below 2^-12, mostly fp16 subnormals)
//    recomputes its rows after the tensor-core pass, in fp32 on CUDA cores.
//  * head_dim 64 or 128: a tile is one or two 64-dim swizzled panels.
//  * Online softmax in the log2 domain; the running maximum is only moved
//    (and O rescaled in TMEM) when it grows by more than 2^8; the final
//    O / l uses the same reference, so the result is unchanged.
//  * Keys past the last query position of the tile are masked; V rows past
//    it are zeroed in shared memory during the conversion (a 0 weight
//    times a NaN in an unused slot would otherwise poison the MMA).
//  * Every wait is bounded; TMEM is freed on every exit path.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kTileM = 128;                          // query rows per unit
constexpr int kTileN = 128;                          // keys per key tile
constexpr int kMaxHeadDim = 128;                     // head_dim 64 uses the first panel of each tile
constexpr int kUnits = 2;                            // q heads per CTA (max)
constexpr int kBlocksPerTile = kTileN / kBlockSize;  // 8
constexpr int kPanelBytes = 128 * 128;               // 128 rows x 128 B (64 bf16)
constexpr int kTileBytes = 2 * kPanelBytes;          // [128][128] bf16 as two swizzled panels
constexpr int kBoxBytes = kBlockSize * 128;          // one 16-row box of one panel

constexpr int kVStages = 3;                          // V waits longest (load + fp16 conversion)
constexpr int OFF_Q = 0;                             // kUnits Q tiles
constexpr int OFF_K = OFF_Q + kUnits * kTileBytes;   // 2 stages
constexpr int OFF_V = OFF_K + 2 * kTileBytes;        // kVStages stages
constexpr int OFF_BAR = OFF_V + kVStages * kTileBytes;
constexpr int NBAR = 20;
constexpr int OFF_INFO = OFF_BAR + NBAR * 8;         // tile info (ints)
constexpr int OFF_TMEM = OFF_INFO + 16 * 4;
constexpr int SMEM_USED = OFF_TMEM + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;         // slack to align the base to 1024 B
static_assert(SMEM_BYTES <= 232448, "shared memory budget (227 KB)");
// One CTA per SM: the CTA allocates all 512 TMEM columns, and tcgen05.alloc
// would wait for a second resident CTA to free them.  A footprint above half
// of the SM's 228 KB of shared memory rules a second CTA out.
static_assert(2 * SMEM_BYTES > 228 * 1024, "the 512-column TMEM allocation needs one CTA per SM");

constexpr int kSoftmaxWarps = 8;                     // per unit: two per TMEM lane quarter
constexpr int kLoadWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kThreads = 32 * 18;
constexpr int kConvWarps = kSoftmaxWarps * kUnits;   // warps 0-15 also convert V tiles

constexpr uint32_t kTmemCols = 512;
// Unit u: S/P at columns [256u, 256u + 128), O at [256u + 128, 256u + 256).
__host__ __device__ constexpr uint32_t col_s(int u) { return static_cast<uint32_t>(u) * 256u; }
__host__ __device__ constexpr uint32_t col_o(int u) { return static_cast<uint32_t>(u) * 256u + 128u; }

constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLog2e = 1.4426950408889634f;

struct PrefillParams {
    const uint8_t* q;       // bf16 [num_tokens][hq][D] (for the exact fallback)
    const uint8_t* k_pool;  // bf16 [num_blocks][hkv][16][D] (for the exact fallback)
    const uint8_t* v_pool;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* qsl;
    float* out;
    unsigned long long* err;
    int32_t num_blocks, hkv, hq, num_seqs, max_blocks, ctx_cap, num_tokens, units;
    // The last split_last row tiles of each prefill sequence (its longest:
    // they hold the most keys) run as two one-head CTAs instead of one
    // two-head CTA (units == 2 only), so that more SMs share them.
    int32_t split_last;
    float scale_log2;
};

// Barrier indices.
enum {
    B_QFULL = 0,
    B_KFULL = 1,   // +stage
    B_KEMPTY = 3,  // +stage
    B_VFULL = 5,   // +V stage
    B_VEMPTY = 8,  // +V stage
    B_SFULL = 11,  // +unit
    B_PFULL = 13,  // +unit (4 arrivals)
    B_ODONE = 15,  // +unit
    B_VCONV = 17,  // +V stage (8 arrivals): V tile converted to fp16
};

// Tile info slots (written by warp 0 before the CTA-wide sync).
enum { I_S = 0, I_ROW0, I_ROWS, I_PMIN, I_PMAX, I_NT, I_KLAST, I_BAD, I_CTX, I_VMAX, I_UNITS, I_H0 };

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// bf16 pair -> fp16 pair (round to nearest even: exact for 2^-14 <= |v| <=
// 65504); `vmax` tracks the largest magnitude seen.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x, float& vmax) {
    const float lo = __uint_as_float(x << 16), hi = __uint_as_float(x & 0xFFFF0000u);
    vmax = fmax3(vmax, fabsf(lo), fabsf(hi));
    return tc::pack_f16x2(lo, hi);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) { return mbar_wait_warp(bar, parity); }

// Compensated fp32 sum (Neumaier): s + c carries the sum of the added
// terms to about one rounding of the largest of them, so small terms added
// to a large accumulator are not lost.
__device__ __forceinline__ void sum2(float& s, float& c, float y) {
    const float t = __fadd_rn(s, y);
    c = __fadd_rn(c, fabsf(s) >= fabsf(y) ? __fadd_rn(__fsub_rn(s, t), y) : __fadd_rn(__fsub_rn(y, t), s));
    s = t;
}

// Exact fallback of a CTA's rows on CUDA cores (fp32 scores, online softmax
// in the log2 domain whose reference moves only when the maximum grows by
// more than 2^8, compensated fp32 sums for P.V and the row sum), for V values
// the fp16 tensor-core P.V cannot carry.  Warp w takes the (row, unit) items
// w, w + 10, ...; lane l owns D/32 consecutive dims of q, K, V and the
// output; keys go in order, read through the block table.
template <int D>
__device__ __noinline__ void redo_rows_exact(const PrefillParams& P, int s, int row0, int rows, int pmin, int h0,
                                             int units, int g, int warp, int lane) {
    constexpr int DPL = D / 32;
    const int32_t* trow = P.block_tables + static_cast<size_t>(s) * P.max_blocks;
    auto load = [](const uint8_t* p, float (&x)[DPL]) {
        if constexpr (DPL == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(p);
            x[0] = bf16lo(u.x), x[1] = bf16hi(u.x), x[2] = bf16lo(u.y), x[3] = bf16hi(u.y);
        } else {
            const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
            x[0] = bf16lo(u), x[1] = bf16hi(u);
        }
    };
    for (int item = warp; item < rows * units; item += kThreads / 32) {
        const int m = item / units, h = h0 + item % units, pos = pmin + m;
        float q[DPL], o[DPL], oc[DPL];
        load(P.q + ((static_cast<size_t>(row0 + m) * P.hq + h) * D + lane * DPL) * 2, q);
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            q[i] *= P.scale_log2;
            o[i] = 0.f;
            oc[i] = 0.f;
        }
        float mx = -INFINITY, l = 0.f, lc = 0.f;
        for (int j = 0; j <= pos; ++j) {
            int phys = __ldg(trow + j / kBlockSize);
            if (phys < 0 || phys >= P.num_blocks) phys = 0;  // reported by the tensor-core pass already
            const size_t at = (((static_cast<size_t>(phys) * P.hkv + g) * kBlockSize + j % kBlockSize) * D +
                               lane * DPL) * 2;
            float k[DPL], v[DPL];
            load(P.k_pool + at, k);
            load(P.v_pool + at, v);
            float part = 0.f;
#pragma unroll
            for (int i = 0; i < DPL; ++i) part = fmaf(q[i], k[i], part);
            const float x = warp_sum(part);
            if (x > mx + kRescaleThreshold) {
                const float alpha = fast_exp2(mx - x);
                l *= alpha;
                lc *= alpha;
#pragma unroll
                for (int i = 0; i < DPL; ++i) {
                    o[i] *= alpha;
                    oc[i] *= alpha;
                }
                mx = x;
            }
            const float p = fast_exp2(x - mx);
            sum2(l, lc, p);
#pragma unroll
            for (int i = 0; i < DPL; ++i) sum2(o[i], oc[i], __fmul_rn(p, v[i]));
        }
        const float lt = l + lc;
        float* orow = P.out + (static_cast<size_t>(row0 + m) * P.hq + h) * D + lane * DPL;
#pragma unroll
        for (int i = 0; i < DPL; ++i) orow[i] = (o[i] + oc[i]) / lt;
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams P) {
    static_assert(D == 64 || D == 128, "head_dim");
    constexpr int kPanels = D / 64;  // 64-dim swizzled panels of a tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    int* info = reinterpret_cast<int*>(smem + OFF_INFO);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const unsigned FULL = 0xffffffffu;

    // ---------------------------------------------------------- setup
    // The launch may overlap the previous kernel on the stream: barrier and
    // TMEM set-up go first, every global access after griddep_wait().
    griddep_launch_dependents();
    if (warp == 0) {
        griddep_wait();
        // Find the sequence and row tile of this CTA: entries are numbered
        // over the prefill sequences (query_len > 1) in order, one per row
        // tile of 128 rows (ceil(qlen/128) tiles), and two for each of the
        // last split_last tiles (one per q head).
        const int tile = blockIdx.x;
        const int split = P.units == 2 ? P.split_last : 0;
        int base = 0, found = -1, e = 0, nt_s = 0;
        for (int s0 = 0; s0 < P.num_seqs && found < 0; s0 += 32) {
            const int s = s0 + lane;
            int nt = 0;
            if (s < P.num_seqs) {
                const int ql = __ldg(P.qsl + s + 1) - __ldg(P.qsl + s);
                nt = ql > 1 ? (ql + kTileM - 1) / kTileM : 0;
            }
            const int ne = nt + min(split, nt);
            int incl = ne;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += t;
            }
            const unsigned hit = __ballot_sync(FULL, base + incl > tile);
            if (hit) {
                const int j = __ffs(hit) - 1;
                found = s0 + j;
                e = tile - (base + __shfl_sync(FULL, incl - ne, j));
                nt_s = __shfl_sync(FULL, nt, j);
            } else {
                base += __shfl_sync(FULL, incl, 31);
            }
        }
        // Entry e of the sequence: row tile e while e < nt - sl (both
        // heads), then tile nt - sl + (e - (nt - sl)) / 2, one head each.
        const int sl = min(split, nt_s);
        int tloc = e, cta_units = P.units, cta_h0 = blockIdx.y * P.units;
        if (sl > 0 && e >= nt_s - sl) {
            const int k = e - (nt_s - sl);
            tloc = nt_s - sl + k / 2;
            cta_units = 1;
            cta_h0 += k % 2;
        }
        if (lane == 0) {
            info[I_UNITS] = cta_units;
            info[I_H0] = cta_h0;
            int bad = 0, s = found, row0 = 0, rows = 0, pmin = 0, pmax = 0, nt = 0, klast = 0, ctx = 0;
            if (s < 0) {
                bad = 1;
            } else {
                const int q0 = __ldg(P.qsl + s);
                const int ql = __ldg(P.qsl + s + 1) - q0;
                ctx = __ldg(P.context_lens + s);
                if (ctx > P.ctx_cap || ql > ctx) {
                    record_error(P.err, kErrRange, static_cast<uint32_t>(s));
                    bad = 1;
                }
                row0 = q0 + tloc * kTileM;
                rows = min(kTileM, ql - tloc * kTileM);
                pmin = ctx - ql + tloc * kTileM;
                pmax = pmin + rows - 1;
                nt = pmax / kTileN + 1;
                klast = pmax + 1 - (nt - 1) * kTileN;
                if (bad) nt = 0;
            }
            info[I_S] = s;
            info[I_ROW0] = row0;
            info[I_ROWS] = (s < 0) ? 0 : rows;
            info[I_PMIN] = pmin;
            info[I_PMAX] = pmax;
            info[I_NT] = nt;
            info[I_KLAST] = klast;
            info[I_BAD] = bad;
            info[I_CTX] = ctx;
            info[I_VMAX] = 0;  // largest |v| the converters see (fp32 bits; non-negative floats order as ints)
        }
    }
    if (threadIdx.x == 32 * kMmaWarp) {
        for (int i = 0; i < NBAR; ++i)
            mbar_init(&bar[i], (i == B_PFULL || i == B_PFULL + 1) ? kSoftmaxWarps
                                : (i >= B_VCONV && i < B_VCONV + kVStages) ? kConvWarps : 1u);
        fence_mbar_init();
    }
    if (warp == kLoadWarp) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
        if (lane == 0) {
            tc::prefetch_tensormap(&tm_q);
            tc::prefetch_tensormap(&tm_k);
            tc::prefetch_tensormap(&tm_v);
        }
    }
    griddep_wait();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int units = info[I_UNITS];
    const int h0 = info[I_H0];                   // q head of unit 0 (unit 1 is h0 + 1)
    const int g = h0 / (P.hq / P.hkv);           // the kv head both units read
    const int s = info[I_S];
    const int row0 = info[I_ROW0];
    const int rows = info[I_ROWS];
    const int pmin = info[I_PMIN];
    const int pmax = info[I_PMAX];
    const int nt = info[I_NT];
    const int klast = info[I_KLAST];
    const int bad = info[I_BAD];
    const int nblk = (pmax + 1 + kBlockSize - 1) / kBlockSize;  // blocks holding keys 0..pmax
    bool ok = true;

    if (warp == kLoadWarp && nt > 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            mbar_arrive_expect_tx(&bar[B_QFULL], static_cast<uint32_t>(units) * kPanels * kPanelBytes);
            for (int u = 0; u < units; ++u) {
                uint8_t* dq = smem + OFF_Q + u * kTileBytes;
#pragma unroll
                for (int pn = 0; pn < kPanels; ++pn)
                    tc::tma_load_3d(dq + pn * kPanelBytes, &tm_q, 64 * pn, h0 + u, row0, &bar[B_QFULL]);
            }
        }
        const int32_t* trow = P.block_tables + static_cast<size_t>(s) * P.max_blocks;
        for (int j = 0; j < nt && ok; ++j) {
            const int st = j & 1;
            const uint32_t ph = (j >> 1) & 1;
            const int nvb = min(kBlocksPerTile, nblk - j * kBlocksPerTile);
            int e = 0;
            if (lane < nvb) {
                e = __ldg(trow + j * kBlocksPerTile + lane);
                if (e < 0 || e >= P.num_blocks) {
                    record_error(P.err, kErrRange, static_cast<uint32_t>(s));
                    e = 0;
                }
            }
            int rowsel[kBlocksPerTile];
#pragma unroll
            for (int b = 0; b < kBlocksPerTile; ++b) rowsel[b] = (__shfl_sync(FULL, e, b) * P.hkv + g) * kBlockSize;
            const uint32_t bytes = static_cast<uint32_t>(nvb) * kPanels * kBoxBytes;
            if (!warp_wait(&bar[B_KEMPTY + st], ph ^ 1)) { ok = false; break; }
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar[B_KFULL + st], bytes);
                uint8_t* dst = smem + OFF_K + st * kTileBytes;
#pragma unroll
                for (int b = 0; b < kBlocksPerTile; ++b) {
                    if (b < nvb) {
#pragma unroll
                        for (int pn = 0; pn < kPanels; ++pn)
                            tc::tma_load_2d(dst + pn * kPanelBytes + b * kBoxBytes, &tm_k, 64 * pn, rowsel[b],
                                            &bar[B_KFULL + st]);
                    }
                }
            }
            const int sv = j % kVStages;
            if (!warp_wait(&bar[B_VEMPTY + sv], ((j / kVStages) & 1) ^ 1)) { ok = false; break; }
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar[B_VFULL + sv], bytes);
                uint8_t* dst = smem + OFF_V + sv * kTileBytes;
#pragma unroll
                for (int b = 0; b < kBlocksPerTile; ++b) {
                    if (b < nvb) {
#pragma unroll
                        for (int pn = 0; pn < kPanels; ++pn)
                            tc::tma_load_2d(dst + pn * kPanelBytes + b * kBoxBytes, &tm_v, 64 * pn, rowsel[b],
                                            &bar[B_VFULL + sv]);
                    }
                }
            }
            __syncwarp();
        }
    } else if (warp == kMmaWarp && nt > 0) {
        // ------------------------------------------------------ MMA issuer
        constexpr uint32_t kIdescQK = tc::idesc_bf16_f32(kTileM, kTileN, 0, 0);
        constexpr uint32_t kIdescPV = tc::idesc_f16_f32(kTileM, D, 0, 1);
        // S_u = Q_u K^T for K tile j into the unit's S/P columns.
        auto qk = [&](int u, int j) {
            const uint32_t sq = smem_addr(smem + OFF_Q + u * kTileBytes);
            const uint32_t sk = smem_addr(smem + OFF_K + (j & 1) * kTileBytes);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t off = (k >> 2) * kPanelBytes + (k & 3) * 32;
                tc::mma_bf16_ss(tmem + col_s(u), tc::smem_desc_sw128(sq + off, 16, 1024),
                                tc::smem_desc_sw128(sk + off, 16, 1024), kIdescQK, k > 0 ? 1u : 0u);
            }
            tc::mma_commit(&bar[B_SFULL + u]);
        };
        // O_u += P_u V for V tile j, both in fp16.  Key step k covers keys
        // 16k..16k+15, held as P in columns [8k, 8k+8) of the unit's S/P
        // block.
        auto pv = [&](int u, int j) {
            const uint32_t svb = smem_addr(smem + OFF_V + (j % kVStages) * kTileBytes);
#pragma unroll
            for (int k = 0; k < kTileN / 16; ++k) {
                const uint64_t vdesc = tc::smem_desc_sw128(svb + k * 2048, kPanelBytes, 1024);
                tc::mma_bf16_ts(tmem + col_o(u), tmem + col_s(u) + 8 * k, vdesc, kIdescPV,
                                (j > 0 || k > 0) ? 1u : 0u);
            }
            tc::mma_commit(&bar[B_ODONE + u]);
        };
        ok = warp_wait(&bar[B_QFULL], 0) && warp_wait(&bar[B_KFULL], 0);
        if (ok) {
            tc::fence_after_sync();
            if (lane == 0) {
                for (int u = 0; u < units; ++u) qk(u, 0);
                tc::mma_commit(&bar[B_KEMPTY]);
            }
            __syncwarp();
        }
        // Per tile, unit by unit: P_u V, then (once P_u has been read) the
        // next tile's S_u.  Unit 1's softmax then runs while unit 0's MMAs
        // execute and the other way round.
        for (int j = 0; j < nt && ok; ++j) {
            const int sv = j % kVStages;
            if (!warp_wait(&bar[B_VCONV + sv], (j / kVStages) & 1)) { ok = false; break; }
            const bool next = j + 1 < nt;
            if (next && !warp_wait(&bar[B_KFULL + ((j + 1) & 1)], ((j + 1) >> 1) & 1)) { ok = false; break; }
            for (int u = 0; u < units && ok; ++u) {
                if (!warp_wait(&bar[B_PFULL + u], j & 1)) { ok = false; break; }
                tc::fence_after_sync();
                if (lane == 0) {
                    pv(u, j);
                    if (u == units - 1) tc::mma_commit(&bar[B_VEMPTY + sv]);  // V tile j read
                }
                __syncwarp();
                if (next) {
                    if (!warp_wait(&bar[B_ODONE + u], j & 1)) { ok = false; break; }  // P_u(j) consumed
                    tc::fence_after_sync();
                    if (lane == 0) qk(u, j + 1);
                    __syncwarp();
                }
            }
            if (!ok) break;
            if (lane == 0 && next) tc::mma_commit(&bar[B_KEMPTY + ((j + 1) & 1)]);
            __syncwarp();
        }
    } else if (warp < kConvWarps) {
        // ------------------------------------------------------ V to fp16
        // Warps 0-15 convert each V tile in place, a sixteenth (128 16-byte
        // chunks at head_dim 128, contiguous) each; the map is elementwise,
        // so the 128-byte swizzle is irrelevant.  On the last tile, rows of
        // keys past the last visible position (unused slots of the last
        // block, blocks never loaded) are zeroed instead: a 0 weight times a
        // NaN would poison the MMA.  A softmax warp converts tile j right
        // before it waits for S of tile j, while the MMAs run.  Spread over
        // all sixteen warps (all four SM sub-partitions), the work stays off
        // the softmax's critical path; two dedicated warps on two
        // sub-partitions slowed it down.
        float vmax = 0.f;
        auto convert_v = [&](int j) -> bool {
            const int sv = j % kVStages;
            if (!warp_wait(&bar[B_VFULL + sv], (j / kVStages) & 1)) return false;
            constexpr int kChunksPerWarp = kPanels * kPanelBytes / 16 / kConvWarps;  // 16-byte chunks
            const uint32_t base = smem_addr(smem + OFF_V + sv * kTileBytes) +
                                  static_cast<uint32_t>(warp) * (kChunksPerWarp * 16u);
            const int nrows = (j == nt - 1) ? klast : kTileN;
#pragma unroll
            for (int n = 0; n < kChunksPerWarp / 32; ++n) {
                const int i = warp * kChunksPerWarp + n * 32 + lane;  // chunk of the tile
                const uint32_t a = base + static_cast<uint32_t>(n * 32 + lane) * 16u;
                if (((i >> 3) & (kTileN - 1)) < nrows) {
                    uint32_t x[4];
                    tc::lds128(a, x);
                    tc::sts128(a, bf16x2_to_f16x2(x[0], vmax), bf16x2_to_f16x2(x[1], vmax),
                               bf16x2_to_f16x2(x[2], vmax), bf16x2_to_f16x2(x[3], vmax));
                } else {
                    tc::sts128(a, 0u, 0u, 0u, 0u);
                }
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_VCONV + sv]);
            return true;
        };
        const int u = warp / kSoftmaxWarps;
        if (u >= units) {
            for (int j = 0; j < nt && ok; ++j) ok = convert_v(j);
        } else {
        // ------------------------------------------------------ softmax rows
        // Eight warps per unit: warps w and w + 4 share TMEM lane quarter
        // w % 4 and take its first and second 16 lanes (16-lane shapes).
        // Thread t holds rows ra = t/4 and ra + 8 of those 16 and columns
        // 8g + 2(t%4) and + 1 of every group g of 8, so a row is spread over
        // the 4 threads of a quad: its maximum and sum take two shuffles,
        // and its P pairs land in the layout of the 16x128b store (P column
        // 4g + t%4 holds keys 8g + 2(t%4) and + 1).
        const int hh = (warp >> 2) & 1;
        const int ma = 32 * (warp & 3) + 16 * hh + lane / 4;  // tile rows ma and ma + 8
        const int mb = ma + 8;
        const int tq = lane & 3;
        const uint32_t tlane = static_cast<uint32_t>(32 * (warp & 3) + 16 * hh) << 16;
        const int h = h0 + u;
        const int pos_a = (ma < rows) ? pmin + ma : pmax;
        const int pos_b = (mb < rows) ? pmin + mb : pmax;
        float mua = -INFINITY, mub = -INFINITY;  // reference maxima of the two rows
        float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);  // row sums of P
        for (int j = 0; j < nt && ok; ++j) {
            // V tile j first (unit 1 gets here while unit 0 still works on
            // tile j), then S of tile j.
            if (!convert_v(j) || !warp_wait(&bar[B_SFULL + u], j & 1)) { ok = false; break; }
            tc::fence_after_sync();
            const int kbase = j * kTileN;
            // Rows grow with the lane, so the tile is fully visible to the
            // warp when its last key is visible to the warp's first row.
            const bool full = kbase + kTileN - 1 <= __shfl_sync(FULL, pos_a, 0);
            uint32_t sr[64];  // groups 0-7, then 8-15
            tc::tmem_ld16x256b_x8(tmem + tlane + col_s(u), *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
            tc::tmem_ld16x256b_x8(tmem + tlane + col_s(u) + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
            tc::tmem_wait_ld();
            // Pass 1: each row's maximum over the tile (raw scores; the scale
            // is positive, so it is applied afterwards).
            float xa0 = -INFINITY, xa1 = -INFINITY, xb0 = -INFINITY, xb1 = -INFINITY;
            if (full) {
#pragma unroll
                for (int g = 0; g < 16; g += 2) {
                    xa0 = fmax3(xa0, __uint_as_float(sr[4 * g]), __uint_as_float(sr[4 * g + 1]));
                    xa1 = fmax3(xa1, __uint_as_float(sr[4 * g + 4]), __uint_as_float(sr[4 * g + 5]));
                    xb0 = fmax3(xb0, __uint_as_float(sr[4 * g + 2]), __uint_as_float(sr[4 * g + 3]));
                    xb1 = fmax3(xb1, __uint_as_float(sr[4 * g + 6]), __uint_as_float(sr[4 * g + 7]));
                }
            } else {
#pragma unroll
                for (int g = 0; g < 16; ++g) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int key = kbase + 8 * g + 2 * tq + c;
                        if (key <= pos_a) xa0 = fmaxf(xa0, __uint_as_float(sr[4 * g + c]));
                        if (key <= pos_b) xb0 = fmaxf(xb0, __uint_as_float(sr[4 * g + 2 + c]));
                    }
                }
            }
            float mxa = fmaxf(xa0, xa1), mxb = fmaxf(xb0, xb1);
            mxa = fmaxf(mxa, __shfl_xor_sync(FULL, mxa, 1));
            mxb = fmaxf(mxb, __shfl_xor_sync(FULL, mxb, 1));
            mxa = fmaxf(mxa, __shfl_xor_sync(FULL, mxa, 2));
            mxb = fmaxf(mxb, __shfl_xor_sync(FULL, mxb, 2));
            const float mta = mxa * P.scale_log2, mtb = mxb * P.scale_log2;
            // A new reference only when the maximum grew by more than 2^8;
            // O is then rescaled by alpha after pass 2 (before P is handed
            // to the MMA warp), l now.
            float alpha_a = 1.f, alpha_b = 1.f;
            bool rescale = false;
            if (j == 0) {
                mua = mta;
                mub = mtb;
            } else {
                const bool need_a = mta > mua + kRescaleThreshold, need_b = mtb > mub + kRescaleThreshold;
                rescale = __any_sync(FULL, need_a || need_b);
                if (need_a) {
                    alpha_a = fast_exp2(mua - mta);
                    mua = mta;
                    la.x *= alpha_a;
                    la.y *= alpha_a;
                }
                if (need_b) {
                    alpha_b = fast_exp2(mub - mtb);
                    mub = mtb;
                    lb.x *= alpha_b;
                    lb.y *= alpha_b;
                }
            }
            // Pass 2: P = exp2(scale * s - reference) as fp16 pairs, written
            // over the first 64 S columns; the row sums in fp32.
            const float2 sc2 = make_float2(P.scale_log2, P.scale_log2);
            const float2 nma = make_float2(-mua, -mua), nmb = make_float2(-mub, -mub);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
            uint32_t w[16];
#pragma unroll
            for (int g = 8 * hf; g < 8 * hf + 8; ++g) {
                const float2 xa = __ffma2_rn(make_float2(__uint_as_float(sr[4 * g]), __uint_as_float(sr[4 * g + 1])),
                                             sc2, nma);
                const float2 xb = __ffma2_rn(
                    make_float2(__uint_as_float(sr[4 * g + 2]), __uint_as_float(sr[4 * g + 3])), sc2, nmb);
                float2 pa = make_float2(fast_exp2(xa.x), fast_exp2(xa.y));
                float2 pb = make_float2(fast_exp2(xb.x), fast_exp2(xb.y));
                if (!full) {  // keys past the row's position (NaN in unused slots included)
                    const int key = kbase + 8 * g + 2 * tq;
                    if (key > pos_a) pa.x = 0.f;
                    if (key + 1 > pos_a) pa.y = 0.f;
                    if (key > pos_b) pb.x = 0.f;
                    if (key + 1 > pos_b) pb.y = 0.f;
                }
                w[2 * (g - 8 * hf)] = tc::pack_f16x2(pa.x, pa.y);
                w[2 * (g - 8 * hf) + 1] = tc::pack_f16x2(pb.x, pb.y);
                la = __fadd2_rn(la, pa);
                lb = __fadd2_rn(lb, pb);
            }
            tc::tmem_st16x128b_x8(tmem + tlane + col_s(u) + 32 * hf, w);
            }
            if (rescale) {
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t r[32];
                    const uint32_t ta = tmem + tlane + col_o(u) + 64 * c;
                    tc::tmem_ld16x256b_x8(ta, r);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        r[4 * g] = __float_as_uint(__uint_as_float(r[4 * g]) * alpha_a);
                        r[4 * g + 1] = __float_as_uint(__uint_as_float(r[4 * g + 1]) * alpha_a);
                        r[4 * g + 2] = __float_as_uint(__uint_as_float(r[4 * g + 2]) * alpha_b);
                        r[4 * g + 3] = __float_as_uint(__uint_as_float(r[4 * g + 3]) * alpha_b);
                    }
                    tc::tmem_st16x256b_x8(ta, r);
                }
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_PFULL + u]);
        }
        if (ok && nt > 0) {
            if (!warp_wait(&bar[B_ODONE + u], (nt - 1) & 1)) {
                ok = false;
            } else {
                tc::fence_after_sync();
                float sa = la.x + la.y, sb = lb.x + lb.y;
                sa += __shfl_xor_sync(FULL, sa, 1);
                sb += __shfl_xor_sync(FULL, sb, 1);
                sa += __shfl_xor_sync(FULL, sa, 2);
                sb += __shfl_xor_sync(FULL, sb, 2);
                const float inva = 1.f / sa, invb = 1.f / sb;
                float* oa = P.out + (static_cast<size_t>(row0 + ma) * P.hq + h) * D;
                float* ob = P.out + (static_cast<size_t>(row0 + mb) * P.hq + h) * D;
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t r[32];
                    tc::tmem_ld16x256b_x8(tmem + tlane + col_o(u) + 64 * c, r);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        const int col = 64 * c + 8 * g + 2 * tq;
                        if (ma < rows)
                            *reinterpret_cast<float2*>(oa + col) =
                                make_float2(__uint_as_float(r[4 * g]) * inva, __uint_as_float(r[4 * g + 1]) * inva);
                        if (mb < rows)
                            *reinterpret_cast<float2*>(ob + col) = make_float2(__uint_as_float(r[4 * g + 2]) * invb,
                                                                               __uint_as_float(r[4 * g + 3]) * invb);
                    }
                }
            }
        } else if (bad && s >= 0) {
            // Zero rows for a sequence whose arguments were out of range.
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int m = e ? mb : ma;
                if (m < rows) {
                    float* orow = P.out + (static_cast<size_t>(row0 + m) * P.hq + h) * D;
                    for (int c = 2 * tq; c < D; c += 8)
                        *reinterpret_cast<float2*>(orow + c) = make_float2(0.f, 0.f);
                }
            }
        }
        }
        // The CTA's largest visible |v|, for the range check after the loop.
        const float wmax = warp_max(vmax);
        if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(&info[I_VMAX]), __float_as_uint(wmax));
    }
    if (!ok) record_error(P.err, kErrTimeout, 0x100u + static_cast<uint32_t>(warp));
    // ---------------------------------------------------------- teardown
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == kLoadWarp) tc::tmem_dealloc(tmem, kTmemCols);
    // V values outside the range where the fp16 P.V holds the tolerance (a
    // visible |v| above 65504 became inf; if every |v| is below 2^-12 most
    // of them are fp16 subnormals): recompute this CTA's rows exactly.
    const float cta_vmax = __uint_as_float(static_cast<unsigned int>(info[I_VMAX]));
    if (nt > 0 && !bad && (cta_vmax > 65504.f || cta_vmax < 0x1p-12f)) {
        const bool all_ok = __syncthreads_and(ok);
        if (all_ok) redo_rows_exact<D>(P, s, row0, rows, pmin, h0, units, g, warp, lane);
    }
}

}  // namespace

// The driver's tensor-map encoder, looked up once through the runtime.
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool make_tile_map(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, cuuint32_t rank,
                   const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    std::memset(map, 0, sizeof(*map));
    const CUresult r = fn(map, dtype, rank, const_cast<void*>(base), dims, strides_bytes, box, elem_strides,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_bf16_map(CUtensorMap* map, const void* base, cuuint32_t rank, const cuuint64_t* dims,
                   const cuuint64_t* strides_bytes, const cuuint32_t* box) {
    return make_tile_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides_bytes, box);
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
    if (a.head_dim != 64 && a.head_dim != kMaxHeadDim) return cudaErrorNotSupported;
    if (a.num_tiles == 0) return cudaSuccess;
    CUtensorMap tq, tk, tv;
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.head_dim), static_cast<cuuint64_t>(a.num_q_heads),
                                    static_cast<cuuint64_t>(a.num_tokens)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.head_dim) * 2,
                                       static_cast<cuuint64_t>(a.num_q_heads) * a.head_dim * 2};
        const cuuint32_t box[3] = {64, 1, kTileM};
        if (!make_bf16_map(&tq, a.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t rows = static_cast<cuuint64_t>(a.num_blocks) * a.num_kv_heads * kBlockSize;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.head_dim), rows > 0 ? rows : 1};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.head_dim) * 2};
        const cuuint32_t box[2] = {64, kBlockSize};
        if (!make_bf16_map(&tk, a.k_pool, 2, dims, strides, box)) return cudaErrorInvalidValue;
        if (!make_bf16_map(&tv, a.v_pool, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    PrefillParams P;
    P.q = static_cast<const uint8_t*>(a.q);
    P.k_pool = static_cast<const uint8_t*>(a.k_pool);
    P.v_pool = static_cast<const uint8_t*>(a.v_pool);
    P.block_tables = a.block_tables;
    P.context_lens = a.context_lens;
    P.qsl = a.query_start_loc;
    P.out = a.out;
    P.err = a.err;
    P.num_blocks = a.num_blocks;
    P.hkv = a.num_kv_heads;
    P.hq = a.num_q_heads;
    P.num_seqs = a.num_seqs;
    P.max_blocks = a.max_blocks_per_seq;
    P.ctx_cap = static_cast<int32_t>(
        std::min<int64_t>(a.max_context_len, static_cast<int64_t>(a.max_blocks_per_seq) * kBlockSize));
    P.num_tokens = a.num_tokens;
    // Two q heads per CTA when a GQA group holds an even number of them.
    P.units = ((a.num_q_heads / a.num_kv_heads) % 2 == 0) ? 2 : 1;
    P.split_last = P.units == 2 ? a.split_last : 0;
    P.scale_log2 = a.scale * kLog2e;
    auto kernel = a.head_dim == 64 ? prefill_kernel<64> : prefill_kernel<kMaxHeadDim>;
    static bool configured[2][64] = {};
    const int which = a.head_dim == 64 ? 0 : 1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[which][dev]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured[which][dev] = true;
    }
    dim3 grid(static_cast<unsigned>(a.num_tiles + (P.units == 2 ? a.split_tiles : 0)),
              static_cast<unsigned>(a.num_q_heads / P.units));
    return launch_overlapped(kernel, grid, dim3(kThreads), SMEM_BYTES, stream, tq, tk, tv, P);
}

}  // namespace pkv
