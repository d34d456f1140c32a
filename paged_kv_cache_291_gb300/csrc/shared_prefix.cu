// shared_prefix.cu -- decode attention over the leading blocks that every
// sequence of a batch shares, read once per kv head for all of them.
//
// [KV2] section 2, "Sharing blocks": requests may point at the same physical
// block (a prompt shared by parallel samples or beams, or a common system
// prompt that the prefix cache maps to the same blocks, [ENG] "Prefix
// Caching").  Plain paged decode reads such a block once per sequence that
// holds it.  Here the first J entries of every block table (the same full
// blocks for every sequence) are attended once per (block, kv head) by the
// queries of the whole batch: per slab that is the product of the batch's
// B x G query rows (G = Hq / Hkv) with 16 keys, a dense contraction, so it
// runs on tensor cores.  The decode kernel then attends each sequence's own
// blocks and merges its state with the states left here (log-sum-exp rule),
// so the result is attention over the whole context.
//
//  * Grid (chunk, kv head, query tile), one cluster of C CTAs per (kv head,
//    query tile): CTA c takes chunk c of the J shared blocks (blocks
//    [c J / C, (c + 1) J / C)) for one kv head and 64 query rows (row r =
//    sequence r / G, q head g G + r % G).
//  * Warp 8 streams the chunk's K and V slabs with tiled TMA copies (one
//    16-row box per 64-dim panel, 128-byte swizzle) into a ring of stages;
//    it reads the chunk's table entries 32 at a time.
//  * Warps 0..7 form two groups of four; group j takes the chunk's blocks
//    j, j + 2, ...: a block's time is set by the latency of its MMA and
//    softmax chains, so two blocks are in flight per CTA.
//    A warp holds 16 query rows as MMA operands (mma.sync m16n8k16, bf16
//    operands, fp32 accumulators) and per block computes
//        S = Q K^T  (16 rows x 16 keys),
//        online softmax in registers (the running maximum moves only when
//        a block's maximum exceeds it by more than 2^8),
//        O += P V   with P split into bf16 hi + lo parts (P to 2^-17
//                   relative; two MMAs per tile).
//    The accumulator layout of S (rows g, g+8 and key pairs 2t, 2t+1 of
//    each 8-key tile, lane = 4 g + t) is the A-operand layout of P for a
//    16-key step, so P never moves between lanes.
//  * The contractions may run over their index in any order, so the
//    operands' dims are permuted: a lane reads whole 16-byte chunks of K
//    and V rows, and the 8 lanes of each shared-memory load phase hit 8
//    different 16-byte bank groups of the swizzled slab.
//  * Each group leaves every row's state of its blocks -- m (the log2-
//    domain reference maximum), l = sum 2^(x - m) and the unnormalised o --
//    in shared memory, and the CTA merges its groups' states (log-sum-exp
//    rule).  After a cluster barrier CTA c merges rows [64 c / C,
//    64 (c + 1) / C) over the C states of the cluster (read through
//    distributed shared memory) and writes one state per (sequence, q head)
//    for the decode kernel.
//  * The shared blocks are taken from sequence 0's table.  Every CTA checks
//    that its sequences' tables hold the same ids over its chunk and that
//    their contexts extend past the prefix; a mismatch is reported as
//    PKV_ERR_RANGE (the results of the call are then not valid).
//  * Every wait is bounded; on expiry the CTA records PKV_ERR_TIMEOUT and
//    unwinds after its copies in flight have landed.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kRowsPerCta = 64;                  // query rows per CTA
constexpr int kGroups = 2;                       // warp groups splitting a chunk's blocks
constexpr int kWarpsPerGroup = kRowsPerCta / 16;  // one warp per 16 query rows
constexpr int kConsumerWarps = kGroups * kWarpsPerGroup;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kStages = 8;
constexpr int kPanelBytes = kBlockSize * 128;  // 16 rows x 64 bf16
constexpr int kMaxChunks = 8;                  // CTAs of one cluster (the portable cluster size)
constexpr int kTargetCtas = 152;               // CTAs a launch aims at (chunks x kv heads x tiles)
constexpr int kMinChunkBlocks = 4;             // fewest shared blocks per chunk
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct PrefixParams {
    const uint8_t* q;              // bf16 [S][Hq][D]
    const int32_t* block_tables;   // [S][max_blocks]
    const int32_t* context_lens;   // [S]
    float2* pre_ml;                // [S][Hq] (m, l) of the shared blocks
    float* pre_o;                  // [S][Hq][D] their unnormalised o
    unsigned long long* err;
    int32_t num_blocks, hkv, hq, num_seqs, max_blocks, shared_blocks;
    float scale_log2;
};

template <int D>
struct PCfg {
    static constexpr int PANELS = D / 64;
    static constexpr int SLAB = PANELS * kPanelBytes;  // one (block, kv head): K or V
    static constexpr int STAGE = 2 * SLAB;
    static constexpr int RING = kStages * STAGE;
    // After the block loop the ring's bytes hold the groups' states:
    // o [kGroups][kRowsPerCta][D] fp32, then (m, l) [kGroups][kRowsPerCta],
    // then the CTA's merged (m, l) [kRowsPerCta] (its o is merged in place
    // into group 0's rows).
    static constexpr int OFF_MO = 0;
    static constexpr int OFF_MML = kGroups * kRowsPerCta * D * 4;
    static constexpr int OFF_CML = OFF_MML + kGroups * kRowsPerCta * 8;
    static constexpr int MERGE = OFF_CML + kRowsPerCta * 8;
    static constexpr int OFF_BAR = RING > MERGE ? RING : MERGE;
    static constexpr int SMEM_USED = OFF_BAR + 2 * kStages * 8 + 16;
    static constexpr int SMEM = SMEM_USED + 1024;  // slack to align the base to 1024 B
    static_assert(STAGE % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
    static_assert(OFF_MML % 16 == 0 && OFF_CML % 8 == 0 && OFF_BAR % 8 == 0, "aligned regions");
    static_assert(kStages % kGroups == 0, "a group's blocks keep to its own stages");
};

// Byte offset of 16-byte chunk c (dims 8c .. 8c+7) of row r in a slab of
// 64-dim panels stored with the 128-byte swizzle: within a row's 128 bytes
// the chunk index is XORed with r mod 8.
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>((c >> 3) * kPanelBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// The chunk of a K (or q) row that quad lane t reads for chunk step i: its
// dims serve k-steps 2i and 2i+1 of S = Q K^T.
__device__ __forceinline__ int kchunk(int t, int i) { return 2 * t + (i & 1) + 8 * (i >> 1); }

__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two floats -> bf16x2 (nearest even), lo in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// A pair of probabilities as bf16 MMA operands: hi = p rounded, lo = the
// rounded rest (p - hi is exact in fp32), so hi + lo = p to 2^-17 relative.
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = bf16x2_rn(a, b);
    lo = bf16x2_rn(a - bf16lo(hi), b - bf16hi(hi));
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}

// Loads from another CTA's shared memory, issued back to back (they only
// run between the two cluster barriers, which order them).
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t a) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
    return v;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a));
    return v;
}

// The producer warp: the chunk's table entries (sequence 0's row) are read
// 32 at a time by the whole warp, the next batch requested before this
// one's copies; lane 0 issues each block's copies once its stage is free.
template <int D>
__device__ void produce(const CUtensorMap* tk, const CUtensorMap* tv, const PrefixParams& P, uint8_t* smem,
                        uint64_t* full, uint64_t* empty, volatile int* abort_flag, int g, int j0, int nblk,
                        int lane) {
    using C = PCfg<D>;
    const unsigned FULL = 0xffffffffu;
    const int32_t* row0 = P.block_tables + j0;
    int k = 0;
    bool bad = false;
    int e = (lane < nblk) ? __ldg(row0 + lane) : 0;
    for (int base = 0; base < nblk && !bad; base += 32) {
        const int e_next = (base + 32 + lane < nblk) ? __ldg(row0 + base + 32 + lane) : 0;
        const int cnt = min(32, nblk - base);
        for (int i = 0; i < cnt; ++i) {
            k = base + i;
            const int st = k % kStages;
            int phys = __shfl_sync(FULL, e, i);
            int ok = 1;
            if (lane == 0) {
                if (*abort_flag || !mbar_wait(&empty[st], ((k / kStages) & 1) ^ 1)) {
                    ok = 0;
                } else {
                    if (phys < 0 || phys >= P.num_blocks) {
                        record_error(P.err, kErrRange, 0u);
                        phys = 0;  // never address an invalid id
                    }
                    const int y = (phys * P.hkv + g) * kBlockSize;  // the slab's first row in the pool's row space
                    uint8_t* dst = smem + st * C::STAGE;
                    mbar_arrive_expect_tx(&full[st], C::STAGE);
#pragma unroll
                    for (int p = 0; p < C::PANELS; ++p) {
                        tc::tma_load_2d(dst + p * kPanelBytes, tk, p * 64, y, &full[st]);
                        tc::tma_load_2d(dst + C::SLAB + p * kPanelBytes, tv, p * 64, y, &full[st]);
                    }
                }
            }
            if (!__shfl_sync(FULL, ok, 0)) {
                bad = true;
                break;
            }
        }
        e = e_next;
    }
    if (bad && lane == 0) {
        *abort_flag = 1;
        record_error(P.err, kErrTimeout, 4u);
        // Blocks 0 .. k-1 were issued; only the last use of each stage can
        // still be in flight.
        for (int kk = max(0, k - kStages); kk < k; ++kk) mbar_wait(&full[kk % kStages], (kk / kStages) & 1);
    }
    __syncwarp();
}

// The tables of this tile's sequences hold sequence 0's ids over the chunk,
// and their contexts reach past the shared prefix.  The kv heads' CTAs of a
// (chunk, tile) share the work: CTA g checks the sequences s = g mod Hkv
// (the chunk's first CTA also their lengths).  It runs after the CTA's
// blocks, off the path to the first MMA.
__device__ void check_shared(const PrefixParams& P, int G, int j0, int nblk, int tid, int nthreads) {
    const int s_lo = blockIdx.z * kRowsPerCta / G;
    const int s_hi = min(P.num_seqs, ((blockIdx.z + 1) * kRowsPerCta + G - 1) / G);
    const int per = nblk + 1;
    const int first = s_lo + (static_cast<int>(blockIdx.y) - s_lo % P.hkv + P.hkv) % P.hkv;
    const int mine = first < s_hi ? (s_hi - 1 - first) / P.hkv + 1 : 0;
    const long long total = static_cast<long long>(mine) * per;
    for (long long x = tid; x < total; x += nthreads) {
        const int s = first + static_cast<int>(x / per) * P.hkv;
        const int k = static_cast<int>(x % per);
        if (k == nblk) {
            if (blockIdx.x == 0 && __ldg(P.context_lens + s) < P.shared_blocks * kBlockSize)
                record_error(P.err, kErrRange, static_cast<uint32_t>(s));
        } else if (__ldg(P.block_tables + static_cast<size_t>(s) * P.max_blocks + j0 + k) !=
                   __ldg(P.block_tables + j0 + k)) {
            record_error(P.err, kErrRange, static_cast<uint32_t>(s));
        }
    }
}

// Consumer warp `warp` (group warp / 4, rows 16 (warp % 4) .. + 15 of the
// tile): the group's blocks of the chunk, then its rows' states into the
// merge area (after all consumer warps are done with the ring).
template <int D>
__device__ void consume(const PrefixParams& P, uint8_t* smem, uint64_t* full, uint64_t* empty,
                        volatile int* abort_flag, int G, int g, int nblk, int warp, int lane) {
    using C = PCfg<D>;
    constexpr int KS = D / 16;  // k-steps of S = Q K^T
    constexpr int NT = D / 8;   // 8-dim n-tiles of O
    const unsigned FULL = 0xffffffffu;
    const int g8 = lane >> 2, t = lane & 3;
    const int group = warp / kWarpsPerGroup, wq = warp % kWarpsPerGroup;
    const int rows = P.num_seqs * G;
    const int rbase = blockIdx.z * kRowsPerCta + wq * 16;

    // Q as A operands: qa[ks] = {rows g8 and g8+8} x {k pairs 2t, 2t+8} of
    // k-step ks; chunk step i gives k-steps 2i (words 0, 1) and 2i + 1
    // (words 2, 3).  Rows past the batch are zero.
    uint32_t qa[KS][4];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int r = rbase + g8 + 8 * rr;
        const bool live = r < rows;
        const size_t qrow = live ? (static_cast<size_t>(r / G) * P.hq + static_cast<size_t>(g) * G + r % G) : 0;
        const uint8_t* qp = P.q + qrow * D * 2;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
            uint4 u = make_uint4(0u, 0u, 0u, 0u);
            if (live) u = __ldg(reinterpret_cast<const uint4*>(qp + kchunk(t, i) * 16));
            qa[2 * i][rr] = u.x;
            qa[2 * i][2 + rr] = u.y;
            qa[2 * i + 1][rr] = u.z;
            qa[2 * i + 1][2 + rr] = u.w;
        }
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows g8, g8 + 8
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    bool ok = true;
    for (int k = group; k < nblk; k += kGroups) {
        const int st = k % kStages;
        if (*abort_flag || !mbar_wait_warp(&full[st], (k / kStages) & 1)) {
            ok = false;
            break;
        }
        const uint8_t* kst = smem + st * C::STAGE;
        const uint8_t* vst = kst + C::SLAB;
        // ---- S = Q K^T: key tile nt holds keys 8 nt .. 8 nt + 7 (B operand
        // column g8 = key 8 nt + g8).
        // Two accumulator sets per key tile (even and odd k-steps) halve the
        // dependent MMA chain.
        float s[2][4], s2[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[nt][j] = s2[nt][j] = 0.f;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const uint4 u = lds128(kst + swz(nt * 8 + g8, kchunk(t, i)));
                mma_bf16(s[nt], qa[2 * i], u.x, u.y);
                mma_bf16(s2[nt], qa[2 * i + 1], u.z, u.w);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[nt][j] += s2[nt][j];
        // ---- online softmax (log2 domain); s[nt] = rows (g8, g8+8) x keys
        // (8 nt + 2t, + 1); a row's 16 keys sit in the 4 lanes of its quad.
        float x[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) x[nt][j] = s[nt][j] * P.scale_log2;
        float mb0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
        float mb1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
        mb0 = fmaxf(mb0, __shfl_xor_sync(FULL, mb0, 1));
        mb1 = fmaxf(mb1, __shfl_xor_sync(FULL, mb1, 1));
        mb0 = fmaxf(mb0, __shfl_xor_sync(FULL, mb0, 2));
        mb1 = fmaxf(mb1, __shfl_xor_sync(FULL, mb1, 2));
        if (mb0 > m0 + kRescaleThreshold) {
            const float a = fast_exp2(m0 - mb0);
            l0 *= a;
#pragma unroll
            for (int n = 0; n < NT; ++n) o[n][0] *= a, o[n][1] *= a;
            m0 = mb0;
        }
        if (mb1 > m1 + kRescaleThreshold) {
            const float a = fast_exp2(m1 - mb1);
            l1 *= a;
#pragma unroll
            for (int n = 0; n < NT; ++n) o[n][2] *= a, o[n][3] *= a;
            m1 = mb1;
        }
        float p[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            p[nt][0] = fast_exp2(x[nt][0] - m0);
            p[nt][1] = fast_exp2(x[nt][1] - m0);
            p[nt][2] = fast_exp2(x[nt][2] - m1);
            p[nt][3] = fast_exp2(x[nt][3] - m1);
        }
        l0 += (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
        l1 += (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
        // P as the A operand of a 16-key step: {row g8, row g8+8} x {keys
        // 2t, 2t+1 (tile 0), keys 8+2t, 8+2t+1 (tile 1)}.
        uint32_t ph[4], pl[4];
        split_pair(p[0][0], p[0][1], ph[0], pl[0]);
        split_pair(p[0][2], p[0][3], ph[1], pl[1]);
        split_pair(p[1][0], p[1][1], ph[2], pl[2]);
        split_pair(p[1][2], p[1][3], ph[3], pl[3]);
        // ---- O += P V.  n-tile 8 hh + e, column n is dim 8 (n + 8 hh) + e:
        // lane (g8, t) reads chunk g8 + 8 hh of V rows 2t, 2t+1, 2t+8, 2t+9
        // and takes element e of each for the B operand.
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
            const int c = g8 + 8 * hh;
            const uint4 ra = lds128(vst + swz(2 * t, c)), rb = lds128(vst + swz(2 * t + 1, c));
            const uint4 rc = lds128(vst + swz(2 * t + 8, c)), rd = lds128(vst + swz(2 * t + 9, c));
            const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
            const uint32_t wc[4] = {rc.x, rc.y, rc.z, rc.w}, wd[4] = {rd.x, rd.y, rd.z, rd.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int n = 8 * hh + 2 * w;
                uint32_t b0 = __byte_perm(wa[w], wb[w], 0x5410), b1 = __byte_perm(wc[w], wd[w], 0x5410);
                mma_bf16(o[n], ph, b0, b1);
                mma_bf16(o[n], pl, b0, b1);
                b0 = __byte_perm(wa[w], wb[w], 0x7632);
                b1 = __byte_perm(wc[w], wd[w], 0x7632);
                mma_bf16(o[n + 1], ph, b0, b1);
                mma_bf16(o[n + 1], pl, b0, b1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (!ok) {
        *abort_flag = 1;
        record_error(P.err, kErrTimeout, 5u);
    }
    l0 += __shfl_xor_sync(FULL, l0, 1);
    l1 += __shfl_xor_sync(FULL, l1, 1);
    l0 += __shfl_xor_sync(FULL, l0, 2);
    l1 += __shfl_xor_sync(FULL, l1, 2);
    // The merge area overlaps the ring: wait until every consumer warp is
    // past its last block (the producer issues nothing after the last one).
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    // ---- the group's state of the warp's 16 rows.  o[8 hh + e][cc + 2 rr]
    // is row g8 + 8 rr, dim 8 (2t + cc + 8 hh) + e.
    float* mo = reinterpret_cast<float*>(smem + C::OFF_MO) + group * kRowsPerCta * D;
    float2* mml = reinterpret_cast<float2*>(smem + C::OFF_MML) + group * kRowsPerCta;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int row = wq * 16 + g8 + 8 * rr;
        if (t == 0) mml[row] = make_float2(rr ? m1 : m0, rr ? l1 : l0);
        float* orow = mo + row * D;
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int j = cc + 2 * rr;
                float4* dst = reinterpret_cast<float4*>(orow + 8 * (2 * t + cc + 8 * hh));
                dst[0] = make_float4(o[8 * hh][j], o[8 * hh + 1][j], o[8 * hh + 2][j], o[8 * hh + 3][j]);
                dst[1] = make_float4(o[8 * hh + 4][j], o[8 * hh + 5][j], o[8 * hh + 6][j], o[8 * hh + 7][j]);
            }
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    // ---- the CTA's state: the groups' states merged (log-sum-exp), o in
    // place over group 0's rows (each float4 by one thread), (m, l) apart.
    constexpr int C4 = D / 4;
    const float2* gml = reinterpret_cast<const float2*>(smem + C::OFF_MML);
    float4* o4 = reinterpret_cast<float4*>(smem + C::OFF_MO);
    float2* cml = reinterpret_cast<float2*>(smem + C::OFF_CML);
    for (int it = warp * 32 + lane; it < kRowsPerCta * C4; it += kConsumerWarps * 32) {
        const int row = it / C4, c4 = it % C4;
        float2 e[kGroups];
        float M = -INFINITY;
#pragma unroll
        for (int gr = 0; gr < kGroups; ++gr) {
            e[gr] = gml[gr * kRowsPerCta + row];
            M = fmaxf(M, e[gr].x);
        }
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int gr = 0; gr < kGroups; ++gr) {
            const float w = (e[gr].x == -INFINITY) ? 0.f : fast_exp2(e[gr].x - M);
            const float4 v = o4[(gr * kRowsPerCta + row) * C4 + c4];
            L = fmaf(e[gr].y, w, L);
            acc.x = fmaf(v.x, w, acc.x);
            acc.y = fmaf(v.y, w, acc.y);
            acc.z = fmaf(v.z, w, acc.z);
            acc.w = fmaf(v.w, w, acc.w);
        }
        o4[row * C4 + c4] = acc;
        if (c4 == 0) cml[row] = make_float2(M, L);
    }
}

// After the cluster barrier: this CTA's share of the tile's live rows,
// merged over the states of every CTA of the cluster (distributed shared
// memory; each source's loads issued together), to global.
template <int D>
__device__ void merge_rows(const PrefixParams& P, const uint8_t* smem, int G, int g, int tid, int nthreads) {
    using C = PCfg<D>;
    constexpr int C4 = D / 4;
    const int chunks = gridDim.x;  // = the cluster size, at most kMaxChunks
    const int rank = blockIdx.x;
    const int live = min(kRowsPerCta, P.num_seqs * G - static_cast<int>(blockIdx.z) * kRowsPerCta);
    const int r_lo = rank * kRowsPerCta / chunks;
    const int r_hi = min(live, (rank + 1) * kRowsPerCta / chunks);
    const float4* o4 = reinterpret_cast<const float4*>(smem + C::OFF_MO);
    const float2* cml = reinterpret_cast<const float2*>(smem + C::OFF_CML);
    for (int it = tid; it < (r_hi - r_lo) * C4; it += nthreads) {
        const int row = r_lo + it / C4;
        const int c4 = it % C4;
        float2 e[kMaxChunks];
        float4 v[kMaxChunks];
        float M = -INFINITY;
#pragma unroll
        for (int src = 0; src < kMaxChunks; ++src) {
            e[src] = make_float2(-INFINITY, 0.f);
            v[src] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (src < chunks) {
                e[src] = ld_cluster_f2(cluster_addr(cml + row, src));
                v[src] = ld_cluster_f4(cluster_addr(o4 + row * C4 + c4, src));
            }
            M = fmaxf(M, e[src].x);
        }
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int src = 0; src < kMaxChunks; ++src) {
            const float w = (e[src].x == -INFINITY) ? 0.f : fast_exp2(e[src].x - M);
            L = fmaf(e[src].y, w, L);
            acc.x = fmaf(v[src].x, w, acc.x);
            acc.y = fmaf(v[src].y, w, acc.y);
            acc.z = fmaf(v[src].z, w, acc.z);
            acc.w = fmaf(v[src].w, w, acc.w);
        }
        const int r = static_cast<int>(blockIdx.z) * kRowsPerCta + row;
        const size_t idx = static_cast<size_t>(r / G) * P.hq + static_cast<size_t>(g) * G + r % G;
        reinterpret_cast<float4*>(P.pre_o + idx * D)[c4] = acc;
        if (c4 == 0) P.pre_ml[idx] = make_float2(M, L);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    shared_prefix_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const PrefixParams P) {
    using C = PCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int g = blockIdx.y;
    const int J = P.shared_blocks;
    const int j0 = static_cast<int>(static_cast<long long>(blockIdx.x) * J / gridDim.x);
    const int j1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * J / gridDim.x);
    const int G = P.hq / P.hkv;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kWarpsPerGroup);  // the warps of the group that takes the stage's block
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    griddep_launch_dependents();
    __syncthreads();
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            tc::prefetch_tensormap(&tm_k);
            tc::prefetch_tensormap(&tm_v);
        }
        griddep_wait();
        produce<D>(&tm_k, &tm_v, P, smem, full, empty, abort_flag, g, j0, j1 - j0, lane);
        check_shared(P, G, j0, j1 - j0, lane, 32);
    } else {
        griddep_wait();
        consume<D>(P, smem, full, empty, abort_flag, G, g, j1 - j0, warp, lane);
    }
    // Every thread of the cluster passes both barriers: the states are
    // complete before any CTA reads them, and no CTA leaves while another
    // may still read its shared memory.
    cluster_sync_all();
    merge_rows<D>(P, smem, G, g, threadIdx.x, kThreads);
    cluster_sync_all();
}

template <int D>
cudaError_t launch_t(const DecodeArgs& a, const DecodeWsLayout& L, cudaStream_t stream) {
    using C = PCfg<D>;
    CUtensorMap tk, tv;
    const cuuint64_t rows = static_cast<cuuint64_t>(a.num_blocks) * a.num_kv_heads * kBlockSize;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), rows > 0 ? rows : 1};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
    const cuuint32_t box[2] = {64, kBlockSize};
    if (!make_bf16_map(&tk, a.k_pool, 2, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_bf16_map(&tv, a.v_pool, 2, dims, strides, box)) return cudaErrorInvalidValue;
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    PrefixParams P;
    P.q = static_cast<const uint8_t*>(a.q);
    P.block_tables = a.block_tables;
    P.context_lens = a.context_lens;
    P.pre_ml = reinterpret_cast<float2*>(ws + L.pre_ml);
    P.pre_o = reinterpret_cast<float*>(ws + L.pre_o);
    P.err = a.err;
    P.num_blocks = a.num_blocks;
    P.hkv = a.num_kv_heads;
    P.hq = a.num_q_heads;
    P.num_seqs = a.num_seqs;
    P.max_blocks = a.max_blocks_per_seq;
    P.shared_blocks = a.skip_blocks;
    P.scale_log2 = a.scale * kLog2e;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(shared_prefix_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int G = a.num_q_heads / a.num_kv_heads;
    const int tiles = static_cast<int>((static_cast<int64_t>(a.num_seqs) * G + kRowsPerCta - 1) / kRowsPerCta);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(a.prefix_chunks);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(a.prefix_chunks), static_cast<unsigned>(a.num_kv_heads),
                       static_cast<unsigned>(tiles));
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap_enabled() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, shared_prefix_kernel<D>, tk, tv, P);
}

}  // namespace

int32_t shared_prefix_chunks(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t shared_blocks) {
    if (shared_blocks <= 0 || num_seqs <= 0 || num_kv_heads <= 0 || num_q_heads < num_kv_heads) return 0;
    const int64_t G = num_q_heads / num_kv_heads;
    const int64_t tiles = (static_cast<int64_t>(num_seqs) * G + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t per_chunk = static_cast<int64_t>(num_kv_heads) * tiles;
    int64_t c = (kTargetCtas + per_chunk - 1) / per_chunk;
    c = std::min<int64_t>(c, std::max<int64_t>(1, shared_blocks / kMinChunkBlocks));
    return static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(c, kMaxChunks)));
}

cudaError_t launch_shared_prefix(const DecodeArgs& a, cudaStream_t stream) {
    if (a.skip_blocks <= 0 || a.prefix_chunks <= 0 || a.num_seqs == 0) return cudaSuccess;
    if (a.kv_e4m3 || a.prefix_chunks > kMaxChunks) return cudaErrorNotSupported;
    const DecodeWsLayout L =
        decode_ws_layout(a.num_seqs, a.num_q_heads, a.num_kv_heads, a.head_dim, a.plan.max_ranges, true);
    if (a.head_dim == 128) return launch_t<128>(a, L, stream);
    if (a.head_dim == 64) return launch_t<64>(a, L, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
