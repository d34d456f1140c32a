// block_manager.cu -- the block bookkeeping of the paged cache, on the device.
//
// "PagedAttention: splitting KV into blocks", section 2 of the serving-engine
// KV blog:
//  * "Blocks and block tables": a request's KV is cut into 16-token blocks
//    that may sit anywhere in free memory; a table maps its logical blocks to
//    physical ones, and a block is allocated at the moment the tokens fill
//    the last one (nothing is reserved ahead).
//  * "Sharing blocks": requests may point at the same block under a
//    reference count; a shared block is copied only when a holder has to
//    append to it (copy-on-write).
// Section 4 ("Prefix cache"): blocks of a finished request go back to the
// free queue tail block first.
//
// The state is caller-owned device memory (pkv_blocks_t): tables, lengths,
// reference counts and a ring of free block ids, least recently freed
// first (with the prefix cache: keys and a key table).  Keeping it on the
// device lets one decode step (append -> copy-on-write copies -> cache write
// -> attention) run without a host round trip, and be captured in a graph.
//
// The semantics are those of processing sequences one after another:
//  * append, in sequence order: a holder of a shared, partly filled last
//    block copies it while the block's count is above 1, so when every holder
//    appends in one call the last one (highest index) writes in place;
//    allocation takes blocks from the ring's head in sequence order, the
//    copy-on-write block first, then new blocks in logical order;
//  * release, in the given row order, each row's blocks last first: a block
//    joins the ring's tail when its count reaches 0, keeping its content and
//    (if registered) its key;
//  * match (prefix cache, section 4): an empty row takes the cached blocks of
//    its leading keys up to the first key not cached, taking a free one back
//    out of the queue; an append that takes a cached block drops its key;
//  * register, in (row, block) order: a block keeps a key it has, and a key
//    already cached (or given earlier in the call) keeps its first block.
// The kernels reach the same result in parallel: per-block counters in a
// scratch array (atomicAdd of holders, atomicMax of the last holder's
// position) decide who copies or frees, and CTA-wide exclusive scans turn the
// per-sequence needs into ring positions.  Every decision is taken on the
// counts as they were when the call started, before anything is written, so
// a call that fails changes nothing.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kBmThreads = 1024;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ int blocks_for(int n) { return (n + kBlockSize - 1) / kBlockSize; }

// Exclusive prefix sum of v over the CTA; *total gets the sum of all v.
// Every thread of the CTA must call it.
__device__ int cta_exclusive_scan(int v, int* wsum, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = (lane < kBmThreads / 32) ? wsum[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(kFull, wi, o);
            if (lane >= o) wi += t;
        }
        wsum[lane] = wi - w;
        if (lane == 31) wsum[32] = wi;
    }
    __syncthreads();
    const int r = wsum[warp] + incl - v;
    *total = wsum[32];
    __syncthreads();
    return r;
}

// The free queue is a ring of 2 * num_blocks entries from `head`; an entry
// at index i holding block b is live iff ring_pos[b] == i.  A block taken
// back by a prefix-cache hit only clears its ring_pos, so its entry goes
// stale; stale entries are skipped when popping and dropped when the ring is
// compacted.
__device__ __forceinline__ int ring_cap(const BlocksArgs& st) { return 2 * st.num_blocks; }

__device__ __forceinline__ bool ring_ok(const BlocksArgs& st, int head, int entries, int nfree) {
    const int cap = ring_cap(st);
    return entries >= 0 && entries <= cap && nfree >= 0 && nfree <= entries && nfree <= st.num_blocks &&
           head >= 0 && (head < cap || cap == 0);
}

__device__ __forceinline__ bool ring_live(const BlocksArgs& st, int idx, int b) {
    return b >= 0 && b < st.num_blocks && st.ring_pos[b] == idx;
}

// ---- prefix-cache table: block ids by key, linear probing, -1 = empty.
__device__ __forceinline__ int key_home(const BlocksArgs& st, const uint8_t* key) {
    return static_cast<int>(*reinterpret_cast<const uint32_t*>(key) & static_cast<uint32_t>(st.table_size - 1));
}

__device__ __forceinline__ bool key_equal(const uint8_t* a, const uint8_t* b) {
    const uint4 a0 = reinterpret_cast<const uint4*>(a)[0], a1 = reinterpret_cast<const uint4*>(a)[1];
    const uint4 b0 = reinterpret_cast<const uint4*>(b)[0], b1 = reinterpret_cast<const uint4*>(b)[1];
    return a0.x == b0.x && a0.y == b0.y && a0.z == b0.z && a0.w == b0.w && a1.x == b1.x && a1.y == b1.y &&
           a1.z == b1.z && a1.w == b1.w;
}

// The cached block holding `key`, or -1.
__device__ int table_find(const BlocksArgs& st, const uint8_t* key) {
    int i = key_home(st, key);
    for (int n = 0; n < st.table_size; ++n) {
        const int v = st.key_table[i];
        if (v < 0) return -1;
        if (key_equal(st.block_keys + static_cast<int64_t>(v) * 32, key)) return v;
        i = (i + 1) & (st.table_size - 1);
    }
    return -1;
}

// Remove block b's entry, shifting the entries after it back so that no
// probe sequence is cut (one thread at a time).
__device__ void table_erase(const BlocksArgs& st, int b) {
    const int mask = st.table_size - 1;
    int i = key_home(st, st.block_keys + static_cast<int64_t>(b) * 32);
    int n = 0;
    while (st.key_table[i] != b) {
        if (st.key_table[i] < 0 || ++n >= st.table_size) return;  // not in the table
        i = (i + 1) & mask;
    }
    int j = i;
    for (n = 0; n < st.table_size; ++n) {
        j = (j + 1) & mask;
        const int v = st.key_table[j];
        if (v < 0) break;
        const int k = key_home(st, st.block_keys + static_cast<int64_t>(v) * 32);
        // v may move to i unless its home lies cyclically in (i, j].
        const bool stays = (i <= j) ? (i < k && k <= j) : (i < k || k <= j);
        if (!stays) {
            st.key_table[i] = v;
            i = j;
        }
    }
    st.key_table[i] = -1;
}

// What row s does in this append, read from the state as it was at entry.
struct AppendRow {
    int q;        // new tokens
    int n0;       // tokens held before
    int b;        // partly filled last block it appends to, or -1
    bool bad;     // the row's inputs are out of range
};

__device__ __forceinline__ AppendRow append_row(const BlocksArgs& st, const int32_t* qsl, int s) {
    AppendRow r{0, 0, -1, false};
    r.q = qsl[s + 1] - qsl[s];
    if (r.q < 0) { r.bad = true; return r; }
    if (r.q == 0) return r;
    r.n0 = st.lens[s];
    const int cap = st.max_blocks * kBlockSize;
    if (r.n0 < 0 || r.n0 > cap - r.q) { r.bad = true; return r; }
    if (r.n0 % kBlockSize) {
        const int b = st.tables[static_cast<int64_t>(s) * st.max_blocks + r.n0 / kBlockSize];
        if (b < 0 || b >= st.num_blocks || st.refs[b] <= 0) { r.bad = true; return r; }
        r.b = b;
    }
    return r;
}

__global__ void __launch_bounds__(kBmThreads, 1)
    blocks_append_kernel(const BlocksArgs st, const int32_t* __restrict__ qsl, int32_t S, int32_t T,
                         int32_t* __restrict__ slots, int32_t* __restrict__ cow_src, int32_t* __restrict__ cow_dst,
                         int32_t* __restrict__ cow_count, unsigned long long* err) {
    __shared__ int wsum[33];
    griddep_launch_dependents();
    griddep_wait();
    const int tid = threadIdx.x;
    int32_t* cnt = st.scratch;                  // holders appending to a block
    int32_t* last = st.scratch + st.num_blocks; // highest such holder

    // A: check the rows; count the holders that append to each partly
    // filled last block.
    int bad = (tid == 0 && S > 0 && (qsl[0] != 0 || qsl[S] != T)) ? 1 : 0;
    for (int s = tid; s < S; s += kBmThreads) {
        const AppendRow r = append_row(st, qsl, s);
        bad |= r.bad;
        if (r.b >= 0) {
            atomicAdd(&cnt[r.b], 1);
            atomicMax(&last[r.b], s);
        }
    }
    bad = __syncthreads_or(bad);

    // B: who copies, and how many blocks each row takes.  Row s copies its
    // last block b when b is shared, unless s is b's last appender and every
    // holder of b appends (then the others have copied and s holds b alone).
    // The counters are read here, before the barrier of the scan that
    // follows, into registers: the last appender settles b after it.
    struct Decision {
        AppendRow r;
        int need, cow;
        bool settles;      // s is b's last appender: it applies b's new count
        int copies;        // copies of b made in this call (valid if settles)
        bool inconsistent; // more holders append to b than hold it
    };
    auto decide = [&](int s) {
        Decision d{};
        d.r = append_row(st, qsl, s);
        if (d.r.bad || d.r.q == 0) return d;
        if (d.r.b >= 0) {
            const int c = cnt[d.r.b], rc = st.refs[d.r.b];
            d.inconsistent = c > rc;
            d.cow = (rc > 1 && !(s == last[d.r.b] && c == rc)) ? 1 : 0;
            d.settles = (s == last[d.r.b]);
            d.copies = rc > 1 ? c - (c == rc ? 1 : 0) : 0;
        }
        d.need = d.cow + blocks_for(d.r.n0 + d.r.q) - blocks_for(d.r.n0);
        return d;
    };
    int need_total = 0, cow_total = 0;
    if (!bad) {
        for (int base = 0; base < S; base += kBmThreads) {
            const int s = base + tid;
            Decision d{};
            if (s < S) d = decide(s);
            if (d.inconsistent) bad = 1;
            int t1, t2;
            cta_exclusive_scan(d.need, wsum, &t1);
            cta_exclusive_scan(d.cow, wsum, &t2);
            need_total += t1;
            cow_total += t2;
        }
    }
    __shared__ int s_last;
    const int head = st.free_state[0], entries = st.free_state[1], nfree = st.free_state[2];
    if (!ring_ok(st, head, entries, nfree)) bad = 1;
    bad = __syncthreads_or(bad);
    const bool short_of_blocks = !bad && need_total > nfree;
    // P: the first need_total live entries from the ring's head, in order,
    // into alloc[].  The ids are checked to be free blocks: nothing is
    // written through an id that was not checked.
    int32_t* alloc = st.scratch + 2 * st.num_blocks;
    int consumed = 0;
    if (!bad && !short_of_blocks && need_total > 0) {
        const int cap = ring_cap(st);
        int taken = 0;
        if (tid == 0) s_last = -1;
        for (int base = 0; base < entries && taken < need_total; base += kBmThreads) {
            const int e = base + tid;
            int live = 0, b = -1;
            if (e < entries) {
                const int idx = (head + e) % cap;
                b = st.free_ring[idx];
                live = ring_live(st, idx, b) ? 1 : 0;
            }
            int t;
            const int rank = cta_exclusive_scan(live, wsum, &t);
            if (live && taken + rank < need_total) {
                alloc[taken + rank] = b;
                if (st.refs[b] != 0) bad = 1;
                if (taken + rank == need_total - 1) s_last = e;
            }
            taken = min(taken + t, need_total);
        }
        bad = __syncthreads_or(bad || (tid == 0 && s_last < 0));
        consumed = s_last + 1;
    } else {
        bad = __syncthreads_or(bad);
    }

    if (bad || short_of_blocks) {
        // Leave the state as it was (the scratch counters back to zero) and
        // make the outputs inert for the calls that follow in the step.
        for (int s = tid; s < S; s += kBmThreads) {
            const AppendRow r = append_row(st, qsl, s);
            if (r.b >= 0) {
                cnt[r.b] = 0;   // every appender of b writes the same zeros
                last[r.b] = 0;
            }
        }
        for (int t = tid; t < T; t += kBmThreads) slots[t] = -1;
        for (int s = tid; s < S; s += kBmThreads) cow_src[s] = cow_dst[s] = -1;
        if (tid == 0) {
            *cow_count = 0;
            record_error(err, bad ? kErrRange : kErrNoBlocks, 0u);
        }
        return;
    }

    // C: take blocks from the ring's head in sequence order and fill the
    // tables.  A copied block's count is settled by its last appender, the
    // block's only writer; every other row that reads it does so in this or
    // an earlier chunk, before that chunk's barrier.
    int carry_need = 0, carry_cow = 0;
    for (int base = 0; base < S; base += kBmThreads) {
        const int s = base + tid;
        Decision d{};
        if (s < S) d = decide(s);
        int t1, t2;
        const int off = carry_need + cta_exclusive_scan(d.need, wsum, &t1);
        const int coff = carry_cow + cta_exclusive_scan(d.cow, wsum, &t2);
        carry_need += t1;
        carry_cow += t2;
        if (s < S && d.r.q > 0) {
            int32_t* row = st.tables + static_cast<int64_t>(s) * st.max_blocks;
            int j = off;
            if (d.cow) {
                const int nb = alloc[j++];
                row[d.r.n0 / kBlockSize] = nb;
                st.refs[nb] = 1;
                cow_src[coff] = d.r.b;
                cow_dst[coff] = nb;
            }
            for (int li = blocks_for(d.r.n0); li < blocks_for(d.r.n0 + d.r.q); ++li) {
                const int nb = alloc[j++];
                row[li] = nb;
                st.refs[nb] = 1;
            }
            if (d.settles) {
                st.refs[d.r.b] -= d.copies;
                cnt[d.r.b] = 0;
                last[d.r.b] = 0;
            }
        }
    }
    __syncthreads();
    // D: slots of the new tokens through the final tables, then the lengths,
    // the ring and the unused pair entries.
    for (int t = tid; t < T; t += kBmThreads) {
        int lo = 0, hi = S - 1;  // the last s with qsl[s] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (qsl[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int pos = st.lens[lo] + (t - qsl[lo]);
        slots[t] = st.tables[static_cast<int64_t>(lo) * st.max_blocks + pos / kBlockSize] * kBlockSize +
                   pos % kBlockSize;
    }
    for (int s = cow_total + tid; s < S; s += kBmThreads) cow_src[s] = cow_dst[s] = -1;
    // The taken blocks leave the free queue; a cached one loses its key (its
    // content is about to be overwritten).
    for (int j = tid; j < need_total; j += kBmThreads) st.ring_pos[alloc[j]] = -1;
    if (tid == 0 && st.key_table != nullptr)
        for (int j = 0; j < need_total; ++j)
            if (st.cached[alloc[j]]) {
                table_erase(st, alloc[j]);
                st.cached[alloc[j]] = 0;
            }
    __syncthreads();
    for (int s = tid; s < S; s += kBmThreads) st.lens[s] += qsl[s + 1] - qsl[s];
    if (tid == 0) {
        st.free_state[0] = ring_cap(st) > 0 ? (head + consumed) % ring_cap(st) : 0;
        st.free_state[1] = entries - consumed;
        st.free_state[2] = nfree - need_total;
        *cow_count = cow_total;
    }
}

__global__ void __launch_bounds__(256) blocks_reset_kernel(const BlocksArgs st) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t ntab = static_cast<int64_t>(st.max_seqs) * st.max_blocks;
    for (int64_t i = first; i < ntab; i += stride) st.tables[i] = -1;
    for (int64_t i = first; i < st.max_seqs; i += stride) st.lens[i] = 0;
    for (int64_t i = first; i < st.num_blocks; i += stride) {
        st.refs[i] = 0;
        st.free_ring[i] = static_cast<int32_t>(i);
        st.free_ring[st.num_blocks + i] = -1;
        st.ring_pos[i] = static_cast<int32_t>(i);
        st.scratch[i] = 0;
        st.scratch[st.num_blocks + i] = 0;
        if (st.cached != nullptr) st.cached[i] = 0;
    }
    if (st.key_table != nullptr)
        for (int64_t i = first; i < st.table_size; i += stride) st.key_table[i] = -1;
    if (first == 0) {
        st.free_state[0] = 0;
        st.free_state[1] = st.num_blocks;
        st.free_state[2] = st.num_blocks;
    }
}

// Whether row r's first blocks_for(len) entries are held blocks.
__device__ __forceinline__ bool row_blocks_held(const BlocksArgs& st, int r, int len) {
    const int32_t* row = st.tables + static_cast<int64_t>(r) * st.max_blocks;
    for (int li = 0; li < blocks_for(len); ++li) {
        const int b = row[li];
        if (b < 0 || b >= st.num_blocks || st.refs[b] <= 0) return false;
    }
    return true;
}

// children[i] takes parents[i]'s blocks (and length); each block gains a
// holder.  Rows are checked in the order: in range, then children distinct
// and not parents, then children empty and parents' blocks held.
__global__ void __launch_bounds__(kBmThreads, 1)
    blocks_fork_kernel(const BlocksArgs st, const int32_t* __restrict__ parents,
                       const int32_t* __restrict__ children, int32_t n, unsigned long long* err) {
    __shared__ int sp[kBlocksMaxRows], sc[kBlocksMaxRows];
    griddep_launch_dependents();
    griddep_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cap = st.max_blocks * kBlockSize;
    int bad = 0;
    for (int i = tid; i < n; i += kBmThreads) {
        sp[i] = parents[i];
        sc[i] = children[i];
        if (sp[i] < 0 || sp[i] >= st.max_seqs || sc[i] < 0 || sc[i] >= st.max_seqs) bad = 1;
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) record_error(err, kErrRange, 0u);
        return;
    }
    int alias = 0;
    for (int i = tid; i < n; i += kBmThreads)
        for (int k = 0; k < n; ++k)
            if ((k != i && sc[k] == sc[i]) || sp[k] == sc[i]) alias = 1;
    if (__syncthreads_or(alias)) {
        if (tid == 0) record_error(err, kErrAlias, 0u);
        return;
    }
    for (int i = tid; i < n; i += kBmThreads) {
        const int len = st.lens[sp[i]];
        if (st.lens[sc[i]] != 0 || len < 0 || len > cap || !row_blocks_held(st, sp[i], len)) bad = 1;
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) record_error(err, kErrRange, 0u);
        return;
    }
    for (int i = warp; i < n; i += kBmThreads / 32) {
        const int len = st.lens[sp[i]];
        const int32_t* src = st.tables + static_cast<int64_t>(sp[i]) * st.max_blocks;
        int32_t* dst = st.tables + static_cast<int64_t>(sc[i]) * st.max_blocks;
        for (int li = lane; li < blocks_for(len); li += 32) {
            const int b = src[li];
            dst[li] = b;
            atomicAdd(&st.refs[b], 1);
        }
        if (lane == 0) st.lens[sc[i]] = len;
    }
}

// Rows drop their blocks: in the given row order, each row's blocks last
// first.  Reference g enumerates that order; the reference that takes a
// block's count to 0 is the block's last one (highest g) when every holder
// of the block is released here, and the freed blocks join the ring's tail in
// g order.
__global__ void __launch_bounds__(kBmThreads, 1)
    blocks_release_kernel(const BlocksArgs st, const int32_t* __restrict__ rows, int32_t n,
                          unsigned long long* err) {
    __shared__ int srow[kBlocksMaxRows];
    __shared__ int sbase[kBlocksMaxRows + 1];
    __shared__ int wsum[33];
    griddep_launch_dependents();
    griddep_wait();
    const int tid = threadIdx.x;
    const int len_cap = st.max_blocks * kBlockSize;
    int32_t* cnt = st.scratch;
    int32_t* last = st.scratch + st.num_blocks;
    int bad = 0;
    for (int i = tid; i < n; i += kBmThreads) {
        srow[i] = rows[i];
        if (srow[i] < 0 || srow[i] >= st.max_seqs) bad = 1;
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) record_error(err, kErrRange, 0u);
        return;
    }
    int alias = 0;
    for (int i = tid; i < n; i += kBmThreads)
        for (int k = 0; k < i; ++k)
            if (srow[k] == srow[i]) alias = 1;
    if (__syncthreads_or(alias)) {
        if (tid == 0) record_error(err, kErrAlias, 0u);
        return;
    }
    // Per-row block counts -> offsets of each row's references.
    int G = 0;
    for (int base = 0; base < n; base += kBmThreads) {
        const int i = base + tid;
        int nb = 0;
        if (i < n) {
            const int len = st.lens[srow[i]];
            if (len < 0 || len > len_cap || !row_blocks_held(st, srow[i], len)) bad = 1;
            else nb = blocks_for(len);
        }
        int t;
        const int off = G + cta_exclusive_scan(nb, wsum, &t);
        if (i < n) sbase[i] = off;
        G += t;
    }
    if (tid == 0) sbase[n] = G;
    if (__syncthreads_or(bad)) {
        if (tid == 0) record_error(err, kErrRange, 0u);
        return;
    }
    // Reference g -> (row i, logical block li, physical block b).
    auto ref_at = [&](int g, int& i, int& li) {
        int lo = 0, hi = n - 1;  // the last i with sbase[i] <= g
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sbase[mid] <= g) lo = mid; else hi = mid - 1;
        }
        i = lo;
        li = (sbase[i + 1] - sbase[i]) - 1 - (g - sbase[i]);
        return st.tables[static_cast<int64_t>(srow[i]) * st.max_blocks + li];
    };
    for (int g = tid; g < G; g += kBmThreads) {
        int i, li;
        const int b = ref_at(g, i, li);
        atomicAdd(&cnt[b], 1);
        atomicMax(&last[b], g);
    }
    __syncthreads();
    for (int g = tid; g < G; g += kBmThreads) {
        int i, li;
        const int b = ref_at(g, i, li);
        if (cnt[b] > st.refs[b]) bad = 1;  // more holders released than hold it
    }
    if (__syncthreads_or(bad)) {
        for (int g = tid; g < G; g += kBmThreads) {
            int i, li;
            const int b = ref_at(g, i, li);
            cnt[b] = 0;
            last[b] = 0;
        }
        if (tid == 0) record_error(err, kErrRange, 0u);
        return;
    }
    const int head = st.free_state[0];
    int entries = st.free_state[1];
    const int nfree = st.free_state[2];
    if (!ring_ok(st, head, entries, nfree)) {  // (G > 0 implies num_blocks > 0)
        for (int g = tid; g < G; g += kBmThreads) {
            int i, li;
            const int b = ref_at(g, i, li);
            cnt[b] = 0;
            last[b] = 0;
        }
        if (tid == 0) record_error(err, kErrRange, 0u);
        return;
    }
    const int cap = ring_cap(st);
    auto frees = [&](int g, int& b) {
        int i, li;
        b = ref_at(g, i, li);
        return g == last[b] && cnt[b] == st.refs[b];
    };
    int freed = 0;
    for (int base = 0; base < G; base += kBmThreads) {
        const int g = base + tid;
        int b, flag = 0;
        if (g < G) flag = frees(g, b) ? 1 : 0;
        freed += __syncthreads_count(flag);
    }
    // The ring holds 2 * num_blocks entries; when the freed blocks would not
    // fit after the stale entries, drop those first, keeping the live ones in
    // order (a window is read before it is written, and every write goes to
    // an index no later than the one it came from).
    if (entries + freed > cap) {
        int kept = 0;
        for (int base = 0; base < entries; base += kBmThreads) {
            const int e = base + tid;
            int b = -1, live = 0;
            if (e < entries) {
                const int idx = (head + e) % cap;
                b = st.free_ring[idx];
                live = ring_live(st, idx, b) ? 1 : 0;
            }
            int t;
            const int rank = cta_exclusive_scan(live, wsum, &t);
            if (live) {
                const int to = (head + kept + rank) % cap;
                st.free_ring[to] = b;
                st.ring_pos[b] = to;
            }
            kept += t;
            __syncthreads();
        }
        entries = kept;
    }
    int pushed = 0;
    for (int base = 0; base < G; base += kBmThreads) {
        const int g = base + tid;
        int b = -1, flag = 0;
        if (g < G) flag = frees(g, b) ? 1 : 0;
        int t;
        const int off = pushed + cta_exclusive_scan(flag, wsum, &t);
        if (flag) {
            const int to = (head + entries + off) % cap;
            st.free_ring[to] = b;
            st.ring_pos[b] = to;
        }
        pushed += t;
    }
    __syncthreads();
    for (int g = tid; g < G; g += kBmThreads) {
        int i, li;
        const int b = ref_at(g, i, li);
        if (g == last[b]) st.refs[b] -= cnt[b];
    }
    __syncthreads();
    for (int g = tid; g < G; g += kBmThreads) {
        int i, li;
        const int b = ref_at(g, i, li);
        cnt[b] = 0;
        last[b] = 0;
        st.tables[static_cast<int64_t>(srow[i]) * st.max_blocks + li] = -1;
    }
    __syncthreads();
    for (int i = tid; i < n; i += kBmThreads) st.lens[srow[i]] = 0;
    if (tid == 0) {
        st.free_state[1] = entries + freed;
        st.free_state[2] = nfree + freed;
    }
}

// Rows s with num_keys[s] > 0 (each empty) take the cached blocks of their
// leading keys, up to the first key that is not cached; a block with no
// holder leaves the free queue.  matched[s] gets the number taken.
__global__ void __launch_bounds__(kBmThreads, 1)
    blocks_match_kernel(const BlocksArgs st, const uint8_t* __restrict__ keys, int32_t key_stride,
                        const int32_t* __restrict__ num_keys, int32_t S, int32_t* __restrict__ matched,
                        unsigned long long* err) {
    __shared__ int sbase[kBlocksMaxRows + 1];
    __shared__ int wsum[33];
    griddep_launch_dependents();
    griddep_wait();
    const int tid = threadIdx.x;
    int bad = 0;
    // Per-row key counts -> offsets of the (row, key) pairs.
    int G = 0;
    for (int base = 0; base < S; base += kBmThreads) {
        const int s = base + tid;
        int n = 0;
        if (s < S) {
            n = num_keys[s];
            if (n < 0 || n > st.max_blocks || n > key_stride || (n > 0 && st.lens[s] != 0)) {
                bad = 1;
                n = 0;
            }
            matched[s] = n;  // lowered to the first miss below
        }
        int t;
        const int off = G + cta_exclusive_scan(n, wsum, &t);
        if (s < S) sbase[s] = off;
        G += t;
    }
    if (tid == 0) sbase[S] = G;
    if (__syncthreads_or(bad)) {
        if (tid == 0) record_error(err, kErrRange, 0u);
        return;
    }
    auto pair_at = [&](int g, int& s, int& i) {
        int lo = 0, hi = S - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sbase[mid] <= g) lo = mid; else hi = mid - 1;
        }
        s = lo;
        i = g - sbase[s];
        return keys + (static_cast<int64_t>(s) * key_stride + i) * 32;
    };
    for (int g = tid; g < G; g += kBmThreads) {
        int s, i;
        if (table_find(st, pair_at(g, s, i)) < 0) atomicMin(&matched[s], i);
    }
    __syncthreads();
    for (int g = tid; g < G; g += kBmThreads) {
        int s, i;
        const uint8_t* key = pair_at(g, s, i);
        if (i >= matched[s]) continue;
        const int b = table_find(st, key);
        st.tables[static_cast<int64_t>(s) * st.max_blocks + i] = b;
        if (atomicAdd(&st.refs[b], 1) == 0) {  // it was free: it leaves the queue
            st.ring_pos[b] = -1;
            atomicSub(&st.free_state[2], 1);
        }
    }
    for (int s = tid; s < S; s += kBmThreads)
        if (num_keys[s] > 0) st.lens[s] = matched[s] * kBlockSize;
}

// The full blocks of rows s < S get their keys, with the result of doing it
// in (row, block) order: a block that already has a key keeps it, a block
// listed twice counts once, and a key already cached, or given to an earlier
// (row, block) of the call, keeps its block.  In parallel: every new key is
// inserted into an empty slot of its probe sequence (atomicCAS), then every
// inserted candidate scans its probe run for entries with an equal key and
// keeps its entry only if it is the earliest of them; the few losers (equal
// prompts computed in the same step) are removed one at a time.
__global__ void __launch_bounds__(kBmThreads, 1)
    blocks_register_kernel(const BlocksArgs st, const uint8_t* __restrict__ keys, int32_t key_stride,
                           const int32_t* __restrict__ num_keys, int32_t S, unsigned long long* err) {
    __shared__ int sbase[kBlocksMaxRows + 1];
    __shared__ int wsum[33];
    __shared__ int s_losers;
    griddep_launch_dependents();
    griddep_wait();
    const int tid = threadIdx.x;
    const int mask = st.table_size - 1;
    int32_t* first = st.scratch;                      // per block: G - (its first candidate), 0 = none
    int32_t* mark = st.scratch + st.num_blocks;       // per block: 1 = its key goes into the table now
    int32_t* losers = st.scratch + 2 * st.num_blocks; // blocks whose entry is removed again
    int bad = 0, G = 0;
    for (int base = 0; base < S; base += kBmThreads) {
        const int s = base + tid;
        int n = 0;
        if (s < S) {
            n = num_keys[s];
            if (n < 0 || n > key_stride || st.lens[s] < 0 || n > st.lens[s] / kBlockSize ||
                st.lens[s] > st.max_blocks * kBlockSize) {
                bad = 1;
                n = 0;
            }
            for (int i = 0; i < n; ++i) {
                const int b = st.tables[static_cast<int64_t>(s) * st.max_blocks + i];
                if (b < 0 || b >= st.num_blocks || st.refs[b] <= 0) bad = 1;
            }
        }
        int t;
        const int off = G + cta_exclusive_scan(n, wsum, &t);
        if (s < S) sbase[s] = off;
        G += t;
    }
    if (tid == 0) {
        sbase[S] = G;
        s_losers = 0;
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) record_error(err, kErrRange, 0u);
        return;
    }
    auto cand = [&](int g, int& b) {
        int lo = 0, hi = S - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sbase[mid] <= g) lo = mid; else hi = mid - 1;
        }
        const int i = g - sbase[lo];
        b = st.tables[static_cast<int64_t>(lo) * st.max_blocks + i];
        return keys + (static_cast<int64_t>(lo) * key_stride + i) * 32;
    };
    // A: the first candidate of each block that has no key yet.
    for (int g = tid; g < G; g += kBmThreads) {
        int b;
        cand(g, b);
        if (!st.cached[b]) atomicMax(&first[b], G - g);
    }
    __syncthreads();
    // B: of those, the ones whose key is not cached yet write it.
    for (int g = tid; g < G; g += kBmThreads) {
        int b;
        const uint8_t* key = cand(g, b);
        if (st.cached[b] || first[b] != G - g || table_find(st, key) >= 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(st.block_keys + static_cast<int64_t>(b) * 32);
        dst[0] = reinterpret_cast<const uint4*>(key)[0];
        dst[1] = reinterpret_cast<const uint4*>(key)[1];
        mark[b] = 1;
    }
    __syncthreads();
    // C: insert them.  (A table of >= 2 * num_blocks slots never fills.)
    for (int g = tid; g < G; g += kBmThreads) {
        int b;
        cand(g, b);
        if (!mark[b] || first[b] != G - g) continue;
        int slot = key_home(st, st.block_keys + static_cast<int64_t>(b) * 32);
        for (int n = 0; n < st.table_size; ++n) {
            if (st.key_table[slot] == -1 && atomicCAS(&st.key_table[slot], -1, b) == -1) break;
            slot = (slot + 1) & mask;
        }
    }
    __syncthreads();
    // D: among entries with equal keys inserted here, the earliest stays.
    for (int g = tid; g < G; g += kBmThreads) {
        int b;
        cand(g, b);
        if (!mark[b] || first[b] != G - g) continue;
        const uint8_t* key = st.block_keys + static_cast<int64_t>(b) * 32;
        int slot = key_home(st, key), earliest = g;
        for (int n = 0; n < st.table_size; ++n) {
            const int v = st.key_table[slot];
            if (v < 0) break;
            if (v != b && mark[v] && key_equal(st.block_keys + static_cast<int64_t>(v) * 32, key))
                earliest = min(earliest, G - first[v]);
            slot = (slot + 1) & mask;
        }
        if (earliest == g) st.cached[b] = 1;
        else losers[atomicAdd(&s_losers, 1)] = b;
    }
    __syncthreads();
    if (tid == 0)
        for (int k = 0; k < s_losers; ++k) table_erase(st, losers[k]);
    __syncthreads();
    for (int g = tid; g < G; g += kBmThreads) {
        int b;
        cand(g, b);
        first[b] = 0;
        mark[b] = 0;
    }
}

}  // namespace

cudaError_t launch_blocks_match(const BlocksArgs& st, const uint8_t* keys, int32_t key_stride,
                                const int32_t* num_keys, int32_t num_seqs, int32_t* matched,
                                unsigned long long* err, cudaStream_t stream) {
    return launch_overlapped(blocks_match_kernel, dim3(1), dim3(kBmThreads), 0, stream, st, keys, key_stride,
                             num_keys, num_seqs, matched, err);
}

cudaError_t launch_blocks_register(const BlocksArgs& st, const uint8_t* keys, int32_t key_stride,
                                   const int32_t* num_keys, int32_t num_seqs, unsigned long long* err,
                                   cudaStream_t stream) {
    return launch_overlapped(blocks_register_kernel, dim3(1), dim3(kBmThreads), 0, stream, st, keys, key_stride,
                             num_keys, num_seqs, err);
}

cudaError_t launch_blocks_reset(const BlocksArgs& st, cudaStream_t stream) {
    const int64_t work = std::max<int64_t>(std::max<int64_t>(static_cast<int64_t>(st.max_seqs) * st.max_blocks,
                                                             st.num_blocks),
                                           st.table_size);
    const int64_t blocks = std::min<int64_t>(std::max<int64_t>((work + 255) / 256, 1), 1024);
    return launch_overlapped(blocks_reset_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, st);
}

cudaError_t launch_blocks_append(const BlocksArgs& st, const int32_t* query_start_loc, int32_t num_seqs,
                                 int32_t num_tokens, int32_t* slot_mapping, int32_t* cow_src, int32_t* cow_dst,
                                 int32_t* cow_count, unsigned long long* err, cudaStream_t stream) {
    return launch_overlapped(blocks_append_kernel, dim3(1), dim3(kBmThreads), 0, stream, st, query_start_loc,
                             num_seqs, num_tokens, slot_mapping, cow_src, cow_dst, cow_count, err);
}

cudaError_t launch_blocks_fork(const BlocksArgs& st, const int32_t* parents, const int32_t* children, int32_t n,
                               unsigned long long* err, cudaStream_t stream) {
    return launch_overlapped(blocks_fork_kernel, dim3(1), dim3(kBmThreads), 0, stream, st, parents, children, n,
                             err);
}

cudaError_t launch_blocks_release(const BlocksArgs& st, const int32_t* rows, int32_t n, unsigned long long* err,
                                  cudaStream_t stream) {
    return launch_overlapped(blocks_release_kernel, dim3(1), dim3(kBmThreads), 0, stream, st, rows, n, err);
}

}  // namespace pkv
