// prefix_cache.cu -- prefix-cache block keys on the device.
//
// "Prefix cache", section 4 of the serving-engine KV blog: every full block
// gets a key hashing the previous block's key, the block's token ids and
// extra information (adapter, multimodal hashes, a per-user cache salt).
// Since the previous key is part of it, a key stands for the whole prefix up
// to its block.  Only full blocks are keyed; the default hash is SHA-256.
//
// Message of block i of a sequence (104 bytes):
//   key_{i-1} (32 bytes) || 16 token ids (little-endian int32) || extra
//   (little-endian int64),
// key_{-1} = the caller's parent key or 32 zero bytes, key_i = SHA-256 of it.
// Keys depend on each other along a sequence, so one thread walks one
// sequence's chain; sequences run in parallel.
//
// SHA-256 is written from its published definition (FIPS 180-4): the
// message is padded with a 1 bit, zeros and the 64-bit big-endian bit length
// to a multiple of 512 bits (104 bytes -> two 64-byte blocks), and each
// block goes through the compression function (message schedule of 64
// words, 64 rounds) that updates the eight state words.
#include <cuda_runtime.h>

#include <cstdint>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

// First 32 bits of the fractional parts of the cube roots of the first 64
// primes (the round constants) and of the square roots of the first 8
// primes (the initial state), as the standard defines them.
__constant__ uint32_t kRound[64] = {
    0x428a2f98, 0x71374491, 0xb5c0fbcf, 0xe9b5dba5, 0x3956c25b, 0x59f111f1, 0x923f82a4, 0xab1c5ed5,
    0xd807aa98, 0x12835b01, 0x243185be, 0x550c7dc3, 0x72be5d74, 0x80deb1fe, 0x9bdc06a7, 0xc19bf174,
    0xe49b69c1, 0xefbe4786, 0x0fc19dc6, 0x240ca1cc, 0x2de92c6f, 0x4a7484aa, 0x5cb0a9dc, 0x76f988da,
    0x983e5152, 0xa831c66d, 0xb00327c8, 0xbf597fc7, 0xc6e00bf3, 0xd5a79147, 0x06ca6351, 0x14292967,
    0x27b70a85, 0x2e1b2138, 0x4d2c6dfc, 0x53380d13, 0x650a7354, 0x766a0abb, 0x81c2c92e, 0x92722c85,
    0xa2bfe8a1, 0xa81a664b, 0xc24b8b70, 0xc76c51a3, 0xd192e819, 0xd6990624, 0xf40e3585, 0x106aa070,
    0x19a4c116, 0x1e376c08, 0x2748774c, 0x34b0bcb5, 0x391c0cb3, 0x4ed8aa4a, 0x5b9cca4f, 0x682e6ff3,
    0x748f82ee, 0x78a5636f, 0x84c87814, 0x8cc70208, 0x90befffa, 0xa4506ceb, 0xbef9a3f7, 0xc67178f2};
__constant__ uint32_t kInit[8] = {0x6a09e667, 0xbb67ae85, 0x3c6ef372, 0xa54ff53a,
                                  0x510e527f, 0x9b05688c, 0x1f83d9ab, 0x5be0cd19};

__device__ __forceinline__ uint32_t rotr(uint32_t x, int n) { return __funnelshift_r(x, x, n); }
__device__ __forceinline__ uint32_t bswap(uint32_t x) { return __byte_perm(x, 0, 0x0123); }

// One 64-byte block (16 big-endian words in w, overwritten by the schedule).
__device__ __forceinline__ void sha256_compress(uint32_t (&h)[8], uint32_t (&w)[16]) {
    uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], k = h[7];
#pragma unroll
    for (int t = 0; t < 64; ++t) {
        if (t >= 16) {
            const uint32_t w15 = w[(t - 15) & 15], w2 = w[(t - 2) & 15];
            const uint32_t s0 = rotr(w15, 7) ^ rotr(w15, 18) ^ (w15 >> 3);
            const uint32_t s1 = rotr(w2, 17) ^ rotr(w2, 19) ^ (w2 >> 10);
            w[t & 15] += s0 + w[(t - 7) & 15] + s1;
        }
        const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
        const uint32_t ch = (e & f) ^ (~e & g);
        const uint32_t t1 = k + S1 + ch + kRound[t] + w[t & 15];
        const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
        const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
        k = g;
        g = f;
        f = e;
        e = d + t1;
        d = c;
        c = b;
        b = a;
        a = t1 + S0 + maj;
    }
    h[0] += a; h[1] += b; h[2] += c; h[3] += d;
    h[4] += e; h[5] += f; h[6] += g; h[7] += k;
}

__global__ void __launch_bounds__(64)
    prefix_keys_kernel(const int32_t* __restrict__ tokens, const int32_t* __restrict__ start,
                       const int64_t* __restrict__ extra, const uint8_t* __restrict__ parents, int32_t S,
                       int32_t max_blocks, uint8_t* __restrict__ keys, unsigned long long* err) {
    griddep_launch_dependents();
    griddep_wait();
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= S) return;
    const int t0 = start[s], t1 = start[s + 1];
    if (t0 < 0 || t1 < t0 || (t1 - t0) / kBlockSize > max_blocks) {
        record_error(err, kErrRange, static_cast<uint32_t>(s));
        return;
    }
    const int nfull = (t1 - t0) / kBlockSize;
    uint32_t prev[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (parents != nullptr) {
        const uint32_t* p = reinterpret_cast<const uint32_t*>(parents + static_cast<int64_t>(s) * 32);
#pragma unroll
        for (int k = 0; k < 8; ++k) prev[k] = bswap(p[k]);  // digest bytes are the big-endian state words
    }
    const uint64_t x = extra != nullptr ? static_cast<uint64_t>(extra[s]) : 0ull;
    uint4* out = reinterpret_cast<uint4*>(keys + static_cast<int64_t>(s) * max_blocks * 32);
    for (int i = 0; i < nfull; ++i) {
        const int32_t* tk = tokens + t0 + i * kBlockSize;
        uint32_t h[8], w[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) h[k] = kInit[k];
        // Block 1: parent key, tokens 0-7.
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = prev[k];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[8 + k] = bswap(static_cast<uint32_t>(tk[k]));
        sha256_compress(h, w);
        // Block 2: tokens 8-15, extra, the 1 bit, zeros, length 104*8 bits.
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = bswap(static_cast<uint32_t>(tk[8 + k]));
        w[8] = bswap(static_cast<uint32_t>(x));
        w[9] = bswap(static_cast<uint32_t>(x >> 32));
        w[10] = 0x80000000u;
        w[11] = w[12] = w[13] = w[14] = 0u;
        w[15] = 104u * 8u;
        sha256_compress(h, w);
        out[2 * i] = make_uint4(bswap(h[0]), bswap(h[1]), bswap(h[2]), bswap(h[3]));
        out[2 * i + 1] = make_uint4(bswap(h[4]), bswap(h[5]), bswap(h[6]), bswap(h[7]));
#pragma unroll
        for (int k = 0; k < 8; ++k) prev[k] = h[k];
    }
}

}  // namespace

cudaError_t launch_prefix_keys(const int32_t* token_ids, const int32_t* token_start_loc, const int64_t* extra,
                               const uint8_t* parent_keys, int32_t num_seqs, int32_t max_blocks, uint8_t* keys,
                               unsigned long long* err, cudaStream_t stream) {
    const int threads = 64;
    const int blocks = (num_seqs + threads - 1) / threads;
    return launch_overlapped(prefix_keys_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                             token_ids, token_start_loc, extra, parent_keys, num_seqs, max_blocks, keys, err);
}

}  // namespace pkv
