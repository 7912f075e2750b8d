// philox.cuh - the dropout decisions of the attention kernels.
//
// Generator: Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as
// 1, 2, 3", SC 2011): 128-bit counter of four 32-bit words, 64-bit key, ten rounds of two
// 32 x 32 -> 64-bit products (one wide multiply each) with the key advanced by two Weyl
// constants between rounds.
// Decisions: score (q, k) of query head bh takes byte (k mod 16) of the 16 output bytes (four
// little-endian 32-bit words) for counter (k div 16, q, bh, offset) and key (seed mod 2^32,
// seed div 2^32), and is dropped when that byte is below the threshold t (drop probability
// t / 256).  The offset is a 32-bit counter word.
#pragma once

#include <cstdint>

namespace fa {

struct DropSpec {
    uint32_t t4;        // threshold t in each byte (t * 0x01010101); 0: no dropout
    float keep_scale;   // 256 / (256 - t)
    uint64_t seed;      // key
    uint64_t offset;    // counter word 3 (below 2^32)
};

// One Philox4x32 round on counter (c0, c1, c2, c3) under round key (k0, k1).
__device__ __forceinline__ void philox4x32_round(uint32_t &c0, uint32_t &c1, uint32_t &c2,
                                                 uint32_t &c3, uint32_t k0, uint32_t k1) {
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c0;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c2;
    const uint32_t hi0 = static_cast<uint32_t>(p0 >> 32), lo0 = static_cast<uint32_t>(p0);
    const uint32_t hi1 = static_cast<uint32_t>(p1 >> 32), lo1 = static_cast<uint32_t>(p1);
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
}

// Keep bits of the 32 scores k = 32 kb .. 32 kb + 31 of query row q: bit j set = key 32 kb + j
// is kept.  The two generator blocks (counters 2 kb and 2 kb + 1) run interleaved, sharing the
// key schedule.
__device__ __forceinline__ uint32_t philox_keep_bits(uint64_t kb, uint64_t q, uint64_t bh,
                                                     const DropSpec &ds) {
    uint32_t a0 = static_cast<uint32_t>(2 * kb), a1 = static_cast<uint32_t>(q),
             a2 = static_cast<uint32_t>(bh), a3 = static_cast<uint32_t>(ds.offset);
    uint32_t b0 = a0 + 1, b1 = a1, b2 = a2, b3 = a3;
    uint32_t k0 = static_cast<uint32_t>(ds.seed), k1 = static_cast<uint32_t>(ds.seed >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        philox4x32_round(a0, a1, a2, a3, k0, k1);
        philox4x32_round(b0, b1, b2, b3, k0, k1);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    const uint32_t w[8] = {a0, a1, a2, a3, b0, b1, b2, b3};
    uint32_t bits = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // bytes 4i .. 4i + 3 of the 32 (keys 32 kb + 4i ..)
        // 0xFF in every byte at or above the threshold; one bit per byte gathered by a product
        // whose partial terms land on distinct bit positions (no carries)
        const uint32_t ge = __vcmpgeu4(w[i], ds.t4) & 0x01010101u;
        bits |= ((ge * 0x01020408u) >> 24) << (4 * i);
    }
    return bits;
}

// Zero the 16-bit halves of `w` (elements 2c and 2c + 1 of a row) whose keep bit is clear.
__device__ __forceinline__ uint32_t keep_halves(uint32_t w, uint32_t bits, int c) {
    const uint32_t lo = (bits >> (2 * c)) & 1u, hi = (bits >> (2 * c + 1)) & 1u;
    return w & ((lo * 0xFFFFu) | (hi * 0xFFFF0000u));
}

}  // namespace fa
