// philox.cuh - the dropout decisions of the attention kernels.
//
// Generator: Philox4x64-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as
// 1, 2, 3", SC 2011): 256-bit counter, 128-bit key, ten rounds of two 64 x 64 -> 128-bit
// products with the key advanced by two Weyl constants between rounds.
// Decisions: score (q, k) of query head bh takes byte (k mod 32) of the 32 output bytes (four
// little-endian 64-bit words) for counter (k div 32, q, bh, 0) and key (seed, offset), and is
// dropped when that byte is below the threshold t (drop probability t / 256).
#pragma once

#include <cstdint>

namespace fa {

struct DropSpec {
    uint32_t t4;        // threshold t in each byte (t * 0x01010101); 0: no dropout
    float keep_scale;   // 256 / (256 - t)
    uint64_t seed, offset;
};

// Keep bits of the 32 scores k = 32 kb .. 32 kb + 31 of query row q: bit j set = key 32 kb + j
// is kept.
__device__ __forceinline__ uint32_t philox_keep_bits(uint64_t kb, uint64_t q, uint64_t bh,
                                                     const DropSpec &ds) {
    uint64_t c0 = kb, c1 = q, c2 = bh, c3 = 0;
    uint64_t k0 = ds.seed, k1 = ds.offset;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t lo0 = 0xD2E7470EE14C6C93ull * c0, hi0 = __umul64hi(0xD2E7470EE14C6C93ull, c0);
        const uint64_t lo1 = 0xCA5A826395121157ull * c2, hi1 = __umul64hi(0xCA5A826395121157ull, c2);
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
        k0 += 0x9E3779B97F4A7C15ull;
        k1 += 0xBB67AE8584CAA73Bull;
    }
    const uint64_t w[4] = {c0, c1, c2, c3};
    uint32_t bits = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // bytes 4i .. 4i + 3
        const uint32_t word = static_cast<uint32_t>(w[i >> 1] >> (32 * (i & 1)));
        // 0xFF in every byte at or above the threshold; one bit per byte gathered by a product
        // whose partial terms land on distinct bit positions (no carries)
        const uint32_t ge = __vcmpgeu4(word, ds.t4) & 0x01010101u;
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
