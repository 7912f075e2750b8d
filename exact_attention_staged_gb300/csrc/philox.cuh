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

constexpr int kPhiloxRounds = 10;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u, kPhiloxW1 = 0xBB67AE85u;  // key increments

struct DropSpec {
    uint32_t t4;        // threshold t in each byte (t * 0x01010101); 0: no dropout
    float keep_scale;   // 256 / (256 - t)
    uint64_t seed;      // key
    uint64_t offset;    // counter word 3 (below 2^32)
    // the key of every round, (k0, k1) = (seed mod 2^32 + r W0, seed div 2^32 + r W1) mod 2^32:
    // the same for every counter, so they are worked out once on the host and read from the
    // kernel's parameter block
    uint32_t round_key[kPhiloxRounds][2];
};

// Fill in the round keys of ds.seed.
__host__ __device__ inline void philox_round_keys(DropSpec &ds) {
    uint32_t k0 = static_cast<uint32_t>(ds.seed), k1 = static_cast<uint32_t>(ds.seed >> 32);
    for (int r = 0; r < kPhiloxRounds; ++r) {
        ds.round_key[r][0] = k0;
        ds.round_key[r][1] = k1;
        k0 += kPhiloxW0;
        k1 += kPhiloxW1;
    }
}

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

// The eight output words of the two generator blocks with counters (2 kb, q, bh, offset) and
// (2 kb + 1, q, bh, offset), run interleaved: their bytes decide the 32 scores
// k = 32 kb .. 32 kb + 31 of query row q (byte k mod 32 of the 32).  kHostKeys: read each round's
// key from ds.round_key (fewer instructions), else advance the key in registers (fewer registers
// held: the dK/dV compute warps run at 96 per thread).
template <bool kHostKeys>
__device__ __forceinline__ void philox_pair(uint64_t kb, uint64_t q, uint64_t bh,
                                            const DropSpec &ds, uint32_t w[8]) {
    uint32_t a0 = static_cast<uint32_t>(2 * kb), a1 = static_cast<uint32_t>(q),
             a2 = static_cast<uint32_t>(bh), a3 = static_cast<uint32_t>(ds.offset);
    uint32_t b0 = a0 + 1, b1 = a1, b2 = a2, b3 = a3;
    uint32_t k0 = static_cast<uint32_t>(ds.seed), k1 = static_cast<uint32_t>(ds.seed >> 32);
#pragma unroll
    for (int r = 0; r < kPhiloxRounds; ++r) {
        if constexpr (kHostKeys) {
            k0 = ds.round_key[r][0];
            k1 = ds.round_key[r][1];
        }
        philox4x32_round(a0, a1, a2, a3, k0, k1);
        philox4x32_round(b0, b1, b2, b3, k0, k1);
        if constexpr (!kHostKeys) {
            k0 += kPhiloxW0;
            k1 += kPhiloxW1;
        }
    }
    w[0] = a0; w[1] = a1; w[2] = a2; w[3] = a3;
    w[4] = b0; w[5] = b1; w[6] = b2; w[7] = b3;
}

// Keep flags of the four bytes of `w`: the top bit of byte b is set when that byte is kept (the
// other bits carry no meaning).  A byte x is kept when x >= t, i.e. when the 8-bit sum
// x + (256 - t) carries out; the carries of all four bytes come from one add of the low seven
// bits of each byte (no carry crosses a byte) and a bitwise majority of the two top bits and
// that sum's top bit.  c4 = (256 - t) * 0x01010101 (t >= 1).  Three instructions.
__device__ __forceinline__ uint32_t keep_flags4(uint32_t w, uint32_t c4) {
    const uint32_t s7 = (w & 0x7F7F7F7Fu) + (c4 & 0x7F7F7F7Fu);
    uint32_t f;
    asm("lop3.b32 %0, %1, %2, %3, 0xE8;" : "=r"(f) : "r"(w), "r"(c4), "r"(s7));  // majority
    return f;
}
__device__ __forceinline__ uint32_t keep_c4(const DropSpec &ds) {
    return (256u - (ds.t4 & 0xFFu)) * 0x01010101u;
}

// Keep bits of the 32 scores k = 32 kb .. 32 kb + 31 of query row q: bit j set = key 32 kb + j
// is kept.
template <bool kHostKeys = true>
__device__ __forceinline__ uint32_t philox_keep_bits(uint64_t kb, uint64_t q, uint64_t bh,
                                                     const DropSpec &ds) {
    uint32_t w[8];
    philox_pair<kHostKeys>(kb, q, bh, ds, w);
    const uint32_t c4 = keep_c4(ds);
    uint32_t bits = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // bytes 4i .. 4i + 3 of the 32 (keys 32 kb + 4i ..)
        // the four top bits to bits 28..31 by a product whose other terms land on distinct
        // lower bits (no carries)
        bits |= (((keep_flags4(w[i], c4) & 0x80808080u) * 0x00204081u) >> 28) << (4 * i);
    }
    return bits;
}

// The same 32 decisions as keep flags: word i holds those of keys 32 kb + 4 i .. + 3, one per
// byte (keep_flags4).
__device__ __forceinline__ void philox_keep_flags(uint64_t kb, uint64_t q, uint64_t bh,
                                                  const DropSpec &ds, uint32_t flags[8]) {
    uint32_t w[8];
    philox_pair<true>(kb, q, bh, ds, w);
    const uint32_t c4 = keep_c4(ds);
#pragma unroll
    for (int i = 0; i < 8; ++i) flags[i] = keep_flags4(w[i], c4);
}

// Mask keeping the 16-bit halves of a packed pair whose keep flags are bytes `byte` and
// `byte` + 1 of `flags` (top bits): prmt copies each selected byte's top bit over its byte.
__device__ __forceinline__ uint32_t keep_pair_mask(uint32_t flags, int byte) {
    const uint32_t sel = (8u | byte) * 0x11u | ((8u | (byte + 1)) * 0x11u) << 8;
    uint32_t m;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(m) : "r"(flags), "r"(sel));
    return m;
}
// All-ones when the keep flag in byte `byte` of `flags` is set, else zero.
__device__ __forceinline__ uint32_t keep_elem_mask(uint32_t flags, int byte) {
    uint32_t m;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(m) : "r"(flags), "r"((8u | byte) * 0x1111u));
    return m;
}

// Transpose of the 32 x 32 bit matrix whose row l is `x` of lane l: returns, to lane r, the word
// whose bit c is bit r of lane c's `x`.  Five butterfly stages; at stage j, lanes l and l ^ j swap
// the j-bit blocks in which they differ (the lane with bit j clear gives its high blocks and takes
// its partner's low ones, shifted up).  Every lane of the warp calls it.
__device__ __forceinline__ uint32_t transpose32_bits(uint32_t x, int lane) {
    const uint32_t m[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
    for (int s = 0; s < 5; ++s) {
        const int j = 16 >> s;
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
        x = (lane & j) == 0 ? (x & m[s]) | ((y & m[s]) << j) : (x & ~m[s]) | ((y >> j) & m[s]);
    }
    return x;
}

}  // namespace fa
