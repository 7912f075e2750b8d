// fa_internal.h - parameter blocks and launchers shared by the C-ABI shim and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "philox.cuh"
#include "sm100.cuh"

namespace fa {

constexpr int kTile = 128;  // query rows / key rows per tile, also the block-mask granularity

// Block-mask bits in shared memory.  A CTA walks one row (forward, dQ: its query tiles' key
// tiles) or one column (dK/dV: its key tile's query tiles) of the [T][T] byte mask, and every
// warp role re-scans it; read from global memory that is one dependent load per tile visited,
// and a column's bytes are T bytes apart, so each one is a round trip to L2.  The CTA copies its
// row or column once, 32 tiles per ballot, as bits; masks wider than kMaskSmemTiles tiles
// (N > 524288) are read from global memory as before.
constexpr int kMaskSmemTiles = 4096;
constexpr int kMaskSmemWords = kMaskSmemTiles / 32;

// Every warp of the CTA calls this (warp-uniform): bit i of bits[] = (src[i * stride] != 0) for
// i < T; warp w writes words w, w + warps, ...
__device__ __forceinline__ void mask_bits_load(uint32_t *bits, const uint8_t *src, long stride,
                                               int T) {
    const int warps = static_cast<int>(blockDim.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    for (int w = static_cast<int>(threadIdx.x >> 5); w < (T + 31) / 32; w += warps) {
        const int i = 32 * w + lane;
        const bool live = i < T && src[static_cast<long>(i) * stride] != 0;
        const uint32_t word = __ballot_sync(0xffffffffu, live);
        if (lane == 0) bits[w] = word;
    }
}
__device__ __forceinline__ bool mask_bit(const uint32_t *bits, int i) {
    return ((bits[i >> 5] >> (i & 31)) & 1u) != 0;
}

// Forward kernels (bf16/fp16 and e4m3 parameter blocks alike): is key tile j live for query tile
// qt?  rowbits: where the query tile's mask row is kept as bits in shared memory when the mask
// is at most kMaskSmemTiles wide; wider masks are read from global memory.
template <class Params>
__device__ __forceinline__ bool tile_live(const Params &p, const uint32_t *rowbits, int qt, int j) {
    if (qt >= p.T) return false;
    if (p.causal && j > qt) return false;
    if (p.mask == nullptr) return true;
    return p.T <= kMaskSmemTiles ? mask_bit(rowbits, j) : p.mask[qt * p.T + j] != 0;
}

// Test hook: OR `bit` into byte `idx` of the tile-visit log, atomically on the containing 32-bit
// word (the log is 4-byte aligned): the dQ and dK/dV passes of one backward call may run at the
// same time and mark neighbouring bytes.
__device__ __forceinline__ void visit_mark(uint8_t *log, size_t idx, uint32_t bit) {
    atomicOr(reinterpret_cast<unsigned int *>(log + (idx & ~static_cast<size_t>(3))),
             bit << (8 * (idx & 3)));
}

// CTA order: heads are taken in groups of `group` so that the tiles streamed by the CTAs that
// run at the same time (K/V of the forward, Q/dO of dK/dV, K/V of dQ) stay within a slice of
// L2; inside a group the work unit (query-tile pair or tile) advances slowest, longest first.
struct CtaOrder {
    int head;  // b * H + h
    int rank;  // 0 = the first (longest) work unit of the head
};
__host__ __device__ inline CtaOrder cta_order(unsigned cta, int BH, int units, int group) {
    // 32-bit arithmetic: the grid has fewer than 2^31 CTAs
    const unsigned per_group = static_cast<unsigned>(group) * static_cast<unsigned>(units);
    const unsigned g = cta / per_group;
    const unsigned r = cta - g * per_group;
    const int left = BH - static_cast<int>(g) * group;
    const unsigned heads = static_cast<unsigned>(left < group ? left : group);
    CtaOrder o;
    o.rank = static_cast<int>(r / heads);
    o.head = static_cast<int>(g) * group + static_cast<int>(r % heads);
    return o;
}

struct FwdParams {
    void *o;                  // [B,H,N,d] output
    float *lse;               // [B,H,N] output
    const uint8_t *mask;      // [T][T] or nullptr
    int BH, N, T;             // heads (B*H), sequence length, tiles per side
    int num_pairs;            // ceil(T / 2): query-tile pairs per head
    int head_group;           // heads per CTA-order group (see cta_order)
    int rep;                  // query heads per K/V head: K/V head of query head bh is bh / rep
    float scale_log2;         // scale * log2(e)
    int causal;
    DropSpec drop;            // dropout on the probabilities (drop.t4 == 0: none)
    Ctl ctl;
};

struct BwdParams {
    void *out0;               // dK (dK/dV kernel, [B,H_kv,N,d]) or dQ (dQ kernel, [B,H,N,d])
    void *out1;               // dV (dK/dV kernel) or unused
    const float *lse;         // [B,H,N]
    const float *delta;       // [B,H,N]
    const uint8_t *mask;      // [T][T] or nullptr
    int BH, N, T;             // query heads (B*H), sequence length, tiles per side
    int head_group;           // CTA-order group size (see cta_order)
    int rep;                  // query heads per K/V head
    // dK/dV only: the rep query heads of a K/V head are split over `splits` CTAs per key tile,
    // `chunk` heads each.  With splits == 1 the kernel writes dK, dV; otherwise each split
    // writes fp32 partial sums to part[(which * splits + split) * kv_elems + ...] (which: 0 dK,
    // 1 dV) and fa_bwd_group_reduce_kernel adds them up.
    int units;                // B * H_kv * splits: the "heads" of the dK/dV CTA order
    int splits, chunk;
    float *part;
    long kv_elems;            // B * H_kv * N * d
    float scale;              // softmax scale (dK and dQ carry it)
    float scale_log2;         // scale * log2(e)
    int causal;
    DropSpec drop;            // the forward's dropout (drop.t4 == 0: none)
    Ctl ctl;
};

// Forward on e4m3 inputs (see fa_fwd_fp8.cu): the FwdParams fields plus the value scales.
struct Fp8FwdParams {
    void *o;                  // [B,H,N,d] bf16 output
    float *lse;               // [B,H,N]
    const uint8_t *mask;      // [T][T] or nullptr
    int BH, N, T, num_pairs, head_group, rep;
    float scale_log2;         // softmax scale * descale_q * descale_k * log2(e)
    float descale_v;          // value of one V unit
    int causal;
    Ctl ctl;
};

struct Fp8Maps {
    CUtensorMap q, k;         // [B*H or B*H_kv, N, d] bytes, boxes d x 128 rows
    CUtensorMap vt;           // [B*H_kv, d, Np] bytes (V transposed), boxes 128 keys x d rows
    CUtensorMap o;            // [B*H, N, d] bf16 output, boxes 64 elements x 128 rows
};

// Decode: a few new query rows per sequence against a KV cache (see fa_decode.cu).
struct DecodeParams {
    const void *q;            // [B,H,Nq,d]
    const void *k, *v;        // [B,H_kv,Nk,d] cache
    void *o;                  // [B,H,Nq,d]
    float *lse;               // [B,H,Nq]
    const int *kv_len;        // [B] cache lengths, or nullptr for Nk
    float *part_o;            // splits > 1: [splits][B*H*Nq][d] unnormalised partial outputs
    float *part_ml;           //             [splits][B*H*Nq][2] running max (log2) and sum
    int B, H, Hkv, Nq, Nk;
    int rows;                 // (H / H_kv) * Nq: query rows that share one K/V head
    int row_groups;           // ceil(rows / 128): work units per K/V head and key range
    int splits, chunk;        // key ranges [s * chunk, (s + 1) * chunk), chunk a multiple of 128
    float scale_log2;         // scale * log2(e)
    int causal;               // new rows end-aligned with the cache
    Ctl ctl;
};

struct DecodeMaps {
    CUtensorMap q;            // [B*H*Nq, d] query rows (one z slice), boxes 64 elements x 128 rows
    CUtensorMap k, v;         // [B*H_kv, Nk, d] cache, boxes 64 elements x 128 keys
};

struct Maps {
    CUtensorMap q, k, v, dout;
    CUtensorMap out0, out1;   // outputs written by TMA: O (forward), dK and dV, or dQ
};

cudaError_t launch_fwd(const Maps &maps, const FwdParams &p, int d, bool bf16,
                       cudaStream_t stream);
// delta[row] = mul * rowsum(dout o o)
cudaError_t launch_bwd_preprocess(const void *o, const void *dout, float *delta, long rows,
                                  int d, bool bf16, float mul, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(const Maps &maps, const BwdParams &p, int d, bool bf16,
                            bool after_dq, cudaStream_t stream);
cudaError_t launch_bwd_dq(const Maps &maps, const BwdParams &p, int d, bool bf16,
                          cudaStream_t stream);
cudaError_t launch_decode(const DecodeMaps &maps, const DecodeParams &p, int d, bool bf16,
                          cudaStream_t stream);
cudaError_t launch_fp8_transpose_v(const uint8_t *v, uint8_t *vt, int BHkv, int N, int Np, int d,
                                   cudaStream_t stream);
cudaError_t launch_fwd_fp8(const Fp8Maps &maps, const Fp8FwdParams &p, int d,
                           cudaStream_t stream);
cudaError_t launch_bwd_group_reduce(const float *part, void *dk, void *dv, int splits,
                                    long kv_elems, bool bf16, cudaStream_t stream);

}  // namespace fa
