// fa_decode.cu - decode: a few new query rows per sequence against a KV cache, sm_103a.
//
// FlashAttention-2 reading notes, section on the KV cache: in the decode phase each step's
// query is 1 x d (a few rows here) against the N cached keys, so the product is a matrix-vector
// one and the kernel is bound by reading K and V from HBM, not by arithmetic.  The work is
// therefore split over the cache, not over queries: CTA (K/V head, key range, row group) runs
// the online softmax (running max m and sum l per row, FlashAttention-2 Algorithm 1) over its
// key range for every query row that reads this K/V head (all query heads of a grouped-query
// group, times the new rows), reading each cached K/V row once.  Key ranges are merged by the
// statistic merge of the FlashAttention paper detail, Technique 1 (m = max(m1, m2),
// l = e^(m1-m) l1 + e^(m2-m) l2, and the outputs weighted the same way).
//
// GB300 mapping: no tensor cores (one to sixteen rows per key: 4 to 64 FLOP per 16-bit K/V
// element pair, far below what would make the MMA pipe the limit); 128 threads per CTA, seven
// CTAs per SM at up to four rows (each CTA's tile loop is a chain of barriers and shuffles, so
// resident CTAs set the rate).  K and V tiles of 16 keys stream through a three-stage ring
// filled by TMA (one thread issues a tile's boxes; completion on the stage's mbarrier), in boxes
// of 64 elements x 16 keys with the 128-byte swizzle: 16-byte chunk c of key row r sits at
// chunk position c ^ (r mod 8), so the 16-byte reads of 8 consecutive key rows (phase A) and the
// 128-byte row reads (phase B) are free of bank conflicts without padding.  Per tile:
//   A   every warp takes a quarter of d, every lane one key and half of that quarter: partial
//       dot products of that key with all rows (query rows broadcast from shared memory, fp32,
//       pre-scaled by scale * log2 e), the two halves summed by one shuffle;
//   A2  warp w owns rows w, w+4, ...: sums the four quarters, masks, takes the tile max with
//       shuffles over 16 lanes, P = 2^(s - m), l = alpha l + sum P;
//   B   every thread owns two output columns of every row and a fixed share of the tile's keys
//       (key group): O_g = alpha O_g + P V over its keys, P read four keys per shared load, so
//       each V element and each probability is read from shared memory once per tile.
// The key groups' partial outputs share the row statistics (alpha is per row and tile), so they
// are summed once, after the last tile.  With one key range the CTA then writes O and LSE;
// otherwise it writes (m, l, unnormalised O) and fa_decode_combine_kernel merges the ranges in
// order (deterministic).
#include "fa_internal.h"

#include <cmath>
#include <type_traits>

namespace fa {
namespace {

constexpr int kThreads = 128;
constexpr int kKeys = 16;     // keys per shared-memory tile (lane = key and column half)
constexpr int kStages = 3;    // K/V tiles in the TMA ring (two in flight while one is used)

template <int D, int RPC>
struct DecLayout {
    static constexpr int kBoxBytes = kKeys * 128;                   // 64 elements x 16 keys
    static constexpr int kTileBytes = kKeys * D * 2;                // D / 64 boxes
    static constexpr int kKOff = 0;                                 // kStages tiles (1024-aligned)
    static constexpr int kVOff = kKOff + kStages * kTileBytes;      // kStages tiles
    static constexpr int kQOff = kVOff + kStages * kTileBytes;      // float [RPC][D]
    static constexpr int kPartOff = kQOff + RPC * D * 4;            // float [4][RPC][kKeys]
    static constexpr int kPOff = kPartOff + 4 * RPC * kKeys * 4;    // float [RPC][kKeys]
    static constexpr int kStatOff = kPOff + RPC * kKeys * 4;        // alpha, m, l [RPC] each
    static constexpr int kBarOff = (kStatOff + 3 * RPC * 4 + 7) / 8 * 8;  // full[kStages]
    static constexpr int kAbortOff = kBarOff + kStages * 8;
    static constexpr int kBytes = kAbortOff + 8;
    static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024 bytes
};

// Byte offset of the 16-byte chunk holding elements [8 c, 8 c + 8) of key row r in a tile of
// 128-byte-swizzled 64-element boxes.
__device__ __forceinline__ int swz_chunk(int r, int c) {
    return (c >> 3) * (kKeys * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

template <bool BF16>
using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;

// reductions over each 16-lane half of a warp (both halves hold the same 16 keys)
__device__ __forceinline__ float half_max(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float half_sum(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// RPC: query rows per CTA (1, 2, 4, 8 or 16), the smallest that holds a K/V head's rows.
template <int D, bool BF16, int RPC>
__global__ void __launch_bounds__(kThreads)
    fa_decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const DecodeParams p) {
    using L = DecLayout<D, RPC>;
    using T = elem_t<BF16>;
    constexpr int kPairs = D / 2;                 // column pairs of O
    constexpr int kRB = kThreads / kPairs;        // key groups in phase B (2 for d=128, 4 for 64)
    constexpr int kKeysB = kKeys / kRB;           // keys per group and tile (16 or 8)
    constexpr int kRowsB = (RPC + kRB - 1) / kRB; // rows per thread in the final merge and store
    static_assert(kKeysB % 4 == 0, "probabilities are read four keys at a time");
    static_assert(kRB * RPC * D * 4 <= L::kBarOff,
                  "the merge buffer reuses the K/V ring, the query rows and the partial dots");
    constexpr int kQuarter = D / 4;               // columns per warp in phase A
    constexpr int kHalf = kQuarter / 2;           // columns per lane in phase A (16 or 8)
    static_assert(kKeys == 16, "phase A maps a warp's lanes to 16 keys x 2 column halves");
    constexpr int kRowsA2 = (RPC + 3) / 4;        // rows per warp in phase A2
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kAbortOff);
    float *qs = reinterpret_cast<float *>(smem + L::kQOff);
    float *part = reinterpret_cast<float *>(smem + L::kPartOff);
    float *ps = reinterpret_cast<float *>(smem + L::kPOff);
    float *alpha_s = reinterpret_cast<float *>(smem + L::kStatOff);
    float *m_s = alpha_s + RPC;
    float *l_s = m_s + RPC;

    // block order: row group fastest, then key range, then K/V head (b * H_kv + g)
    unsigned bid = blockIdx.x;
    const int rg = static_cast<int>(bid % static_cast<unsigned>(p.row_groups));
    bid /= static_cast<unsigned>(p.row_groups);
    const int split = static_cast<int>(bid % static_cast<unsigned>(p.splits));
    const int kvh = static_cast<int>(bid / static_cast<unsigned>(p.splits));
    const int b = kvh / p.Hkv;
    const int r0 = rg * RPC;
    const int nrows = min(RPC, p.rows - r0);
    int len = p.kv_len != nullptr ? p.kv_len[b] : p.Nk;
    len = max(0, min(len, p.Nk));
    const int k_begin = split * p.chunk;
    const int k_end = min(k_begin + p.chunk, len);
    const int ntiles = k_end > k_begin ? (k_end - k_begin + kKeys - 1) / kKeys : 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kl = lane & (kKeys - 1), half = lane >> 4;  // phase A / A2: key, column half
    // CTA row r is group row r0 + r: query head kvh * rep + (r0 + r) / Nq, new row (r0 + r) % Nq,
    // i.e. global row ((b * H + h) * Nq + i) = kvh * rows + r0 + r
    const long grow0 = static_cast<long>(kvh) * p.rows + r0;
    if (tid == 0) {
        for (int s2 = 0; s2 < kStages; ++s2) mbar_init(&full[s2], 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    __syncthreads();
    // Thread 0 fills stage t % kStages with the K and V boxes of tile t (keys past the cache's
    // capacity read as zeros; keys past the range or the sequence length are masked in A2).
    auto load_tile = [&](int t) {
        if (tid != 0 || t >= ntiles) return;
        const int key0 = k_begin + kKeys * t;
        const int stage = t % kStages;
        mbar_arrive_expect_tx(&full[stage], 2 * L::kTileBytes);
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
            tma_load_3d(smem + L::kKOff + stage * L::kTileBytes + b * L::kBoxBytes, &tmk, b * 64,
                        key0, kvh, &full[stage]);
            tma_load_3d(smem + L::kVOff + stage * L::kTileBytes + b * L::kBoxBytes, &tmv, b * 64,
                        key0, kvh, &full[stage]);
        }
    };
#pragma unroll
    for (int t = 0; t < kStages - 1; ++t) load_tile(t);
    // the range merge queued after this grid may take its SM slots early (it waits for this
    // grid's completion before it reads a partial result)
    if (tid == 0) griddep_launch_dependents();

    const T *qrows = reinterpret_cast<const T *>(p.q) + static_cast<size_t>(grow0) * D;
    for (int i = tid; i < RPC * D; i += kThreads)
        qs[i] = i < nrows * D ? static_cast<float>(qrows[i]) * p.scale_log2 : 0.f;

    float m_run[kRowsA2], l_run[kRowsA2];
#pragma unroll
    for (int i = 0; i < kRowsA2; ++i) {
        m_run[i] = -INFINITY;
        l_run[i] = 0.f;
    }
    const int cp = tid % kPairs, rs = tid / kPairs;  // column pair; key group (phase B)
    float2 acc[RPC];  // this thread's two output columns of every row, over its key group
#pragma unroll
    for (int r = 0; r < RPC; ++r) acc[r] = make_float2(0.f, 0.f);

    int t = 0;
    for (; t < ntiles; ++t) {
        const int stage = t % kStages;
        // tile t has landed; every thread is done with tile t - 1, whose stage is refilled
        if (!mbar_wait(&full[stage], (t / kStages) & 1, p.ctl, abort_flag)) *abort_flag = 1;
        __syncthreads();
        if (*abort_flag) break;  // a wait ran out: every thread leaves the loop here
        load_tile(t + kStages - 1);

        {  // A: partial dots of key `kl` over columns [c0, c0 + D/8), c0 = warp * D/4 + half * D/8
            const uint8_t *ktile = smem + L::kKOff + stage * L::kTileBytes;
            const int c0 = warp * kQuarter + half * kHalf;
            float2 dot[RPC];  // even and odd columns summed apart (paired fp32 FMAs)
#pragma unroll
            for (int r = 0; r < RPC; ++r) dot[r] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c8 = 0; c8 < kHalf / 8; ++c8) {
                const uint4 kw =
                    *reinterpret_cast<const uint4 *>(ktile + swz_chunk(kl, (c0 >> 3) + c8));
                const float2 k0 = unpack2<BF16>(kw.x), k1 = unpack2<BF16>(kw.y),
                             k2 = unpack2<BF16>(kw.z), k3 = unpack2<BF16>(kw.w);
#pragma unroll
                for (int r = 0; r < RPC; ++r) {  // rows past nrows hold zeros
                    const float4 *qv =
                        reinterpret_cast<const float4 *>(qs + r * D + warp * kQuarter +
                                                         half * kHalf + c8 * 8);
                    const float4 a = qv[0], c = qv[1];
                    float2 d = dot[r];
                    d = ffma2(make_float2(a.x, a.y), k0, d);
                    d = ffma2(make_float2(a.z, a.w), k1, d);
                    d = ffma2(make_float2(c.x, c.y), k2, d);
                    d = ffma2(make_float2(c.z, c.w), k3, d);
                    dot[r] = d;
                }
            }
#pragma unroll
            for (int r = 0; r < RPC; ++r) {  // the two column halves of key kl summed
                float sp = dot[r].x + dot[r].y;
                sp += __shfl_xor_sync(0xffffffffu, sp, 16);
                if (half == 0) part[(warp * RPC + r) * kKeys + kl] = sp;
            }
        }
        __syncthreads();
        {  // A2: warp w owns rows w, w + 4, w + 8, w + 12
            const int key = k_begin + kKeys * t + kl;
#pragma unroll
            for (int i = 0; i < kRowsA2; ++i) {
                const int r = warp + 4 * i;
                if (r < nrows) {
                    const int gr = r0 + r;
                    const int last = p.causal ? len - p.Nq + gr % p.Nq : len - 1;
                    float s = part[r * kKeys + kl] + part[(RPC + r) * kKeys + kl] +
                              part[(2 * RPC + r) * kKeys + kl] +
                              part[(3 * RPC + r) * kKeys + kl];
                    if (key >= k_end || key > last) s = -INFINITY;
                    const float m_new = fmaxf(m_run[i], half_max(s));
                    float alpha = 1.f, pr = 0.f;
                    if (m_new != -INFINITY) {  // ex2(-inf) = 0 covers masked keys, first tile
                        alpha = ex2(m_run[i] - m_new);
                        pr = ex2(s - m_new);
                    }
                    l_run[i] = l_run[i] * alpha + half_sum(pr);
                    m_run[i] = m_new;
                    if (half == 0) ps[r * kKeys + kl] = pr;
                    if (lane == 0) alpha_s[r] = alpha;
                }
            }
        }
        __syncthreads();
        {  // B: O_g = alpha O_g + P V over this thread's key group, two columns, every row
            const uint8_t *vtile = smem + L::kVOff + stage * L::kTileBytes;
            const float *pg = ps + rs * kKeysB;
#pragma unroll
            for (int r = 0; r < RPC; ++r) {
                if (r < nrows) {
                    const float a = alpha_s[r];
                    acc[r] = fmul2(acc[r], make_float2(a, a));
                }
            }
#pragma unroll
            for (int k4 = 0; k4 < kKeysB; k4 += 4) {
                float2 vv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int key = rs * kKeysB + k4 + u;  // row of the tile
                    vv[u] = unpack2<BF16>(*reinterpret_cast<const uint32_t *>(
                        vtile + swz_chunk(key, cp >> 2) + (cp & 3) * 4));
                }
#pragma unroll
                for (int r = 0; r < RPC; ++r) {
                    if (r < nrows) {  // rows past nrows have no probabilities this tile
                        const float4 p4 = *reinterpret_cast<const float4 *>(pg + r * kKeys + k4);
                        float2 o = acc[r];
                        o = ffma2(make_float2(p4.x, p4.x), vv[0], o);
                        o = ffma2(make_float2(p4.y, p4.y), vv[1], o);
                        o = ffma2(make_float2(p4.z, p4.z), vv[2], o);
                        o = ffma2(make_float2(p4.w, p4.w), vv[3], o);
                        acc[r] = o;
                    }
                }
            }
        }
    }
    if (*abort_flag) {
        // let the copies still in flight land before shared memory is reused or released
        if (tid == 0)
            for (int u = t; u < min(ntiles, t + kStages - 1); ++u)
                drain_wait(&full[u % kStages], (u / kStages) & 1, p.ctl);
        __syncthreads();
        return;
    }

#pragma unroll
    for (int i = 0; i < kRowsA2; ++i) {
        const int r = warp + 4 * i;
        if (r < nrows && lane == 0) {
            m_s[r] = m_run[i];
            l_s[r] = l_run[i];
        }
    }
    __syncthreads();  // every thread is past its last read of the K/V ring
    // merge of the key groups: group g's partial output of row r at red[(g * RPC + r) * D]
    float *red = reinterpret_cast<float *>(smem);
#pragma unroll
    for (int r = 0; r < RPC; ++r)
        if (r < nrows) reinterpret_cast<float2 *>(red + (rs * RPC + r) * D)[cp] = acc[r];
    __syncthreads();
    const long total_rows = static_cast<long>(p.B) * p.H * p.Nq;
#pragma unroll
    for (int j = 0; j < kRowsB; ++j) {
        const int r = rs + kRB * j;
        if (r >= nrows) continue;
        float2 o = make_float2(0.f, 0.f);
#pragma unroll
        for (int g = 0; g < kRB; ++g) {  // fixed order: deterministic
            const float2 x = reinterpret_cast<const float2 *>(red + (g * RPC + r) * D)[cp];
            o.x += x.x;
            o.y += x.y;
        }
        const long grow = grow0 + r;
        const float m = m_s[r], l = l_s[r];
        if (p.splits == 1) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            reinterpret_cast<uint32_t *>(reinterpret_cast<T *>(p.o) + grow * D)[cp] =
                pack2<BF16>(o.x * inv, o.y * inv);
            if (cp == 0)
                p.lse[grow] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        } else {
            const long prow = static_cast<long>(split) * total_rows + grow;
            reinterpret_cast<float2 *>(p.part_o + prow * D)[cp] = o;
            if (cp == 0) reinterpret_cast<float2 *>(p.part_ml)[prow] = make_float2(m, l);
        }
    }
}

// Merge of the key ranges of every row, in range order: M = max m_s, w_s = 2^(m_s - M),
// l = sum w_s l_s, O = sum w_s O_s / l, LSE = (M + log2 l) ln 2.  One CTA of four warps per
// row: warp q sums the q-th quarter of the ranges in order, the four partial sums are added in
// the order q = 0..3 (deterministic).
template <int D, bool BF16>
__global__ void __launch_bounds__(128) fa_decode_combine_kernel(const DecodeParams p) {
    using T = elem_t<BF16>;
    constexpr int kCols = D / 32;
    constexpr int kBatch = 8;  // ranges whose partial outputs are in flight at once
    __shared__ float red_o[4][D];
    __shared__ float red_l[4];
    const long total_rows = static_cast<long>(p.B) * p.H * p.Nq;
    const long row = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // launched to overlap the tail of the range kernel: its partial results are complete and
    // visible only past this point
    griddep_wait();
    const float2 *ml = reinterpret_cast<const float2 *>(p.part_ml);
    // every warp finds M over all ranges, 32 at a time, lane s holding range s
    float M = -INFINITY;
    for (int s0 = 0; s0 < p.splits; s0 += 32) {
        const int s = s0 + lane;
        const float m = s < p.splits ? ml[static_cast<long>(s) * total_rows + row].x : -INFINITY;
        M = fmaxf(M, m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const int per = (p.splits + 3) / 4;
    const int sb = min(p.splits, warp * per), se = min(p.splits, sb + per);
    float lsum = 0.f, acc[kCols];
#pragma unroll
    for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
    for (int s0 = sb; s0 < se; s0 += 32) {
        const int s = s0 + lane;
        float w = 0.f, lw = 0.f;  // the weights come from the lanes
        if (s < se) {
            const float2 st = ml[static_cast<long>(s) * total_rows + row];
            if (st.x != -INFINITY) {  // an empty range (also covers M = -inf) weighs nothing
                w = ex2(st.x - M);
                lw = w * st.y;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
        lsum += lw;
        // a batch of ranges' partial outputs loaded before any is used, so their latencies
        // overlap; a range past the warp's last one reads as zero with weight zero
        const int n = min(32, se - s0);
        for (int i0 = 0; i0 < n; i0 += kBatch) {
            float x[kBatch][kCols];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = i0 + u;
                const float *src = p.part_o +
                                   (static_cast<long>(s0 + min(i, n - 1)) * total_rows + row) * D +
                                   lane * kCols;
#pragma unroll
                for (int c = 0; c < kCols; ++c) x[u][c] = i < n ? src[c] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const float wi = __shfl_sync(0xffffffffu, w, i0 + u);
#pragma unroll
                for (int c = 0; c < kCols; ++c) acc[c] = fmaf(wi, x[u][c], acc[c]);
            }
        }
    }
    if (lane == 0) red_l[warp] = lsum;
#pragma unroll
    for (int c = 0; c < kCols; ++c) red_o[warp][lane * kCols + c] = acc[c];
    __syncthreads();
    if (warp != 0) return;
    const float l = red_l[0] + red_l[1] + red_l[2] + red_l[3];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T *dst = reinterpret_cast<T *>(p.o) + row * D + lane * kCols;
#pragma unroll
    for (int c = 0; c < kCols; c += 2) {
        float o2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int col = lane * kCols + c + e;
            o2[e] = red_o[0][col] + red_o[1][col] + red_o[2][col] + red_o[3][col];
        }
        reinterpret_cast<uint32_t *>(dst + c)[0] = pack2<BF16>(o2[0] * inv, o2[1] * inv);
    }
    if (lane == 0) p.lse[row] = l > 0.f ? (M + __log2f(l)) * 0.69314718055994531f : -INFINITY;
}

template <int D, bool BF16, int RPC>
cudaError_t launch_decode_rpc(const DecodeMaps &m, const DecodeParams &p, cudaStream_t stream) {
    using L = DecLayout<D, RPC>;
    auto kern = fa_decode_kernel<D, BF16, RPC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kAlloc);
    if (e != cudaSuccess) return e;
    const long grid = static_cast<long>(p.B) * p.Hkv * p.splits * p.row_groups;
    kern<<<static_cast<unsigned>(grid), kThreads, L::kAlloc, stream>>>(m.k, m.v, p);
    return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_decode_t(const DecodeMaps &m, const DecodeParams &p, cudaStream_t stream) {
    const int rpc = p.rows >= 16 ? 16 : p.rows;  // rows per CTA: the row group size
    cudaError_t e;
    if (rpc <= 1) e = launch_decode_rpc<D, BF16, 1>(m, p, stream);
    else if (rpc <= 2) e = launch_decode_rpc<D, BF16, 2>(m, p, stream);
    else if (rpc <= 4) e = launch_decode_rpc<D, BF16, 4>(m, p, stream);
    else if (rpc <= 8) e = launch_decode_rpc<D, BF16, 8>(m, p, stream);
    else e = launch_decode_rpc<D, BF16, 16>(m, p, stream);
    if (e != cudaSuccess || p.splits == 1) return e;
    // programmatic stream serialization: the merge's CTAs (small: 128 threads, 2 KB) are
    // scheduled beside the range kernel's last CTAs instead of after its completion
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long>(p.B) * p.H * p.Nq));
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fa_decode_combine_kernel<D, BF16>, p);
}

}  // namespace

cudaError_t launch_decode(const DecodeMaps &m, const DecodeParams &p, int d, bool bf16,
                          cudaStream_t stream) {
    if (d == 64) return bf16 ? launch_decode_t<64, true>(m, p, stream)
                             : launch_decode_t<64, false>(m, p, stream);
    return bf16 ? launch_decode_t<128, true>(m, p, stream)
                : launch_decode_t<128, false>(m, p, stream);
}

}  // namespace fa
