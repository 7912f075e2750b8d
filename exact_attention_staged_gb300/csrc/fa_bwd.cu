// fa_bwd.cu - exact-attention backward for sm_103a (tcgen05 + TMA + TMEM).
//
// FlashAttention-2 reading notes, Algorithm 2 (backward), with the scores and probabilities
// recomputed on chip from Q, K and the stored logsumexp (P_ij = exp(S_ij - L_i), eq. (16)) and
// the softmax Jacobian dS = P o (dP - D) (eq. (17)), where D_i = rowsum(dO_i o O_i) is computed
// first (Algorithm 2's precomputation; FlashAttention paper detail, "Technique 2").
// The atomic dQ update of Algorithm 2 is replaced by a second, query-stationary pass, so every
// output element is written once by one CTA: the result is deterministic.
//
//   preprocess   D = rowsum(dO o O), one group of lanes per row, fp32.
//   dK/dV        CTA = one 128-row key tile j of one head (K_j, V_j stay in smem).  For every
//                live query tile i (causal: i >= j; block mask: M[i][j] != 0):
//                  S^T = K_j Q_i^T, dP^T = V_j dO_i^T     (SS MMAs into TMEM)
//                  P^T = exp2(S^T * scale*log2e - L * log2e)  (one key row per thread)
//                  dV += P^T dO_i                         (TS MMA, P^T in TMEM)
//                  dS^T = P^T o (dP^T - D)
//                  dK += dS^T Q_i                         (TS MMA, dS^T in TMEM)
//                and finally dK *= scale.
//   dQ           CTA = one 128-row query tile i.  For every live key tile j:
//                  S = Q_i K_j^T, dP = dO_i V_j^T, P = exp2(...), dS = P o (dP - D_i),
//                  dQ += dS K_j (TS MMA), and finally dQ *= scale.
// TMEM (512 columns): [0,128) S or S^T (then P / dS packed over its first 64 columns),
// [128,256) dP or dP^T (dS^T packed over its first 64 columns), then the d-wide accumulators.
#include "fa_internal.h"

#include <cmath>
#include <type_traits>

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    const uint32_t a = smem_u32(p);
    return p + ((1024u - (a & 1023u)) & 1023u);
}

__device__ __forceinline__ bool tile_live(const BwdParams &p, int qt, int kt) {
    if (p.causal && kt > qt) return false;
    if (p.mask != nullptr && p.mask[qt * p.T + kt] == 0) return false;
    return true;
}

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, const Ctl &ctl) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(a, parity)) {
        if (global_timer_ns() - t0 > ctl.wait_limit_ns) return;
    }
}

// LSE in log2 units for the exponent; rows that are out of range or fully masked (LSE = -inf)
// get +inf so that every recomputed probability of theirs is exactly 0.
__device__ __forceinline__ float lse_log2(const BwdParams &p, int bh, int row) {
    if (row >= p.N) return INFINITY;
    const float v = p.lse[static_cast<size_t>(bh) * p.N + row];
    return v == -INFINITY ? INFINITY : v * kLog2e;
}

template <bool BF16>
using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;

// Store 32 fp32 values (times `mul`) of one row as 16-bit values, 64 bytes.
template <bool BF16>
__device__ __forceinline__ void store_row32(void *dst, const uint32_t *v, float mul) {
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
        w[e] = pack2<BF16>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
    uint4 *d = reinterpret_cast<uint4 *>(dst);
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
    d[2] = make_uint4(w[8], w[9], w[10], w[11]);
    d[3] = make_uint4(w[12], w[13], w[14], w[15]);
}

// ================================================================================ preprocess
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_preprocess_kernel(const void *o, const void *dout,
                                                                float *delta, long rows) {
    constexpr int kLanes = D / 8;  // 8 elements (16 bytes) per lane
    const long gid = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long row = gid / kLanes;
    const int part = static_cast<int>(gid % kLanes);
    float acc = 0.f;
    if (row < rows) {
        const uint4 a = reinterpret_cast<const uint4 *>(o)[row * kLanes + part];
        const uint4 b = reinterpret_cast<const uint4 *>(dout)[row * kLanes + part];
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
        const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = unpack2<BF16>(aw[e]);
            const float2 y = unpack2<BF16>(bw[e]);
            acc = fmaf(x.x, y.x, acc);
            acc = fmaf(x.y, y.y, acc);
        }
    }
#pragma unroll
    for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && part == 0) delta[row] = acc;
}

// ================================================================================ dK / dV
template <int D>
struct DkvLayout {
    static constexpr int kTileBytes = kTile * D * 2;
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = kTile * 128;
    static constexpr int kStages = (D == 128) ? 2 : 4;
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kTileBytes;
    static constexpr int kStageOff = 2 * kTileBytes;
    // per stage: Q tile, dO tile, then 128 floats of L*log2e and 128 floats of D
    static constexpr int kStageBytes = 2 * kTileBytes + 1024;
    static constexpr int kBarOff = kStageOff + kStages * kStageBytes;
    // kv_full, full[S], empty[S], s_full, p_ready, ds_ready, final, drain
    static constexpr int kNumBars = 1 + 2 * kStages + 5;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kAlloc = kMiscOff + 16 + 1024;
    static constexpr int kThreads = 192;
};

template <int D, bool BF16>
__global__ void __launch_bounds__(192, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv,
                       const __grid_constant__ CUtensorMap tmdo, const BwdParams p) {
    using L = DkvLayout<D>;
    constexpr uint32_t kIdescSS = idesc_f16(128, 128, BF16, false);
    constexpr uint32_t kIdescTS = idesc_f16(128, D, BF16, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *kv_full = bars;
    uint64_t *full = bars + 1;
    uint64_t *empty = full + L::kStages;
    uint64_t *s_full = empty + L::kStages;
    uint64_t *p_ready = s_full + 1;
    uint64_t *ds_ready = p_ready + 1;
    uint64_t *fin = ds_ready + 1;
    uint64_t *drain = fin + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);

    const int warp = warp_id(), lane = lane_id();
    const int bh = blockIdx.x % p.BH;
    const int kt = static_cast<int>(blockIdx.x / p.BH);  // key tile
    const int i0 = p.causal ? kt : 0;                    // first query tile that can see it

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(&full[s], 2);  // TMA bytes + the producer warp's L/D stores
            mbar_init(&empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_ready, 128);
        mbar_init(ds_ready, 128);
        mbar_init(fin, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer warp
        if (lane == 0) {
            mbar_arrive_expect_tx(kv_full, 2 * L::kTileBytes);
            for (int b = 0; b < L::kBoxes; ++b) {
                tma_load_3d(smem + L::kKOff + b * L::kBoxBytes, &tmk, b * 64, kt * kTile, bh,
                            kv_full);
                tma_load_3d(smem + L::kVOff + b * L::kBoxBytes, &tmv, b * 64, kt * kTile, bh,
                            kv_full);
            }
        }
        int n = 0;
        bool ok = true;
        for (int i = i0; i < p.T && ok; ++i) {
            if (!tile_live(p, i, kt)) continue;
            const int s = n % L::kStages;
            const uint32_t par = ((n / L::kStages) & 1) ^ 1;
            int got = 0;
            if (lane == 0) got = mbar_wait(&empty[s], par, p.ctl, abort_flag) ? 1 : 0;
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
                ok = false;
                break;
            }
            uint8_t *st = smem + L::kStageOff + s * L::kStageBytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[s], 2 * L::kTileBytes);
                for (int b = 0; b < L::kBoxes; ++b) {
                    tma_load_3d(st + b * L::kBoxBytes, &tmq, b * 64, i * kTile, bh, &full[s]);
                    tma_load_3d(st + L::kTileBytes + b * L::kBoxBytes, &tmdo, b * 64, i * kTile,
                                bh, &full[s]);
                }
            }
            float *sl = reinterpret_cast<float *>(st + 2 * L::kTileBytes);
            float *sd = sl + 128;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = lane + 32 * e;
                const int row = i * kTile + c;
                sl[c] = lse_log2(p, bh, row);
                sd[c] = row < p.N ? p.delta[static_cast<size_t>(bh) * p.N + row] : 0.f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[s]);
            ++n;
        }
        if (lane == 0 && (!ok || *abort_flag)) {
            drain_wait(kv_full, 0, p.ctl);
            const int first = n > L::kStages ? n - L::kStages : 0;
            for (int l = first; l < n; ++l)
                drain_wait(&full[l % L::kStages], (l / L::kStages) & 1, p.ctl);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t sK = smem_u32(smem + L::kKOff);
            const uint32_t sV = smem_u32(smem + L::kVOff);
            const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;
            bool ok = mbar_wait(kv_full, 0, p.ctl, abort_flag);
            int n = 0;
            for (int i = i0; ok && i < p.T; ++i) {
                if (!tile_live(p, i, kt)) continue;
                const int s = n % L::kStages;
                if (!mbar_wait(&full[s], (n / L::kStages) & 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sQ = smem_u32(smem + L::kStageOff + s * L::kStageBytes);
                const uint32_t sdO = sQ + L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {  // S^T = K Q^T
                    const uint32_t off = (kk >> 2) * L::kBoxBytes + (kk & 3) * 32;
                    umma_ss(tS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024),
                            kIdescSS, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {  // dP^T = V dO^T
                    const uint32_t off = (kk >> 2) * L::kBoxBytes + (kk & 3) * 32;
                    umma_ss(tdP, sdesc_sw128(sV + off, 16, 1024),
                            sdesc_sw128(sdO + off, 16, 1024), kIdescSS, kk > 0 ? 1u : 0u);
                }
                umma_commit(s_full);
                if (p.ctl.visit_log != nullptr)
                    p.ctl.visit_log[(static_cast<size_t>(bh) * p.T + i) * p.T + kt] |= 2;
                if (!mbar_wait(p_ready, n & 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)  // dV += P^T dO
                    umma_ts(tdV, tS + kk * 8, sdesc_sw128(sdO + kk * 2048, L::kBoxBytes, 1024),
                            kIdescTS, (n > 0 || kk > 0) ? 1u : 0u);
                if (!mbar_wait(ds_ready, n & 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)  // dK += dS^T Q
                    umma_ts(tdK, tdP + kk * 8, sdesc_sw128(sQ + kk * 2048, L::kBoxBytes, 1024),
                            kIdescTS, (n > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&empty[s]);
                ++n;
            }
            if (ok && n > 0) umma_commit(fin);
            umma_commit(drain);
            drain_wait(drain, 0, p.ctl);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- compute group
        const int quad = warp & 3;
        const int row = quad * 32 + lane;  // key row within the tile
        const int k_row = kt * kTile + row;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_base, tdP = tS + 128, tdV = tS + 256, tdK = tS + 256 + D;
        const float sl2 = p.scale_log2;
        int n = 0;
        bool ok = true;
        for (int i = i0; i < p.T; ++i) {
            if (!tile_live(p, i, kt)) continue;
            const int s = n % L::kStages;
            // the stage's L and D values were stored by the producer warp before its arrive
            if (!mbar_wait_warp(&full[s], (n / L::kStages) & 1, p.ctl, abort_flag) ||
                !mbar_wait_warp(s_full, n & 1, p.ctl, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float *sl =
                reinterpret_cast<const float *>(smem + L::kStageOff + s * L::kStageBytes +
                                                2 * L::kTileBytes);
            const float *sd = sl + 128;
            const bool diag = p.causal && i == kt;  // only this tile needs the causal compare
            uint32_t pk[64];                        // P^T of this row, packed 16-bit pairs
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld32(tS + 32 * c, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int q0 = 32 * c + 2 * e;
                    float a = ex2(fmaf(__uint_as_float(r[2 * e]), sl2, -sl[q0]));
                    float b = ex2(fmaf(__uint_as_float(r[2 * e + 1]), sl2, -sl[q0 + 1]));
                    if (diag) {  // query q sees key k only when k <= q
                        if (q0 < row) a = 0.f;
                        if (q0 + 1 < row) b = 0.f;
                    }
                    pk[16 * c + e] = pack2<BF16>(a, b);
                }
            }
            tmem_st32(tS, pk);
            tmem_st32(tS + 32, pk + 32);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(p_ready);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld32(tdP + 32 * c, r);
                tmem_wait_ld();
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int q0 = 32 * c + 2 * e;
                    const float2 pp = unpack2<BF16>(pk[16 * c + e]);
                    const float a = pp.x * (__uint_as_float(r[2 * e]) - sd[q0]);
                    const float b = pp.y * (__uint_as_float(r[2 * e + 1]) - sd[q0 + 1]);
                    w[e] = pack2<BF16>(a, b);
                }
                tmem_st16(tdP + 16 * c, w);  // over columns already read
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(ds_ready);
            ++n;
        }
        if (ok && n > 0) {
            ok = mbar_wait_warp(fin, 0, p.ctl, abort_flag);
            tc_fence_after();
        }
        if (ok) {
            const bool valid = k_row < p.N;
            using T = elem_t<BF16>;
            T *dk = reinterpret_cast<T *>(p.out0) + (static_cast<size_t>(bh) * p.N + k_row) * D;
            T *dv = reinterpret_cast<T *>(p.out1) + (static_cast<size_t>(bh) * p.N + k_row) * D;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t a[32], b[32];
                if (n > 0) {
                    tmem_ld32(tdV + 32 * cc, a);
                    tmem_ld32(tdK + 32 * cc, b);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) a[e] = b[e] = 0u;
                }
                if (valid) {
                    store_row32<BF16>(dv + 32 * cc, a, 1.f);
                    store_row32<BF16>(dk + 32 * cc, b, p.scale);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ================================================================================ dQ
template <int D>
struct DqLayout {
    static constexpr int kTileBytes = kTile * D * 2;
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = kTile * 128;
    static constexpr int kStages = (D == 128) ? 2 : 4;
    static constexpr int kQOff = 0;
    static constexpr int kdOOff = kTileBytes;
    static constexpr int kStageOff = 2 * kTileBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;  // K tile, V tile
    static constexpr int kBarOff = kStageOff + kStages * kStageBytes;
    // q_full, full[S], empty[S], s_full, ds_ready, final, drain
    static constexpr int kNumBars = 1 + 2 * kStages + 4;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kAlloc = kMiscOff + 16 + 1024;
    static constexpr int kThreads = 192;
};

template <int D, bool BF16>
__global__ void __launch_bounds__(192, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmdo, const BwdParams p) {
    using L = DqLayout<D>;
    constexpr uint32_t kIdescSS = idesc_f16(128, 128, BF16, false);
    constexpr uint32_t kIdescTS = idesc_f16(128, D, BF16, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *q_full = bars;
    uint64_t *full = bars + 1;
    uint64_t *empty = full + L::kStages;
    uint64_t *s_full = empty + L::kStages;
    uint64_t *ds_ready = s_full + 1;
    uint64_t *fin = ds_ready + 1;
    uint64_t *drain = fin + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);

    const int warp = warp_id(), lane = lane_id();
    const int bh = blockIdx.x % p.BH;
    const int qt = p.T - 1 - static_cast<int>(blockIdx.x / p.BH);  // long rows first
    const int jend = p.causal ? qt + 1 : p.T;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(ds_ready, 128);
        mbar_init(fin, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, 2 * L::kTileBytes);
            for (int b = 0; b < L::kBoxes; ++b) {
                tma_load_3d(smem + L::kQOff + b * L::kBoxBytes, &tmq, b * 64, qt * kTile, bh,
                            q_full);
                tma_load_3d(smem + L::kdOOff + b * L::kBoxBytes, &tmdo, b * 64, qt * kTile, bh,
                            q_full);
            }
            int n = 0;
            bool ok = true;
            for (int j = 0; j < jend && ok; ++j) {
                if (!tile_live(p, qt, j)) continue;
                const int s = n % L::kStages;
                if (!mbar_wait(&empty[s], ((n / L::kStages) & 1) ^ 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                uint8_t *st = smem + L::kStageOff + s * L::kStageBytes;
                mbar_arrive_expect_tx(&full[s], 2 * L::kTileBytes);
                for (int b = 0; b < L::kBoxes; ++b) {
                    tma_load_3d(st + b * L::kBoxBytes, &tmk, b * 64, j * kTile, bh, &full[s]);
                    tma_load_3d(st + L::kTileBytes + b * L::kBoxBytes, &tmv, b * 64, j * kTile,
                                bh, &full[s]);
                }
                ++n;
            }
            if (!ok || *abort_flag) {
                drain_wait(q_full, 0, p.ctl);
                const int first = n > L::kStages ? n - L::kStages : 0;
                for (int l = first; l < n; ++l)
                    drain_wait(&full[l % L::kStages], (l / L::kStages) & 1, p.ctl);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t sQ = smem_u32(smem + L::kQOff);
            const uint32_t sdO = smem_u32(smem + L::kdOOff);
            const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256;
            bool ok = mbar_wait(q_full, 0, p.ctl, abort_flag);
            int n = 0;
            for (int j = 0; ok && j < jend; ++j) {
                if (!tile_live(p, qt, j)) continue;
                const int s = n % L::kStages;
                if (!mbar_wait(&full[s], (n / L::kStages) & 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sK = smem_u32(smem + L::kStageOff + s * L::kStageBytes);
                const uint32_t sV = sK + L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {  // S = Q K^T
                    const uint32_t off = (kk >> 2) * L::kBoxBytes + (kk & 3) * 32;
                    umma_ss(tS, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024),
                            kIdescSS, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {  // dP = dO V^T
                    const uint32_t off = (kk >> 2) * L::kBoxBytes + (kk & 3) * 32;
                    umma_ss(tdP, sdesc_sw128(sdO + off, 16, 1024),
                            sdesc_sw128(sV + off, 16, 1024), kIdescSS, kk > 0 ? 1u : 0u);
                }
                umma_commit(s_full);
                if (p.ctl.visit_log != nullptr)
                    p.ctl.visit_log[(static_cast<size_t>(bh) * p.T + qt) * p.T + j] |= 4;
                if (!mbar_wait(ds_ready, n & 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)  // dQ += dS K
                    umma_ts(tdQ, tS + kk * 8, sdesc_sw128(sK + kk * 2048, L::kBoxBytes, 1024),
                            kIdescTS, (n > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&empty[s]);
                ++n;
            }
            if (ok && n > 0) umma_commit(fin);
            umma_commit(drain);
            drain_wait(drain, 0, p.ctl);
        }
        __syncwarp();
    } else {
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int q_row = qt * kTile + row;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_base, tdP = tS + 128, tdQ = tS + 256;
        const float sl2 = p.scale_log2;
        const float lrow = lse_log2(p, bh, q_row);
        const float drow = q_row < p.N ? p.delta[static_cast<size_t>(bh) * p.N + q_row] : 0.f;
        int n = 0;
        bool ok = true;
        for (int j = 0; j < jend; ++j) {
            if (!tile_live(p, qt, j)) continue;
            if (!mbar_wait_warp(s_full, n & 1, p.ctl, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int kv0 = j * kTile;
            const bool need_mask = (p.causal && j == qt) || (kv0 + kTile > p.N);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t a[32], b[32];
                tmem_ld32(tS + 32 * c, a);
                tmem_ld32(tdP + 32 * c, b);
                tmem_wait_ld();
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float pa = ex2(fmaf(__uint_as_float(a[2 * e]), sl2, -lrow));
                    float pb = ex2(fmaf(__uint_as_float(a[2 * e + 1]), sl2, -lrow));
                    if (need_mask) {
                        const int col = kv0 + 32 * c + 2 * e;
                        if (col >= p.N || (p.causal && col > q_row)) pa = 0.f;
                        if (col + 1 >= p.N || (p.causal && col + 1 > q_row)) pb = 0.f;
                    }
                    w[e] = pack2<BF16>(pa * (__uint_as_float(b[2 * e]) - drow),
                                       pb * (__uint_as_float(b[2 * e + 1]) - drow));
                }
                tmem_st16(tS + 16 * c, w);  // over columns already read
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(ds_ready);
            ++n;
        }
        if (ok && n > 0) {
            ok = mbar_wait_warp(fin, 0, p.ctl, abort_flag);
            tc_fence_after();
        }
        if (ok) {
            const bool valid = q_row < p.N;
            using T = elem_t<BF16>;
            T *dq = reinterpret_cast<T *>(p.out0) + (static_cast<size_t>(bh) * p.N + q_row) * D;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t a[32];
                if (n > 0) {
                    tmem_ld32(tdQ + 32 * cc, a);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) a[e] = 0u;
                }
                if (valid) store_row32<BF16>(dq + 32 * cc, a, p.scale);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool BF16>
cudaError_t launch_pre_t(const void *o, const void *dout, float *delta, long rows,
                         cudaStream_t stream) {
    const long threads = rows * (D / 8);
    const long blocks = (threads + 255) / 256;
    fa_bwd_preprocess_kernel<D, BF16>
        <<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o, dout, delta, rows);
    return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_dkdv_t(const Maps &m, const BwdParams &p, cudaStream_t stream) {
    using L = DkvLayout<D>;
    auto kern = fa_bwd_dkdv_kernel<D, BF16>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(static_cast<long>(p.BH) * p.T), L::kThreads, L::kAlloc,
           stream>>>(m.q, m.k, m.v, m.dout, p);
    return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_dq_t(const Maps &m, const BwdParams &p, cudaStream_t stream) {
    using L = DqLayout<D>;
    auto kern = fa_bwd_dq_kernel<D, BF16>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(static_cast<long>(p.BH) * p.T), L::kThreads, L::kAlloc,
           stream>>>(m.q, m.k, m.v, m.dout, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess(const void *o, const void *dout, float *delta, long rows,
                                  int d, bool bf16, cudaStream_t stream) {
    if (d == 64) return bf16 ? launch_pre_t<64, true>(o, dout, delta, rows, stream)
                             : launch_pre_t<64, false>(o, dout, delta, rows, stream);
    return bf16 ? launch_pre_t<128, true>(o, dout, delta, rows, stream)
                : launch_pre_t<128, false>(o, dout, delta, rows, stream);
}

cudaError_t launch_bwd_dkdv(const Maps &maps, const BwdParams &p, int d, bool bf16,
                            cudaStream_t stream) {
    if (d == 64) return bf16 ? launch_dkdv_t<64, true>(maps, p, stream)
                             : launch_dkdv_t<64, false>(maps, p, stream);
    return bf16 ? launch_dkdv_t<128, true>(maps, p, stream)
                : launch_dkdv_t<128, false>(maps, p, stream);
}

cudaError_t launch_bwd_dq(const Maps &maps, const BwdParams &p, int d, bool bf16,
                          cudaStream_t stream) {
    if (d == 64) return bf16 ? launch_dq_t<64, true>(maps, p, stream)
                             : launch_dq_t<64, false>(maps, p, stream);
    return bf16 ? launch_dq_t<128, true>(maps, p, stream)
                : launch_dq_t<128, false>(maps, p, stream);
}

}  // namespace fa
