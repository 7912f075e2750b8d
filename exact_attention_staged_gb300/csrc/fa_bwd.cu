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
// In both, two groups of four warps split every 128 x 128 score tile into two 64-wide halves
// and alternate on the tensor core, the way the forward's two query tiles do.
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
// CTA = one 128-row key tile, 320 threads: warp 0 loads, warp 1 issues MMAs, warps 2..5
// (group 0) and 6..9 (group 1) each own one 64-query half of every 128 x 128 score tile.
// TMEM: S^T half h at [64h, 64h+64), dP^T half h at [128+64h, ...), dV at [256, 256+d),
// dK at [256+d, 256+2d).  P^T_h and dS^T_h are packed over the first 32 columns of S^T_h and
// dP^T_h.  MMA order per query tile n (next tile n+1), for h = 0, 1:
//   dV += P^T_h dO_h;  dK += dS^T_h Q_h;  S^T_h(n+1);  dP^T_h(n+1)
// so while one group exponentiates, the tensor core works on the other group's half.
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
    // kv_full, full[S], empty[S], s_full[2], dp_full[2], p_ready[2], ds_ready[2], final, drain
    static constexpr int kNumBars = 1 + 2 * kStages + 10;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kAlloc = kMiscOff + 16 + 1024;
    static constexpr int kThreads = 320;
};

template <int D, bool BF16>
__global__ void __launch_bounds__(320, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv,
                       const __grid_constant__ CUtensorMap tmdo, const BwdParams p) {
    using L = DkvLayout<D>;
    constexpr uint32_t kIdescSS = idesc_f16(128, 64, BF16, false);  // S^T_h, dP^T_h
    constexpr uint32_t kIdescTS = idesc_f16(128, D, BF16, true);    // dV, dK
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *kv_full = bars;
    uint64_t *full = bars + 1;
    uint64_t *empty = full + L::kStages;
    uint64_t *s_full = empty + L::kStages;  // [2]
    uint64_t *dp_full = s_full + 2;         // [2]
    uint64_t *p_ready = dp_full + 2;        // [2]
    uint64_t *ds_ready = p_ready + 2;       // [2]
    uint64_t *fin = ds_ready + 2;
    uint64_t *drain = fin + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);

    const int warp = warp_id(), lane = lane_id();
    const CtaOrder ord = cta_order(blockIdx.x, p.BH, p.T, p.head_group);
    const int bh = ord.head;
    const int kt = ord.rank;              // key tile; tile 0 sees the most query tiles when causal
    const int i0 = p.causal ? kt : 0;     // first query tile that can see it

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(&full[s], 2);  // TMA bytes + the producer warp's L/D stores
            mbar_init(&empty[s], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&s_full[h], 1);
            mbar_init(&dp_full[h], 1);
            mbar_init(&p_ready[h], 128);
            mbar_init(&ds_ready[h], 128);
        }
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
            const uint32_t tdV = tmem + 256, tdK = tmem + 256 + D;
            auto stage_q = [&](int st) {
                return smem_u32(smem + L::kStageOff + st * L::kStageBytes);
            };
            // S^T_h = K Q_h^T and dP^T_h = V dO_h^T, Q_h / dO_h = query rows [64h, 64h+64)
            const SDesc dK0 = sdesc_make(sK, 16, 1024), dV0 = sdesc_make(sV, 16, 1024);
            const SDesc dQk0 = sdesc_make(stage_q(0), 16, 1024);
            const SDesc dQm0 = sdesc_make(stage_q(0), L::kBoxBytes, 1024);
            auto issue_sdp = [&](int st, int h) {
                const uint32_t qoff = st * L::kStageBytes + h * 64 * 128;
                const SDesc bq = sdesc_add(dQk0, qoff), bdo = sdesc_add(dQk0, qoff + L::kTileBytes);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * L::kBoxBytes + (kk & 3) * 32;
                    mma_ss(tmem + 64 * h, sdesc_add(dK0, off), sdesc_add(bq, off), kIdescSS,
                           kk > 0 ? 1u : 0u);
                }
                umma_commit(&s_full[h]);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * L::kBoxBytes + (kk & 3) * 32;
                    mma_ss(tmem + 128 + 64 * h, sdesc_add(dV0, off), sdesc_add(bdo, off), kIdescSS,
                           kk > 0 ? 1u : 0u);
                }
                umma_commit(&dp_full[h]);
            };
            auto next_live = [&](int i) {
                for (++i; i < p.T; ++i)
                    if (tile_live(p, i, kt)) return i;
                return p.T;
            };
            bool ok = mbar_wait(kv_full, 0, p.ctl, abort_flag);
            int i = next_live(i0 - 1);
            int n = 0;
            if (ok && i < p.T) {
                ok = mbar_wait(&full[0], 0, p.ctl, abort_flag);
                if (ok) {
                    tc_fence_after();
                    issue_sdp(0, 0);
                    issue_sdp(0, 1);
                    if (p.ctl.visit_log != nullptr)
                        p.ctl.visit_log[(static_cast<size_t>(bh) * p.T + i) * p.T + kt] |= 2;
                }
            }
            while (ok && i < p.T) {
                const int s = n % L::kStages;
                const int s2 = (n + 1) % L::kStages;
                const int nxt = next_live(i);
                const SDesc bQm = sdesc_add(dQm0, s * L::kStageBytes);
                const SDesc bdOm = sdesc_add(bQm, L::kTileBytes);
                for (int h = 0; h < 2 && ok; ++h) {
                    if (!mbar_wait(&p_ready[h], n & 1, p.ctl, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // dV += P^T_h dO_h (K = 64 queries)
                        mma_ts(tdV, tmem + 64 * h + kk * 8, sdesc_add(bdOm, h * 8192 + kk * 2048),
                               kIdescTS, (n > 0 || h > 0 || kk > 0) ? 1u : 0u);
                    if (!mbar_wait(&ds_ready[h], n & 1, p.ctl, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // dK += dS^T_h Q_h
                        mma_ts(tdK, tmem + 128 + 64 * h + kk * 8, sdesc_add(bQm, h * 8192 + kk * 2048),
                               kIdescTS, (n > 0 || h > 0 || kk > 0) ? 1u : 0u);
                    if (h == 1) umma_commit(&empty[s]);
                    if (nxt < p.T) {
                        if (h == 0) {
                            if (!mbar_wait(&full[s2], ((n + 1) / L::kStages) & 1, p.ctl,
                                           abort_flag)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            if (p.ctl.visit_log != nullptr)
                                p.ctl.visit_log[(static_cast<size_t>(bh) * p.T + nxt) * p.T +
                                                kt] |= 2;
                        }
                        issue_sdp(s2, h);
                    }
                }
                i = nxt;
                ++n;
            }
            if (ok && n > 0) umma_commit(fin);
            umma_commit(drain);
            drain_wait(drain, 0, p.ctl);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- compute groups
        const int h = (warp - 2) >> 2;    // query half of every tile this group owns
        const int quad = warp & 3;
        const int row = quad * 32 + lane;  // key row within the tile
        const int k_row = kt * kTile + row;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_base + 64 * h, tdP = tS + 128;
        const float sl2 = p.scale_log2;
        int n = 0;
        bool ok = true;
        for (int i = i0; i < p.T; ++i) {
            if (!tile_live(p, i, kt)) continue;
            const int s = n % L::kStages;
            // the stage's L and D values were stored by the producer warp before its arrive
            if (!mbar_wait_warp(&full[s], (n / L::kStages) & 1, p.ctl, abort_flag) ||
                !mbar_wait_warp(&s_full[h], n & 1, p.ctl, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float *sl =
                reinterpret_cast<const float *>(smem + L::kStageOff + s * L::kStageBytes +
                                                2 * L::kTileBytes) + 64 * h;
            const float *sd = sl + 128;
            // query q sees key k only when k <= q: only the diagonal tile needs the compare
            const bool diag = p.causal && i == kt;
            uint32_t pk[32];  // P^T of this row's 64 queries, packed 16-bit pairs
            {
                uint32_t r[64];
                tmem_ld32(tS, r);
                tmem_ld32(tS + 32, r + 32);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int q0 = 2 * e;
                    float a = ex2(fmaf(__uint_as_float(r[q0]), sl2, -sl[q0]));
                    float b = ex2(fmaf(__uint_as_float(r[q0 + 1]), sl2, -sl[q0 + 1]));
                    if (diag) {
                        if (64 * h + q0 < row) a = 0.f;
                        if (64 * h + q0 + 1 < row) b = 0.f;
                    }
                    pk[e] = pack2<BF16>(a, b);
                }
            }
            tmem_st32(tS, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_ready[h]);
            if (!mbar_wait_warp(&dp_full[h], n & 1, p.ctl, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            {
                uint32_t r[64];
                tmem_ld32(tdP, r);
                tmem_ld32(tdP + 32, r + 32);
                tmem_wait_ld();
                uint32_t w[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int q0 = 2 * e;
                    const float2 pp = unpack2<BF16>(pk[e]);
                    w[e] = pack2<BF16>(pp.x * (__uint_as_float(r[q0]) - sd[q0]),
                                       pp.y * (__uint_as_float(r[q0 + 1]) - sd[q0 + 1]));
                }
                tmem_st32(tdP, w);  // over columns already read
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&ds_ready[h]);
            ++n;
        }
        if (ok && n > 0) {
            ok = mbar_wait_warp(fin, 0, p.ctl, abort_flag);
            tc_fence_after();
        }
        if (ok) {
            // group 0 writes dV, group 1 writes dK (times the softmax scale)
            const bool valid = k_row < p.N;
            using T = elem_t<BF16>;
            T *dst = reinterpret_cast<T *>(h == 0 ? p.out1 : p.out0) +
                     (static_cast<size_t>(bh) * p.N + k_row) * D;
            const uint32_t tacc = tmem + lane_base + 256 + h * D;
            const float mul = h == 0 ? 1.f : p.scale;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t a[32];
                if (n > 0) {
                    tmem_ld32(tacc + 32 * cc, a);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) a[e] = 0u;
                }
                if (valid) store_row32<BF16>(dst + 32 * cc, a, mul);
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
// CTA = one 128-row query tile, 320 threads: warp 0 loads, warp 1 issues MMAs, warps 2..5
// (group 0) and 6..9 (group 1) each own one 64-key half of every 128 x 128 score tile.
// TMEM: S half h at [64h, 64h+64), dP half h at [128+64h, ...), dQ at [256, 256+d); dS_h is
// packed over the first 32 columns of S_h.  MMA order per key tile n (next n+1), h = 0, 1:
//   dQ += dS_h K_h;  S_h(n+1);  dP_h(n+1)
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
    // q_full, full[S], empty[S], s_full[2], dp_full[2], ds_ready[2], final, drain
    static constexpr int kNumBars = 1 + 2 * kStages + 8;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kAlloc = kMiscOff + 16 + 1024;
    static constexpr int kThreads = 320;
};

template <int D, bool BF16>
__global__ void __launch_bounds__(320, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmdo, const BwdParams p) {
    using L = DqLayout<D>;
    constexpr uint32_t kIdescSS = idesc_f16(128, 64, BF16, false);  // S_h, dP_h
    constexpr uint32_t kIdescTS = idesc_f16(128, D, BF16, true);    // dQ
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *q_full = bars;
    uint64_t *full = bars + 1;
    uint64_t *empty = full + L::kStages;
    uint64_t *s_full = empty + L::kStages;  // [2]
    uint64_t *dp_full = s_full + 2;         // [2]
    uint64_t *ds_ready = dp_full + 2;       // [2]
    uint64_t *fin = ds_ready + 2;
    uint64_t *drain = fin + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);

    const int warp = warp_id(), lane = lane_id();
    const CtaOrder ord = cta_order(blockIdx.x, p.BH, p.T, p.head_group);
    const int bh = ord.head;
    const int qt = p.T - 1 - ord.rank;  // long rows first
    const int jend = p.causal ? qt + 1 : p.T;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&s_full[h], 1);
            mbar_init(&dp_full[h], 1);
            mbar_init(&ds_ready[h], 128);
        }
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
            const uint32_t tdQ = tmem + 256;
            auto stage_k = [&](int st) {
                return smem_u32(smem + L::kStageOff + st * L::kStageBytes);
            };
            // S_h = Q K_h^T and dP_h = dO V_h^T, K_h / V_h = key rows [64h, 64h+64)
            const SDesc dQa = sdesc_make(sQ, 16, 1024), ddOa = sdesc_make(sdO, 16, 1024);
            const SDesc dK0 = sdesc_make(stage_k(0), 16, 1024);
            const SDesc dKm0 = sdesc_make(stage_k(0), L::kBoxBytes, 1024);
            auto issue_sdp = [&](int st, int h) {
                const uint32_t koff = st * L::kStageBytes + h * 64 * 128;
                const SDesc bk = sdesc_add(dK0, koff), bv = sdesc_add(dK0, koff + L::kTileBytes);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * L::kBoxBytes + (kk & 3) * 32;
                    mma_ss(tmem + 64 * h, sdesc_add(dQa, off), sdesc_add(bk, off), kIdescSS,
                           kk > 0 ? 1u : 0u);
                }
                umma_commit(&s_full[h]);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * L::kBoxBytes + (kk & 3) * 32;
                    mma_ss(tmem + 128 + 64 * h, sdesc_add(ddOa, off), sdesc_add(bv, off), kIdescSS,
                           kk > 0 ? 1u : 0u);
                }
                umma_commit(&dp_full[h]);
            };
            auto next_live = [&](int j) {
                for (++j; j < jend; ++j)
                    if (tile_live(p, qt, j)) return j;
                return jend;
            };
            bool ok = mbar_wait(q_full, 0, p.ctl, abort_flag);
            int j = next_live(-1);
            int n = 0;
            if (ok && j < jend) {
                ok = mbar_wait(&full[0], 0, p.ctl, abort_flag);
                if (ok) {
                    tc_fence_after();
                    issue_sdp(0, 0);
                    issue_sdp(0, 1);
                    if (p.ctl.visit_log != nullptr)
                        p.ctl.visit_log[(static_cast<size_t>(bh) * p.T + qt) * p.T + j] |= 4;
                }
            }
            while (ok && j < jend) {
                const int s = n % L::kStages;
                const int s2 = (n + 1) % L::kStages;
                const int nxt = next_live(j);
                const SDesc bKm = sdesc_add(dKm0, s * L::kStageBytes);
                for (int h = 0; h < 2 && ok; ++h) {
                    if (!mbar_wait(&ds_ready[h], n & 1, p.ctl, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // dQ += dS_h K_h (K = 64 keys)
                        mma_ts(tdQ, tmem + 64 * h + kk * 8, sdesc_add(bKm, h * 8192 + kk * 2048),
                               kIdescTS, (n > 0 || h > 0 || kk > 0) ? 1u : 0u);
                    if (h == 1) umma_commit(&empty[s]);
                    if (nxt < jend) {
                        if (h == 0) {
                            if (!mbar_wait(&full[s2], ((n + 1) / L::kStages) & 1, p.ctl,
                                           abort_flag)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            if (p.ctl.visit_log != nullptr)
                                p.ctl.visit_log[(static_cast<size_t>(bh) * p.T + qt) * p.T +
                                                nxt] |= 4;
                        }
                        issue_sdp(s2, h);
                    }
                }
                j = nxt;
                ++n;
            }
            if (ok && n > 0) umma_commit(fin);
            umma_commit(drain);
            drain_wait(drain, 0, p.ctl);
        }
        __syncwarp();
    } else {
        const int h = (warp - 2) >> 2;  // key half of every tile this group owns
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int q_row = qt * kTile + row;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_base + 64 * h, tdP = tS + 128;
        const float sl2 = p.scale_log2;
        const float lrow = lse_log2(p, bh, q_row);
        const float drow = q_row < p.N ? p.delta[static_cast<size_t>(bh) * p.N + q_row] : 0.f;
        int n = 0;
        bool ok = true;
        for (int j = 0; j < jend; ++j) {
            if (!tile_live(p, qt, j)) continue;
            if (!mbar_wait_warp(&s_full[h], n & 1, p.ctl, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int kv0 = j * kTile + 64 * h;
            const bool need_mask = (p.causal && j == qt) || (kv0 + 64 > p.N);
            float pr[64];  // P of this row's 64 keys, fp32, while the tensor core is on dP
            {
                uint32_t a[64];
                tmem_ld32(tS, a);
                tmem_ld32(tS + 32, a + 32);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    float pv = ex2(fmaf(__uint_as_float(a[e]), sl2, -lrow));
                    if (need_mask) {
                        const int col = kv0 + e;
                        if (col >= p.N || (p.causal && col > q_row)) pv = 0.f;
                    }
                    pr[e] = pv;
                }
            }
            if (!mbar_wait_warp(&dp_full[h], n & 1, p.ctl, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            {
                uint32_t b[64];
                tmem_ld32(tdP, b);
                tmem_ld32(tdP + 32, b + 32);
                tmem_wait_ld();
                uint32_t w[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    w[e] = pack2<BF16>(pr[2 * e] * (__uint_as_float(b[2 * e]) - drow),
                                       pr[2 * e + 1] * (__uint_as_float(b[2 * e + 1]) - drow));
                tmem_st32(tS, w);  // over columns already read
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&ds_ready[h]);
            ++n;
        }
        if (ok && n > 0) {
            ok = mbar_wait_warp(fin, 0, p.ctl, abort_flag);
            tc_fence_after();
        }
        if (ok) {
            // each group writes half of dQ's columns (times the softmax scale)
            const bool valid = q_row < p.N;
            using T = elem_t<BF16>;
            T *dq = reinterpret_cast<T *>(p.out0) + (static_cast<size_t>(bh) * p.N + q_row) * D +
                    h * (D / 2);
            const uint32_t tacc = tmem + lane_base + 256 + h * (D / 2);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t a[32];
                if (n > 0) {
                    tmem_ld32(tacc + 32 * cc, a);
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
