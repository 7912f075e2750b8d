// fa_decode.cu - decode: a few new query rows per sequence against a KV cache, sm_103a.
//
// FlashAttention-2 reading notes, section on the KV cache: in the decode phase each step's
// query is a few rows against the N cached keys, so the work is bound by reading K and V from
// HBM, not by arithmetic, and it is split over the cache: a work unit is (K/V head, key range,
// group of up to 128 query rows) and runs the online softmax (running max m and sum l per row,
// FlashAttention-2 Algorithm 1) over its key range for every query row that reads this K/V head
// (all query heads of a grouped-query group, times the new rows), reading each cached K/V row
// once.  Key ranges are merged by the statistic merge of the FlashAttention paper detail,
// Technique 1 (m = max(m1, m2), l = e^(m1-m) l1 + e^(m2-m) l2, and the outputs weighted the same
// way), in range order.
//
// GB300 mapping: the products run on the tensor cores even though a unit has only a handful of
// real query rows, so that the SM's own pipes are left with the softmax alone and the kernel can
// stream K and V at the HBM rate: the unit's query rows are the first rows of a 128-row A tile
// (a group's rows are consecutive rows of Q, loaded by TMA; the tile's other rows belong to the
// next groups or read as zeros, and their results are never stored), S = Q K_j^T is a 128 x 128
// tcgen05 MMA into tensor memory, one softmax thread per row (as in the forward) turns it into
// P~ = 2^(S scale log2 e - m) over S, and O += P~ V_j takes P~ from tensor memory.  Per CTA
// (192 threads, one per SM): warp 0 loads (Q of each unit, K_j and V_j of 128 keys into a ring),
// warp 1 issues the MMAs, warps 2..5 run the softmax of their 32-row quarter (only quarters
// holding real rows do the arithmetic).  S has two buffers, so S_{j+1} is computed while the
// softmax of S_j runs.  The grid has one CTA per unit, and the CTAs that start walk the units
// of those that have not (cluster launch control, as in the forward), so the ring streams across
// unit boundaries.
#include "fa_internal.h"

#include <cmath>
#include <type_traits>

namespace fa {
namespace {

constexpr int kDecTile = 128;  // keys per K/V tile, rows per query tile (the MMA's M)

template <int D>
struct DecLayout {
    static constexpr int kTileBytes = kDecTile * D * 2;   // one 128 x d tile of 16-bit values
    static constexpr int kBoxes = D / 64;                 // 128-byte-wide TMA boxes per tile row
    static constexpr int kBoxBytes = kDecTile * 128;      // 16 KB
    static constexpr int kStages = (D == 128) ? 3 : 6;    // K/V tile pairs in the ring
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = kTileBytes;           // [stage][K, V]
    static constexpr int kBarOff = kRingOff + kStages * 2 * kTileBytes;
    // q_full, q_empty, kv_full[S], kv_empty[S], s_full[2], p_full[2], pv_done, o_final,
    // unit_full[2], unit_empty[2], sched, drain
    static constexpr int kNumBars = 2 + 2 * kStages + 12;
    static constexpr int kSchedOff = (kBarOff + kNumBars * 8 + 15) / 16 * 16;  // 16-byte answer
    static constexpr int kUnitOff = kSchedOff + 16;      // int unit[2]
    static constexpr int kMiscOff = kUnitOff + 8;        // TMEM base, abort flag
    static constexpr int kBytes = kMiscOff + 8;
    static constexpr int kAlloc = kBytes + 1024;         // room to align the base to 1024 bytes
    static constexpr int kThreads = 192;
    static constexpr uint32_t kTmemCols = 512;           // S_0, S_1 (2 x 128) + O (d)
    static_assert(kAlloc <= 232448, "shared memory per CTA");
};

template <bool BF16>
using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;

// One work unit: a key range of one K/V head for one group of its query rows.
struct DecUnit {
    int kvh, split, r0, nrows;  // K/V head (b * H_kv + g); range; first group row; real rows
    int len;                    // keys of the sequence (kv_len clamped to [0, Nk])
    int k_begin, k_end, ntiles; // the range [k_begin, k_end) in 128-key tiles
    long grow0;                 // global row of the group's first row
};
__device__ __forceinline__ DecUnit dec_unit(const DecodeParams &p, int unit) {
    unsigned bid = static_cast<unsigned>(unit);  // row group fastest, then key range, then K/V head
    DecUnit u;
    const int rg = static_cast<int>(bid % static_cast<unsigned>(p.row_groups));
    bid /= static_cast<unsigned>(p.row_groups);
    u.split = static_cast<int>(bid % static_cast<unsigned>(p.splits));
    u.kvh = static_cast<int>(bid / static_cast<unsigned>(p.splits));
    const int b = u.kvh / p.Hkv;
    u.r0 = rg * kDecTile;
    u.nrows = min(kDecTile, p.rows - u.r0);
    int len = p.kv_len != nullptr ? p.kv_len[b] : p.Nk;
    u.len = max(0, min(len, p.Nk));
    u.k_begin = u.split * p.chunk;
    u.k_end = min(u.k_begin + p.chunk, u.len);
    u.ntiles = u.k_end > u.k_begin ? (u.k_end - u.k_begin + kDecTile - 1) / kDecTile : 0;
    // group row r is query head kvh * rep + (r0 + r) / Nq, new row (r0 + r) % Nq, i.e. global
    // row ((b * H + h) * Nq + i) = kvh * rows + r0 + r
    u.grow0 = static_cast<long>(u.kvh) * p.rows + u.r0;
    return u;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(192, 1)
    fa_decode_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const DecodeParams p) {
    using L = DecLayout<D>;
    constexpr uint32_t kIdescS = idesc_f16(128, 128, BF16, false);
    constexpr uint32_t kIdescPV = idesc_f16(128, D, BF16, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *q_full = bars;
    uint64_t *q_empty = bars + 1;
    uint64_t *kv_full = bars + 2;
    uint64_t *kv_empty = kv_full + L::kStages;
    uint64_t *s_full = kv_empty + L::kStages;  // [2]: one per S buffer
    uint64_t *p_full = s_full + 2;             // [2]: one per S buffer
    uint64_t *pv_done = p_full + 2;
    uint64_t *o_final = pv_done + 1;
    uint64_t *unit_full = o_final + 1;         // [2]
    uint64_t *unit_empty = unit_full + 2;      // [2]
    uint64_t *sched = unit_empty + 2;
    uint64_t *drain = sched + 1;
    void *sched_answer = smem + L::kSchedOff;
    volatile int *unit_slot = reinterpret_cast<volatile int *>(smem + L::kUnitOff);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);
    const long total_rows = static_cast<long>(p.B) * p.H * p.Nq;

    const int warp = warp_id(), lane = lane_id();
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 4);   // the four softmax warps
            mbar_init(&unit_full[b], 1);
            mbar_init(&unit_empty[b], 5);  // the MMA warp and the four softmax warps
        }
        mbar_init(pv_done, 1);
        mbar_init(o_final, 1);
        mbar_init(sched, 1);
        mbar_init(drain, 1);
        unit_slot[0] = static_cast<int>(blockIdx.x);  // the first unit is this CTA's own
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the range merge queued after this grid may take its SM slots early (it waits for this
    // grid's completion before it reads a partial result)
    if (threadIdx.x == 0) griddep_launch_dependents();

    if (warp == 0) {
        // ---------------------------------------------------------------- load warp
        // The whole warp walks the units; lane 0 issues the copies and requests.
        if (lane == 0) mbar_arrive(&unit_full[0]);
        int unit = static_cast<int>(blockIdx.x);
        int n = 0;     // K/V tile pairs issued
        int nq = 0;    // Q tiles issued
        int nreq = 0;  // scheduler requests made
        bool more = true;
        bool ok = true;
        for (int k = 0;; ++k) {
            const DecUnit u = dec_unit(p, unit);
            auto load_q = [&]() {  // the Q tile is free once the previous unit's last S is done
                if (nq > 0 && !mbar_wait_warp(q_empty, (nq - 1) & 1, p.ctl, abort_flag))
                    return false;
                if (lane == 0) {
                    mbar_arrive_expect_tx(q_full, L::kTileBytes);
                    for (int b = 0; b < L::kBoxes; ++b)
                        tma_load_3d(smem + L::kQOff + b * L::kBoxBytes, &tmq, b * 64,
                                    static_cast<int>(u.grow0), 0, q_full);
                }
                ++nq;
                return true;
            };
            bool q_done = false;
            for (int t = 0; t < u.ntiles && ok; ++t) {
                const int s = n % L::kStages;
                if (!mbar_wait_warp(&kv_empty[s], ((n / L::kStages) & 1) ^ 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    // keys past the cache's capacity read as zeros; keys past the range or the
                    // sequence length are masked in the softmax
                    const int key0 = u.k_begin + kDecTile * t;
                    uint8_t *kd = smem + L::kRingOff + s * 2 * L::kTileBytes;
                    mbar_arrive_expect_tx(&kv_full[s], 2 * L::kTileBytes);
                    for (int b = 0; b < L::kBoxes; ++b) {
                        tma_load_3d(kd + b * L::kBoxBytes, &tmk, b * 64, key0, u.kvh, &kv_full[s]);
                        tma_load_3d(kd + L::kTileBytes + b * L::kBoxBytes, &tmv, b * 64, key0,
                                    u.kvh, &kv_full[s]);
                    }
                }
                ++n;
                // the first K/V tile goes ahead of Q: its slot frees before the Q tile does
                if (!q_done) {
                    ok = load_q();
                    q_done = true;
                }
            }
            if (ok && !q_done) ok = load_q();  // a unit without keys still takes its Q turn
            if (!ok) break;
            // next unit: a CTA of this grid that has not started, cancelled for us
            int next = -1;
            if (more) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(sched, 16);
                    clc_try_cancel(sched_answer, sched);
                }
                ++nreq;
                if (!mbar_wait_warp(sched, (nreq - 1) & 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                next = clc_cancelled_x(sched_answer);
                if (next >= static_cast<int>(gridDim.x)) next = -1;
                more = next >= 0;
            }
            // publish it (or the end) in slot (k + 1) & 1, once unit k - 1 has released it
            const int e2 = (k + 1) & 1;
            if (k >= 1 && !mbar_wait_warp(&unit_empty[e2], ((k + 1) / 2 - 1) & 1, p.ctl,
                                          abort_flag)) {
                ok = false;
                break;
            }
            __syncwarp();
            if (lane == 0) {
                unit_slot[e2] = next;
                mbar_arrive(&unit_full[e2]);
            }
            if (next < 0) break;
            unit = next;
        }
        if (!ok || *abort_flag) {
            // let every copy and request still in flight land before shared memory goes away
            if (lane == 0) {
                if (nq > 0) drain_wait(q_full, (nq - 1) & 1, p.ctl);
                if (nreq > 0) drain_wait(sched, (nreq - 1) & 1, p.ctl);
                for (int l = n > L::kStages ? n - L::kStages : 0; l < n; ++l)
                    drain_wait(&kv_full[l % L::kStages], (l / L::kStages) & 1, p.ctl);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        const SDesc dq = sdesc_make(smem_u32(smem + L::kQOff), 16, 1024);       // Q: K-major
        const SDesc dk0 = sdesc_make(smem_u32(smem + L::kRingOff), 16, 1024);   // K: K-major
        const SDesc dv0 = sdesc_make(smem_u32(smem + L::kRingOff + L::kTileBytes), L::kBoxBytes,
                                     1024);                                      // V: MN-major
        int n = 0;  // K/V tile pairs used (all units): tile n's S goes into buffer n % 2
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int e = k & 1;
            if (!mbar_wait_warp(&unit_full[e], (k >> 1) & 1, p.ctl, abort_flag)) {
                ok = false;
                break;
            }
            const int unit = unit_slot[e];
            if (unit < 0) break;
            const DecUnit u = dec_unit(p, unit);
            if (!mbar_wait_warp(q_full, k & 1, p.ctl, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            auto issue_s = [&](int t) -> bool {  // S of the unit's tile t (ring tile n + t)
                const int g = n + t;
                const int s = g % L::kStages;
                if (!mbar_wait_warp(&kv_full[s], (g / L::kStages) & 1, p.ctl, abort_flag))
                    return false;
                tc_fence_after();
                const SDesc b = sdesc_add(dk0, s * 2 * L::kTileBytes);
                if constexpr (D == 128)
                    mma_ss_chain_k128(tmem + (g & 1) * 128, dq, b, kIdescS, 0u);
                else
                    mma_ss_chain_k64(tmem + (g & 1) * 128, dq, b, kIdescS, 0u);
                umma_commit_el(&s_full[g & 1]);
                if (t == u.ntiles - 1) umma_commit_el(q_empty);  // the unit's last S: Q is free
                return true;
            };
            if (u.ntiles == 0) {
                umma_commit_el(q_empty);
            } else if (!issue_s(0)) {
                ok = false;
                break;
            }
            for (int t = 0; ok && t < u.ntiles; ++t) {
                if (t + 1 < u.ntiles && !issue_s(t + 1)) {  // S_{t+1} ahead of PV_t
                    ok = false;
                    break;
                }
                const int g = n + t;
                if (!mbar_wait_warp(&p_full[g & 1], (g >> 1) & 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int s = g % L::kStages;
                mma_ts_chain_k128(tmem + 256, tmem + (g & 1) * 128,
                                  sdesc_add(dv0, s * 2 * L::kTileBytes), kIdescPV, t > 0 ? 1u : 0u);
                umma_commit_el(pv_done);
                umma_commit_el(&kv_empty[s]);
            }
            if (!ok) break;
            n += u.ntiles;
            if (u.ntiles > 0) umma_commit_el(o_final);
            __syncwarp();
            if (lane == 0) mbar_arrive(&unit_empty[e]);
        }
        // every MMA issued above completes before the CTA releases TMEM and smem
        umma_commit_el(drain);
        drain_wait(drain, 0, p.ctl);
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- softmax warps
        using T = elem_t<BF16>;
        const int quad = warp & 3;  // a warp may touch TMEM lanes [32*(warp%4), +32)
        const int row = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tO = tmem + lane_base + 256;
        const float sl2 = p.scale_log2;
        int g = 0;     // K/V tiles consumed (all units)
        int nfin = 0;  // units with keys (o_final phases)
        for (int k = 0;; ++k) {
            const int e = k & 1;
            if (!mbar_wait_warp(&unit_full[e], (k >> 1) & 1, p.ctl, abort_flag)) break;
            const int unit = unit_slot[e];
            if (unit < 0) break;
            const DecUnit u = dec_unit(p, unit);
            const bool busy = quad * 32 < u.nrows;  // this quarter holds real rows
            // the last key this row may see: its own position when causal (new rows end-aligned
            // with the cache), the sequence's last key otherwise
            const int gr = u.r0 + row;
            const int last = p.causal ? u.len - p.Nq + gr % p.Nq : u.len - 1;
            float m = -INFINITY;  // running (reference) max of the scaled scores, log2 units
            float l = 0.f;        // running sum of exp2(score - m)
            bool ok = true;
            for (int t = 0; t < u.ntiles; ++t, ++g) {
                if (!mbar_wait_warp(&s_full[g & 1], (g >> 1) & 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (busy) {
                    const uint32_t tS = tmem + lane_base + (g & 1) * 128;
                    uint32_t r[128];
                    tmem_ld32(tS + 0, r + 0);
                    tmem_ld32(tS + 32, r + 32);
                    tmem_ld32(tS + 64, r + 64);
                    tmem_ld32(tS + 96, r + 96);
                    tmem_wait_ld();
                    const int kv0 = u.k_begin + kDecTile * t;
                    const int lim = min(u.k_end - 1, last);  // keys above lim are masked
                    if (kv0 + kDecTile - 1 > lim) {
#pragma unroll
                        for (int c = 0; c < 128; ++c)
                            if (kv0 + c > lim) r[c] = __float_as_uint(-INFINITY);
                    }
                    const float m_tile = row_max128(r) * sl2;
                    const float m_new = fmaxf(m, m_tile);
                    const bool old_finite = m != -INFINITY;
                    const bool grow = m_new > m + 8.0f;
                    float alpha = 1.f;
                    if (grow) {
                        if (old_finite) alpha = ex2(m - m_new);
                        l *= alpha;
                        m = m_new;
                    }
                    const bool rescale = grow && old_finite;
                    const float mu = m == -INFINITY ? 0.f : m;  // a row with nothing unmasked yet
                    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                     make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    const float2 sc2 = make_float2(sl2, sl2), mu2 = make_float2(-mu, -mu);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t pk[32];
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            const float2 x = ffma2(make_float2(__uint_as_float(r[64 * h + 2 * c]),
                                                               __uint_as_float(r[64 * h + 2 * c + 1])),
                                                   sc2, mu2);
                            const float2 ev = make_float2(ex2(x.x), ex2(x.y));
                            acc[c & 3] = fadd2(acc[c & 3], ev);
                            pk[c] = pack2<BF16>(ev.x, ev.y);
                        }
                        tmem_st32(tS + 32 * h, pk);
                    }
                    const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
                    const float2 a = fadd2(a01, a23);
                    l += a.x + a.y;
                    if (__any_sync(0xffffffffu, rescale)) {
                        // O holds the products up to PV_{t-1}, which S_t did not wait for: let
                        // it complete before O is rescaled (the next PV waits for p_full)
                        if (!mbar_wait_warp(pv_done, (g - 1) & 1, p.ctl, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int cc = 0; cc < D / 32; ++cc) {
                            uint32_t o[32];
                            tmem_ld32(tO + cc * 32, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int x = 0; x < 32; ++x)
                                o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
                            tmem_st32(tO + cc * 32, o);
                        }
                    }
                }
                mbar_arrive_warp_after_st(&p_full[g & 1]);
            }
            if (!ok) break;
            if (u.ntiles > 0) {
                if (!mbar_wait_warp(o_final, nfin & 1, p.ctl, abort_flag)) break;
                ++nfin;
                tc_fence_after();
            }
            // rows of this unit: O = O~ / l and LSE, or the range's partial (m, l, O~); the
            // tensor-memory loads are warp-wide, the stores only for real rows
            if (busy) {
                const bool real = row < u.nrows;
                const long grow = u.grow0 + row;
                const long prow = static_cast<long>(u.split) * total_rows + grow;
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    if (u.ntiles > 0) {
                        tmem_ld32(tO + cc * 32, o);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int x = 0; x < 32; ++x) o[x] = 0u;
                    }
                    if (!real) continue;
                    if (p.splits == 1) {
                        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.o) +
                                                               grow * D + cc * 32);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint32_t w[4];
#pragma unroll
                            for (int x = 0; x < 4; ++x)
                                w[x] = pack2<BF16>(__uint_as_float(o[8 * q4 + 2 * x]) * inv,
                                                   __uint_as_float(o[8 * q4 + 2 * x + 1]) * inv);
                            dst[q4] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    } else {
                        float4 *dst = reinterpret_cast<float4 *>(p.part_o + prow * D + cc * 32);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            dst[q4] = make_float4(__uint_as_float(o[4 * q4]), __uint_as_float(o[4 * q4 + 1]),
                                                  __uint_as_float(o[4 * q4 + 2]),
                                                  __uint_as_float(o[4 * q4 + 3]));
                    }
                }
                if (real) {
                    if (p.splits == 1)
                        p.lse[grow] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
                    else
                        reinterpret_cast<float2 *>(p.part_ml)[prow] = make_float2(m, l);
                }
            }
            // O has been read out (the next unit's first PV waits for this warp's next p_full
            // arrival); the unit slot is no longer needed
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&unit_empty[e]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
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

template <int D, bool BF16>
cudaError_t launch_decode_t(const DecodeMaps &m, const DecodeParams &p, cudaStream_t stream) {
    using L = DecLayout<D>;
    auto kern = fa_decode_kernel<D, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kAlloc);
    if (e != cudaSuccess) return e;
    const long grid = static_cast<long>(p.B) * p.Hkv * p.splits * p.row_groups;
    kern<<<static_cast<unsigned>(grid), L::kThreads, L::kAlloc, stream>>>(m.q, m.k, m.v, p);
    e = cudaGetLastError();
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
