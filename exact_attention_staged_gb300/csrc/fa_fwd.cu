// fa_fwd.cu - fused exact-attention forward for sm_103a (tcgen05 + TMA + TMEM).
//
// Computes, per (batch, head) and per 128-row query tile Q_i, the FlashAttention-2 forward
// ("FlashAttention-2: better parallelism and work partitioning" reading notes, Algorithm 1):
// S_ij = Q_i K_j^T on the tensor cores into tensor memory, the online softmax statistics
// (m, l) in fp32 with one thread per row, P~_ij = exp(S_ij - m) rounded to the input type,
// O~_i += P~_ij V_j on the tensor cores, and once per row O_i = O~_i / l_i and
// L_i = m_i + ln(l_i) (delayed normalisation eq. (10)-(11), logsumexp eq. (15)).  Neither S nor
// P ever leaves the SM.  Causal tiles above the diagonal and tiles whose block-mask entry is
// zero are never loaded nor multiplied (FlashAttention-2 notes, causal masking section;
// FlashAttention post, "Block-Sparse FlashAttention").
//
// GB300 mapping (prior art on the pages is A100 mma.sync with warp split-Q; not used here):
//   work unit = two query tiles of one head (256 rows); the grid has one CTA per unit, but a
//   CTA that runs keeps taking the units of CTAs that have not started (cluster launch
//   control), so in practice one CTA per SM walks a sequence of units; 384 threads:
//     warp 0       load warp: per unit the Q tiles, then K_j and V_j into a ring of smem slots;
//                  it also asks the hardware for the next unit and publishes it (with the
//                  unit's block-mask rows) in one of two unit slots
//     warp 1       MMA issuer (one elected lane): S_t = Q_t K_j^T (SS), O_t += P_t V_j (TS, P in
//                  TMEM); warps 2, 3 idle, so that warps 0..3 form a warpgroup that hands
//                  registers to the softmax warpgroups (setmaxnreg: 64 vs 216 per thread)
//     warps 4..7   softmax for query tile 0, one TMEM lane (= query row) per thread; at the end
//                  of a unit each thread stores its row of O and its LSE
//     warps 8..11  softmax for query tile 1
//   TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+d), O_1 [256+d,256+2d).
//   P_t is written as packed 16-bit pairs over the first 64 columns of S_t and read from
//   there by the PV MMA, so P never touches shared memory.
//   MMA issue order per key tile j: PV_0(j-1), S_0(j), PV_1(j-1), S_1(j): while one softmax
//   group exponentiates, the tensor core works on the other group's products.
//   The row max is a tree of three-input maxima; exponent arguments and row sums use paired
//   fp32 instructions (f32x2).  The running max is kept in log2 units; O and l are rescaled
//   only when the max grows by more than 8 (a factor 256).  This is exact: O~ and l always share the same reference max, and the
//   final O~/l and L = m + log2(l) (converted to natural log) do not depend on which max it is.
#include "fa_internal.h"

#include <cmath>
#include <type_traits>

namespace fa {
namespace {

// Block-mask rows are copied to shared memory as bits when the mask is at most this many tiles
// wide (two rows for each of the two unit slots); wider masks are read from global memory.
constexpr int kFwdMaskTiles = 2048;
constexpr int kFwdMaskWords = kFwdMaskTiles / 32;

template <int D>
struct FwdLayout {
    static constexpr int kTileBytes = kTile * D * 2;  // one 128 x d tile of 16-bit values
    static constexpr int kBoxes = D / 64;             // 128-byte-wide TMA boxes per tile row
    static constexpr int kBoxBytes = kTile * 128;     // 16 KB
    static constexpr int kSlots = (D == 128) ? 4 : 8; // K/V ring slots
    static constexpr int kQSets = (D == 128) ? 1 : 2; // Q tile pairs: units k, k + 1 at d = 64
    static constexpr int kQOff = 0;                   // [kQSets][Q_0, Q_1]
    static constexpr int kSlotOff = kQSets * 2 * kTileBytes;
    static constexpr int kBarOff = kSlotOff + kSlots * kTileBytes;
    // q_full[2], q_empty[2], full[kSlots], empty[kSlots], s_full[2], p_full[2], o_final[2],
    // unit_full[2], unit_empty[2], sched, drain
    static constexpr int kNumBars = 4 + 2 * kSlots + 12;
    static constexpr int kSchedOff = (kBarOff + kNumBars * 8 + 15) / 16 * 16;  // 16-byte answer
    static constexpr int kUnitOff = kSchedOff + 16;   // int unit[2]: the two unit slots
    static constexpr int kMiscOff = kUnitOff + 8;     // TMEM base, abort flag
    static constexpr int kMaskOff = kMiscOff + 8;     // bits [unit slot][query tile][words]
    static constexpr int kBytes = kMaskOff + 4 * kFwdMaskWords * 4;
    static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024 bytes
    static constexpr int kThreads = 384;
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kAlloc <= 232448, "shared memory per CTA");
};

// One work unit: two consecutive query tiles of one query head.
struct FwdUnit {
    int bh, qt0, qt1, jend, kvh;
    bool has1;
};
__device__ __forceinline__ FwdUnit fwd_unit(const FwdParams &p, int unit) {
    const CtaOrder ord = cta_order(static_cast<unsigned>(unit), p.BH, p.num_pairs, p.head_group);
    FwdUnit u;
    u.bh = ord.head;
    const int pair = p.num_pairs - 1 - ord.rank;  // long rows first
    u.qt0 = 2 * pair;
    u.qt1 = 2 * pair + 1;
    u.has1 = u.qt1 < p.T;
    u.jend = p.causal ? min(u.has1 ? u.qt1 : u.qt0, p.T - 1) + 1 : p.T;
    u.kvh = u.bh / p.rep;  // K/V head shared by this query head's group
    return u;
}

// Is key tile j live for query tile qt?  bits: the query tile's mask row in shared memory.
__device__ __forceinline__ bool fwd_live(const FwdParams &p, const uint32_t *bits, int qt, int j) {
    if (qt >= p.T) return false;
    if (p.causal && j > qt) return false;
    if (p.mask == nullptr) return true;
    return p.T <= kFwdMaskTiles ? mask_bit(bits, j) : p.mask[qt * p.T + j] != 0;
}

// One warp copies the mask rows of query tiles qt0 and qt1 as bits: lane i reads bytes i, i + 32,
// ... (each warp-wide read is 32 consecutive bytes) and a ballot turns 32 of them into a word;
// eight words' reads are issued before the first ballot, so a row of up to 128 tiles costs one
// round trip to memory.
__device__ __forceinline__ void fwd_mask_rows(const FwdParams &p, uint32_t *bits0, int qt0,
                                              uint32_t *bits1, int qt1) {
    if (p.mask == nullptr || p.T > kFwdMaskTiles) return;
    const int lane = lane_id();
    const int words = (p.T + 31) / 32;
    for (int r = 0; r < 2; ++r) {
        const int qt = r == 0 ? qt0 : qt1;
        if (qt >= p.T) continue;
        uint32_t *bits = r == 0 ? bits0 : bits1;
        const uint8_t *src = p.mask + static_cast<long>(qt) * p.T;
        for (int w0 = 0; w0 < words; w0 += 8) {
            uint8_t b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int idx = 32 * (w0 + i) + lane;
                b[i] = (w0 + i < words && idx < p.T) ? src[idx] : 0;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t word = __ballot_sync(0xffffffffu, b[i] != 0);
                if (lane == 0 && w0 + i < words) bits[w0 + i] = word;
            }
        }
    }
}

// Persistent forward.  The grid has one CTA per unit (query-tile pair) in the CTA order; the
// CTAs that start run unit after unit, each next unit taken from the hardware's queue of CTAs
// not yet started (cluster launch control), so the CTA's setup is paid once per SM and the
// next unit's loads and first products overlap the end of the current one.  Unit slots in
// shared memory carry the unit index and its mask rows from the load warp to the MMA warp and
// the softmax groups.  Q is reloaded once the last S of the unit that used its buffer has been
// computed (two Q buffers at d = 64, so the next unit's Q lands while the current one runs), and
// each softmax thread stores its row of O straight from registers, so a unit's epilogue holds
// up neither the other query tile nor the next unit's products.
template <int D, bool BF16, bool DROP>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const FwdParams p) {
    using L = FwdLayout<D>;
    constexpr uint32_t kIdescPV = idesc_f16(128, D, BF16, true);
    constexpr uint32_t kIdescS = idesc_f16(128, 128, BF16, false);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *q_full = bars;
    uint64_t *q_empty = bars + 2;
    uint64_t *full = bars + 4;
    uint64_t *empty = full + L::kSlots;
    uint64_t *s_full = empty + L::kSlots;
    uint64_t *p_full = s_full + 2;
    uint64_t *o_final = p_full + 2;
    uint64_t *unit_full = o_final + 2;
    uint64_t *unit_empty = unit_full + 2;
    uint64_t *sched = unit_empty + 2;
    uint64_t *drain = sched + 1;
    void *sched_answer = smem + L::kSchedOff;
    volatile int *unit_slot = reinterpret_cast<volatile int *>(smem + L::kUnitOff);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);
    uint32_t *mask_bits = reinterpret_cast<uint32_t *>(smem + L::kMaskOff);
    // mask row of query tile t (0, 1) of the unit in slot e
    auto mrow = [&](int e, int t) { return mask_bits + (2 * e + t) * kFwdMaskWords; };

    const int warp = warp_id(), lane = lane_id();
    if (threadIdx.x == 0) {
        for (int q = 0; q < 2; ++q) {
            mbar_init(&q_full[q], 1);
            mbar_init(&q_empty[q], 1);
        }
        for (int s = 0; s < L::kSlots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 4);  // one arrival per softmax warp
            mbar_init(&o_final[t], 1);
            mbar_init(&unit_full[t], 1);
            mbar_init(&unit_empty[t], 9);  // the MMA warp and the eight softmax warps
        }
        mbar_init(sched, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        // the first unit is this CTA's own
        const FwdUnit u = fwd_unit(p, blockIdx.x);
        fwd_mask_rows(p, mrow(0, 0), u.qt0, mrow(0, 1), u.qt1);
        if (lane == 0) {
            unit_slot[0] = static_cast<int>(blockIdx.x);
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // a backward pre-pass queued after this grid with programmatic stream serialization may
    // start on the SMs this grid's last CTAs leave idle; it waits for this grid before reading
    if (threadIdx.x == 0) griddep_launch_dependents();
    // warpgroup 0 (load warp, MMA warp, two idle warps) gives registers to the two softmax
    // warpgroups: 128 x 64 + 256 x 216 = 63488 of the 384 x 168 = 64512 the CTA is launched with
    if (warp < 4) {
        regs_dec<64>();
        if (warp == 0) {
            // ---------------------------------------------------------------- load warp
            // The whole warp walks the units; lane 0 issues the copies and requests.
            int unit = static_cast<int>(blockIdx.x);
            if (lane == 0) mbar_arrive(&unit_full[0]);  // slot 0, filled before the CTA barrier
            int k = 0;          // units of this CTA so far
            int n = 0;          // K/V tiles issued into the ring
            int nq = 0;         // Q loads issued
            int nreq = 0;       // scheduler requests made
            bool more = true;   // the hardware may still hand out a unit
            bool ok = true;
            for (;;) {
                const FwdUnit u = fwd_unit(p, unit);
                const int e = k & 1;
                const uint32_t *m0 = mrow(e, 0), *m1 = mrow(e, 1);
                auto load_q = [&]() {
                    // the Q set of this unit is free once the last S of the unit that used it
                    // before (kQSets units back) has been computed
                    const int qs = nq % L::kQSets;
                    if (nq >= L::kQSets && !mbar_wait_warp(&q_empty[qs], (nq / L::kQSets - 1) & 1,
                                                           p.ctl, abort_flag))
                        return false;
                    if (lane == 0) {
                        uint8_t *sQ = smem + L::kQOff + qs * 2 * L::kTileBytes;
                        mbar_arrive_expect_tx(&q_full[qs], (u.has1 ? 2 : 1) * L::kTileBytes);
                        for (int t = 0; t < (u.has1 ? 2 : 1); ++t)
                            for (int b = 0; b < L::kBoxes; ++b)
                                tma_load_3d(sQ + t * L::kTileBytes + b * L::kBoxBytes, &tmq,
                                            b * 64, (u.qt0 + t) * kTile, u.bh, &q_full[qs]);
                    }
                    ++nq;
                    return true;
                };
                // with two Q sets the unit's Q goes first; with one, after the first K/V pair,
                // whose slots free before the Q set does
                bool q_done = false;
                if constexpr (L::kQSets > 1) {
                    ok = load_q();
                    q_done = true;
                }
                for (int j = 0; j < u.jend && ok; ++j) {
                    if (!fwd_live(p, m0, u.qt0, j) && !fwd_live(p, m1, u.qt1, j)) continue;
                    for (int kv = 0; kv < 2; ++kv) {
                        const int s = n % L::kSlots;
                        const uint32_t par = ((n / L::kSlots) & 1) ^ 1;
                        if (!mbar_wait_warp(&empty[s], par, p.ctl, abort_flag)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0 && !(p.ctl.fault_mode == 1 && n == 0)) {
                            mbar_arrive_expect_tx(&full[s], L::kTileBytes);
                            uint8_t *dst = smem + L::kSlotOff + s * L::kTileBytes;
                            for (int b = 0; b < L::kBoxes; ++b)
                                tma_load_3d(dst + b * L::kBoxBytes, kv ? &tmv : &tmk, b * 64,
                                            j * kTile, u.kvh, &full[s]);
                        }
                        ++n;
                    }
                    // the first K/V pair goes ahead of Q: its slots free before Q's does
                    if (ok && !q_done) {
                        ok = load_q();
                        q_done = true;
                    }
                }
                if (ok && !q_done) ok = load_q();  // a unit with nothing live still gets its Q
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
                ++k;
                // publish it (or the end) in slot k & 1, once unit k - 2 has released the slot
                const int e2 = k & 1;
                if (k >= 2 && !mbar_wait_warp(&unit_empty[e2], ((k >> 1) - 1) & 1, p.ctl,
                                              abort_flag)) {
                    ok = false;
                    break;
                }
                if (next >= 0) {
                    const FwdUnit un = fwd_unit(p, next);
                    fwd_mask_rows(p, mrow(e2, 0), un.qt0, mrow(e2, 1), un.qt1);
                }
                __threadfence_block();
                __syncwarp();
                if (lane == 0) {
                    unit_slot[e2] = next;
                    mbar_arrive(&unit_full[e2]);
                }
                if (next < 0) break;
                unit = next;
            }
            if (!ok || *abort_flag) {
                // let every copy and request still in flight land before the CTA's shared
                // memory goes away
                if (lane == 0) {
                    for (int l = nq > L::kQSets ? nq - L::kQSets : 0; l < nq; ++l)
                        drain_wait(&q_full[l % L::kQSets], (l / L::kQSets) & 1, p.ctl);
                    if (nreq > 0) drain_wait(sched, (nreq - 1) & 1, p.ctl);
                    const int first = n > L::kSlots ? n - L::kSlots : 0;
                    for (int l = first; l < n; ++l) {
                        if (p.ctl.fault_mode == 1 && l == 0) continue;
                        drain_wait(&full[l % L::kSlots], (l / L::kSlots) & 1, p.ctl);
                    }
                }
            }
            __syncwarp();
        } else if (warp == 1) {
            // ---------------------------------------------------------------- MMA issuer
            // the whole warp runs this loop in lockstep; one elected lane issues each MMA/commit
            const uint32_t sQ = smem_u32(smem + L::kQOff);
            const uint32_t sSlots = smem_u32(smem + L::kSlotOff);
            // descriptors of the Q tiles and of slot 0; a slot or k-step only adds an offset
            const SDesc dq0 = sdesc_make(sQ, 16, 1024);
            const SDesc dk0 = sdesc_make(sSlots, 16, 1024);                // K: K-major
            const SDesc dv0 = sdesc_make(sSlots, L::kBoxBytes, 1024);      // V: MN-major
            auto issue_s = [&](int qs, int t, int ks) {
                const SDesc a = sdesc_add(dq0, (qs * 2 + t) * L::kTileBytes);
                const SDesc b = sdesc_add(dk0, ks * L::kTileBytes);
                if constexpr (D == 128)
                    mma_ss_chain_k128(tmem + t * 128, a, b, kIdescS, 0u);
                else
                    mma_ss_chain_k64(tmem + t * 128, a, b, kIdescS, 0u);
            };
            auto issue_pv = [&](int t, int vs, bool accumulate) {
                mma_ts_chain_k128(tmem + 256 + t * D, tmem + t * 128,
                                  sdesc_add(dv0, vs * L::kTileBytes), kIdescPV,
                                  accumulate ? 1u : 0u);
            };
            int n = 0;                 // K/V tiles consumed from the ring
            int pcnt[2] = {0, 0};      // PV products issued (p_full phases), per query tile
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int e = k & 1;
                if (!mbar_wait_warp(&unit_full[e], (k >> 1) & 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                const int unit = unit_slot[e];
                if (unit < 0) break;
                const FwdUnit u = fwd_unit(p, unit);
                const uint32_t *m0 = mrow(e, 0), *m1 = mrow(e, 1);
                // the unit's last step with a live tile: Q is free once its S are computed
                int jlast = u.jend - 1;
                while (jlast >= 0 && !fwd_live(p, m0, u.qt0, jlast) && !fwd_live(p, m1, u.qt1, jlast))
                    --jlast;
                const int qs = k % L::kQSets;
                if (!mbar_wait_warp(&q_full[qs], (k / L::kQSets) & 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int p0[2] = {pcnt[0], pcnt[1]};  // PV products before this unit
                int prev_j = -1;
                bool prev_live[2] = {false, false};
                int prev_vs = 0;
                uint32_t prev_vpar = 0;
                for (int j = 0; ok && j <= jlast; ++j) {
                    const bool lv[2] = {fwd_live(p, m0, u.qt0, j), fwd_live(p, m1, u.qt1, j)};
                    if (!lv[0] && !lv[1]) continue;
                    const int ks = n % L::kSlots;
                    const uint32_t kpar = (n / L::kSlots) & 1;
                    const int vs = (n + 1) % L::kSlots;
                    const uint32_t vpar = ((n + 1) / L::kSlots) & 1;
                    if (!mbar_wait_warp(&full[ks], kpar, p.ctl, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    bool v_ready = false;
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (prev_j >= 0 && prev_live[t]) {
                            if (!v_ready) {
                                if (!mbar_wait_warp(&full[prev_vs], prev_vpar, p.ctl, abort_flag)) {
                                    ok = false;
                                    break;
                                }
                                v_ready = true;
                            }
                            if (!mbar_wait_warp(&p_full[t], pcnt[t] & 1, p.ctl, abort_flag)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            issue_pv(t, prev_vs, pcnt[t] > p0[t]);
                            ++pcnt[t];
                        }
                        if (lv[t]) {
                            issue_s(qs, t, ks);
                            umma_commit_el(&s_full[t]);
                            if (p.ctl.visit_log != nullptr && lane == 0)
                                visit_mark(p.ctl.visit_log,
                                           (static_cast<size_t>(u.bh) * p.T + (u.qt0 + t)) * p.T + j,
                                           1u);
                        }
                    }
                    if (!ok) break;
                    if (j == jlast) umma_commit_el(&q_empty[qs]);
                    if (prev_j >= 0) umma_commit_el(&empty[prev_vs]);
                    umma_commit_el(&empty[ks]);
                    prev_j = j;
                    prev_live[0] = lv[0];
                    prev_live[1] = lv[1];
                    prev_vs = vs;
                    prev_vpar = vpar;
                    n += 2;
                }
                if (ok && prev_j >= 0) {
                    bool v_ready = false;
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (!prev_live[t]) continue;
                        if (!v_ready) {
                            ok = mbar_wait_warp(&full[prev_vs], prev_vpar, p.ctl, abort_flag);
                            v_ready = true;
                            if (!ok) break;
                        }
                        if (!mbar_wait_warp(&p_full[t], pcnt[t] & 1, p.ctl, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_pv(t, prev_vs, pcnt[t] > p0[t]);
                        ++pcnt[t];
                    }
                    if (ok) umma_commit_el(&empty[prev_vs]);
                }
                if (!ok) break;
                if (jlast < 0) umma_commit_el(&q_empty[qs]);  // nothing live: Q is free at once
                // O_t of this unit is final (the softmax group waits only when it had steps)
                for (int t = 0; t < 2; ++t)
                    if (pcnt[t] > p0[t]) umma_commit_el(&o_final[t]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&unit_empty[e]);
            }
            // every MMA issued above completes before the CTA releases TMEM and smem
            umma_commit_el(drain);
            drain_wait(drain, 0, p.ctl);
            __syncwarp();
        }
    } else {
        regs_inc<216>();
        // ---------------------------------------------------------------- softmax groups
        const int t = (warp - 4) >> 2;
        const int quad = warp & 3;  // a warp may touch TMEM lanes [32*(warp%4), +32)
        const int row = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_base + t * 128;
        const uint32_t tO = tmem + lane_base + 256 + t * D;
        const float sl2 = p.scale_log2;
        int scnt = 0;  // score tiles consumed by this group (s_full / p_full phases)
        int nfin = 0;  // units whose O_t the MMA warp finished (o_final phases)
        // Each warp walks the units on its own (no group barrier): a warp that gives up sets the
        // CTA's abort flag, so the other warps' next waits give up too.
        for (int k = 0;; ++k) {
            const int e = k & 1;
            if (!mbar_wait_warp(&unit_full[e], (k >> 1) & 1, p.ctl, abort_flag)) break;
            const int unit = unit_slot[e];
            if (unit < 0) break;
            const FwdUnit u = fwd_unit(p, unit);
            const int qt = t == 0 ? u.qt0 : u.qt1;
            const uint32_t *mr = mrow(e, t);
            const int q_row = qt * kTile + row;
            float m = -INFINITY;  // running (reference) max of the scaled scores, log2 units
            float l = 0.f;        // running sum of exp2(score - m)
            int cu = 0;           // score tiles of this unit
            bool ok = true;
            for (int j = 0; j < u.jend; ++j) {
                if (!fwd_live(p, mr, qt, j)) continue;
                // dropout: keep flags of the 64 keys of one half of the tile (keys 32w .. 32w + 31
                // in keep[w % 2]); the first half's are drawn while the tensor core still works
                // on S, the second half's once the first half's P is stored
                uint32_t keep[2][8];
                if constexpr (DROP) {
                    philox_keep_flags(4u * j, q_row, u.bh, p.drop, keep[0]);
                    philox_keep_flags(4u * j + 1, q_row, u.bh, p.drop, keep[1]);
                }
                if (!mbar_wait_warp(&s_full[t], scnt & 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t r[128];
                tmem_ld32(tS + 0, r + 0);
                tmem_ld32(tS + 32, r + 32);
                tmem_ld32(tS + 64, r + 64);
                tmem_ld32(tS + 96, r + 96);
                tmem_wait_ld();
                const int kv0 = j * kTile;
                const bool need_mask = (p.causal && j == qt) || (kv0 + kTile > p.N);
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) {
                        const int col = kv0 + c;
                        if (col >= p.N || (p.causal && col > q_row)) r[c] = __float_as_uint(-INFINITY);
                    }
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
                // P~ = 2^(s * scale * log2(e) - mu) in pairs; l sums every probability (only PV
                // sees the dropped ones); masked scores (-inf) give exactly 0
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
                const float2 sc2 = make_float2(sl2, sl2), mu2 = make_float2(-mu, -mu);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if constexpr (DROP) {
                        if (h == 1) {
                            philox_keep_flags(4u * j + 2, q_row, u.bh, p.drop, keep[0]);
                            philox_keep_flags(4u * j + 3, q_row, u.bh, p.drop, keep[1]);
                        }
                    }
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float2 x = ffma2(make_float2(__uint_as_float(r[64 * h + 2 * c]),
                                                           __uint_as_float(r[64 * h + 2 * c + 1])),
                                               sc2, mu2);
                        const float2 ev = make_float2(ex2(x.x), ex2(x.y));
                        acc[c & 3] = fadd2(acc[c & 3], ev);
                        pk[c] = pack2<BF16>(ev.x, ev.y);
                        if constexpr (DROP)  // keys 64h + 2c, + 1: bytes 2(c % 2), + 1 of word (c % 16) / 2
                                             // of chunk c / 16 of this half
                            pk[c] &= keep_pair_mask(keep[c >> 4][(c & 15) >> 1], 2 * (c & 1));
                    }
                    tmem_st32(tS + 32 * h, pk);
                }
                const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
                const float2 a = fadd2(a01, a23);
                l += a.x + a.y;
                if (__any_sync(0xffffffffu, rescale)) {
                    // The previous PV into O_t has completed (its commit preceded this S_t) and
                    // the next one waits for p_full, so O_t is ours to rescale here.
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(tO + cc * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
                        tmem_st32(tO + cc * 32, o);
                    }
                }
                mbar_arrive_warp_after_st(&p_full[t]);
                ++scnt;
                ++cu;
            }
            if (ok && cu > 0) {
                ok = mbar_wait_warp(&o_final[t], nfin & 1, p.ctl, abort_flag);
                ++nfin;
                tc_fence_after();
            }
            if (!ok) break;
            // O_t = O~_t / l, each thread its own row, stored straight from registers: no
            // staging tile and no barrier, so the group goes on to the next unit at once.  The
            // tensor-memory loads are warp-wide; only the stores depend on the row being < N.
            {
                const bool in = q_row < p.N;
                const float inv = l > 0.f ? (DROP ? p.drop.keep_scale : 1.f) / l : 0.f;
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.o) +
                                                       (static_cast<size_t>(u.bh) * p.N + q_row) * D * 2);
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    if (cu > 0) {
                        tmem_ld32(tO + cc * 32, o);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int x = 0; x < 32; ++x) o[x] = 0u;
                    }
                    if (in) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t w[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                w[i] = pack2<BF16>(__uint_as_float(o[8 * q + 2 * i]) * inv,
                                                   __uint_as_float(o[8 * q + 2 * i + 1]) * inv);
                            dst[cc * 4 + q] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                if (in)
                    p.lse[static_cast<size_t>(u.bh) * p.N + q_row] =
                        l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            }
            // O_t has been read out of tensor memory (the next unit's first PV into it waits
            // for this warp's next p_full arrival); the unit's slot is no longer needed
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

template <int D, bool BF16>
cudaError_t launch_fwd_t(const Maps &maps, const FwdParams &p, cudaStream_t stream) {
    using L = FwdLayout<D>;
    auto kern = p.drop.t4 != 0 ? fa_fwd_kernel<D, BF16, true> : fa_fwd_kernel<D, BF16, false>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    const long grid = static_cast<long>(p.BH) * p.num_pairs;
    kern<<<static_cast<unsigned>(grid), L::kThreads, L::kAlloc, stream>>>(maps.q, maps.k, maps.v,
                                                                           p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const Maps &maps, const FwdParams &p, int d, bool bf16,
                       cudaStream_t stream) {
    if (d == 64) return bf16 ? launch_fwd_t<64, true>(maps, p, stream)
                             : launch_fwd_t<64, false>(maps, p, stream);
    return bf16 ? launch_fwd_t<128, true>(maps, p, stream)
                : launch_fwd_t<128, false>(maps, p, stream);
}

}  // namespace fa
