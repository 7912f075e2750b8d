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
//   CTA = two query tiles of one head (256 rows), 384 threads, one CTA per SM:
//     warp 0       TMA producer: Q tiles once, then K_j and V_j into a ring of smem slots
//     warp 1       MMA issuer (one elected lane): S_t = Q_t K_j^T (SS), O_t += P_t V_j (TS, P in
//                  TMEM); warps 2, 3 idle, so that warps 0..3 form a warpgroup that hands
//                  registers to the softmax warpgroups (setmaxnreg: 64 vs 216 per thread)
//     warps 4..7   softmax for query tile 0, one TMEM lane (= query row) per thread
//     warps 8..11  softmax for query tile 1
//   TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+d), O_1 [256+d,256+2d).
//   P_t is written as packed 16-bit pairs over the first 64 columns of S_t and read from
//   there by the PV MMA, so P never touches shared memory.
//   MMA issue order per key tile j: PV_0(j-1), S_0(j), PV_1(j-1), S_1(j): while one softmax
//   group exponentiates, the tensor core works on the other group's products.
//   The row max is a tree of three-input maxima; exponent arguments and row sums use paired
//   fp32 instructions (f32x2).  The running max is kept in log2 units; O and l are rescaled only when the max grows by more
//   than 8 (a factor 256).  This is exact: O~ and l always share the same reference max, and the
//   final O~/l and L = m + log2(l) (converted to natural log) do not depend on which max it is.
#include "fa_internal.h"

#include <cmath>
#include <type_traits>

namespace fa {
namespace {

template <int D>
struct FwdLayout {
    static constexpr int kTileBytes = kTile * D * 2;  // one 128 x d tile of 16-bit values
    static constexpr int kBoxes = D / 64;             // 128-byte-wide TMA boxes per tile row
    static constexpr int kBoxBytes = kTile * 128;     // 16 KB
    static constexpr int kSlots = (D == 128) ? 4 : 8; // K/V ring slots
    static constexpr int kQOff = 0;
    static constexpr int kSlotOff = 2 * kTileBytes;
    static constexpr int kBarOff = kSlotOff + kSlots * kTileBytes;
    // q_full, full[kSlots], empty[kSlots], s_full[2], p_full[2], o_final[2], drain
    static constexpr int kNumBars = 1 + 2 * kSlots + 7;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kMaskOff = kMiscOff + 16;  // block-mask bits of the two query tiles
    static constexpr int kBytes = kMaskOff + 2 * kMaskSmemWords * 4;
    static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024 bytes
    static constexpr int kThreads = 384;
    static constexpr uint32_t kTmemCols = 512;
};

template <int D, bool BF16, bool DROP>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv,
                  const __grid_constant__ CUtensorMap tmo, const FwdParams p) {
    using L = FwdLayout<D>;
    constexpr uint32_t kIdescPV = idesc_f16(128, D, BF16, true);
    constexpr uint32_t kIdescS = idesc_f16(128, 128, BF16, false);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *q_full = bars;
    uint64_t *full = bars + 1;
    uint64_t *empty = full + L::kSlots;
    uint64_t *s_full = empty + L::kSlots;
    uint64_t *p_full = s_full + 2;
    uint64_t *o_final = p_full + 2;
    uint64_t *drain = o_final + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);

    const int warp = warp_id(), lane = lane_id();
    const CtaOrder ord = cta_order(blockIdx.x, p.BH, p.num_pairs, p.head_group);
    const int bh = ord.head;
    const int pair = p.num_pairs - 1 - ord.rank;  // long rows first
    const int qt0 = 2 * pair, qt1 = 2 * pair + 1;
    const bool has1 = qt1 < p.T;
    const int jend = p.causal ? min(has1 ? qt1 : qt0, p.T - 1) + 1 : p.T;
    const int kvh = bh / p.rep;  // K/V head shared by this query head's group

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < L::kSlots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 4);  // one arrival per softmax warp
            mbar_init(&o_final[t], 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, L::kTmemCols);
        tmem_relinquish();
    }
    // mask rows of qt0 and qt1, kMaskSmemWords words each
    uint32_t *const mrow0 = reinterpret_cast<uint32_t *>(smem + L::kMaskOff);
    uint32_t *const mrow1 = mrow0 + kMaskSmemWords;
    if (p.mask != nullptr && p.T <= kMaskSmemTiles) {
        mask_bits_load(mrow0, p.mask + static_cast<long>(qt0) * p.T, 1, p.T);
        if (has1) mask_bits_load(mrow1, p.mask + static_cast<long>(qt1) * p.T, 1, p.T);
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
            // ---------------------------------------------------------------- TMA producer
            if (lane == 0) {
                uint8_t *sQ = smem + L::kQOff;
                mbar_arrive_expect_tx(q_full, (has1 ? 2 : 1) * L::kTileBytes);
                for (int t = 0; t < (has1 ? 2 : 1); ++t)
                    for (int b = 0; b < L::kBoxes; ++b)
                        tma_load_3d(sQ + t * L::kTileBytes + b * L::kBoxBytes, &tmq, b * 64,
                                    (qt0 + t) * kTile, bh, q_full);
                int n = 0;
                bool ok = true;
                for (int j = 0; j < jend && ok; ++j) {
                    if (!tile_live(p, mrow0, qt0, j) && !tile_live(p, mrow1, qt1, j)) continue;
                    for (int kv = 0; kv < 2; ++kv) {
                        const int s = n % L::kSlots;
                        const uint32_t par = ((n / L::kSlots) & 1) ^ 1;
                        if (!mbar_wait(&empty[s], par, p.ctl, abort_flag)) {
                            ok = false;
                            break;
                        }
                        if (!(p.ctl.fault_mode == 1 && n == 0)) {
                            mbar_arrive_expect_tx(&full[s], L::kTileBytes);
                            uint8_t *dst = smem + L::kSlotOff + s * L::kTileBytes;
                            for (int b = 0; b < L::kBoxes; ++b)
                                tma_load_3d(dst + b * L::kBoxBytes, kv ? &tmv : &tmk, b * 64,
                                            j * kTile, kvh, &full[s]);
                        }
                        ++n;
                    }
                }
                if (!ok || *abort_flag) {
                    // let every copy still in flight land before the CTA's shared memory goes away
                    drain_wait(q_full, 0, p.ctl);
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
            {
                const uint32_t sQ = smem_u32(smem + L::kQOff);
                const uint32_t sSlots = smem_u32(smem + L::kSlotOff);
                bool ok = mbar_wait_warp(q_full, 0, p.ctl, abort_flag);
                tc_fence_after();
                int n = 0;
                int cnt[2] = {0, 0};
                int prev_j = -1;
                bool prev_live[2] = {false, false};
                int prev_vs = 0;
                uint32_t prev_vpar = 0;

                // descriptors of the Q tiles and of slot 0; a slot or k-step only adds an offset
                const SDesc dq0 = sdesc_make(sQ, 16, 1024);
                const SDesc dk0 = sdesc_make(sSlots, 16, 1024);                // K: K-major
                const SDesc dv0 = sdesc_make(sSlots, L::kBoxBytes, 1024);      // V: MN-major
                auto issue_s = [&](int t, int ks) {
                    const SDesc a = sdesc_add(dq0, t * L::kTileBytes);
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

                for (int j = 0; ok && j < jend; ++j) {
                    const bool lv[2] = {tile_live(p, mrow0, qt0, j), tile_live(p, mrow1, qt1, j)};
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
                            if (!mbar_wait_warp(&p_full[t], cnt[t] & 1, p.ctl, abort_flag)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            issue_pv(t, prev_vs, cnt[t] > 0);
                            ++cnt[t];
                        }
                        if (lv[t]) {
                            issue_s(t, ks);
                            umma_commit_el(&s_full[t]);
                            if (p.ctl.visit_log != nullptr && lane == 0)
                                visit_mark(p.ctl.visit_log,
                                           (static_cast<size_t>(bh) * p.T + (qt0 + t)) * p.T + j, 1u);
                        }
                    }
                    if (!ok) break;
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
                        if (!mbar_wait_warp(&p_full[t], cnt[t] & 1, p.ctl, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_pv(t, prev_vs, cnt[t] > 0);
                        ++cnt[t];
                    }
                    if (ok) umma_commit_el(&empty[prev_vs]);
                }
                if (ok) {
                    for (int t = 0; t < 2; ++t)
                        if (cnt[t] > 0) umma_commit_el(&o_final[t]);
                }
                // every MMA issued above completes before the CTA releases TMEM and smem
                umma_commit_el(drain);
                drain_wait(drain, 0, p.ctl);
            }
            __syncwarp();
        }
    } else {
        regs_inc<216>();
        // ---------------------------------------------------------------- softmax groups
        const int t = (warp - 4) >> 2;
        const int quad = warp & 3;  // a warp may touch TMEM lanes [32*(warp%4), +32)
        const int row = quad * 32 + lane;
        const int qt = t == 0 ? qt0 : qt1;
        const uint32_t *mrow = t == 0 ? mrow0 : mrow1;
        const int q_row = qt * kTile + row;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_base + t * 128;
        const uint32_t tO = tmem + lane_base + 256 + t * D;
        const float sl2 = p.scale_log2;
        float m = -INFINITY;  // running (reference) max of the scaled scores, log2 units
        float l = 0.f;        // running sum of exp2(score - m)
        int cnt = 0;
        bool ok = true;
        for (int j = 0; j < jend; ++j) {
            if (!tile_live(p, mrow, qt, j)) continue;
            uint32_t keep[4];  // dropout: keep bits of keys 32w .. 32w + 31 of this tile, drawn
            if constexpr (DROP) {  // while the tensor core still works on S
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    keep[w] = philox_keep_bits(4u * j + w, q_row, bh, p.drop);
            }
            if (!mbar_wait_warp(&s_full[t], cnt & 1, p.ctl, abort_flag)) {
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
            // P~ = 2^(s * scale * log2(e) - mu) in pairs; l sums every probability (only PV sees
            // the dropped ones); masked scores (-inf) give exactly 0
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
            const float2 sc2 = make_float2(sl2, sl2), mu2 = make_float2(-mu, -mu);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float2 x = ffma2(make_float2(__uint_as_float(r[64 * h + 2 * c]),
                                                       __uint_as_float(r[64 * h + 2 * c + 1])),
                                           sc2, mu2);
                    const float2 e = make_float2(ex2(x.x), ex2(x.y));
                    acc[c & 3] = fadd2(acc[c & 3], e);
                    pk[c] = pack2<BF16>(e.x, e.y);
                    if constexpr (DROP) pk[c] = keep_halves(pk[c], keep[2 * h + (c >> 4)], c & 15);
                }
                tmem_st32(tS + 32 * h, pk);
            }
            const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
            const float2 a = fadd2(a01, a23);
            const float rs0 = a.x, rs1 = a.y;
            l += rs0 + rs1;
            if (__any_sync(0xffffffffu, rescale)) {
                // The previous PV into O_t has completed (its commit preceded this S_t) and the
                // next one waits for p_full, so O_t is ours to rescale here.
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tO + cc * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(tO + cc * 32, o);
                }
            }
            mbar_arrive_warp_after_st(&p_full[t]);
            ++cnt;
        }
        if (ok && cnt > 0) {
            ok = mbar_wait_warp(&o_final[t], 0, p.ctl, abort_flag);
            tc_fence_after();
        }
        // A tile without live key tiles stages zeros: its Q tile must have landed first.
        if (ok && cnt == 0) ok = mbar_wait_warp(q_full, 0, p.ctl, abort_flag);
        // O_t = O~_t / l is staged as a 16-bit tile over Q_t (no MMA reads Q_t any more: every
        // S_t was issued before the final PV_t) and written by TMA.  All four warps of the group
        // reach the named barrier, whether or not their waits succeeded.
        uint8_t *stage = smem + L::kQOff + t * L::kTileBytes;
        if (ok) {
            const float inv = l > 0.f ? (DROP ? p.drop.keep_scale : 1.f) / l : 0.f;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                if (cnt > 0) {
                    tmem_ld32(tO + cc * 32, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                st_box_row<BF16, 32>(stage + (cc >> 1) * L::kBoxBytes, row, (cc & 1) * 32, o, inv);
            }
            fence_proxy_async_smem();
            if (q_row < p.N)
                p.lse[static_cast<size_t>(bh) * p.N + q_row] =
                    l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
        named_sync(1 + t, 128);
        if (quad == 0 && lane == 0 && ok && *abort_flag == 0 && qt * kTile < p.N) {
            for (int b = 0; b < L::kBoxes; ++b)
                tma_store_3d(&tmo, stage + b * L::kBoxBytes, b * 64, qt * kTile, bh);
            bulk_commit();
            bulk_wait_read_all();
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
                                                                           maps.out0, p);
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
