// fa_fwd_fp8.cu - exact-attention forward on e4m3 (8-bit float) inputs for sm_103a.
//
// The FlashAttention-2 forward of fa_fwd.cu ("FlashAttention-2: better parallelism and work
// partitioning" reading notes, Algorithm 1) with Q, K, V given as e4m3 codes and one scale per
// tensor: S = (Q8 K8^T) * descale_q * descale_k on the tensor cores (tcgen05.mma kind::f8f6f4,
// twice the bf16 rate), the online softmax in fp32 exactly as in fa_fwd.cu, P~ rounded to e4m3
// in tensor memory, O~ += P~ V8 (kind::f8f6f4 again) and O = O~ * descale_v / l, stored as bf16.
//
// Two 8-bit specifics:
//  * The PV product needs V with the key index contiguous (K-major B operand), so a pre-pass
//    (fa_fp8_transpose_v_kernel) writes V^T, [d][N rounded up to 16] per K/V head, zero past N.
//  * P~ is stored as e4m3, whose range is 2^-9 .. 448.  The running max is raised lazily only
//    when it grows by more than kTau = 4 (log2 units) and P~ = 2^(s - m + kOff) with kOff = 4,
//    so P~ <= 2^8 and the largest probabilities of a row sit near the top of the e4m3 range,
//    leaving 17 binades below them before values flush to zero.  l sums the unrounded P~, so O
//    and L = m - kOff + log2(l) are unchanged by the offset.
//
// CTA and TMEM layout as fa_fwd.cu: two query tiles (256 rows), 384 threads (TMA warp, MMA
// warp, two idle warps whose registers go to the softmax warpgroups, 2 x 4 softmax warps), S_t
// at columns [128 t, 128 t + 128), O_t at 256 + t d; P~_t packed four per column over the
// first 32 columns of S_t.  O_t (bf16, twice the size of the e4m3 Q_t tile) is staged in the
// box layout of its tensor map over K/V ring slots 2t and 2t + 1, idle once every MMA of the CTA
// has completed, and written by TMA.
#include "fa_internal.h"

#include <cmath>

namespace fa {
namespace {

constexpr float kTau = 4.f;  // lazy-rescale threshold (log2 units)
constexpr float kOff = 4.f;  // P~ = 2^(s - m + kOff) <= 2^(kTau + kOff) = 256 <= 448

template <int D>
struct Fp8Layout {
    static constexpr int kTileBytes = kTile * D;  // Q or K tile (128 x d), or V^T tile (d x 128)
    static constexpr int kSlots = (D == 128) ? 8 : 16;  // K and V^T ring
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
};

// Q and K tiles: 128 rows of d bytes (128-byte swizzle at d = 128, 64-byte at d = 64).
template <int D>
__device__ __forceinline__ SDesc qk_desc(uint32_t saddr) {
    if constexpr (D == 128) return sdesc_make(saddr, 16, 1024);
    else return sdesc_make_sw64(saddr, 16, 512);
}

template <int D>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmq,
                      const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmvt,
                      const __grid_constant__ CUtensorMap tmo, const Fp8FwdParams p) {
    using L = Fp8Layout<D>;
    constexpr uint32_t kIdescS = idesc_e4m3(128, 128);
    constexpr uint32_t kIdescPV = idesc_e4m3(128, D);
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
    const int kvh = bh / p.rep;

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
        tma_prefetch_desc(&tmvt);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
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
                    tma_load_3d(sQ + t * L::kTileBytes, &tmq, 0, (qt0 + t) * kTile, bh, q_full);
                int n = 0;
                bool ok = true;
                for (int j = 0; j < jend && ok; ++j) {
                    if (!tile_live(p, mrow0, qt0, j) && !tile_live(p, mrow1, qt1, j)) continue;
                    for (int kv = 0; kv < 2; ++kv) {  // K_j, then V^T_j
                        const int s = n % L::kSlots;
                        const uint32_t par = ((n / L::kSlots) & 1) ^ 1;
                        if (!mbar_wait(&empty[s], par, p.ctl, abort_flag)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[s], L::kTileBytes);
                        uint8_t *dst = smem + L::kSlotOff + s * L::kTileBytes;
                        if (kv == 0)
                            tma_load_3d(dst, &tmk, 0, j * kTile, kvh, &full[s]);
                        else
                            tma_load_3d(dst, &tmvt, j * kTile, 0, kvh, &full[s]);
                        ++n;
                    }
                }
                if (!ok || *abort_flag) {
                    drain_wait(q_full, 0, p.ctl);
                    const int first = n > L::kSlots ? n - L::kSlots : 0;
                    for (int l = first; l < n; ++l)
                        drain_wait(&full[l % L::kSlots], (l / L::kSlots) & 1, p.ctl);
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
                const SDesc dq0 = qk_desc<D>(sQ);
                const SDesc dk0 = qk_desc<D>(sSlots);
                const SDesc dv0 = sdesc_make(sSlots, 16, 1024);  // V^T: 128-byte key rows
                auto issue_s = [&](int t, int ks) {  // S_t = Q_t K^T: d / 32 steps of 32 bytes
                    const SDesc a = sdesc_add(dq0, t * L::kTileBytes);
                    const SDesc b = sdesc_add(dk0, ks * L::kTileBytes);
                    if constexpr (D == 128)
                        mma_ss_f8_chain_k128(tmem + t * 128, a, b, kIdescS, 0u);
                    else
                        mma_ss_f8_chain_k64(tmem + t * 128, a, b, kIdescS, 0u);
                };
                auto issue_pv = [&](int t, int vs, bool accumulate) {  // 4 steps of 32 keys
                    mma_ts_f8_chain_k128(tmem + 256 + t * D, tmem + t * 128,
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
                // both tiles' o_final complete once every MMA issued above has: the ring is then
                // idle, and each softmax group stages its O over two of its slots
                if (ok) {
                    umma_commit_el(&o_final[0]);
                    umma_commit_el(&o_final[1]);
                }
                umma_commit_el(drain);
                drain_wait(drain, 0, p.ctl);
            }
            __syncwarp();
        }
    } else {
        regs_inc<216>();
        // ---------------------------------------------------------------- softmax groups
        const int t = (warp - 4) >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int qt = t == 0 ? qt0 : qt1;
        const uint32_t *mrow = t == 0 ? mrow0 : mrow1;
        const int q_row = qt * kTile + row;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_base + t * 128;
        const uint32_t tO = tmem + lane_base + 256 + t * D;
        const float sl2 = p.scale_log2;
        float m = -INFINITY;  // running (reference) max of the scaled scores, log2 units
        float l = 0.f;        // running sum of 2^(score - m + kOff)
        int cnt = 0;
        bool ok = true;
        for (int j = 0; j < jend; ++j) {
            if (!tile_live(p, mrow, qt, j)) continue;
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
            const float m_new = fmaxf(m, row_max128(r) * sl2);
            const bool old_finite = m != -INFINITY;
            const bool grow = m_new > m + kTau;
            float alpha = 1.f;
            if (grow) {
                if (old_finite) alpha = ex2(m - m_new);
                l *= alpha;
                m = m_new;
            }
            const bool rescale = grow && old_finite;
            const float bias = m == -INFINITY ? 0.f : kOff - m;  // nothing unmasked yet: P~ = 0
            float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            const float2 sc2 = make_float2(sl2, sl2), b2 = make_float2(bias, bias);
            uint32_t pk[32];
#pragma unroll
            for (int w = 0; w < 32; ++w) {
                const float2 x01 = ffma2(make_float2(__uint_as_float(r[4 * w]),
                                                     __uint_as_float(r[4 * w + 1])), sc2, b2);
                const float2 x23 = ffma2(make_float2(__uint_as_float(r[4 * w + 2]),
                                                     __uint_as_float(r[4 * w + 3])), sc2, b2);
                const float2 e01 = make_float2(ex2(x01.x), ex2(x01.y));
                const float2 e23 = make_float2(ex2(x23.x), ex2(x23.y));
                acc[0] = fadd2(acc[0], e01);
                acc[1] = fadd2(acc[1], e23);
                pk[w] = pack4_e4m3(e01.x, e01.y, e23.x, e23.y);
            }
            tmem_st32(tS, pk);
            const float2 a = fadd2(acc[0], acc[1]);
            l += a.x + a.y;
            if (__any_sync(0xffffffffu, rescale)) {
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
        if (ok) {
            ok = mbar_wait_warp(&o_final[t], 0, p.ctl, abort_flag);
            tc_fence_after();
        }
        // O_t = O~_t * descale_v / l staged as bf16 boxes over ring slots 2t, 2t + 1 and written
        // by TMA.  All four warps of the group reach the named barrier, whether or not their
        // waits succeeded.
        constexpr int kBoxBytes = kTile * 128;
        uint8_t *stage = smem + L::kSlotOff + t * 2 * L::kTileBytes;
        if (ok) {
            const float inv = l > 0.f ? p.descale_v / l : 0.f;
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
                st_box_row<true, 32>(stage + (cc >> 1) * kBoxBytes, row, (cc & 1) * 32, o, inv);
            }
            fence_proxy_async_smem();
            if (q_row < p.N)
                p.lse[static_cast<size_t>(bh) * p.N + q_row] =
                    l > 0.f ? (m - kOff + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
        named_sync(1 + t, 128);
        if (quad == 0 && lane == 0 && ok && *abort_flag == 0 && qt * kTile < p.N) {
            for (int b = 0; b < D / 64; ++b)
                tma_store_3d(&tmo, stage + b * kBoxBytes, b * 64, qt * kTile, bh);
            bulk_commit();
            bulk_wait_read_all();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// V [BHkv][N][d] bytes -> V^T [BHkv][d][Np] bytes, zero for keys N .. Np - 1.  One 64 x 64 byte
// tile per CTA through shared memory, both sides read and written 16 bytes per thread.
__global__ void __launch_bounds__(256) fa_fp8_transpose_v_kernel(const uint8_t *v, uint8_t *vt,
                                                                int N, int Np, int d) {
    __shared__ uint8_t tile[64][64 + 4];
    const int k0 = blockIdx.x * 64, d0 = blockIdx.y * 64;
    const size_t head = blockIdx.z;
    const int t = threadIdx.x;
    {
        const int key = k0 + t / 4, ch = t % 4;
        uint4 x = make_uint4(0, 0, 0, 0);
        if (key < N)
            x = *reinterpret_cast<const uint4 *>(v + (head * N + key) * d + d0 + ch * 16);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
            *reinterpret_cast<uint32_t *>(&tile[t / 4][ch * 16 + 4 * e]) = w[e];
    }
    __syncthreads();
    {
        const int dim = t / 4, ch = t % 4;
        const int key = k0 + ch * 16;
        if (key < Np) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                w[e] = static_cast<uint32_t>(tile[ch * 16 + 4 * e][dim]) |
                       (static_cast<uint32_t>(tile[ch * 16 + 4 * e + 1][dim]) << 8) |
                       (static_cast<uint32_t>(tile[ch * 16 + 4 * e + 2][dim]) << 16) |
                       (static_cast<uint32_t>(tile[ch * 16 + 4 * e + 3][dim]) << 24);
            *reinterpret_cast<uint4 *>(vt + (head * d + d0 + dim) * Np + key) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

template <int D>
cudaError_t launch_fwd_fp8_t(const Fp8Maps &maps, const Fp8FwdParams &p, cudaStream_t stream) {
    using L = Fp8Layout<D>;
    auto kern = fa_fwd_fp8_kernel<D>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    const long grid = static_cast<long>(p.BH) * p.num_pairs;
    kern<<<static_cast<unsigned>(grid), L::kThreads, L::kAlloc, stream>>>(maps.q, maps.k,
                                                                           maps.vt, maps.o, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8_transpose_v(const uint8_t *v, uint8_t *vt, int BHkv, int N, int Np, int d,
                                   cudaStream_t stream) {
    dim3 grid(static_cast<unsigned>((Np + 63) / 64), static_cast<unsigned>(d / 64),
              static_cast<unsigned>(BHkv));
    fa_fp8_transpose_v_kernel<<<grid, 256, 0, stream>>>(v, vt, N, Np, d);
    return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const Fp8Maps &maps, const Fp8FwdParams &p, int d,
                           cudaStream_t stream) {
    if (d == 64) return launch_fwd_fp8_t<64>(maps, p, stream);
    return launch_fwd_fp8_t<128>(maps, p, stream);
}

}  // namespace fa
