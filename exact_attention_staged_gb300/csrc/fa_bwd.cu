// fa_bwd.cu - exact-attention backward for sm_103a (tcgen05 + TMA + TMEM).
//
// FlashAttention-2 reading notes, Algorithm 2 (backward), with the scores and probabilities
// recomputed on chip from Q, K and the stored logsumexp (P_ij = exp(S_ij - L_i), eq. (16)) and
// the softmax Jacobian dS = P o (dP - D) (eq. (17)), where D_i = rowsum(dO_i o O_i) is computed
// first (Algorithm 2's precomputation; FlashAttention paper detail, "Technique 2").
// The atomic dQ update of Algorithm 2 is replaced by a second, query-stationary pass, so every
// output element is written once by one CTA: the result is deterministic.
//
//   preprocess   D = rowsum(dO o O) (times a given factor), one group of lanes per row, fp32.
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
// In both, four groups of four warps split every 128 x 128 score tile into four 32-wide column
// quarters (one TMEM lane quadrant per warp of a group), and the MMA warps run one tile ahead so
// the groups' exponentials overlap the tensor core (see each kernel's comment for its order).
// With dropout (keep scale s = 256 / (256 - t), keep decisions Z regenerated as in the forward):
// dV takes the dropped P (Z o P) and the factor s at the end; dP is masked to Z o dP, and since
// dS = P o (s Z o dP - D) = s P o (Z o dP - D / s), the preprocess writes D / s and dK, dQ take
// the factor s at the end with the softmax scale.
#include "fa_internal.h"

#include <cmath>
#include <type_traits>

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// bits: where the CTA keeps its mask column (dK/dV, bit = qt) or row (dQ, bit = kt) in shared
// memory when the mask is at most kMaskSmemTiles wide (a constant address: nothing stays live in
// a register between calls); wider masks are read from global memory
__device__ __forceinline__ bool tile_live(const BwdParams &p, const uint32_t *bits, int qt, int kt,
                                          int bit) {
    if (p.causal && kt > qt) return false;
    if (p.mask == nullptr) return true;
    return p.T <= kMaskSmemTiles ? mask_bit(bits, bit) : p.mask[qt * p.T + kt] != 0;
}

// The dK/dV kernel walks the (query head, query tile) pairs of its key tile kt in order, query
// tiles fastest: advance (hq, i) to the next live pair; hq reaches hq_end when none is left.
__device__ __forceinline__ void next_unit(const BwdParams &p, const uint32_t *bits, int kt, int i0,
                                          int hq_end, int &hq, int &i) {
    for (;;) {
        if (++i >= p.T) {
            if (++hq >= hq_end) return;
            i = i0;
        }
        if (tile_live(p, bits, i, kt, i)) return;
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

// Store 32 fp32 values (times `mul`) of one row as fp32, 128 bytes.
__device__ __forceinline__ void store_row32_f32(float *dst, const uint32_t *v, float mul) {
    float4 *d = reinterpret_cast<float4 *>(dst);
#pragma unroll
    for (int e = 0; e < 8; ++e)
        d[e] = make_float4(__uint_as_float(v[4 * e]) * mul, __uint_as_float(v[4 * e + 1]) * mul,
                           __uint_as_float(v[4 * e + 2]) * mul, __uint_as_float(v[4 * e + 3]) * mul);
}

// Compute-group geometry shared by both backward kernels: four groups of four warps (one
// warp per TMEM lane quadrant each), group g owning columns [32g, 32g+32) of every 128-wide
// score tile.  The CTA also has a load warp and one (dK/dV) or two (dQ) MMA-issuing warps.
constexpr int kGroups = 4;
constexpr int kGroupCols = kTile / kGroups;  // 32
constexpr int kComputeThreads = kGroups * 128;
constexpr int kComputeWarps = kComputeThreads / 32;

// ================================================================================ preprocess
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_preprocess_kernel(const void *o, const void *dout,
                                                                float *delta, long rows, float mul) {
    constexpr int kLanes = D / 8;  // 8 elements (16 bytes) per lane
    // queued right after the forward with programmatic stream serialization: O is complete and
    // visible only past this point
    griddep_wait();
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
    if (row < rows && part == 0) delta[row] = acc * mul;
}

// ================================================================================ dK / dV
// CTA = one 128-row key tile of one K/V head, 576 threads: warp 0 loads, warp 1 issues the MMAs, warps 2..17
// are four compute groups, group g owning query columns [32g, 32g+32) of every score tile.
// Shared memory: K_j and V_j (stationary), a ring of slots that receives Q_0, dO_0, Q_1, dO_1,
// ... in that order (each released as soon as its last MMA is done), and a two-entry ring of
// the tiles' L (logsumexp) and D values, fetched with cp.async so the load warp never stalls.
// TMEM: S^T [0,128), dP^T [128,256), dV [256,256+d), dK [256+d,256+2d).  Group g packs its
// P^T columns into [32g, 32g+16) and its dS^T columns into [128+32g, 128+32g+16).
// MMA order, one query tile of lookahead: dV(n), S^T(n+1), dK(n), dP^T(n+1), dV(n+1), ...
// So the exponentials of tile n+1 overlap dK(n) and dP^T(n+1), and dS(n+1) overlaps dV(n+1)
// and S^T(n+2).  One issuing thread keeps this order exact on the tensor pipe.
// Head dimension 64: dV and dK take 128 columns, so a second S^T buffer fits at [384, 512)
// (tile n uses buffer n % 2) and S^T(n+1) is issued before dV(n), which still reads P^T(n) from
// the other buffer: S^T(n+1), dV(n), dK(n), dP^T(n+1).  The compute warps then find the next
// tile's scores ready when they finish dS(n) (at d = 64 a tile's four GEMMs take half the tensor
// time of d = 128 against the same element-wise work, and with one buffer the MMA warp waited
// about 750 cycles per tile for the probabilities).
// Grouped-query attention (FlashAttention-2 reading notes, MQA/GQA section): the query tiles
// of every query head that shares this K/V head stream through the same pipeline, one head
// after the other, so dK and dV are summed over the group in TMEM.  When there are too few K/V
// heads to fill the GPU, the group is split over several CTAs whose fp32 partial sums a second
// kernel adds up (fa_bwd_group_reduce_kernel).
template <int D>
struct DkvLayout {
    static constexpr int kTileBytes = kTile * D * 2;
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = kTile * 128;
    static constexpr int kSlots = (D == 128) ? 5 : 10;  // Q / dO ring
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kTileBytes;
    static constexpr int kSlotOff = 2 * kTileBytes;
    static constexpr int kLdOff = kSlotOff + kSlots * kTileBytes;  // 2 x (128 L + 128 D floats)
    static constexpr int kBarOff = kLdOff + 2 * 1024;
    // kv_full, full[S], empty[S], ld_full[2], ld_empty[2], s_full[2], dp_full, p_ready[2],
    // ds_ready, final, drain
    static constexpr int kNumBars = 1 + 2 * kSlots + 4 + 8;
    static constexpr bool kDbl = D == 64;  // two S^T buffers (see the kernel comment)
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kMaskOff = kMiscOff + 16;  // block-mask bits of the CTA's column / row
    static constexpr int kAlloc = kMaskOff + kMaskSmemWords * 4;  // 1024-aligned base (checked)
    static constexpr int kThreads = 64 + kComputeThreads;
    static constexpr int kComputeWarp0 = 2;
};

template <int D, bool BF16, bool DROP>
__global__ void __launch_bounds__(64 + kComputeThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv,
                       const __grid_constant__ CUtensorMap tmdo,
                       const __grid_constant__ CUtensorMap tmdk,
                       const __grid_constant__ CUtensorMap tmdv, const BwdParams p) {
    using L = DkvLayout<D>;
    constexpr uint32_t kIdescSS = idesc_f16(128, 128, BF16, false);  // S^T, dP^T
    constexpr uint32_t kIdescTS = idesc_f16(128, D, BF16, true);     // dV, dK
    extern __shared__ uint8_t smem[];
    if (smem_u32(smem) & 1023u) {  // layouts assume a 1024-aligned base; never observed
        if (threadIdx.x == 0) atomicExch(p.ctl.status, kErrInternal);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *kv_full = bars;
    uint64_t *full = bars + 1;
    uint64_t *empty = full + L::kSlots;
    uint64_t *ld_full = empty + L::kSlots;  // [2]
    uint64_t *ld_empty = ld_full + 2;       // [2]
    uint64_t *s_full = ld_empty + 2;        // [2]: one per S^T buffer (d = 64), else [0] only
    uint64_t *dp_full = s_full + 2;
    uint64_t *p_ready = dp_full + 1;        // [2]: one per S^T buffer (d = 64), else [0] only
    uint64_t *ds_ready = p_ready + 2;
    uint64_t *fin = ds_ready + 1;
    uint64_t *drain = fin + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);
    float *ld_ring = reinterpret_cast<float *>(smem + L::kLdOff);

    const int warp = warp_id(), lane = lane_id();
    const CtaOrder ord = cta_order(blockIdx.x, p.units, p.T, p.head_group);
    const int kvh = ord.head / p.splits;               // b * H_kv + K/V head
    const int split = ord.head - kvh * p.splits;
    const int hq0 = kvh * p.rep + split * p.chunk;     // first query head (b * H + h)
    const int hq_end = min(hq0 + p.chunk, (kvh + 1) * p.rep);
    const int kt = ord.rank;           // key tile; tile 0 sees the most query tiles when causal
    const int i0 = p.causal ? kt : 0;  // first query tile that can see it

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int s = 0; s < L::kSlots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int e = 0; e < 2; ++e) {
            mbar_init(&ld_full[e], 32);   // one cp.async completion per lane of the load warp
            mbar_init(&ld_empty[e], kComputeWarps);  // every compute warp, after its dS
        }
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(dp_full, 1);
        mbar_init(&p_ready[0], kComputeWarps);
        mbar_init(&p_ready[1], kComputeWarps);
        mbar_init(ds_ready, kComputeWarps);
        mbar_init(fin, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    uint32_t *const mcol = reinterpret_cast<uint32_t *>(smem + L::kMaskOff);  // column kt
    if (p.mask != nullptr && p.T <= kMaskSmemTiles) mask_bits_load(mcol, p.mask + kt, p.T, p.T);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------------- load warp
        if (lane == 0) {
            mbar_arrive_expect_tx(kv_full, 2 * L::kTileBytes);
            for (int b = 0; b < L::kBoxes; ++b) {
                tma_load_3d(smem + L::kKOff + b * L::kBoxBytes, &tmk, b * 64, kt * kTile, kvh,
                            kv_full);
                tma_load_3d(smem + L::kVOff + b * L::kBoxBytes, &tmv, b * 64, kt * kTile, kvh,
                            kv_full);
            }
        }
        int n = 0;  // query tiles issued
        bool ok = true;
        int hq = hq0, i = i0 - 1;
        next_unit(p, mcol, kt, i0, hq_end, hq, i);
        for (; hq < hq_end && ok; next_unit(p, mcol, kt, i0, hq_end, hq, i)) {
            for (int x = 0; x < 2 && ok; ++x) {  // Q_i then dO_i
                const int l = 2 * n + x;
                const int s = l % L::kSlots;
                int got = 0;
                if (lane == 0) {
                    got = mbar_wait(&empty[s], ((l / L::kSlots) & 1) ^ 1, p.ctl, abort_flag);
                    // test hook: fault mode 2 leaves the first Q tile unloaded
                    if (got && !(p.ctl.fault_mode == 2 && l == 0)) {
                        mbar_arrive_expect_tx(&full[s], L::kTileBytes);
                        uint8_t *dst = smem + L::kSlotOff + s * L::kTileBytes;
                        for (int b = 0; b < L::kBoxes; ++b)
                            tma_load_3d(dst + b * L::kBoxBytes, x ? &tmdo : &tmq, b * 64,
                                        i * kTile, hq, &full[s]);
                    }
                }
                ok = __shfl_sync(0xffffffffu, got, 0) != 0;
            }
            if (!ok) break;
            // L and D of tile i into ring entry n % 2, once tile n - 2 has released it
            const int e = n & 1;
            int got = 0;
            if (lane == 0) got = mbar_wait(&ld_empty[e], ((n >> 1) & 1) ^ 1, p.ctl, abort_flag);
            if (!__shfl_sync(0xffffffffu, got, 0)) {
                ok = false;
                break;
            }
            float *dl = ld_ring + e * 256;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int c = lane + 32 * k;
                const int row = i * kTile + c;
                const bool in = row < p.N;
                const size_t off = static_cast<size_t>(hq) * p.N + (in ? row : 0);
                cp_async_4(dl + c, p.lse + off, in);
                cp_async_4(dl + 128 + c, p.delta + off, in);
            }
            cp_async_arrive_noinc(&ld_full[e]);
            ++n;
        }
        if (lane == 0 && (!ok || *abort_flag)) {
            drain_wait(kv_full, 0, p.ctl);
            const int issued = 2 * n;
            const int first = issued > L::kSlots ? issued - L::kSlots : 0;
            for (int l = first; l < issued; ++l) {
                if (p.ctl.fault_mode == 2 && l == 0) continue;  // never loaded
                drain_wait(&full[l % L::kSlots], (l / L::kSlots) & 1, p.ctl);
            }
        }
        cp_async_wait_all();
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        // the whole warp runs this loop in lockstep; one elected lane issues each MMA/commit
        {
            const uint32_t sSlot = smem_u32(smem + L::kSlotOff);
            const uint32_t tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;
            // S^T buffer of query tile n, and the barrier that says it holds S^T(n)
            auto tS_of = [&](int n) { return tmem + ((L::kDbl && (n & 1)) ? 384u : 0u); };
            auto sbar_of = [&](int n) { return &s_full[L::kDbl ? (n & 1) : 0]; };
            const SDesc dK0 = sdesc_make(smem_u32(smem + L::kKOff), 16, 1024);
            const SDesc dV0 = sdesc_make(smem_u32(smem + L::kVOff), 16, 1024);
            const SDesc dSk = sdesc_make(sSlot, 16, 1024);            // slot as K-major B
            const SDesc dSm = sdesc_make(sSlot, L::kBoxBytes, 1024);  // slot as MN-major B
            auto slot_of = [&](int l) { return l % L::kSlots; };
            auto full_wait = [&](int l) {
                return mbar_wait_warp(&full[slot_of(l)], (l / L::kSlots) & 1, p.ctl, abort_flag);
            };
            auto issue_ss = [&](uint32_t d, SDesc a, int l) {  // 128 x 128 x d, A stationary
                const SDesc b = sdesc_add(dSk, slot_of(l) * L::kTileBytes);
                if constexpr (D == 128)
                    mma_ss_chain_k128(d, a, b, kIdescSS, 0u);
                else
                    mma_ss_chain_k64(d, a, b, kIdescSS, 0u);
            };
            auto issue_ts = [&](uint32_t d, uint32_t a_col, int l, bool acc) {  // K = 128 queries
                mma_ts_chain_k128_g32(d, a_col, sdesc_add(dSm, slot_of(l) * L::kTileBytes),
                                      kIdescTS, acc ? 1u : 0u);
            };
            auto log_visit = [&](int hq, int i) {
                if (p.ctl.visit_log != nullptr && lane == 0)
                    visit_mark(p.ctl.visit_log, (static_cast<size_t>(hq) * p.T + i) * p.T + kt, 2u);
            };
            bool ok = mbar_wait_warp(kv_full, 0, p.ctl, abort_flag);
            int hq = hq0, i = i0 - 1;
            next_unit(p, mcol, kt, i0, hq_end, hq, i);
            int n = 0;
            if (ok && hq < hq_end) {
                ok = full_wait(0) && full_wait(1);
                if (ok) {
                    issue_ss(tS_of(0), dK0, 0);
                    umma_commit_el(sbar_of(0));
                    issue_ss(tdP, dV0, 1);
                    umma_commit_el(dp_full);
                    log_visit(hq, i);
                }
            }
            while (ok && hq < hq_end) {
                int nhq = hq, ni = i;
                next_unit(p, mcol, kt, i0, hq_end, nhq, ni);
                const bool more = nhq < hq_end;
                const int lq = 2 * n, ldo = 2 * n + 1;  // this tile's Q and dO loads
                auto issue_next_s = [&]() -> bool {  // S^T(n+1) = K Q^T
                    if (!more) return true;
                    if (!full_wait(lq + 2)) return false;
                    issue_ss(tS_of(n + 1), dK0, lq + 2);
                    umma_commit_el(sbar_of(n + 1));
                    log_visit(nhq, ni);
                    return true;
                };
                if (L::kDbl && !issue_next_s()) {  // into the other buffer, ahead of dV(n)
                    ok = false;
                    break;
                }
                // at d = 64 a compute warp may post P^T(n+1) (its S^T was issued ahead of dV(n))
                // before a slower warp has posted P^T(n): each S^T buffer has its own barrier
                if (!mbar_wait_warp(&p_ready[L::kDbl ? (n & 1) : 0],
                                    L::kDbl ? ((n >> 1) & 1) : (n & 1), p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_ts(tdV, tS_of(n), ldo, n > 0);  // dV += P^T dO
                umma_commit_el(&empty[slot_of(ldo)]);
                if (!L::kDbl && !issue_next_s()) {  // over P^T(n), after dV(n) has read it
                    ok = false;
                    break;
                }
                if (!mbar_wait_warp(ds_ready, n & 1, p.ctl, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_ts(tdK, tdP, lq, n > 0);  // dK += dS^T Q
                umma_commit_el(&empty[slot_of(lq)]);
                if (more) {
                    if (!full_wait(ldo + 2)) {
                        ok = false;
                        break;
                    }
                    issue_ss(tdP, dV0, ldo + 2);  // dP^T(n+1) = V dO^T
                    umma_commit_el(dp_full);
                }
                hq = nhq;
                i = ni;
                ++n;
            }
            if (ok && n > 0) umma_commit_el(fin);
            umma_commit_el(drain);
            drain_wait(drain, 0, p.ctl);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- compute groups
        const int g = (warp - L::kComputeWarp0) >> 2;  // query columns [32g, 32g+32)
        const int quad = warp & 3;
        const int row = quad * 32 + lane;  // key row within the tile
        const int k_row = kt * kTile + row;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS0 = tmem + lane_base + kGroupCols * g, tdP = tS0 + 128;
        const float sl2 = p.scale_log2;
        int n = 0;
        bool ok = true;
        int hq = hq0, i = i0 - 1;
        next_unit(p, mcol, kt, i0, hq_end, hq, i);
        for (; hq < hq_end; next_unit(p, mcol, kt, i0, hq_end, hq, i)) {
            const int e = n & 1;
            uint32_t keep = 0;  // dropout: bit c set = query 32g + c of tile i keeps this key row
            if constexpr (DROP) {
                // lane l draws the bits of query 32g + l for the warp's 32 key rows (one
                // generator block) before the scores are ready; a bit transpose hands lane r the
                // bits of its own key row
                const uint32_t mine = philox_keep_bits<false>(
                    static_cast<uint64_t>(kt) * 4 + quad,
                    static_cast<uint64_t>(i * kTile + kGroupCols * g + lane),
                    static_cast<uint64_t>(hq), p.drop);
                keep = transpose32_bits(mine, lane);
            }
            // keep bits 4w .. 4w + 3 as keep flags (to the top bits of bytes 0 .. 3): the
            // product's other terms land on distinct lower bits, so no carry reaches a top bit
            auto kf = [&](int w) { return ((keep >> (4 * w)) & 0xFu) * 0x10204080u; };
            // S^T of this tile: buffer n % 2 at d = 64, the only one otherwise
            const uint32_t tS = tS0 + ((L::kDbl && (n & 1)) ? 384u : 0u);
            uint64_t *const sbar = &s_full[L::kDbl ? (n & 1) : 0];
            const uint32_t spar = L::kDbl ? ((n >> 1) & 1) : (n & 1);
            if (!mbar_wait_warp(&ld_full[e], (n >> 1) & 1, p.ctl, abort_flag) ||
                !mbar_wait_warp(sbar, spar, p.ctl, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float4 *lv = reinterpret_cast<const float4 *>(ld_ring + e * 256 + kGroupCols * g);
            const float4 *dv = lv + 32;  // D values 128 floats after L
            // query q sees key k only when k <= q (causal) and q < N
            const int q_base = i * kTile + kGroupCols * g;
            const bool need_mask = (p.causal && i == kt) || (q_base + kGroupCols > p.N);
            uint32_t pk[16];  // P^T of this row's 32 queries, packed 16-bit pairs (for dV)
            float pf[32];     // the same in fp32 (for dS)
            {
                uint32_t r[32];
                tmem_ld32(tS, r);
                tmem_wait_ld();
                const float2 sc2 = make_float2(sl2, sl2);
                const float2 nl2e = make_float2(-kLog2e, -kLog2e);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 lq = lv[c];
                    const float2 x01 = ffma2(make_float2(__uint_as_float(r[4 * c]),
                                                         __uint_as_float(r[4 * c + 1])),
                                             sc2, fmul2(make_float2(lq.x, lq.y), nl2e));
                    const float2 x23 = ffma2(make_float2(__uint_as_float(r[4 * c + 2]),
                                                         __uint_as_float(r[4 * c + 3])),
                                             sc2, fmul2(make_float2(lq.z, lq.w), nl2e));
                    float pv[4] = {ex2(x01.x), ex2(x01.y), ex2(x23.x), ex2(x23.y)};
                    if (need_mask) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int q = q_base + 4 * c + u;
                            if (q >= p.N || (p.causal && q < k_row)) pv[u] = 0.f;
                        }
                    }
                    pk[2 * c] = pack2<BF16>(pv[0], pv[1]);
                    pk[2 * c + 1] = pack2<BF16>(pv[2], pv[3]);
#pragma unroll
                    for (int u = 0; u < 4; ++u) pf[4 * c + u] = pv[u];
                }
            }
            if constexpr (DROP) {  // dV sees the dropped probabilities, dS all of them
                uint32_t pkd[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) pkd[c] = pk[c] & keep_pair_mask(kf(c >> 1), 2 * (c & 1));
                tmem_st16(tS, pkd);
            } else {
                tmem_st16(tS, pk);
            }
            mbar_arrive_warp_after_st(&p_ready[L::kDbl ? (n & 1) : 0]);
            if (!mbar_wait_warp(dp_full, n & 1, p.ctl, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            {
                uint32_t r[32];
                tmem_ld32(tdP, r);
                tmem_wait_ld();
                if constexpr (DROP) {  // dP of a dropped score is 0, of a kept one dP / (1 - p)
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        r[c] &= static_cast<uint32_t>(static_cast<int32_t>(keep << (31 - c)) >> 31);
                }
                uint32_t w[16];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 dq = dv[c];
                    const float2 s01 = fmul2(make_float2(pf[4 * c], pf[4 * c + 1]),
                                             fsub2(make_float2(__uint_as_float(r[4 * c]),
                                                               __uint_as_float(r[4 * c + 1])),
                                                   make_float2(dq.x, dq.y)));
                    const float2 s23 = fmul2(make_float2(pf[4 * c + 2], pf[4 * c + 3]),
                                             fsub2(make_float2(__uint_as_float(r[4 * c + 2]),
                                                               __uint_as_float(r[4 * c + 3])),
                                                   make_float2(dq.z, dq.w)));
                    w[2 * c] = pack2<BF16>(s01.x, s01.y);
                    w[2 * c + 1] = pack2<BF16>(s23.x, s23.y);
                }
                tmem_st16(tdP, w);  // over columns already read
            }
            mbar_arrive_warp_after_st(ds_ready);
            mbar_arrive_warp(&ld_empty[e]);
            ++n;
        }
        if (ok && n > 0) {
            ok = mbar_wait_warp(fin, 0, p.ctl, abort_flag);
            tc_fence_after();
        }
        // groups 0, 1 hold the two column halves of dV; groups 2, 3 those of dK (x scale).
        // With one split they are staged as 16-bit tiles in the (now idle) first two ring slots
        // and written by TMA; a split K/V group writes fp32 partial sums directly.  Every compute
        // warp reaches the named barrier, whether or not its waits succeeded.
        const int half = g & 1;
        const uint32_t tacc = tmem + lane_base + 256 + (g < 2 ? 0 : D) + half * (D / 2);
        const float mul = (DROP ? p.drop.keep_scale : 1.f) * (g < 2 ? 1.f : p.scale);
        if (p.part == nullptr) {
            if (ok) {
                uint8_t *stage = smem + L::kSlotOff + (g < 2 ? 0 : 1) * L::kTileBytes;
#pragma unroll
                for (int cc = 0; cc < D / 64; ++cc) {
                    uint32_t a[32];
                    if (n > 0) {
                        tmem_ld32(tacc + 32 * cc, a);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int e2 = 0; e2 < 32; ++e2) a[e2] = 0u;
                    }
                    const int col = half * (D / 2) + 32 * cc;
                    st_box_row<BF16, 32>(stage + (col >> 6) * L::kBoxBytes, row, col & 63, a, mul);
                }
                fence_proxy_async_smem();
            }
            named_sync(1, kComputeThreads);
            if (warp == L::kComputeWarp0 && lane == 0 && ok && *abort_flag == 0) {
                const uint8_t *sdv = smem + L::kSlotOff, *sdk = sdv + L::kTileBytes;
                for (int b2 = 0; b2 < L::kBoxes; ++b2) {
                    tma_store_3d(&tmdv, sdv + b2 * L::kBoxBytes, b2 * 64, kt * kTile, kvh);
                    tma_store_3d(&tmdk, sdk + b2 * L::kBoxBytes, b2 * 64, kt * kTile, kvh);
                }
                bulk_commit();
                bulk_wait_read_all();
            }
        } else if (ok) {
            const bool valid = k_row < p.N;
            const size_t row_off = (static_cast<size_t>(kvh) * p.N + k_row) * D + half * (D / 2);
            float *dstf = p.part + (static_cast<size_t>(g < 2 ? 1 : 0) * p.splits + split) *
                                       p.kv_elems + row_off;
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t a[32];
                if (n > 0) {
                    tmem_ld32(tacc + 32 * cc, a);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e2 = 0; e2 < 32; ++e2) a[e2] = 0u;
                }
                if (valid) store_row32_f32(dstf + 32 * cc, a, mul);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // Launched to overlap the tail of the dQ pass (see launch_dkdv_t), this grid must not
    // complete before that pass has: whatever the caller queues next may overwrite what dQ reads.
    if (threadIdx.x == 0) griddep_wait();
}

// ================================================================================ dQ
// CTA = one 128-row query tile, 608 threads: warp 0 loads, warp 1 issues S and dQ, warp 2
// issues dP, warps 3..18 are four compute groups, group g owning key columns [32g, 32g+32) of
// every score tile.  Two issuers: the MMA pipe holds only about two MMAs, and the two chains
// (S and dQ; dP) need no order between them, so one thread's waits no longer idle the pipe.
// Shared memory: Q_i and dO_i (stationary) and a ring of slots receiving K_0, V_0, K_1, V_1, ...
// TMEM: two S buffers [0,128) and [128,256) (tile n uses buffer n % 2), dP [256,384),
// dQ [384,384+d).  Group g packs its dS columns into the first 16 columns of its S quarter.
// MMA order: warp 1 runs dQ(n), S(n+2), dQ(n+1), ...; warp 2 runs dP(n+1), dP(n+2), ... as soon
// as every group has loaded dP(n) from TMEM (dp_read), so dP(n+1) overlaps the dS(n)
// arithmetic.  The next tile's S is already in TMEM while the groups work on
// tile n+1, and S(n+2) overwrites buffer n % 2 only after dQ(n) has read it.  Each S buffer has
// its own dS-ready barrier, so neither issuer can fall two phases behind one.
template <int D>
struct DqLayout {
    static constexpr int kTileBytes = kTile * D * 2;
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = kTile * 128;
    static constexpr int kSlots = (D == 128) ? 5 : 10;  // K / V ring
    static constexpr int kQOff = 0;
    static constexpr int kdOOff = kTileBytes;
    static constexpr int kSlotOff = 2 * kTileBytes;
    static constexpr int kBarOff = kSlotOff + kSlots * kTileBytes;
    // q_full, full[S], empty[S], s_full[2], dp_full, ds_ready[2], final, drain[2], dp_read
    static constexpr int kNumBars = 1 + 2 * kSlots + 9;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kMaskOff = kMiscOff + 16;  // block-mask bits of the CTA's column / row
    static constexpr int kAlloc = kMaskOff + kMaskSmemWords * 4;  // 1024-aligned base (checked)
    static constexpr int kThreads = 96 + kComputeThreads;
    static constexpr int kComputeWarp0 = 3;
};

template <int D, bool BF16, bool DROP>
__global__ void __launch_bounds__(96 + kComputeThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmdo,
                     const __grid_constant__ CUtensorMap tmdq, const BwdParams p) {
    using L = DqLayout<D>;
    constexpr uint32_t kIdescSS = idesc_f16(128, 128, BF16, false);  // S, dP
    constexpr uint32_t kIdescTS = idesc_f16(128, D, BF16, true);     // dQ
    extern __shared__ uint8_t smem[];
    if (smem_u32(smem) & 1023u) {  // layouts assume a 1024-aligned base; never observed
        if (threadIdx.x == 0) atomicExch(p.ctl.status, kErrInternal);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *q_full = bars;
    uint64_t *full = bars + 1;
    uint64_t *empty = full + L::kSlots;
    uint64_t *s_full = empty + L::kSlots;  // [2]
    uint64_t *dp_full = s_full + 2;
    uint64_t *ds_ready = dp_full + 1;       // [2], one per S buffer
    uint64_t *fin = ds_ready + 2;
    uint64_t *drain = fin + 1;              // [2]
    uint64_t *dp_read = drain + 2;          // every compute thread has loaded dP(n) from TMEM
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);

    const int warp = warp_id(), lane = lane_id();
    const CtaOrder ord = cta_order(blockIdx.x, p.BH, p.T, p.head_group);
    const int bh = ord.head;
    const int kvh = bh / p.rep;         // K/V head of this query head's group
    const int qt = p.T - 1 - ord.rank;  // long rows first
    const int jend = p.causal ? qt + 1 : p.T;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < L::kSlots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(dp_full, 1);
        mbar_init(&ds_ready[0], kComputeWarps);
        mbar_init(&ds_ready[1], kComputeWarps);
        mbar_init(dp_read, kComputeWarps);
        mbar_init(fin, 1);
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    uint32_t *const mrow = reinterpret_cast<uint32_t *>(smem + L::kMaskOff);  // row qt
    if (p.mask != nullptr && p.T <= kMaskSmemTiles)
        mask_bits_load(mrow, p.mask + static_cast<long>(qt) * p.T, 1, p.T);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the dK/dV pass queued after this one reads nothing it writes: let it take the SMs that
    // this grid's last CTAs leave idle
    if (threadIdx.x == 0) griddep_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, 2 * L::kTileBytes);
            for (int b = 0; b < L::kBoxes; ++b) {
                tma_load_3d(smem + L::kQOff + b * L::kBoxBytes, &tmq, b * 64, qt * kTile, bh,
                            q_full);
                tma_load_3d(smem + L::kdOOff + b * L::kBoxBytes, &tmdo, b * 64, qt * kTile, bh,
                            q_full);
            }
            int l = 0;  // loads issued: K_n is load 2n, V_n load 2n + 1
            bool ok = true;
            for (int j = 0; j < jend && ok; ++j) {
                if (!tile_live(p, mrow, qt, j, j)) continue;
                for (int x = 0; x < 2; ++x, ++l) {
                    const int s = l % L::kSlots;
                    if (!mbar_wait(&empty[s], ((l / L::kSlots) & 1) ^ 1, p.ctl, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (p.ctl.fault_mode == 3 && l == 0) continue;  // test hook: K_0 unloaded
                    mbar_arrive_expect_tx(&full[s], L::kTileBytes);
                    uint8_t *dst = smem + L::kSlotOff + s * L::kTileBytes;
                    for (int b = 0; b < L::kBoxes; ++b)
                        tma_load_3d(dst + b * L::kBoxBytes, x ? &tmv : &tmk, b * 64, j * kTile,
                                    kvh, &full[s]);
                }
            }
            if (!ok || *abort_flag) {
                drain_wait(q_full, 0, p.ctl);
                const int first = l > L::kSlots ? l - L::kSlots : 0;
                for (int m = first; m < l; ++m) {
                    if (p.ctl.fault_mode == 3 && m == 0) continue;  // never loaded
                    drain_wait(&full[m % L::kSlots], (m / L::kSlots) & 1, p.ctl);
                }
            }
        }
        __syncwarp();
    } else if (warp <= 2) {
        // each issuing warp runs its loop in lockstep; one elected lane issues each MMA/commit
        {
            const bool sq = warp == 1;  // warp 1: S and dQ; warp 2: dP
            const uint32_t sSlot = smem_u32(smem + L::kSlotOff);
            const uint32_t tdP = tmem + 256, tdQ = tmem + 384;
            const SDesc dQa = sdesc_make(smem_u32(smem + L::kQOff), 16, 1024);
            const SDesc ddOa = sdesc_make(smem_u32(smem + L::kdOOff), 16, 1024);
            const SDesc dSk = sdesc_make(sSlot, 16, 1024);            // slot as K-major B
            const SDesc dSm = sdesc_make(sSlot, L::kBoxBytes, 1024);  // slot as MN-major B
            auto slot_of = [&](int l) { return l % L::kSlots; };
            auto full_wait = [&](int l) {
                return mbar_wait_warp(&full[slot_of(l)], (l / L::kSlots) & 1, p.ctl, abort_flag);
            };
            auto issue_ss = [&](uint32_t d, SDesc a, int l) {  // 128 x 128 x d
                const SDesc b = sdesc_add(dSk, slot_of(l) * L::kTileBytes);
                if constexpr (D == 128)
                    mma_ss_chain_k128(d, a, b, kIdescSS, 0u);
                else
                    mma_ss_chain_k64(d, a, b, kIdescSS, 0u);
            };
            auto next_live = [&](int j) {
                for (++j; j < jend; ++j)
                    if (tile_live(p, mrow, qt, j, j)) return j;
                return jend;
            };
            auto ds_wait = [&](int n) {
                return mbar_wait_warp(&ds_ready[n & 1], (n >> 1) & 1, p.ctl, abort_flag);
            };
            bool ok = mbar_wait_warp(q_full, 0, p.ctl, abort_flag);
            int j = next_live(-1);
            int j1 = j < jend ? next_live(j) : jend;  // tile n + 1
            int n = 0;
            if (sq) {
                // S(0) -> buffer 0, S(1) -> buffer 1; then per tile: dQ(n), S(n+2)
                if (ok && j < jend) {
                    ok = full_wait(0);
                    if (ok) {
                        tc_fence_after();
                        issue_ss(tmem, dQa, 0);
                        umma_commit_el(&s_full[0]);
                        if (p.ctl.visit_log != nullptr && lane == 0)
                            visit_mark(p.ctl.visit_log, (static_cast<size_t>(bh) * p.T + qt) * p.T + j, 4u);
                    }
                    if (ok && j1 < jend) {
                        ok = full_wait(2);
                        if (ok) {
                            tc_fence_after();
                            issue_ss(tmem + 128, dQa, 2);
                            umma_commit_el(&s_full[1]);
                            if (p.ctl.visit_log != nullptr && lane == 0)
                                visit_mark(p.ctl.visit_log, (static_cast<size_t>(bh) * p.T + qt) * p.T + j1, 4u);
                        }
                    }
                }
                while (ok && j < jend) {
                    const int j2 = j1 < jend ? next_live(j1) : jend;  // tile n + 2
                    const uint32_t buf = tmem + 128 * (n & 1);
                    if (!ds_wait(n)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    {  // dQ += dS K_n, K = 128 keys
                        mma_ts_chain_k128_g32(tdQ, buf, sdesc_add(dSm, slot_of(2 * n) * L::kTileBytes),
                                              kIdescTS, n > 0 ? 1u : 0u);
                        umma_commit_el(&empty[slot_of(2 * n)]);
                    }
                    if (j2 < jend) {  // S(n+2) into this buffer, after dQ(n) read it
                        if (!full_wait(2 * n + 4)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_ss(buf, dQa, 2 * n + 4);
                        umma_commit_el(&s_full[n & 1]);
                        if (p.ctl.visit_log != nullptr && lane == 0)
                            visit_mark(p.ctl.visit_log, (static_cast<size_t>(bh) * p.T + qt) * p.T + j2, 4u);
                    }
                    j = j1;
                    j1 = j2;
                    ++n;
                }
                if (ok && n > 0) umma_commit_el(fin);
            } else {
                // dP(0); then per tile: once the groups are done with dP(n), dP(n+1)
                if (ok && j < jend) {
                    ok = full_wait(1);
                    if (ok) {
                        tc_fence_after();
                        issue_ss(tdP, ddOa, 1);
                        umma_commit_el(dp_full);
                        umma_commit_el(&empty[slot_of(1)]);
                    }
                }
                while (ok && j < jend) {
                    // dP(n+1) may overwrite the dP buffer once every compute thread has loaded
                    // dP(n) (dS goes to the S buffer), so it runs while dS(n) is computed
                    if (!mbar_wait_warp(dp_read, n & 1, p.ctl, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (j1 < jend) {
                        if (!full_wait(2 * n + 3)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_ss(tdP, ddOa, 2 * n + 3);
                        umma_commit_el(dp_full);
                        umma_commit_el(&empty[slot_of(2 * n + 3)]);
                    }
                    j = j1;
                    j1 = j1 < jend ? next_live(j1) : jend;
                    ++n;
                }
            }
            umma_commit_el(&drain[sq ? 0 : 1]);
            drain_wait(&drain[sq ? 0 : 1], 0, p.ctl);
        }
        __syncwarp();
    } else {
        const int g = (warp - L::kComputeWarp0) >> 2;  // key columns [32g, 32g+32)
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int q_row = qt * kTile + row;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tdP = tmem + lane_base + 256 + kGroupCols * g;
        const float sl2 = p.scale_log2;
        const float lrow = lse_log2(p, bh, q_row);
        const float drow = q_row < p.N ? p.delta[static_cast<size_t>(bh) * p.N + q_row] : 0.f;
        int n = 0;
        bool ok = true;
        for (int j = 0; j < jend; ++j) {
            if (!tile_live(p, mrow, qt, j, j)) continue;
            const int b = n & 1;
            const uint32_t tS = tmem + lane_base + 128 * b + kGroupCols * g;
            uint32_t keep[8];  // dropout: keep flag of key 128 j + 32 g + e in byte e % 4 of word e / 4
            if constexpr (DROP)
                philox_keep_flags(static_cast<uint64_t>(j) * 4 + g, static_cast<uint64_t>(q_row),
                                  static_cast<uint64_t>(bh), p.drop, keep);
            if (!mbar_wait_warp(&s_full[b], (n >> 1) & 1, p.ctl, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int kv0 = j * kTile + kGroupCols * g;
            const bool need_mask = (p.causal && j == qt) || (kv0 + kGroupCols > p.N);
            float pr[32];  // P of this row's 32 keys, while the tensor core is on dP
            {
                uint32_t a[32];
                tmem_ld32(tS, a);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 x = ffma2(make_float2(__uint_as_float(a[e]),
                                                       __uint_as_float(a[e + 1])),
                                           make_float2(sl2, sl2), make_float2(-lrow, -lrow));
                    pr[e] = ex2(x.x);
                    pr[e + 1] = ex2(x.y);
                }
                if (need_mask) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int col = kv0 + e;
                        if (col >= p.N || (p.causal && col > q_row)) pr[e] = 0.f;
                    }
                }
            }
            if (!mbar_wait_warp(dp_full, n & 1, p.ctl, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            {
                uint32_t bv[32];
                tmem_ld32(tdP, bv);
                tmem_wait_ld();
                mbar_arrive_warp(dp_read);  // the dP buffer is free for dP(n+1)
                if constexpr (DROP) {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        bv[e] &= keep_elem_mask(keep[e >> 2], e & 3);
                }
                uint32_t w[16];
                const float2 d2 = make_float2(drow, drow);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float2 ds = fmul2(make_float2(pr[2 * e], pr[2 * e + 1]),
                                            fsub2(make_float2(__uint_as_float(bv[2 * e]),
                                                              __uint_as_float(bv[2 * e + 1])),
                                                  d2));
                    w[e] = pack2<BF16>(ds.x, ds.y);
                }
                tmem_st16(tS, w);  // over columns already read
            }
            mbar_arrive_warp_after_st(&ds_ready[b]);
            ++n;
        }
        if (ok && n > 0) {
            ok = mbar_wait_warp(fin, 0, p.ctl, abort_flag);
            tc_fence_after();
        }
        // group g holds dQ columns [g*d/4, (g+1)*d/4) (times the softmax scale): staged as a
        // 16-bit tile in the (now idle) first K/V ring slot and written by TMA.  Every compute
        // warp reaches the named barrier, whether or not its waits succeeded.
        if (ok) {
            uint8_t *stage = smem + L::kSlotOff;
            const uint32_t tacc = tmem + lane_base + 384 + g * (D / 4);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t a[16];
                if (n > 0) {
                    tmem_ld16(tacc + 16 * cc, a);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) a[e] = 0u;
                }
                const int col = g * (D / 4) + 16 * cc;
                st_box_row<BF16, 16>(stage + (col >> 6) * L::kBoxBytes, row, col & 63, a,
                                     DROP ? p.scale * p.drop.keep_scale : p.scale);
            }
            fence_proxy_async_smem();
        }
        named_sync(1, kComputeThreads);
        if (warp == L::kComputeWarp0 && lane == 0 && ok && *abort_flag == 0) {
            for (int b2 = 0; b2 < L::kBoxes; ++b2)
                tma_store_3d(&tmdq, smem + L::kSlotOff + b2 * L::kBoxBytes, b2 * 64, qt * kTile,
                             bh);
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

// ================================================================================ group reduce
// dK, dV of grouped-query attention whose K/V groups were split over several dK/dV CTAs:
// the sum of the splits' fp32 partials, always added in split order (deterministic), rounded
// once to the 16-bit output type.  8 consecutive elements per thread.
template <bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_group_reduce_kernel(const float *part, void *dk,
                                                                  void *dv, int splits,
                                                                  long kv_elems) {
    const long per = kv_elems / 8;
    const long gid = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (gid >= 2 * per) return;
    const int which = gid >= per ? 1 : 0;  // 0 dK, 1 dV
    const long e = (gid - which * per) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < splits; ++s) {
        const float4 *src = reinterpret_cast<const float4 *>(
            part + (static_cast<long>(which) * splits + s) * kv_elems + e);
        const float4 a = src[0], b = src[1];
        acc[0] += a.x;
        acc[1] += a.y;
        acc[2] += a.z;
        acc[3] += a.w;
        acc[4] += b.x;
        acc[5] += b.y;
        acc[6] += b.z;
        acc[7] += b.w;
    }
    uint4 w;
    w.x = pack2<BF16>(acc[0], acc[1]);
    w.y = pack2<BF16>(acc[2], acc[3]);
    w.z = pack2<BF16>(acc[4], acc[5]);
    w.w = pack2<BF16>(acc[6], acc[7]);
    reinterpret_cast<uint4 *>(static_cast<elem_t<BF16> *>(which ? dv : dk) + e)[0] = w;
}

// Launched with programmatic stream serialization: when the forward kernel is the grid queued
// just before (the usual order, forward then backward), this small kernel's CTAs are scheduled
// beside its last CTAs instead of after its completion; it waits for that grid before reading.
template <int D, bool BF16>
cudaError_t launch_pre_t(const void *o, const void *dout, float *delta, long rows, float mul,
                         cudaStream_t stream) {
    const long threads = rows * (D / 8);
    const long blocks = (threads + 255) / 256;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fa_bwd_preprocess_kernel<D, BF16>, o, dout, delta, rows, mul);
}

// after_dq: the launch directly follows the dQ pass of the same backward call on `stream`; it is
// made with programmatic stream serialization, so its CTAs start on the SMs the dQ grid's last
// CTAs leave idle (the two passes share no output; every CTA of this grid waits for the dQ grid
// before it exits).
template <int D, bool BF16>
cudaError_t launch_dkdv_t(const Maps &m, const BwdParams &p, bool after_dq, cudaStream_t stream) {
    using L = DkvLayout<D>;
    auto kern = p.drop.t4 != 0 ? fa_bwd_dkdv_kernel<D, BF16, true>
                               : fa_bwd_dkdv_kernel<D, BF16, false>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long>(p.units) * p.T));
    cfg.blockDim = dim3(L::kThreads);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_dq ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, m.q, m.k, m.v, m.dout, m.out0, m.out1, p);
}

template <int D, bool BF16>
cudaError_t launch_dq_t(const Maps &m, const BwdParams &p, cudaStream_t stream) {
    using L = DqLayout<D>;
    auto kern = p.drop.t4 != 0 ? fa_bwd_dq_kernel<D, BF16, true> : fa_bwd_dq_kernel<D, BF16, false>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(static_cast<long>(p.BH) * p.T), L::kThreads, L::kAlloc,
           stream>>>(m.q, m.k, m.v, m.dout, m.out0, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess(const void *o, const void *dout, float *delta, long rows,
                                  int d, bool bf16, float mul, cudaStream_t stream) {
    if (d == 64) return bf16 ? launch_pre_t<64, true>(o, dout, delta, rows, mul, stream)
                             : launch_pre_t<64, false>(o, dout, delta, rows, mul, stream);
    return bf16 ? launch_pre_t<128, true>(o, dout, delta, rows, mul, stream)
                : launch_pre_t<128, false>(o, dout, delta, rows, mul, stream);
}

cudaError_t launch_bwd_group_reduce(const float *part, void *dk, void *dv, int splits,
                                    long kv_elems, bool bf16, cudaStream_t stream) {
    const long threads = 2 * (kv_elems / 8);
    const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
    if (bf16)
        fa_bwd_group_reduce_kernel<true><<<blocks, 256, 0, stream>>>(part, dk, dv, splits, kv_elems);
    else
        fa_bwd_group_reduce_kernel<false><<<blocks, 256, 0, stream>>>(part, dk, dv, splits,
                                                                      kv_elems);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const Maps &maps, const BwdParams &p, int d, bool bf16,
                            bool after_dq, cudaStream_t stream) {
    if (d == 64) return bf16 ? launch_dkdv_t<64, true>(maps, p, after_dq, stream)
                             : launch_dkdv_t<64, false>(maps, p, after_dq, stream);
    return bf16 ? launch_dkdv_t<128, true>(maps, p, after_dq, stream)
                : launch_dkdv_t<128, false>(maps, p, after_dq, stream);
}

cudaError_t launch_bwd_dq(const Maps &maps, const BwdParams &p, int d, bool bf16,
                          cudaStream_t stream) {
    if (d == 64) return bf16 ? launch_dq_t<64, true>(maps, p, stream)
                             : launch_dq_t<64, false>(maps, p, stream);
    return bf16 ? launch_dq_t<128, true>(maps, p, stream)
                : launch_dq_t<128, false>(maps, p, stream);
}

}  // namespace fa
