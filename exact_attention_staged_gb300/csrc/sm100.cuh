// sm100.cuh - inline-PTX building blocks for sm_100-family (sm_103a) kernels:
// mbarriers with bounded waits, TMA tile loads, tcgen05 tensor-memory allocation, UMMA
// (tcgen05.mma kind::f16) issue and commit, tensor-memory loads and stores.
//
// Everything here is written against the public PTX ISA.  Operand layouts used by the
// attention kernels:
//   * shared-memory tiles are [rows][64 elements] boxes of 128 bytes per row written by TMA
//     with the 128-byte swizzle, 1024-byte aligned (8-row swizzle atoms of 1024 bytes);
//   * "K-major" operand: the contraction index runs along the 128-byte row;
//   * "MN-major" operand: the output index runs along the 128-byte row and the contraction
//     index runs over rows.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fa {

// ------------------------------------------------------------------------------------------
// control block shared by every kernel: status word, wait bound, hooks
struct Ctl {
    int *status;                      // device status word (FA_ERR_TIMEOUT written on give-up)
    unsigned long long wait_limit_ns; // bound on any single pipeline wait
    uint8_t *visit_log;               // optional per-tile visit bits (nullptr = off)
    int fault_mode;                   // test hook: 1 = forward load warp skips one tile
};

constexpr int kErrTimeout = -4;
constexpr int kErrInternal = -5;  // shared memory misplaced: the kernel did not run

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }
__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }

// ------------------------------------------------------------------------------------------
// mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: the hardware parks the waiting thread until the phase
// completes or the hint (ns) runs out, so a waiting warp does not spin through issue slots that
// the warp sharing its scheduler needs.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false (and records a timeout in
// the status word and in the CTA's abort flag) when the bound runs out, or when another warp
// of the CTA has already given up.  Never traps.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const Ctl &ctl,
                                          volatile int *abort_flag) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(a, parity, 20000u)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > ctl.wait_limit_ns) {
            *abort_flag = 1;
            atomicExch(ctl.status, kErrTimeout);
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag: used only to drain copies and MMAs in flight before
// a CTA that gave up releases its shared and tensor memory.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, const Ctl &ctl) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(a, parity)) {
        if (global_timer_ns() - t0 > ctl.wait_limit_ns) return;
    }
}

// First 1024-byte-aligned address at or after p (the 128-byte swizzle's pattern repeats every
// 1024 bytes, so swizzled tiles start on such a boundary).
__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    const uint32_t a = smem_u32(p);
    return p + ((1024u - (a & 1023u)) & 1023u);
}

// Warp-uniform form of mbar_wait for warps that go on to warp-collective operations
// (tcgen05.ld/st, vote): either every lane of the warp proceeds or none does.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, const Ctl &ctl,
                                               volatile int *abort_flag) {
    const bool ok = mbar_wait(bar, parity, ctl, abort_flag);
    return __all_sync(0xffffffffu, ok) != 0;
}

// ------------------------------------------------------------------------------------------
// TMA: 3-D tiled load (x = element within a row, y = row, z = head) into shared memory,
// completing on an mbarrier with the byte count.
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, int x, int y,
                                            int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// TMA: 3-D tiled store of one box from shared memory (bulk-group completion).  The box is in
// the map's swizzled layout; rows (y) or heads (z) past the tensor's extent are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *smem_src, int x,
                                             int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------------------------------
// cp.async: 4-byte copies global -> shared (zero-filled when `valid` is false), with completion
// reported to an mbarrier so the issuing warp never waits on the global load.
__device__ __forceinline__ void cp_async_4(void *smem_dst, const void *gsrc, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(smem_dst)),
                 "l"(gsrc), "r"(valid ? 4 : 0)
                 : "memory");
}
// 16-byte cp.async through L2 only (streamed data); valid == false writes 16 zero bytes.
__device__ __forceinline__ void cp_async_16(void *smem_dst, const void *gsrc, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
                 "l"(gsrc), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Arrive on `bar` (without raising its expected count) once this thread's cp.async are done.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// ------------------------------------------------------------------------------------------
// tensor memory
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Instruction descriptor for tcgen05.mma kind::f16 with an fp32 accumulator.
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format (0 = f16, 1 = bf16),
//   15 A major (0 = K), 16 B major (0 = K, 1 = MN), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// The same descriptor as two 32-bit halves, so that the MMA issue loop only adds a k-step's
// start-address offset (bytes >> 4) to the low word: no 64-bit arithmetic per MMA.  Valid while
// the start address stays below 256 KB, which every shared-memory address does.
struct SDesc {
    uint32_t lo, hi;
};
__device__ __forceinline__ SDesc sdesc_make(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    SDesc d;
    d.lo = ((saddr & 0x3FFFFu) >> 4) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
    d.hi = ((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
    return d;
}
// As sdesc_make with the 64-byte swizzle (layout type 4): rows of 64 bytes, 8-row atoms of 512.
__device__ __forceinline__ SDesc sdesc_make_sw64(uint32_t saddr, uint32_t lbo_bytes,
                                                 uint32_t sbo_bytes) {
    SDesc d;
    d.lo = ((saddr & 0x3FFFFu) >> 4) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
    d.hi = ((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | (4u << 29);
    return d;
}
__device__ __forceinline__ SDesc sdesc_add(SDesc d, uint32_t byte_offset) {
    d.lo += byte_offset >> 4;
    return d;
}

// e4m3 x e4m3 -> fp32 (tcgen05.mma kind::f8f6f4, K = 32 per instruction): A and B format
// E4M3 (0) in bits 7-9 and 10-12, both operands K-major, D f32 in bits 4-5, N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// e4m3 GEMM chains with one election (as the f16 chains below): 128 x N x 128 from two
// K-major 128-byte-swizzled tiles, 4 k-steps of 32 bytes.
__device__ __forceinline__ void mma_ss_f8_chain_k128(uint32_t d_tmem, SDesc a, SDesc b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b32 al, bl;\n\t.reg .b64 da, db;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.ne.b32 t, %5, 0;\n\t"  // the instruction descriptor is never 0
        "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, p;\n\t"
        "add.u32 al, %1, 2;\n\tadd.u32 bl, %3, 2;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, t;\n\t"
        "add.u32 al, %1, 4;\n\tadd.u32 bl, %3, 4;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, t;\n\t"
        "add.u32 al, %1, 6;\n\tadd.u32 bl, %3, 6;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, t;\n\t"
        "}" ::"r"(d_tmem), "r"(a.lo), "r"(a.hi), "r"(b.lo), "r"(b.hi), "r"(idesc),
        "r"(accumulate));
}
// The same over 64 contraction bytes (2 k-steps).
__device__ __forceinline__ void mma_ss_f8_chain_k64(uint32_t d_tmem, SDesc a, SDesc b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b32 al, bl;\n\t.reg .b64 da, db;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.ne.b32 t, %5, 0;\n\t"  // the instruction descriptor is never 0
        "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, p;\n\t"
        "add.u32 al, %1, 2;\n\tadd.u32 bl, %3, 2;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, t;\n\t"
        "}" ::"r"(d_tmem), "r"(a.lo), "r"(a.hi), "r"(b.lo), "r"(b.hi), "r"(idesc),
        "r"(accumulate));
}
// 128 x N x 128 with A (four e4m3 per column) in tensor memory, 8 columns per k-step, and a
// K-major B whose k-steps are 32 bytes apart.
__device__ __forceinline__ void mma_ts_f8_chain_k128(uint32_t d_tmem, uint32_t a_tmem, SDesc b,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b32 at, bl;\n\t.reg .b64 db;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "setp.ne.b32 t, %4, 0;\n\t"  // the instruction descriptor is never 0
        "mov.b64 db, {%2, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], db, %4, p;\n\t"
        "add.u32 at, %1, 8;\n\tadd.u32 bl, %2, 2;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 16;\n\tadd.u32 bl, %2, 4;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 24;\n\tadd.u32 bl, %2, 6;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [at], db, %4, t;\n\t"
        "}" ::"r"(d_tmem), "r"(a_tmem), "r"(b.lo), "r"(b.hi), "r"(idesc), "r"(accumulate));
}

// Four fp32 values to e4m3 (round to nearest, saturating to +-448) in one word, e0 in the
// lowest byte (the lowest contraction index).  PTX cvt ... e4m3x2 puts its first source in
// the upper byte of the pair.
__device__ __forceinline__ uint32_t pack4_e4m3(float e0, float e1, float e2, float e3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(e1), "f"(e0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(e3), "f"(e2));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Whole GEMM chains in one instruction sequence with a single election: fewer issue slots per
// MMA for the issuing warp, which shares its sub-partition with busy element-wise warps.  The
// whole warp runs the issue loop in lockstep (every lane computes the warp-uniform operands)
// and one lane chosen by elect.sync issues: keeping the issuing warp converged lets its
// address arithmetic and waits run at full rate next to busy compute warps, which a
// single-lane issue path inside a divergent branch does not (measured on GB300: 74 vs 64
// cycles per 128 x 128 x 16 MMA taking A from tensor memory, with three busy warps alongside).
// 128 x N x 128 from two K-major 128-byte-swizzled tiles of two 64-wide boxes each (16 KB
// apart): D (+)= A B^T over 8 k-steps; only the first k-step uses `accumulate`.
__device__ __forceinline__ void mma_ss_chain_k128(uint32_t d_tmem, SDesc a, SDesc b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b32 al, bl;\n\t.reg .b64 da, db;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.ne.b32 t, %5, 0;\n\t"  // the instruction descriptor is never 0
        "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t"
        "add.u32 al, %1, 2;\n\tadd.u32 bl, %3, 2;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t"
        "add.u32 al, %1, 4;\n\tadd.u32 bl, %3, 4;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t"
        "add.u32 al, %1, 6;\n\tadd.u32 bl, %3, 6;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t"
        "add.u32 al, %1, 1024;\n\tadd.u32 bl, %3, 1024;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t"
        "add.u32 al, %1, 1026;\n\tadd.u32 bl, %3, 1026;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t"
        "add.u32 al, %1, 1028;\n\tadd.u32 bl, %3, 1028;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t"
        "add.u32 al, %1, 1030;\n\tadd.u32 bl, %3, 1030;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t"
        "}" ::"r"(d_tmem), "r"(a.lo), "r"(a.hi), "r"(b.lo), "r"(b.hi), "r"(idesc),
        "r"(accumulate));
}
// The same over one 64-wide box (4 k-steps).
__device__ __forceinline__ void mma_ss_chain_k64(uint32_t d_tmem, SDesc a, SDesc b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b32 al, bl;\n\t.reg .b64 da, db;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.ne.b32 t, %5, 0;\n\t"  // the instruction descriptor is never 0
        "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t"
        "add.u32 al, %1, 2;\n\tadd.u32 bl, %3, 2;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t"
        "add.u32 al, %1, 4;\n\tadd.u32 bl, %3, 4;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t"
        "add.u32 al, %1, 6;\n\tadd.u32 bl, %3, 6;\n\t"
        "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, t;\n\t"
        "}" ::"r"(d_tmem), "r"(a.lo), "r"(a.hi), "r"(b.lo), "r"(b.hi), "r"(idesc),
        "r"(accumulate));
}
// 128 x N x 128 with A (16-bit pairs) in tensor memory, 8 columns per k-step, and an
// MN-major B whose k-steps are 2048 bytes apart: D (+)= A B over 8 k-steps.
__device__ __forceinline__ void mma_ts_chain_k128(uint32_t d_tmem, uint32_t a_tmem, SDesc b,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b32 at, bl;\n\t.reg .b64 db;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "setp.ne.b32 t, %4, 0;\n\t"  // the instruction descriptor is never 0
        "mov.b64 db, {%2, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t"
        "add.u32 at, %1, 8;\n\tadd.u32 bl, %2, 128;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 16;\n\tadd.u32 bl, %2, 256;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 24;\n\tadd.u32 bl, %2, 384;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 32;\n\tadd.u32 bl, %2, 512;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 40;\n\tadd.u32 bl, %2, 640;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 48;\n\tadd.u32 bl, %2, 768;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 56;\n\tadd.u32 bl, %2, 896;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "}" ::"r"(d_tmem), "r"(a_tmem), "r"(b.lo), "r"(b.hi), "r"(idesc), "r"(accumulate));
}
// As mma_ts_chain_k128 with A packed by groups of 32 contraction indices, each group's
// 16 columns 32 columns apart (k-step k at column 32 (k / 2) + 8 (k % 2)).
__device__ __forceinline__ void mma_ts_chain_k128_g32(uint32_t d_tmem, uint32_t a_tmem, SDesc b,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b32 at, bl;\n\t.reg .b64 db;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "setp.ne.b32 t, %4, 0;\n\t"  // the instruction descriptor is never 0
        "mov.b64 db, {%2, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t"
        "add.u32 at, %1, 8;\n\tadd.u32 bl, %2, 128;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 32;\n\tadd.u32 bl, %2, 256;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 40;\n\tadd.u32 bl, %2, 384;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 64;\n\tadd.u32 bl, %2, 512;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 72;\n\tadd.u32 bl, %2, 640;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 96;\n\tadd.u32 bl, %2, 768;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "add.u32 at, %1, 104;\n\tadd.u32 bl, %2, 896;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %4, t;\n\t"
        "}" ::"r"(d_tmem), "r"(a_tmem), "r"(b.lo), "r"(b.hi), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit_el(uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        ::"r"(smem_u32(bar))
        : "memory");
}

// Each thread of the warp reads its own lane (row) of tensor memory, 32 consecutive 32-bit
// columns starting at taddr's column.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Register rebalancing between warpgroups (all four warps of a warpgroup execute it): the
// counts are immediates, multiples of 8 in [24, 256], and the CTA's total must stay within the
// registers it was launched with.
template <int N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Programmatic dependent launch (PTX griddepcontrol).  launch_dependents: this CTA no longer
// holds back the grid launched after it with programmatic stream serialization (that grid starts
// once every CTA of this one has signalled or exited).  wait: block until the grids this one was
// allowed to overlap have completed and their memory operations are visible; returns at once
// for a grid launched without that attribute.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Cluster launch control (PTX clusterlaunchcontrol, sm_100 and later).  try_cancel asks the
// hardware to cancel one CTA of this grid that has not started yet; the 16-byte answer lands in
// shared memory (16-byte aligned) and completes 16 transaction bytes on `bar`, whose expected
// count the caller has raised.  A CTA that wins a cancelled CTA's index does that CTA's work,
// so a grid of one CTA per work unit runs as a persistent grid that the hardware keeps fed in
// launch order.  After a failed answer (nothing left to cancel) no further request is made.
__device__ __forceinline__ void clc_try_cancel(void *resp16, uint64_t *bar) {
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128"
        " [%0], [%1];" ::"r"(smem_u32(resp16)),
        "r"(smem_u32(bar))
        : "memory");
}
// x index of the CTA an answer cancelled, or -1 when it cancelled none.
__device__ __forceinline__ int clc_cancelled_x(const void *resp16) {
    uint32_t ok, x;
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b128 r;\n\t"
        "ld.shared.b128 r, [%2];\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "mov.u32 %1, 0;\n\t"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
        : "=r"(ok), "=r"(x)
        : "r"(smem_u32(resp16))
        : "memory");
    return ok ? static_cast<int>(x) : -1;
}

// 2^x on the special-function unit (PTX ex2.approx, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max of three values in one instruction (PTX max.f32 with three sources, sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Largest of the 128 scores of a row: eight independent chains of three-input maxima.
__device__ __forceinline__ float row_max128(const uint32_t *r) {
    float a[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        a[k] = fmax3(__uint_as_float(r[k]), __uint_as_float(r[8 + k]), __uint_as_float(r[16 + k]));
#pragma unroll
    for (int c = 24; c < 120; c += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k)
            a[k] = fmax3(a[k], __uint_as_float(r[c + k]), __uint_as_float(r[c + 8 + k]));
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = fmaxf(a[k], __uint_as_float(r[120 + k]));
    return fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
}

// Paired fp32 arithmetic (PTX f32x2 forms, sm_100 and later): one instruction for two lanes of
// work, round to nearest.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// One mbarrier arrival per warp once every lane is past this point, its tensor-memory loads
// waited for (the barrier is initialised with the number of arriving warps).
__device__ __forceinline__ void mbar_arrive_warp(uint64_t *bar) {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
// The same after every lane's prior tensor-memory stores have completed.
__device__ __forceinline__ void mbar_arrive_warp_after_st(uint64_t *bar) {
    tmem_wait_st();
    mbar_arrive_warp(bar);
}

// Pack two fp32 values into one 32-bit word of two 16-bit values, round to nearest even;
// `lo` lands in the low half (the lower contraction index).
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

// NV (16 or 32) consecutive values of one row (times mul) as 16-bit values into a 128-row x
// 64-element box laid out as a TMA tile with the 128-byte swizzle (16-byte chunk c of row r at
// r * 128 + (c ^ (r % 8)) * 16; the box is 1024-byte aligned).  col: the first element's column
// within the box, a multiple of 8.
template <bool BF16, int NV>
__device__ __forceinline__ void st_box_row(uint8_t *box, int row, int col, const uint32_t *v,
                                           float mul) {
    uint32_t w[NV / 2];
#pragma unroll
    for (int e = 0; e < NV / 2; ++e)
        w[e] = pack2<BF16>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
#pragma unroll
    for (int q = 0; q < NV / 8; ++q) {
        const int chunk = ((col >> 3) + q) ^ (row & 7);
        *reinterpret_cast<uint4 *>(box + row * 128 + chunk * 16) =
            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    if constexpr (BF16) {
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&w);
        return __bfloat1622float2(h);
    } else {
        __half2 h = *reinterpret_cast<__half2 *>(&w);
        return __half22float2(h);
    }
}

}  // namespace fa
