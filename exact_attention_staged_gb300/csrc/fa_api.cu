// fa_api.cu - the C ABI of libfa.so: argument validation, TMA tensor maps, launches, and the
// per-device status word that bounded pipeline waits report into.  See include/fa.h.
#include "fa.h"
#include "fa_internal.h"

#include <cmath>
#include <cstdio>
#include <cudaTypedefs.h>
#include <mutex>

namespace {

__device__ int g_fa_status;  // one per device: FA_OK or the first device-side error

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s

std::mutex g_mu;
int *g_status_ptr[kMaxDevices] = {};
int g_arch_ok[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other
uint8_t *g_visit_log = nullptr;
size_t g_visit_bytes = 0;
unsigned long long g_wait_ns = kDefaultWaitNs;
int g_fault_mode = 0;
int g_dkdv_splits = 0;  // 0: automatic
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Device status word address and architecture check, once per device.
int device_setup(int *dev_out, int **status_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_arch_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (g_arch_ok[dev] != 1) return FA_ERR_UNSUPPORTED;
    if (g_status_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return FA_ERR_CUDA;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return FA_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *dev_out = dev;
    *status_out = g_status_ptr[dev];
    return FA_OK;
}

// Snapshot of the debug hooks for one launch; the visit log must cover every tile of it.
int make_ctl(int *status, int BH, int T, fa::Ctl *out) {
    std::lock_guard<std::mutex> lk(g_mu);
    // the marks are 32-bit atomic ORs: the log covers every tile, rounded up to whole words
    const size_t need = static_cast<size_t>(BH) * static_cast<size_t>(T) * static_cast<size_t>(T);
    if (g_visit_log != nullptr && g_visit_bytes < (need + 3) / 4 * 4) return FA_ERR_INVALID;
    fa::Ctl &c = *out;
    c.status = status;
    c.wait_limit_ns = g_wait_ns;
    c.visit_log = g_visit_log;
    c.fault_mode = g_fault_mode;
    return FA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int B, int H, int N, int d, int dtype, float scale) {
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID;
    if (static_cast<long long>(B) * H * N >= (1ll << 31)) return FA_ERR_INVALID;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_INVALID;
    if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

// A block mask has T x T entries (T = ceil(N / 128)); the kernels index it with 32-bit
// arithmetic, so T may not exceed 46340 (T^2 < 2^31, N <= 5931520).
constexpr int kMaxMaskTiles = 46340;
int check_mask(const uint8_t *mask, int N) {
    return mask != nullptr && (N + 127) / 128 > kMaxMaskTiles ? FA_ERR_INVALID : FA_OK;
}

int check_ptrs(std::initializer_list<const void *> ptrs) {
    for (const void *p : ptrs)
        if (p == nullptr || !aligned16(p)) return FA_ERR_INVALID;
    return FA_OK;
}

// [B*H, N, d] 16-bit tensor, 64 x box_rows boxes (128 bytes x box_rows rows), 128-byte swizzle.
int make_map(CUtensorMap *m, const void *base, int BH, int N, int d, int dtype,
             int box_rows = 128) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m,
                          dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// 3-D byte tensor (e4m3 codes): dims x (contiguous), y, z; box box_x bytes x box_y rows with
// the swizzle that matches box_x (128 or 64 bytes).
int make_map_bytes(CUtensorMap *m, const void *base, long x, long y, long z, int box_x,
                   int box_y) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(x), static_cast<cuuint64_t>(y),
                          static_cast<cuuint64_t>(z)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(x), static_cast<cuuint64_t>(x * y)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_x), static_cast<cuuint32_t>(box_y), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          box_x == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

int tiles_of(int N) { return (N + fa::kTile - 1) / fa::kTile; }

// Dropout decisions: drop probability p -> byte threshold t = nearest integer to 256 p (ties to
// even), valid for 0 <= t <= 255; t = 0 turns dropout off.  The offset is a 32-bit counter word
// of the generator.
constexpr fa::DropSpec kNoDrop = {0u, 1.f, 0ull, 0ull, {}};
int make_drop(float p, unsigned long long seed, unsigned long long offset, fa::DropSpec *out) {
    if (!(p >= 0.f && p < 1.f)) return FA_ERR_INVALID;
    if (offset > 0xFFFFFFFFull) return FA_ERR_INVALID;  // a 32-bit counter word
    const long t = std::lrint(static_cast<double>(p) * 256.0);
    if (t < 0 || t > 255) return FA_ERR_INVALID;
    out->t4 = static_cast<uint32_t>(t) * 0x01010101u;
    out->keep_scale = static_cast<float>(256.0 / (256.0 - static_cast<double>(t)));
    out->seed = seed;
    out->offset = offset;
    fa::philox_round_keys(*out);
    return FA_OK;
}

int check_heads(int H, int Hkv) {
    return (Hkv >= 1 && Hkv <= H && H % Hkv == 0) ? FA_OK : FA_ERR_INVALID;
}

// CTA-order group size: `units` work-unit heads, each streaming `tensors_per_unit` [N, d]
// 16-bit tensors; the group's streamed tiles stay near 32 MiB, a quarter of the L2.
int head_group(int units, int N, int d, double tensors_per_unit) {
    const double per_unit = 2.0 * N * d * tensors_per_unit;
    int g = static_cast<int>((32.0 * 1024 * 1024) / per_unit);
    if (g < 1) g = 1;
    if (g > units) g = units;
    return g;
}

// How the dK/dV kernel spreads the H / H_kv query heads of one K/V head: over `splits` CTAs
// per key tile, `chunk` heads each, aiming at no fewer than kDkvTargetCtas CTAs (a few per SM)
// so that few K/V heads (MQA) still fill the GPU.  One split needs no partial sums.
constexpr long kDkvTargetCtas = 512;
struct DkvSplit {
    int splits, chunk;
};
DkvSplit dkdv_split(int B, int H, int Hkv, int N) {
    const int rep = H / Hkv;
    int s = 1;
    if (rep > 1) {
        int forced;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            forced = g_dkdv_splits;
        }
        if (forced > 0) {
            s = forced;
        } else {
            const long units = static_cast<long>(B) * Hkv * tiles_of(N);
            s = static_cast<int>((kDkvTargetCtas + units - 1) / units);
        }
        if (s > rep) s = rep;
        if (s < 1) s = 1;
    }
    const int chunk = (rep + s - 1) / s;
    return {(rep + chunk - 1) / chunk, chunk};
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

size_t delta_bytes(int B, int H, int N) {
    return round256(static_cast<size_t>(B) * H * N * sizeof(float));
}

size_t part_bytes(const DkvSplit &sp, int B, int Hkv, int N, int d) {
    if (sp.splits == 1) return 0;
    return 2ull * sp.splits * static_cast<size_t>(B) * Hkv * N * d * sizeof(float);
}

int fwd_common(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
               int Hkv, int N, int d, int dtype, float scale, int causal, const uint8_t *mask,
               const fa::DropSpec &drop, void *stream) {
    int rc = check_shape(B, H, N, d, dtype, scale);
    if (rc != FA_OK) return rc;
    rc = check_mask(mask, N);
    if (rc != FA_OK) return rc;
    rc = check_heads(H, Hkv);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({q, k, v, o, lse});
    if (rc != FA_OK) return rc;
    int dev = 0, *status = nullptr;
    rc = device_setup(&dev, &status);
    if (rc != FA_OK) return rc;
    fa::Maps maps;
    const int BH = B * H;
    // the forward stores O row by row from registers: no output map
    if (make_map(&maps.q, q, BH, N, d, dtype) || make_map(&maps.k, k, B * Hkv, N, d, dtype) ||
        make_map(&maps.v, v, B * Hkv, N, d, dtype))
        return FA_ERR_CUDA;
    maps.out0 = maps.out1 = maps.q;
    fa::FwdParams p;
    p.o = o;
    p.lse = lse;
    p.mask = mask;
    p.BH = BH;
    p.N = N;
    p.T = tiles_of(N);
    p.num_pairs = (p.T + 1) / 2;
    p.rep = H / Hkv;
    p.head_group = head_group(BH, N, d, 2.0 / p.rep);  // K and V, shared by rep query heads
    p.scale_log2 = scale * 1.4426950408889634f;
    p.causal = causal ? 1 : 0;
    p.drop = drop;
    if (make_ctl(status, BH, p.T, &p.ctl) != FA_OK) return FA_ERR_INVALID;
    cudaError_t e = fa::launch_fwd(maps, p, d, dtype == FA_BF16, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int bwd_params(const void *q, const void *k, const void *v, const void *dout, const float *lse,
               const float *delta, int B, int H, int Hkv, int N, int d, int dtype, float scale,
               int causal, const uint8_t *mask, const fa::DropSpec &drop, fa::Maps *maps,
               fa::BwdParams *p) {
    int rc = check_shape(B, H, N, d, dtype, scale);
    if (rc != FA_OK) return rc;
    rc = check_mask(mask, N);
    if (rc != FA_OK) return rc;
    rc = check_heads(H, Hkv);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({q, k, v, dout, lse, delta});
    if (rc != FA_OK) return rc;
    int dev = 0, *status = nullptr;
    rc = device_setup(&dev, &status);
    if (rc != FA_OK) return rc;
    const int BH = B * H;
    if (make_map(&maps->q, q, BH, N, d, dtype) || make_map(&maps->k, k, B * Hkv, N, d, dtype) ||
        make_map(&maps->v, v, B * Hkv, N, d, dtype) ||
        make_map(&maps->dout, dout, BH, N, d, dtype))
        return FA_ERR_CUDA;
    p->out0 = nullptr;
    p->out1 = nullptr;
    p->lse = lse;
    p->delta = delta;
    p->mask = mask;
    p->BH = BH;
    p->N = N;
    p->T = tiles_of(N);
    p->rep = H / Hkv;
    p->head_group = head_group(BH, N, d, 2.0 / p->rep);  // dQ: K and V per query head
    p->units = BH;
    p->splits = 1;
    p->chunk = p->rep;
    p->part = nullptr;
    p->kv_elems = static_cast<long>(B) * Hkv * N * d;
    p->scale = scale;
    p->scale_log2 = scale * 1.4426950408889634f;
    p->causal = causal ? 1 : 0;
    p->drop = drop;
    return make_ctl(status, BH, p->T, &p->ctl);
}

// dK/dV (+ the group reduce when the K/V groups are split, sp.splits > 1); part: room for
// part_bytes(sp, ...) of fp32 partial sums, or nullptr with one split.
// after_dq: queued right after the dQ pass of the same call (see fa::launch_bwd_dkdv).
int run_dkdv(const void *q, const void *k, const void *v, const void *dout, const float *lse,
             const float *delta, void *dk, void *dv, const DkvSplit &sp, float *part, int B,
             int H, int Hkv, int N, int d, int dtype, float scale, int causal,
             const uint8_t *mask, const fa::DropSpec &drop, bool after_dq, void *stream) {
    fa::Maps maps;
    fa::BwdParams p;
    int rc = bwd_params(q, k, v, dout, lse, delta, B, H, Hkv, N, d, dtype, scale, causal, mask,
                        drop, &maps, &p);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({dk, dv});
    if (rc != FA_OK) return rc;
    if (sp.splits < 1 || sp.chunk < 1 || sp.splits * sp.chunk < H / Hkv) return FA_ERR_INVALID;
    if (sp.splits > 1 && (part == nullptr || !aligned16(part))) return FA_ERR_INVALID;
    p.out0 = dk;
    p.out1 = dv;
    p.splits = sp.splits;
    p.chunk = sp.chunk;
    p.units = B * Hkv * sp.splits;
    p.part = sp.splits > 1 ? part : nullptr;
    p.head_group = head_group(p.units, N, d, 2.0 * sp.chunk);  // Q and dO of chunk heads
    if (sp.splits == 1) {  // dK, dV written by TMA; split groups write fp32 partials instead
        if (make_map(&maps.out0, dk, B * Hkv, N, d, dtype) ||
            make_map(&maps.out1, dv, B * Hkv, N, d, dtype))
            return FA_ERR_CUDA;
    } else {
        maps.out0 = maps.k;
        maps.out1 = maps.v;
    }
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = fa::launch_bwd_dkdv(maps, p, d, dtype == FA_BF16, after_dq, st);
    if (e == cudaSuccess && sp.splits > 1)
        e = fa::launch_bwd_group_reduce(part, dk, dv, sp.splits, p.kv_elems, dtype == FA_BF16, st);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int run_dq(const void *q, const void *k, const void *v, const void *dout, const float *lse,
           const float *delta, void *dq, int B, int H, int Hkv, int N, int d, int dtype,
           float scale, int causal, const uint8_t *mask, const fa::DropSpec &drop, void *stream) {
    fa::Maps maps;
    fa::BwdParams p;
    int rc = bwd_params(q, k, v, dout, lse, delta, B, H, Hkv, N, d, dtype, scale, causal, mask,
                        drop, &maps, &p);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({dq});
    if (rc != FA_OK) return rc;
    if (make_map(&maps.out0, dq, B * H, N, d, dtype)) return FA_ERR_CUDA;
    maps.out1 = maps.q;
    p.out0 = dq;
    cudaError_t e =
        fa::launch_bwd_dq(maps, p, d, dtype == FA_BF16, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int run_preprocess(const void *o, const void *dout, float *delta, int B, int H, int N, int d,
                   int dtype, void *stream, float mul = 1.f) {
    int rc = check_shape(B, H, N, d, dtype, 1.f);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({o, dout, delta});
    if (rc != FA_OK) return rc;
    int dev = 0, *status = nullptr;
    rc = device_setup(&dev, &status);
    if (rc != FA_OK) return rc;
    cudaError_t e = fa::launch_bwd_preprocess(o, dout, delta, static_cast<long>(B) * H * N, d,
                                              dtype == FA_BF16, mul,
                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// The whole backward: D, then dQ and dK/dV.  delta: B*H*N floats; sp, part: see run_dkdv.
// The two passes read the same inputs and write disjoint outputs, so with one dK/dV split the
// dK/dV grid is queued after the dQ grid with programmatic stream serialization: its CTAs fill
// the SMs that the dQ grid's last wave leaves idle.  Split K/V groups keep the plain order
// dK/dV, group reduce, dQ.
int run_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
            const float *lse, void *dq, void *dk, void *dv, float *delta, const DkvSplit &sp,
            float *part, int B, int H, int Hkv, int N, int d, int dtype, float scale, int causal,
            const uint8_t *mask, const fa::DropSpec &drop, void *stream) {
    // with dropout the passes take D / s (s = 256 / (256 - t) the keep scale): dS = s P o (Z o dP
    // - D / s), so a kept dP needs no multiply and dK, dQ take the factor s at the end
    const float dmul =
        drop.t4 != 0 ? static_cast<float>((256.0 - static_cast<double>(drop.t4 & 0xFFu)) / 256.0)
                     : 1.f;
    int rc = run_preprocess(o, dout, delta, B, H, N, d, dtype, stream, dmul);
    if (rc != FA_OK) return rc;
    if (sp.splits == 1) {
        rc = run_dq(q, k, v, dout, lse, delta, dq, B, H, Hkv, N, d, dtype, scale, causal, mask,
                    drop, stream);
        if (rc != FA_OK) return rc;
        return run_dkdv(q, k, v, dout, lse, delta, dk, dv, sp, part, B, H, Hkv, N, d, dtype,
                        scale, causal, mask, drop, true, stream);
    }
    rc = run_dkdv(q, k, v, dout, lse, delta, dk, dv, sp, part, B, H, Hkv, N, d, dtype, scale,
                  causal, mask, drop, false, stream);
    if (rc != FA_OK) return rc;
    return run_dq(q, k, v, dout, lse, delta, dq, B, H, Hkv, N, d, dtype, scale, causal, mask,
                  drop, stream);
}

// fa_bwd_gqa / fa_bwd_dropout: validation, workspace split, run_bwd.
int bwd_entry(const void *q, const void *k, const void *v, const void *o, const void *dout,
              const float *lse, void *dq, void *dk, void *dv, void *workspace,
              size_t workspace_bytes, int B, int H, int H_kv, int N, int d, int dtype,
              float scale, int causal, const uint8_t *block_mask, const fa::DropSpec &drop,
              void *stream) {
    int rc = check_shape(B, H, N, d, dtype, scale);
    if (rc != FA_OK) return rc;
    rc = check_mask(block_mask, N);
    if (rc != FA_OK) return rc;
    rc = check_heads(H, H_kv);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({q, k, v, o, dout, lse, dq, dk, dv, workspace});
    if (rc != FA_OK) return rc;
    const size_t need_delta = delta_bytes(B, H, N);
    const DkvSplit sp = dkdv_split(B, H, H_kv, N);  // once: the size check and the launch agree
    const size_t need_part = part_bytes(sp, B, H_kv, N, d);
    if (workspace_bytes < need_delta + need_part) return FA_ERR_INVALID;
    float *delta = static_cast<float *>(workspace);
    float *part = need_part ? reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                                        need_delta)
                            : nullptr;
    return run_bwd(q, k, v, o, dout, lse, dq, dk, dv, delta, sp, part, B, H, H_kv, N, d, dtype,
                   scale, causal, block_mask, drop, stream);
}

// Key ranges of decode: a unit is (K/V head, key range, group of up to 128 query rows) and the
// grid runs one CTA per SM that walks the units, so the ranges are cut to give each SM about
// eight units (the last ones then finish within about an eighth of a unit of each other) but
// never shorter than four 128-key tiles.
constexpr long kDecodeUnitsTarget = 8 * 152;
struct DecodeSplit {
    int splits, chunk, row_groups;
};
DecodeSplit decode_split(int B, int H, int Hkv, int Nq, int Nk) {
    const int rows = (H / Hkv) * Nq;
    const int row_groups = (rows + 127) / 128;
    const long units = static_cast<long>(B) * Hkv * row_groups;
    long s = (kDecodeUnitsTarget + units - 1) / units;
    const long max_s = (Nk + 511) / 512;
    if (s > max_s) s = max_s;
    if (s < 1) s = 1;
    int chunk = static_cast<int>((Nk + s - 1) / s);
    chunk = (chunk + 127) / 128 * 128;
    return {(Nk + chunk - 1) / chunk, chunk, row_groups};
}

size_t decode_part_bytes(const DecodeSplit &sp, int B, int H, int Nq, int d) {
    if (sp.splits == 1) return 0;
    const size_t rows = static_cast<size_t>(B) * H * Nq * sp.splits;
    return rows * d * sizeof(float) + rows * 2 * sizeof(float);
}

// Scratch of fa_bwd_noalloc: the D values (one float per query row) of one backward call.
// Host code must not pass this name to a kernel: on the host it only stands in for the
// symbol; noalloc_scratch() looks up its device address once per device.
static __device__ __align__(256) float g_noalloc_delta[FA_NOALLOC_MAX_ROWS];
float *g_noalloc_ptr[kMaxDevices] = {};

int noalloc_scratch(int dev, float **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_delta) != cudaSuccess || p == nullptr)
            return FA_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_noalloc_ptr[dev];
    return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int N,
           int d, int dtype, float scale, int causal, void *stream) {
    return fwd_common(q, k, v, o, lse, B, H, H, N, d, dtype, scale, causal, nullptr, kNoDrop,
                      stream);
}

int fa_fwd_blocksparse(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                       int H, int N, int d, int dtype, float scale, int causal,
                       const uint8_t *block_mask, void *stream) {
    if (block_mask == nullptr) return FA_ERR_INVALID;
    return fwd_common(q, k, v, o, lse, B, H, H, N, d, dtype, scale, causal, block_mask, kNoDrop,
                      stream);
}

int fa_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
               int H_kv, int N, int d, int dtype, float scale, int causal,
               const uint8_t *block_mask, void *stream) {
    return fwd_common(q, k, v, o, lse, B, H, H_kv, N, d, dtype, scale, causal, block_mask,
                      kNoDrop, stream);
}

int fa_fwd_dropout(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                   int H, int H_kv, int N, int d, int dtype, float scale, int causal,
                   const uint8_t *block_mask, float p_drop, unsigned long long seed,
                   unsigned long long offset, void *stream) {
    fa::DropSpec drop;
    if (make_drop(p_drop, seed, offset, &drop) != FA_OK) return FA_ERR_INVALID;
    return fwd_common(q, k, v, o, lse, B, H, H_kv, N, d, dtype, scale, causal, block_mask, drop,
                      stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
    (void)d;
    if (B < 1 || H < 1 || N < 1) return 0;
    return delta_bytes(B, H, N);
}

size_t fa_bwd_gqa_workspace_bytes(int B, int H, int H_kv, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || check_heads(H, H_kv) != FA_OK) return 0;
    return delta_bytes(B, H, N) + part_bytes(dkdv_split(B, H, H_kv, N), B, H_kv, N, d);
}

int fa_bwd_preprocess(const void *o, const void *dout, float *delta, int B, int H, int N, int d,
                      int dtype, void *stream) {
    return run_preprocess(o, dout, delta, B, H, N, d, dtype, stream);
}

int fa_bwd_dkdv(const void *q, const void *k, const void *v, const void *dout, const float *lse,
                const float *delta, void *dk, void *dv, int B, int H, int N, int d, int dtype,
                float scale, int causal, const uint8_t *block_mask, void *stream) {
    return run_dkdv(q, k, v, dout, lse, delta, dk, dv, DkvSplit{1, 1}, nullptr, B, H, H, N, d,
                    dtype, scale, causal, block_mask, kNoDrop, false, stream);
}

int fa_bwd_dq(const void *q, const void *k, const void *v, const void *dout, const float *lse,
              const float *delta, void *dq, int B, int H, int N, int d, int dtype, float scale,
              int causal, const uint8_t *block_mask, void *stream) {
    return run_dq(q, k, v, dout, lse, delta, dq, B, H, H, N, d, dtype, scale, causal, block_mask,
                  kNoDrop, stream);
}

int fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
           const float *lse, void *dq, void *dk, void *dv, void *workspace,
           size_t workspace_bytes, int B, int H, int N, int d, int dtype, float scale,
           int causal, const uint8_t *block_mask, void *stream) {
    return fa_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, H, N,
                      d, dtype, scale, causal, block_mask, stream);
}

int fa_bwd_gqa(const void *q, const void *k, const void *v, const void *o, const void *dout,
               const float *lse, void *dq, void *dk, void *dv, void *workspace,
               size_t workspace_bytes, int B, int H, int H_kv, int N, int d, int dtype,
               float scale, int causal, const uint8_t *block_mask, void *stream) {
    return bwd_entry(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, H_kv,
                     N, d, dtype, scale, causal, block_mask, kNoDrop, stream);
}

int fa_bwd_dropout(const void *q, const void *k, const void *v, const void *o, const void *dout,
                   const float *lse, void *dq, void *dk, void *dv, void *workspace,
                   size_t workspace_bytes, int B, int H, int H_kv, int N, int d, int dtype,
                   float scale, int causal, const uint8_t *block_mask, float p_drop,
                   unsigned long long seed, unsigned long long offset, void *stream) {
    fa::DropSpec drop;
    if (make_drop(p_drop, seed, offset, &drop) != FA_OK) return FA_ERR_INVALID;
    return bwd_entry(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, H_kv,
                     N, d, dtype, scale, causal, block_mask, drop, stream);
}

int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const void *dout,
                   const float *lse, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                   int dtype, float scale, int causal, const uint8_t *block_mask, void *stream) {
    int rc = check_shape(B, H, N, d, dtype, scale);
    if (rc != FA_OK) return rc;
    rc = check_mask(block_mask, N);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({q, k, v, o, dout, lse, dq, dk, dv});
    if (rc != FA_OK) return rc;
    if (static_cast<size_t>(B) * H * N > FA_NOALLOC_MAX_ROWS) return FA_ERR_INVALID;
    int dev = 0, *status = nullptr;
    rc = device_setup(&dev, &status);
    if (rc != FA_OK) return rc;
    float *delta = nullptr;
    rc = noalloc_scratch(dev, &delta);
    if (rc != FA_OK) return rc;
    return run_bwd(q, k, v, o, dout, lse, dq, dk, dv, delta, DkvSplit{1, 1}, nullptr, B, H, H, N,
                   d, dtype, scale, causal, block_mask, kNoDrop, stream);
}

size_t fa_fwd_fp8_workspace_bytes(int B, int H_kv, int N, int d) {
    if (B < 1 || H_kv < 1 || N < 1 || (d != 64 && d != 128)) return 0;
    const size_t np = (static_cast<size_t>(N) + 15) / 16 * 16;
    return round256(static_cast<size_t>(B) * H_kv * d * np);
}

int fa_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
               int H_kv, int N, int d, float scale, float descale_q, float descale_k,
               float descale_v, int causal, const uint8_t *block_mask, void *workspace,
               size_t workspace_bytes, void *stream) {
    int rc = check_shape(B, H, N, d, FA_BF16, scale);
    if (rc != FA_OK) return rc;
    rc = check_mask(block_mask, N);
    if (rc != FA_OK) return rc;
    rc = check_heads(H, H_kv);
    if (rc != FA_OK) return rc;
    for (float x : {descale_q, descale_k, descale_v})
        if (!(std::isfinite(x) && x > 0.f)) return FA_ERR_INVALID;
    rc = check_ptrs({q, k, v, o, lse, workspace});
    if (rc != FA_OK) return rc;
    if (workspace_bytes < fa_fwd_fp8_workspace_bytes(B, H_kv, N, d)) return FA_ERR_INVALID;
    int dev = 0, *status = nullptr;
    rc = device_setup(&dev, &status);
    if (rc != FA_OK) return rc;
    const int Np = (N + 15) / 16 * 16;
    uint8_t *vt = static_cast<uint8_t *>(workspace);
    fa::Fp8Maps maps;
    if (make_map_bytes(&maps.q, q, d, N, static_cast<long>(B) * H, d, fa::kTile) ||
        make_map_bytes(&maps.k, k, d, N, static_cast<long>(B) * H_kv, d, fa::kTile) ||
        make_map_bytes(&maps.vt, vt, Np, d, static_cast<long>(B) * H_kv, fa::kTile, d) ||
        make_map(&maps.o, o, B * H, N, d, FA_BF16))
        return FA_ERR_CUDA;
    fa::Fp8FwdParams p;
    p.o = o;
    p.lse = lse;
    p.mask = block_mask;
    p.BH = B * H;
    p.N = N;
    p.T = tiles_of(N);
    p.num_pairs = (p.T + 1) / 2;
    p.rep = H / H_kv;
    p.head_group = head_group(p.BH, N, d, 1.0 / p.rep);  // K and V^T: d bytes per row each
    p.scale_log2 = scale * descale_q * descale_k * 1.4426950408889634f;
    p.descale_v = descale_v;
    p.causal = causal ? 1 : 0;
    if (make_ctl(status, p.BH, p.T, &p.ctl) != FA_OK) return FA_ERR_INVALID;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = fa::launch_fp8_transpose_v(static_cast<const uint8_t *>(v), vt, B * H_kv, N,
                                               Np, d, st);
    if (e == cudaSuccess) e = fa::launch_fwd_fp8(maps, p, d, st);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_decode_workspace_bytes(int B, int H, int H_kv, int Nq, int Nk, int d) {
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || check_heads(H, H_kv) != FA_OK) return 0;
    return decode_part_bytes(decode_split(B, H, H_kv, Nq, Nk), B, H, Nq, d);
}

int fa_decode(const void *q, const void *k, const void *v, void *o, float *lse,
              const int *kv_len, int B, int H, int H_kv, int Nq, int Nk, int d, int dtype,
              float scale, int causal, void *workspace, size_t workspace_bytes, void *stream) {
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID;
    if (static_cast<long long>(B) * H * Nq >= (1ll << 31) ||
        static_cast<long long>(B) * H_kv * Nk >= (1ll << 31))
        return FA_ERR_INVALID;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_INVALID;
    if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID;
    if (check_heads(H, H_kv) != FA_OK) return FA_ERR_INVALID;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    int rc = check_ptrs({q, k, v, o, lse});
    if (rc != FA_OK) return rc;
    if (kv_len != nullptr && (reinterpret_cast<uintptr_t>(kv_len) & 3u) != 0) return FA_ERR_INVALID;
    const DecodeSplit sp = decode_split(B, H, H_kv, Nq, Nk);
    const size_t need = decode_part_bytes(sp, B, H, Nq, d);
    if (need > 0 && (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need))
        return FA_ERR_INVALID;
    int dev = 0, *status = nullptr;
    rc = device_setup(&dev, &status);
    if (rc != FA_OK) return rc;
    fa::DecodeParams p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.kv_len = kv_len;
    p.part_o = need > 0 ? static_cast<float *>(workspace) : nullptr;
    p.part_ml = need > 0 ? static_cast<float *>(workspace) +
                               static_cast<size_t>(B) * H * Nq * sp.splits * d
                         : nullptr;
    p.B = B;
    p.H = H;
    p.Hkv = H_kv;
    p.Nq = Nq;
    p.Nk = Nk;
    p.rows = (H / H_kv) * Nq;
    p.row_groups = sp.row_groups;
    p.splits = sp.splits;
    p.chunk = sp.chunk;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.causal = causal ? 1 : 0;
    if (make_ctl(status, 0, 0, &p.ctl) != FA_OK) return FA_ERR_INVALID;
    fa::DecodeMaps maps;
    if (make_map(&maps.q, q, 1, B * H * Nq, d, dtype) || make_map(&maps.k, k, B * H_kv, Nk, d, dtype) ||
        make_map(&maps.v, v, B * H_kv, Nk, d, dtype))
        return FA_ERR_CUDA;
    cudaError_t e = fa::launch_decode(maps, p, d, dtype == FA_BF16,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_sync_status(void *stream) {
    int dev = 0, *status = nullptr;
    int rc = device_setup(&dev, &status);
    if (rc != FA_OK) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    int h = 0;
    if (cudaMemcpyFromSymbol(&h, g_fa_status, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
    const int zero = 0;
    if (h != 0 && cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(int)) != cudaSuccess)
        return FA_ERR_CUDA;
    return h;
}

const char *fa_status_string(int code) {
    switch (code) {
        case FA_OK: return "ok";
        case FA_ERR_INVALID: return "invalid argument";
        case FA_ERR_UNSUPPORTED: return "unsupported head dimension or device";
        case FA_ERR_CUDA: return "CUDA runtime error";
        case FA_ERR_TIMEOUT: return "device pipeline wait timed out";
        case FA_ERR_INTERNAL: return "kernel found its shared memory misaligned";
        default: return "unknown status";
    }
}

int fa_debug_set_visit_log(uint8_t *buf, size_t bytes) {
    if (bytes != 0 && (buf == nullptr || (reinterpret_cast<uintptr_t>(buf) & 3u) != 0))
        return FA_ERR_INVALID;
    std::lock_guard<std::mutex> lk(g_mu);
    g_visit_log = bytes ? buf : nullptr;
    g_visit_bytes = bytes;
    return FA_OK;
}

int fa_debug_set_wait_limit_ns(unsigned long long ns) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_wait_ns = ns ? ns : kDefaultWaitNs;
    return FA_OK;
}

int fa_debug_set_dkdv_splits(int splits) {
    if (splits < 0) return FA_ERR_INVALID;
    std::lock_guard<std::mutex> lk(g_mu);
    g_dkdv_splits = splits;
    return FA_OK;
}

int fa_debug_set_fault(int mode) {
    if (mode < 0 || mode > 3) return FA_ERR_INVALID;
    std::lock_guard<std::mutex> lk(g_mu);
    g_fault_mode = mode;
    return FA_OK;
}

}  // extern "C"
