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
    if (g_visit_log != nullptr &&
        g_visit_bytes < static_cast<size_t>(BH) * static_cast<size_t>(T) * static_cast<size_t>(T))
        return FA_ERR_INVALID;
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

int check_ptrs(std::initializer_list<const void *> ptrs) {
    for (const void *p : ptrs)
        if (p == nullptr || !aligned16(p)) return FA_ERR_INVALID;
    return FA_OK;
}

// [B*H, N, d] 16-bit tensor, 64 x 128 boxes (128 bytes x 128 rows), 128-byte swizzle.
int make_map(CUtensorMap *m, const void *base, int BH, int N, int d, int dtype) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m,
                          dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

int tiles_of(int N) { return (N + fa::kTile - 1) / fa::kTile; }

// Heads per CTA-order group: the streamed tiles of one head (two [N, d] 16-bit tensors) times
// the group stay near 32 MiB, a quarter of the L2.
int head_group(int BH, int N, int d) {
    const double per_head = 4.0 * N * d;
    int g = static_cast<int>((32.0 * 1024 * 1024) / per_head);
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    return g;
}

int fwd_common(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
               int N, int d, int dtype, float scale, int causal, const uint8_t *mask,
               void *stream) {
    int rc = check_shape(B, H, N, d, dtype, scale);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({q, k, v, o, lse});
    if (rc != FA_OK) return rc;
    int dev = 0, *status = nullptr;
    rc = device_setup(&dev, &status);
    if (rc != FA_OK) return rc;
    fa::Maps maps;
    const int BH = B * H;
    if (make_map(&maps.q, q, BH, N, d, dtype) || make_map(&maps.k, k, BH, N, d, dtype) ||
        make_map(&maps.v, v, BH, N, d, dtype))
        return FA_ERR_CUDA;
    fa::FwdParams p;
    p.o = o;
    p.lse = lse;
    p.mask = mask;
    p.BH = BH;
    p.N = N;
    p.T = tiles_of(N);
    p.num_pairs = (p.T + 1) / 2;
    p.head_group = head_group(BH, N, d);
    p.scale_log2 = scale * 1.4426950408889634f;
    p.causal = causal ? 1 : 0;
    if (make_ctl(status, BH, p.T, &p.ctl) != FA_OK) return FA_ERR_INVALID;
    cudaError_t e = fa::launch_fwd(maps, p, d, dtype == FA_BF16, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int bwd_params(const void *q, const void *k, const void *v, const void *dout, const float *lse,
               const float *delta, int B, int H, int N, int d, int dtype, float scale,
               int causal, const uint8_t *mask, fa::Maps *maps, fa::BwdParams *p) {
    int rc = check_shape(B, H, N, d, dtype, scale);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({q, k, v, dout, lse, delta});
    if (rc != FA_OK) return rc;
    int dev = 0, *status = nullptr;
    rc = device_setup(&dev, &status);
    if (rc != FA_OK) return rc;
    const int BH = B * H;
    if (make_map(&maps->q, q, BH, N, d, dtype) || make_map(&maps->k, k, BH, N, d, dtype) ||
        make_map(&maps->v, v, BH, N, d, dtype) || make_map(&maps->dout, dout, BH, N, d, dtype))
        return FA_ERR_CUDA;
    p->out0 = nullptr;
    p->out1 = nullptr;
    p->lse = lse;
    p->delta = delta;
    p->mask = mask;
    p->BH = BH;
    p->N = N;
    p->T = tiles_of(N);
    p->head_group = head_group(BH, N, d);
    p->scale = scale;
    p->scale_log2 = scale * 1.4426950408889634f;
    p->causal = causal ? 1 : 0;
    return make_ctl(status, BH, p->T, &p->ctl);
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
    return fwd_common(q, k, v, o, lse, B, H, N, d, dtype, scale, causal, nullptr, stream);
}

int fa_fwd_blocksparse(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                       int H, int N, int d, int dtype, float scale, int causal,
                       const uint8_t *block_mask, void *stream) {
    if (block_mask == nullptr) return FA_ERR_INVALID;
    return fwd_common(q, k, v, o, lse, B, H, N, d, dtype, scale, causal, block_mask, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
    (void)d;
    if (B < 1 || H < 1 || N < 1) return 0;
    const size_t bytes = static_cast<size_t>(B) * H * N * sizeof(float);
    return (bytes + 255) / 256 * 256;
}

int fa_bwd_preprocess(const void *o, const void *dout, float *delta, int B, int H, int N, int d,
                      int dtype, void *stream) {
    int rc = check_shape(B, H, N, d, dtype, 1.f);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({o, dout, delta});
    if (rc != FA_OK) return rc;
    int dev = 0, *status = nullptr;
    rc = device_setup(&dev, &status);
    if (rc != FA_OK) return rc;
    cudaError_t e = fa::launch_bwd_preprocess(o, dout, delta, static_cast<long>(B) * H * N, d,
                                              dtype == FA_BF16, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_bwd_dkdv(const void *q, const void *k, const void *v, const void *dout, const float *lse,
                const float *delta, void *dk, void *dv, int B, int H, int N, int d, int dtype,
                float scale, int causal, const uint8_t *block_mask, void *stream) {
    fa::Maps maps;
    fa::BwdParams p;
    int rc = bwd_params(q, k, v, dout, lse, delta, B, H, N, d, dtype, scale, causal, block_mask,
                        &maps, &p);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({dk, dv});
    if (rc != FA_OK) return rc;
    p.out0 = dk;
    p.out1 = dv;
    cudaError_t e =
        fa::launch_bwd_dkdv(maps, p, d, dtype == FA_BF16, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_bwd_dq(const void *q, const void *k, const void *v, const void *dout, const float *lse,
              const float *delta, void *dq, int B, int H, int N, int d, int dtype, float scale,
              int causal, const uint8_t *block_mask, void *stream) {
    fa::Maps maps;
    fa::BwdParams p;
    int rc = bwd_params(q, k, v, dout, lse, delta, B, H, N, d, dtype, scale, causal, block_mask,
                        &maps, &p);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({dq});
    if (rc != FA_OK) return rc;
    p.out0 = dq;
    cudaError_t e =
        fa::launch_bwd_dq(maps, p, d, dtype == FA_BF16, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
           const float *lse, void *dq, void *dk, void *dv, void *workspace,
           size_t workspace_bytes, int B, int H, int N, int d, int dtype, float scale,
           int causal, const uint8_t *block_mask, void *stream) {
    int rc = check_shape(B, H, N, d, dtype, scale);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({q, k, v, o, dout, lse, dq, dk, dv, workspace});
    if (rc != FA_OK) return rc;
    if (workspace_bytes < fa_bwd_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID;
    float *delta = static_cast<float *>(workspace);
    rc = fa_bwd_preprocess(o, dout, delta, B, H, N, d, dtype, stream);
    if (rc != FA_OK) return rc;
    rc = fa_bwd_dkdv(q, k, v, dout, lse, delta, dk, dv, B, H, N, d, dtype, scale, causal,
                     block_mask, stream);
    if (rc != FA_OK) return rc;
    return fa_bwd_dq(q, k, v, dout, lse, delta, dq, B, H, N, d, dtype, scale, causal, block_mask,
                     stream);
}

int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const void *dout,
                   const float *lse, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                   int dtype, float scale, int causal, const uint8_t *block_mask, void *stream) {
    int rc = check_shape(B, H, N, d, dtype, scale);
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
    rc = fa_bwd_preprocess(o, dout, delta, B, H, N, d, dtype, stream);
    if (rc != FA_OK) return rc;
    rc = fa_bwd_dkdv(q, k, v, dout, lse, delta, dk, dv, B, H, N, d, dtype, scale, causal,
                     block_mask, stream);
    if (rc != FA_OK) return rc;
    return fa_bwd_dq(q, k, v, dout, lse, delta, dq, B, H, N, d, dtype, scale, causal, block_mask,
                     stream);
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
        default: return "unknown status";
    }
}

int fa_debug_set_visit_log(uint8_t *buf, size_t bytes) {
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

int fa_debug_set_fault(int mode) {
    if (mode != 0 && mode != 1) return FA_ERR_INVALID;
    std::lock_guard<std::mutex> lk(g_mu);
    g_fault_mode = mode;
    return FA_OK;
}

}  // extern "C"
