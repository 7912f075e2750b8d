// fa_internal.h - parameter blocks and launchers shared by the C-ABI shim and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sm100.cuh"

namespace fa {

constexpr int kTile = 128;  // query rows / key rows per tile, also the block-mask granularity

struct FwdParams {
    void *o;                  // [B,H,N,d] output
    float *lse;               // [B,H,N] output
    const uint8_t *mask;      // [T][T] or nullptr
    int BH, N, T;             // heads (B*H), sequence length, tiles per side
    int num_pairs;            // ceil(T / 2): query-tile pairs per head
    float scale_log2;         // scale * log2(e)
    int causal;
    Ctl ctl;
};

struct BwdParams {
    void *out0;               // dK (dK/dV kernel) or dQ (dQ kernel)
    void *out1;               // dV (dK/dV kernel) or unused
    const float *lse;         // [B,H,N]
    const float *delta;       // [B,H,N]
    const uint8_t *mask;      // [T][T] or nullptr
    int BH, N, T;
    float scale;              // softmax scale (dK and dQ carry it)
    float scale_log2;         // scale * log2(e)
    int causal;
    Ctl ctl;
};

struct Maps {
    CUtensorMap q, k, v, dout;
};

cudaError_t launch_fwd(const Maps &maps, const FwdParams &p, int d, bool bf16,
                       cudaStream_t stream);
cudaError_t launch_bwd_preprocess(const void *o, const void *dout, float *delta, long rows,
                                  int d, bool bf16, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(const Maps &maps, const BwdParams &p, int d, bool bf16,
                            cudaStream_t stream);
cudaError_t launch_bwd_dq(const Maps &maps, const BwdParams &p, int d, bool bf16,
                          cudaStream_t stream);

}  // namespace fa
