// Internal launch interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>

namespace kda {

struct BwdArgs {
    const void *q, *k;
    const float *g, *beta, *dAqk, *dAkk;
    float *dq, *dk, *db, *dg;
    int B, T, H;
    bool fp16;  // q/k element type: false = bf16, true = fp16
};

// All-FP32 SIMT kernel (one CTA per unit).
cudaError_t launch_intra_fp32(const BwdArgs &a, cudaStream_t stream);

// Tensor-core (tcgen05 TF32) kernel.
cudaError_t launch_intra_tc(const BwdArgs &a, cudaStream_t stream);

}  // namespace kda
