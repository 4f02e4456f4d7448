// Internal launch interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>

namespace kda {

struct BwdArgs {
    const void *q, *k;
    const float *g, *beta, *dAqk, *dAkk;
    void *dq, *dk;  // fp32, or the q/k element type when emit_io is set
    float *db, *dg;
    int B, T, H;    // H = heads of q and k
    bool fp16;      // q/k element type: false = bf16, true = fp16
    // extended options (tensor-core path only)
    int HV = 0;     // heads of g, beta, dA and every output (0 = H); a multiple of H
    const float *dq_in = nullptr, *dk_in = nullptr, *dg_in = nullptr, *db_in = nullptr;
    bool fold_dg = false;  // dg as its inclusive reverse cumsum inside each chunk
    bool emit_io = false;  // dq, dk written in the q/k element type
    bool factor_diag = false;  // diagonal blocks' lower-left quadrant through row 8
    bool split = false;        // cross sums in split TF32 (FP32-level accuracy)
    unsigned *dbg = nullptr;   // bounds-checked debug build: the caller's flag word
    // variable-length sequences packed along T (B == 1): sequence n holds tokens
    // [cu_seqlens[n], cu_seqlens[n+1]); chunk c of the launch is chunk
    // chunk_indices[2c+1] of sequence chunk_indices[2c]
    const int *cu_seqlens = nullptr, *chunk_indices = nullptr;
    int num_seqs = 0, num_chunks = 0;
};

// Forward: the score matrices Aqk, Akk ([B,T,H,64] fp32, zeros outside the support).
struct FwdArgs {
    const void *q, *k;
    const float *g, *beta;
    float *Aqk, *Akk;
    int B, T, H;  // H = heads of q and k
    bool fp16;
    int HV = 0;   // heads of g, beta and the outputs (0 = H); a multiple of H
    // variable-length sequences, as in BwdArgs
    const int *cu_seqlens = nullptr, *chunk_indices = nullptr;
    int num_seqs = 0, num_chunks = 0;
    unsigned *dbg = nullptr;  // bounds-checked debug build: the caller's flag word
};

// Tensor-core (tcgen05 TF32) forward kernel.
cudaError_t launch_intra_fwd(const FwdArgs &a, cudaStream_t stream);

// All-FP32 SIMT kernel (persistent, one CTA per SM).
cudaError_t launch_intra_fp32(const BwdArgs &a, cudaStream_t stream);

// Tensor-core (tcgen05 TF32) kernel.
cudaError_t launch_intra_tc(const BwdArgs &a, cudaStream_t stream);

}  // namespace kda
