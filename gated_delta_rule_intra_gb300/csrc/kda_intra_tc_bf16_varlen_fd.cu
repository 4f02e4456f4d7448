// Instantiations of the tensor-core kernel: __nv_bfloat16 q/k, variable-length sequences,
// the diagonal blocks' lower-left quadrant factorized through row 8.
#include "kda_intra_tc.cuh"

namespace kda {
cudaError_t launch_tc_bf16_varlen_fd(const BwdArgs &a, cudaStream_t stream) {
    return tcimpl::launch_io<__nv_bfloat16, true, true>(a, stream);
}
}  // namespace kda
