// Instantiations of the tensor-core kernel: __half q/k, variable-length sequences,
// the diagonal blocks' lower-left quadrant factorized through row 8.
#include "kda_intra_tc.cuh"

namespace kda {
cudaError_t launch_tc_fp16_varlen_fd(const BwdArgs &a, cudaStream_t stream) {
    return tcimpl::launch_io<__half, true, true>(a, stream);
}
}  // namespace kda
