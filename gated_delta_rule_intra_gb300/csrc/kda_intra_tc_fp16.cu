// Instantiations of the tensor-core kernel: __half q/k, fixed-length sequences,
// one exp2 per (r, s, d) in the diagonal blocks.
#include "kda_intra_tc.cuh"

namespace kda {
cudaError_t launch_tc_fp16(const BwdArgs &a, cudaStream_t stream) {
    return tcimpl::launch_io<__half, false, false>(a, stream);
}
}  // namespace kda
