// Instantiations of the tensor-core kernel: __nv_bfloat16 q/k, variable-length sequences,
// one exp2 per (r, s, d) in the diagonal blocks.
#include "kda_intra_tc.cuh"

namespace kda {
cudaError_t launch_tc_bf16_varlen(const BwdArgs &a, cudaStream_t stream) {
    return tcimpl::launch_io<__nv_bfloat16, true, false>(a, stream);
}
}  // namespace kda
