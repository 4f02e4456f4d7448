// Instantiation of the tensor-core kernel with split-TF32 cross sums: __nv_bfloat16 q/k,
// fixed-length sequences.
#include "kda_intra_tc.cuh"

namespace kda {
cudaError_t launch_tc_bf16_split(const BwdArgs &a, cudaStream_t stream) {
    return tcimpl::launch_split<__nv_bfloat16>(a, stream);
}
}  // namespace kda
