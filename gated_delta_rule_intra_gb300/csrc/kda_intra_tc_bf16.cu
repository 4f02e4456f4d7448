// Instantiations of the tensor-core kernel for __nv_bfloat16 q/k.
#include "kda_intra_tc.cuh"

namespace kda {
cudaError_t launch_tc_bf16(const BwdArgs &a, cudaStream_t stream) {
    return tcimpl::launch_io<__nv_bfloat16>(a, stream);
}
}  // namespace kda
