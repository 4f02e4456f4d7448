// Instantiations of the tensor-core kernel for __half q/k.
#include "kda_intra_tc.cuh"

namespace kda {
cudaError_t launch_tc_fp16(const BwdArgs &a, cudaStream_t stream) {
    return tcimpl::launch_io<__half>(a, stream);
}
}  // namespace kda
