// Instantiation of the tensor-core kernel with split-TF32 cross sums: __half q/k,
// fixed-length sequences.
#include "kda_intra_tc.cuh"

namespace kda {
cudaError_t launch_tc_fp16_split(const BwdArgs &a, cudaStream_t stream) {
    return tcimpl::launch_split<__half>(a, stream);
}
}  // namespace kda
