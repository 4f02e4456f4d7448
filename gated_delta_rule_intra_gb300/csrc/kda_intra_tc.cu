// Tensor-core path of the KDA intra-chunk backward (placeholder: routes to the
// all-FP32 kernel until the tcgen05 kernel lands).
#include "kda_launch.h"

namespace kda {
cudaError_t launch_intra_tc(const BwdArgs &a, cudaStream_t stream) {
    return launch_intra_fp32(a, stream);
}
}  // namespace kda
