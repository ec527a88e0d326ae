// Tensor-core (tcgen05, 3xTF32) implicit-GEMM path -- placeholder until the kernel lands.
#include "convt3d_internal.h"

namespace convt3d {
cudaError_t launch_tc(const convt3d_plan_s &, const float *, const float *, const float *, const float *,
                      const float *, float *, double *, uint32_t *, cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace convt3d
