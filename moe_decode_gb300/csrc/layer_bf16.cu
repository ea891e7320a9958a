// bf16 routed experts: instantiation and launch of the persistent layer kernel.
#include "launch.h"
#include "launch_common.cuh"
#include "layer_kernel.cuh"

namespace moe {
cudaError_t launch_layer_bf16(const LayerParams& p, cudaStream_t stream, bool pdl, bool coop) {
    const bool io = p.gamma != nullptr || p.residual != 0;
    return launch_persistent(io ? moe_layer_kernel<0, true> : moe_layer_kernel<0, false>, block_threads(0), p,
                             stream, pdl, coop);
}
}  // namespace moe
