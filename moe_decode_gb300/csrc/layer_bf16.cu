// bf16 routed experts: instantiation and launch of the persistent layer kernel.
#include "launch.h"
#include "launch_common.cuh"
#include "layer_kernel.cuh"

namespace moe {
cudaError_t launch_layer_bf16(const LayerParams& p, cudaStream_t stream, bool pdl, bool coop) {
    const bool io = p.gamma != nullptr || p.residual != 0;
    const bool one = p.M == 1 && p.mode == kModeLayer;
    auto* kernel = io ? (one ? moe_layer_kernel<0, true, true> : moe_layer_kernel<0, true, false>)
                      : (one ? moe_layer_kernel<0, false, true> : moe_layer_kernel<0, false, false>);
    return launch_persistent(kernel, block_threads(0), p, stream, pdl, coop);
}
}  // namespace moe
