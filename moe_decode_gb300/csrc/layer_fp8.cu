// FP8 e4m3 routed experts (one fp32 scale per 128 elements of a row, decoded
// in registers): instantiation and launch of the persistent layer kernel.
#include "launch.h"
#include "launch_common.cuh"
#include "layer_kernel.cuh"

namespace moe {
cudaError_t launch_layer_fp8(const LayerParams& p, cudaStream_t stream, bool pdl, bool coop) {
    const bool io = p.gamma != nullptr || p.residual != 0;
    const bool one = p.M == 1 && p.mode == kModeLayer;
    auto* kernel = io ? (one ? moe_layer_kernel<2, true, true> : moe_layer_kernel<2, true, false>)
                      : (one ? moe_layer_kernel<2, false, true> : moe_layer_kernel<2, false, false>);
    return launch_persistent(kernel, block_threads(2), p, stream, pdl, coop);
}
}  // namespace moe
