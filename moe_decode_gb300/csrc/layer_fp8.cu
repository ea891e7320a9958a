// FP8 e4m3 routed experts (one fp32 scale per 128 elements of a row, decoded
// in registers): instantiation and launch of the persistent layer kernel.
#include "launch.h"
#include "launch_common.cuh"
#include "layer_kernel.cuh"

namespace moe {
cudaError_t launch_layer_fp8(const LayerParams& p, cudaStream_t stream, bool pdl, bool coop) {
    const bool io = p.gamma != nullptr || p.residual != 0;
    return launch_persistent(io ? moe_layer_kernel<2, true> : moe_layer_kernel<2, false>, block_threads(2), p,
                             stream, pdl, coop);
}
}  // namespace moe
