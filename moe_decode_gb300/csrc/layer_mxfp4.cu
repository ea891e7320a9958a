// MXFP4 routed experts (e2m1 codes, e8m0 scale per 32 elements, decoded in
// registers): instantiation and launch of the persistent layer kernel, and the
// stand-alone dequantisation kernel that uses the same decode.
#include "launch.h"
#include "launch_common.cuh"
#include "layer_kernel.cuh"

namespace moe {
cudaError_t launch_layer_mxfp4(const LayerParams& p, cudaStream_t stream, bool pdl, bool coop) {
    const bool io = p.gamma != nullptr || p.residual != 0;
    const bool one = p.M == 1 && p.mode == kModeLayer;
    auto* kernel = io ? (one ? moe_layer_kernel<1, true, true> : moe_layer_kernel<1, true, false>)
                      : (one ? moe_layer_kernel<1, false, true> : moe_layer_kernel<1, false, false>);
    return launch_persistent(kernel, block_threads(1), p, stream, pdl, coop);
}

__global__ void mxfp4_dequant_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                     int64_t rows, int K, float* __restrict__ out) {
    const int64_t n = rows * (int64_t)K;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / K;
        const int c = (int)(i - r * K);
        uint32_t w[4];
        e2m1x8_to_f16x2(codes[r * (K / 2) + c / 2], w);  // the kernels' decode
        const float2 v = f16x2_to_f32(w[0]);
        out[i] = ((c & 1) ? v.y : v.x) * e8m0_to_f32(scales[r * (K / 32) + c / 32]);
    }
}

cudaError_t launch_mxfp4_dequant(const uint8_t* codes, const uint8_t* scales, int64_t rows, int K, float* out,
                                 cudaStream_t stream) {
    const int64_t n = rows * (int64_t)K;
    if (n == 0) return cudaSuccess;
    int blocks = (int)((n + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    mxfp4_dequant_kernel<<<blocks, 256, 0, stream>>>(codes, scales, rows, K, out);
    return cudaGetLastError();
}
}  // namespace moe
