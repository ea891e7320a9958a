// One-token split-K layer (bf16 experts with transposed down projections):
// instantiation and launch, and the load-time transpose that prepares the
// transposed down projections.
#include "launch.h"
#include "launch_common.cuh"
#include "layer_splitk.cuh"

namespace moe {
cudaError_t launch_layer_splitk(const LayerParams& p, cudaStream_t stream, bool pdl, bool coop) {
    const bool io = p.gamma != nullptr || p.residual != 0;
    const int nvec = p.H / 8;
    // the fewest output vectors per unit thread that cover H
    auto* kernel = nvec <= kUnitThreads     ? (io ? moe_layer_splitk_kernel<true, 1> : moe_layer_splitk_kernel<false, 1>)
                   : nvec <= 2 * kUnitThreads ? (io ? moe_layer_splitk_kernel<true, 2> : moe_layer_splitk_kernel<false, 2>)
                                              : (io ? moe_layer_splitk_kernel<true, 3> : moe_layer_splitk_kernel<false, 3>);
    return launch_persistent(kernel, block_threads(0), p, stream, pdl, coop);
}

// dst[m][c][r] = src[m][r][c] for m < n, r < R, c < C (bf16 bits), through a
// 32 x 32 shared-memory tile (the padding column keeps the transposed reads
// free of bank conflicts).
__global__ void transpose_bf16_kernel(const uint16_t* __restrict__ src, int R, int C, uint16_t* __restrict__ dst) {
    __shared__ uint16_t tile[32][33];
    const size_t m = blockIdx.z;
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    const uint16_t* s = src + m * (size_t)R * C;
    uint16_t* d = dst + m * (size_t)R * C;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int r = r0 + i, c = c0 + threadIdx.x;
        if (r < R && c < C) tile[i][threadIdx.x] = s[(size_t)r * C + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int c = c0 + i, r = r0 + threadIdx.x;
        if (r < R && c < C) d[(size_t)c * R + r] = tile[threadIdx.x][i];
    }
}

cudaError_t launch_transpose_bf16(const uint16_t* src, int64_t n, int R, int C, uint16_t* dst, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    for (int64_t m0 = 0; m0 < n; m0 += 65535) {
        const unsigned nz = (unsigned)(n - m0 < 65535 ? n - m0 : 65535);
        const dim3 grid((unsigned)((C + 31) / 32), (unsigned)((R + 31) / 32), nz);
        transpose_bf16_kernel<<<grid, dim3(32, 8), 0, stream>>>(src + m0 * (size_t)R * C, R, C,
                                                                 dst + m0 * (size_t)R * C);
    }
    return cudaGetLastError();
}
}  // namespace moe
