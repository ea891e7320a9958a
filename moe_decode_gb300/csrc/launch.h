// Host-side launch entry points of the layer kernel (one per weight format).
#pragma once
#include <cuda_runtime.h>

#include "layer_params.h"
#include "lm_params.h"

namespace moe {
cudaError_t launch_layer_bf16(const LayerParams& p, cudaStream_t stream, bool pdl, bool coop);
cudaError_t launch_layer_mxfp4(const LayerParams& p, cudaStream_t stream, bool pdl, bool coop);
cudaError_t launch_layer_fp8(const LayerParams& p, cudaStream_t stream, bool pdl, bool coop);
cudaError_t launch_layer_splitk(const LayerParams& p, cudaStream_t stream, bool pdl, bool coop);
cudaError_t launch_transpose_bf16(const uint16_t* src, int64_t n, int R, int C, uint16_t* dst, cudaStream_t stream);
cudaError_t launch_mxfp4_dequant(const uint8_t* codes, const uint8_t* scales, int64_t rows, int K, float* out,
                                 cudaStream_t stream);
cudaError_t launch_lm_head(const LmParams& p, int wt, cudaStream_t stream, bool pdl);
cudaError_t launch_fp8_quantize(const uint16_t* w, int64_t rows, int K, int block, uint8_t* codes, float* scales,
                                cudaStream_t stream);
cudaError_t launch_fp8_dequant(const uint8_t* codes, const float* scales, int64_t rows, int K, int block, float* out,
                               cudaStream_t stream);
}  // namespace moe
