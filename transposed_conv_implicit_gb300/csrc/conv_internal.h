// Declarations shared by the host dispatcher and the kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include "conv_params.h"

namespace convgb300 {

// Launches the implicit-GEMM kernel instance for (kind, output dtype, loader).
cudaError_t launch_conv_igemm(int kind, bool out_bf16, const ConvKernelParams& p, int grid,
                              size_t smem_bytes, cudaStream_t stream);

// The gather-loader instances (their own translation unit).
cudaError_t launch_conv_igemm_gather(int kind, bool out_bf16, const ConvKernelParams& p, int grid,
                                     size_t smem_bytes, cudaStream_t stream);

// One TMA im2col load into shared memory, copied out un-swizzled (test hook).
cudaError_t launch_im2col_probe(const CUtensorMap& map, int c, int w, int h, int n, int off_w,
                                int off_h, uint32_t row_bytes, void* out, unsigned int* status,
                                long long limit_cycles, cudaStream_t stream);

}  // namespace convgb300
