// Instances of the implicit-GEMM kernel with the gather A loader.
#include "conv_launch.cuh"

namespace convgb300 {

cudaError_t launch_conv_igemm_gather(int kind, bool out_bf16, const ConvKernelParams& p, int grid,
                                     size_t smem_bytes, cudaStream_t stream) {
  return launch_family<true>(kind, out_bf16, p, grid, smem_bytes, stream);
}

}  // namespace convgb300
