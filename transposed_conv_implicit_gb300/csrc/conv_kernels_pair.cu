// Instances of the implicit-GEMM kernel for CTA pairs (cta_group::2 MMAs).
#include "conv_launch.cuh"

namespace convgb300 {

cudaError_t launch_conv_igemm_pair(int kind, bool out_bf16, const ConvKernelParams& p, int grid,
                                   size_t smem_bytes, cudaStream_t stream) {
  return launch_family<false, true>(kind, out_bf16, p, grid, smem_bytes, stream);
}

}  // namespace convgb300
