// Instances of the implicit-GEMM kernel for the stream-K schedule (TMA
// loaders, single CTAs): equal shares of the (tile, k-block) iterations per
// SM, split tiles summed through fp32 partial tiles in the workspace.
#include "conv_launch.cuh"

namespace convgb300 {

cudaError_t launch_conv_igemm_streamk(int kind, bool out_bf16, const ConvKernelParams& p, int grid,
                                      size_t smem_bytes, cudaStream_t stream) {
  return launch_family<false, false, true>(kind, out_bf16, p, grid, smem_bytes, stream);
}

}  // namespace convgb300
