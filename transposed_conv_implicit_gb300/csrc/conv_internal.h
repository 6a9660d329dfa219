// Declarations shared by the host dispatcher and the kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include "conv_params.h"

namespace convgb300 {

// Launches the implicit-GEMM kernel instance for (kind, output dtype, loader).
cudaError_t launch_conv_igemm(int kind, bool out_bf16, const ConvKernelParams& p, int grid,
                              size_t smem_bytes, cudaStream_t stream);

// Direct (CUDA-core) grouped convolution for channel groups too narrow for
// the tensor cores.  The filter is the packed one: flat [F][K] with
// k = (r*S + s)*c_group + c, or, when w_runs is set, the gather layout
// [F][r][run_elems] with run index s*c_group + c.
struct DirectParams {
  const void* x;
  const void* w;
  const void* src;
  void* y;
  int N, H, W, C, Ho, Wo, F, R, S;
  int c_group, f_group;
  int stride_h, stride_w, pad_h, pad_w, dil_h, dil_w;
  int w_runs, run_elems, kdim;
  int has_residual, epilogue;
  float beta;
  FastDiv div_wo, div_ho;  // pixel index -> (n, oy, ox)
};

size_t direct_smem_bytes(int r, int s, int c_group);

// in_dtype: 0 bf16, 1 f16, 2 e4m3 (bf16 out).
cudaError_t launch_conv_direct(int in_dtype, bool out_bf16, const DirectParams& p, int num_sms,
                               cudaStream_t stream);

// The gather-loader instances (their own translation unit).
cudaError_t launch_conv_igemm_gather(int kind, bool out_bf16, const ConvKernelParams& p, int grid,
                                     size_t smem_bytes, cudaStream_t stream);

// One TMA im2col load into shared memory, copied out un-swizzled (test hook).
cudaError_t launch_im2col_probe(const CUtensorMap& map, int c, int w, int h, int n, int off_w,
                                int off_h, uint32_t row_bytes, void* out, unsigned int* status,
                                long long limit_cycles, cudaStream_t stream);

}  // namespace convgb300
