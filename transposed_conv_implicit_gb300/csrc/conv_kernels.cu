// Instances of the implicit-GEMM kernel with the TMA loaders, and the im2col
// probe, with their launchers.
#include "conv_launch.cuh"

namespace convgb300 {

namespace {

__global__ void im2col_probe_kernel(const __grid_constant__ CUtensorMap map, int c, int w, int h,
                                    int n, int off_w, int off_h, uint32_t row_bytes,
                                    uint8_t* __restrict__ out, unsigned int* status,
                                    long long limit_cycles) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tile = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t bytes = kBM * row_bytes;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(smem_u32(&bar), bytes);
    tma_load_im2col_4d(smem_u32(tile), &map, smem_u32(&bar), c, w, h, n,
                       static_cast<uint16_t>(off_w), static_cast<uint16_t>(off_h));
  }
  const bool ok = mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, status, 1u, limit_cycles);
  if (!__syncthreads_and(ok)) {
    if (threadIdx.x == 0) mbar_wait_drain(smem_u32(&bar), 0, limit_cycles);
    __syncthreads();
    return;
  }
  // The TMA swizzle XORs the 16-byte chunk index with address bits 7 and up.
  const uint32_t mask = row_bytes / 16 - 1;
  for (uint32_t q = threadIdx.x; q < bytes / 16; q += blockDim.x) {
    const uint32_t logical = q * 16;
    const uint32_t phys = logical ^ (((logical >> 7) & mask) << 4);
    reinterpret_cast<uint4*>(out)[q] = *reinterpret_cast<const uint4*>(tile + phys);
  }
}

}  // namespace

cudaError_t launch_conv_igemm(int kind, bool out_bf16, const ConvKernelParams& p, int grid,
                              size_t smem_bytes, cudaStream_t stream) {
  if (p.gather) return launch_conv_igemm_gather(kind, out_bf16, p, grid, smem_bytes, stream);
  if (p.pair) return launch_conv_igemm_pair(kind, out_bf16, p, grid, smem_bytes, stream);
  if (p.streamk) return launch_conv_igemm_streamk(kind, out_bf16, p, grid, smem_bytes, stream);
  return launch_family<false>(kind, out_bf16, p, grid, smem_bytes, stream);
}

cudaError_t launch_im2col_probe(const CUtensorMap& map, int c, int w, int h, int n, int off_w,
                                int off_h, uint32_t row_bytes, void* out, unsigned int* status,
                                long long limit_cycles, cudaStream_t stream) {
  const size_t smem = 1024 + static_cast<size_t>(kBM) * row_bytes;
  im2col_probe_kernel<<<1, 128, smem, stream>>>(map, c, w, h, n, off_w, off_h, row_bytes,
                                                static_cast<uint8_t*>(out), status, limit_cycles);
  return cudaGetLastError();
}

}  // namespace convgb300
