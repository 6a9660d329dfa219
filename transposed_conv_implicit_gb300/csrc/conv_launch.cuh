// Launcher of one implicit-GEMM kernel instance (shared by the kernel
// translation units).
#pragma once

#include <atomic>

#include "conv_internal.h"
#include "conv_kernel.cuh"

namespace convgb300 {

constexpr int kMaxDevices = 64;

template <int kKind, typename OutT, bool kGather, bool kPair = false, bool kStreamK = false>
cudaError_t launch_instance(const ConvKernelParams& p, int grid, size_t smem_bytes,
                            cudaStream_t stream) {
  // The dynamic shared-memory limit is a per-device function attribute: raise
  // it once per device to the largest size requested so far.
  static std::atomic<size_t> configured[kMaxDevices];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (configured[dev].load(std::memory_order_relaxed) < smem_bytes) {
    err = cudaFuncSetAttribute(conv_igemm_kernel<kKind, OutT, kGather, kPair, kStreamK>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem_bytes));
    if (err != cudaSuccess) return err;
    configured[dev].store(smem_bytes, std::memory_order_relaxed);
  }
  // Programmatic stream serialization: the kernel may be scheduled while the
  // previous kernel of the stream drains; it waits (griddepcontrol.wait)
  // before touching global memory, so stream order is preserved.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (kPair) {  // clusters of two CTAs (grid is even)
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  err = cudaLaunchKernelEx(&cfg, conv_igemm_kernel<kKind, OutT, kGather, kPair, kStreamK>, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

template <bool kGather, bool kPair = false, bool kStreamK = false>
cudaError_t launch_family(int kind, bool out_bf16, const ConvKernelParams& p, int grid,
                          size_t smem_bytes, cudaStream_t stream) {
  if (kind == kKindF8)
    return launch_instance<kKindF8, __nv_bfloat16, kGather, kPair, kStreamK>(p, grid, smem_bytes,
                                                                            stream);
  if (out_bf16)
    return launch_instance<kKindF16, __nv_bfloat16, kGather, kPair, kStreamK>(p, grid, smem_bytes,
                                                                             stream);
  return launch_instance<kKindF16, __half, kGather, kPair, kStreamK>(p, grid, smem_bytes, stream);
}

}  // namespace convgb300
