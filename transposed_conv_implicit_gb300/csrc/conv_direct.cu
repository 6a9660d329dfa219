// Direct (CUDA-core) kernel for grouped convolutions whose channel groups are
// too narrow for the tensor-core path: depthwise convs, channel multipliers,
// and groups of a few channels ("dispatch_amd_4wave_conv2d", Args:
// num_groups).  Per output element it sums R*S*C_in/G products in fp32, then
// applies the same epilogue as the implicit GEMM: + beta*source, the
// activation, one round-to-nearest-even to the output dtype.
//
// A CTA covers 64 output channels of a run of pixels: the filter slice of
// those channels is staged once in shared memory as fp32, laid out
// [(r*S + s)*C/G + c][64], and each thread computes 8 consecutive output
// channels of one pixel.  Neighbouring threads take neighbouring pixels, so
// the input rows they share stay in L1.  The kernel is memory-bound: every
// input element is read from HBM about once and every output written once.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "conv_internal.h"

namespace convgb300 {

namespace {

constexpr int kDirectThreads = 256;
constexpr int kDirectChannels = 64;  // output channels per CTA
constexpr int kDirectVec = 8;        // output channels per thread

template <typename T>
__device__ __forceinline__ float load_f32(const T* p);
template <>
__device__ __forceinline__ float load_f32<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <>
__device__ __forceinline__ float load_f32<__half>(const __half* p) {
  return __half2float(*p);
}
template <>
__device__ __forceinline__ float load_f32<__nv_fp8_e4m3>(const __nv_fp8_e4m3* p) {
  return static_cast<float>(*p);
}

template <typename OutT>
__device__ __forceinline__ OutT store_rn(float v);
template <>
__device__ __forceinline__ __nv_bfloat16 store_rn<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ __half store_rn<__half>(float v) {
  return __float2half_rn(v);
}

__device__ __forceinline__ float direct_activation(float v, int act) {
  if (act == kEpiRelu) return fmaxf(v, 0.0f);
  if (act == kEpiSilu) return v / (1.0f + __expf(-v));
  return v;
}

__device__ __forceinline__ int div_fixed(int x, const FastDiv& f) {
  const uint32_t u = static_cast<uint32_t>(x);
  return static_cast<int>((static_cast<uint64_t>(__umulhi(u, f.mul)) + u) >> f.shift);
}

// Filter element W(r, s, c, f) of the packed filter: flat [F][(r*S + s)*Cg + c],
// or (gather layout) [F][r][run] with run index s*Cg + c.
__device__ __forceinline__ long long packed_index(const DirectParams& p, int f, int r, int s,
                                                  int c) {
  const long long row = static_cast<long long>(f) * p.kdim;
  if (p.w_runs) return row + static_cast<long long>(r) * p.run_elems + s * p.c_group + c;
  return row + (static_cast<long long>(r) * p.S + s) * p.c_group + c;
}

template <typename InT, typename OutT>
__global__ void __launch_bounds__(kDirectThreads)
    conv_direct_kernel(const __grid_constant__ DirectParams p) {
  extern __shared__ float wsm[];  // [taps * Cg][kDirectChannels]
  const int taps = p.R * p.S;
  const int kloc = taps * p.c_group;
  const int f_base = blockIdx.y * kDirectChannels;
  const InT* __restrict__ w = static_cast<const InT*>(p.w);
  for (int i = threadIdx.x; i < kloc * kDirectChannels; i += blockDim.x) {
    const int k = i / kDirectChannels, fl = i - k * kDirectChannels;
    const int f = f_base + fl;
    const int tap = k / p.c_group, c = k - tap * p.c_group;
    const int r = tap / p.S, s = tap - r * p.S;
    wsm[i] = f < p.F ? load_f32<InT>(w + packed_index(p, f, r, s, c)) : 0.0f;
  }
  __syncthreads();

  const InT* __restrict__ x = static_cast<const InT*>(p.x);
  const int slot = threadIdx.x % (kDirectChannels / kDirectVec);
  const int fl0 = slot * kDirectVec;
  const int f0 = f_base + fl0;
  if (f0 >= p.F) return;
  const int nf = min(kDirectVec, p.F - f0);
  // Depthwise with multiplier 1: output channel f reads input channel f, so
  // the 8 channels are one vector.
  const bool vec_in = p.c_group == 1 && p.f_group == 1 && nf == kDirectVec &&
                      (p.C * static_cast<int>(sizeof(InT))) % 16 == 0 && sizeof(InT) == 2;
  const bool k3x3 = p.R == 3 && p.S == 3;
  // (The host keeps N*Ho*Wo below 2^31.)
  const int pixels = p.N * p.Ho * p.Wo;
  const int pix_per_cta = kDirectThreads / (kDirectChannels / kDirectVec);
  for (int pix = blockIdx.x * pix_per_cta + threadIdx.x / (kDirectChannels / kDirectVec);
       pix < pixels; pix += gridDim.x * pix_per_cta) {
    const int t = div_fixed(pix, p.div_wo);
    const int ox = pix - t * p.Wo;
    const int n = div_fixed(t, p.div_ho);
    const int oy = t - n * p.Ho;
    float acc[kDirectVec];
#pragma unroll
    for (int j = 0; j < kDirectVec; ++j) acc[j] = 0.0f;
    if (k3x3 && vec_in) {
      // 3x3 depthwise: all nine input vectors are loaded before any use, so
      // their latencies overlap.
      uint4 in[9];
#pragma unroll
      for (int r = 0; r < 3; ++r)
#pragma unroll
        for (int s = 0; s < 3; ++s) {
          const int iy = oy * p.stride_h - p.pad_h + r * p.dil_h;
          const int ix = ox * p.stride_w - p.pad_w + s * p.dil_w;
          in[r * 3 + s] = make_uint4(0u, 0u, 0u, 0u);
          if (iy >= 0 && iy < p.H && ix >= 0 && ix < p.W)
            in[r * 3 + s] = __ldg(reinterpret_cast<const uint4*>(
                x + ((static_cast<long long>(n) * p.H + iy) * p.W + ix) * p.C + f0));
        }
#pragma unroll
      for (int tap = 0; tap < 9; ++tap) {
        const InT* v = reinterpret_cast<const InT*>(&in[tap]);
        const float* wk = wsm + tap * kDirectChannels + fl0;
        const float4 wa = *reinterpret_cast<const float4*>(wk);
        const float4 wb = *reinterpret_cast<const float4*>(wk + 4);
        const float wv[kDirectVec] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int j = 0; j < kDirectVec; ++j) acc[j] = fmaf(load_f32<InT>(v + j), wv[j], acc[j]);
      }
    }
    for (int r = 0; !(k3x3 && vec_in) && r < p.R; ++r) {
      const int iy = oy * p.stride_h - p.pad_h + r * p.dil_h;
      if (iy < 0 || iy >= p.H) continue;
      for (int s = 0; s < p.S; ++s) {
        const int ix = ox * p.stride_w - p.pad_w + s * p.dil_w;
        if (ix < 0 || ix >= p.W) continue;
        const InT* px = x + ((static_cast<long long>(n) * p.H + iy) * p.W + ix) * p.C;
        const float* wk = wsm + (r * p.S + s) * p.c_group * kDirectChannels + fl0;
        if (vec_in) {
          const uint4 raw = __ldg(reinterpret_cast<const uint4*>(px + f0));
          const InT* v = reinterpret_cast<const InT*>(&raw);
          const float4 wa = *reinterpret_cast<const float4*>(wk);
          const float4 wb = *reinterpret_cast<const float4*>(wk + 4);
          const float wv[kDirectVec] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
          for (int j = 0; j < kDirectVec; ++j) acc[j] = fmaf(load_f32<InT>(v + j), wv[j], acc[j]);
        } else {
#pragma unroll
          for (int j = 0; j < kDirectVec; ++j) {
            if (j < nf) {
              const int g = (f0 + j) / p.f_group;
              const InT* pg = px + g * p.c_group;
              for (int c = 0; c < p.c_group; ++c)
                acc[j] = fmaf(load_f32<InT>(pg + c), wk[c * kDirectChannels + j], acc[j]);
            }
          }
        }
      }
    }
    const long long o = static_cast<long long>(pix) * p.F + f0;
    OutT* y = static_cast<OutT*>(p.y) + o;
    const OutT* src = p.has_residual ? static_cast<const OutT*>(p.src) + o : nullptr;
    if (nf == kDirectVec && (p.F * 2) % 16 == 0) {
      uint4 out;
      OutT* o = reinterpret_cast<OutT*>(&out);
      uint4 sraw = make_uint4(0u, 0u, 0u, 0u);
      if (src) sraw = __ldg(reinterpret_cast<const uint4*>(src));
      const OutT* sv = reinterpret_cast<const OutT*>(&sraw);
#pragma unroll
      for (int j = 0; j < kDirectVec; ++j) {
        float v = acc[j];
        if (src) v = fmaf(p.beta, load_f32<OutT>(sv + j), v);
        o[j] = store_rn<OutT>(direct_activation(v, p.epilogue));
      }
      *reinterpret_cast<uint4*>(y) = out;
    } else {
      for (int j = 0; j < nf; ++j) {
        float v = acc[j];
        if (src) v = fmaf(p.beta, load_f32<OutT>(src + j), v);
        y[j] = store_rn<OutT>(direct_activation(v, p.epilogue));
      }
    }
  }
}

template <typename InT, typename OutT>
cudaError_t launch_direct(const DirectParams& p, int num_sms, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(p.R) * p.S * p.c_group * kDirectChannels * sizeof(float);
  cudaError_t err = cudaFuncSetAttribute(conv_direct_kernel<InT, OutT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const long long pixels = static_cast<long long>(p.N) * p.Ho * p.Wo;
  const int pix_per_cta = kDirectThreads / (kDirectChannels / kDirectVec);
  const int cblocks = (p.F + kDirectChannels - 1) / kDirectChannels;
  long long want = (pixels + pix_per_cta - 1) / pix_per_cta;
  // Enough CTAs to fill every SM several times; the loop strides over the rest.
  const long long cap = std::max<long long>(1, static_cast<long long>(num_sms) * 16 / cblocks);
  const dim3 grid(static_cast<unsigned>(std::min(want, cap)), static_cast<unsigned>(cblocks));
  conv_direct_kernel<InT, OutT><<<grid, kDirectThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t direct_smem_bytes(int r, int s, int c_group) {
  return static_cast<size_t>(r) * s * c_group * kDirectChannels * sizeof(float);
}

cudaError_t launch_conv_direct(int in_dtype, bool out_bf16, const DirectParams& p, int num_sms,
                               cudaStream_t stream) {
  if (in_dtype == 2) return launch_direct<__nv_fp8_e4m3, __nv_bfloat16>(p, num_sms, stream);
  if (out_bf16) return launch_direct<__nv_bfloat16, __nv_bfloat16>(p, num_sms, stream);
  return launch_direct<__half, __half>(p, num_sms, stream);
}

}  // namespace convgb300
