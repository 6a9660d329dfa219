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
#include "ptx.cuh"

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

long long dw_tile_count(const DirectParams& p) {
  return static_cast<long long>(p.N) * ((p.Ho + kDwRows - 1) / kDwRows) *
         ((p.Wo + kDwCols - 1) / kDwCols) * ((p.F + kDirectChannels - 1) / kDirectChannels);
}

bool dw_tiles_apply(const DirectParams& p) {
  if (!(p.R == 3 && p.S == 3 && p.stride_h == 1 && p.stride_w == 1 && p.dil_h == 1 &&
        p.dil_w == 1 && p.c_group == 1 && p.f_group == 1 && p.C % kDirectVec == 0))
    return false;
  return dw_tile_count(p) < (1ll << 31);
}

// 3x3 depthwise with multiplier 1, stride 1, dilation 1, 16-bit inputs, C a
// multiple of 8.  A tile is kDwRows output rows x kDwCols output columns x 64
// channels; its input (kDwRows + 2 rows x kDwCols + 2 columns x 64 channels,
// zero outside the image) arrives in shared memory as one TMA box; the CTA
// keeps the boxes of its next kDwBufs - 1 tiles in flight while it computes
// this one.  Thread (slot, px) owns 4 channels of output column px, with their
// nine filter taps in registers: it walks down the tile's input rows, reads
// the three taps of each row from shared memory (converted to fp32 once) and
// adds them into the three output rows that row touches (a rolling set of
// fp32 accumulators); an output row is stored once its third input row is in.
constexpr int kDwBoxRows = kDwRows + 2;
constexpr int kDwBoxCols = kDwCols + 2;
constexpr uint32_t kDwBoxBytes = kDwBoxRows * kDwBoxCols * kDirectChannels * 2;

constexpr int kDwThreads = 512;
constexpr int kDwBufs = 2;  // input boxes in flight per CTA (one being read)
constexpr int kDwVec = 4;  // channels per thread

// Four 16-bit inputs (8 bytes) -> four floats.
template <typename InT>
__device__ __forceinline__ void dw_unpack(uint2 raw, float (&f)[kDwVec]) {
  const InT* v = reinterpret_cast<const InT*>(&raw);
#pragma unroll
  for (int j = 0; j < kDwVec; ++j) f[j] = load_f32<InT>(v + j);
}

template <typename OutT>
__device__ __forceinline__ void dw_store(const DirectParams& p, const float (&acc)[kDwVec], int n,
                                         int oy, int ox, int f0) {
  if (ox >= p.Wo || f0 >= p.F) return;
  const long long o = ((static_cast<long long>(n) * p.Ho + oy) * p.Wo + ox) * p.F + f0;
  uint2 sraw = make_uint2(0u, 0u);
  if (p.has_residual) sraw = __ldg(reinterpret_cast<const uint2*>(static_cast<const OutT*>(p.src) + o));
  const OutT* sv = reinterpret_cast<const OutT*>(&sraw);
  uint2 out;
  OutT* ov = reinterpret_cast<OutT*>(&out);
#pragma unroll
  for (int j = 0; j < kDwVec; ++j) {
    float v = acc[j];
    if (p.has_residual) v = fmaf(p.beta, load_f32<OutT>(sv + j), v);
    ov[j] = store_rn<OutT>(direct_activation(v, p.epilogue));
  }
  *reinterpret_cast<uint2*>(static_cast<OutT*>(p.y) + o) = out;
}

struct DwTile {
  int cb, n, oy0, x0;
};

__device__ __forceinline__ DwTile dw_decode(const DirectParams& p, int t) {
  const int n_xseg = (p.Wo + kDwCols - 1) / kDwCols;
  const int n_yblk = (p.Ho + kDwRows - 1) / kDwRows;
  const int per_cb = p.N * n_yblk * n_xseg;
  DwTile d;
  d.cb = t / per_cb;
  int rest = t - d.cb * per_cb;
  const int xs = rest % n_xseg;
  rest /= n_xseg;
  d.oy0 = (rest % n_yblk) * kDwRows;
  d.n = rest / n_yblk;
  d.x0 = xs * kDwCols;
  return d;
}

template <typename InT, typename OutT>
__global__ void __launch_bounds__(kDwThreads, 1)
    conv_dw3x3_kernel(const __grid_constant__ DirectParams p, int tiles) {
  extern __shared__ uint8_t dw_smem_raw[];
  // [kDwBufs buffers][box], from a 128-byte aligned base (TMA destinations)
  uint8_t* boxes = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dw_smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  __shared__ __align__(8) uint64_t bar[kDwBufs];
  __shared__ int abort_flag;
  const int slot = threadIdx.x & 15;  // channels [4*slot, 4*slot+4) of the tile's 64
  const int px = threadIdx.x >> 4;    // output column of the tile (0..31)
  const InT* __restrict__ w = static_cast<const InT*>(p.w);
  if (threadIdx.x == 0) {
    for (int b = 0; b < kDwBufs; ++b) mbar_init(smem_u32(&bar[b]), 1);
    abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&p.map_x);
  }
  __syncthreads();
  int issued[kDwBufs] = {};  // boxes issued per buffer (thread 0)
  auto issue = [&](int t, int buf) {  // thread 0: the input box of tile t
    // (fault_mode 1, a test hook: CTA 0 never loads its first tile.)
    if (p.fault_mode == 1 && blockIdx.x == 0 && t == static_cast<int>(blockIdx.x)) return;
    const DwTile d = dw_decode(p, t);
    const uint32_t b = smem_u32(&bar[buf]);
    ++issued[buf];
    fence_proxy_async_shared();  // earlier generic reads of the buffer come first
    mbar_arrive_expect_tx(b, kDwBoxBytes);
    tma_load_4d(smem_u32(boxes + buf * kDwBoxBytes), &p.map_x, b, d.cb * kDirectChannels,
                d.x0 - p.pad_w, d.oy0 - p.pad_h, d.n);
  };
  // Tile i of this CTA (t = blockIdx.x + i * gridDim.x) uses buffer i % kDwBufs.
  if (threadIdx.x == 0)
    for (int j = 0; j < kDwBufs - 1; ++j) {
      const long long tj = blockIdx.x + static_cast<long long>(j) * gridDim.x;
      if (tj < tiles) issue(static_cast<int>(tj), j);
    }
  float wr[9][kDwVec];  // this thread's filter taps, in registers
  int cb_loaded = -1;
  int i = 0;
  for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
    const int buf = i % kDwBufs;
    const DwTile d = dw_decode(p, t);
    const int f0 = d.cb * kDirectChannels + slot * kDwVec;
    if (d.cb != cb_loaded) {
#pragma unroll
      for (int tap = 0; tap < 9; ++tap)
#pragma unroll
        for (int j = 0; j < kDwVec; ++j)
          wr[tap][j] = f0 + j < p.F ? load_f32<InT>(w + packed_index(p, f0 + j, tap / 3, tap % 3, 0))
                                    : 0.0f;
      cb_loaded = d.cb;
    }
    // Tile i + kDwBufs - 1 goes into the buffer read in the previous
    // iteration, which every thread has finished (the __syncthreads at its end).
    const long long tn = t + static_cast<long long>(kDwBufs - 1) * gridDim.x;
    if (threadIdx.x == 0 && tn < tiles) issue(static_cast<int>(tn), (i + kDwBufs - 1) % kDwBufs);
    if (threadIdx.x == 0) {
      if (!mbar_wait_bounded(smem_u32(&bar[buf]), static_cast<uint32_t>((i / kDwBufs) & 1), &abort_flag,
                             p.status, kStatusProducerTimeout, p.timeout_cycles))
        abort_flag = 1;
    }
    __syncthreads();  // the box is in (thread 0 saw its barrier complete)
    if (abort_flag) break;
    const int ox = d.x0 + px;
    const int rows = min(kDwRows, p.Ho - d.oy0);
    const uint8_t* col = boxes + buf * kDwBoxBytes + (px * kDirectChannels + slot * kDwVec) * 2;
    float a0[kDwVec], a1[kDwVec], a2[kDwVec];  // output rows k, k-1, k-2
#pragma unroll
    for (int j = 0; j < kDwVec; ++j) a0[j] = a1[j] = a2[j] = 0.0f;
    for (int k = 0; k < rows + 2; ++k) {
      const uint8_t* rowp = col + k * (kDwBoxCols * kDirectChannels * 2);
      float in[3][kDwVec];  // taps s = 0, 1, 2 of this input row
      dw_unpack<InT>(*reinterpret_cast<const uint2*>(rowp), in[0]);
      dw_unpack<InT>(*reinterpret_cast<const uint2*>(rowp + kDirectChannels * 2), in[1]);
      dw_unpack<InT>(*reinterpret_cast<const uint2*>(rowp + 2 * kDirectChannels * 2), in[2]);
      // Filter row 0 feeds output row k, row 1 row k-1, row 2 row k-2.
#pragma unroll
      for (int s = 0; s < 3; ++s)
#pragma unroll
        for (int j = 0; j < kDwVec; ++j) {
          a0[j] = fmaf(in[s][j], wr[s][j], a0[j]);
          a1[j] = fmaf(in[s][j], wr[3 + s][j], a1[j]);
          a2[j] = fmaf(in[s][j], wr[6 + s][j], a2[j]);
        }
      if (k >= 2) dw_store<OutT>(p, a2, d.n, d.oy0 + k - 2, ox, f0);
#pragma unroll
      for (int j = 0; j < kDwVec; ++j) {
        a2[j] = a1[j];
        a1[j] = a0[j];
        a0[j] = 0.0f;
      }
    }
    __syncthreads();  // done with this buffer
  }
  // A box still in flight (after an abort) lands before the CTA exits.
  if (threadIdx.x == 0 && abort_flag) {
    for (int b = 0; b < kDwBufs; ++b)
      if (issued[b] > 0)
        mbar_wait_drain(smem_u32(&bar[b]), static_cast<uint32_t>((issued[b] - 1) & 1),
                        p.timeout_cycles / 8 + 1);
  }
}

template <typename InT, typename OutT>
cudaError_t launch_direct(const DirectParams& p, int num_sms, cudaStream_t stream) {
  if (sizeof(InT) == 2 && dw_tiles_apply(p)) {
    const long long tiles = dw_tile_count(p);
    const size_t smem = 128 + kDwBufs * kDwBoxBytes;
    cudaError_t err = cudaFuncSetAttribute(conv_dw3x3_kernel<InT, OutT>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const unsigned grid = static_cast<unsigned>(std::min<long long>(tiles, num_sms));
    conv_dw3x3_kernel<InT, OutT><<<grid, kDwThreads, smem, stream>>>(p, static_cast<int>(tiles));
    return cudaGetLastError();
  }
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

bool direct_uses_dw_tiles(int in_dtype, const DirectParams& p) {
  return in_dtype != 2 && dw_tiles_apply(p);
}

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
