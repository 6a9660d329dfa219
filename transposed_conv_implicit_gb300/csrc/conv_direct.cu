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
#include <atomic>

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
         ((p.Wo + p.dw_cols - 1) / p.dw_cols) * ((p.F + kDirectChannels - 1) / kDirectChannels);
}

bool dw_tiles_apply(const DirectParams& p) {
  if (!(p.R == 3 && p.S == 3 && p.stride_h == 1 && p.stride_w == 1 && p.dil_h == 1 &&
        p.dil_w == 1 && p.c_group == 1 && p.f_group == 1 && p.C % kDirectVec == 0))
    return false;
  if (p.dw_cols != 28 && p.dw_cols != 32) return false;
  return dw_tile_count(p) < (1ll << 31);
}

// 3x3 depthwise with multiplier 1, stride 1, dilation 1, 16-bit inputs, C a
// multiple of 8.  A tile is kDwRows output rows x kCols output columns x 64
// channels (kCols = 28 or 32, dw_tile_cols); its input (kDwRows + 2 rows x
// kCols + 2 columns x 64 channels, zero outside the image) arrives in shared
// memory as one TMA box, loaded by the CTA's last warp into a ring of two
// buffers (full and empty barriers per buffer: a compute warp waits for the
// box and releases it when done, so the warps run free of each other).  Thread (slot, pair, half)
// owns 4 channels of output columns 2*pair and 2*pair + 1 in output rows
// [8*half, 8*half + 8) of the tile, with the nine filter taps in registers as
// two channel pairs: it walks down its ten input rows, converts the four
// input columns of each row to fp32 once and adds them, two channels per
// packed fp32 FMA, into the three output rows that row touches; an output row
// is stored once its third input row is in.  Every output is the same fp32
// chain of nine FMAs in filter order (r, s) as in the plain direct kernel.
constexpr int kDwBoxRows = kDwRows + 2;
constexpr int kDwHalfRows = kDwRows / 2;  // output rows per thread
constexpr int kDwVec = 4;                 // channels per thread
constexpr int kDwPixBytes = kDirectChannels * 2;  // one box pixel: 64 16-bit channels

template <int kCols>
constexpr uint32_t dw_box_bytes() {
  return static_cast<uint32_t>(kDwBoxRows * (kCols + 2) * kDwPixBytes);
}
// Input boxes per CTA: one being read, one in flight.  (Three boxes of 28
// columns fit as well, and ran the 32x112x112x64 conv 35.8 us against 34.4.)
template <int kCols>
constexpr int dw_bufs() {
  return 2;
}

// Four 16-bit inputs (8 bytes) -> channels 0-1 and 2-3 as float pairs.
template <typename InT>
__device__ __forceinline__ void dw_unpack2(uint2 raw, float2& lo, float2& hi);
template <>
__device__ __forceinline__ void dw_unpack2<__nv_bfloat16>(uint2 raw, float2& lo, float2& hi) {
  // A bfloat16 is the high half of the float with the same value.
  lo = make_float2(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u));
  hi = make_float2(__uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
}
template <>
__device__ __forceinline__ void dw_unpack2<__half>(uint2 raw, float2& lo, float2& hi) {
  lo = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
  hi = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
}

// Four outputs (channel pairs lo, hi) at y: + beta * source (when src is
// given), the activation, one round-to-nearest-even each, 8 bytes.
template <int kAct>
__device__ __forceinline__ float dw_act(float v) {
  if (kAct == kEpiRelu) return fmaxf(v, 0.0f);
  if (kAct == kEpiSilu) return v / (1.0f + __expf(-v));
  return v;
}

template <typename OutT>
__device__ __forceinline__ uint32_t dw_pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t dw_pack2<__nv_bfloat16>(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t dw_pack2<__half>(float a, float b) {
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <typename OutT, int kAct>
__device__ __forceinline__ void dw_store2(float2 lo, float2 hi, OutT* y, const OutT* src,
                                          float beta) {
  float v[kDwVec] = {lo.x, lo.y, hi.x, hi.y};
  if (src) {
    const uint2 sraw = __ldg(reinterpret_cast<const uint2*>(src));
    const OutT* sv = reinterpret_cast<const OutT*>(&sraw);
#pragma unroll
    for (int j = 0; j < kDwVec; ++j) v[j] = fmaf(beta, load_f32<OutT>(sv + j), v[j]);
  }
  *reinterpret_cast<uint2*>(y) = make_uint2(dw_pack2<OutT>(dw_act<kAct>(v[0]), dw_act<kAct>(v[1])),
                                            dw_pack2<OutT>(dw_act<kAct>(v[2]), dw_act<kAct>(v[3])));
}

struct DwTile {
  int cb, n, oy0, x0;
};

__device__ __forceinline__ DwTile dw_decode(const DirectParams& p, int t) {
  const int n_xseg = (p.Wo + p.dw_cols - 1) / p.dw_cols;
  const int n_yblk = (p.Ho + kDwRows - 1) / kDwRows;
  const int per_cb = p.N * n_yblk * n_xseg;
  DwTile d;
  d.cb = t / per_cb;
  int rest = t - d.cb * per_cb;
  const int xs = rest % n_xseg;
  rest /= n_xseg;
  d.oy0 = (rest % n_yblk) * kDwRows;
  d.n = rest / n_yblk;
  d.x0 = xs * p.dw_cols;
  return d;
}

template <typename InT, typename OutT, int kCols, int kAct>
__global__ void __launch_bounds__(16 * kCols + 32, 1)
    conv_dw3x3_kernel(const __grid_constant__ DirectParams p, int tiles) {
  constexpr uint32_t kBoxBytes = dw_box_bytes<kCols>();
  constexpr int kDwBufs = dw_bufs<kCols>();
  static_assert(kDwBufs >= 2, "two input boxes must fit");
  constexpr int kPairs = kCols / 2;
  constexpr int kRowBytes = (kCols + 2) * kDwPixBytes;
  constexpr int kComputeWarps = 16 * kCols / 32;  // the last warp loads the boxes
  extern __shared__ uint8_t dw_smem_raw[];
  // [kDwBufs buffers][box], from a 128-byte aligned base (TMA destinations)
  uint8_t* boxes = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dw_smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  __shared__ __align__(8) uint64_t full[kDwBufs];   // box landed
  __shared__ __align__(8) uint64_t empty[kDwBufs];  // every compute warp is done with it
  __shared__ int abort_flag;
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);
  if (threadIdx.x == 0) {
    for (int b = 0; b < kDwBufs; ++b) {
      mbar_init(smem_u32(&full[b]), 1);
      mbar_init(smem_u32(&empty[b]), kComputeWarps);
    }
    abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&p.map_x);
  }
  __syncthreads();
  if (warp == kComputeWarps) {
    // Loader: tile i of this CTA (t = blockIdx.x + i * gridDim.x) goes into
    // buffer i % kDwBufs once the compute warps have released its previous tile.
    if (lane == 0) {
      int issued[kDwBufs] = {};
      int i = 0;
      for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
        const int buf = i % kDwBufs;
        if (i >= kDwBufs &&
            !mbar_wait_bounded(smem_u32(&empty[buf]), static_cast<uint32_t>((i / kDwBufs - 1) & 1),
                               &abort_flag, p.status, kStatusProducerTimeout, p.timeout_cycles))
          break;
        // (fault_mode 1, a test hook: CTA 0 never loads its first tile.)
        if (p.fault_mode == 1 && blockIdx.x == 0 && i == 0) continue;
        const DwTile d = dw_decode(p, t);
        const uint32_t b = smem_u32(&full[buf]);
        ++issued[buf];
        fence_proxy_async_shared();  // the compute warps' reads of the buffer come first
        mbar_arrive_expect_tx(b, kBoxBytes);
        tma_load_4d(smem_u32(boxes + buf * kBoxBytes), &p.map_x, b, d.cb * kDirectChannels,
                    d.x0 - p.pad_w, d.oy0 - p.pad_h, d.n);
      }
      // After an abort, the boxes still in flight land before the CTA exits.
      if (abort_flag)
        for (int b = 0; b < kDwBufs; ++b)
          if (issued[b] > 0)
            mbar_wait_drain(smem_u32(&full[b]), static_cast<uint32_t>((issued[b] - 1) & 1),
                            p.timeout_cycles / 8 + 1);
    }
    return;
  }
  const int slot = threadIdx.x & 15;  // channels [4*slot, 4*slot+4) of the tile's 64
  const int pair = (threadIdx.x >> 4) % kPairs;  // output columns 2*pair, 2*pair + 1
  const int half = (threadIdx.x >> 4) / kPairs;  // output rows [8*half, 8*half + 8)
  const InT* __restrict__ w = static_cast<const InT*>(p.w);
  float2 wl[9], wh[9];  // this thread's filter taps r*3 + s: channels 0-1 and 2-3
  int cb_loaded = -1;
  int i = 0;
  for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
    const int buf = i % kDwBufs;
    const DwTile d = dw_decode(p, t);
    const int f0 = d.cb * kDirectChannels + slot * kDwVec;
    if (d.cb != cb_loaded) {
      float wv[9][kDwVec];
#pragma unroll
      for (int tap = 0; tap < 9; ++tap)
#pragma unroll
        for (int j = 0; j < kDwVec; ++j)
          wv[tap][j] = f0 + j < p.F ? load_f32<InT>(w + packed_index(p, f0 + j, tap / 3, tap % 3, 0))
                                    : 0.0f;
#pragma unroll
      for (int tap = 0; tap < 9; ++tap) {
        wl[tap] = make_float2(wv[tap][0], wv[tap][1]);
        wh[tap] = make_float2(wv[tap][2], wv[tap][3]);
      }
      cb_loaded = d.cb;
    }
    if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&full[buf]),
                                                   static_cast<uint32_t>((i / kDwBufs) & 1),
                                                   &abort_flag, p.status, kStatusProducerTimeout,
                                                   p.timeout_cycles)))
      break;
    const int oy_first = d.oy0 + kDwHalfRows * half;  // this thread's first output row
    const int ox0 = d.x0 + 2 * pair;
    const bool store_ok[2] = {ox0 < p.Wo && f0 < p.F, ox0 + 1 < p.Wo && f0 < p.F};
    const long long o_row0 =
        ((static_cast<long long>(d.n) * p.Ho + oy_first) * p.Wo + ox0) * p.F + f0;
    const long long o_row_step = static_cast<long long>(p.Wo) * p.F;
    // Box row kDwHalfRows*half + k, columns 2*pair .. 2*pair + 3, this thread's channels.
    const uint8_t* src_rows =
        boxes + buf * kBoxBytes + (kDwHalfRows * half) * kRowBytes + (2 * pair) * kDwPixBytes + slot * 8;
    float2 acc[3][2][2];  // [output row % 3][column q][channel pair]
    OutT* yrow = static_cast<OutT*>(p.y) + o_row0;  // this thread's output row o = 0
    const OutT* srow = p.has_residual ? static_cast<const OutT*>(p.src) + o_row0 : nullptr;
#pragma unroll
    for (int k = 0; k < kDwHalfRows + 2; ++k) {
      float2 in[4][2];  // input columns 2*pair + c, channel pairs
#pragma unroll
      for (int c = 0; c < 4; ++c)
        dw_unpack2<InT>(*reinterpret_cast<const uint2*>(src_rows + k * kRowBytes + c * kDwPixBytes),
                        in[c][0], in[c][1]);
      // Filter row r takes this input row into output row k - r (of this
      // thread's 8); an output row starts at its r = 0 input row.
#pragma unroll
      for (int r = 0; r < 3; ++r) {
        const int o = k - r;
        if (o < 0 || o >= kDwHalfRows) continue;
        float2(&a)[2][2] = acc[o % 3];
        if (r == 0) {
#pragma unroll
          for (int q = 0; q < 2; ++q) a[q][0] = a[q][1] = make_float2(0.0f, 0.0f);
        }
#pragma unroll
        for (int s = 0; s < 3; ++s)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            a[q][0] = __ffma2_rn(in[q + s][0], wl[r * 3 + s], a[q][0]);
            a[q][1] = __ffma2_rn(in[q + s][1], wh[r * 3 + s], a[q][1]);
          }
      }
      const int o = k - 2;  // complete after this input row
      if (o >= 0) {
        if (oy_first + o < p.Ho) {
#pragma unroll
          for (int q = 0; q < 2; ++q)
            if (store_ok[q])
              dw_store2<OutT, kAct>(acc[o % 3][q][0], acc[o % 3][q][1], yrow + q * p.F,
                                    srow ? srow + q * p.F : nullptr, p.beta);
        }
        yrow += o_row_step;
        if (srow) srow += o_row_step;
      }
    }
    __syncwarp();  // every lane of this warp is done with the buffer
    if (lane == 0) mbar_arrive(smem_u32(&empty[buf]));
  }
}

// The dynamic shared-memory limit is a per-device function attribute: raise
// it once per device (slots in `configured`) to the largest size requested.
template <typename Kernel>
cudaError_t raise_smem_limit(Kernel kernel, std::atomic<size_t> (&configured)[64], size_t smem) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured[dev].load(std::memory_order_relaxed) >= smem) return cudaSuccess;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  if (err == cudaSuccess) configured[dev].store(smem, std::memory_order_relaxed);
  return err;
}

template <typename InT, typename OutT, int kCols, int kAct>
cudaError_t launch_dw_tiles_act(const DirectParams& p, int num_sms, cudaStream_t stream) {
  static std::atomic<size_t> configured[64];
  const long long tiles = dw_tile_count(p);
  const size_t smem = 128 + dw_bufs<kCols>() * dw_box_bytes<kCols>();
  cudaError_t err = raise_smem_limit(conv_dw3x3_kernel<InT, OutT, kCols, kAct>, configured, smem);
  if (err != cudaSuccess) return err;
  const unsigned grid = static_cast<unsigned>(std::min<long long>(tiles, num_sms));
  conv_dw3x3_kernel<InT, OutT, kCols, kAct>
      <<<grid, 16 * kCols + 32, smem, stream>>>(p, static_cast<int>(tiles));
  return cudaGetLastError();
}

template <typename InT, typename OutT, int kCols>
cudaError_t launch_dw_tiles(const DirectParams& p, int num_sms, cudaStream_t stream) {
  if (p.epilogue == kEpiRelu) return launch_dw_tiles_act<InT, OutT, kCols, kEpiRelu>(p, num_sms, stream);
  if (p.epilogue == kEpiSilu) return launch_dw_tiles_act<InT, OutT, kCols, kEpiSilu>(p, num_sms, stream);
  return launch_dw_tiles_act<InT, OutT, kCols, kEpiNone>(p, num_sms, stream);
}

template <typename InT, typename OutT>
cudaError_t launch_direct(const DirectParams& p, int num_sms, cudaStream_t stream) {
  if constexpr (sizeof(InT) == 2) {
    if (dw_tiles_apply(p))
      return p.dw_cols == 28 ? launch_dw_tiles<InT, OutT, 28>(p, num_sms, stream)
                             : launch_dw_tiles<InT, OutT, 32>(p, num_sms, stream);
  }
  static std::atomic<size_t> configured[64];
  const size_t smem = static_cast<size_t>(p.R) * p.S * p.c_group * kDirectChannels * sizeof(float);
  cudaError_t err = raise_smem_limit(conv_direct_kernel<InT, OutT>, configured, smem);
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

int dw_tile_cols(int wo) {
  const int waste28 = (wo + 27) / 28 * 28 - wo;
  const int waste32 = (wo + 31) / 32 * 32 - wo;
  return waste28 < waste32 ? 28 : 32;
}

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
