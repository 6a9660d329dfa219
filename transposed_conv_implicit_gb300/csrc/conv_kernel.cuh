// Implicit-GEMM convolution kernel for sm_103a (tcgen05 + TMA im2col).
//
// One kernel serves the forward convolution and every stride phase of the
// transposed convolution.  The GEMM view ("dispatch_fused_im2col_conv2d_apple",
// description): rows m are output pixels (n, oy, ox), columns are output
// channels, and the contraction index is k = (r*S + s)*C_in + c.  The A operand
// (the im2col matrix) is never materialised: each 128-pixel x (one filter tap,
// bk channels) block is fetched straight from the NHWC input by a TMA im2col
// load, with the hardware zero-filling pixels that fall in the padding.  The B
// operand is the filter pre-packed once into a K-major [C_out][K] matrix.
//
// Warp roles (192 threads, one persistent CTA per SM):
//   warp 0      TMA producer: one elected lane streams (A, B) k-blocks into an
//               S-stage shared-memory ring guarded by full/empty mbarriers;
//   warp 1      TMEM owner and MMA issuer: one lane issues tcgen05.mma
//               (M=128, N=bn) into a double-buffered fp32 TMEM accumulator;
//   warps 2-5   epilogue: tcgen05.ld the accumulator, add beta*source, apply
//               the activation, round once to the output dtype and store.
// Every wait is bounded in time; on expiry the CTA records a status bit,
// stops, lets in-flight copies and MMAs land, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "conv_params.h"
#include "ptx.cuh"

namespace convgb300 {

struct TileInfo {
  int phase;
  int m0;       // first row (pixel) of the tile within its phase grid
  int n0;       // first output channel
  int kblocks;  // k-blocks in this tile's contraction
};

__device__ __forceinline__ TileInfo decode_tile(const ConvKernelParams& p, int t) {
  int ph = 0;
  while (ph + 1 < p.num_phases && t >= p.tile_start[ph + 1]) ++ph;
  const int local = t - p.tile_start[ph];
  TileInfo ti;
  ti.phase = ph;
  ti.n0 = (local % p.n_tiles) * p.bn;
  ti.m0 = (local / p.n_tiles) * kBM;
  ti.kblocks = p.taps_h[ph] * p.taps_w[ph] * p.c_blocks;
  return ti;
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) {
  return __half2float(v);
}

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ __half from_f32<__half>(float v) {
  return __float2half_rn(v);
}

// v = acc (+ beta*source); v = act(v); one round-to-nearest-even to OutT.
// `nvalid` < 16 masks the columns beyond C_out (the edge tile).
template <typename OutT>
__device__ __forceinline__ void epilogue_16(const ConvKernelParams& p, long long off,
                                            const uint32_t (&acc)[16], int nvalid) {
  float f[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(acc[j]);
  const bool full_vec = (nvalid == 16) && p.vec_ok;
  if (p.has_residual) {
    const OutT* src = static_cast<const OutT*>(p.src) + off;
    if (full_vec) {
      uint4 raw[2];
      raw[0] = __ldg(reinterpret_cast<const uint4*>(src));
      raw[1] = __ldg(reinterpret_cast<const uint4*>(src) + 1);
      const OutT* s = reinterpret_cast<const OutT*>(raw);
#pragma unroll
      for (int j = 0; j < 16; ++j) f[j] += p.beta * to_f32<OutT>(s[j]);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < nvalid) f[j] += p.beta * to_f32<OutT>(src[j]);
    }
  }
  if (p.epilogue == kEpiRelu) {
#pragma unroll
    for (int j = 0; j < 16; ++j) f[j] = fmaxf(f[j], 0.0f);
  } else if (p.epilogue == kEpiSilu) {
#pragma unroll
    for (int j = 0; j < 16; ++j) f[j] = f[j] / (1.0f + __expf(-f[j]));
  }
  OutT* dst = static_cast<OutT*>(p.out) + off;
  if (full_vec) {
    uint4 raw[2];
    OutT* o = reinterpret_cast<OutT*>(raw);
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j] = from_f32<OutT>(f[j]);
    reinterpret_cast<uint4*>(dst)[0] = raw[0];
    reinterpret_cast<uint4*>(dst)[1] = raw[1];
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < nvalid) dst[j] = from_f32<OutT>(f[j]);
  }
}

template <int kKind, typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
    conv_igemm_kernel(const __grid_constant__ ConvKernelParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int stages = p.stages;
  const uint32_t sw = p.sw_bytes;
  const uint32_t a_bytes = kBM * sw;
  const uint32_t b_bytes = static_cast<uint32_t>(p.bn) * sw;

  uint8_t* a_base = smem;
  uint8_t* b_base = smem + stages * a_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(b_base + stages * b_bytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + stages;
  uint64_t* tfull = bars + 2 * stages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned int* status = p.status;
  const uint64_t limit = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), kEpilogueWarps);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    for (int ph = 0; ph < p.num_phases; ++ph) tma_prefetch_desc(&p.map_a[ph]);
    tma_prefetch_desc(&p.map_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t acc_cols = p.tmem_cols / 2;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        const TileInfo ti = decode_tile(p, t);
        const int ph = ti.phase;
        const int hw = p.grid_h[ph] * p.grid_w[ph];
        const int n_img = ti.m0 / hw;
        const int rem = ti.m0 - n_img * hw;
        const int j = rem / p.grid_w[ph];
        const int i = rem - j * p.grid_w[ph];
        const int h0 = p.base_h[ph] + j * p.step_h;
        const int w0 = p.base_w[ph] + i * p.step_w;
        const int tw = p.taps_w[ph];
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          const int tap = kb / p.c_blocks;
          const int cb = kb - tap * p.c_blocks;
          const int uh = tap / tw;
          const int uw = tap - uh * tw;
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, status,
                                 kStatusProducerTimeout, limit)) {
            ok = false;
            break;
          }
          if (p.fault_mode == 1 && blockIdx.x == 0 && issued == 0) {
            // Test hook: leave this stage un-armed; its consumer can only time out.
            ++issued;
            if (++stage == stages) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, a_bytes + b_bytes);
          tma_load_im2col_4d(smem_u32(a_base + stage * a_bytes), &p.map_a[ph], fb, cb * p.bk, w0,
                             h0, n_img, static_cast<uint16_t>(uw * p.dil_w),
                             static_cast<uint16_t>(uh * p.dil_h));
          tma_load_3d(smem_u32(b_base + stage * b_bytes), &p.map_b, fb, kb * p.bk, ti.n0,
                      p.b_index[ph]);
          ++issued;
          if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every copy still in flight land before the CTA exits.
        const long long first = issued > stages ? issued - stages : 0;
        for (long long q = first; q < issued; ++q)
          mbar_wait_drain(smem_u32(&full[q % stages]), static_cast<uint32_t>((q / stages) & 1),
                          limit / 8 + 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++it) {
        const TileInfo ti = decode_tile(p, t);
        const int acc = it & 1;
        if (!mbar_wait_bounded(smem_u32(&tempty[acc]), static_cast<uint32_t>(((it >> 1) & 1) ^ 1),
                               abort_flag, status, kStatusMmaTimeout, limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (ti.kblocks == 0) {  // a phase with no filter taps: the epilogue writes act(0)
          mbar_arrive(smem_u32(&tfull[acc]));
          continue;
        }
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * acc_cols;
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, status,
                                 kStatusMmaTimeout, limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(a_base + stage * a_bytes);
          const uint32_t b_addr = smem_u32(b_base + stage * b_bytes);
          for (uint32_t kk = 0; kk < sw / 32; ++kk) {
            const uint64_t adesc = smem_desc_kmajor(a_addr + kk * 32, sw);
            const uint64_t bdesc = smem_desc_kmajor(b_addr + kk * 32, sw);
            const uint32_t accumulate = (kb | static_cast<int>(kk)) != 0;
            if (kKind == kKindF16)
              mma_f16(d_tmem, adesc, bdesc, p.idesc, accumulate);
            else
              mma_f8(d_tmem, adesc, bdesc, p.idesc, accumulate);
          }
          mma_commit(smem_u32(&empty[stage]));
          if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&tfull[acc]));
      }
      if (!ok) {
        // Every MMA already issued must finish before TMEM is released.
        mma_commit(smem_u32(drain));
        mbar_wait_drain(smem_u32(drain), 0, limit / 8 + 1);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may read: [32*quarter, 32*quarter+32)
    const int row = quarter * 32 + lane;
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    int it = 0;
    for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++it) {
      const TileInfo ti = decode_tile(p, t);
      const int acc = it & 1;
      bool ok = mbar_wait_bounded(smem_u32(&tfull[acc]), static_cast<uint32_t>((it >> 1) & 1),
                                  abort_flag, status, kStatusEpilogueTimeout, limit);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
      const int ph = ti.phase;
      const int m = ti.m0 + row;
      const bool valid = m < p.rows[ph];
      long long out_off = 0;
      if (valid) {
        const int hw = p.grid_h[ph] * p.grid_w[ph];
        const int n_img = m / hw;
        const int rem = m - n_img * hw;
        const int j = rem / p.grid_w[ph];
        const int i = rem - j * p.grid_w[ph];
        const long long oy = static_cast<long long>(p.out_step_h) * j + p.out_off_h[ph];
        const long long ox = static_cast<long long>(p.out_step_w) * i + p.out_off_w[ph];
        out_off = ((static_cast<long long>(n_img) * p.Ho + oy) * p.Wo + ox) * p.Cout;
      }
      const uint32_t taddr = tmem_base + lane_field + static_cast<uint32_t>(acc) * acc_cols;
      for (int c0 = 0; c0 < p.bn; c0 += 16) {
        uint32_t v[16];
        if (ti.kblocks > 0) {
          tmem_ld_32x32b_x16(taddr + static_cast<uint32_t>(c0), v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0u;
        }
        const int ch = ti.n0 + c0;
        if (valid && ch < p.Cout) {
          const int nvalid = p.Cout - ch < 16 ? p.Cout - ch : 16;
          epilogue_16<OutT>(p, out_off + ch, v, nvalid);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace convgb300
