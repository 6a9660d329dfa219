// Row-tap kernel: forward convolution with few output channels (an RGB head,
// C_out = 3) on the tensor cores ("dispatch_amd_4wave_conv2d", Args: the
// masked edge tile that keeps small C_out on the matrix units).
//
// With C_out this small an implicit GEMM over K = R*S*C_in spends one MMA of
// the narrowest width (N = 16) per filter tap and channel block, and loads
// every input pixel R*S times.  Here the filter taps along S and the output
// channels share the N dimension instead:
//
//   P_iy[j][r][(f, s)] = sum_c x[n][iy][x0 - pad_w + j][c] * W(r, s, c, f)
//
// is one MMA per K-step over a segment of 128 input pixels j of input row iy,
// N = R groups of g16 columns (group r: the S*F products of filter row r).
// Output row oy = iy + pad_h - r takes group r, so each input row is loaded
// and multiplied once.  A tile is `band` output rows of one 128-pixel
// segment; its accumulators sit side by side in tensor memory in decreasing
// row order -- output row q at column g16 * (Qhi - q) -- so that the MMA for
// band input row k, issued at output row k's column, covers rows k, k-1, ...,
// k-R+1 with its R groups.  Output row k's group receives its first product
// from input row k: the first K-step of that row writes it afresh (its own
// N = g16 MMA without accumulate) and accumulates the other groups.
//
// Epilogue: output row q is complete once band input row q + R - 1 has been
// multiplied.  Lane j of its group holds the products (f, s) of input pixel
// x0 - pad_w + j; output pixel x0 + i sums tap s from lane i + s.  The lanes
// go through shared memory so that each thread can read its neighbours'
// values; then + beta*source, the activation and one round-to-nearest-even.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "conv_internal.h"
#include "ptx.cuh"
#include "segment_copy.cuh"

namespace convgb300 {

namespace {

constexpr int kRtWarps = 10;  // producer, MMA, 8 epilogue warps (two groups of 4)
constexpr int kRtThreads = 32 * kRtWarps;
constexpr uint32_t kRtStageBytes = 128 * 128;  // 128 pixels x 128-byte channel block

template <typename OutT>
__device__ __forceinline__ OutT rt_round(float v);
template <>
__device__ __forceinline__ __nv_bfloat16 rt_round<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ __half rt_round<__half>(float v) {
  return __float2half_rn(v);
}

__device__ __forceinline__ float rt_activation(float v, int act) {
  if (act == kEpiRelu) return fmaxf(v, 0.0f);
  if (act == kEpiSilu) return v / (1.0f + __expf(-v));
  return v;
}

__device__ __forceinline__ float rt_to_float(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float rt_to_float(__half v) { return __half2float(v); }

struct RtTile {
  int n, oy0, x0, rows;
};

__device__ __forceinline__ RtTile rt_decode(const RowTapParams& p, int t) {
  RtTile ti;
  const int seg = t % p.n_seg;
  const int rest = t / p.n_seg;
  const int band = rest % p.n_band;
  ti.n = rest / p.n_band;
  ti.oy0 = band * p.band;
  ti.x0 = seg * p.seg_w;
  ti.rows = min(p.band, p.Ho - ti.oy0);
  return ti;
}

// Issued from the converged MMA warp: one elected lane issues.
template <int kKind>
__device__ __forceinline__ void rt_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  if (kKind == kKindF16)
    mma_f16_warp(d, a, b, idesc, accumulate);
  else
    mma_f8_warp(d, a, b, idesc, accumulate);
}

// bar.sync over `count` threads that also ANDs a predicate across them, so
// that every thread of an epilogue group takes the same branch afterwards.
__device__ __forceinline__ bool group_barrier_all(uint32_t id, uint32_t count, bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(count)
      : "memory");
  return out != 0;
}

template <int kKind, typename OutT>
__global__ void __launch_bounds__(kRtThreads, 1)
    conv_rowtap_kernel(const __grid_constant__ RowTapParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int stages = p.stages;
  const int bk = 128 / (kKind == kKindF16 ? 2 : 1);  // channels per 128-byte block
  const int sf = p.S * p.F;                           // products per filter row
  const int brows = p.R * p.g16;                      // B rows per channel block
  uint8_t* a_ring = smem;
  uint8_t* b_res = smem + p.off_b;
  float* part = reinterpret_cast<float*>(smem + p.off_part);
  uint8_t* ostage = smem + p.off_stage;                   // [group] output row segment
  uint8_t* sstage = ostage + 2 * p.stage_bytes;           // [group] residual source segment
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* full = bars;
  uint64_t* empty = bars + stages;
  uint64_t* bres_full = bars + 2 * stages;
  uint64_t* rowfull = bres_full + 1;  // [buffer][output row of the band]
  uint64_t* tempty = rowfull + 2 * kRowTapMaxBand;
  uint64_t* drain = tempty + 2;
  uint64_t* epi_done = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned int* status = p.status;
  const long long limit = p.timeout_cycles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(bres_full), 1);
    for (int i = 0; i < 2 * kRowTapMaxBand; ++i) mbar_init(smem_u32(&rowfull[i]), 1);
    mbar_init(smem_u32(&tempty[0]), 8);
    mbar_init(smem_u32(&tempty[1]), 8);
    mbar_init(smem_u32(drain), 1);
    mbar_init(smem_u32(epi_done), 8);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // B rows that no filter box writes (each group's rows sf .. g16-1) are zero.
  {
    uint32_t* bw = reinterpret_cast<uint32_t*>(b_res);
    const int words = p.c_blocks * brows * 32;
    for (int i = threadIdx.x; i < words; i += blockDim.x) {
      const int row = (i >> 5) % brows;
      if (row % p.g16 >= sf) bw[i] = 0u;
    }
    fence_proxy_async_shared();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.map_x);
    tma_prefetch_desc(&p.map_w);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Set-up above may overlap the previous kernel of the stream; every global
  // memory access below comes after it has completed.
  grid_dependency_wait();
  grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the loads (warp-uniform operands); lane 0 issues.
    {
      const uint32_t lead = lane == 0 ? 1u : 0u;
      bool ok = true;
      const uint32_t b_blk = static_cast<uint32_t>(brows) * 128u;
      mbar_arrive_expect_tx_if(lead, smem_u32(bres_full),
                               static_cast<uint32_t>(p.c_blocks * p.R * sf) * 128u);
      for (int cb = 0; cb < p.c_blocks; ++cb)
        for (int r = 0; r < p.R; ++r)
          tma_load_4d_if(lead, smem_u32(b_res + cb * b_blk + r * p.g16 * 128), &p.map_w,
                         smem_u32(bres_full), cb * bk, 0, r, 0);
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      const int bps = p.blocks_per_stage;
      const uint32_t stage_bytes = static_cast<uint32_t>(bps) * kRtStageBytes;
      for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x) {
        const RtTile ti = rt_decode(p, t);
        const int kin = ti.rows + p.R - 1;
        for (int k = 0; ok && k < kin; ++k) {
          const int iy = ti.oy0 - p.pad_h + k;  // rows outside the image arrive as zeros
          for (int cb0 = 0; cb0 < p.c_blocks; cb0 += bps) {
            if (!__all_sync(0xFFFFFFFFu,
                            mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag,
                                              status, kStatusProducerTimeout, limit))) {
              ok = false;
              break;
            }
            const uint32_t fb = smem_u32(&full[stage]);
            // (fault_mode 1, a test hook: CTA 0 leaves its first stage un-armed.)
            if (!(p.fault_mode == 1 && blockIdx.x == 0 && issued == 0)) {
              mbar_arrive_expect_tx_if(lead, fb, stage_bytes);
              for (int i = 0; i < bps; ++i)
                tma_load_4d_if(lead, smem_u32(a_ring + stage * stage_bytes + i * kRtStageBytes),
                               &p.map_x, fb, (cb0 + i) * bk, ti.x0 - p.pad_w, iy, ti.n);
            }
            ++issued;
            if (++stage == stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // Let every copy still in flight land before the CTA exits.
        mbar_wait_drain(smem_u32(bres_full), 0, limit / 8 + 1);
        for (long long q = issued - stages; q < issued; ++q)
          if (q >= 0)
            mbar_wait_drain(smem_u32(&full[q % stages]), static_cast<uint32_t>((q / stages) & 1),
                            limit / 8 + 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The converged warp walks the MMAs; one elected lane issues each.
    {
      bool ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(bres_full), 0, abort_flag,
                                                          status, kStatusMmaTimeout, limit));
      tc_fence_after();
      const uint64_t desc_hi = smem_desc_kmajor(0, 128);
      const uint32_t a_lo0 = smem_u32(a_ring) >> 4;
      const uint32_t b_lo0 = smem_u32(b_res) >> 4;
      const uint32_t b_blk = (static_cast<uint32_t>(brows) * 128u) >> 4;
      const uint32_t g_lo = (static_cast<uint32_t>(p.g16) * 128u) >> 4;  // one B group
      const uint32_t g16 = static_cast<uint32_t>(p.g16);
      const uint32_t idesc_all = p.idesc_all, idesc_one = p.idesc_one, idesc_rest = p.idesc_rest;
      const bool multi_row = p.R > 1;
      const int R = p.R, c_blocks = p.c_blocks, total_tiles = p.total_tiles, band = p.band;
      const int bps = p.blocks_per_stage;
      const uint32_t stage_lo = (static_cast<uint32_t>(bps) * kRtStageBytes) >> 4;
      const uint32_t cols_per_buf = p.cols_per_buf;
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x, ++it) {
        const RtTile ti = rt_decode(p, t);
        const int buf = it & 1;
        if (!__all_sync(0xFFFFFFFFu,
                        mbar_wait_bounded(smem_u32(&tempty[buf]),
                                          static_cast<uint32_t>(((it >> 1) & 1) ^ 1), abort_flag,
                                          status, kStatusMmaTimeout, limit))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = tmem_base + static_cast<uint32_t>(buf) * cols_per_buf;
        const int kin = ti.rows + R - 1;
        for (int k = 0; ok && k < kin; ++k) {
          // Output row k's column; the MMA's R groups cover rows k .. k-R+1.
          const uint32_t d = base + g16 * static_cast<uint32_t>(kin - 1 - k);
          for (int cb0 = 0; cb0 < c_blocks; cb0 += bps) {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&full[stage]), phase,
                                                           abort_flag, status, kStatusMmaTimeout,
                                                           limit))) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int i = 0; i < bps; ++i) {
              const int cb = cb0 + i;
              const uint32_t a_lo = a_lo0 + static_cast<uint32_t>(stage) * stage_lo +
                                    static_cast<uint32_t>(i) * (kRtStageBytes >> 4);
              const uint32_t b_lo = b_lo0 + static_cast<uint32_t>(cb) * b_blk;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t a = desc_hi | static_cast<uint64_t>(a_lo + 2u * kk);
                const uint64_t b = desc_hi | static_cast<uint64_t>(b_lo + 2u * kk);
                if (kk == 0 && cb == 0) {
                  rt_mma<kKind>(d, a, b, idesc_one, 0u);  // output row k: first product
                  if (multi_row)
                    rt_mma<kKind>(d + g16, a, desc_hi | static_cast<uint64_t>(b_lo + g_lo),
                                  idesc_rest, 1u);
                } else {
                  rt_mma<kKind>(d, a, b, idesc_all, 1u);
                }
              }
            }
            mma_commit_warp(smem_u32(&empty[stage]));
            if (++stage == stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok && k >= R - 1)
            mma_commit_warp(smem_u32(&rowfull[buf * kRowTapMaxBand + k - (R - 1)]));
        }
        // A short band (the image's last) still completes every row barrier
        // of the buffer once, so that their phases stay in step with its uses.
        for (int q = ti.rows; ok && q < band; ++q)
          mma_commit_warp(smem_u32(&rowfull[buf * kRowTapMaxBand + q]));
      }
      if (!ok) {
        // Every MMA already issued must finish before TMEM is released.
        mma_commit_warp(smem_u32(drain));
        mbar_wait_drain(smem_u32(drain), 0, limit / 8 + 1);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Two groups of four warps take alternate output rows; warp w reads TMEM
    // lanes [32*(w%4), 32*(w%4)+32): input pixel j of the segment.
    const int grp = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int j = quarter * 32 + lane;
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t bar_id = 1 + static_cast<uint32_t>(grp);
    float* pg = part + grp * 2 * p.g16 * 128;
    const OutT* src = static_cast<const OutT*>(p.src);
    OutT* y = static_cast<OutT*>(p.out);
    int it = 0;
    int rb = 0;  // part buffer of the group's next row
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x, ++it) {
      const RtTile ti = rt_decode(p, t);
      const int buf = it & 1;
      const uint32_t base =
          tmem_base + lane_field + static_cast<uint32_t>(buf) * p.cols_per_buf;
      const int qhi = ti.rows + p.R - 2;
      for (int q = grp; q < ti.rows; q += 2) {
        bool mine = mbar_wait_bounded(smem_u32(&rowfull[buf * kRowTapMaxBand + q]),
                                      static_cast<uint32_t>((it >> 1) & 1), abort_flag, status,
                                      kStatusEpilogueTimeout, limit);
        float* pb = pg + rb * p.g16 * 128;
        rb ^= 1;
        if (__all_sync(0xFFFFFFFFu, mine)) {
          tc_fence_after();
          const uint32_t taddr = base + static_cast<uint32_t>(p.g16 * (qhi - q));
          uint32_t v[16];
          tmem_ld_32x32b_x16(taddr, v);
          tmem_wait_ld_regs(v);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (e < sf) pb[e * 128 + j] = __uint_as_float(v[e]);
          if (p.g16 == 32) {
            tmem_ld_32x32b_x16(taddr + 16u, v);
            tmem_wait_ld_regs(v);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (16 + e < sf) pb[(16 + e) * 128 + j] = __uint_as_float(v[e]);
          }
        } else {
          mine = false;
        }
        // Every thread of the group reaches this barrier, whatever its waits returned.
        if (!group_barrier_all(bar_id, 128, mine)) {
          ok = false;
          break;
        }
        // The row segment's outputs are contiguous in the NHWC output
        // (npx pixels x F channels).  They are assembled in shared memory at
        // the same 16-byte phase as their global address, so that the copy
        // out (and the residual source's copy in) moves aligned 16-byte words;
        // only the few bytes before the first and after the last 16-byte
        // boundary move as single elements.
        const int npx = min(p.seg_w, p.Wo - ti.x0);
        const long long o0 =
            ((static_cast<long long>(ti.n) * p.Ho + ti.oy0 + q) * p.Wo + ti.x0) * p.F;
        const int nel = npx * p.F;
        const uintptr_t gbeg = reinterpret_cast<uintptr_t>(y + o0);
        const int phase16 = static_cast<int>(gbeg & 15u);  // bytes before the first boundary's 16-byte word
        uint8_t* ost = ostage + grp * p.stage_bytes;
        if (p.has_residual) {
          // Source segment in, same layout (into the group's source stage).
          uint8_t* sst = sstage + grp * p.stage_bytes;
          copy_segment16<true>(reinterpret_cast<const uint8_t*>(src + o0), sst, phase16,
                                nel * static_cast<int>(sizeof(OutT)), j, 128);
          named_barrier(bar_id, 128);
        }
        if (j < npx) {
          const OutT* sv = reinterpret_cast<const OutT*>(sstage + grp * p.stage_bytes + phase16);
          OutT* ov = reinterpret_cast<OutT*>(ost + phase16);
          for (int f = 0; f < p.F; ++f) {
            float a = 0.0f;
            const float* pf = pb + f * p.S * 128 + j;
            for (int s = 0; s < p.S; ++s) a += pf[s * 128 + s];
            if (p.has_residual) a = fmaf(p.beta, rt_to_float(sv[j * p.F + f]), a);
            ov[j * p.F + f] = rt_round<OutT>(rt_activation(a, p.epilogue));
          }
        }
        named_barrier(bar_id, 128);
        copy_segment16<false>(reinterpret_cast<uint8_t*>(y + o0), ost, phase16,
                               nel * static_cast<int>(sizeof(OutT)), j, 128);
      }
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[buf]));
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(epi_done));
  }
  __syncthreads();
  if (warp == 1) {
    // TMEM is released once every epilogue warp's last tcgen05.ld is complete.
    if (lane == 0) mbar_wait_drain(smem_u32(epi_done), 0, limit);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

template <int kKind, typename OutT>
cudaError_t launch_rowtap(const RowTapParams& p, int grid, size_t smem_bytes,
                          cudaStream_t stream) {
  static std::atomic<size_t> configured[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured[dev].load(std::memory_order_relaxed) < smem_bytes) {
    err = cudaFuncSetAttribute(conv_rowtap_kernel<kKind, OutT>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem_bytes));
    if (err != cudaSuccess) return err;
    configured[dev].store(smem_bytes, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kRtThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, conv_rowtap_kernel<kKind, OutT>, p);
}

}  // namespace

cudaError_t launch_conv_rowtap(int in_dtype, bool out_bf16, const RowTapParams& p, int grid,
                               size_t smem_bytes, cudaStream_t stream) {
  if (in_dtype == 2) return launch_rowtap<kKindF8, __nv_bfloat16>(p, grid, smem_bytes, stream);
  if (out_bf16) return launch_rowtap<kKindF16, __nv_bfloat16>(p, grid, smem_bytes, stream);
  return launch_rowtap<kKindF16, __half>(p, grid, smem_bytes, stream);
}

}  // namespace convgb300
