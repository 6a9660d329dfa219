// Implicit-GEMM convolution kernel for sm_103a (tcgen05 + TMA).
//
// One kernel serves the forward convolution and every stride phase of the
// transposed convolution.  The GEMM view ("dispatch_fused_im2col_conv2d_apple",
// description): rows m are output pixels (n, oy, ox), columns are output
// channels, and the contraction index is k = (r*S + s)*C_in + c.  The A operand
// (the im2col matrix) is never materialised; one of three loaders brings each
// k-block of it into shared memory straight from the NHWC input:
//   - TMA im2col: one 128-pixel x (one filter tap, bk channels) box per
//     k-block, the hardware zero-filling pixels that fall in the padding;
//   - row window (stride-1 forward convs whose padded output row fits in
//     128 MMA rows): one tiled box of the tile's input rows with halo per
//     channel block, read by every filter tap at a row offset;
//   - gather (channel rows TMA cannot address, e.g. C_in = 3): the producer
//     warps load 16-byte pieces of the input with plain loads and write them
//     into the swizzled stage.
// The B operand is the filter pre-packed once into a K-major [C_out][K]
// matrix; when it fits, it is loaded into shared memory with the first tile
// and kept there.
//
// Warp roles (384 threads, one persistent CTA per SM, or one per SM of a
// CTA pair):
//   warps 0, 10  producers: k-block `seq` belongs to producer seq % nprod;
//   (and 11)     the whole warp walks the k-blocks and one lane issues its
//                TMA loads into an S-stage shared-memory ring guarded by
//                full/empty mbarriers.  Warp 11 is the third TMA producer
//                unless it issues MMAs (below); in gather mode warps 0, 10
//                and 11 each build every third k-block, the whole warp
//                writing it;
//   warp 1       TMEM owner and MMA issuer: the converged warp walks the
//                k-blocks and one elected lane issues each tcgen05.mma
//                (M=128 per half, N=bn; M=256 over both CTAs of a pair, from
//                rank 0) into a double-buffered fp32 TMEM accumulator; with
//                two 128-row halves and the TMA loaders warp 11 issues the
//                second half's MMAs;
//   warps 2-9    epilogue, two warpgroups taking alternate (half, column
//                chunk) items: tcgen05.ld the accumulator, add beta*source,
//                apply the activation, round once to the output dtype and
//                store.  With a TMA epilogue the residual source is loaded by
//                TMA ahead of use into swizzled shared memory, and results are
//                staged there and written by TMA stores (which also clip the
//                ragged M tail and the C_out edge tile).
// Every wait is bounded in time; on expiry the CTA records a status bit,
// stops, lets in-flight copies and MMAs land, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "conv_params.h"
#include "ptx.cuh"
#include "segment_copy.cuh"

namespace convgb300 {

struct TileInfo {
  int phase;
  int group;    // channel group (forward convs with num_groups > 1), else 0
  int m0;       // first row (pixel) of the tile within its phase grid
  int n0;       // first output channel
  int kblocks;  // k-blocks in this tile's contraction
};

// x / f.d for 0 <= x < 2^31 (see FastDiv).
__device__ __forceinline__ int fast_div(int x, const FastDiv& f) {
  const uint32_t u = static_cast<uint32_t>(x);
  return static_cast<int>((static_cast<uint64_t>(__umulhi(u, f.mul)) + u) >> f.shift);
}

__device__ __forceinline__ TileInfo decode_tile(const ConvKernelParams& p, int t) {
  if (p.window) {  // one C_out tile; m0 carries the tile index
    TileInfo ti;
    ti.phase = 0;
    ti.group = 0;
    ti.n0 = 0;
    ti.m0 = t;
    ti.kblocks = p.c_blocks;
    return ti;
  }
  int group = 0;
  if (p.groups > 1) {
    group = fast_div(t, p.div_tpg);
    t -= group * p.tiles_per_group;
  }
  int ph = 0;
  while (ph + 1 < p.num_phases && t >= p.tile_start[ph + 1]) ++ph;
  const int local = t - p.tile_start[ph];
  TileInfo ti;
  ti.phase = ph;
  ti.group = group;
  const int mt = fast_div(local, p.div_ntiles);
  ti.n0 = (local - mt * p.n_tiles) * p.bn;
  ti.m0 = mt * ((kBM * p.m_halves) << p.pair);  // a pair's tile spans both CTAs' rows
  ti.kblocks = p.taps_h[ph] * p.taps_w[ph] * p.c_blocks;
  return ti;
}

// ---------------------------------------------------------------- work items
// A CTA's (or CTA pair's) work: whole tiles cta, cta + nctas, ...
// (data-parallel), or, with stream-K, its equal share of the iteration
// sequence (tile by tile, k-block by k-block), cut at tile boundaries.
struct Work {
  TileInfo ti;
  int tile;
  int kb0, kb1;  // k-blocks [kb0, kb1) of the tile
};

struct WorkWalk {
  long long pos, end;  // stream-K iteration range
  int t, step;         // data-parallel tile walk
};

__device__ __forceinline__ long long sk_share_begin(const ConvKernelParams& p, int cta, int nctas) {
  return p.sk_iters * cta / nctas;
}

// The CTA whose share holds iteration `pos`: the last c with share_begin(c) <= pos.
__device__ __forceinline__ int sk_owner(const ConvKernelParams& p, long long pos, int nctas) {
  return static_cast<int>(((pos + 1) * nctas - 1) / p.sk_iters);
}

// kStreamK: the kernel instance runs the stream-K schedule (a separate
// instance, so that the whole-tile instances carry none of its code).
template <bool kStreamK>
__device__ __forceinline__ WorkWalk work_begin(const ConvKernelParams& p, int cta, int nctas) {
  WorkWalk w;
  w.t = cta;
  w.step = nctas;
  w.pos = kStreamK ? sk_share_begin(p, cta, nctas) : 0;
  w.end = kStreamK ? sk_share_begin(p, cta + 1, nctas) : 0;
  return w;
}

// First iteration of tile `tile` (stream-K).
__device__ __forceinline__ long long sk_tile_iter(const ConvKernelParams& p, int tile, int phase) {
  return p.sk_iter_start[phase] +
         static_cast<long long>(tile - p.tile_start[phase]) * p.sk_kpt[phase];
}

template <bool kStreamK>
__device__ __forceinline__ bool work_next(const ConvKernelParams& p, WorkWalk& w, Work& out) {
  if constexpr (kStreamK) {
    if (w.pos >= w.end) return false;
    int ph = 0;
    while (ph + 1 < p.num_phases && w.pos >= p.sk_iter_start[ph + 1]) ++ph;
    const int local = static_cast<int>(w.pos - p.sk_iter_start[ph]);
    const int tl = fast_div(local, p.sk_div_kpt[ph]);
    out.tile = p.tile_start[ph] + tl;
    out.ti = decode_tile(p, out.tile);
    out.kb0 = local - tl * p.sk_kpt[ph];
    const long long room = w.end - w.pos;
    out.kb1 = room < out.ti.kblocks - out.kb0 ? out.kb0 + static_cast<int>(room) : out.ti.kblocks;
    w.pos += out.kb1 - out.kb0;
    return true;
  }
  if (w.t >= p.total_tiles) return false;
  out.tile = w.t;
  out.ti = decode_tile(p, w.t);
  out.kb0 = 0;
  out.kb1 = out.ti.kblocks;
  w.t += w.step;
  return true;
}

// The role of a work item in its tile's epilogue.
constexpr int kSkWhole = 0;    // the whole tile: the ordinary epilogue
constexpr int kSkPartial = 1;  // starts inside the tile: accumulators go to the partial slot
constexpr int kSkFinish = 2;   // the tile's first k-blocks, others follow: add their partials

__device__ __forceinline__ int work_role(const Work& w) {
  if (w.kb0 != 0) return kSkPartial;
  return w.kb1 < w.ti.kblocks ? kSkFinish : kSkWhole;
}

// Partial slot layout: [16-column group][quarter k of the group][128 rows][4
// floats], so each 16-byte store or load instruction of a warp (32 rows, one
// (group, k)) touches 512 consecutive bytes: whole sectors and lines.
__device__ __forceinline__ float4* sk_slot_at(const ConvKernelParams& p, int cta, int group, int k,
                                              int row) {
  return reinterpret_cast<float4*>(p.sk_partials + static_cast<size_t>(cta) * p.sk_slot_floats) +
         (static_cast<size_t>(group) * 4 + k) * kBM + row;
}

// Contributor: 16 accumulator columns of one row into the slot.
__device__ __forceinline__ void sk_store16(const ConvKernelParams& p, int cta, int group, int row,
                                           const uint32_t* v) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    *sk_slot_at(p, cta, group, k, row) =
        make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                    __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
}

// Finisher: waits (bounded) until every CTA holding later k-blocks of the
// work item's tile has raised the flag of epilogue warp `ew` for this launch.
// Returns false on timeout (status bit and abort flag raised) or abort.
__device__ __forceinline__ bool sk_wait_partials(const ConvKernelParams& p, const Work& w, int ew,
                                                 int nctas, volatile int* abort_flag,
                                                 long long limit) {
  const long long first = sk_tile_iter(p, w.tile, w.ti.phase);
  const long long end = first + w.ti.kblocks;
  const long long t0 = cycle_count();
  for (long long pos = first + w.kb1; pos < end;) {
    const int c = sk_owner(p, pos, nctas);
    const unsigned int* flag = p.sk_flags + static_cast<size_t>(c) * kEpilogueWarps + ew;
    while (ld_acquire_gpu(flag) != p.sk_epoch) {
      if (*abort_flag) return false;
      if (cycle_count() - t0 > limit) {
        *abort_flag = 1;
        atomicOr(p.status, kStatusStreamKTimeout);
        return false;
      }
    }
    pos = sk_share_begin(p, c + 1, nctas);
  }
  return true;
}

// Finisher: sets v to the sum of every later contributor's partial of the
// 16-column groups [g0, g0 + ngroups) (ngroups <= kGroups) of row `row`
// (v[16 * k + j] is column j of group g0 + k, as float bits).  The first
// contributor's loads land straight in v, all in flight together; further
// contributors (rare: tiles split three ways or more) add group by group.
template <int kGroups>
__device__ __forceinline__ void sk_sum_partials(const ConvKernelParams& p, const Work& w, int g0,
                                                int ngroups, int row, int nctas,
                                                uint32_t (&v)[16 * kGroups]) {
  const long long first = sk_tile_iter(p, w.tile, w.ti.phase);
  const long long end = first + w.ti.kblocks;
  long long pos = first + w.kb1;
  int c = sk_owner(p, pos, nctas);
#pragma unroll
  for (int k = 0; k < kGroups; ++k)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 a = k < ngroups ? __ldcg(sk_slot_at(p, c, g0 + k, j, row))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
      v[16 * k + 4 * j] = __float_as_uint(a.x);
      v[16 * k + 4 * j + 1] = __float_as_uint(a.y);
      v[16 * k + 4 * j + 2] = __float_as_uint(a.z);
      v[16 * k + 4 * j + 3] = __float_as_uint(a.w);
    }
  for (pos = sk_share_begin(p, c + 1, nctas); pos < end; pos = sk_share_begin(p, c + 1, nctas)) {
    c = sk_owner(p, pos, nctas);
#pragma unroll
    for (int k = 0; k < kGroups; ++k) {
      if (k < ngroups) {
        float4 a[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] = __ldcg(sk_slot_at(p, c, g0 + k, j, row));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = 16 * k + 4 * j;
          v[e] = __float_as_uint(__uint_as_float(v[e]) + a[j].x);
          v[e + 1] = __float_as_uint(__uint_as_float(v[e + 1]) + a[j].y);
          v[e + 2] = __float_as_uint(__uint_as_float(v[e + 2]) + a[j].z);
          v[e + 3] = __float_as_uint(__uint_as_float(v[e + 3]) + a[j].w);
        }
      }
    }
  }
}

// v[16 * k + j] += TMEM column 16 * k + j (from taddr), k < ngroups: 16 columns
// per load, so only 16 more registers are live.
template <int kGroups>
__device__ __forceinline__ void tmem_add_groups(uint32_t taddr, int ngroups,
                                                uint32_t (&v)[16 * kGroups]) {
#pragma unroll
  for (int k = 0; k < kGroups; ++k) {
    if (k < ngroups) {
      uint32_t t[16];
      tmem_ld_32x32b_x16(taddr + static_cast<uint32_t>(16 * k), t);
      tmem_wait_ld_regs(t);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        v[16 * k + j] = __float_as_uint(__uint_as_float(v[16 * k + j]) + __uint_as_float(t[j]));
    }
  }
}

// Contributor: after the warp's partial stores, publish them (flag = epoch).
__device__ __forceinline__ void sk_publish(const ConvKernelParams& p, int cta, int ew, int lane) {
  __threadfence();
  __syncwarp();
  if (lane == 0 && p.fault_mode != 2)  // (fault_mode 2, a test hook: never publish)
    st_release_gpu(p.sk_flags + static_cast<size_t>(cta) * kEpilogueWarps + ew, p.sk_epoch);
}

// Image and first output row of row-window tile t.
__device__ __forceinline__ void window_origin(const ConvKernelParams& p, int t, int& n_img,
                                              int& oy0) {
  n_img = fast_div(t, p.div_win_rb);
  oy0 = (t - n_img * p.win_row_blocks) * (p.win_rows * p.m_halves);
}

// (image, grid row, grid column) of GEMM row m in phase ph.
__device__ __forceinline__ void grid_pos(const ConvKernelParams& p, int ph, int m, int& n_img,
                                         int& j, int& i) {
  n_img = fast_div(m, p.div_ghw[ph]);
  const int rem = m - n_img * static_cast<int>(p.div_ghw[ph].d);
  j = fast_div(rem, p.div_gw[ph]);
  i = rem - j * p.grid_w[ph];
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

__device__ __forceinline__ float activation(float v, int epilogue) {
  if (epilogue == kEpiRelu) return fmaxf(v, 0.0f);
  if (epilogue == kEpiSilu) return v / (1.0f + __expf(-v));
  return v;
}

// Byte offset of 16-byte piece q of row r in a [rows][row_bytes] tile stored
// with the TMA swizzle whose span equals row_bytes (32, 64 or 128): the
// piece index is XOR-ed with address bits 7 and up.
__device__ __forceinline__ uint32_t swizzled_offset(uint32_t r, uint32_t q, uint32_t row_bytes) {
  const uint32_t lin = r * row_bytes + q * 16;
  return lin ^ (((lin >> 7) & (row_bytes / 16 - 1)) << 4);
}

// Two floats -> two packed 16-bit outputs (one conversion instruction).
template <typename OutT>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Two packed 16-bit values -> two floats.
template <typename OutT>
__device__ __forceinline__ float2 unpack2(uint32_t w);
template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}
template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

template <int kAct>
__device__ __forceinline__ float act_fixed(float v) {
  if (kAct == kEpiRelu) return fmaxf(v, 0.0f);
  if (kAct == kEpiSilu) return v / (1.0f + __expf(-v));
  return v;
}

// One epilogue work item for this thread's row: kCw accumulator columns in
// v, plus beta * source read from `buf` when kRes, activation kAct, one
// rounding, written to `buf` at the same swizzled positions.
template <typename OutT, int kCw, int kAct, bool kRes>
__device__ __forceinline__ void process_row(const uint32_t (&v)[64], uint8_t* buf, uint32_t row,
                                            float beta) {
  constexpr uint32_t kRowBytes = kCw * 2;
  constexpr int kPieces = kCw / 8;
  uint4 src[kPieces];
  uint32_t off[kPieces];
#pragma unroll
  for (int k = 0; k < kPieces; ++k) {
    off[k] = swizzled_offset(row, k, kRowBytes);
    if (kRes) src[k] = *reinterpret_cast<const uint4*>(buf + off[k]);
  }
#pragma unroll
  for (int k = 0; k < kPieces; ++k) {
    float f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(v[k * 8 + e]);
    if (kRes) {
      const uint32_t w[4] = {src[k].x, src[k].y, src[k].z, src[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 sv = unpack2<OutT>(w[e]);
        f[2 * e] = fmaf(beta, sv.x, f[2 * e]);
        f[2 * e + 1] = fmaf(beta, sv.y, f[2 * e + 1]);
      }
    }
    uint4 out;
    out.x = pack2<OutT>(act_fixed<kAct>(f[0]), act_fixed<kAct>(f[1]));
    out.y = pack2<OutT>(act_fixed<kAct>(f[2]), act_fixed<kAct>(f[3]));
    out.z = pack2<OutT>(act_fixed<kAct>(f[4]), act_fixed<kAct>(f[5]));
    out.w = pack2<OutT>(act_fixed<kAct>(f[6]), act_fixed<kAct>(f[7]));
    *reinterpret_cast<uint4*>(buf + off[k]) = out;
  }
}

template <typename OutT, int kCw>
__device__ __forceinline__ void process_row_act(const uint32_t (&v)[64], uint8_t* buf,
                                                uint32_t row, float beta, int act, bool res) {
  if (res) {
    if (act == kEpiRelu) process_row<OutT, kCw, kEpiRelu, true>(v, buf, row, beta);
    else if (act == kEpiSilu) process_row<OutT, kCw, kEpiSilu, true>(v, buf, row, beta);
    else process_row<OutT, kCw, kEpiNone, true>(v, buf, row, beta);
  } else {
    if (act == kEpiRelu) process_row<OutT, kCw, kEpiRelu, false>(v, buf, row, beta);
    else if (act == kEpiSilu) process_row<OutT, kCw, kEpiSilu, false>(v, buf, row, beta);
    else process_row<OutT, kCw, kEpiNone, false>(v, buf, row, beta);
  }
}

// Direct-store epilogue for 16 columns (used when no TMA store map applies).
template <typename OutT>
__device__ __forceinline__ void epilogue_16_direct(const ConvKernelParams& p, long long off,
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
#pragma unroll
  for (int j = 0; j < 16; ++j) f[j] = activation(f[j], p.epilogue);
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

// Direct epilogue of few output channels through a shared-memory stage
// (seg_store): the warp's 32 rows, from GEMM row mw0, are one contiguous run
// of nrows * C_out outputs; each lane computes its row's C_out values from
// acc (+ beta * source, read through the source stage), the warp then writes
// the run with 16-byte words.  `st` holds the output stage, then the source
// stage.
template <typename OutT>
__device__ __forceinline__ void epilogue_seg_warp(const ConvKernelParams& p, int mw0, int lane,
                                                  const uint32_t (&acc)[16], uint8_t* st) {
  const int nrows = min(32, p.rows[0] - mw0);
  if (nrows <= 0) return;
  const int cout = p.Cout;
  const long long first = static_cast<long long>(mw0) * cout;
  uint8_t* gout = reinterpret_cast<uint8_t*>(static_cast<OutT*>(p.out) + first);
  const int phase16 = static_cast<int>(reinterpret_cast<uintptr_t>(gout) & 15u);
  const int bytes = nrows * cout * static_cast<int>(sizeof(OutT));
  uint8_t* st_src = st + p.seg_slot_bytes;
  if (p.has_residual) {
    copy_segment16<true>(
        reinterpret_cast<const uint8_t*>(static_cast<const OutT*>(p.src) + first), st_src,
        phase16, bytes, lane, 32);
    __syncwarp();
  }
  if (lane < nrows) {
    const OutT* sv = reinterpret_cast<const OutT*>(st_src + phase16) + lane * cout;
    OutT* ov = reinterpret_cast<OutT*>(st + phase16) + lane * cout;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      if (c < cout) {
        float f = __uint_as_float(acc[c]);
        if (p.has_residual) f = fmaf(p.beta, to_f32<OutT>(sv[c]), f);
        ov[c] = from_f32<OutT>(activation(f, p.epilogue));
      }
    }
  }
  __syncwarp();
  copy_segment16<false>(gout, st, phase16, bytes, lane, 32);
  __syncwarp();  // the stage is free again
}

// Issues the TMA loads of the residual-source chunks that epilogue group
// `grp` owns in one tile: work item q = h * nchunks + c (128-row half h,
// column chunk c) belongs to group q % 2.  The buffer is laid out
// [half][chunk][128][cw]; completion is tracked by `bar`.
__device__ __forceinline__ void issue_source_items(const ConvKernelParams& p, const TileInfo& ti,
                                                   uint8_t* buf, uint32_t bar, int grp) {
  const uint32_t chunk_bytes = kBM * p.cw * 2;
  const int nchunks = p.bn / p.cw;
  const int nitems = nchunks * p.m_halves;
  const int mine = (nitems - grp + kEpilogueGroups - 1) / kEpilogueGroups;
  if (mine <= 0) return;
  // A row-window half fills only its win_half_rows rows of the chunk buffer.
  const uint32_t box_bytes =
      p.epi_mode == 3 ? static_cast<uint32_t>(p.win_half_rows) * p.cw * 2 : chunk_bytes;
  mbar_arrive_expect_tx(bar, box_bytes * mine);
  for (int q = grp; q < nitems; q += kEpilogueGroups) {
    const int h = q / nchunks;
    const int c = q - h * nchunks;
    const int mh = ti.m0 + h * kBM;
    const uint32_t dst = smem_u32(buf + q * p.src_chunk_bytes);
    if (p.epi_mode == 1) {
      tma_load_3d(dst, &p.map_src[ti.phase], bar, ti.n0 + c * p.cw, ti.group, mh);
    } else if (p.epi_mode == 3) {
      int n_img, oy0;
      window_origin(p, ti.m0, n_img, oy0);
      tma_load_4d(dst, &p.map_src[0], bar, ti.n0 + c * p.cw, 0, oy0 + h * p.win_rows, n_img);
    } else {
      int n_img, j, i;
      grid_pos(p, ti.phase, mh, n_img, j, i);
      tma_load_4d(dst, &p.map_src[ti.phase], bar, ti.n0 + c * p.cw, i, j, n_img);
    }
  }
}

// Issues the MMAs of one k-block: kSteps K-steps of 32 bytes per operand row,
// kHalves 128-row halves of A sharing the B operand.  Descriptors are built
// from precomputed high bits plus an address field advanced by adds only: the
// issuing warp is latency-bound, so nothing here divides or branches.  Every
// lane of the (converged) MMA warp runs this; one lane issues each MMA.
// kPair: one M = 256 MMA over both CTAs of a pair (issued by rank 0).
template <int kKind, int kSteps, int kHalves, bool kPair = false>
__device__ __forceinline__ void issue_kblock(uint32_t d_tmem, uint64_t desc_hi, uint32_t a_lo,
                                             uint32_t b_lo, uint32_t half_lo, uint32_t bn_cols,
                                             uint32_t idesc, uint32_t first_accumulate) {
#pragma unroll
  for (int kk = 0; kk < kSteps; ++kk) {
    const uint64_t bdesc = desc_hi | static_cast<uint64_t>(b_lo + 2u * kk);
    const uint32_t accumulate = kk == 0 ? first_accumulate : 1u;
#pragma unroll
    for (int h = 0; h < kHalves; ++h) {
      const uint64_t adesc = desc_hi | static_cast<uint64_t>(a_lo + h * half_lo + 2u * kk);
      if (kPair) {
        if (kKind == kKindF16)
          mma_f16_pair_warp(d_tmem + h * bn_cols, adesc, bdesc, idesc, accumulate);
        else
          mma_f8_pair_warp(d_tmem + h * bn_cols, adesc, bdesc, idesc, accumulate);
      } else {
        if (kKind == kKindF16)
          mma_f16_warp(d_tmem + h * bn_cols, adesc, bdesc, idesc, accumulate);
        else
          mma_f8_warp(d_tmem + h * bn_cols, adesc, bdesc, idesc, accumulate);
      }
    }
  }
}

// The MMA role for one (kSteps, kHalves) specialisation.  Tiles t0, t0 +
// step, ...  kPair: rank 0 of a CTA pair issues M = 256 MMAs over both CTAs'
// operands (each holds bn/2 rows of B) and commits to both CTAs' barriers.
// `half`: with two issuing warps (mma_split) each issues the MMAs of one
// 128-row half (kHalves = 1), into that half's accumulator columns; -1: this
// warp issues every half.
template <int kKind, int kSteps, int kHalves, bool kPair = false, bool kStreamK = false>
__device__ __forceinline__ bool mma_role(const ConvKernelParams& p, uint32_t tmem_base,
                                         uint8_t* a_ring, uint8_t* b_ring, uint8_t* b_res,
                                         uint64_t* full, uint64_t* empty, uint64_t* tfull,
                                         uint64_t* tempty, int half, volatile int* abort_flag,
                                         unsigned int* status, long long limit, int t0,
                                         int step) {
  const int stages = p.stages;
  const uint32_t sw = p.sw_bytes;
  const uint32_t a_bytes = kBM * p.m_halves * sw;  // stage stride: every half of A
  const uint32_t b_bytes = static_cast<uint32_t>(kPair ? p.bn / 2 : p.bn) * sw;
  const uint64_t desc_hi = smem_desc_kmajor(0, sw);  // address field zero
  const uint32_t h0 = half < 0 ? 0u : static_cast<uint32_t>(half);
  const uint32_t a_lo0 = (smem_u32(a_ring) >> 4) + h0 * ((kBM * sw) >> 4);
  const uint32_t b_lo0 = smem_u32(p.b_resident ? b_res : b_ring) >> 4;
  const uint32_t a_step = a_bytes >> 4;
  const uint32_t b_step = b_bytes >> 4;
  const uint32_t half_lo = (kBM * sw) >> 4;
  const uint32_t bn_cols = static_cast<uint32_t>(p.bn);
  const uint32_t idesc = p.idesc;
  const uint32_t full0 = smem_u32(full), empty0 = smem_u32(empty);
  // Loop-invariant parameters in registers: the tcgen05 asm statements below
  // clobber memory, which would otherwise make the compiler re-read them.
  const bool b_resident = p.b_resident != 0;
  const uint32_t acc_stride = p.acc_stride;
  const int total_tiles = p.total_tiles;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t a_lo = a_lo0;
  uint32_t bs_lo = b_lo0;  // streamed B: advances with the ring
  bool ok = true;
  int it = 0;
  (void)total_tiles;
  WorkWalk walk = work_begin<kStreamK>(p, t0, step);
  Work wk;
  for (; ok && work_next<kStreamK>(p, walk, wk); ++it) {
    const TileInfo& ti = wk.ti;
    const int acc = it & 1;
    if (!__all_sync(0xFFFFFFFFu,
                    mbar_wait_bounded(smem_u32(&tempty[acc]),
                                      static_cast<uint32_t>(((it >> 1) & 1) ^ 1), abort_flag,
                                      status, kStatusMmaTimeout, limit, 0u, kPair))) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (ti.kblocks == 0) {  // a phase with no filter taps: the epilogue writes act(0)
      if (kPair) {
        mma_commit_pair_warp(smem_u32(&tfull[acc]));
      } else if ((threadIdx.x & 31) == 0) {
        mbar_arrive(smem_u32(&tfull[acc]));
      }
      __syncwarp();
      continue;
    }
    const uint32_t d_tmem =
        tmem_base + static_cast<uint32_t>(acc) * acc_stride + h0 * bn_cols;
    // Resident B: block kb of the tile sits at index kb.
    uint32_t br_lo = b_lo0 + static_cast<uint32_t>(wk.kb0) * b_step;
    const int kblocks = wk.kb1 - wk.kb0;
    for (int kb = 0; kb < kblocks; ++kb) {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(full0 + 8u * stage, phase, abort_flag,
                                                     status, kStatusMmaTimeout, limit, 0u,
                                                     kPair))) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_kblock<kKind, kSteps, kHalves, kPair>(d_tmem, desc_hi, a_lo,
                                                  b_resident ? br_lo : bs_lo, half_lo, bn_cols,
                                                  idesc, kb != 0 ? 1u : 0u);
      if (kPair)
        mma_commit_pair_warp(empty0 + 8u * stage);
      else
        mma_commit_warp(empty0 + 8u * stage);
      br_lo += b_step;
      a_lo += a_step;
      bs_lo += b_step;
      if (++stage == stages) {
        stage = 0;
        phase ^= 1u;
        a_lo = a_lo0;
        bs_lo = b_lo0;
      }
    }
    if (!ok) break;
    if (kPair)
      mma_commit_pair_warp(smem_u32(&tfull[acc]));
    else
      mma_commit_warp(smem_u32(&tfull[acc]));
  }
  return ok;
}

// The MMA role of the row-window loader: one A box per channel block holds
// the tile's input rows with halo; tap (r, s) of half h starts at box row
// h*win_half_rows + r*win_pitch + s.  The filter is resident: block
// (tap, cb) of the packed filter sits at index tap*c_blocks + cb.
template <int kKind, int kSteps, int kHalves>
__device__ __forceinline__ bool mma_role_window(const ConvKernelParams& p, uint32_t tmem_base,
                                                uint8_t* a_ring, uint8_t* b_res, uint64_t* full,
                                                uint64_t* empty, uint64_t* tfull, uint64_t* tempty,
                                                int half, volatile int* abort_flag,
                                                unsigned int* status, long long limit, int t0,
                                                int step) {
  const int stages = p.stages;
  const uint32_t sw = p.sw_bytes;  // 128 in this mode
  const uint32_t b_bytes = static_cast<uint32_t>(p.bn) * sw;
  const uint64_t desc_hi = smem_desc_kmajor(0, sw);
  const uint32_t row_lo = sw >> 4;  // one box row in descriptor address units
  const uint32_t half_lo = static_cast<uint32_t>(p.win_half_rows) * row_lo;
  const uint32_t h0 = half < 0 ? 0u : static_cast<uint32_t>(half);
  const uint32_t a_lo0 = (smem_u32(a_ring) >> 4) + h0 * half_lo;
  const uint32_t b_lo0 = smem_u32(b_res) >> 4;
  const uint32_t a_step = p.win_stage_bytes >> 4;
  const uint32_t b_step = b_bytes >> 4;
  const uint32_t bn_cols = static_cast<uint32_t>(p.bn);
  const uint32_t idesc = p.idesc;
  const uint32_t full0 = smem_u32(full), empty0 = smem_u32(empty);
  const int taps_s = p.win_S;
  const int taps = p.win_R * p.win_S;
  // Loop-invariant parameters in registers (the tcgen05 asm clobbers memory).
  const int c_blocks = p.c_blocks, total_tiles = p.total_tiles;
  const uint32_t acc_stride = p.acc_stride;
  const uint32_t b_tap_step = static_cast<uint32_t>(c_blocks) * b_step;  // next tap, same block
  const uint32_t a_row_skip = static_cast<uint32_t>(p.win_pitch - taps_s) * row_lo;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t a_lo = a_lo0;
  bool ok = true;
  int it = 0;
  for (int t = t0; ok && t < total_tiles; t += step, ++it) {
    const int acc = it & 1;
    if (!__all_sync(0xFFFFFFFFu,
                    mbar_wait_bounded(smem_u32(&tempty[acc]),
                                      static_cast<uint32_t>(((it >> 1) & 1) ^ 1), abort_flag,
                                      status, kStatusMmaTimeout, limit))) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * acc_stride + h0 * bn_cols;
    for (int cb = 0; cb < c_blocks; ++cb) {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(full0 + 8u * stage, phase, abort_flag,
                                                     status, kStatusMmaTimeout, limit))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // Tap (r, s) reads box row r*pitch + s and filter block tap*c_blocks + cb.
      uint32_t tap_lo = a_lo;
      uint32_t b_lo = b_lo0 + static_cast<uint32_t>(cb) * b_step;
      int s = 0;
      for (int tap = 0; tap < taps; ++tap) {
        issue_kblock<kKind, kSteps, kHalves>(d_tmem, desc_hi, tap_lo, b_lo, half_lo, bn_cols,
                                             idesc, (cb | tap) != 0 ? 1u : 0u);
        b_lo += b_tap_step;
        tap_lo += row_lo;
        if (++s == taps_s) {
          s = 0;
          tap_lo += a_row_skip;
        }
      }
      mma_commit_warp(empty0 + 8u * stage);
      a_lo += a_step;
      if (++stage == stages) {
        stage = 0;
        phase ^= 1u;
        a_lo = a_lo0;
      }
    }
    if (!ok) break;
    mma_commit_warp(smem_u32(&tfull[acc]));
  }
  return ok;
}

// ---------------------------------------------------------------- gather A loader
// Builds the A operand with plain loads for inputs whose channel rows a TMA
// box cannot address.  An A row (output pixel) of the contraction is the
// sequence of runs r = 0 .. R-1; run r holds the input bytes under filter row
// r and taps s = 0 .. S-1, which for dil_w = 1 are S adjacent pixels, i.e.
// S*C_in*elt contiguous bytes of the NHWC input, zero-padded to g_run_bytes.
// A k-block is 128 bytes of that sequence, so each of its 16-byte pieces lies
// inside one run: it is the bytes at one input address, with the pixels left
// or right of the image (and the run's padding) zeroed.

constexpr int kGatherBatch = 8;  // rows per lane whose loads are in flight together

// Mask keeping bytes [lo, hi) of a 16-byte piece (lo, hi clamped to [0, 16]).
__device__ __forceinline__ uint4 byte_range_mask(int lo, int hi) {
  uint32_t m[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int a = min(max(lo - 4 * j, 0), 4);
    const int b = min(max(hi - 4 * j, 0), 4);
    const uint32_t below_b = b == 4 ? 0xFFFFFFFFu : ((1u << (8 * b)) - 1u);
    const uint32_t below_a = a == 4 ? 0xFFFFFFFFu : ((1u << (8 * a)) - 1u);
    m[j] = b > a ? (below_b & ~below_a) : 0u;
  }
  return make_uint4(m[0], m[1], m[2], m[3]);
}

__device__ __forceinline__ uint4 and4(uint4 a, uint4 b) {
  return make_uint4(a.x & b.x, a.y & b.y, a.z & b.z, a.w & b.w);
}

// Bytes [sh, sh + 16) of the 32 bytes (w0, w1), sh in [0, 16).
__device__ __forceinline__ uint4 shift_pair(uint4 w0, uint4 w1, int sh) {
  const uint32_t v[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  const int wq = sh >> 2;
  uint32_t t[6], u[5];
#pragma unroll
  for (int j = 0; j < 6; ++j) t[j] = (wq & 2) ? v[j + 2] : v[j];
#pragma unroll
  for (int j = 0; j < 5; ++j) u[j] = (wq & 1) ? t[j + 1] : t[j];
  const uint32_t bits = static_cast<uint32_t>(sh & 3) * 8u;
  return make_uint4(__funnelshift_r(u[0], u[1], bits), __funnelshift_r(u[1], u[2], bits),
                    __funnelshift_r(u[2], u[3], bits), __funnelshift_r(u[3], u[4], bits));
}

// First padded input row (see g_pr) that the tile starting at GEMM row m0
// reads, and how many consecutive padded rows it spans.
__device__ __forceinline__ void gather_tile_rows(const ConvKernelParams& p, int m0, int& g_first,
                                                 int& count) {
  const int m_last = min(m0 + kBM * p.m_halves, p.rows[0]) - 1;
  int na, oya, nb, oyb, xa, xb;
  grid_pos(p, 0, m0, na, oya, xa);
  grid_pos(p, 0, m_last, nb, oyb, xb);
  g_first = na * p.g_pr + oya * p.step_h;
  count = nb * p.g_pr + oyb * p.step_h + (p.g_runs - 1) * p.dil_h - g_first + 1;
}

// Row table of the tile whose first GEMM row is m0, one 16-byte entry per
// row: {row index of filter row 0 -- in the input tensor, n*H + iy0, or,
// with staging, the staging slot --, iy0, ix0, row < M}.  Built once per
// tile by each producer warp, so that its k-blocks need no division and
// every row's work is independent of the others'.
__device__ __forceinline__ void gather_row_table(const ConvKernelParams& p, int4* tab, int m0,
                                                 int g_first, int lane) {
  const int rows = kBM * p.m_halves;
  const FastDiv div_hw = p.div_ghw[0], div_wo = p.div_gw[0];
  const int Wo = p.Wo, hw = p.Ho * p.Wo, M = p.rows[0];
  const int step_h = p.step_h, step_w = p.step_w, base_h = p.base_h[0], base_w = p.base_w[0];
  const int staged = p.g_stage, g_pr = p.g_pr, g_h = p.g_h;
  for (int i = lane; i < rows; i += 32) {
    const int m = m0 + i;
    const int n = fast_div(m, div_hw);
    const int rem = m - n * hw;
    const int oy = fast_div(rem, div_wo);
    const int ox = rem - oy * Wo;
    const int iy0 = oy * step_h + base_h;
    const int ix0 = ox * step_w + base_w;
    const int row = staged ? n * g_pr + oy * step_h - g_first : n * g_h + iy0;
    tab[i] = make_int4(row, iy0, ix0, m < M ? 1 : 0);
  }
  __syncwarp();
}

// Zeroes the margins of every slot of both staging buffers (the bulk copies
// only ever write the rows between them).
__device__ __forceinline__ void gather_zero_margins(const ConvKernelParams& p, uint8_t* gstage,
                                                    int lane) {
  const int slots = 2 * p.g_slots;
  const int left = p.g_slot_pad / 16;
  const int right = (p.g_slot_bytes - p.g_slot_pad - p.g_row_bytes) / 16;
  const int per = left + right;
  for (int i = lane; i < slots * per; i += 32) {
    const int j = i / per, k = i - j * per;
    const int buf = j / p.g_slots, slot = j - buf * p.g_slots;
    const int off = k < left ? 16 * k : p.g_slot_pad + p.g_row_bytes + 16 * (k - left);
    *reinterpret_cast<uint4*>(gstage + buf * p.g_stage_bytes + slot * p.g_slot_bytes + off) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  __syncwarp();
}

// Issues the bulk copies of the input rows the tile starting at GEMM row m0
// reads into a staging buffer (slot j = padded row g_first + j, rows in the
// padding are not copied), completing on `bar`.  The whole warp takes part:
// lane l copies slots l, l + 32, ...
__device__ __forceinline__ void gather_stage_tile(const ConvKernelParams& p, int m0, uint8_t* buf,
                                                  uint32_t bar, int lane) {
  int g_first, count;
  gather_tile_rows(p, m0, g_first, count);
  count = min(count, p.g_slots);  // the host's bound makes this a no-op
  const int pad_h = -p.base_h[0], g_pr = p.g_pr, g_n = p.g_n, g_h = p.g_h;
  const int row_bytes = p.g_row_bytes, slot_bytes = p.g_slot_bytes, slot_pad = p.g_slot_pad;
  const uint8_t* const input = p.g_input;
  const FastDiv div_pr = p.g_div_pr;
  for (int j0 = 0; j0 < count; j0 += 32) {
    // Each pass raises the transaction count by its bytes before its copies;
    // the phase completes after the final arrival below.
    const int j = j0 + lane;
    const int g = g_first + j;
    const int n = fast_div(g, div_pr);
    const int iy = g - n * g_pr - pad_h;
    const bool copy = j < count && n < g_n && iy >= 0 && iy < g_h;
    const uint32_t bytes = __reduce_add_sync(0xFFFFFFFFu, copy ? static_cast<uint32_t>(row_bytes) : 0u);
    if (lane == 0 && bytes) mbar_expect_tx(bar, bytes);
    __syncwarp();
    if (copy)
      bulk_load(smem_u32(buf + static_cast<size_t>(j) * slot_bytes + slot_pad),
                input + (static_cast<long long>(n) * g_h + iy) * row_bytes,
                static_cast<uint32_t>(row_bytes), bar);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// Fills one A stage (128 * m_halves rows x 128 bytes, 128-byte swizzle) with
// k-block kb, from the tile's row table and either the input in global
// memory or the tile's staged input rows (kStaged; `stage` is their
// shared-memory address).  Lane l writes piece l % 8 of rows l / 8, l / 8 + 4, ...
// A piece keeps only the bytes of its run that lie inside the image: bytes
// past the run's end (its padding) are cleared by a per-lane mask, pixels
// left or right of the image by a byte mask on the (rare) edge rows, and
// rows in the padding or past M are zero.
template <bool kStaged>
__device__ __forceinline__ void gather_a_kblock(const ConvKernelParams& p, const int4* tab,
                                                uint32_t stage, uint8_t* a_stage, int kb,
                                                int lane) {
  // Every parameter the loop needs, in registers (the loop's stores could
  // otherwise make the compiler re-read them).
  const int g_h = p.g_h, g_w = p.g_w, g_s = p.g_s, g_slots = p.g_slots;
  const int slot_bytes = p.g_slot_bytes, slot_pad = p.g_slot_pad;
  const uint8_t* const input = p.g_input;
  const int q = lane & 7;
  const int kbyte = kb * 128 + 16 * q;
  const int u = fast_div(kbyte, p.g_div_run);  // filter row of this piece's run
  const int jb = kbyte - u * p.g_run_bytes;
  const bool piece_ok = u < p.g_runs && jb < p.g_run_len_bytes;
  const uint4 run_mask = byte_range_mask(0, p.g_run_len_bytes - jb);
  const int pix_bytes = p.g_c * p.g_elt;
  const long long row_bytes = static_cast<long long>(g_w) * pix_bytes;
  const int dy = u * p.dil_h;
  const int rows = kBM * p.m_halves;
  for (int i0 = lane >> 3; i0 < rows; i0 += 4 * kGatherBatch) {
    long long addr[kGatherBatch];
    bool ok[kGatherBatch], edge[kGatherBatch];
    int e_lo[kGatherBatch], e_hi[kGatherBatch];
#pragma unroll
    for (int g = 0; g < kGatherBatch; ++g) {
      const int4 row = tab[i0 + 4 * g];
      const int iy = row.y + dy;
      // (Staged rows: the slot also stays inside the buffer, whatever the tile.)
      ok[g] = piece_ok && row.w != 0 && static_cast<unsigned>(iy) < static_cast<unsigned>(g_h) &&
              (!kStaged || static_cast<unsigned>(row.x + dy) < static_cast<unsigned>(g_slots));
      // Bytes of the run inside the image: taps s with 0 <= ix0 + s < W.
      edge[g] = row.z < 0 || row.z + g_s > g_w;
      e_lo[g] = max(max(0, -row.z) * pix_bytes - jb, 0);
      e_hi[g] = min(min(g_s, g_w - row.z) * pix_bytes - jb, 16);
      addr[g] = kStaged ? static_cast<long long>((row.x + dy) * slot_bytes + slot_pad + row.z * pix_bytes + jb)
                        : (row.x + dy) * row_bytes + static_cast<long long>(row.z) * pix_bytes + jb;
    }
    if (kStaged) {
      // Five 4-byte words from the one holding the piece's first byte; the
      // slot's zero margins supply the pixels left or right of the image.
      uint32_t w[kGatherBatch][5];
#pragma unroll
      for (int g = 0; g < kGatherBatch; ++g) {
        const uint32_t a = stage + (static_cast<uint32_t>(addr[g]) & ~3u);
#pragma unroll
        for (int k = 0; k < 5; ++k) w[g][k] = ok[g] ? lds32(a + 4u * k) : 0u;
      }
#pragma unroll
      for (int g = 0; g < kGatherBatch; ++g) {
        const uint32_t bits = (static_cast<uint32_t>(addr[g]) & 3u) * 8u;
        const uint4 v = and4(make_uint4(__funnelshift_r(w[g][0], w[g][1], bits),
                                        __funnelshift_r(w[g][1], w[g][2], bits),
                                        __funnelshift_r(w[g][2], w[g][3], bits),
                                        __funnelshift_r(w[g][3], w[g][4], bits)),
                             run_mask);
        const uint32_t row = static_cast<uint32_t>(i0 + 4 * g);
        *reinterpret_cast<uint4*>(a_stage + swizzled_offset(row, static_cast<uint32_t>(q), 128u)) =
            v;
      }
    } else {
      // Only aligned 16-byte words that hold a kept byte are read, so every
      // load stays inside the input's 16-byte granules.
      uint4 w0[kGatherBatch], w1[kGatherBatch];
#pragma unroll
      for (int g = 0; g < kGatherBatch; ++g) {
        const long long f = addr[g] & ~15ll;
        w0[g] = make_uint4(0u, 0u, 0u, 0u);
        w1[g] = make_uint4(0u, 0u, 0u, 0u);
        if (ok[g] && e_hi[g] > e_lo[g]) {
          if (addr[g] + e_lo[g] < f + 16) w0[g] = __ldg(reinterpret_cast<const uint4*>(input + f));
          if (addr[g] + e_hi[g] > f + 16)
            w1[g] = __ldg(reinterpret_cast<const uint4*>(input + f + 16));
        }
      }
#pragma unroll
      for (int g = 0; g < kGatherBatch; ++g) {
        uint4 v = and4(shift_pair(w0[g], w1[g], static_cast<int>(addr[g] & 15)), run_mask);
        if (__any_sync(0xFFFFFFFFu, edge[g]) && edge[g])
          v = and4(v, byte_range_mask(e_lo[g], e_hi[g]));
        if (!ok[g]) v = make_uint4(0u, 0u, 0u, 0u);
        const uint32_t row = static_cast<uint32_t>(i0 + 4 * g);
        *reinterpret_cast<uint4*>(a_stage + swizzled_offset(row, static_cast<uint32_t>(q), 128u)) =
            v;
      }
    }
  }
}

// Producer role of the gather loader (one of kGatherProducers warps, `role`):
// the whole warp builds the A k-blocks whose sequence number is congruent to
// its role; lane 0 also streams the B k-block (or, on the first tile, the
// resident filter block) by TMA.  The stage's full barrier completes with
// lane 0's arrival after the warp's shared-memory writes are fenced for the
// tensor cores, plus the B bytes.  With row staging, role 0's lanes also
// issue the bulk copies of the next tile's input rows into the other staging
// buffer once every builder warp has released it; each warp waits for a
// tile's rows before its first k-block there and releases the buffer after
// its last.
__device__ __forceinline__ void gather_producer(const ConvKernelParams& p, int role, int lane,
                                                uint8_t* a_ring, uint8_t* b_ring, uint8_t* b_res,
                                                int4* tab, uint8_t* gstage, uint64_t* full,
                                                uint64_t* empty, uint64_t* gst_full,
                                                uint64_t* gst_empty, volatile int* abort_flag,
                                                unsigned int* status, long long limit) {
  const int stages = p.stages;
  const uint32_t a_bytes = kBM * p.m_halves * 128u;
  const uint32_t b_bytes = static_cast<uint32_t>(p.bn) * 128u;
  int stage = 0;
  uint32_t phase = 0;
  long long seq = 0, last_issued = -1;
  bool ok = true, first_tile = true;
  int staged[2] = {0, 0};  // staging uses issued per buffer (warp 0, lane 0)
  int sel = 0;             // seq % kGatherProducers
  int it = 0;
  for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x, ++it) {
    const TileInfo ti = decode_tile(p, t);
    const bool load_res = p.b_resident && first_tile;
    const int sb = it & 1;
    if (p.g_stage) {
      if (role == 0) {
        if (first_tile) {
          gather_zero_margins(p, gstage, lane);
          gather_stage_tile(p, ti.m0, gstage, smem_u32(&gst_full[0]), lane);
          ++staged[0];
        }
        const int tn = t + static_cast<int>(gridDim.x);
        if (tn < p.total_tiles) {
          // The other buffer last held tile it-1: every builder warp must be done with it.
          const int nb = sb ^ 1;
          int w = 1;
          if (lane == 0)
            w = mbar_wait_bounded(smem_u32(&gst_empty[nb]),
                                  static_cast<uint32_t>(((it + 1) >> 1) & 1) ^ 1u, abort_flag,
                                  status, kStatusProducerTimeout, limit) ? 1 : 0;
          if (__shfl_sync(0xFFFFFFFFu, w, 0)) {
            gather_stage_tile(p, decode_tile(p, tn).m0, gstage + nb * p.g_stage_bytes,
                              smem_u32(&gst_full[nb]), lane);
            ++staged[nb];
          } else {
            ok = false;
          }
        }
      }
      if (!ok) break;
      // Every warp waits for the tile's rows, even one without a k-block
      // here, so that no warp can release a buffer use twice.
      int w = 1;
      if (lane == 0)
        w = mbar_wait_bounded(smem_u32(&gst_full[sb]), static_cast<uint32_t>((it >> 1) & 1),
                              abort_flag, status, kStatusProducerTimeout, limit) ? 1 : 0;
      if (!__shfl_sync(0xFFFFFFFFu, w, 0)) {
        ok = false;
        break;
      }
    }
    first_tile = false;
    int g_first = 0, count = 0;
    if (p.g_stage) gather_tile_rows(p, ti.m0, g_first, count);
    const uint32_t stage_u32 = smem_u32(gstage + sb * p.g_stage_bytes);
    bool have_table = false;
    for (int kb = 0; kb < ti.kblocks; ++kb, ++seq) {
      const bool mine = sel == role;  // k-block seq belongs to warp seq % kGatherProducers
      if (++sel == kGatherProducers) sel = 0;
      if (mine) {
        if (!have_table) {
          gather_row_table(p, tab, ti.m0, g_first, lane);
          have_table = true;
        }
        int w = 1;
        if (lane == 0)
          w = mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, status,
                                kStatusProducerTimeout, limit, p.wait_hint_ns) ? 1 : 0;
        w = __shfl_sync(0xFFFFFFFFu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
        last_issued = seq;
        if (!(p.fault_mode == 1 && blockIdx.x == 0 && seq == 0)) {
          // (fault_mode 1, a test hook: CTA 0 leaves its first stage un-armed.)
          const uint32_t fb = smem_u32(&full[stage]);
          if (lane == 0) {
            if (!p.b_resident) {
              mbar_expect_tx(fb, b_bytes);
              tma_load_3d(smem_u32(b_ring + stage * b_bytes), &p.map_b, fb, kb * p.bk, ti.n0, 0);
            } else if (load_res) {
              mbar_expect_tx(fb, b_bytes);
              tma_load_3d(smem_u32(b_res + kb * b_bytes), &p.map_b, fb, kb * p.bk, 0, 0);
            }
          }
          if (p.g_stage)
            gather_a_kblock<true>(p, tab, stage_u32, a_ring + stage * a_bytes, kb, lane);
          else
            gather_a_kblock<false>(p, tab, 0u, a_ring + stage * a_bytes, kb, lane);
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(fb);
        }
      }
      if (++stage == stages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (p.g_stage && ok) {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&gst_empty[sb]));
    }
  }
  if (!ok && lane == 0) {
    // Let this warp's copies in flight land before exiting: B k-blocks, and
    // (warp 0) the latest row staging of each buffer.
    for (long long q = last_issued - stages + 1; q <= last_issued; ++q)
      if (q >= 0 && q % kGatherProducers == role)
        mbar_wait_drain(smem_u32(&full[q % stages]), static_cast<uint32_t>((q / stages) & 1),
                        limit / 8 + 1);
    for (int b = 0; b < 2; ++b)
      if (staged[b] > 0)
        mbar_wait_drain(smem_u32(&gst_full[b]), static_cast<uint32_t>((staged[b] - 1) & 1),
                        limit / 8 + 1);
  }
}

// kGather selects the producer role: the gather loader, or the TMA loaders
// (im2col and row window).  The two are separate instances so that neither
// carries the other's registers.
// kPair: the CTAs run as clusters of two.  A pair works on one tile of 256
// rows: rank r's producers load rows [128r, 128r + 128) of A and filter rows
// [r*bn/2, (r+1)*bn/2) of B into its own shared memory, rank 0 issues M = 256
// MMAs over both (tcgen05 cta_group::2), and each CTA's epilogue stores its
// 128 rows from its own TMEM.  TMA im2col loader, streamed filter only.
template <int kKind, typename OutT, bool kGather, bool kPair = false, bool kStreamK = false>
__global__ void __launch_bounds__(kThreads, 1)
    conv_igemm_kernel(const __grid_constant__ ConvKernelParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int stages = p.stages;
  const uint32_t sw = p.sw_bytes;
  const uint32_t a_bytes = kBM * p.m_halves * sw;
  const uint32_t b_bytes = static_cast<uint32_t>(kPair ? p.bn / 2 : p.bn) * sw;
  // Tile walk: CTAs (or CTA pairs) take tiles tile0, tile0 + tile_step, ...
  const uint32_t rank = kPair ? cluster_rank() : 0u;
  const int tile0 = kPair ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int tile_step = kPair ? static_cast<int>(num_clusters_x()) : static_cast<int>(gridDim.x);
  const int m_off = static_cast<int>(rank) * kBM;  // this CTA's rows within a pair's tile

  uint8_t* a_ring = smem + p.off_a;
  uint8_t* b_ring = smem + p.off_b;
  uint8_t* b_res = smem + p.off_bres;
  uint8_t* src_base = smem + p.off_src;
  uint8_t* stg_base = smem + p.off_stg;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* full = bars;
  uint64_t* empty = bars + stages;
  uint64_t* tfull = bars + 2 * stages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* bres_full = drain + 1;
  uint64_t* src_full = bres_full + 1;  // [buffer][group]
  uint64_t* epi_done = src_full + 4;   // every epilogue warp has finished with TMEM
  uint64_t* gst_full = epi_done + 1;   // gather row staging: [buffer]
  uint64_t* gst_empty = gst_full + 2;
  uint64_t* drain2 = gst_empty + 2;    // the second MMA issuer's drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain2 + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned int* status = p.status;
  const long long limit = p.timeout_cycles;

  if (threadIdx.x == 0) {
    // Stage-empty and accumulator-full phases take one commit per MMA issuer.
    const uint32_t issuers = p.mma_split ? 2u : 1u;
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), issuers);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull[a]), issuers);
      mbar_init(smem_u32(&tempty[a]), kEpilogueWarps * (kPair ? 2 : 1));
      mbar_init(smem_u32(&src_full[2 * a]), 1);
      mbar_init(smem_u32(&src_full[2 * a + 1]), 1);
    }
    mbar_init(smem_u32(drain), 1);
    mbar_init(smem_u32(drain2), 1);
    mbar_init(smem_u32(bres_full), 1);
    mbar_init(smem_u32(epi_done), kEpilogueWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&gst_full[b]), 1);
      mbar_init(smem_u32(&gst_empty[b]), kGatherProducers);  // every builder warp
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    if (kPair) {
      tmem_alloc_pair(smem_u32(tmem_slot), p.tmem_cols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
      tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    if (!kGather)
      for (int ph = 0; ph < p.num_phases; ++ph) tma_prefetch_desc(&p.map_a[ph]);
    tma_prefetch_desc(&p.map_b);
  }
  tc_fence_before();
  __syncthreads();
  // Both CTAs of a pair have initialised their barriers before either
  // signals one of the other's.
  if (kPair) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Set-up above may overlap the previous kernel in the stream.  Every role
  // waits for that kernel to complete before its first global memory access
  // or bounded wait; a TMA producer waits only right before its first copy,
  // so walking to it (parameters only, no memory) overlaps that kernel too.
  grid_launch_dependents();

  const bool split_issuer = !kGather && !kPair && p.mma_split;  // warp 11 issues MMAs
  const bool tma_producer =
      !kGather && (warp == 0 || warp == kProducer2Warp || (warp == kProducer3Warp && !split_issuer));
  // (Not with the gather loader: its builder warps ran the RGB stem 78 -> 85
  // us when the epilogue warps waited after their zero pass.)
  const bool staged_epilogue =
      !kGather && warp >= 2 && warp < 2 + kEpilogueWarps && p.epi_mode != 0;
  if (!tma_producer && !staged_epilogue) grid_dependency_wait();
  if (warp == 0 || warp == kProducer2Warp || (warp == kProducer3Warp && !split_issuer)) {
    // ------------------------------------------------------------ producers
    // The producer warps walk the same k-block sequence; with the TMA loaders
    // k-block `seq` is issued by producer seq % nprod, so two or three TMA
    // issue streams overlap; the gather loader's three warps (0, 10, 11)
    // build every third k-block each.
    if constexpr (kGather) {
      const int role = warp == 0 ? 0 : (warp == kProducer2Warp ? 1 : 2);
      int4* tab = reinterpret_cast<int4*>(smem + p.off_gtab) + role * kBM * p.m_halves;
      gather_producer(p, role, lane, a_ring, b_ring, b_res, tab, smem + p.off_gstage, full, empty,
                      gst_full, gst_empty, abort_flag, status, limit);
    } else {
      // The whole warp walks the k-blocks (operands stay warp-uniform); lane 0
      // issues the copies.  K-block `seq` belongs to producer seq % nprod:
      // warps 0 and 10, and warp 11 too when it issues no MMAs (one TMA
      // issue stream cannot keep up with a converged MMA warp).
      const uint32_t lead = lane == 0 ? 1u : 0u;
      const int nprod = split_issuer ? 2 : 3;
      const int role = warp == 0 ? 0 : (warp == kProducer2Warp ? 1 : 2);
      int rr = 0;  // seq % nprod
      bool dep_done = false;  // grid_dependency_wait() passed
      int stage = 0;
      uint32_t phase = 0;
      long long seq = 0;
      long long last_issued = -1;
      bool ok = true;
      const uint32_t stage_tx = a_bytes + (p.b_resident ? 0u : b_bytes);
      bool first_tile = true;  // a resident filter is loaded k-block by k-block with it
      if (p.window) {
        // One tiled box of input rows (with halo) per channel block; the
        // first tile also brings every tap's filter block of that channel block.
        const uint32_t box_bytes = static_cast<uint32_t>(p.win_pitch * p.win_box_rows) * sw;
        const int taps = p.win_R * p.win_S;
        for (int t = tile0; t < p.total_tiles && ok; t += tile_step) {
          int n_img, oy0;
          window_origin(p, t, n_img, oy0);
          for (int cb = 0; cb < p.c_blocks; ++cb, ++seq) {
            if (rr == role) {
              if (!__all_sync(0xFFFFFFFFu,
                              mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag,
                                                status, kStatusProducerTimeout, limit,
                                                p.wait_hint_ns))) {
                ok = false;
                break;
              }
              if (!dep_done) {
                grid_dependency_wait();
                dep_done = true;
              }
              last_issued = seq;
              if (!(p.fault_mode == 1 && blockIdx.x == 0 && seq == 0)) {
                const uint32_t fb = smem_u32(&full[stage]);
                // The first tile also brings every tap's filter block of this
                // channel block, on the same barrier.  (Each block on its own
                // barrier, so that tap 0's MMAs could start earlier, measured
                // slower: the ResNet 3x3 conv ran 19.0 against 16.7 us.)
                mbar_arrive_expect_tx_if(lead, fb, box_bytes + (first_tile ? b_bytes * taps : 0u));
                tma_load_4d_if(lead, smem_u32(a_ring + stage * p.win_stage_bytes), &p.map_a[0], fb,
                               cb * p.bk, -p.win_pad_w, oy0 - p.win_pad_h, n_img);
                if (first_tile)
                  for (int tap = 0; tap < taps; ++tap)
                    tma_load_3d_if(lead, smem_u32(b_res + (tap * p.c_blocks + cb) * b_bytes),
                                   &p.map_b, fb, tap * p.c_in + cb * p.bk, 0, 0);
              }
            }
            if (++rr == nprod) rr = 0;
            if (++stage == stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          first_tile = false;
        }
      }
      // A pair's rank 0 arms its stage barrier for both CTAs' bytes; rank 1's
      // copies count on rank 0's barrier.
      const uint32_t arm_tx = kPair ? 2u * stage_tx : stage_tx;
      WorkWalk walk = work_begin<kStreamK>(p, tile0, tile_step);
      Work wk;
      while (!p.window && ok && work_next<kStreamK>(p, walk, wk)) {
        const int t = wk.tile;
        TileInfo ti = wk.ti;
        ti.m0 += m_off;
        const int ph = ti.phase;
        int n_img, j, i;
        grid_pos(p, ph, ti.m0, n_img, j, i);
        const int h0 = p.base_h[ph] + j * p.step_h;
        const int w0 = p.base_w[ph] + i * p.step_w;
        const int tw = p.taps_w[ph];
        const CUtensorMap* amap = &p.map_a[ph];
        // Filter slot: the stride phase, or the channel group.
        const int bz = p.groups > 1 ? ti.group : p.b_index[ph];
        const int c_base = ti.group * p.c_group;  // first input channel of the group
        // The work item's first k-block: channel block cb of tap (uh, uw).
        int cb = 0, uw = 0, uh = 0;
        int bk_k = 0;  // k coordinate of this k-block in the packed filter: tap*C_in + cb*bk
        if (kStreamK && wk.kb0 != 0) {
          const int tap = wk.kb0 / p.c_blocks;
          cb = wk.kb0 - tap * p.c_blocks;
          uh = tap / tw;
          uw = tap - uh * tw;
          bk_k = tap * p.c_in + cb * p.bk;
        }
        const bool load_res = p.b_resident && first_tile;
        first_tile = false;
        // This CTA's next tile: its A boxes are prefetched into L2 alongside
        // this tile's loads, so they come from L2 rather than HBM later.
        const int tn = t + tile_step;
        const bool pf = p.l2_prefetch && tn < p.total_tiles;
        int pf_n = 0, pf_h0 = 0, pf_w0 = 0;
        const CUtensorMap* pf_map = amap;
        if (pf) {
          TileInfo tin = decode_tile(p, tn);
          tin.m0 += m_off;
          int pj, pi;
          grid_pos(p, tin.phase, tin.m0, pf_n, pj, pi);
          pf_h0 = p.base_h[tin.phase] + pj * p.step_h;
          pf_w0 = p.base_w[tin.phase] + pi * p.step_w;
          pf_map = &p.map_a[tin.phase];
          if (tin.kblocks != ti.kblocks || tin.n0 != 0 || tin.m0 == ti.m0 || tin.group != ti.group)
            pf_n = -1;  // skip
        }
        for (int kb = wk.kb0; kb < wk.kb1; ++kb, ++seq) {
          if (rr == role) {
            if (!__all_sync(0xFFFFFFFFu,
                            mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag,
                                              status, kStatusProducerTimeout, limit,
                                              p.wait_hint_ns, kPair))) {
              ok = false;
              break;
            }
            if (!dep_done) {
              grid_dependency_wait();
              dep_done = true;
            }
            last_issued = seq;
            if (kPair && p.fault_mode == 1 && tile0 == 0 && seq == 0) {
              // (Test hook: both CTAs of cluster 0 leave their first stage
              // un-armed and unloaded, so nothing of it is ever in flight.)
            } else if (kPair) {
              const uint32_t fb = smem_u32(&full[stage]);
              const int n_b = ti.n0 + static_cast<int>(rank) * (p.bn / 2);
              if (rank == 0) {
                mbar_arrive_expect_tx_if(lead, fb, arm_tx);
                tma_load_im2col_4d_if(lead, smem_u32(a_ring + stage * a_bytes), amap, fb,
                                      c_base + cb * p.bk, w0, h0, n_img,
                                      static_cast<uint16_t>(uw * p.dil_w),
                                      static_cast<uint16_t>(uh * p.dil_h));
                tma_load_3d_if(lead, smem_u32(b_ring + stage * b_bytes), &p.map_b, fb, bk_k, n_b,
                               bz);
              } else {
                const uint32_t fb0 = map_to_rank(fb, 0);
                tma_load_im2col_4d_pair_if(lead, smem_u32(a_ring + stage * a_bytes), amap, fb0,
                                           c_base + cb * p.bk, w0, h0, n_img,
                                           static_cast<uint16_t>(uw * p.dil_w),
                                           static_cast<uint16_t>(uh * p.dil_h));
                tma_load_3d_pair_if(lead, smem_u32(b_ring + stage * b_bytes), &p.map_b, fb0, bk_k,
                                    n_b, bz);
              }
            } else if (!(p.fault_mode == 1 && blockIdx.x == 0 && seq == 0)) {
              // (fault_mode 1, a test hook: CTA 0 leaves its first stage un-armed.)
              const uint32_t fb = smem_u32(&full[stage]);
              mbar_arrive_expect_tx_if(lead, fb, stage_tx + (load_res ? b_bytes : 0u));
              tma_load_im2col_4d_if(lead, smem_u32(a_ring + stage * a_bytes), amap, fb,
                                    c_base + cb * p.bk, w0, h0, n_img,
                                    static_cast<uint16_t>(uw * p.dil_w),
                                    static_cast<uint16_t>(uh * p.dil_h));
              if (!p.b_resident)
                tma_load_3d_if(lead, smem_u32(b_ring + stage * b_bytes), &p.map_b, fb, bk_k, ti.n0,
                               bz);
              else if (load_res)
                tma_load_3d_if(lead, smem_u32(b_res + kb * b_bytes), &p.map_b, fb, bk_k, 0, bz);
            }
            if (pf && pf_n >= 0)
              tma_prefetch_im2col_4d_if(lead, pf_map, c_base + cb * p.bk, pf_w0, pf_h0, pf_n,
                                        static_cast<uint16_t>(uw * p.dil_w),
                                        static_cast<uint16_t>(uh * p.dil_h));
          }
          if (++rr == nprod) rr = 0;
          if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
          }
          bk_k += p.bk;
          if (++cb == p.c_blocks) {
            cb = 0;
            bk_k += p.c_tail;  // the last block of a tap may reach past C_in: realign
            if (++uw == tw) {
              uw = 0;
              ++uh;
            }
          }
        }
      }
      if (!ok && rank == 0) {
        // Let every copy this producer still has in flight land before exiting.
        // (A pair's rank-0 barriers count rank 1's copies too.)
        for (long long q = last_issued - stages + 1; q <= last_issued; ++q)
          if (q >= 0 && static_cast<int>(q % nprod) == role)
            mbar_wait_drain(smem_u32(&full[q % stages]), static_cast<uint32_t>((q / stages) & 1),
                            limit / 8 + 1);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == kProducer3Warp) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues; with mma_split (two 128-row halves, no gather loader,
    // no pair) warp 11 issues the second half's MMAs beside it.  Each issuer
    // is a converged warp with one elected lane per MMA: a lone lane of a
    // diverged warp issued one MMA every ~100 cycles (187 with a barrier
    // wait and commit per 4), a converged warp keeps the tensor core busy
    // (64 cycles per N = 128 MMA), but its per-k-block wait and commit still
    // cost ~90 cycles, which the second warp hides for N <= 128.  (In a pair
    // only rank 0 issues.)
    if (rank == 0) {  // the whole warp: one elected lane issues each MMA
      bool ok;
      const int ks = static_cast<int>(sw / 32);
      const int half = p.mma_split ? (warp == 1 ? 0 : 1) : -1;
      uint64_t* my_drain = warp == 1 ? drain : drain2;
      if (!kPair && p.window) {
        ok = (p.m_halves == 2 && half < 0)
                 ? mma_role_window<kKind, 4, 2>(p, tmem_base, a_ring, b_res, full, empty, tfull,
                                                tempty, half, abort_flag, status, limit, tile0,
                                                tile_step)
                 : mma_role_window<kKind, 4, 1>(p, tmem_base, a_ring, b_res, full, empty, tfull,
                                                tempty, half, abort_flag, status, limit, tile0,
                                                tile_step);
        if (!ok) {
          mma_commit_warp(smem_u32(my_drain));
          mbar_wait_drain(smem_u32(my_drain), 0, limit / 8 + 1);
        }
      } else {
#define CONV_MMA_ROLE(KS, MH)                                                                   \
  mma_role<kKind, KS, MH, kPair, kStreamK>(p, tmem_base, a_ring, b_ring, b_res, full, empty,       \
                                           tfull, tempty, half, abort_flag, status, limit, tile0,  \
                                           tile_step)
      if (!kPair && p.m_halves == 2 && half < 0)
        ok = ks == 4 ? CONV_MMA_ROLE(4, 2) : (ks == 2 ? CONV_MMA_ROLE(2, 2) : CONV_MMA_ROLE(1, 2));
      else
        ok = ks == 4 ? CONV_MMA_ROLE(4, 1) : (ks == 2 ? CONV_MMA_ROLE(2, 1) : CONV_MMA_ROLE(1, 1));
#undef CONV_MMA_ROLE
      if (!ok) {
        // Every MMA already issued must finish before TMEM is released.
        if (kPair)
          mma_commit_pair_warp(smem_u32(my_drain));
        else
          mma_commit_warp(smem_u32(my_drain));
        mbar_wait_drain(smem_u32(my_drain), 0, limit / 8 + 1);
      }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Two warpgroups (warps 2-5 and 6-9).  Each warp reads the TMEM lane
    // quarter its warp index allows; group g takes the work items q % 2 == g
    // of every tile (item = one 128-row half x one chunk of cw columns).
    const int grp = (warp - 2) / 4;
    const int quarter = warp & 3;  // TMEM lanes this warp may read: [32*quarter, 32*quarter+32)
    const int row = quarter * 32 + lane;
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    const bool leader = (warp == 2 + 4 * grp) && lane == 0;
    const uint32_t bar_id = 1 + grp;
    int it = 0;
    // (A pair's rank 1 takes rows 128..255 of each tile: m_off.)
    // Hands accumulator buffer `acc` back to the MMA issuer (lane 0, after
    // tcgen05.fence::before_thread_sync and __syncwarp).
    auto release_acc = [&](int acc) {
      if (kPair && rank != 0)
        mbar_arrive_remote(map_to_rank(smem_u32(&tempty[acc]), 0));
      else
        mbar_arrive(smem_u32(&tempty[acc]));
    };
    const int ew = warp - 2;  // epilogue warp index: its stream-K flag
    if (p.epi_mode != 0) {
      const uint32_t row_bytes = static_cast<uint32_t>(p.cw) * 2;
      const uint32_t chunk_bytes = kBM * row_bytes;
      const int nchunks = p.bn / p.cw;
      const int nitems = nchunks * p.m_halves;
      const uint32_t src_tile_bytes = p.src_chunk_bytes * nitems;
      const bool in_place = p.has_residual != 0;  // outputs overwrite the source chunk, stored from there
      uint8_t* stg_grp = stg_base + grp * (p.stg_bufs * chunk_bytes);
      int store_seq = 0;
      int src_issued[2] = {0, 0};  // source loads issued per buffer (leader only)
      if (!in_place) {
        // While the first tile's MMAs run, pass zeros through this
        // epilogue's row code into the (still unused) staging buffer: its
        // instructions are then cached when the first accumulator lands.  A
        // conv of one tile per CTA otherwise fetches them cold at its end.
        uint32_t zeros[64];
#pragma unroll
        for (int k = 0; k < 64; ++k) zeros[k] = 0u;
        if (row < p.valid_rows) {
          if (p.cw == 64)
            process_row_act<OutT, 64>(zeros, stg_grp, static_cast<uint32_t>(row), p.beta,
                                      p.epilogue, false);
          else if (p.cw == 32)
            process_row_act<OutT, 32>(zeros, stg_grp, static_cast<uint32_t>(row), p.beta,
                                      p.epilogue, false);
          else
            process_row_act<OutT, 16>(zeros, stg_grp, static_cast<uint32_t>(row), p.beta,
                                      p.epilogue, false);
        }
        named_barrier(bar_id, 128);
      }
      if (!kGather) grid_dependency_wait();  // (the pass above touched shared memory only)
      // Work items in order; the source prefetch peeks at the next one.
      WorkWalk walk = work_begin<kStreamK>(p, tile0, tile_step);
      Work cur{};
      bool have = work_next<kStreamK>(p, walk, cur);
      if (p.has_residual && leader && have) {
        TileInfo t0i = cur.ti;
        t0i.m0 += m_off;
        issue_source_items(p, t0i, src_base, smem_u32(&src_full[grp]), grp);
        ++src_issued[0];
      }
      for (; have; ++it, have = work_next<kStreamK>(p, walk, cur)) {
        TileInfo ti = cur.ti;
        ti.m0 += m_off;
        const int role = kStreamK ? work_role(cur) : kSkWhole;
        const int acc = it & 1;
        const int sbuf = p.src_bufs == 2 ? acc : 0;
        if (p.has_residual && leader && p.src_bufs == 2) {
          WorkWalk ahead = walk;
          Work nx;
          if (work_next<kStreamK>(p, ahead, nx)) {
            nx.ti.m0 += m_off;
            // The other buffer last held item it-1, whose stores must have read it.
            bulk_wait_read_all();
            issue_source_items(p, nx.ti, src_base + (acc ^ 1) * src_tile_bytes,
                               smem_u32(&src_full[2 * (acc ^ 1) + grp]), grp);
            ++src_issued[acc ^ 1];
          }
        }
        bool ok = mbar_wait_bounded(smem_u32(&tfull[acc]), static_cast<uint32_t>((it >> 1) & 1),
                                    abort_flag, status, kStatusEpilogueTimeout, limit,
                                    p.wait_hint_ns, kPair);
        if (ok && p.has_residual && grp < nitems) {
          const uint32_t par = static_cast<uint32_t>(p.src_bufs == 2 ? (it >> 1) & 1 : it & 1);
          ok = mbar_wait_bounded(smem_u32(&src_full[2 * sbuf + grp]), par, abort_flag, status,
                                 kStatusEpilogueTimeout, limit, p.wait_hint_ns);
        }
        if (ok && role == kSkFinish)
          ok = sk_wait_partials(p, cur, ew, tile_step, abort_flag, limit);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
        tc_fence_after();
        uint8_t* src_tile = src_base + sbuf * src_tile_bytes;
        const uint32_t tacc = tmem_base + lane_field + static_cast<uint32_t>(acc) * p.acc_stride;
        if (grp >= nitems) {  // nothing for this group in this tile
          tc_fence_before();
          __syncwarp();
          if (lane == 0) release_acc(acc);
        }
        for (int q = grp; q < nitems; q += kEpilogueGroups) {
          const int h = q / nchunks;
          const int c = q - h * nchunks;
          const int mh = ti.m0 + h * kBM;
          uint32_t v[64];
          // 16-column groups of this chunk within the tile's partial slot.
          const int g0 = h * (p.bn / 16) + c * (p.cw / 16);
          if (role == kSkFinish) {
            // The later k-blocks' partials first, then this CTA's accumulators.
            sk_sum_partials<4>(p, cur, g0, p.cw / 16, row, tile_step, v);
            tmem_add_groups<4>(tacc + static_cast<uint32_t>(h * p.bn + c * p.cw), p.cw / 16, v);
          } else if (ti.kblocks > 0) {
            const uint32_t taddr = tacc + static_cast<uint32_t>(h * p.bn + c * p.cw);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (k < p.cw / 16)
                tmem_ld_32x32b_x16(taddr + static_cast<uint32_t>(k * 16),
                                   *reinterpret_cast<uint32_t(*)[16]>(&v[k * 16]));
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (k < p.cw / 16)
                tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[16]>(&v[k * 16]));
          } else {
#pragma unroll
            for (int k = 0; k < 64; ++k) v[k] = 0u;
          }
          if (q + kEpilogueGroups >= nitems) {
            // This group's last TMEM read of the tile: hand the buffer back early.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release_acc(acc);
          }
          if (role == kSkPartial) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (k < p.cw / 16)
                sk_store16(p, static_cast<int>(blockIdx.x), g0 + k, row, &v[k * 16]);
            continue;  // no output from a partial
          }
          uint8_t* buf;
          if (in_place) {
            buf = src_tile + q * p.src_chunk_bytes;
          } else {
            buf = stg_grp + (p.stg_bufs == 2 ? (store_seq & 1) : 0) * chunk_bytes;
            if (leader) {
              if (p.stg_bufs == 2)
                bulk_wait_read_le1();
              else
                bulk_wait_read_all();
            }
            named_barrier(bar_id, 128);
          }
          // Lanes past valid_rows (the junk rows of a row-window half) are
          // never stored: they neither read nor write the buffer.
          if (row < p.valid_rows) {
            if (p.cw == 64)
              process_row_act<OutT, 64>(v, buf, static_cast<uint32_t>(row), p.beta, p.epilogue,
                                        in_place);
            else if (p.cw == 32)
              process_row_act<OutT, 32>(v, buf, static_cast<uint32_t>(row), p.beta, p.epilogue,
                                        in_place);
            else
              process_row_act<OutT, 16>(v, buf, static_cast<uint32_t>(row), p.beta, p.epilogue,
                                        in_place);
          }
          fence_proxy_async_shared();
          named_barrier(bar_id, 128);
          if (leader) {
            if (p.epi_mode == 1) {
              tma_store_3d(&p.map_out[ti.phase], smem_u32(buf), ti.n0 + c * p.cw, ti.group, mh);
            } else if (p.epi_mode == 3) {
              int n_img, oy0;
              window_origin(p, ti.m0, n_img, oy0);
              tma_store_4d(&p.map_out[0], smem_u32(buf), ti.n0 + c * p.cw, 0,
                           oy0 + h * p.win_rows, n_img);
            } else {
              int n_img, gj, gi;
              grid_pos(p, ti.phase, mh, n_img, gj, gi);
              tma_store_4d(&p.map_out[ti.phase], smem_u32(buf), ti.n0 + c * p.cw, gi, gj, n_img);
            }
            bulk_commit_group();
          }
          ++store_seq;
        }
        if (role == kSkPartial) sk_publish(p, static_cast<int>(blockIdx.x), ew, lane);
        if (p.has_residual && leader && p.src_bufs == 1) {
          WorkWalk ahead = walk;
          Work nx;
          if (work_next<kStreamK>(p, ahead, nx)) {
            nx.ti.m0 += m_off;
            // Single source buffer: fetch the next item's source once this
            // item's stores (which read it) are done reading.
            bulk_wait_read_all();
            issue_source_items(p, nx.ti, src_base, smem_u32(&src_full[grp]), grp);
            ++src_issued[0];
          }
        }
      }
      // Before the CTA exits, its stores must have read their shared-memory
      // sources; their global writes complete with the grid (a dependent
      // kernel's griddepcontrol.wait sees them).
      if (leader) bulk_wait_read_all();
      // On abort, source loads issued for tiles never processed must land
      // before the CTA exits: wait for the latest phase of each buffer.
      if (leader && p.has_residual && *abort_flag && grp < nitems) {
        for (int b = 0; b < 2; ++b)
          if (src_issued[b] > 0)
            mbar_wait_drain(smem_u32(&src_full[2 * b + grp]),
                            static_cast<uint32_t>((src_issued[b] - 1) & 1), limit / 8 + 1);
      }
    } else {
      WorkWalk walk = work_begin<kStreamK>(p, tile0, tile_step);
      Work wk;
      for (; work_next<kStreamK>(p, walk, wk); ++it) {
        TileInfo ti = wk.ti;
        ti.m0 += m_off;
        const int role = kStreamK ? work_role(wk) : kSkWhole;
        const int acc = it & 1;
        bool ok = mbar_wait_bounded(smem_u32(&tfull[acc]), static_cast<uint32_t>((it >> 1) & 1),
                                    abort_flag, status, kStatusEpilogueTimeout, limit,
                                    p.wait_hint_ns, kPair);
        if (ok && role == kSkFinish)
          ok = sk_wait_partials(p, wk, ew, tile_step, abort_flag, limit);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
        tc_fence_after();
        const int ph = ti.phase;
        // Group g takes the 16-column chunks j with j % 2 == g of every half.
        for (int h = 0; h < p.m_halves; ++h) {
          const int m = ti.m0 + h * kBM + row;
          const bool valid = m < p.rows[ph];
          long long out_off = 0;
          if (valid) {
            int n_img, j, i;
            grid_pos(p, ph, m, n_img, j, i);
            const long long oy = static_cast<long long>(p.out_step_h) * j + p.out_off_h[ph];
            const long long ox = static_cast<long long>(p.out_step_w) * i + p.out_off_w[ph];
            out_off = ((static_cast<long long>(n_img) * p.Ho + oy) * p.Wo + ox) * p.Cout +
                      static_cast<long long>(ti.group) * p.f_group;
          }
          const uint32_t taddr = tmem_base + lane_field + static_cast<uint32_t>(acc) * p.acc_stride +
                                 static_cast<uint32_t>(h * p.bn);
          for (int c0 = grp * 16; c0 < p.bn; c0 += 16 * kEpilogueGroups) {
            uint32_t v[16];
            const int g = h * (p.bn / 16) + c0 / 16;  // 16-column group within the tile
            if (role == kSkFinish) {
              sk_sum_partials<1>(p, wk, g, 1, row, tile_step, v);
              tmem_add_groups<1>(taddr + static_cast<uint32_t>(c0), 1, v);
            } else if (ti.kblocks > 0) {
              tmem_ld_32x32b_x16(taddr + static_cast<uint32_t>(c0), v);
              tmem_wait_ld_regs(v);
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = 0u;
            }
            if (role == kSkPartial) {
              sk_store16(p, static_cast<int>(blockIdx.x), g, row, v);
              continue;
            }
            if (p.seg_store) {  // (one 16-column chunk: group 0's warps only)
              epilogue_seg_warp<OutT>(p, ti.m0 + h * kBM + quarter * 32, lane, v,
                                      smem + p.off_seg + quarter * 2 * p.seg_slot_bytes);
              continue;
            }
            // Columns past the group's (or the conv's) last output channel are not stored.
            const int ch = ti.n0 + c0;
            if (valid && ch < p.f_group) {
              const int nvalid = p.f_group - ch < 16 ? p.f_group - ch : 16;
              epilogue_16_direct<OutT>(p, out_off + ch, v, nvalid);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(acc);
        if (role == kSkPartial) sk_publish(p, static_cast<int>(blockIdx.x), ew, lane);
      }
    }
  }

  if (warp >= 2 && warp < 2 + kEpilogueWarps) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(epi_done));
  }
  __syncthreads();
  // Neither CTA of a pair exits (or frees TMEM) while the other may still
  // signal one of its barriers or read its TMEM.
  if (kPair) cluster_sync();
  if (warp == 1) {
    // TMEM is released only once every epilogue warp has signalled that its
    // last tcgen05.ld is complete.
    if (lane == 0) mbar_wait_drain(smem_u32(epi_done), 0, limit);
    __syncwarp();
    tc_fence_after();
    if (kPair)
      tmem_dealloc_pair(tmem_base, p.tmem_cols);
    else
      tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace convgb300
