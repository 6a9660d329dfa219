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
  // 3x3 depthwise tiles: tiled {C, W, H, N} over the input, box {64, dw_cols +
  // 2, kDwRows + 2, 1} (encoded only for that kernel).
  CUtensorMap map_x;
  unsigned int* status;     // workspace status word (bounded waits)
  long long timeout_cycles;
  int fault_mode;           // test hook: 1 = CTA 0 never loads its first depthwise tile
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
  int dw_cols;             // output columns per depthwise tile (dw_tile_cols)
};

size_t direct_smem_bytes(int r, int s, int c_group);

// True when the 3x3 depthwise tile kernel runs this conv (its input map must
// then be encoded): 16-bit inputs, multiplier 1, stride 1, dilation 1, C % 8 == 0.
bool direct_uses_dw_tiles(int in_dtype, const DirectParams& p);
constexpr int kDwRows = 16;   // output rows per depthwise tile
// Output columns per depthwise tile: 28 or 32, whichever leaves fewer unused
// columns in the last tile of a row (32 on a tie).
int dw_tile_cols(int wo);

// in_dtype: 0 bf16, 1 f16, 2 e4m3 (bf16 out).
cudaError_t launch_conv_direct(int in_dtype, bool out_bf16, const DirectParams& p, int num_sms,
                               cudaStream_t stream);

// Row-tap kernel for forward convs with few output channels (S * C_out <= 32,
// e.g. an RGB head): the filter taps along S and the output channels share
// the MMA's N dimension, so each input-row segment is multiplied once by the
// filter rows of all R taps and its products accumulate, in tensor memory,
// into the R output rows it touches; the epilogue sums the S taps across
// neighbouring pixels.  Stride 1, dilation 1, one channel group.
constexpr int kRowTapMaxBand = 24;  // output rows per tile (upper bound)

struct RowTapParams {  // aligned like CUtensorMap
  CUtensorMap map_x;   // tiled {C_in, W, H, N}, box {bk, 128, 1, 1}, 128-B swizzle
  CUtensorMap map_w;   // tiled {C_in, S, R, F} over the packed filter, box {bk, S, 1, F}
  int N, H, W, Ho, Wo, F, R, S;
  int pad_h, pad_w;
  int c_blocks;        // 128-byte channel blocks of C_in (the last one zero-filled past C_in)
  int g16;             // TMEM columns (B rows) per filter row r: S*F rounded up to 16
  int band;            // output rows per tile
  int seg_w;           // output columns per tile: 128 - (S - 1)
  int n_seg, n_band, total_tiles;
  int stages;
  int blocks_per_stage;  // channel blocks of one input row segment per A stage (1 or c_blocks)
  uint32_t idesc_all;  // N = R * g16
  uint32_t idesc_one;  // N = g16
  uint32_t idesc_rest; // N = (R - 1) * g16 (R > 1)
  uint32_t cols_per_buf, tmem_cols;
  uint32_t off_b, off_part, off_bar;  // shared-memory offsets (A ring at 0)
  uint32_t off_stage;  // output and source row-segment stages, two epilogue groups each
  int stage_bytes;     // bytes per segment stage: 128 * F * elt + 16, rounded to 16
  int has_residual, epilogue;
  float beta;
  const void* src;
  void* out;
  unsigned int* status;
  long long timeout_cycles;
  int fault_mode;      // test hook: 1 = CTA 0 leaves its first A stage un-armed
};

// Launches the row-tap kernel; in_dtype: 0 bf16, 1 f16, 2 e4m3 (bf16 out).
cudaError_t launch_conv_rowtap(int in_dtype, bool out_bf16, const RowTapParams& p, int grid,
                               size_t smem_bytes, cudaStream_t stream);

// The CTA-pair instances (cta_group::2; their own translation unit).
cudaError_t launch_conv_igemm_pair(int kind, bool out_bf16, const ConvKernelParams& p, int grid,
                                   size_t smem_bytes, cudaStream_t stream);

// The stream-K instances (TMA loaders, single CTAs; their own translation unit).
cudaError_t launch_conv_igemm_streamk(int kind, bool out_bf16, const ConvKernelParams& p, int grid,
                                      size_t smem_bytes, cudaStream_t stream);

// The gather-loader instances (their own translation unit).
cudaError_t launch_conv_igemm_gather(int kind, bool out_bf16, const ConvKernelParams& p, int grid,
                                     size_t smem_bytes, cudaStream_t stream);

// One TMA im2col load into shared memory, copied out un-swizzled (test hook).
cudaError_t launch_im2col_probe(const CUtensorMap& map, int c, int w, int h, int n, int off_w,
                                int off_h, uint32_t row_bytes, void* out, unsigned int* status,
                                long long limit_cycles, cudaStream_t stream);

}  // namespace convgb300
