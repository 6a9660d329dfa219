/*
 * conv_gb300.h -- C ABI of libconvgb300.so: NHWC 2-D convolution as an
 * implicit GEMM on one NVIDIA GB300 GPU (sm_103a), plus transposed
 * convolution.  No torch types; plain pointers, sizes and a CUDA stream.
 *
 * Operations follow the Modular "nn/conv" kernel API pages:
 *  - "dispatch_amd_4wave_conv2d" (Parameters, Args, description): dtype
 *    gates, FCRS/RSCF filter (filter_is_fcrs), stride/dilation/symmetric
 *    padding/num_groups gates, D = Conv(A, B) + beta * source with an NHWC
 *    source of the output's shape, read only when has_residual is set, and an
 *    optional fused elementwise epilogue.
 *  - "dispatch_fused_im2col_conv2d_apple" (description): the im2col matrix
 *    (M = N*Ho*Wo, N = C_out, K = R*S*C_in) is gathered on the fly and never
 *    materialised; the filter is transposed once to a (C_out, K) NK matrix;
 *    small C_out (down to 1) runs on the matrix units through a masked edge
 *    tile.
 *  - "conv_transposed_gpu" (description, Args): transposed convolution (the
 *    backward-data pass of the forward convolution) over an NHWC input and an
 *    RSFC filter, with an optional elementwise epilogue.
 *
 * Conventions for every entry point:
 *  - Tensors are NHWC, dense, row-major, channels fastest.  All tensor
 *    pointers are DEVICE pointers, 16-byte aligned.
 *  - The caller owns all memory (input, filter, packed filter, output,
 *    source, workspace).  The library never allocates device memory at run
 *    time; it keeps host-side state (driver entry points, per-device
 *    attributes) and one static device array used only by conv2d_fwd_noalloc.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Outputs are valid once the stream has been synchronised.
 *  - Validation failures return before any launch and write nothing.
 *    Unsupported cases return CONV_ERR_NOT_SUPPORTED: there is no fallback.
 *  - Workspaces start with a CONV_STATUS_BYTES status region that the caller
 *    must zero once before first use (e.g. cudaMemsetAsync).  Kernels only OR
 *    error bits into it; conv_check_device_status() reads and clears it.
 */
#ifndef CONV_GB300_H
#define CONV_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CONV_OK = 0,
  CONV_ERR_INVALID_VALUE = 1,        /* null pointer, bad size, inconsistent shape */
  CONV_ERR_NOT_SUPPORTED = 2,        /* a gate failed (dtype, stride, padding, ...) */
  CONV_ERR_MISALIGNED = 3,           /* a tensor pointer is not 16-byte aligned */
  CONV_ERR_WORKSPACE_TOO_SMALL = 4,  /* workspace or packed-filter buffer too small */
  CONV_ERR_CUDA = 5,                 /* a CUDA runtime/driver call or launch failed */
  CONV_ERR_DEVICE_TIMEOUT = 6        /* a bounded wait inside a kernel ran out */
} conv_status_t;

typedef enum {
  CONV_DTYPE_BF16 = 0,
  CONV_DTYPE_F16 = 1,
  CONV_DTYPE_F8E4M3 = 2              /* OCP float8 e4m3 ("fn"), per-tensor scale 1 */
} conv_dtype_t;

typedef enum {
  CONV_EPI_NONE = 0,
  CONV_EPI_RELU = 1,                 /* max(v, 0) */
  CONV_EPI_SILU = 2                  /* v * sigmoid(v) */
} conv_epilogue_t;

#define CONV_STATUS_BYTES 256

/* Human-readable name of a status code (static string). */
const char* conv_status_string(conv_status_t status);

/* ------------------------------------------------------------------------
 * Filter packing ("dispatch_fused_im2col_conv2d_apple", description: the
 * filter is transposed once to the (C_out, K = R*S*C_in) NK matrix).
 *
 * Packed layout: packed[f][k], k = (r*S + s)*C_in + c, K-major, element type
 * = dtype.  For channel counts the gather loader serves (c_in * elt not a
 * multiple of 16 bytes, or under 32) each filter row r is one run of
 * S*C_in elements zero-padded to a multiple of 16 bytes:
 * packed[f][r*RP + s*C_in + c], RP = ceil(S*C_in*elt / 16) * 16 / elt.
 * For a grouped conv pack with c_in = C_in / num_groups (the filter's own
 * channel extent).
 * `filter` is FCRS [C_out][C_in][R][S] when filter_is_fcrs is
 * nonzero, else RSCF [R][S][C_in][C_out] ("dispatch_amd_4wave_conv2d",
 * Parameters: filter_is_fcrs).  Returns CONV_ERR_WORKSPACE_TOO_SMALL when
 * packed_bytes < conv2d_packed_filter_bytes(...).
 * ------------------------------------------------------------------------ */
size_t conv2d_packed_filter_bytes(int r, int s, int c_in, int c_out, conv_dtype_t dtype);

conv_status_t conv2d_pack_filter(const void* filter, int r, int s, int c_in, int c_out,
                                 int filter_is_fcrs, conv_dtype_t dtype, void* packed,
                                 size_t packed_bytes, void* stream);

/* Workspace for conv2d_fwd: the status region plus room for the packed
 * filter.  conv2d_fwd_packed needs only CONV_STATUS_BYTES. */
size_t conv2d_workspace_size(int r, int s, int c_in, int c_out, conv_dtype_t dtype);

/* Extra workspace that enables the stream-K schedule on the current device:
 * for convolutions whose output tiles fill less than one wave of the GPU's
 * SMs, every SM takes an equal share of the (tile, k-block) iterations, and
 * a tile split between CTAs is summed through fp32 partial tiles kept in the
 * workspace (one slot of up to 128 KB per SM, plus flags).  A workspace of
 * at least (conv2d_workspace_size or CONV_STATUS_BYTES for the packed entry
 * points, or conv_transposed_workspace_size) + this many bytes lets every
 * forward and transposed call use it where the planner expects a gain; a
 * smaller workspace only disables it.  Launches that use stream-K keep
 * their partials and flags in the workspace: launches that may overlap on
 * the GPU need separate workspaces.  Returns 0 when no device is current.
 * No counterpart on the pages: a schedule of the implicit GEMM's tiles. */
size_t conv_streamk_workspace_size(void);

/* ------------------------------------------------------------------------
 * Forward convolution ("dispatch_amd_4wave_conv2d", signature and Args):
 *   y[n][oy][ox][f] = act( sum_{r,s,c} x[n][oy*st - p + r][ox*st - p + s][c] * W(r,s,c,f)
 *                          + (has_residual ? beta * source[n][oy][ox][f] : 0) )
 * with x taken as zero outside the image, fp32 accumulation and one
 * round-to-nearest-even to out_dtype at the end.
 *
 *  input   [n][h][w][c_in], in_dtype
 *  filter  FCRS or RSCF (see conv2d_pack_filter), same dtype as the input
 *  output  [n][ho][wo][c_out], out_dtype = BF16 for F8E4M3 inputs, else in_dtype
 *  stride, dilation, symmetric_padding: {h, w} pairs
 *  source  [n][ho][wo][c_out], out_dtype; read only when has_residual != 0
 *          (then it must be non-NULL); beta is ignored otherwise
 *
 * Gates (CONV_ERR_NOT_SUPPORTED otherwise): in_dtype in {BF16, F16, F8E4M3};
 * out_dtype as above; stride (1,1) or (2,2); dilation d_h, d_w in [1, 32];
 * padding per axis 0 <= p_h <= d_h*(r-1), 0 <= p_w <= d_w*(s-1) (a TMA map
 * also needs the padded corners within [-128, 127]);
 * r, s <= 32.  Any c_in: channel rows of c_in * sizeof(in_dtype) bytes that
 * are a multiple of 16 and at least 32 are loaded by TMA; other channel
 * counts (e.g. c_in = 3) by the gather loader, which needs d_w == 1.
 * num_groups = G splits input and output channels into G equal groups
 * (output group g reads input group g; the filter is FCRS
 * [c_out][c_in/G][r][s] or RSCF [r][s][c_in/G][c_out]).  Groups of whole TMA
 * channel blocks ((c_in/G) * sizeof(in_dtype) a multiple of 16 bytes, at
 * least 32) run on the tensor cores; narrower ones (depthwise, channel
 * multipliers) on CUDA cores, which need r * s * (c_in/G) * 256 bytes of
 * shared memory <= 200 KB (else CONV_ERR_NOT_SUPPORTED); channels not
 * divisible by G are CONV_ERR_INVALID_VALUE.
 * CONV_ERR_INVALID_VALUE: null pointers, non-positive sizes, ho/wo not equal
 * to floor((h + 2p - (r-1) - 1)/stride) + 1, has_residual with NULL source,
 * unknown epilogue.
 * conv2d_fwd packs the filter into the workspace on every call;
 * conv2d_fwd_packed takes a filter already packed by conv2d_pack_filter.
 * Which kernel runs is the library's choice and does not change results
 * beyond fp32 summation order: the implicit GEMM (single CTAs, or CTA pairs
 * sharing 256-row tiles for wide, many-tile convs), the row-tap kernel for
 * stride-1 convs with s * c_out <= 32 (e.g. an RGB head), or the CUDA-core
 * kernels for narrow channel groups.
 * ------------------------------------------------------------------------ */
conv_status_t conv2d_fwd(const void* input, int n, int h, int w, int c_in, conv_dtype_t in_dtype,
                         const void* filter, int r, int s, int c_out, int filter_is_fcrs,
                         void* output, int ho, int wo, conv_dtype_t out_dtype,
                         const int stride[2], const int dilation[2],
                         const int symmetric_padding[2], int num_groups, int has_residual,
                         const void* source, float beta, conv_epilogue_t epilogue,
                         void* workspace, size_t workspace_bytes, void* stream);

conv_status_t conv2d_fwd_packed(const void* input, int n, int h, int w, int c_in,
                                conv_dtype_t in_dtype, const void* packed_filter, int r, int s,
                                int c_out, void* output, int ho, int wo, conv_dtype_t out_dtype,
                                const int stride[2], const int dilation[2],
                                const int symmetric_padding[2], int num_groups, int has_residual,
                                const void* source, float beta, conv_epilogue_t epilogue,
                                void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Transposed convolution ("conv_transposed_gpu", description and Args): the
 * backward-data pass of the forward convolution, written as the scatter
 *   Y[n][iy*st_h - p_h + r*d_h][ix*st_w - p_w + s*d_w][f] += x[n][iy][ix][c] * w[r][s][f][c]
 * over the RSFC filter w [R][S][C_out][C_in] (F = output channels, C = input
 * channels; the same memory as the RSCF filter of the forward convolution
 * whose backward-data this is), then y = act(Y + beta*source).
 * It is computed as stride_h*stride_w dense implicit GEMMs, one per output
 * phase (oy mod stride_h, ox mod stride_w), with no zero insertion: the taps
 * r of phase a are those with r*d = a + p (mod stride) (with g = gcd(d,
 * stride), every stride/g-th tap, or none), read at input dilation d/g.
 * Phases are launched four at a time (a stride of 3 or 4 takes several
 * launches of the same kernel; they write disjoint output pixels).
 *
 *  input  [n][h][w][c_in]; output [n][ho][wo][c_out]
 *  ho - ((h-1)*stride_h - 2*p_h + d_h*(r-1) + 1) must lie in [0, stride_h)
 *  (the extra rows play the role of an output padding), likewise wo.
 * Gates: dtypes as conv2d_fwd; stride_h, stride_w >= 1 with
 * stride_h*stride_w <= 16 (per-axis strides may differ); dilation 1..32 per
 * axis; 0 <= p <= d*(r-1) per axis; c_in * sizeof(in_dtype) a multiple of 16
 * bytes and at least 32 bytes; r, s <= 32.
 * conv_transposed packs the filter into the workspace on every call;
 * conv_transposed_packed takes the result of conv_transposed_pack_filter
 * (dilation 1) or conv_transposed_pack_filter_dilated, which must have been
 * called with the same stride, dilation and padding.
 * Packed layout: [stride_h*stride_w phases][c_out][K_max], phase (a, b) at
 * index a*stride_w + b, with k = (u*T_w + v)*c_in + c over the phase's taps.
 * The _dilated sizes and packing take the dilation; the others assume (1, 1).
 * ------------------------------------------------------------------------ */
size_t conv_transposed_packed_filter_bytes(int r, int s, int c_in, int c_out,
                                           const int stride[2], const int padding[2],
                                           conv_dtype_t dtype);

size_t conv_transposed_packed_filter_bytes_dilated(int r, int s, int c_in, int c_out,
                                                   const int stride[2], const int dilation[2],
                                                   const int padding[2], conv_dtype_t dtype);

size_t conv_transposed_workspace_size(int r, int s, int c_in, int c_out, const int stride[2],
                                      const int padding[2], conv_dtype_t dtype);

size_t conv_transposed_workspace_size_dilated(int r, int s, int c_in, int c_out,
                                              const int stride[2], const int dilation[2],
                                              const int padding[2], conv_dtype_t dtype);

conv_status_t conv_transposed_pack_filter(const void* filter_rsfc, int r, int s, int c_in,
                                          int c_out, const int stride[2], const int padding[2],
                                          conv_dtype_t dtype, void* packed, size_t packed_bytes,
                                          void* stream);

conv_status_t conv_transposed_pack_filter_dilated(const void* filter_rsfc, int r, int s, int c_in,
                                                  int c_out, const int stride[2],
                                                  const int dilation[2], const int padding[2],
                                                  conv_dtype_t dtype, void* packed,
                                                  size_t packed_bytes, void* stream);

conv_status_t conv_transposed(const void* input, int n, int h, int w, int c_in,
                              conv_dtype_t in_dtype, const void* filter_rsfc, int r, int s,
                              int c_out, void* output, int ho, int wo, conv_dtype_t out_dtype,
                              const int stride[2], const int dilation[2], const int padding[2],
                              int has_residual, const void* source, float beta,
                              conv_epilogue_t epilogue, void* workspace, size_t workspace_bytes,
                              void* stream);

conv_status_t conv_transposed_packed(const void* input, int n, int h, int w, int c_in,
                                     conv_dtype_t in_dtype, const void* packed_filter, int r,
                                     int s, int c_out, void* output, int ho, int wo,
                                     conv_dtype_t out_dtype, const int stride[2],
                                     const int dilation[2], const int padding[2], int has_residual,
                                     const void* source, float beta, conv_epilogue_t epilogue,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * conv2d_fwd without any device allocation.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory --
 * for example code running under a host framework that owns every device
 * allocation, or a real-time loop whose policy forbids cudaMalloc after
 * start-up -- and so cannot provide conv2d_fwd's workspace.
 *
 * Arguments, gates and results are those of conv2d_fwd called with a
 * workspace of exactly conv2d_workspace_size bytes (raw FCRS/RSCF filter; the
 * caller still passes input, filter, output and source): the same plan, so
 * the same output bits.  The packed
 * filter and the status word go to a library-owned scratch array of 8 MiB
 * (CONV_NOALLOC_SCRATCH_BYTES) that lives in device memory of every GPU that
 * loads the library until the process exits.  Filters whose packed size plus
 * CONV_STATUS_BYTES exceeds it return CONV_ERR_WORKSPACE_TOO_SMALL before
 * any CUDA call (the packed filter spans C_in / num_groups channels, so
 * grouped and depthwise filters are sized as conv2d_fwd sizes them; a
 * num_groups that does not divide C_in returns CONV_ERR_INVALID_VALUE).
 * Each call looks up the scratch address of the current device (a host-side
 * query); the first call on a device may also load the library's device
 * code there, so make that first call before any stream capture.  Every
 * call shares the one array: calls that overlap on the GPU (different
 * streams, or devices sharing nothing but the library) race, so serialise
 * them.  The status word is cleared at the start of each call; a bounded
 * wait that runs out inside the kernel leaves the output incomplete and is
 * not reported by this entry point (use conv2d_fwd with a workspace and
 * conv_check_device_status when that report is needed).
 * ------------------------------------------------------------------------ */
#define CONV_NOALLOC_SCRATCH_BYTES (8u << 20)

conv_status_t conv2d_fwd_noalloc(const void* input, int n, int h, int w, int c_in,
                                 conv_dtype_t in_dtype, const void* filter, int r, int s, int c_out,
                                 int filter_is_fcrs, void* output, int ho, int wo,
                                 conv_dtype_t out_dtype, const int stride[2], const int dilation[2],
                                 const int symmetric_padding[2], int num_groups, int has_residual,
                                 const void* source, float beta, conv_epilogue_t epilogue,
                                 void* stream);

/* ------------------------------------------------------------------------
 * Device-side failure report.  Synchronises `stream`, reads the status
 * region of `workspace`, clears it, and returns CONV_ERR_DEVICE_TIMEOUT if a
 * bounded wait inside a kernel ran out since the last check (the kernel then
 * stopped early, released its tensor memory and returned; its output is
 * incomplete), CONV_ERR_CUDA if the stream reports an error, else CONV_OK.
 * `detail` (may be NULL) receives the raw status bits.
 * ------------------------------------------------------------------------ */
conv_status_t conv_check_device_status(void* workspace, void* stream, unsigned int* detail);

#ifdef __cplusplus
}
#endif

#endif /* CONV_GB300_H */
