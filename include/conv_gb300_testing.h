/*
 * conv_gb300_testing.h -- test hooks exported by libconvgb300.so.
 *
 * These entry points are not part of the convolution API.  They exist so the
 * test suite can (a) look at exactly what one TMA im2col load of the
 * convolution kernel places in shared memory, and (b) exercise the kernels'
 * bounded-wait failure path without faulting or hanging a GPU.
 */
#ifndef CONV_GB300_TESTING_H
#define CONV_GB300_TESTING_H

#include <stddef.h>

#include "conv_gb300.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Make the next launches of the convolution kernel misbehave on purpose, in
 * a way that only exercises its bounded waits:
 *   mode 0: normal operation (the default);
 *   mode 1: CTA 0's producer skips the arrive of its first k-block, so the
 *           MMA warp's wait on it can only end by running out of time (for
 *           CTA pairs: both CTAs of the first pair leave their first stage
 *           un-armed and unloaded);
 *   mode 2: stream-K launches never publish their partial tiles, so the CTAs
 *           that finish split tiles wait for them until the limit runs out.
 * timeout_ns sets the per-wait limit of subsequent launches (0 = default,
 * one second).  The kernel then records CONV_ERR_DEVICE_TIMEOUT in the
 * workspace status word, releases its tensor memory and returns; nothing
 * traps.  Process-wide; not thread-safe. */
void conv_testing_set_wait_fault(int mode, unsigned long long timeout_ns);

/* Run ONE TMA im2col load exactly as the forward convolution kernel would
 * issue it for the output tile starting at GEMM row m0, filter tap (tap_r,
 * tap_s) and input-channel block starting at c0, and copy the loaded
 * 128 x bk tile (un-swizzled, row = pixel, bk channels per row) to
 * out_tile (device, 128 * bk * sizeof(dtype) bytes).  bk is what the
 * convolution would use for this c_in and dtype; it is returned in *bk_out.
 * Shapes and gates as conv2d_fwd; channel counts served by the gather loader
 * (no im2col map) return CONV_ERR_NOT_SUPPORTED.  Synchronous. */
conv_status_t conv_testing_im2col_tile(const void* input, int n, int h, int w, int c_in,
                                       conv_dtype_t dtype, int r, int s, const int stride[2],
                                       const int symmetric_padding[2], int m0, int tap_r,
                                       int tap_s, int c0, void* out_tile, int* bk_out,
                                       void* status_workspace, void* stream);

/* The tile and shared-memory configuration the dispatcher picks for a
 * forward convolution through conv2d_fwd_packed with a workspace of
 * workspace_bytes: out[0] = bn (tile width along C_out), out[1] = bk
 * (channels per k-block), out[2] = pipeline stages, out[3] = dynamic shared
 * memory bytes, out[4] = total tiles, out[5] = grid size (CTAs), out[6] =
 * TMEM columns, out[7] = epilogue mode (0 direct stores, 1 TMA 2-D, 2 TMA
 * phase grid, 3 TMA row window), out[8] = filter resident in shared memory,
 * out[9] = residual source buffers, out[10] = output staging buffers,
 * out[11] = A loader (0 TMA im2col, 1 row window, 2 gather, 3 row-tap).  For
 * the row-tap kernel (few output channels: the filter taps along S and the
 * output channels share the MMA's N) out[0] = R * g16 (MMA width), out[9] =
 * 128-byte channel blocks per A stage (all of an input row segment's, or
 * one), out[10] = output rows per tile.  out[12] = 1 when CTA pairs (clusters of two CTAs
 * sharing 256-row tiles through cta_group::2 MMAs) run the conv.  out[13] = 1
 * when the stream-K schedule runs it.  Host-only. */
conv_status_t conv_testing_fwd_plan(int n, int h, int w, int c_in, conv_dtype_t dtype, int r,
                                    int s, int c_out, const int stride[2],
                                    const int symmetric_padding[2], int has_residual, int num_sms,
                                    size_t workspace_bytes, int out[14]);

/* Read the CONV_* tuning overrides from the environment again (the library
 * reads them once, on first use) and invalidate every cached prepared call.
 * For tests that change an override between calls; not to be called while
 * other threads are inside the library. */
void conv_testing_reload_tuning(void);

/* Process-wide counts of calls that found their prepared launch in the
 * library's cache (same entry point, arguments, device and tuning) and of
 * calls that had to plan and encode afresh.  Either pointer may be NULL. */
void conv_testing_cache_stats(unsigned long long* hits, unsigned long long* misses);

#ifdef __cplusplus
}
#endif

#endif /* CONV_GB300_TESTING_H */
