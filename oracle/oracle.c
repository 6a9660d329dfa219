/*
 * CPU oracle for NHWC 2-D convolution and transposed convolution.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * helper with the CUDA library; the two meet only through the seeded input
 * generator, which holds none of the method's arithmetic.
 *
 * Everything is computed in fp64, single-threaded, with plain loops in the
 * order the definitions are written.  No blocking, no reordering, no fusion.
 *
 * Definitions followed (pages of the Modular "nn/conv" kernel API docs):
 *
 *  - "dispatch_amd_4wave_conv2d", Parameters and Args: NHWC input, FCRS or
 *    RSCF filter (filter_is_fcrs), NHWC output, stride, dilation, symmetric
 *    padding; description: D = Conv(A, B) + beta * source, source NHWC with
 *    the output's shape and read only when has_residual is set.
 *  - "dispatch_fused_im2col_conv2d_apple", description: the GEMM view
 *    M = N*Ho*Wo, N = C_out, K = R*S*C_in; Args: [R,S,C_in,C_out] and
 *    [C_out,C_in,R,S] filter layouts.
 *  - "conv_transposed_gpu", description and Args: transposed convolution is
 *    the backward-data pass of the forward convolution, NHWC input, RSFC
 *    filter.  Read as the scatter form
 *        Y[n, iy*sh - ph + r*dh, ix*sw - pw + s*dw, f] += x[n,iy,ix,c] * w[r][s][f][c]
 *    with F the transposed conv's output channels and C its input channels.
 *
 * The oracle does not round its result to the output dtype: it returns the
 * exact fp64 value of act(conv + beta*source) over the decoded inputs.
 *
 * Readings where the pages are silent (stated once, used throughout):
 *  - num_groups = G splits input and output channels into G equal groups;
 *    output group g reads input group g only, and the filter's channel
 *    extent is C_in/G (FCRS [C_out][C_in/G][R][S], RSCF [R][S][C_in/G][C_out]);
 *  - residual before activation: y = act(conv + beta*source);
 *  - activations: none, ReLU = max(v, 0), SiLU = v / (1 + exp(-v));
 *  - output size of the forward conv: floor((H + 2p - d(R-1) - 1)/s) + 1.
 *
 * Every function here is pinned by CPU tests to something other than itself
 * (library convolutions, closed forms, adjoint identity, brute force).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

enum { ORACLE_BF16 = 0, ORACLE_F16 = 1, ORACLE_F8E4M3 = 2 };
enum { ORACLE_ACT_NONE = 0, ORACLE_ACT_RELU = 1, ORACLE_ACT_SILU = 2 };

/* ---------------------------------------------------------------------------
 * Bit-exact decoders, written from the formats' definitions.
 *   bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits.
 *   IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits.
 *   OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
 *   infinities; S.1111.111 is NaN; largest finite 448.
 * Exponent field 0 encodes subnormals (no implicit leading one).
 * ------------------------------------------------------------------------- */
static double decode_fields(uint32_t sign, uint32_t e, uint32_t m, int mbits, int bias)
{
    double mag;
    if (e == 0)
        mag = ldexp((double)m, 1 - bias - mbits);
    else
        mag = ldexp((double)((1u << mbits) | m), (int)e - bias - mbits);
    return sign ? -mag : mag;
}

double oracle_decode_one(uint32_t bits, int dtype)
{
    if (dtype == ORACLE_BF16) {
        uint32_t s = (bits >> 15) & 1u, e = (bits >> 7) & 0xFFu, m = bits & 0x7Fu;
        if (e == 0xFFu) return m ? NAN : (s ? -INFINITY : INFINITY);
        return decode_fields(s, e, m, 7, 127);
    }
    if (dtype == ORACLE_F16) {
        uint32_t s = (bits >> 15) & 1u, e = (bits >> 10) & 0x1Fu, m = bits & 0x3FFu;
        if (e == 0x1Fu) return m ? NAN : (s ? -INFINITY : INFINITY);
        return decode_fields(s, e, m, 10, 15);
    }
    if (dtype == ORACLE_F8E4M3) {
        uint32_t s = (bits >> 7) & 1u, e = (bits >> 3) & 0xFu, m = bits & 0x7u;
        if (e == 0xFu && m == 0x7u) return NAN;
        return decode_fields(s, e, m, 3, 7);
    }
    return NAN;
}

/* Decode `count` raw elements (2-byte little-endian words for bf16/f16, bytes
 * for fp8) into fp64.  Returns 0, or -1 for an unknown dtype. */
int oracle_decode(const void *src, int dtype, int64_t count, double *dst)
{
    if (dtype == ORACLE_BF16 || dtype == ORACLE_F16) {
        const uint16_t *p = (const uint16_t *)src;
        for (int64_t i = 0; i < count; ++i) dst[i] = oracle_decode_one(p[i], dtype);
        return 0;
    }
    if (dtype == ORACLE_F8E4M3) {
        const uint8_t *p = (const uint8_t *)src;
        for (int64_t i = 0; i < count; ++i) dst[i] = oracle_decode_one(p[i], dtype);
        return 0;
    }
    return -1;
}

double oracle_activation(double v, int act)
{
    if (act == ORACLE_ACT_RELU) return v > 0.0 ? v : 0.0;
    if (act == ORACLE_ACT_SILU) return v / (1.0 + exp(-v));
    return v;
}

/* Filter element W(r, s, c, f) of a forward filter stored FCRS or RSCF, C
 * being the filter's channel extent (C_in / groups). */
static double fwd_filter(const double *w, int64_t R, int64_t S, int64_t C, int64_t F,
                         int fcrs, int64_t r, int64_t s, int64_t c, int64_t f)
{
    if (fcrs) return w[((f * C + c) * R + r) * S + s];   /* [C_out][C_in/G][R][S] */
    return w[((r * S + s) * C + c) * F + f];             /* [R][S][C_in/G][C_out] */
}

/* One forward output element: the plain correlation sum over (r, s, c), input
 * taken as zero outside [0,H) x [0,W).  With G groups, output channel f
 * belongs to group g = f / (F/G) and sums only the input channels
 * g*(C/G) + c, c < C/G, against filter channel c. */
static double fwd_point(const double *x, int64_t H, int64_t W, int64_t C, int64_t G,
                        const double *w, int64_t R, int64_t S, int64_t F, int fcrs,
                        int sh, int sw, int ph, int pw, int dh, int dw,
                        int64_t n, int64_t oy, int64_t ox, int64_t f)
{
    const int64_t Cg = C / G, g = f / (F / G);
    double acc = 0.0;
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t s = 0; s < S; ++s) {
            int64_t iy = oy * sh - ph + r * dh;
            int64_t ix = ox * sw - pw + s * dw;
            if (iy < 0 || iy >= H || ix < 0 || ix >= W) continue;
            for (int64_t c = 0; c < Cg; ++c)
                acc += x[((n * H + iy) * W + ix) * C + g * Cg + c] *
                       fwd_filter(w, R, S, Cg, F, fcrs, r, s, c, f);
        }
    }
    return acc;
}

/* Full forward convolution, direct seven-loop form.
 * y[n][oy][ox][f] = act( sum_{r,s,c} X(n, oy*sh-ph+r*dh, ox*sw-pw+s*dw, c) * W(r,s,c,f)
 *                        + (has_res ? beta * src[n][oy][ox][f] : 0) ),
 * with G channel groups ("dispatch_amd_4wave_conv2d", Args: num_groups), read
 * in the usual way: C and F split into G equal groups, group g of the output
 * sees group g of the input only, and the filter's channel extent is C/G. */
int oracle_conv2d_fwd(const double *x, int64_t N, int64_t H, int64_t W, int64_t C, int64_t G,
                      const double *w, int64_t R, int64_t S, int64_t F, int fcrs,
                      int sh, int sw, int ph, int pw, int dh, int dw,
                      int64_t Ho, int64_t Wo,
                      int has_res, const double *src, double beta, int act,
                      double *y)
{
    if (N < 0 || H <= 0 || W <= 0 || C <= 0 || R <= 0 || S <= 0 || F <= 0) return -1;
    if (sh <= 0 || sw <= 0 || dh <= 0 || dw <= 0 || Ho < 0 || Wo < 0) return -1;
    if (G <= 0 || C % G != 0 || F % G != 0) return -1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t oy = 0; oy < Ho; ++oy)
            for (int64_t ox = 0; ox < Wo; ++ox)
                for (int64_t f = 0; f < F; ++f) {
                    int64_t o = ((n * Ho + oy) * Wo + ox) * F + f;
                    double v = fwd_point(x, H, W, C, G, w, R, S, F, fcrs, sh, sw, ph, pw, dh,
                                         dw, n, oy, ox, f);
                    if (has_res) v += beta * src[o];
                    y[o] = oracle_activation(v, act);
                }
    return 0;
}

/* The same definition evaluated only at the flat NHWC output indices `pts`
 * (each in [0, N*Ho*Wo*F)); out[i] is the value at pts[i]. */
int oracle_conv2d_fwd_points(const double *x, int64_t N, int64_t H, int64_t W, int64_t C,
                             int64_t G, const double *w, int64_t R, int64_t S, int64_t F,
                             int fcrs, int sh, int sw, int ph, int pw, int dh, int dw,
                             int64_t Ho, int64_t Wo,
                             int has_res, const double *src, double beta, int act,
                             const int64_t *pts, int64_t npts, double *out)
{
    if (G <= 0 || C % G != 0 || F % G != 0) return -1;
    int64_t total = N * Ho * Wo * F;
    for (int64_t i = 0; i < npts; ++i) {
        int64_t o = pts[i];
        if (o < 0 || o >= total) return -1;
        int64_t f = o % F, t = o / F;
        int64_t ox = t % Wo; t /= Wo;
        int64_t oy = t % Ho;
        int64_t n = t / Ho;
        double v = fwd_point(x, H, W, C, G, w, R, S, F, fcrs, sh, sw, ph, pw, dh, dw, n, oy, ox,
                             f);
        if (has_res) v += beta * src[o];
        out[i] = oracle_activation(v, act);
    }
    return 0;
}

/* Transposed convolution, direct scatter form over an RSFC filter
 * w[r][s][f][c] (F = output channels, C = input channels):
 *   Y[n, iy*sh-ph+r*dh, ix*sw-pw+s*dw, f] += x[n,iy,ix,c] * w[r][s][f][c]
 * for targets inside [0,Ho) x [0,Wo); then y = act(Y + beta*src). */
int oracle_conv_transposed(const double *x, int64_t N, int64_t H, int64_t W, int64_t C,
                           const double *w, int64_t R, int64_t S, int64_t F,
                           int sh, int sw, int ph, int pw, int dh, int dw,
                           int64_t Ho, int64_t Wo,
                           int has_res, const double *src, double beta, int act,
                           double *y)
{
    if (N < 0 || H <= 0 || W <= 0 || C <= 0 || R <= 0 || S <= 0 || F <= 0) return -1;
    if (sh <= 0 || sw <= 0 || dh <= 0 || dw <= 0 || Ho < 0 || Wo < 0) return -1;
    int64_t total = N * Ho * Wo * F;
    for (int64_t i = 0; i < total; ++i) y[i] = 0.0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t iy = 0; iy < H; ++iy)
            for (int64_t ix = 0; ix < W; ++ix)
                for (int64_t r = 0; r < R; ++r)
                    for (int64_t s = 0; s < S; ++s) {
                        int64_t oy = iy * sh - ph + r * dh;
                        int64_t ox = ix * sw - pw + s * dw;
                        if (oy < 0 || oy >= Ho || ox < 0 || ox >= Wo) continue;
                        for (int64_t c = 0; c < C; ++c) {
                            double xv = x[((n * H + iy) * W + ix) * C + c];
                            for (int64_t f = 0; f < F; ++f)
                                y[((n * Ho + oy) * Wo + ox) * F + f] +=
                                    xv * w[((r * S + s) * F + f) * C + c];
                        }
                    }
    for (int64_t o = 0; o < total; ++o) {
        double v = y[o];
        if (has_res) v += beta * src[o];
        y[o] = oracle_activation(v, act);
    }
    return 0;
}

/* The scatter definition evaluated at selected outputs: every (iy, r) with
 * iy*sh - ph + r*dh == oy and every (ix, s) with ix*sw - pw + s*dw == ox
 * contributes.  The pairs are found by testing the scatter condition for
 * each input row / column, so this is the same sum as above, restricted. */
int oracle_conv_transposed_points(const double *x, int64_t N, int64_t H, int64_t W, int64_t C,
                                  const double *w, int64_t R, int64_t S, int64_t F,
                                  int sh, int sw, int ph, int pw, int dh, int dw,
                                  int64_t Ho, int64_t Wo,
                                  int has_res, const double *src, double beta, int act,
                                  const int64_t *pts, int64_t npts, double *out)
{
    int64_t total = N * Ho * Wo * F;
    for (int64_t i = 0; i < npts; ++i) {
        int64_t o = pts[i];
        if (o < 0 || o >= total) return -1;
        int64_t f = o % F, t = o / F;
        int64_t ox = t % Wo; t /= Wo;
        int64_t oy = t % Ho;
        int64_t n = t / Ho;
        double acc = 0.0;
        for (int64_t r = 0; r < R; ++r)
            for (int64_t iy = 0; iy < H; ++iy) {
                if (iy * sh - ph + r * dh != oy) continue;
                for (int64_t s = 0; s < S; ++s)
                    for (int64_t ix = 0; ix < W; ++ix) {
                        if (ix * sw - pw + s * dw != ox) continue;
                        for (int64_t c = 0; c < C; ++c)
                            acc += x[((n * H + iy) * W + ix) * C + c] *
                                   w[((r * S + s) * F + f) * C + c];
                    }
            }
        if (has_res) acc += beta * src[o];
        out[i] = oracle_activation(acc, act);
    }
    return 0;
}
