"""Pins for the CPU oracle: each check ties it to something other than itself.

Library routines (PyTorch fp64 CPU conv2d / conv_transpose2d, numpy matmul,
torch/numpy dtype casts), hand-worked fixtures under tests/golden, closed forms,
linearity, the adjoint identity and brute-force restatements.  A plausible
mistake in the oracle (a dropped term, a wrong sign or index, a transposed
operand or layout, an off-by-one in padding) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(12345)


def _torch_fwd(x, w, filter_is_fcrs, stride, pad, dil, groups=1):
    """PyTorch's own fp64 CPU conv2d (cross-correlation, FCRS weight [F, C/G, R, S])."""
    xt = torch.from_numpy(x).permute(0, 3, 1, 2)
    wt = torch.from_numpy(w)
    if not filter_is_fcrs:                       # RSCF [R,S,C/G,F] -> [F,C/G,R,S]
        wt = wt.permute(3, 2, 0, 1)
    y = F.conv2d(xt, wt.contiguous(), stride=stride, padding=pad, dilation=dil, groups=groups)
    return y.permute(0, 2, 3, 1).contiguous().numpy()


def _torch_convT(x, w_rsfc, stride, pad, dil, out_hw):
    """PyTorch's own fp64 CPU conv_transpose2d; its weight is [C_in, C_out, R, S]."""
    N, H, W, C = x.shape
    R, S, Fo, _ = w_rsfc.shape
    base = [(H - 1) * stride[0] - 2 * pad[0] + dil[0] * (R - 1) + 1,
            (W - 1) * stride[1] - 2 * pad[1] + dil[1] * (S - 1) + 1]
    opad = (out_hw[0] - base[0], out_hw[1] - base[1])
    xt = torch.from_numpy(x).permute(0, 3, 1, 2)
    wt = torch.from_numpy(w_rsfc).permute(3, 2, 0, 1).contiguous()
    y = F.conv_transpose2d(xt, wt, stride=stride, padding=pad, output_padding=opad, dilation=dil)
    return y.permute(0, 2, 3, 1).contiguous().numpy()


# ----------------------------------------------------------------------------- decoders

def test_decode_bf16_every_pattern_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_decode_f16_every_pattern_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_decode_e4m3_every_pattern_matches_torch():
    bits = np.arange(256, dtype=np.uint8)
    ours = oracle.decode(bits, "f8e4m3")
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_decode_e4m3_spec_values():
    spec = json.load(open(os.path.join(GOLDEN, "e4m3_values.json")))
    for b, v in spec["values"]:
        got = oracle.decode_one(b, "f8e4m3")
        assert got == v and math.copysign(1, got) == math.copysign(1, v), (b, got, v)
    for b in spec["nan"]:
        assert math.isnan(oracle.decode_one(b, "f8e4m3"))


# ----------------------------------------------------------------------------- hand-worked

def test_hand_worked_forward():
    g = json.load(open(os.path.join(GOLDEN, "hand_conv2d_fwd.json")))
    x = np.array(g["x"], dtype=np.float64)[None, :, :, None]
    w = np.array(g["w"], dtype=np.float64)[:, :, None, None]        # RSCF
    for case in g["cases"]:
        st, p = case["stride"], case["pad"]
        y = oracle.conv2d_fwd(x, w, filter_is_fcrs=False, stride=(st, st), padding=(p, p))
        assert np.array_equal(y[0, :, :, 0], np.array(case["y"], dtype=np.float64)), case


def test_hand_worked_transposed():
    g = json.load(open(os.path.join(GOLDEN, "hand_conv_transposed.json")))
    x = np.array(g["x"], dtype=np.float64)[None, :, :, None]
    w = np.array(g["w"], dtype=np.float64)[:, :, None, None]        # RSFC
    for case in g["cases"]:
        st, p = case["stride"], case["pad"]
        y = oracle.conv_transposed(x, w, out_hw=tuple(case["out_hw"]), stride=(st, st), padding=(p, p))
        assert np.array_equal(y[0, :, :, 0], np.array(case["y"], dtype=np.float64)), case


# ----------------------------------------------------------------------------- library special cases

FWD_CASES = [
    # N, H, W, C, F, R, S, stride, pad, dil, fcrs
    (1, 5, 7, 3, 4, 3, 3, (1, 1), (1, 1), (1, 1), True),
    (2, 6, 5, 2, 3, 3, 3, (2, 2), (1, 1), (1, 1), False),
    (1, 8, 8, 4, 2, 5, 5, (2, 2), (2, 2), (1, 1), True),
    (2, 7, 9, 3, 5, 1, 1, (1, 1), (0, 0), (1, 1), False),
    (1, 9, 6, 2, 2, 3, 2, (1, 2), (0, 1), (1, 1), True),
    (1, 9, 9, 2, 3, 3, 3, (1, 1), (2, 2), (2, 1), False),
    (3, 4, 4, 5, 1, 2, 2, (2, 2), (0, 0), (1, 1), True),
    (1, 11, 10, 1, 3, 4, 3, (2, 1), (2, 0), (1, 2), False),
]


@pytest.mark.parametrize("case", FWD_CASES)
def test_forward_matches_torch_conv2d(case):
    N, H, W, C, Fo, R, S, st, pd, dl, fcrs = case
    x = RNG.standard_normal((N, H, W, C))
    w = RNG.standard_normal((Fo, C, R, S) if fcrs else (R, S, C, Fo))
    ours = oracle.conv2d_fwd(x, w, filter_is_fcrs=fcrs, stride=st, padding=pd, dilation=dl)
    ref = _torch_fwd(x, w, fcrs, st, pd, dl)
    assert ours.shape == ref.shape
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-12)


def test_fcrs_and_rscf_describe_the_same_filter():
    x = RNG.standard_normal((1, 6, 6, 3))
    w_rscf = RNG.standard_normal((3, 3, 3, 4))
    w_fcrs = np.ascontiguousarray(w_rscf.transpose(3, 2, 0, 1))
    a = oracle.conv2d_fwd(x, w_rscf, filter_is_fcrs=False, padding=(1, 1))
    b = oracle.conv2d_fwd(x, w_fcrs, filter_is_fcrs=True, padding=(1, 1))
    assert np.array_equal(a, b)


TR_CASES = [
    # N, H, W, C, F, R, S, stride, pad, dil, extra output (output_padding)
    (1, 4, 4, 3, 2, 4, 4, (2, 2), (1, 1), (1, 1), (0, 0)),
    (2, 3, 5, 2, 3, 3, 3, (2, 2), (1, 1), (1, 1), (1, 1)),
    (1, 5, 4, 2, 2, 3, 3, (1, 1), (1, 1), (1, 1), (0, 0)),
    (1, 3, 3, 4, 3, 5, 5, (2, 2), (2, 2), (1, 1), (1, 0)),
    (2, 4, 3, 1, 2, 2, 3, (2, 1), (0, 1), (1, 1), (0, 0)),
    (1, 4, 4, 2, 2, 3, 3, (1, 1), (0, 0), (2, 2), (0, 0)),
    # stride 2 with dilation 2 (taps reach only every other output phase)
    (2, 4, 5, 2, 3, 4, 4, (2, 2), (1, 1), (2, 2), (0, 1)),
    # strides 3 and 4, dilation 2 with stride 3, per-axis stride and dilation
    (1, 3, 4, 2, 2, 3, 3, (3, 3), (1, 1), (1, 1), (2, 0)),
    (1, 3, 3, 3, 2, 4, 4, (4, 4), (0, 0), (1, 1), (0, 3)),
    (2, 3, 3, 2, 2, 3, 3, (3, 3), (2, 2), (2, 2), (1, 1)),
    (1, 4, 3, 2, 3, 3, 2, (1, 2), (1, 0), (3, 1), (0, 1)),
]


@pytest.mark.parametrize("case", TR_CASES)
def test_transposed_matches_torch_conv_transpose2d(case):
    N, H, W, C, Fo, R, S, st, pd, dl, extra = case
    Ho = (H - 1) * st[0] - 2 * pd[0] + dl[0] * (R - 1) + 1 + extra[0]
    Wo = (W - 1) * st[1] - 2 * pd[1] + dl[1] * (S - 1) + 1 + extra[1]
    x = RNG.standard_normal((N, H, W, C))
    w = RNG.standard_normal((R, S, Fo, C))
    ours = oracle.conv_transposed(x, w, out_hw=(Ho, Wo), stride=st, padding=pd, dilation=dl)
    ref = _torch_convT(x, w, st, pd, dl, (Ho, Wo))
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-12)


def test_1x1_conv_is_matmul():
    x = RNG.standard_normal((2, 5, 6, 7))
    w = RNG.standard_normal((1, 1, 7, 9))
    y = oracle.conv2d_fwd(x, w, filter_is_fcrs=False)
    ref = (x.reshape(-1, 7) @ w.reshape(7, 9)).reshape(2, 5, 6, 9)
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)


def test_delta_filter_reproduces_input():
    x = RNG.standard_normal((2, 6, 7, 4))
    for R in (1, 3, 5):
        w = np.zeros((R, R, 4, 4))
        for c in range(4):
            w[R // 2, R // 2, c, c] = 1.0
        y = oracle.conv2d_fwd(x, w, filter_is_fcrs=False, padding=(R // 2, R // 2))
        assert np.array_equal(y, x)


def _im2col_gemm(x, w_rscf, st, pd):
    """Explicit (materialised) im2col matrix [M, R*S*C] times the NK filter, with k = (r*S+s)*C + c."""
    N, H, W, C = x.shape
    R, S, _, Fo = w_rscf.shape
    Ho = (H + 2 * pd - R) // st + 1
    Wo = (W + 2 * pd - S) // st + 1
    xp = np.zeros((N, H + 2 * pd, W + 2 * pd, C))
    xp[:, pd:pd + H, pd:pd + W, :] = x
    A = np.zeros((N * Ho * Wo, R * S * C))
    m = 0
    for n in range(N):
        for oy in range(Ho):
            for ox in range(Wo):
                A[m] = xp[n, oy * st:oy * st + R, ox * st:ox * st + S, :].reshape(-1)
                m += 1
    return (A @ w_rscf.reshape(R * S * C, Fo)).reshape(N, Ho, Wo, Fo)


@pytest.mark.parametrize("st,pd", [(1, 0), (1, 1), (2, 1), (2, 2), (1, 2)])
def test_direct_equals_explicit_im2col_gemm_exactly(st, pd):
    x = RNG.integers(-2, 3, (2, 7, 6, 3)).astype(np.float64)
    w = RNG.integers(-1, 2, (3, 3, 3, 5)).astype(np.float64)
    y = oracle.conv2d_fwd(x, w, filter_is_fcrs=False, stride=(st, st), padding=(pd, pd))
    assert np.array_equal(y, _im2col_gemm(x, w, st, pd))


def _valid_taps(out_idx, stride, pad, R, extent):
    """Closed form: number of r in [0,R) with 0 <= out*stride - pad + r < extent."""
    lo = max(0, pad - out_idx * stride)
    hi = min(R, extent + pad - out_idx * stride)
    return max(0, hi - lo)


@pytest.mark.parametrize("st,pd,R", [(1, 1, 3), (2, 1, 3), (2, 2, 5), (1, 0, 2), (1, 2, 3)])
def test_all_ones_closed_form(st, pd, R):
    C = 5
    x = np.ones((1, 9, 8, C))
    w = np.ones((R, R, C, 2))
    y = oracle.conv2d_fwd(x, w, filter_is_fcrs=False, stride=(st, st), padding=(pd, pd))
    for oy in range(y.shape[1]):
        for ox in range(y.shape[2]):
            want = C * _valid_taps(oy, st, pd, R, 9) * _valid_taps(ox, st, pd, R, 8)
            assert y[0, oy, ox, 0] == want and y[0, oy, ox, 1] == want


# ----------------------------------------------------------------------------- algebraic identities

def test_linearity_in_input_and_filter():
    x1, x2 = RNG.standard_normal((2, 2, 6, 5, 3))
    w1, w2 = RNG.standard_normal((2, 3, 3, 3, 4))
    a, b = 0.75, -1.5
    kw = dict(filter_is_fcrs=False, stride=(2, 2), padding=(1, 1))
    lhs = oracle.conv2d_fwd(a * x1 + b * x2, w1, **kw)
    rhs = a * oracle.conv2d_fwd(x1, w1, **kw) + b * oracle.conv2d_fwd(x2, w1, **kw)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
    lhs = oracle.conv2d_fwd(x1, a * w1 + b * w2, **kw)
    rhs = a * oracle.conv2d_fwd(x1, w1, **kw) + b * oracle.conv2d_fwd(x1, w2, **kw)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("st,pd,R,H", [(1, 1, 3, 6), (2, 1, 3, 7), (2, 1, 4, 8), (2, 2, 5, 9), (1, 0, 2, 5)])
def test_adjoint_identity(st, pd, R, H):
    """<conv(x; w as RSCF), y> == <x, convT(y; the same memory read as RSFC)>."""
    C, Fo = 3, 4
    x = RNG.standard_normal((2, H, H + 1, C))
    w = RNG.standard_normal((R, R, C, Fo))          # RSCF of the forward conv == RSFC of its transpose
    fwd = oracle.conv2d_fwd(x, w, filter_is_fcrs=False, stride=(st, st), padding=(pd, pd))
    y = RNG.standard_normal(fwd.shape)
    back = oracle.conv_transposed(y, w, out_hw=(H, H + 1), stride=(st, st), padding=(pd, pd))
    lhs = float(np.sum(fwd * y))
    rhs = float(np.sum(x * back))
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(lhs))


@pytest.mark.parametrize("pd,R", [(0, 3), (1, 3), (2, 5), (1, 2)])
def test_stride1_transposed_is_flipped_forward_conv(pd, R):
    C, Fo = 3, 2
    x = RNG.standard_normal((1, 6, 5, C))
    w = RNG.standard_normal((R, R, Fo, C))          # RSFC
    Ho, Wo = 6 - 1 - 2 * pd + R, 5 - 1 - 2 * pd + R
    y = oracle.conv_transposed(x, w, out_hw=(Ho, Wo), padding=(pd, pd))
    w_flip = np.ascontiguousarray(w[::-1, ::-1].transpose(0, 1, 3, 2))   # RSCF, C -> F
    q = R - 1 - pd
    ref = oracle.conv2d_fwd(x, w_flip, filter_is_fcrs=False, padding=(q, q))
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- residual and epilogue

def test_zero_filter_gives_beta_times_source():
    x = RNG.standard_normal((1, 5, 5, 2))
    w = np.zeros((3, 3, 2, 3))
    src = RNG.standard_normal((1, 5, 5, 3))
    y = oracle.conv2d_fwd(x, w, filter_is_fcrs=False, padding=(1, 1), source=src, beta=-2.0)
    assert np.array_equal(y, -2.0 * src)


def test_residual_then_activation_order():
    x = RNG.standard_normal((1, 5, 5, 2))
    w = RNG.standard_normal((3, 3, 2, 3))
    src = RNG.standard_normal((1, 5, 5, 3))
    plain = oracle.conv2d_fwd(x, w, filter_is_fcrs=False, padding=(1, 1))
    y = oracle.conv2d_fwd(x, w, filter_is_fcrs=False, padding=(1, 1), source=src, beta=0.5, act="relu")
    np.testing.assert_allclose(y, np.maximum(plain + 0.5 * src, 0.0), rtol=1e-14, atol=1e-14)


def test_transposed_zero_filter_gives_beta_times_source():
    """conv_transposed_gpu, description (backward-data; the epilogue follows the
    conv): with a zero filter the transposed conv contributes nothing, so the
    output is exactly beta*source, for the scatter form and the point form."""
    x = RNG.standard_normal((2, 3, 4, 3))
    w = np.zeros((4, 4, 5, 3))                       # RSFC
    Ho, Wo = (3 - 1) * 2 - 2 + 4 + 1, (4 - 1) * 2 - 2 + 4   # s = 2, p = 1, output padding (1, 0)
    src = RNG.standard_normal((2, Ho, Wo, 5))
    kw = dict(out_hw=(Ho, Wo), stride=(2, 2), padding=(1, 1), source=src, beta=-2.0)
    y = oracle.conv_transposed(x, w, **kw)
    assert np.array_equal(y, -2.0 * src)
    pts = np.arange(y.size)
    assert np.array_equal(oracle.conv_transposed_points(x, w, pts, **kw), (-2.0 * src).reshape(-1))


@pytest.mark.parametrize("act", ["relu", "silu"])
def test_transposed_residual_then_activation_matches_torch(act):
    """act(conv_transpose2d(x) + beta*source) from PyTorch's fp64 conv_transpose2d,
    at stride 2 with an output padding: the residual is added before the
    activation, and beta scales only the source."""
    from scipy.special import expit
    x = RNG.standard_normal((2, 4, 3, 3))
    w = RNG.standard_normal((4, 4, 2, 3))            # RSFC
    Ho, Wo = (4 - 1) * 2 - 2 + 4 + 1, (3 - 1) * 2 - 2 + 4 + 1
    src = RNG.standard_normal((2, Ho, Wo, 2))
    beta = 0.75
    plain = _torch_convT(x, w, (2, 2), (1, 1), (1, 1), (Ho, Wo))
    v = plain + beta * src
    ref = np.maximum(v, 0.0) if act == "relu" else v * expit(v)
    kw = dict(out_hw=(Ho, Wo), stride=(2, 2), padding=(1, 1), source=src, beta=beta, act=act)
    y = oracle.conv_transposed(x, w, **kw)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    pts = np.arange(y.size)
    np.testing.assert_allclose(oracle.conv_transposed_points(x, w, pts, **kw), ref.reshape(-1),
                               rtol=1e-12, atol=1e-12)


def test_activations_against_library():
    from scipy.special import expit
    v = np.linspace(-30, 30, 601)
    silu = np.array([oracle.activation(t, "silu") for t in v])
    np.testing.assert_allclose(silu, v * expit(v), rtol=1e-14, atol=1e-300)
    relu = np.array([oracle.activation(t, "relu") for t in v])
    assert np.array_equal(relu, np.maximum(v, 0))
    assert oracle.activation(-3.25, "none") == -3.25


# ----------------------------------------------------------------------------- point evaluators

def test_forward_points_match_full():
    x = RNG.standard_normal((2, 7, 6, 3))
    w = RNG.standard_normal((4, 3, 3, 3))            # FCRS
    src = RNG.standard_normal((2, 4, 3, 4))
    kw = dict(filter_is_fcrs=True, stride=(2, 2), padding=(1, 1), source=src, beta=0.25, act="silu")
    full = oracle.conv2d_fwd(x, w, **kw)
    pts = np.arange(full.size)
    assert np.array_equal(oracle.conv2d_fwd_points(x, w, pts, **kw), full.reshape(-1))


@pytest.mark.parametrize("st,pd,R", [(2, 1, 4), (2, 1, 3), (1, 1, 3), (2, 2, 5)])
def test_transposed_points_match_scatter(st, pd, R):
    x = RNG.standard_normal((2, 4, 5, 3))
    w = RNG.standard_normal((R, R, 2, 3))
    Ho, Wo = (4 - 1) * st - 2 * pd + R, (5 - 1) * st - 2 * pd + R + (st - 1)
    src = RNG.standard_normal((2, Ho, Wo, 2))
    kw = dict(out_hw=(Ho, Wo), stride=(st, st), padding=(pd, pd), source=src, beta=1.5, act="relu")
    full = oracle.conv_transposed(x, w, **kw)
    pts = np.arange(full.size)
    np.testing.assert_allclose(oracle.conv_transposed_points(x, w, pts, **kw), full.reshape(-1),
                               rtol=1e-13, atol=1e-13)


def test_tolerance_formula():
    tol = oracle.tolerance(np.array([0.0, -2.0]), 576, 3.0, 0.5, "bf16")
    np.testing.assert_allclose(tol, [2e-3 * 24 * 1.5, 0.02 + 2e-3 * 24 * 1.5])
    tol8 = oracle.tolerance(np.array([1.0]), 2880, 1.0, 1.0, "f8e4m3")
    np.testing.assert_allclose(tol8, [0.02 + 2e-3 * math.sqrt(2880)])


# ----------------------------------------------------------------------------- channel groups

GROUP_CASES = [
    # N, H, W, C, F, G, R, S, stride, pad, dil, fcrs
    (1, 6, 7, 4, 6, 2, 3, 3, (1, 1), (1, 1), (1, 1), True),
    (2, 7, 6, 8, 8, 4, 3, 3, (2, 2), (1, 1), (1, 1), False),
    (1, 8, 8, 6, 6, 6, 3, 3, (1, 1), (1, 1), (1, 1), True),      # depthwise
    (1, 9, 8, 6, 12, 3, 5, 3, (2, 1), (2, 1), (1, 2), False),
    (2, 5, 5, 4, 2, 2, 1, 1, (1, 1), (0, 0), (1, 1), True),      # 1x1, one output per group
]


@pytest.mark.parametrize("case", GROUP_CASES)
def test_grouped_forward_matches_torch(case):
    N, H, W, C, Fo, G, R, S, st, pd, dl, fcrs = case
    x = RNG.standard_normal((N, H, W, C))
    w = RNG.standard_normal((Fo, C // G, R, S) if fcrs else (R, S, C // G, Fo))
    ours = oracle.conv2d_fwd(x, w, filter_is_fcrs=fcrs, stride=st, padding=pd, dilation=dl,
                             groups=G)
    ref = _torch_fwd(x, w, fcrs, st, pd, dl, groups=G)
    assert ours.shape == ref.shape
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-12)
    pts = np.arange(0, ours.size, 3, dtype=np.int64)
    got = oracle.conv2d_fwd_points(x, w, pts, filter_is_fcrs=fcrs, stride=st, padding=pd,
                                   dilation=dl, groups=G)
    np.testing.assert_array_equal(got, ours.reshape(-1)[pts])


def test_grouped_forward_is_independent_convs_side_by_side():
    """Group g of the output is the ungrouped conv of group g of the input with
    group g of the filter, computed on integers so the comparison is exact."""
    G, Cg, Fg = 3, 2, 4
    x = RNG.integers(-3, 4, size=(2, 6, 5, G * Cg)).astype(np.float64)
    w = RNG.integers(-2, 3, size=(3, 3, Cg, G * Fg)).astype(np.float64)   # RSCF
    y = oracle.conv2d_fwd(x, w, filter_is_fcrs=False, padding=(1, 1), groups=G)
    for g in range(G):
        part = oracle.conv2d_fwd(x[..., g * Cg:(g + 1) * Cg], w[..., g * Fg:(g + 1) * Fg],
                                 filter_is_fcrs=False, padding=(1, 1))
        assert np.array_equal(y[..., g * Fg:(g + 1) * Fg], part)


def test_grouped_forward_rejects_indivisible_channels():
    x = np.zeros((1, 4, 4, 6))
    with pytest.raises(ValueError):
        oracle.conv2d_fwd(x, np.zeros((4, 3, 3, 3)), filter_is_fcrs=True, groups=4)
