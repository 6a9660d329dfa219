"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Small cases are compared on every output element; the full-size workloads,
run in the launch configuration the benchmark times, are compared on sampled
outputs that the oracle evaluates one by one.  Integer-valued cases must
match bit for bit.  The bound is the one in tests/_harness.py.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from tests import _harness as H
from transposed_conv_implicit_gb300 import synthetic
from transposed_conv_implicit_gb300.synthetic import ConvCase, Dist, WORKLOADS

pytestmark = pytest.mark.gpu


def _fwd(name, dt, N, Hh, W, C, F, R, st, pd, *, layout="RSCF", res=False, beta=0.0, epi="none",
         seed=1, xd=None, wd=None, S=None, dil=1, pad_w=None, dil_w=None, groups=1):
    S = R if S is None else S
    return ConvCase(name, "fwd", dt, N, Hh, W, C, F, R, S, st, pd, layout,
                    xd or Dist("normal", 1.0), wd or Dist("normal", groups / (R * S * C)),
                    seed=seed, dilation=dil, has_residual=res, beta=beta,
                    src_dist=Dist("normal", 1.0) if res else None, epilogue=epi, pad_w=pad_w,
                    dilation_w=dil_w, groups=groups)


def _tr(name, dt, N, Hh, W, C, F, R, st, pd, extra=0, *, res=False, beta=0.0, epi="none", seed=1,
        xd=None, wd=None, dil=1, st_w=None, extra_w=None):
    sw = st if st_w is None else st_w
    Ho = (Hh - 1) * st - 2 * pd + dil * (R - 1) + 1 + extra
    Wo = (W - 1) * sw - 2 * pd + dil * (R - 1) + 1 + (extra if extra_w is None else extra_w)
    return ConvCase(name, "transposed", dt, N, Hh, W, C, F, R, R, st, pd, "RSFC",
                    xd or Dist("normal", 1.0), wd or Dist("normal", 1.0 / (R * R * C)), seed=seed,
                    has_residual=res, beta=beta, src_dist=Dist("normal", 1.0) if res else None,
                    epilogue=epi, out_hw=(Ho, Wo), dilation=dil, stride_w=st_w)


# Several M tiles with a ragged tail (N*Ho*Wo not a multiple of 128), edge
# tiles along C_out (1, 3, 17, 272 = 2 x 144 with a ragged second tile), each
# stride/padding/filter-size gate value, both forward layouts, all dtypes,
# residual with several betas and every epilogue.
SMALL_FWD = [
    _fwd("b_3x3_s1p1", "bf16", 2, 13, 13, 64, 64, 3, 1, 1),
    _fwd("b_3x3_s2p1", "bf16", 2, 13, 11, 64, 128, 3, 2, 1, layout="FCRS"),
    _fwd("b_5x5_s2p2", "bf16", 2, 11, 12, 32, 48, 5, 2, 2),
    _fwd("b_5x5_s1p2_res", "bf16", 1, 12, 14, 32, 32, 5, 1, 2, res=True, beta=-2.0),
    _fwd("b_3x3_s1p0", "bf16", 2, 12, 9, 48, 24, 3, 1, 0),
    _fwd("b_3x3_s2p2", "bf16", 1, 15, 15, 64, 80, 3, 2, 2, epi="relu"),
    _fwd("b_1x1_s1p0", "bf16", 2, 9, 15, 128, 96, 1, 1, 0, layout="FCRS"),
    _fwd("b_1x1_s2p0", "bf16", 2, 10, 10, 64, 64, 1, 2, 0),
    _fwd("b_cout1", "bf16", 2, 11, 11, 64, 1, 3, 1, 1),
    _fwd("b_cout3_head", "bf16", 1, 20, 20, 128, 3, 3, 1, 1),
    _fwd("b_cout17_res", "bf16", 2, 10, 10, 32, 17, 3, 1, 1, res=True, beta=0.5),
    _fwd("b_cout272", "bf16", 1, 12, 12, 64, 272, 3, 1, 1, layout="FCRS"),
    _fwd("b_cout512_silu", "bf16", 1, 12, 12, 64, 512, 3, 1, 1, epi="silu"),
    _fwd("b_cin16", "bf16", 1, 16, 16, 16, 16, 3, 1, 1),
    _fwd("b_cin48_64B", "bf16", 2, 9, 9, 48, 32, 3, 2, 1),
    _fwd("b_res_relu", "bf16", 2, 13, 13, 64, 64, 3, 1, 1, res=True, beta=1.0, epi="relu"),
    _fwd("b_rect_3x5", "bf16", 1, 13, 17, 64, 64, 3, 1, 1, S=5),
    _fwd("h_3x3_s1p1", "f16", 2, 13, 13, 64, 64, 3, 1, 1),
    _fwd("h_5x5_s2p2", "f16", 2, 17, 17, 128, 128, 5, 2, 2),
    _fwd("h_res_silu", "f16", 1, 14, 14, 64, 40, 3, 1, 1, res=True, beta=0.75, epi="silu"),
    _fwd("h_cout3", "f16", 1, 15, 15, 32, 3, 3, 2, 1, layout="FCRS"),
    _fwd("h_cin16", "f16", 2, 9, 9, 16, 32, 3, 1, 1),
    _fwd("e_3x3_s1p1_res", "f8e4m3", 2, 11, 11, 320, 320, 3, 1, 1, layout="FCRS", res=True,
         beta=0.5, wd=Dist("normal", 1.0 / math.sqrt(2880))),
    _fwd("e_3x3_s2p1", "f8e4m3", 2, 13, 13, 64, 64, 3, 2, 1),
    _fwd("e_1x1", "f8e4m3", 1, 12, 12, 128, 48, 1, 1, 0),
    _fwd("e_5x5_p2_relu", "f8e4m3", 1, 12, 12, 32, 16, 5, 1, 2, epi="relu"),
    _fwd("e_cout3", "f8e4m3", 1, 16, 16, 128, 3, 3, 1, 1),
    _fwd("e_cin32_32B", "f8e4m3", 2, 10, 10, 32, 64, 3, 1, 1, layout="FCRS"),
    _fwd("b_cin24_partial_block", "bf16", 2, 9, 10, 24, 32, 3, 1, 1),
    _fwd("b_cin80_partial_block", "bf16", 1, 11, 11, 80, 48, 3, 2, 1, res=True, beta=1.0),
    _fwd("e_cin160_partial_block", "f8e4m3", 1, 10, 10, 160, 64, 3, 1, 1, layout="FCRS"),
    _fwd("b_window_cin160_partial", "bf16", 2, 10, 9, 160, 48, 3, 1, 1),
    _fwd("b_window_rowblocks_res", "bf16", 2, 21, 20, 64, 64, 3, 1, 1, res=True, beta=1.0),
    _fwd("b_window_5x5_p2", "bf16", 1, 17, 19, 64, 96, 5, 1, 2, res=True, beta=-0.5, epi="silu"),
    _fwd("h_window_cout128", "f16", 2, 14, 12, 64, 128, 3, 1, 1, epi="relu"),
    _fwd("b_window_cout256", "bf16", 1, 9, 11, 128, 256, 3, 1, 1, layout="FCRS"),
    _fwd("b_single_partial_tile", "bf16", 1, 5, 7, 64, 64, 3, 1, 1),
    _fwd("b_exact_one_tile", "bf16", 2, 8, 8, 64, 64, 3, 1, 1),
    _fwd("b_tiny_image", "bf16", 3, 2, 3, 32, 16, 3, 2, 2),
    # Gather loader: channel rows TMA cannot address (C_in * elt % 16 != 0 or < 32).
    _fwd("b_gather_c3_stem3x3_s2", "bf16", 2, 17, 19, 3, 32, 3, 2, 1),
    _fwd("b_gather_c3_7x7_s2p3", "bf16", 2, 23, 21, 3, 64, 7, 2, 3, layout="FCRS"),
    _fwd("h_gather_c5_res_silu", "f16", 1, 13, 11, 5, 40, 3, 1, 1, res=True, beta=0.5, epi="silu"),
    _fwd("b_gather_c8_16B", "bf16", 2, 10, 10, 8, 16, 3, 1, 1),
    _fwd("b_gather_c20_fcrs", "bf16", 2, 9, 11, 20, 48, 3, 2, 1, layout="FCRS"),
    _fwd("e_gather_c3_5x5", "f8e4m3", 2, 12, 12, 3, 32, 5, 1, 2),
    _fwd("e_gather_c16_res", "f8e4m3", 1, 11, 11, 16, 64, 3, 1, 1, res=True, beta=0.5),
    _fwd("b_gather_c3_dil_h2", "bf16", 1, 15, 15, 3, 16, 3, 1, 2, dil=2, dil_w=1),
    _fwd("b_gather_c1_1x1", "bf16", 2, 9, 9, 1, 16, 1, 1, 0),
    _fwd("b_gather_c6_cout300", "bf16", 1, 10, 10, 6, 300, 3, 1, 1, epi="relu"),
    _fwd("h_gather_c3_tail_rows", "f16", 3, 7, 5, 3, 24, 3, 1, 1),
    # ... with input rows staged by bulk copies (W * C_in * elt a multiple of 16 bytes),
    # including tiles that span two or more images.
    _fwd("b_stage_c3_7x7_s2p3", "bf16", 3, 16, 16, 3, 64, 7, 2, 3),
    _fwd("h_stage_c5_res", "f16", 2, 12, 8, 5, 24, 3, 1, 1, res=True, beta=0.5),
    _fwd("e_stage_c3_s2", "f8e4m3", 2, 20, 16, 3, 32, 3, 2, 1),
    _fwd("b_stage_c3_dil_h3", "bf16", 1, 30, 16, 3, 16, 3, 1, 3, dil=3, dil_w=1, pad_w=1),
    _fwd("b_stage_c6_tiny_images", "bf16", 6, 4, 8, 6, 32, 3, 1, 1, epi="silu"),
    _fwd("b_stage_c8_cout200", "bf16", 2, 14, 14, 8, 200, 3, 2, 1),
    # Dilation (TMA im2col tap offsets) and padding per axis.
    _fwd("b_dil2_same", "bf16", 2, 15, 14, 64, 64, 3, 1, 2, dil=2),
    _fwd("h_dil3_s2", "f16", 1, 20, 20, 32, 48, 3, 2, 2, dil=3),
    _fwd("b_dil_w2_only", "bf16", 1, 12, 13, 32, 32, 3, 1, 1, dil=1, dil_w=2),
    _fwd("b_pad3_7x7_s2", "bf16", 1, 20, 20, 32, 32, 7, 2, 3),
    _fwd("b_window_7x7_p3", "bf16", 1, 14, 14, 64, 16, 7, 1, 3, res=True, beta=1.0),
    _fwd("b_pad_h1_w0", "bf16", 2, 10, 12, 64, 64, 3, 1, 1, pad_w=0),
    _fwd("e_pad_h0_w2_5x5", "f8e4m3", 1, 12, 12, 64, 32, 5, 2, 0, pad_w=2),
    # Channel groups: per-group channel offsets, filter slots and output clipping.
    _fwd("b_groups2", "bf16", 2, 11, 10, 64, 64, 3, 1, 1, groups=2),
    _fwd("b_groups4_fg24_res", "bf16", 1, 12, 12, 128, 96, 3, 1, 1, groups=4, res=True, beta=1.0),
    _fwd("h_groups2_s2_fcrs", "f16", 2, 13, 13, 64, 128, 3, 2, 1, groups=2, layout="FCRS"),
    _fwd("e_groups8", "f8e4m3", 1, 10, 10, 256, 64, 3, 1, 1, groups=8, epi="relu"),
    _fwd("b_groups2_fg3_direct", "bf16", 1, 9, 9, 64, 6, 3, 1, 1, groups=2),
    _fwd("b_groups32_1x1", "bf16", 2, 8, 8, 1024, 512, 1, 1, 0, groups=32, epi="silu"),
    # Narrow groups on the direct CUDA-core kernel: depthwise (vector path),
    # channel multipliers, groups of 4 and 40 channels, both filter layouts.
    _fwd("b_depthwise_3x3", "bf16", 2, 12, 12, 64, 64, 3, 1, 1, groups=64),
    _fwd("b_depthwise_s2_res_relu", "bf16", 2, 13, 11, 128, 128, 3, 2, 1, groups=128, res=True,
         beta=0.5, epi="relu", layout="FCRS"),
    _fwd("h_depthwise_mult2", "f16", 1, 10, 10, 32, 64, 3, 1, 1, groups=32),
    _fwd("b_groups16_cg4", "bf16", 2, 9, 9, 64, 64, 3, 1, 1, groups=16, layout="FCRS"),
    _fwd("e_depthwise_5x5", "f8e4m3", 1, 12, 12, 64, 64, 5, 1, 2, groups=64, epi="silu"),
    _fwd("b_depthwise_7x7_dil2", "bf16", 1, 20, 20, 32, 32, 7, 1, 6, groups=32, dil=2),
    _fwd("b_groups2_cg40_flat", "bf16", 1, 9, 9, 80, 48, 3, 1, 1, groups=2),
    _fwd("b_depthwise_c3", "bf16", 2, 9, 9, 3, 3, 3, 1, 1, groups=3),
    # 3x3 depthwise, stride 1, on the tile kernel: ragged 28-column tiles and
    # 8-row halves, several channel blocks (one partial), padding 0/1/2,
    # residual, both 16-bit types.
    _fwd("b_dw3x3_w70_res", "bf16", 3, 19, 70, 64, 64, 3, 1, 1, groups=64, res=True, beta=0.5,
         epi="relu"),
    _fwd("h_dw3x3_c72_p0", "f16", 1, 13, 35, 72, 72, 3, 1, 0, groups=72, layout="FCRS"),
    _fwd("b_dw3x3_c200_p2_silu", "bf16", 2, 6, 33, 200, 200, 3, 1, 2, groups=200, epi="silu"),
    _fwd("b_dw3x3_tall_narrow", "bf16", 1, 41, 3, 16, 16, 3, 1, 1, groups=16),
    # Widths whose tiles are 32 columns (64 and 96: no column left over)
    # rather than 28 (every case above).
    _fwd("b_dw3x3_w64_res", "bf16", 2, 18, 64, 64, 64, 3, 1, 1, groups=64, res=True, beta=0.5,
         epi="relu"),
    _fwd("h_dw3x3_w96_c136_silu", "f16", 1, 9, 96, 136, 136, 3, 1, 1, groups=136, epi="silu"),
    # Row-tap kernel (few output channels, stride 1): two or more 126-pixel
    # segments with a ragged last one, short last bands, g16 = 16 and 32,
    # R = 1, 3 and 5, S = 1 and 3, padding 0..2, several channel blocks.
    _fwd("rt_b_w150_res_silu", "bf16", 2, 13, 150, 64, 3, 3, 1, 1, res=True, beta=0.5, epi="silu"),
    _fwd("rt_h_cout1_w20", "f16", 1, 9, 20, 128, 1, 3, 1, 1, layout="FCRS"),
    _fwd("rt_e_cout5", "f8e4m3", 2, 10, 40, 128, 5, 3, 1, 1, epi="relu"),
    _fwd("rt_b_cout8_g32", "bf16", 1, 11, 30, 64, 8, 3, 1, 1, res=True, beta=-1.0),
    _fwd("rt_b_5x5_p2_cout3", "bf16", 1, 12, 140, 64, 3, 5, 1, 2, epi="relu"),
    _fwd("rt_b_3x3_p0_cout2", "bf16", 2, 9, 12, 128, 2, 3, 1, 0),
    _fwd("rt_h_1x3_cout4", "f16", 1, 6, 133, 64, 4, 1, 1, 0, S=3, pad_w=1),
    _fwd("rt_b_3x1_cout10", "bf16", 1, 14, 17, 64, 10, 3, 1, 1, S=1, pad_w=0, layout="FCRS"),
    _fwd("rt_b_cin256_cout3", "bf16", 1, 8, 8, 256, 3, 3, 1, 1),
    _fwd("rt_e_cout10_g32", "f8e4m3", 1, 9, 27, 256, 10, 3, 1, 1, res=True, beta=0.5),
]

SMALL_TR = [
    _tr("t_h_4x4_s2p1_relu", "f16", 2, 9, 8, 64, 64, 4, 2, 1, epi="relu"),
    _tr("t_b_3x3_s2p1_op1", "bf16", 2, 7, 7, 64, 32, 3, 2, 1, extra=1),
    _tr("t_b_3x3_s2p1_op0", "bf16", 1, 9, 9, 32, 48, 3, 2, 1),
    _tr("t_b_3x3_s1p1", "bf16", 2, 9, 10, 64, 64, 3, 1, 1),
    _tr("t_h_5x5_s2p2_res", "f16", 1, 8, 8, 128, 40, 5, 2, 2, res=True, beta=0.5),
    _tr("t_b_2x2_s2p0", "bf16", 2, 8, 8, 64, 16, 2, 2, 0),
    _tr("t_b_1x1_s2_zero_tap_phase", "bf16", 1, 9, 9, 32, 16, 1, 2, 0, extra=1, epi="relu"),
    _tr("t_e_4x4_s2p1", "f8e4m3", 2, 8, 8, 64, 64, 4, 2, 1),
    _tr("t_h_cout3", "f16", 1, 10, 10, 64, 3, 4, 2, 1),
    _tr("t_h_cout256_silu", "f16", 1, 6, 6, 64, 256, 4, 2, 1, epi="silu"),
    _tr("t_h_cin80_partial_block", "f16", 1, 7, 7, 80, 32, 4, 2, 1),
    # Dilation and general strides: with dilation 2 at stride 2 half the
    # output phases have no taps; strides 3 and 4 have 9 and 16 phases (three
    # and four launches of four phases); stride 3 with dilation 2 (gcd 1);
    # per-axis strides; C_out 17 on the direct epilogue; fp8 with a residual.
    _tr("t_h_4x4_s2p1_d2", "f16", 2, 7, 6, 64, 32, 4, 2, 1, dil=2, epi="relu"),
    _tr("t_b_3x3_s3p1", "bf16", 2, 6, 5, 64, 48, 3, 3, 1, extra=2),
    _tr("t_b_4x4_s4p0", "bf16", 1, 5, 6, 32, 64, 4, 4, 0, extra=1),
    _tr("t_h_3x3_s3p2_d2", "f16", 1, 6, 6, 64, 32, 3, 3, 2, dil=2, extra=1),
    _tr("t_b_3x3_s12", "bf16", 2, 7, 6, 64, 32, 3, 1, 1, st_w=2, extra=0, extra_w=1),
    _tr("t_h_cout17_s3", "f16", 1, 5, 7, 64, 17, 3, 3, 0, extra=1),
    _tr("t_e_5x5_s2p3_d2_res", "f8e4m3", 1, 6, 6, 64, 64, 5, 2, 3, dil=2, res=True, beta=0.5),
]


@pytest.mark.parametrize("case", SMALL_FWD + SMALL_TR, ids=lambda c: c.name)
def test_small_case_every_element(case):
    inp = synthetic.make_inputs(case)
    out = H.run_gpu(case, inp)
    torch.cuda.synchronize()
    got = H.decode(out.cpu(), case.out_dtype)
    ref = H.oracle_full(case, inp)
    H.assert_parity(case, inp, got, ref)


@pytest.mark.parametrize("case", [c for c in SMALL_FWD if c.name in (
    "b_cout1", "b_cout3_head", "e_cout3", "rt_b_cout8_g32", "rt_h_1x3_cout4")],
    ids=lambda c: c.name)
def test_masked_edge_tile_without_row_tap(case, tuning):
    """The same small-C_out convs on the implicit GEMM's masked edge tile (the
    row-tap kernel switched off)."""
    tuning("CONV_ROWTAP", "-1")
    inp = synthetic.make_inputs(case)
    out = H.run_gpu(case, inp)
    torch.cuda.synchronize()
    H.assert_parity(case, inp, H.decode(out.cpu(), case.out_dtype), H.oracle_full(case, inp))


@pytest.mark.parametrize("case", [c for c in SMALL_FWD + SMALL_TR if c.name in (
    "b_3x3_s2p1", "b_cout17_res", "e_3x3_s1p1_res", "t_h_4x4_s2p1_relu", "t_b_3x3_s2p1_op1",
    "b_gather_c3_7x7_s2p3", "e_gather_c3_5x5", "b_groups4_fg24_res", "h_groups2_s2_fcrs", "b_depthwise_s2_res_relu",
    "b_groups16_cg4", "rt_b_w150_res_silu", "rt_e_cout5")],
    ids=lambda c: c.name)
def test_unpacked_entry_point_equals_packed(case):
    """conv2d_fwd / conv_transposed pack in the workspace; the result must be
    bit-identical to the prepacked entry points."""
    inp = synthetic.make_inputs(case)
    a = H.run_gpu(case, inp, packed=True).cpu()
    b = H.run_gpu(case, inp, packed=False).cpu()
    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def _int_case(name, kind, dt, N, Hh, W, C, F, R, st, pd, **kw):
    xd = Dist("int", 2 if dt != "bf16" else 1)
    wd = Dist("int", 1)
    if kind == "fwd":
        return _fwd(name, dt, N, Hh, W, C, F, R, st, pd, xd=xd, wd=wd, **kw)
    return _tr(name, dt, N, Hh, W, C, F, R, st, pd, xd=xd, wd=wd, **kw)


INT_CASES = [
    _int_case("int_b_3x3", "fwd", "bf16", 2, 13, 13, 16, 16, 3, 1, 1),
    _int_case("int_b_s2_res", "fwd", "bf16", 2, 11, 11, 16, 24, 3, 2, 1, res=False),
    _int_case("int_h_5x5", "fwd", "f16", 1, 12, 12, 64, 32, 5, 2, 2, layout="FCRS"),
    _int_case("int_e_3x3", "fwd", "f8e4m3", 2, 10, 10, 32, 64, 3, 1, 1),
    _int_case("int_h_tr", "transposed", "f16", 2, 8, 8, 64, 32, 4, 2, 1),
    _int_case("int_e_tr", "transposed", "f8e4m3", 1, 7, 7, 32, 16, 3, 2, 1, extra=1),
    _int_case("int_b_tr_s3_d2", "transposed", "bf16", 1, 5, 6, 32, 16, 3, 3, 2, extra=1, dil=2),
    _int_case("int_b_gather_c3", "fwd", "bf16", 2, 11, 13, 3, 16, 7, 2, 3),
    _int_case("int_b_stage_c3", "fwd", "bf16", 2, 16, 16, 3, 16, 7, 2, 3),
    _int_case("int_e_gather_c5", "fwd", "f8e4m3", 1, 9, 9, 5, 32, 3, 1, 1),
    _int_case("int_h_dil2", "fwd", "f16", 1, 12, 12, 16, 16, 3, 1, 2, dil=2),
    _int_case("int_b_groups4", "fwd", "bf16", 1, 10, 10, 64, 32, 3, 1, 1, groups=4),
    _int_case("int_h_depthwise", "fwd", "f16", 2, 9, 9, 32, 32, 3, 1, 1, groups=32),
    _int_case("int_b_rowtap", "fwd", "bf16", 1, 12, 140, 64, 3, 3, 1, 1),
    _int_case("int_b_dw3x3_w40", "fwd", "bf16", 2, 17, 40, 128, 128, 3, 1, 1, groups=128),
    _int_case("int_h_dw3x3_w64", "fwd", "f16", 1, 20, 64, 64, 64, 3, 1, 1, groups=64),
    _int_case("int_e_rowtap_g32", "fwd", "f8e4m3", 1, 9, 30, 128, 9, 3, 1, 1),
]


@pytest.mark.parametrize("case", INT_CASES, ids=lambda c: c.name)
def test_integer_inputs_bit_exact(case):
    """Integer inputs: every product and partial sum is exact in fp32 and the
    result is exactly representable in the output dtype, so the GPU must equal
    the oracle exactly."""
    inp = synthetic.make_inputs(case)
    ref = H.oracle_full(case, inp)
    limit = 256 if case.out_dtype == "bf16" else 2048
    assert np.abs(ref).max() <= limit
    out = H.run_gpu(case, inp)
    got = H.decode(out.cpu(), case.out_dtype)
    mism = np.argwhere(got != ref)
    assert mism.size == 0, mism[:5].tolist()


PAIR_CASES = ("b_3x3_s2p1", "h_5x5_s2p2", "e_3x3_s1p1_res", "b_cout512_silu", "b_cout272",
              "e_3x3_s2p1", "h_res_silu", "b_5x5_s2p2", "b_cout17_res", "b_cin80_partial_block",
              "e_cin160_partial_block", "b_tiny_image", "b_1x1_s2p0", "t_h_4x4_s2p1_relu",
              "t_b_3x3_s2p1_op1", "t_h_cout256_silu", "t_b_1x1_s2_zero_tap_phase",
              "t_h_cin80_partial_block", "t_e_4x4_s2p1", "int_b_s2_res", "int_h_5x5", "int_h_tr",
              "int_e_tr")


def _pair_cases():
    return [c for c in SMALL_FWD + SMALL_TR + INT_CASES if c.name in PAIR_CASES]


@pytest.mark.parametrize("case", _pair_cases(), ids=lambda c: c.name)
def test_cta_pair_every_element(case, tuning):
    """CTA pairs forced on (clusters of two CTAs, cta_group::2 MMAs over
    256-row tiles): every element against the oracle; integer cases bit-exact."""
    tuning("CONV_PAIR", "1")
    inp = synthetic.make_inputs(case)
    out = H.run_gpu(case, inp)
    torch.cuda.synchronize()
    got = H.decode(out.cpu(), case.out_dtype)
    ref = H.oracle_full(case, inp)
    if case.name.startswith("int_"):
        mism = np.argwhere(got != ref)
        assert mism.size == 0, mism[:5].tolist()
    else:
        H.assert_parity(case, inp, got, ref)


# One MMA warp for both 128-row halves of a 256-row tile (CONV_MMA_SPLIT=0):
# the converged warp issues the two halves' MMAs of every K-step itself,
# instead of warps 1 and 11 taking one half each.
SPLIT_OFF_CASES = ("b_3x3_s2p1", "h_5x5_s2p2", "b_cout17_res", "int_b_3x3", "int_h_5x5",
                   "int_b_s2_res", "t_h_4x4_s2p1_relu", "t_h_5x5_s2p2_res",
                   # the row-window loader's MMA role, both halves from one warp
                   "b_res_relu", "b_window_rowblocks_res", "h_res_silu")


def _split_off_cases():
    return [c for c in SMALL_FWD + SMALL_TR + INT_CASES if c.name in SPLIT_OFF_CASES]


@pytest.mark.parametrize("case", _split_off_cases(), ids=lambda c: c.name)
def test_single_mma_warp_for_both_halves(case, tuning):
    tuning("CONV_MMA_SPLIT", "0")
    inp = synthetic.make_inputs(case)
    out = H.run_gpu(case, inp)
    torch.cuda.synchronize()
    got = H.decode(out.cpu(), case.out_dtype)
    ref = H.oracle_full(case, inp)
    if case.name.startswith("int_"):
        mism = np.argwhere(got != ref)
        assert mism.size == 0, mism[:5].tolist()
    else:
        H.assert_parity(case, inp, got, ref)


# Stream-K forced on (CONV_STREAMK=1, a workspace with room for its partial
# tiles).  On these small convs most SMs hold one or two k-blocks of the
# iteration sequence, so every tile is split between several CTAs: the
# finisher adds many partials.  Ragged M tails, several C_out tiles, the
# direct-store epilogue (C_out 3 and 17), a residual source, partial channel
# blocks, fp8, and transposed convs whose phases have equal or unequal K.
STREAMK_CASES = (
    "b_3x3_s2p1", "b_5x5_s2p2", "b_5x5_s1p2_res", "b_3x3_s1p0", "b_1x1_s2p0", "b_cout17_res",
    "b_cout272", "b_cout512_silu", "b_cin48_64B", "h_5x5_s2p2", "h_cout3", "e_3x3_s1p1_res",
    "e_3x3_s2p1", "e_5x5_p2_relu", "b_cin80_partial_block", "e_cin160_partial_block",
    "b_window_cout256", "b_tiny_image", "b_pad3_7x7_s2", "t_h_4x4_s2p1_relu", "t_b_3x3_s2p1_op1",
    "t_b_3x3_s2p1_op0", "t_h_5x5_s2p2_res", "t_b_2x2_s2p0", "t_e_4x4_s2p1", "t_h_cout3",
    "t_h_cout256_silu", "t_h_cin80_partial_block", "int_b_3x3", "int_b_s2_res", "int_h_5x5",
    "int_e_3x3", "int_h_tr", "int_e_tr")


def _streamk_cases():
    return [c for c in SMALL_FWD + SMALL_TR + INT_CASES if c.name in STREAMK_CASES]


def streamk_workspace(device="cuda"):
    import transposed_conv_implicit_gb300 as cg
    return cg.new_workspace(cg.CONV_STATUS_BYTES + cg.conv_streamk_workspace_size(), device)


def plan_of(case, workspace_bytes):
    """The dispatcher's plan for a forward case through conv2d_fwd_packed on this device."""
    import ctypes
    from transposed_conv_implicit_gb300 import _lib
    out = (ctypes.c_int * 14)()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st = _lib.lib().conv_testing_fwd_plan(
        case.N, case.H, case.W, case.C_in, _lib.DTYPE_CODES[case.dtype], case.R, case.S, case.C_out,
        _lib.pair((case.stride,) * 2), _lib.pair(case.pads), int(case.has_residual), sms,
        workspace_bytes, out)
    assert st == 0
    return list(out)


@pytest.mark.parametrize("case", _streamk_cases(), ids=lambda c: c.name)
def test_streamk_every_element(case, tuning):
    """Stream-K forced on: every element against the oracle, integer cases
    bit-exact, and a clean status word."""
    import transposed_conv_implicit_gb300 as cg
    tuning("CONV_STREAMK", "1")
    ws = streamk_workspace()
    if case.kind == "fwd":
        assert plan_of(case, ws.numel())[13] == 1
    inp = synthetic.make_inputs(case)
    out = H.run_gpu(case, inp, workspace=ws)
    status, bits = cg.conv_check_device_status(ws)
    assert status == 0 and bits == 0
    got = H.decode(out.cpu(), case.out_dtype)
    ref = H.oracle_full(case, inp)
    if case.name.startswith("int_"):
        mism = np.argwhere(got != ref)
        assert mism.size == 0, mism[:5].tolist()
    else:
        H.assert_parity(case, inp, got, ref)


def test_streamk_chosen_for_a_deep_contraction():
    """The planner's own choice (no override): 32 output rows over a
    contraction of 9216 leave most SMs idle with whole tiles, so stream-K
    spreads the k-blocks over all of them; every element against the oracle."""
    import transposed_conv_implicit_gb300 as cg
    case = _fwd("b_deepk_s2", "bf16", 2, 8, 8, 1024, 256, 3, 2, 1, res=True, beta=-1.0, epi="relu")
    ws = streamk_workspace()
    assert plan_of(case, ws.numel())[13] == 1
    inp = synthetic.make_inputs(case)
    out = H.run_gpu(case, inp, workspace=ws)
    status, bits = cg.conv_check_device_status(ws)
    assert status == 0 and bits == 0
    H.assert_parity(case, inp, H.decode(out.cpu(), "bf16"), H.oracle_full(case, inp))


@pytest.mark.parametrize("name", list(WORKLOADS), ids=str)
def test_full_size_workload_sampled(name):
    """Full-size workloads in the launch configuration the benchmark times
    (packed filter, a workspace with stream-K room), sampled outputs checked
    against the oracle point by point; every output must be finite."""
    case = WORKLOADS[name]
    inp = synthetic.make_inputs(case)
    out = H.run_gpu(case, inp, workspace=streamk_workspace()).cpu()
    flat = H.decode(out, case.out_dtype).reshape(-1)
    assert np.isfinite(flat).all()
    pts = H.sample_points(case, 3000, seed=11)
    ref = H.oracle_points(case, inp, pts)
    H.assert_parity(case, inp, flat[pts], ref, "sampled")


def test_window_one_half_tiles_several_per_cta():
    """The ResNet-50 bottleneck expansion (1x1, 64 -> 256 channels, + residual,
    ReLU) on 56x56 images: row-window tiles of one 128-row half (C_out > 128),
    more tiles than CTAs, so each CTA's epilogue walks several tiles; sampled
    outputs against the oracle."""
    case = _fwd("b_1x1_expand_res", "bf16", 8, 56, 56, 64, 256, 1, 1, 0, res=True, beta=1.0,
                epi="relu", seed=21)
    plan = plan_of(case, streamk_workspace().numel())
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert plan[11] == 1 and plan[0] == 256 and plan[4] > sms  # row window, N = 256, > 1 wave
    inp = synthetic.make_inputs(case)
    out = H.run_gpu(case, inp, workspace=streamk_workspace()).cpu()
    flat = H.decode(out, case.out_dtype).reshape(-1)
    assert np.isfinite(flat).all()
    pts = H.sample_points(case, 3000, seed=12)
    H.assert_parity(case, inp, flat[pts], H.oracle_points(case, inp, pts), "sampled")


def test_rgb_head_two_accumulator_buffers(tuning):
    """The full-size RGB head with 9-row bands: 285 tiles, so CTAs walk two
    tiles on two TMEM accumulator buffers (the default, 18-row bands in one
    wave, keeps one); sampled outputs against the oracle."""
    tuning("CONV_ROWTAP_BAND", "9")
    case = WORKLOADS["vae_head_bf16"]
    plan = plan_of(case, streamk_workspace().numel())
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert plan[11] == 3 and plan[10] == 9 and plan[4] > sms
    inp = synthetic.make_inputs(case)
    out = H.run_gpu(case, inp, workspace=streamk_workspace()).cpu()
    flat = H.decode(out, case.out_dtype).reshape(-1)
    assert np.isfinite(flat).all()
    pts = H.sample_points(case, 3000, seed=13)
    H.assert_parity(case, inp, flat[pts], H.oracle_points(case, inp, pts), "sampled")


def test_tiny_workload_every_element():
    case = WORKLOADS["tiny_bf16"]
    inp = synthetic.make_inputs(case)
    out = H.run_gpu(case, inp).cpu()
    H.assert_parity(case, inp, H.decode(out, case.out_dtype), H.oracle_full(case, inp))


def test_output_canaries_untouched():
    """Writes stay inside the output: guard bands around it keep their NaN
    pattern and no NaN is left inside."""
    case = _fwd("canary", "bf16", 2, 11, 9, 64, 17, 3, 2, 1, res=True, beta=1.0)
    inp = synthetic.make_inputs(case)
    n = int(np.prod(case.out_shape))
    guard = 4096
    buf = torch.full((n + 2 * guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + n].view(case.out_shape)
    H.run_gpu(case, inp, out=out)
    torch.cuda.synchronize()
    host = buf.cpu()
    assert torch.isnan(host[:guard]).all() and torch.isnan(host[guard + n:]).all()
    assert not torch.isnan(host[guard:guard + n]).any()
    H.assert_parity(case, inp, H.decode(out.cpu(), "bf16"), H.oracle_full(case, inp))


def test_repeated_calls_are_deterministic():
    case = SMALL_FWD[0]
    inp = synthetic.make_inputs(case)
    a = H.run_gpu(case, inp).cpu()
    b = H.run_gpu(case, inp).cpu()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_status_clean_after_runs():
    import transposed_conv_implicit_gb300 as cg
    case = SMALL_FWD[0]
    inp = synthetic.make_inputs(case)
    ws = cg.new_workspace(cg.CONV_STATUS_BYTES, "cuda")
    H.run_gpu(case, inp, workspace=ws)
    status, bits = cg.conv_check_device_status(ws)
    assert status == 0 and bits == 0
