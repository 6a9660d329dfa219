"""Shared test plumbing: run a ConvCase on the GPU through the binding, and on
the CPU oracle, and compare element by element with the parity bound

    |gpu - oracle| <= rel*|oracle| + 2e-3*sqrt(K)*max|a|*max|b|
    rel = 1e-2 (bf16/fp16 inputs), 2e-2 (fp8-e4m3 inputs),

K the contraction length one output sees (R*S*C_in forward;
ceil(R/stride)*ceil(S/stride)*C_in transposed), max|a|, max|b| over the
decoded input and filter.  The oracle never sees anything the GPU produced.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from transposed_conv_implicit_gb300 import synthetic


def decode(t: torch.Tensor, dtype: str) -> np.ndarray:
    return oracle.decode(synthetic.raw_bits(t), dtype)


def _max_taps(extent, stride, dilation, pad):
    """Most filter taps r in [0, extent) that reach one output index of a
    transposed conv: o = i*stride - pad + r*dilation for some input i, i.e.
    r*dilation = o + pad (mod stride), maximised over the output phase o."""
    return max(sum(1 for r in range(extent) if (r * dilation - a - pad) % stride == 0)
               for a in range(stride))


def contraction_length(case) -> int:
    if case.kind == "transposed":
        (sh, sw), (dh, dw), (ph, pw) = case.strides, case.dilations, case.pads
        return max(1, _max_taps(case.R, sh, dh, ph) * _max_taps(case.S, sw, dw, pw)) * case.C_in
    return case.R * case.S * case.C_in // case.groups


def oracle_full(case, inp):
    x = decode(inp["x"], case.dtype)
    w = decode(inp["w"], case.dtype)
    src = decode(inp["src"], case.out_dtype) if inp["src"] is not None else None
    st, pd, dl = case.strides, case.pads, case.dilations
    if case.kind == "transposed":
        return oracle.conv_transposed(x, w, out_hw=(case.Ho, case.Wo), stride=st, padding=pd,
                                      dilation=dl, source=src, beta=case.beta, act=case.epilogue)
    return oracle.conv2d_fwd(x, w, filter_is_fcrs=case.filter_layout == "FCRS", stride=st,
                             padding=pd, dilation=dl, source=src, beta=case.beta,
                             act=case.epilogue, out_hw=(case.Ho, case.Wo), groups=case.groups)


def oracle_points(case, inp, pts):
    x = decode(inp["x"], case.dtype)
    w = decode(inp["w"], case.dtype)
    src = decode(inp["src"], case.out_dtype) if inp["src"] is not None else None
    st, pd, dl = case.strides, case.pads, case.dilations
    if case.kind == "transposed":
        return oracle.conv_transposed_points(x, w, pts, out_hw=(case.Ho, case.Wo), stride=st,
                                             padding=pd, dilation=dl, source=src, beta=case.beta,
                                             act=case.epilogue)
    return oracle.conv2d_fwd_points(x, w, pts, filter_is_fcrs=case.filter_layout == "FCRS",
                                    stride=st, padding=pd, dilation=dl, source=src,
                                    beta=case.beta, act=case.epilogue, out_hw=(case.Ho, case.Wo),
                                    groups=case.groups)


def sample_points(case, count, seed=0):
    """Flat NHWC output indices: a seeded random sample plus the first and last
    pixel, the first/last channel of every sampled pixel, and the last tile."""
    total = case.N * case.Ho * case.Wo * case.C_out
    rng = np.random.default_rng(seed)
    pts = set(rng.integers(0, total, size=min(count, total)).tolist())
    C = case.C_out
    npix = case.N * case.Ho * case.Wo
    for pix in (0, npix - 1, npix // 2, max(0, npix - 128)):
        for c in (0, C - 1):
            pts.add(pix * C + c)
    for pix in rng.integers(0, npix, size=64).tolist():
        pts.add(pix * C)
        pts.add(pix * C + C - 1)
    return np.array(sorted(pts), dtype=np.int64)


def run_gpu(case, inp, *, packed=True, device="cuda:0", out=None, workspace=None):
    """Run the case through the binding; returns the output tensor (device)."""
    import transposed_conv_implicit_gb300 as cg
    x = inp["x"].to(device)
    w = inp["w"].to(device)
    src = inp["src"].to(device) if inp["src"] is not None else None
    if out is None:
        out = torch.empty(case.out_shape, dtype=synthetic.TORCH_DTYPES[case.out_dtype], device=device)
    st, pd, dl = case.strides, case.pads, case.dilations
    kw = dict(has_residual=case.has_residual, source=src, beta=case.beta, epilogue=case.epilogue,
              workspace=workspace)
    if case.kind == "transposed":
        if packed:
            pk = cg.conv_transposed_pack_filter(w, stride=st, padding=pd, dilation=dl)
            cg.conv_transposed_packed(x, pk, out, r=case.R, s=case.S, stride=st, dilation=dl,
                                      padding=pd, **kw)
        else:
            cg.conv_transposed(x, w, out, stride=st, dilation=dl, padding=pd, **kw)
    else:
        fcrs = case.filter_layout == "FCRS"
        if packed:
            pk = cg.conv2d_pack_filter(w, filter_is_fcrs=fcrs)
            cg.conv2d_fwd_packed(x, pk, out, r=case.R, s=case.S, stride=st, dilation=dl,
                                 symmetric_padding=pd, num_groups=case.groups, **kw)
        else:
            cg.conv2d_fwd(x, w, out, stride=st, dilation=dl, symmetric_padding=pd,
                          filter_is_fcrs=fcrs, num_groups=case.groups, **kw)
    return out


def assert_parity(case, inp, gpu_vals: np.ndarray, ref: np.ndarray, what=""):
    x = decode(inp["x"], case.dtype)
    w = decode(inp["w"], case.dtype)
    tol = oracle.tolerance(ref, contraction_length(case), float(np.abs(x).max()),
                           float(np.abs(w).max()), case.dtype)
    err = np.abs(gpu_vals - ref)
    bad = ~(err <= tol)              # NaN in the GPU output counts as a failure
    if bad.any():
        idx = np.flatnonzero(bad.reshape(-1))[:8]
        raise AssertionError(
            "%s %s: %d/%d outside the bound; first flat indices %s gpu %s oracle %s tol %s" % (
                case.name, what, int(bad.sum()), bad.size, idx.tolist(),
                gpu_vals.reshape(-1)[idx].tolist(), ref.reshape(-1)[idx].tolist(),
                tol.reshape(-1)[idx].tolist()))
    return float((err / np.maximum(tol, 1e-30)).max())
