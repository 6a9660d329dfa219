"""conv2d_fwd_noalloc: the forward convolution for callers that cannot
allocate device memory (it keeps the packed filter and status word in a
library-owned static device array instead of a caller workspace).

Checked through the C ABI on two calls in a row, with different shapes, so
the second call runs on scratch the first one left behind:
  - bit for bit against conv2d_fwd: both run the same plan and kernels, so
    the raw output bits must be identical;
  - element by element against the CPU oracle within the parity bound the
    other GPU tests use.
A grouped (tensor-core) and a depthwise (CUDA-core) case exercise the size
gate, which sizes the packed filter by C_in / num_groups.  This file is
collected last so that a stop-at-first-failure run has already run every
other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests import _harness as H
from transposed_conv_implicit_gb300 import _lib, synthetic
from transposed_conv_implicit_gb300.synthetic import ConvCase, Dist

pytestmark = pytest.mark.gpu

CASES = [
    ConvCase("noalloc_a", "fwd", "bf16", 2, 13, 11, 64, 96, 3, 3, 2, 1, "FCRS", Dist("normal", 1.0),
             Dist("normal", 1.0 / 576), seed=4242, has_residual=True, beta=0.5,
             src_dist=Dist("normal", 1.0), epilogue="relu"),
    ConvCase("noalloc_b", "fwd", "f8e4m3", 1, 12, 12, 128, 48, 3, 3, 1, 1, "RSCF",
             Dist("normal", 1.0), Dist("normal", 1.0 / 1152), seed=4343),
    # Channel groups of 64 on the tensor cores.
    ConvCase("noalloc_g4", "fwd", "bf16", 1, 10, 9, 256, 128, 3, 3, 1, 1, "RSCF",
             Dist("normal", 1.0), Dist("normal", 1.0 / 576), seed=4444, groups=4),
    # Depthwise, 64 channels, on the CUDA-core kernel.
    ConvCase("noalloc_dw", "fwd", "bf16", 2, 9, 10, 64, 64, 3, 3, 1, 1, "RSCF",
             Dist("normal", 1.0), Dist("normal", 2.0 / 9), seed=4545, groups=64,
             has_residual=True, beta=-1.0, src_dist=Dist("normal", 1.0)),
]


def _run(entry, case, inp):
    dev = "cuda:0"
    x, w = inp["x"].to(dev), inp["w"].to(dev)
    src = inp["src"].to(dev) if inp["src"] is not None else None
    out = torch.full(case.out_shape, float("nan"), dtype=synthetic.TORCH_DTYPES[case.out_dtype],
                     device=dev)
    lib = _lib.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    st, pd, dl = _lib.pair((case.stride,) * 2), _lib.pair(case.pads), _lib.pair(case.dilations)
    args = (ctypes.c_void_p(x.data_ptr()), case.N, case.H, case.W, case.C_in,
            _lib.DTYPE_CODES[case.dtype], ctypes.c_void_p(w.data_ptr()), case.R, case.S, case.C_out,
            int(case.filter_layout == "FCRS"), ctypes.c_void_p(out.data_ptr()), case.Ho, case.Wo,
            _lib.DTYPE_CODES[case.out_dtype], st, dl, pd, case.groups, int(case.has_residual),
            ctypes.c_void_p(src.data_ptr() if src is not None else 0), float(case.beta),
            _lib.EPILOGUE_CODES[case.epilogue])
    if entry == "noalloc":
        status = lib.conv2d_fwd_noalloc(*args, stream)
    else:
        nbytes = lib.conv2d_workspace_size(case.R, case.S, case.C_in // case.groups, case.C_out,
                                           _lib.DTYPE_CODES[case.dtype])
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        status = lib.conv2d_fwd(*args, ctypes.c_void_p(ws.data_ptr()), nbytes, stream)
    assert status == 0, lib.conv_status_string(status)
    torch.cuda.synchronize(dev)
    return out.cpu()


def test_noalloc_matches_conv2d_fwd_and_oracle_on_two_calls_in_a_row():
    for case in CASES:   # each call reuses the scratch the previous one wrote
        inp = synthetic.make_inputs(case)
        ref_out = _run("fwd", case, inp)
        got_out = _run("noalloc", case, inp)
        assert torch.equal(got_out.view(torch.uint8),
                           ref_out.view(torch.uint8)), case.name
        got = H.decode(got_out, case.out_dtype)
        assert np.isfinite(got).all()
        H.assert_parity(case, inp, got, H.oracle_full(case, inp), "noalloc vs oracle")
