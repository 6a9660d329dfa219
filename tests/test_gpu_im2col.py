"""The A-operand loader in isolation: one TMA im2col load, exactly as the
convolution kernel issues it, compared bit for bit with a numpy gather of the
same NHWC input ("dispatch_fused_im2col_conv2d_apple", description: the A
operand is gathered from the NHWC input on the fly).

Row i of the tile is output pixel m0 + i, holding input channels
[c0, c0 + bk) of the input pixel under filter tap (r, s); pixels in the
padding (and rows past the last image) are zero.
"""
import ctypes

import numpy as np
import pytest
import torch

from transposed_conv_implicit_gb300 import _lib, synthetic

pytestmark = pytest.mark.gpu

CASES = [
    # dtype, N, H, W, C, R, stride, pad, m0, tap_r, tap_s, c0
    ("bf16", 2, 13, 13, 64, 3, 1, 1, 0, 0, 0, 0),
    ("bf16", 2, 13, 13, 64, 3, 1, 1, 128, 2, 1, 0),
    ("bf16", 2, 13, 13, 64, 3, 1, 1, 256, 1, 2, 0),
    ("bf16", 2, 13, 11, 64, 3, 2, 1, 0, 2, 2, 0),
    ("bf16", 3, 12, 12, 64, 3, 2, 1, 64, 0, 1, 0),
    ("bf16", 2, 9, 10, 128, 5, 2, 2, 32, 4, 3, 64),
    ("bf16", 2, 9, 9, 64, 3, 1, 0, 48, 1, 1, 0),
    ("bf16", 1, 16, 16, 16, 3, 1, 1, 128, 2, 0, 0),
    ("f16", 2, 10, 10, 128, 5, 1, 2, 100, 0, 4, 64),
    ("f8e4m3", 2, 9, 9, 320, 3, 1, 1, 70, 1, 2, 256),   # last block reaches past C_in: zero tail
    ("bf16", 1, 9, 9, 80, 3, 1, 1, 3, 2, 1, 64),           # 64-B rows, partial last block
    ("f8e4m3", 1, 11, 11, 128, 3, 2, 1, 0, 2, 0, 0),
]


def _expected(xbits, m0, tap_r, tap_s, c0, bk, stride, pad, R):
    N, H, W, C = xbits.shape
    Ho = (H + 2 * pad - R) // stride + 1
    Wo = (W + 2 * pad - R) // stride + 1
    out = np.zeros((128, bk), dtype=xbits.dtype)
    for i in range(128):
        m = m0 + i
        n, rem = divmod(m, Ho * Wo)
        oy, ox = divmod(rem, Wo)
        iy = oy * stride - pad + tap_r
        ix = ox * stride - pad + tap_s
        if n < N and 0 <= iy < H and 0 <= ix < W:
            hi = min(c0 + bk, C)
            out[i, :hi - c0] = xbits[n, iy, ix, c0:hi]      # channels past C_in read as zero
    return out


@pytest.mark.parametrize("case", CASES)
def test_im2col_tile_matches_numpy_gather(case):
    dt, N, H, W, C, R, st, pd, m0, tr, ts, c0 = case
    gen = torch.Generator().manual_seed(7)
    x = torch.randn((N, H, W, C), generator=gen).to(synthetic.TORCH_DTYPES[dt])
    xbits = synthetic.raw_bits(x)
    xd = x.cuda()
    out = torch.zeros(128 * 128, dtype=torch.uint8, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    bk = ctypes.c_int(0)
    lib = _lib.lib()
    status = lib.conv_testing_im2col_tile(
        ctypes.c_void_p(xd.data_ptr()), N, H, W, C, _lib.DTYPE_CODES[dt], R, R, _lib.pair((st, st)),
        _lib.pair((pd, pd)), m0, tr, ts, c0, ctypes.c_void_p(out.data_ptr()), ctypes.byref(bk),
        ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == 0, lib.conv_status_string(status)
    assert int(ws[:4].view(torch.int32).item()) == 0
    elt = synthetic.ELT_BYTES[dt]
    got = out[:128 * bk.value * elt].cpu().numpy().view(xbits.dtype).reshape(128, bk.value)
    want = _expected(xbits, m0, tr, ts, c0, bk.value, st, pd, R)
    mism = np.argwhere(got != want)
    assert mism.size == 0, "first mismatching (row, channel): %s" % mism[:6].tolist()
