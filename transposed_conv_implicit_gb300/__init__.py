"""GB300-native implicit-GEMM NHWC convolution and transposed convolution.

A thin Python binding over libconvgb300.so (include/conv_gb300.h).  The
functions keep the C names and only marshal arguments: torch tensors supply
device pointers, shapes and the current CUDA stream; every step of the
computation runs in the library's sm_103a kernels.  Nothing here computes a
convolution on the CPU, and a missing library raises instead of falling back.

Layouts: input [N,H,W,C_in]; forward filter FCRS [C_out,C_in,R,S] or RSCF
[R,S,C_in,C_out]; transposed filter RSFC [R,S,C_out,C_in]; output
[N,Ho,Wo,C_out]; all dense.  Dtypes: bfloat16, float16, float8_e4m3fn
(output bfloat16 for fp8 inputs).
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import (CONV_ERR_CUDA, CONV_ERR_DEVICE_TIMEOUT, CONV_ERR_INVALID_VALUE,
                   CONV_ERR_MISALIGNED, CONV_ERR_NOT_SUPPORTED, CONV_ERR_WORKSPACE_TOO_SMALL,
                   CONV_OK, CONV_STATUS_BYTES, ExtensionMissing)

__all__ = [
    "conv2d_fwd", "conv2d_fwd_packed", "conv2d_pack_filter", "conv2d_packed_filter_bytes",
    "conv2d_workspace_size", "conv_streamk_workspace_size", "conv_transposed",
    "conv_transposed_packed",
    "conv_transposed_pack_filter", "conv_transposed_packed_filter_bytes",
    "conv_transposed_workspace_size", "conv_check_device_status", "conv_status_string",
    "ConvError", "ExtensionMissing", "new_workspace", "dtype_name", "library_path",
]


class ConvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, conv_status_string(status)))


def library_path() -> str:
    return _lib.LIB_PATH


def conv_status_string(status: int) -> str:
    return _lib.lib().conv_status_string(int(status)).decode()


def dtype_name(t) -> str:
    import torch
    names = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float8_e4m3fn: "f8e4m3"}
    if t.dtype not in names:
        raise ConvError(CONV_ERR_NOT_SUPPORTED, "dtype %s" % t.dtype)
    return names[t.dtype]


def _code(t) -> int:
    return _lib.DTYPE_CODES[dtype_name(t)]


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, where: str):
    if status != CONV_OK:
        raise ConvError(status, where)


def _need_dense(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ConvError(CONV_ERR_INVALID_VALUE, "tensors must be dense (contiguous)")


def new_workspace(nbytes: int, device):
    """A zeroed uint8 device buffer (the status region must start at zero)."""
    import torch
    return torch.zeros(max(int(nbytes), CONV_STATUS_BYTES), dtype=torch.uint8, device=device)


def conv2d_packed_filter_bytes(r, s, c_in, c_out, dtype: str) -> int:
    return _lib.lib().conv2d_packed_filter_bytes(r, s, c_in, c_out, _lib.DTYPE_CODES[dtype])


def conv2d_workspace_size(r, s, c_in, c_out, dtype: str) -> int:
    return _lib.lib().conv2d_workspace_size(r, s, c_in, c_out, _lib.DTYPE_CODES[dtype])


def conv_streamk_workspace_size() -> int:
    """Extra workspace bytes that enable the stream-K schedule on the current device."""
    return _lib.lib().conv_streamk_workspace_size()


def conv2d_pack_filter(filter, *, filter_is_fcrs: bool, out=None, stream=None):
    """Pack an FCRS/RSCF filter into the K-major [C_out][K] matrix (returns `out`).

    K = R*S*C_in, or, for channel counts the gather loader serves, R runs of
    S*C_in padded to 16 bytes; conv2d_packed_filter_bytes gives the size."""
    import torch
    _need_dense(filter)
    if filter_is_fcrs:
        c_out, c_in, r, s = filter.shape
    else:
        r, s, c_in, c_out = filter.shape
    if out is None:
        nbytes = conv2d_packed_filter_bytes(r, s, c_in, c_out, dtype_name(filter))
        out = torch.empty((c_out, nbytes // (c_out * filter.element_size())), dtype=filter.dtype,
                          device=filter.device)
    _check(_lib.lib().conv2d_pack_filter(_ptr(filter), r, s, c_in, c_out, int(bool(filter_is_fcrs)),
                                         _code(filter), _ptr(out), out.numel() * out.element_size(),
                                         _stream(stream, filter.device)), "conv2d_pack_filter")
    return out


def _fwd_common(input, output, stride, dilation, symmetric_padding, source):
    _need_dense(input, output, source)
    n, h, w, c_in = input.shape
    _, ho, wo, c_out = output.shape
    return n, h, w, c_in, ho, wo, c_out, _lib.pair(stride), _lib.pair(dilation), _lib.pair(symmetric_padding)


def conv2d_fwd(input, filter, output, *, stride=(1, 1), dilation=(1, 1), symmetric_padding=(0, 0),
               num_groups=1, filter_is_fcrs=False, has_residual=False, source=None, beta=0.0,
               epilogue="none", workspace=None, stream=None):
    """output = act(conv(input, filter) + beta*source); packs the filter into the workspace."""
    n, h, w, c_in, ho, wo, c_out, st, dl, pd = _fwd_common(input, output, stride, dilation,
                                                             symmetric_padding, source)
    _need_dense(filter)
    if filter_is_fcrs:
        f_out, f_in, r, s = filter.shape
    else:
        r, s, f_in, f_out = filter.shape
    if f_in * int(num_groups) != c_in or f_out != c_out:
        raise ConvError(CONV_ERR_INVALID_VALUE, "filter shape does not match input/output/groups")
    if workspace is None:
        workspace = new_workspace(conv2d_workspace_size(r, s, c_in, c_out, dtype_name(input)),
                                  input.device)
    _check(_lib.lib().conv2d_fwd(
        _ptr(input), n, h, w, c_in, _code(input), _ptr(filter), r, s, c_out, int(bool(filter_is_fcrs)),
        _ptr(output), ho, wo, _code(output), st, dl, pd, int(num_groups), int(bool(has_residual)),
        _ptr(source), float(beta), _lib.EPILOGUE_CODES[epilogue], _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream, input.device)), "conv2d_fwd")
    return output


def conv2d_fwd_packed(input, packed_filter, output, *, r, s, stride=(1, 1), dilation=(1, 1),
                      symmetric_padding=(0, 0), num_groups=1, has_residual=False, source=None,
                      beta=0.0, epilogue="none", workspace=None, stream=None):
    """As conv2d_fwd with a filter packed by conv2d_pack_filter."""
    n, h, w, c_in, ho, wo, c_out, st, dl, pd = _fwd_common(input, output, stride, dilation,
                                                             symmetric_padding, source)
    _need_dense(packed_filter)
    groups = max(int(num_groups), 1)
    if (packed_filter.numel() * packed_filter.element_size()
            != conv2d_packed_filter_bytes(r, s, c_in // groups, c_out, dtype_name(input))):
        raise ConvError(CONV_ERR_INVALID_VALUE, "packed filter size does not match")
    if workspace is None:
        workspace = new_workspace(CONV_STATUS_BYTES, input.device)
    _check(_lib.lib().conv2d_fwd_packed(
        _ptr(input), n, h, w, c_in, _code(input), _ptr(packed_filter), r, s, c_out, _ptr(output), ho,
        wo, _code(output), st, dl, pd, int(num_groups), int(bool(has_residual)), _ptr(source),
        float(beta), _lib.EPILOGUE_CODES[epilogue], _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream, input.device)),
        "conv2d_fwd_packed")
    return output


def conv_transposed_packed_filter_bytes(r, s, c_in, c_out, stride, padding, dtype: str,
                                        dilation=(1, 1)) -> int:
    return _lib.lib().conv_transposed_packed_filter_bytes_dilated(
        r, s, c_in, c_out, _lib.pair(stride), _lib.pair(dilation), _lib.pair(padding),
        _lib.DTYPE_CODES[dtype])


def conv_transposed_workspace_size(r, s, c_in, c_out, stride, padding, dtype: str,
                                   dilation=(1, 1)) -> int:
    return _lib.lib().conv_transposed_workspace_size_dilated(
        r, s, c_in, c_out, _lib.pair(stride), _lib.pair(dilation), _lib.pair(padding),
        _lib.DTYPE_CODES[dtype])


def conv_transposed_pack_filter(filter_rsfc, *, stride, padding, dilation=(1, 1), out=None,
                                stream=None):
    """Pack an RSFC filter into per-phase K-major matrices (returns `out`).

    The packing depends on stride, dilation and padding: conv_transposed_packed
    must be called with the same three."""
    import torch
    _need_dense(filter_rsfc)
    r, s, c_out, c_in = filter_rsfc.shape
    dt = dtype_name(filter_rsfc)
    nbytes = conv_transposed_packed_filter_bytes(r, s, c_in, c_out, stride, padding, dt, dilation)
    if nbytes == 0:
        raise ConvError(CONV_ERR_NOT_SUPPORTED, "conv_transposed_pack_filter")
    if out is None:
        out = torch.empty(nbytes // filter_rsfc.element_size(), dtype=filter_rsfc.dtype,
                          device=filter_rsfc.device)
    _check(_lib.lib().conv_transposed_pack_filter_dilated(
        _ptr(filter_rsfc), r, s, c_in, c_out, _lib.pair(stride), _lib.pair(dilation),
        _lib.pair(padding), _code(filter_rsfc), _ptr(out), out.numel() * out.element_size(),
        _stream(stream, filter_rsfc.device)), "conv_transposed_pack_filter")
    return out


def conv_transposed(input, filter_rsfc, output, *, stride=(1, 1), dilation=(1, 1), padding=(0, 0),
                    has_residual=False, source=None, beta=0.0, epilogue="none", workspace=None,
                    stream=None):
    """Transposed conv (backward-data of the forward conv) with an RSFC filter."""
    n, h, w, c_in, ho, wo, c_out, st, dl, pd = _fwd_common(input, output, stride, dilation, padding,
                                                             source)
    _need_dense(filter_rsfc)
    r, s, f_out, f_in = filter_rsfc.shape
    if f_in != c_in or f_out != c_out:
        raise ConvError(CONV_ERR_INVALID_VALUE, "filter shape does not match input/output")
    if workspace is None:
        workspace = new_workspace(conv_transposed_workspace_size(r, s, c_in, c_out, stride, padding,
                                                                 dtype_name(input), dilation),
                                  input.device)
    _check(_lib.lib().conv_transposed(
        _ptr(input), n, h, w, c_in, _code(input), _ptr(filter_rsfc), r, s, c_out, _ptr(output), ho, wo,
        _code(output), st, dl, pd, int(bool(has_residual)), _ptr(source), float(beta),
        _lib.EPILOGUE_CODES[epilogue], _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream, input.device)), "conv_transposed")
    return output


def conv_transposed_packed(input, packed_filter, output, *, r, s, stride=(1, 1), dilation=(1, 1),
                           padding=(0, 0), has_residual=False, source=None, beta=0.0,
                           epilogue="none", workspace=None, stream=None):
    """As conv_transposed with a filter packed by conv_transposed_pack_filter."""
    n, h, w, c_in, ho, wo, c_out, st, dl, pd = _fwd_common(input, output, stride, dilation, padding,
                                                             source)
    _need_dense(packed_filter)
    if workspace is None:
        workspace = new_workspace(CONV_STATUS_BYTES, input.device)
    _check(_lib.lib().conv_transposed_packed(
        _ptr(input), n, h, w, c_in, _code(input), _ptr(packed_filter), r, s, c_out, _ptr(output), ho,
        wo, _code(output), st, dl, pd, int(bool(has_residual)), _ptr(source), float(beta),
        _lib.EPILOGUE_CODES[epilogue], _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream, input.device)), "conv_transposed_packed")
    return output


def conv_check_device_status(workspace, stream=None):
    """Synchronise, read and clear the workspace status word: returns (status, raw bits)."""
    bits = ctypes.c_uint(0)
    status = _lib.lib().conv_check_device_status(_ptr(workspace), _stream(stream, workspace.device),
                                                 ctypes.byref(bits))
    return status, bits.value


class BoundCall:
    """A C-ABI call with its arguments marshalled once (pointers, shapes,
    stream).  Calling it issues the same asynchronous launch again; the
    tensors it was bound to must stay alive."""

    def __init__(self, fn, args, name, keep):
        self._fn, self._args, self._name, self._keep = fn, args, name, keep

    def __call__(self):
        status = self._fn(*self._args)
        if status != CONV_OK:
            raise ConvError(status, self._name)


def bind_conv2d_fwd_packed(input, packed_filter, output, *, r, s, stride=(1, 1), dilation=(1, 1),
                           symmetric_padding=(0, 0), num_groups=1, has_residual=False, source=None,
                           beta=0.0, epilogue="none", workspace=None, stream=None) -> BoundCall:
    """conv2d_fwd_packed with its arguments bound, for repeated launches."""
    n, h, w, c_in, ho, wo, c_out, st, dl, pd = _fwd_common(input, output, stride, dilation,
                                                             symmetric_padding, source)
    if workspace is None:
        workspace = new_workspace(CONV_STATUS_BYTES, input.device)
    args = (_ptr(input), n, h, w, c_in, _code(input), _ptr(packed_filter), r, s, c_out, _ptr(output),
            ho, wo, _code(output), st, dl, pd, int(num_groups), int(bool(has_residual)), _ptr(source),
            float(beta), _lib.EPILOGUE_CODES[epilogue], _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream, input.device))
    return BoundCall(_lib.lib().conv2d_fwd_packed, args, "conv2d_fwd_packed",
                     (input, packed_filter, output, source, workspace))


def bind_conv_transposed_packed(input, packed_filter, output, *, r, s, stride=(1, 1),
                                dilation=(1, 1), padding=(0, 0), has_residual=False, source=None,
                                beta=0.0, epilogue="none", workspace=None, stream=None) -> BoundCall:
    """conv_transposed_packed with its arguments bound, for repeated launches."""
    n, h, w, c_in, ho, wo, c_out, st, dl, pd = _fwd_common(input, output, stride, dilation, padding,
                                                             source)
    if workspace is None:
        workspace = new_workspace(CONV_STATUS_BYTES, input.device)
    args = (_ptr(input), n, h, w, c_in, _code(input), _ptr(packed_filter), r, s, c_out, _ptr(output),
            ho, wo, _code(output), st, dl, pd, int(bool(has_residual)), _ptr(source), float(beta),
            _lib.EPILOGUE_CODES[epilogue], _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream, input.device))
    return BoundCall(_lib.lib().conv_transposed_packed, args, "conv_transposed_packed",
                     (input, packed_filter, output, source, workspace))
