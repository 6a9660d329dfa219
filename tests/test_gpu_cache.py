"""The prepared-call cache: a call repeated with the same arguments reuses
its prepared launch (plan, encoded tensor maps, grid), and any change that
could alter that launch -- an argument, a pointer, the tuning overrides --
prepares afresh.  Results are bit-identical either way."""
import ctypes

import pytest
import torch

from tests import _harness as H
from transposed_conv_implicit_gb300 import _lib, synthetic
from transposed_conv_implicit_gb300.synthetic import ConvCase, Dist

pytestmark = pytest.mark.gpu

CASE = ConvCase("cache_res", "fwd", "bf16", 2, 12, 10, 64, 48, 3, 3, 1, 1, "RSCF",
                Dist("normal", 1.0), Dist("normal", 1.0 / 576), seed=5151, has_residual=True,
                beta=0.5, src_dist=Dist("normal", 1.0))


def _stats():
    hits, misses = ctypes.c_ulonglong(0), ctypes.c_ulonglong(0)
    _lib.lib().conv_testing_cache_stats(ctypes.byref(hits), ctypes.byref(misses))
    return hits.value, misses.value


def test_repeated_calls_hit_and_changes_miss(tuning):
    import transposed_conv_implicit_gb300 as cg
    inp = synthetic.make_inputs(CASE)
    dev = "cuda:0"
    x, w, src = inp["x"].to(dev), inp["w"].to(dev), inp["src"].to(dev)
    pk = cg.conv2d_pack_filter(w, filter_is_fcrs=False)
    ws = cg.new_workspace(cg.CONV_STATUS_BYTES, dev)
    out = torch.empty(CASE.out_shape, dtype=torch.bfloat16, device=dev)

    def call(beta=0.5, o=out):
        cg.conv2d_fwd_packed(x, pk, o, r=3, s=3, symmetric_padding=(1, 1), has_residual=True,
                             source=src, beta=beta, workspace=ws)
        torch.cuda.synchronize()
        return o.clone()

    first = call()
    h0, m0 = _stats()
    again = [call() for _ in range(3)]
    h1, m1 = _stats()
    assert (h1 - h0, m1 - m0) == (3, 0)
    for a in again:
        assert torch.equal(a.view(torch.int16), first.view(torch.int16))
    call(beta=0.25)                                       # another beta: a new entry
    other = torch.empty_like(out)
    call(o=other)                                         # another output pointer: a new entry
    h2, m2 = _stats()
    assert (h2 - h1, m2 - m1) == (0, 2)
    tuning("CONV_MAX_STAGES", "3")                        # new tuning: prepared afresh
    third = call()
    h3, m3 = _stats()
    assert (h3 - h2, m3 - m2) == (0, 1)
    assert torch.equal(third.view(torch.int16), first.view(torch.int16))
    H.assert_parity(CASE, inp, H.decode(first.cpu(), "bf16"), H.oracle_full(CASE, inp))
