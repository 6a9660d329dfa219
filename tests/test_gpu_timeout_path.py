"""The kernels' bounded-wait failure path, exercised without faulting the GPU.

The test hook makes CTA 0's producer leave its first pipeline stage un-armed
(for CTA pairs: both CTAs of the first pair leave it un-armed and unloaded),
so the MMA warp's wait on that stage can only end by running out of time (a
few milliseconds here).  The kernel must then record the timeout in the
workspace status word, stop its other roles, let its copies in flight land,
release its tensor memory and return; the host reads CONV_ERR_DEVICE_TIMEOUT
from conv_check_device_status.  A normal launch afterwards, in the same
context, must still produce the right answer.
"""
import ctypes

import pytest
import torch

import transposed_conv_implicit_gb300 as cg
from tests import _harness as H
from tests.test_gpu_parity import _fwd, _tr, streamk_workspace
from transposed_conv_implicit_gb300 import _lib, synthetic

pytestmark = pytest.mark.gpu

TIMEOUT_NS = 5_000_000   # 5 ms per wait

CASES = [
    # the row-window loader with a residual source in flight
    _fwd("window_res", "bf16", 2, 13, 13, 64, 64, 3, 1, 1, res=True, beta=1.0),
    # the im2col loader, several C_out tiles, direct epilogue
    _fwd("im2col_s2", "bf16", 2, 13, 11, 64, 272, 3, 2, 1, layout="FCRS"),
    # per-phase maps of the transposed convolution, fp8 kind
    _tr("transposed_e4m3", "f8e4m3", 2, 8, 8, 64, 64, 4, 2, 1),
    # the row-tap kernel (few output channels)
    _fwd("rowtap_head", "bf16", 1, 20, 140, 128, 3, 3, 1, 1),
    # the depthwise 3x3 tile kernel (CUDA cores, TMA boxes)
    _fwd("depthwise_tiles", "bf16", 2, 20, 40, 64, 64, 3, 1, 1, groups=64),
]


# Cases run again on CTA pairs (clusters of two CTAs sharing 256-row tiles):
# there rank 1's epilogue and producers time out in turn once rank 0's MMA
# warp stops, and both CTAs meet at the exit cluster barrier.
PAIR_CASES = [
    _fwd("pair_e4m3_s2", "f8e4m3", 2, 13, 13, 64, 64, 3, 2, 1),
    _fwd("pair_cout512_silu", "bf16", 1, 12, 12, 64, 512, 3, 1, 1, epi="silu"),
    # direct-store epilogue with a residual source
    _fwd("pair_cout17_res", "bf16", 2, 10, 10, 32, 17, 3, 1, 1, res=True, beta=0.5),
    _tr("pair_transposed_relu", "f16", 2, 9, 8, 64, 64, 4, 2, 1, epi="relu"),
]


# Stream-K forced on with the partials never published (fault mode 2): the
# CTAs that finish split tiles wait for them until the limit runs out.  The
# launch after it must be right again: its flags carry a new launch value, so
# the stale partial slots and flags of the failed launch are never taken.
STREAMK_CASES = [
    _fwd("sk_s2_res", "bf16", 2, 13, 11, 64, 96, 3, 2, 1, res=True, beta=0.5),
    _tr("sk_transposed", "f16", 2, 8, 8, 64, 64, 4, 2, 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_timeout_is_reported_and_context_survives(case):
    _timeout_then_normal(case)


@pytest.mark.parametrize("case", STREAMK_CASES, ids=lambda c: c.name)
def test_streamk_partial_timeout_is_reported_and_context_survives(case, tuning):
    tuning("CONV_STREAMK", "1")
    ws = streamk_workspace("cuda:0")
    _timeout_then_normal(case, mode=2, ws=ws)


@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: c.name)
def test_cta_pair_timeout_is_reported_and_context_survives(case, tuning):
    tuning("CONV_PAIR", "1")
    if case.kind == "fwd":   # the planner must put it on CTA pairs on this device
        plan = (ctypes.c_int * 14)()
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        st = _lib.lib().conv_testing_fwd_plan(
            case.N, case.H, case.W, case.C_in, _lib.DTYPE_CODES[case.dtype], case.R, case.S,
            case.C_out, _lib.pair((case.stride,) * 2), _lib.pair(case.pads), int(case.has_residual),
            sms, 256, plan)
        assert st == 0 and plan[12] == 1, list(plan)
    _timeout_then_normal(case)


def _timeout_then_normal(case, mode=1, ws=None):
    inp = synthetic.make_inputs(case)
    if ws is None:
        ws = cg.new_workspace(cg.CONV_STATUS_BYTES, "cuda:0")
    lib = _lib.lib()
    try:
        lib.conv_testing_set_wait_fault(mode, TIMEOUT_NS)
        H.run_gpu(case, inp, workspace=ws)
        status, bits = cg.conv_check_device_status(ws)
    finally:
        lib.conv_testing_set_wait_fault(0, 0)
    assert status == cg.CONV_ERR_DEVICE_TIMEOUT, cg.conv_status_string(status)
    # Which role's wait ran out first (MMA = 2, epilogue = 4, producer = 1,
    # a stream-K partial = 8) depends on timing; at least one did, and
    # nothing else was recorded.  Fault mode 2 always leaves the partial's.
    assert bits != 0 and bits & ~15 == 0, bits
    if mode == 2:
        assert bits & 8, bits

    # The status was cleared by the check; a normal launch is right again.
    out = H.run_gpu(case, inp, workspace=ws)
    status, bits = cg.conv_check_device_status(ws)
    assert status == cg.CONV_OK and bits == 0
    ref = H.oracle_full(case, inp)
    got = H.decode(out.cpu(), case.out_dtype)
    H.assert_parity(case, inp, got, ref, "after a timed-out launch")
    torch.cuda.synchronize()
