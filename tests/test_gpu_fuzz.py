"""Seeded random shapes inside the documented gates, every element against
the fp64 oracle: forward convs over dtypes, channel counts (TMA channel
blocks, partial blocks and the gather loader's narrow rows), filter sizes,
strides, padding, dilation, channel groups, residual sources and epilogues,
and transposed convs over strides (per axis), dilation and output padding.
The shapes stay small enough for the oracle; the planner picks the loader,
tile shape, CTA pairs and kernel as it would for a user."""
import random

import pytest
import torch

from tests import _harness as H
from tests.test_gpu_parity import _fwd, _tr
from transposed_conv_implicit_gb300 import synthetic

pytestmark = pytest.mark.gpu

ELT = {"bf16": 2, "f16": 2, "f8e4m3": 1}


def _fwd_cases(n_cases, seed):
    rng = random.Random(seed)
    cases = []
    while len(cases) < n_cases:
        dt = rng.choice(["bf16", "f16", "f8e4m3"])
        c_in = rng.choice([3, 5, 8, 16, 24, 32, 48, 64, 80, 96, 128, 160, 192, 320])
        groups = 1
        if rng.random() < 0.2:
            groups = rng.choice([g for g in (2, 4, 8, 16) if c_in % g == 0] or [1])
        c_out = rng.choice([1, 3, 8, 16, 17, 32, 48, 64, 96, 128, 160, 200, 256, 300])
        if c_out % groups:
            c_out = groups * max(1, c_out // groups)
        r = rng.choice([1, 3, 3, 5])
        s_ = rng.choice([r, r, 1, 3])
        st = rng.choice([1, 1, 2])
        row_bytes = c_in // groups * ELT[dt]
        gather = groups == 1 and (row_bytes % 16 != 0 or row_bytes < 32)
        dil = 1 if gather else rng.choice([1, 1, 2])
        pd = rng.randint(0, dil * (r - 1))
        if s_ != r:
            pd = min(pd, dil * (s_ - 1))   # symmetric padding must suit both axes
        n = rng.choice([1, 2])
        h = rng.randint(dil * (r - 1) + 1, 20)
        w = rng.randint(dil * (s_ - 1) + 1, rng.choice([20, 40, 140]))
        ho = (h + 2 * pd - dil * (r - 1) - 1) // st + 1
        wo = (w + 2 * pd - dil * (s_ - 1) - 1) // st + 1
        if ho < 1 or wo < 1:
            continue
        work = n * ho * wo * c_out * r * s_ * c_in // groups
        if work > 60_000_000:
            continue
        # (Channel groups narrower than whole 128-byte blocks run on the
        # direct kernel, whose fp32 filter slice must fit in 200 KB: the gate.)
        if groups > 1 and r * s_ * (c_in // groups) * 64 * 4 > 200 * 1024:
            continue
        res = rng.random() < 0.4
        epi = rng.choice(["none", "relu", "silu"])
        layout = rng.choice(["RSCF", "FCRS"])
        name = "fz_f_%d_%s_c%d_f%d_g%d_%dx%d_s%d_p%d_d%d" % (len(cases), dt, c_in, c_out, groups,
                                                               r, s_, st, pd, dil)
        cases.append(_fwd(name, dt, n, h, w, c_in, c_out, r, st, pd, layout=layout, res=res,
                          beta=rng.choice([0.5, 1.0, -0.75]) if res else 0.0, epi=epi,
                          seed=rng.randint(1, 10_000), S=s_, dil=dil, groups=groups))
    return cases


def _tr_cases(n_cases, seed):
    rng = random.Random(seed)
    cases = []
    while len(cases) < n_cases:
        dt = rng.choice(["bf16", "f16", "f8e4m3"])
        c_in = rng.choice([c for c in (16, 32, 48, 64, 96, 128, 256) if c * ELT[dt] >= 32])
        c_out = rng.choice([3, 8, 16, 32, 40, 64, 128])
        r = rng.choice([2, 3, 4, 5])
        st = rng.choice([1, 2, 2, 3])
        st_w = rng.choice([st, st, 1, 2])
        if st * st_w > 16:
            continue
        dil = rng.choice([1, 1, 2])
        pd = rng.randint(0, dil * (r - 1))
        n = rng.choice([1, 2])
        h, w = rng.randint(2, 10), rng.randint(2, 12)
        extra = rng.randint(0, st - 1)
        extra_w = rng.randint(0, st_w - 1)
        ho = (h - 1) * st - 2 * pd + dil * (r - 1) + 1 + extra
        wo = (w - 1) * st_w - 2 * pd + dil * (r - 1) + 1 + extra_w
        if ho < 1 or wo < 1:
            continue
        res = rng.random() < 0.3
        epi = rng.choice(["none", "relu", "silu"])
        name = "fz_t_%d_%s_c%d_f%d_%dx%d_s%dx%d_p%d_d%d" % (len(cases), dt, c_in, c_out, r, r, st,
                                                            st_w, pd, dil)
        cases.append(_tr(name, dt, n, h, w, c_in, c_out, r, st, pd, extra, res=res,
                         beta=rng.choice([0.5, 1.0]) if res else 0.0, epi=epi,
                         seed=rng.randint(1, 10_000), dil=dil, st_w=st_w, extra_w=extra_w))
    return cases


FUZZ_CASES = _fwd_cases(64, seed=20261203) + _tr_cases(32, seed=20261204)


@pytest.mark.parametrize("case", FUZZ_CASES, ids=lambda c: c.name)
def test_random_shape_every_element(case):
    inp = synthetic.make_inputs(case)
    out = H.run_gpu(case, inp)
    torch.cuda.synchronize()
    got = H.decode(out.cpu(), case.out_dtype)
    ref = H.oracle_full(case, inp)
    H.assert_parity(case, inp, got, ref)
