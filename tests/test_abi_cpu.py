"""The C ABI without a GPU: the library builds, loads and exports every symbol
the headers declare, and host-side validation returns the documented status
codes before any CUDA call (the pointers here are never dereferenced).

Gates from "dispatch_amd_4wave_conv2d" (Parameters, Args) and the transposed
conv's shape rule; see include/conv_gb300.h.
"""
import ctypes
import os
import re

import pytest

import transposed_conv_implicit_gb300 as cg
from transposed_conv_implicit_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, NOTSUP, MISALIGNED, WS_SMALL = 0, 1, 2, 3, 4
BF16, F16, F8 = 0, 1, 2

# Fake, 16-byte-aligned device addresses: validation never dereferences them.
A, B, C, D, WS = (ctypes.c_void_p(0x10000 * k) for k in (1, 2, 3, 4, 5))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.lib()


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert "conv2d_fwd" in declared and "conv_transposed" in declared
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(_lib.EXPORTS) == declared


def test_status_strings(lib):
    for code, name in [(0, "CONV_OK"), (1, "CONV_ERR_INVALID_VALUE"), (2, "CONV_ERR_NOT_SUPPORTED"),
                       (3, "CONV_ERR_MISALIGNED"), (4, "CONV_ERR_WORKSPACE_TOO_SMALL"),
                       (5, "CONV_ERR_CUDA"), (6, "CONV_ERR_DEVICE_TIMEOUT")]:
        assert lib.conv_status_string(code).decode() == name


def test_sizes(lib):
    assert lib.conv2d_packed_filter_bytes(3, 3, 64, 64, BF16) == 3 * 3 * 64 * 64 * 2
    assert lib.conv2d_packed_filter_bytes(3, 3, 320, 320, F8) == 3 * 3 * 320 * 320
    assert lib.conv2d_workspace_size(3, 3, 64, 64, BF16) == 256 + 73728
    assert lib.conv2d_packed_filter_bytes(0, 3, 64, 64, BF16) == 0
    # 4x4 filter, stride 2: four phases of 2x2 taps -> K = 4*C_in per phase.
    assert lib.conv_transposed_packed_filter_bytes(4, 4, 256, 128, _lib.pair((2, 2)),
                                                   _lib.pair((1, 1)), F16) == 4 * 128 * 1024 * 2
    # 3x3 filter, stride 2, pad 1: phase taps 1x1,1x2,2x1,2x2 -> K_max = 4*C_in.
    assert lib.conv_transposed_packed_filter_bytes(3, 3, 64, 32, _lib.pair((2, 2)),
                                                   _lib.pair((1, 1)), BF16) == 4 * 32 * 256 * 2
    assert lib.conv_transposed_packed_filter_bytes(3, 3, 64, 32, _lib.pair((1, 1)),
                                                   _lib.pair((1, 1)), BF16) == 32 * 576 * 2


def fwd(lib, *, inp=A, n=2, h=8, w=8, c=64, dt=BF16, flt=B, r=3, s=3, f=64, fcrs=0, out=C,
        ho=None, wo=None, odt=None, stride=(1, 1), dil=(1, 1), pad=(1, 1), groups=1, res=0,
        src=None, beta=0.0, epi=0, ws=WS, ws_bytes=1 << 20, packed=False):
    odt = (BF16 if dt == F8 else dt) if odt is None else odt
    if ho is None:
        ho = (h + 2 * pad[0] - r) // stride[0] + 1 if stride[0] > 0 else 1
    if wo is None:
        wo = (w + 2 * pad[1] - s) // stride[1] + 1 if stride[1] > 0 else 1
    src = ctypes.c_void_p(0) if src is None else src
    tail = (_lib.pair(stride), _lib.pair(dil), _lib.pair(pad), groups, res, src, beta, epi, ws,
            ws_bytes, None)
    if packed:
        return lib.conv2d_fwd_packed(inp, n, h, w, c, dt, flt, r, s, f, out, ho, wo, odt, *tail)
    return lib.conv2d_fwd(inp, n, h, w, c, dt, flt, r, s, f, fcrs, out, ho, wo, odt, *tail)


@pytest.mark.parametrize("kw,want", [
    (dict(inp=ctypes.c_void_p(0)), INVALID),
    (dict(out=ctypes.c_void_p(0)), INVALID),
    (dict(ws=ctypes.c_void_p(0)), INVALID),
    (dict(res=1), INVALID),                                   # residual without a source
    (dict(inp=ctypes.c_void_p(0x10008)), MISALIGNED),
    (dict(res=1, src=ctypes.c_void_p(0x20004)), MISALIGNED),
    (dict(n=0), INVALID),
    (dict(c=-64), INVALID),
    (dict(ho=7), INVALID),                                    # inconsistent output size
    (dict(epi=3), INVALID),
    (dict(stride=(3, 3)), NOTSUP),
    (dict(stride=(1, 2)), NOTSUP),
    (dict(dil=(33, 33)), NOTSUP),
    (dict(c=20, dil=(1, 2)), NOTSUP),                          # gather loader needs dil_w = 1
    (dict(pad=(1, 3)), NOTSUP),                               # pad beyond the filter extent - 1
    (dict(pad=(3, 3)), NOTSUP),
    (dict(r=1, s=1, pad=(1, 1)), NOTSUP),
    (dict(c=60, f=60, groups=4, r=8, s=8, h=16, w=16), NOTSUP),  # direct kernel's filter slice > 200 KB
    (dict(groups=3), INVALID),                                # 64 channels do not split in 3
    (dict(groups=0), INVALID),
    (dict(dt=F8, odt=F8), NOTSUP),                            # fp8 must write bf16
    (dict(dt=BF16, odt=F16), NOTSUP),
    (dict(dt=7), NOTSUP),
    (dict(r=33, s=33, h=40, w=40), NOTSUP),
    (dict(ws_bytes=1000), WS_SMALL),                          # cannot hold the packed filter
    (dict(ws_bytes=100, packed=True), WS_SMALL),
])
def test_forward_validation(lib, kw, want):
    assert fwd(lib, **kw) == want


def tr(lib, *, n=2, h=8, w=8, c=64, dt=F16, r=4, s=4, f=32, ho=None, wo=None, stride=(2, 2),
       dil=(1, 1), pad=(1, 1), res=0, src=None, epi=0, ws_bytes=1 << 22, odt=None):
    odt = (BF16 if dt == F8 else dt) if odt is None else odt
    if ho is None:
        ho = (h - 1) * stride[0] - 2 * pad[0] + dil[0] * (r - 1) + 1
    if wo is None:
        wo = (w - 1) * stride[1] - 2 * pad[1] + dil[1] * (s - 1) + 1
    src = ctypes.c_void_p(0) if src is None else src
    return lib.conv_transposed(A, n, h, w, c, dt, B, r, s, f, C, ho, wo, odt, _lib.pair(stride),
                               _lib.pair(dil), _lib.pair(pad), res, src, 0.0, epi, WS, ws_bytes,
                               None)


@pytest.mark.parametrize("kw,want", [
    (dict(ho=13), INVALID),                   # below (h-1)s - 2p + r
    (dict(ho=18), INVALID),                   # output padding must be < stride
    # Accepted shapes stop at the (deliberately too small) workspace, past every shape gate.
    (dict(dil=(2, 2), ws_bytes=512), WS_SMALL),
    (dict(stride=(2, 1), ws_bytes=512), WS_SMALL),   # per-axis strides
    (dict(stride=(3, 3), ws_bytes=512), WS_SMALL),   # 9 phases: three launches
    (dict(stride=(4, 4), pad=(0, 0), ws_bytes=512), WS_SMALL),
    (dict(dil=(33, 1)), NOTSUP),
    (dict(pad=(4, 4)), NOTSUP),               # pad > dil*(r-1)
    (dict(dil=(2, 2), pad=(7, 7)), NOTSUP),
    (dict(stride=(5, 4)), NOTSUP),            # 20 phases
    (dict(stride=(0, 2)), NOTSUP),
    (dict(c=8), NOTSUP),
    (dict(dt=F8, odt=F16), NOTSUP),
    (dict(res=1), INVALID),
    (dict(ws_bytes=512), WS_SMALL),
])
def test_transposed_validation(lib, kw, want):
    assert tr(lib, **kw) == want


def test_transposed_packed_sizes_with_dilation_and_stride(lib):
    """Packed layout [stride_h*stride_w phases][c_out][K_max]: with stride 2 and
    dilation 2 one output phase per axis gets every tap and the other none
    (K_max = 4*4*64); stride 4 with a 4x4 filter gives 16 phases of one tap."""
    nb = lambda r, s, c, f, st, dl, pd, dt: lib.conv_transposed_packed_filter_bytes_dilated(
        r, s, c, f, _lib.pair(st), _lib.pair(dl), _lib.pair(pd), dt)
    assert nb(4, 4, 64, 32, (2, 2), (2, 2), (1, 1), F16) == 4 * 32 * (16 * 64) * 2
    assert nb(4, 4, 64, 32, (4, 4), (1, 1), (0, 0), F16) == 16 * 32 * 64 * 2
    assert nb(3, 3, 64, 16, (3, 3), (2, 2), (2, 2), F8) == 9 * 16 * 64 * 1   # gcd(2, 3) = 1: one tap each
    assert nb(4, 4, 64, 32, (2, 2), (1, 1), (1, 1), F16) == \
        lib.conv_transposed_packed_filter_bytes(4, 4, 64, 32, _lib.pair((2, 2)), _lib.pair((1, 1)), F16)
    assert nb(4, 4, 64, 32, (5, 4), (1, 1), (1, 1), F16) == 0                 # 20 phases
    assert lib.conv_transposed_workspace_size_dilated(
        4, 4, 64, 32, _lib.pair((2, 2)), _lib.pair((2, 2)), _lib.pair((1, 1)), F16) == 256 + 4 * 32 * 1024 * 2


def test_pack_validation(lib):
    assert lib.conv2d_pack_filter(B, 3, 3, 64, 64, 0, BF16, D, 100, None) == WS_SMALL
    assert lib.conv2d_pack_filter(None, 3, 3, 64, 64, 0, BF16, D, 1 << 20, None) == INVALID
    assert lib.conv2d_pack_filter(ctypes.c_void_p(0x20002), 3, 3, 64, 64, 0, BF16, D, 1 << 20,
                                  None) == MISALIGNED
    assert lib.conv_transposed_pack_filter(B, 4, 4, 64, 32, _lib.pair((2, 2)), _lib.pair((1, 1)),
                                           F16, D, 64, None) == WS_SMALL
    assert lib.conv_transposed_pack_filter(B, 4, 4, 64, 32, _lib.pair((5, 4)), _lib.pair((1, 1)),
                                           F16, D, 1 << 20, None) == NOTSUP   # 20 phases
    assert lib.conv_transposed_pack_filter_dilated(
        B, 4, 4, 64, 32, _lib.pair((2, 2)), _lib.pair((2, 2)), _lib.pair((7, 1)), F16, D, 1 << 20,
        None) == NOTSUP                                                        # pad > dil*(r-1)
    assert lib.conv_transposed_pack_filter_dilated(
        B, 4, 4, 64, 32, _lib.pair((3, 3)), _lib.pair((2, 2)), _lib.pair((1, 1)), F16, D, 64,
        None) == WS_SMALL                                                      # accepted shape


def _plan(lib, n, h, w, c, dt, r, f, st, pd, res=0, sms=148, ws=256):
    out = (ctypes.c_int * 14)()
    assert lib.conv_testing_fwd_plan(n, h, w, c, dt, r, r, f, _lib.pair((st, st)), _lib.pair((pd, pd)),
                                     res, sms, ws, out) == OK
    keys = ("bn", "bk", "stages", "smem", "tiles", "grid", "tmem", "epi", "bres", "srcb", "stgb",
            "loader", "pair", "streamk")
    return dict(zip(keys, list(out)))


def test_tile_plans_for_the_workloads(lib):
    """The dispatcher's tile choices for the benchmark shapes (152 SMs)."""
    p = _plan(lib, 32, 56, 56, 64, BF16, 3, 64, 1, 1, res=1, sms=152)   # ResNet 3x3 + residual:
    assert (p["bn"], p["bk"], p["tiles"], p["tmem"]) == (64, 64, 448, 256)   # row windows of 4 rows
    assert (p["epi"], p["bres"]) == (3, 1)                 # window TMA epilogue, filter resident
    assert p["smem"] <= 227 * 1024 and p["stages"] >= 2
    p = _plan(lib, 32, 56, 56, 64, BF16, 3, 128, 2, 1, sms=152)          # downsample: 147 KB filter
    assert (p["bn"], p["tiles"], p["epi"], p["bres"]) == (128, 98, 1, 0) and p["stages"] >= 4
    p = _plan(lib, 16, 64, 64, 320, F8, 3, 320, 1, 1, res=1, sms=152)    # fp8: 2 x 160 columns,
    assert (p["bn"], p["bk"], p["tiles"], p["tmem"], p["epi"]) == (160, 128, 512, 512, 1)  # 128-ch blocks
    assert p["pair"] == 1                                  # on CTA pairs: 256-row tiles
    p = _plan(lib, 1, 512, 512, 128, BF16, 3, 3, 1, 1, sms=152)          # C_out = 3: row-tap kernel,
    assert (p["loader"], p["bn"], p["bk"], p["stgb"]) == (3, 48, 64, 18)  # N = 3 rows x 16, bands of 18
    assert p["tiles"] == 5 * 29 and p["grid"] == 145 and p["tmem"] == 512   # one wave: 5 segments x 29 bands
    p = _plan(lib, 1, 16, 16, 16, BF16, 3, 16, 1, 1, sms=152)            # 32-byte channel rows
    assert (p["bn"], p["bk"], p["grid"]) == (16, 16, p["tiles"])
    for args in [(1, 256, 256, 512, BF16, 3, 512, 1, 1), (8, 128, 128, 128, F16, 5, 128, 2, 2)]:
        q = _plan(lib, *args, sms=152)
        assert q["smem"] <= 227 * 1024 and q["stages"] >= 3 and q["tmem"] <= 512


def test_row_tap_gate(lib, tuning):
    """Few output channels (S * C_out <= 32), stride 1, dilation 1, 128-byte
    channel blocks and more than one tap take the row-tap kernel; the rest,
    or CONV_ROWTAP=-1, the implicit GEMM's masked edge tile."""
    assert _plan(lib, 1, 40, 40, 64, BF16, 3, 10, 1, 1)["loader"] == 3      # S * C_out = 30
    assert _plan(lib, 1, 40, 40, 128, F8, 3, 8, 1, 1)["loader"] == 3        # fp8: 128 channels
    q = _plan(lib, 1, 40, 40, 64, BF16, 3, 8, 1, 1)                          # g16 = 32: N = 96,
    assert (q["loader"], q["bn"]) == (3, 96) and q["stgb"] <= 4              # bands of <= 4 rows
    assert _plan(lib, 1, 40, 40, 64, BF16, 3, 11, 1, 1)["loader"] != 3      # S * C_out = 33
    assert _plan(lib, 1, 40, 40, 64, BF16, 3, 3, 2, 1)["loader"] != 3       # stride 2
    assert _plan(lib, 1, 40, 40, 32, BF16, 3, 3, 1, 1)["loader"] != 3       # 64-byte channel rows
    assert _plan(lib, 1, 40, 40, 64, BF16, 1, 3, 1, 0)["loader"] != 3       # a single tap
    tuning("CONV_ROWTAP", "-1")
    p = _plan(lib, 1, 512, 512, 128, BF16, 3, 3, 1, 1, sms=152)              # masked 16-wide tile
    assert (p["loader"], p["bn"], p["bk"], p["tiles"], p["epi"], p["bres"]) == (0, 16, 64, 1024, 0, 1)


def test_row_tap_plan_invariants(lib, tuning):
    """Over many eligible shapes: the band fits the TMEM budget (two buffers
    of g16 * (band + 2R - 2) columns within the allocation), the tile count
    covers every output row and column segment, and shared memory fits."""
    import random
    tuning("CONV_ROWTAP", None)
    tuning("CONV_ROWTAP_BAND", None)
    rng = random.Random(7)
    seen = multi = 0
    for _ in range(300):
        r = rng.choice([1, 2, 3, 5, 7])
        s_ = rng.choice([1, 2, 3, 5])
        if r * s_ < 2:
            continue
        dt = rng.choice([BF16, F16, F8])
        c = (128 // (1 if dt == F8 else 2)) * rng.choice([1, 2, 3])
        f = rng.randint(1, 32 // s_)
        n, h, w = rng.randint(1, 3), rng.randint(r, 70), rng.randint(s_, 300)
        pd = rng.randint(0, r - 1) if r == s_ else 0
        out = (ctypes.c_int * 14)()
        st = lib.conv_testing_fwd_plan(n, h, w, c, dt, r, s_, f, _lib.pair((1, 1)), _lib.pair((pd, pd)),
                                       0, 152, 256, out)
        assert st == OK
        if out[11] != 3:
            continue
        seen += 1
        mma_n, band, tiles, tmem, smem = out[0], out[10], out[4], out[6], out[3]
        g16 = mma_n // r
        assert g16 in (16, 32) and g16 >= s_ * f
        # Two accumulator buffers, or one (taller bands) when every CTA has one tile.
        cols = g16 * (band + 2 * r - 2)
        assert 1 <= band <= 24 and cols <= tmem <= 512
        assert 2 * cols <= tmem or (tiles <= 152 and out[5] == tiles)
        ho, wo = h + 2 * pd - r + 1, w + 2 * pd - s_ + 1
        seg = 128 - (s_ - 1)
        assert tiles == n * -(-ho // band) * -(-wo // seg)
        assert smem <= 227 * 1024 and out[2] >= 2
        # An A stage holds one channel block, or every block of the input row
        # segment (then at least four such stages fit).
        c_blocks = c * (1 if dt == F8 else 2) // 128
        blocks = out[9]
        assert blocks in (1, c_blocks)
        assert blocks == 1 or out[2] >= 4
        assert out[2] * blocks * 128 * 128 <= smem
        multi += blocks > 1
    assert seen > 100 and multi > 20


def test_cta_pair_plan_invariants(lib, tuning):
    """CTA pairs forced on over many shapes: 256-row tiles over every C_out
    tile, an even grid of at most the SMs, accumulators of 2 x bn columns
    within TMEM, shared memory within the limit; never with the row window
    or the gather loader."""
    import random
    tuning("CONV_PAIR", "1")
    rng = random.Random(11)
    seen = 0
    for _ in range(300):
        dt = rng.choice([BF16, F16, F8])
        c = rng.choice([32, 64, 96, 128, 256, 320])
        f = rng.choice([32, 48, 64, 128, 200, 256, 320, 512])
        r = rng.choice([1, 3, 5])
        st = rng.choice([1, 2])
        pd = rng.randint(0, r - 1)
        n, h, w = rng.randint(1, 4), rng.randint(r, 90), rng.randint(r, 90)
        sms = rng.choice([8, 20, 152])
        out = (ctypes.c_int * 14)()
        if lib.conv_testing_fwd_plan(n, h, w, c, dt, r, r, f, _lib.pair((st, st)), _lib.pair((pd, pd)),
                                     rng.randint(0, 1), sms, 256, out) != OK:
            continue
        p = dict(zip(("bn", "bk", "stages", "smem", "tiles", "grid", "tmem", "epi", "bres", "srcb",
                      "stgb", "loader", "pair"), list(out)))
        if not p["pair"]:
            assert p["loader"] != 0 or p["bn"] < 32 or p["loader"] == 3
            continue
        seen += 1
        assert p["loader"] == 0 and p["bres"] == 0 and p["bn"] >= 32
        ho, wo = (h + 2 * pd - r) // st + 1, (w + 2 * pd - r) // st + 1
        nt = -(-f // p["bn"])
        assert p["tiles"] == -(-(n * ho * wo) // 256) * nt
        assert p["grid"] % 2 == 0 and 2 <= p["grid"] <= sms and p["grid"] <= 2 * p["tiles"]
        assert 2 * p["bn"] <= p["tmem"] <= 512
        assert p["smem"] <= 227 * 1024 and p["stages"] >= 2
    assert seen > 100


def test_cta_pair_plans(lib, tuning):
    """CTA pairs (cta_group::2, 256-row tiles shared by two CTAs) when every
    pair of SMs gets at least 4 tiles and bn = 256; CONV_PAIR=1/0 force."""
    tuning("CONV_PAIR", None)
    vae = (1, 256, 256, 512, BF16, 3, 512, 1, 1)
    p = _plan(lib, *vae, sms=152)
    assert (p["pair"], p["bn"], p["tiles"], p["grid"], p["tmem"]) == (1, 256, 512, 152, 512)
    f5 = (8, 128, 128, 128, 1, 5, 128, 2, 2)                     # 128 pair tiles < 4 x 76
    assert _plan(lib, *f5, sms=152)["pair"] == 0
    assert _plan(lib, *vae, sms=1000)["pair"] == 0              # too few tiles per pair
    tuning("CONV_PAIR", "1")
    q = _plan(lib, *f5, sms=152)
    assert (q["pair"], q["tiles"], q["grid"], q["tmem"]) == (1, 128, 152, 256)
    assert _plan(lib, 3, 30, 30, 64, BF16, 3, 48, 2, 1, sms=5)["grid"] == 4  # even grid: 2 pairs
    assert _plan(lib, 32, 56, 56, 64, BF16, 3, 64, 1, 1, res=1, sms=152)["pair"] == 0  # row window
    assert _plan(lib, 32, 224, 224, 3, BF16, 7, 64, 2, 2, sms=152)["pair"] == 0       # gather
    assert _plan(lib, 2, 9, 9, 64, BF16, 3, 16, 2, 1, sms=152)["pair"] == 0           # bn < 32
    tuning("CONV_PAIR", "0")
    assert _plan(lib, *vae, sms=152)["pair"] == 0


def test_measured_planner_choices(lib, tuning):
    """Plans the measurements picked (each alternative was timed on GB300 and
    ran slower): 256-row gather tiles for the RGB stem (77.8 vs 90.1 us on
    128-row tiles), CTA pairs for the fp8 conv's 160-column tiles (64.5 vs
    61.7 us) with a 7-stage ring and one residual buffer (5 stages and two
    buffers: 60.8 vs 59.3 us), 256-row bn = 128 tiles for the wave-quantised
    fwd5x5 (128-row: 30.5 vs 27.0 us; CTA pairs 31.2)."""
    for name in ("CONV_TILE_M", "CONV_TILE_N", "CONV_PAIR", "CONV_SRC_BUFS", "CONV_MAX_STAGES"):
        tuning(name, None)
    stem = _plan(lib, 32, 224, 224, 3, BF16, 7, 64, 2, 3, sms=152)
    assert (stem["loader"], stem["tiles"], stem["tmem"]) == (2, 32 * 112 * 112 // 256, 256)
    fp8 = _plan(lib, 16, 64, 64, 320, F8, 3, 320, 1, 1, res=1, sms=152)
    assert (fp8["stages"], fp8["srcb"], fp8["pair"]) == (7, 1, 1)
    f5 = _plan(lib, 8, 128, 128, 128, F16, 5, 128, 2, 2, sms=152)
    assert (f5["bn"], f5["tiles"], f5["pair"]) == (128, 128, 0)
    tuning("CONV_SRC_BUFS", "1")   # the override still caps the buffers
    assert _plan(lib, 16, 64, 64, 320, F8, 3, 320, 1, 1, res=1, sms=152)["srcb"] == 1


def test_binding_raises_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(_lib.ExtensionMissing):
        cg.conv_status_string(0)


def test_noalloc_rejects_filters_beyond_its_scratch(lib):
    # 5x5x2048x2048 bf16 packs to 210 MB, far beyond the 8 MiB scratch: rejected before any CUDA call.
    status = lib.conv2d_fwd_noalloc(A, 1, 8, 8, 2048, BF16, B, 5, 5, 2048, 0, C, 8, 8, BF16,
                                    _lib.pair((1, 1)), _lib.pair((1, 1)), _lib.pair((2, 2)), 1, 0,
                                    None, 0.0, 0, None)
    assert status == WS_SMALL
    assert _lib.CONV_NOALLOC_SCRATCH_BYTES == 8 << 20


def test_noalloc_sizes_grouped_filters_by_channels_per_group(lib):
    """A depthwise 3x3 filter over 1024 channels packs to 1024 x 9 x 1 values
    (18 KB), well within the scratch; sized by the total C_in it would claim
    ~18.9 MB and be rejected.  The output size is deliberately inconsistent so
    that the call stops in conv2d_fwd's shape check and never launches,
    whether or not a GPU is present (without one the scratch lookup fails
    first with CONV_ERR_CUDA)."""
    assert lib.conv2d_workspace_size(3, 3, 1, 1024, BF16) <= _lib.CONV_NOALLOC_SCRATCH_BYTES
    assert lib.conv2d_workspace_size(3, 3, 1024, 1024, BF16) > _lib.CONV_NOALLOC_SCRATCH_BYTES
    status = lib.conv2d_fwd_noalloc(A, 1, 8, 8, 1024, BF16, B, 3, 3, 1024, 0, C, 9, 8, BF16,
                                    _lib.pair((1, 1)), _lib.pair((1, 1)), _lib.pair((1, 1)), 1024, 0,
                                    None, 0.0, 0, None)
    assert status in (INVALID, cg.CONV_ERR_CUDA)
    # A group count that does not divide C_in is rejected before any CUDA call.
    status = lib.conv2d_fwd_noalloc(A, 1, 8, 8, 1024, BF16, B, 3, 3, 1024, 0, C, 8, 8, BF16,
                                    _lib.pair((1, 1)), _lib.pair((1, 1)), _lib.pair((1, 1)), 3, 0,
                                    None, 0.0, 0, None)
    assert status == INVALID


def test_gather_loader_plans(lib):
    """Channel rows TMA cannot address (C_in * elt not a multiple of 16 bytes,
    or under 32) go to the gather loader: 128-byte k-blocks over runs of
    S taps x C_in channels padded to 16 bytes."""
    # RGB stem, 7x7 stride 2: runs of 7*3*2 = 42 -> 48 bytes, K = 7*48 = 336 B = 3 k-blocks
    p = _plan(lib, 32, 224, 224, 3, BF16, 7, 64, 2, 2, sms=152)
    assert (p["loader"], p["bk"], p["bn"], p["bres"]) == (2, 64, 64, 1)
    assert p["smem"] <= 227 * 1024 and p["stages"] >= 2
    for c, dt in [(8, BF16), (20, BF16), (1, F16), (16, F8), (5, F8), (3, F16)]:
        q = _plan(lib, 2, 9, 9, c, dt, 3, 24, 1, 1)
        assert q["loader"] == 2 and q["bk"] == 128 // (1 if dt == F8 else 2)
    # TMA-addressable channel rows keep the TMA loaders.
    assert _plan(lib, 2, 9, 9, 24, BF16, 3, 24, 2, 1)["loader"] == 0
    assert _plan(lib, 2, 9, 9, 64, BF16, 3, 64, 1, 1)["loader"] == 1


def test_gather_packed_filter_bytes(lib):
    # per output channel: R runs of ceil16(S * C_in * elt) bytes
    assert lib.conv2d_packed_filter_bytes(7, 7, 3, 64, BF16) == 64 * 7 * 48
    assert lib.conv2d_packed_filter_bytes(3, 3, 20, 8, BF16) == 8 * 3 * 128
    assert lib.conv2d_packed_filter_bytes(3, 3, 5, 4, F8) == 4 * 3 * 16
    assert lib.conv2d_packed_filter_bytes(1, 1, 8, 16, BF16) == 16 * 16
    assert lib.conv2d_workspace_size(7, 7, 3, 64, BF16) == 256 + 64 * 7 * 48


def _cache_stats(lib):
    hits, misses = ctypes.c_ulonglong(0), ctypes.c_ulonglong(0)
    lib.conv_testing_cache_stats(ctypes.byref(hits), ctypes.byref(misses))
    return hits.value, misses.value


def test_failed_calls_are_never_cached(lib):
    """The prepared-call cache stores only successful preparations: a call
    rejected by validation (or unable to reach a device) misses every time."""
    h0, m0 = _cache_stats(lib)
    for _ in range(3):
        status = lib.conv2d_fwd_packed(A, 1, 8, 8, 64, BF16, B, 3, 3, 64, C, 9, 8, BF16,
                                       _lib.pair((1, 1)), _lib.pair((1, 1)), _lib.pair((1, 1)), 1, 0,
                                       None, 0.0, 0, WS, 256, None)
        assert status == INVALID   # Ho = 9 does not match the shape
    h1, m1 = _cache_stats(lib)
    assert (h1 - h0, m1 - m0) == (0, 3)


SK_WS = 256 + 152 * 8 * 4 + 152 * 128 * 1024 + 4096   # status + stream-K room for 152 SMs


def test_streamk_planner(lib, tuning):
    """Stream-K (every SM an equal share of the (tile, k-block) iterations,
    split tiles summed through fp32 partial slots) is chosen by its cost model
    only where few tiles carry a long contraction; it needs the workspace
    room; CONV_STREAMK=1 forces it where it applies (never with the row
    window, the gather loader or CTA pairs) and 0 forbids it."""
    tuning("CONV_STREAMK", None)
    tuning("CONV_PAIR", None)
    # Few tiles, long contraction: 2 x 8 x 8 x 1024 -> 256, 3x3 s2 (32 rows, K = 9216).
    deep = (2, 8, 8, 1024, BF16, 3, 256, 2, 1)
    p = _plan(lib, *deep, sms=152, ws=SK_WS)
    assert p["streamk"] == 1 and p["grid"] == 152 and p["bres"] == 0
    assert _plan(lib, *deep, sms=152, ws=256)["streamk"] == 0          # no workspace room
    # The benchmark convs keep whole tiles (the fix-up outweighs the balance).
    for conv in [(32, 56, 56, 64, BF16, 3, 128, 2, 1), (8, 128, 128, 128, F16, 5, 128, 2, 2),
                 (1, 16, 16, 16, BF16, 3, 16, 1, 1), (16, 64, 64, 320, F8, 3, 320, 1, 1),
                 (1, 256, 256, 512, BF16, 3, 512, 1, 1)]:
        assert _plan(lib, *conv, sms=152, ws=SK_WS)["streamk"] == 0, conv
    tuning("CONV_STREAMK", "1")
    q = _plan(lib, 8, 128, 128, 128, F16, 5, 128, 2, 2, sms=152, ws=SK_WS)
    assert (q["streamk"], q["grid"], q["tiles"]) == (1, 152, 128)
    assert _plan(lib, 32, 56, 56, 64, BF16, 3, 64, 1, 1, sms=152, ws=SK_WS)["streamk"] == 0  # window
    assert _plan(lib, 32, 224, 224, 3, BF16, 7, 64, 2, 3, sms=152, ws=SK_WS)["streamk"] == 0  # gather
    tuning("CONV_PAIR", "1")
    assert _plan(lib, 8, 128, 128, 128, F16, 5, 128, 2, 2, sms=152, ws=SK_WS)["streamk"] == 0  # pairs
    tuning("CONV_PAIR", None)
    tuning("CONV_STREAMK", "0")
    assert _plan(lib, *deep, sms=152, ws=SK_WS)["streamk"] == 0
