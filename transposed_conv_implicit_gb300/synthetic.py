"""Seeded synthetic inputs for the convolution workloads.

This module only draws random numbers and describes shapes.  It holds none of
the convolution arithmetic, so both the CUDA path and the CPU oracle may take
their inputs from it.

Recipe (the same for every workload): one ``torch.Generator`` seeded with the
workload's seed draws, in this order, the input, the filter and (if the
workload has a residual) the source, each as fp32 on the CPU, then casts each
to its storage dtype with round-to-nearest-even.  ``N(0, v)`` means mean 0 and
VARIANCE v; ``U[-1, 1]`` is uniform.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Tuple

import torch

TORCH_DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16, "f8e4m3": torch.float8_e4m3fn}
ELT_BYTES = {"bf16": 2, "f16": 2, "f8e4m3": 1}


@dataclasses.dataclass(frozen=True)
class Dist:
    kind: str          # "normal" (parameter = variance) or "uniform" (parameter = half-width)
    param: float

    def draw(self, shape, gen: torch.Generator) -> torch.Tensor:
        if self.kind == "normal":
            return torch.randn(shape, generator=gen, dtype=torch.float32) * math.sqrt(self.param)
        if self.kind == "uniform":
            return (torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0) * self.param
        if self.kind == "int":      # integers in [-param, param]: exact in every dtype used here
            p = int(self.param)
            return torch.randint(-p, p + 1, shape, generator=gen).to(torch.float32)
        raise ValueError(self.kind)


@dataclasses.dataclass(frozen=True)
class ConvCase:
    """One convolution problem: shapes, layouts, distributions and seed.

    kind "fwd": input [N,H,W,C_in], filter FCRS [C_out,C_in,R,S] or RSCF
    [R,S,C_in,C_out], output [N,Ho,Wo,C_out].
    kind "transposed": input [N,H,W,C_in], filter RSFC [R,S,C_out,C_in],
    output [N,Ho,Wo,C_out] with Ho/Wo given by ``out_hw``.
    """
    name: str
    kind: str
    dtype: str
    N: int
    H: int
    W: int
    C_in: int
    C_out: int
    R: int
    S: int
    stride: int
    pad: int
    filter_layout: str
    x_dist: Dist
    w_dist: Dist
    seed: int
    dilation: int = 1
    has_residual: bool = False
    beta: float = 0.0
    src_dist: Optional[Dist] = None
    epilogue: str = "none"
    out_hw: Optional[Tuple[int, int]] = None
    pad_w: Optional[int] = None        # padding along W when it differs from `pad` (H)
    dilation_w: Optional[int] = None   # dilation along W when it differs from `dilation` (H)
    groups: int = 1                    # channel groups (forward): filter channels = C_in / groups
    stride_w: Optional[int] = None     # stride along W when it differs from `stride` (H; transposed)

    @property
    def strides(self) -> Tuple[int, int]:
        """(stride_h, stride_w)."""
        return (self.stride, self.stride if self.stride_w is None else self.stride_w)

    @property
    def pads(self) -> Tuple[int, int]:
        """(pad_h, pad_w)."""
        return (self.pad, self.pad if self.pad_w is None else self.pad_w)

    @property
    def dilations(self) -> Tuple[int, int]:
        """(dil_h, dil_w)."""
        return (self.dilation, self.dilation if self.dilation_w is None else self.dilation_w)

    @property
    def out_dtype(self) -> str:
        return "bf16" if self.dtype == "f8e4m3" else self.dtype

    @property
    def Ho(self) -> int:
        if self.out_hw is not None:
            return self.out_hw[0]
        return (self.H + 2 * self.pad - self.dilation * (self.R - 1) - 1) // self.stride + 1

    @property
    def Wo(self) -> int:
        if self.out_hw is not None:
            return self.out_hw[1]
        return (self.W + 2 * self.pads[1] - self.dilations[1] * (self.S - 1) - 1) // self.stride + 1

    @property
    def filter_shape(self):
        if self.filter_layout == "FCRS":
            return (self.C_out, self.C_in // self.groups, self.R, self.S)
        if self.filter_layout == "RSCF":
            return (self.R, self.S, self.C_in // self.groups, self.C_out)
        if self.filter_layout == "RSFC":
            return (self.R, self.S, self.C_out, self.C_in)
        raise ValueError(self.filter_layout)

    @property
    def out_shape(self):
        return (self.N, self.Ho, self.Wo, self.C_out)

    @property
    def flops(self) -> int:
        """Algorithmic FLOPs: 2*N*Ho*Wo*C_out*R*S*C_in forward; 2*N*H*W*C_in*C_out*R*S
        transposed (the scatter count, no zero insertion)."""
        if self.kind == "transposed":
            return 2 * self.N * self.H * self.W * self.C_in * self.C_out * self.R * self.S
        return 2 * self.N * self.Ho * self.Wo * self.C_out * self.R * self.S * self.C_in // self.groups

    @property
    def bytes(self) -> int:
        """Algorithmic bytes: input, filter and output once, plus the source once."""
        e_in, e_out = ELT_BYTES[self.dtype], ELT_BYTES[self.out_dtype]
        b = self.N * self.H * self.W * self.C_in * e_in
        b += self.R * self.S * self.C_in // self.groups * self.C_out * e_in
        b += self.N * self.Ho * self.Wo * self.C_out * e_out
        if self.has_residual:
            b += self.N * self.Ho * self.Wo * self.C_out * e_out
        return b


def make_inputs(case: ConvCase, device="cpu"):
    """Return dict(x, w, src) of tensors in their storage dtypes (src None if no residual)."""
    gen = torch.Generator()
    gen.manual_seed(case.seed)
    td = TORCH_DTYPES[case.dtype]
    x = case.x_dist.draw((case.N, case.H, case.W, case.C_in), gen).to(td)
    w = case.w_dist.draw(case.filter_shape, gen).to(td)
    src = None
    if case.has_residual:
        src = case.src_dist.draw(case.out_shape, gen).to(TORCH_DTYPES[case.out_dtype])
    if device != "cpu":
        x, w = x.to(device), w.to(device)
        src = src.to(device) if src is not None else None
    return {"x": x, "w": w, "src": src}


def raw_bits(t: torch.Tensor):
    """Storage bits of a CPU tensor as a numpy array (uint16 or uint8)."""
    t = t.contiguous().cpu()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view("uint16")
    return t.view(torch.uint8).numpy()


def _n(v):
    return Dist("normal", v)


# The benchmark workloads.  Filter-layout choices where a workload leaves it
# open: RSCF (the forward default).  N(0, v): v is the variance.
WORKLOADS = {
    "tiny_bf16": ConvCase("tiny_bf16", "fwd", "bf16", 1, 16, 16, 16, 16, 3, 3, 1, 1, "RSCF",
                          Dist("uniform", 1.0), Dist("uniform", 1.0), seed=1001),
    "resnet_bf16": ConvCase("resnet_bf16", "fwd", "bf16", 32, 56, 56, 64, 64, 3, 3, 1, 1, "RSCF",
                            _n(1.0), _n(2.0 / (9 * 64)), seed=1002, has_residual=True, beta=1.0,
                            src_dist=_n(1.0)),
    "resnet_down_bf16": ConvCase("resnet_down_bf16", "fwd", "bf16", 32, 56, 56, 64, 128, 3, 3, 2, 1,
                                 "RSCF", _n(1.0), _n(2.0 / (9 * 64)), seed=1012),
    "fp8_res": ConvCase("fp8_res", "fwd", "f8e4m3", 16, 64, 64, 320, 320, 3, 3, 1, 1, "FCRS",
                        _n(1.0), _n(1.0 / math.sqrt(9 * 320)), seed=1003, has_residual=True,
                        beta=0.5, src_dist=_n(1.0)),
    "vae_silu_bf16": ConvCase("vae_silu_bf16", "fwd", "bf16", 1, 256, 256, 512, 512, 3, 3, 1, 1, "RSCF",
                              _n(1.0), _n(1.0 / (9 * 512)), seed=1004, epilogue="silu"),
    "vae_head_bf16": ConvCase("vae_head_bf16", "fwd", "bf16", 1, 512, 512, 128, 3, 3, 3, 1, 1, "RSCF",
                              _n(1.0), _n(1.0 / (9 * 128)), seed=1014),
    "convT_f16": ConvCase("convT_f16", "transposed", "f16", 8, 32, 32, 256, 128, 4, 4, 2, 1, "RSFC",
                          _n(1.0), _n(1.0 / (16 * 256)), seed=1005, epilogue="relu", out_hw=(64, 64)),
    "fwd5x5_f16": ConvCase("fwd5x5_f16", "fwd", "f16", 8, 128, 128, 128, 128, 5, 5, 2, 2, "RSCF",
                           _n(1.0), _n(1.0 / (25 * 128)), seed=1015),
    # RGB stem: 3 input channels (6-byte pixels) need the gather A loader.
    "stem_c3_bf16": ConvCase("stem_c3_bf16", "fwd", "bf16", 32, 224, 224, 3, 64, 7, 7, 2, 3, "RSCF",
                             _n(1.0), _n(2.0 / (49 * 3)), seed=1020, epilogue="relu"),
    # Depthwise 3x3 (one channel per group): the direct CUDA-core kernel.
    "dw_bf16": ConvCase("dw_bf16", "fwd", "bf16", 32, 112, 112, 64, 64, 3, 3, 1, 1, "RSCF",
                        _n(1.0), _n(2.0 / 9), seed=1021, epilogue="relu", groups=64),
}

# The ResNet-style block: the stride-1 residual conv and the stride-2 downsample.
RESNET_BLOCK = ("resnet_bf16", "resnet_down_bf16")

# Every convolution of the benchmark configurations, in their order.
BASELINE_SET = ("tiny_bf16", "resnet_bf16", "resnet_down_bf16", "fp8_res", "vae_silu_bf16",
                "vae_head_bf16", "convT_f16", "fwd5x5_f16")
