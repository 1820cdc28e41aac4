"""Seeded synthetic inputs for the fused Conv2D workloads.

This module holds shapes, value distributions and random-number draws only:
no convolution arithmetic.  Both the CUDA path's tests/benchmark and the CPU
oracle take their inputs from here.  The output geometry (needed for the
side input's shape) is passed in by the caller, who computes it with its
own rule.

Generation follows one fixed recipe: a CPU ``torch.Generator`` seeded with
the workload's seed, drawing in the order x, w, bias, side; int8 values with
``torch.randint`` over an inclusive range, normal values with
``torch.randn`` scaled by the stated standard deviation.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                 # "int8" or "bf16"
    N: int
    H: int
    W: int
    C: int
    K: int
    R: int
    S: int
    stride: int
    padding: str               # "SAME" or "VALID"
    x_dist: tuple              # ("uniform", lo, hi) inclusive, or ("normal", std)
    w_dist: tuple
    bias_std: float
    conv_scale: float
    side_scale: float
    has_side: bool
    relu: bool
    seed: int
    note: str = field(default="", compare=False)
    # (top, bottom, left, right) for a transposed convolution (deconvolution
    # forward, stride `stride`); None for a forward convolution
    transposed_pads: tuple | None = field(default=None, compare=False)


# The five workload shapes of the fused int8/bf16 conv benchmark suite.
WORKLOADS = {
    "small_i8_16x16x32": Workload(
        "small_i8_16x16x32", "int8", 1, 16, 16, 32, 32, 3, 3, 1, "SAME",
        ("uniform", -8, 7), ("uniform", -8, 7), 1.0, 0.05, 0.0, False, True, 0,
        "int8, N=1 16x16x32, 3x3x32x32, stride 1 SAME, side scale 0, ReLU"),
    "resnet_i8_56x56x64": Workload(
        "resnet_i8_56x56x64", "int8", 32, 56, 56, 64, 64, 3, 3, 1, "SAME",
        ("uniform", -128, 127), ("uniform", -128, 127), 1.0, 0.002, 0.5, True, True, 1,
        "int8 residual block conv, N=32 56x56x64, 3x3, side input, ReLU"),
    "proj1x1s2_i8_28x28x256": Workload(
        "proj1x1s2_i8_28x28x256", "int8", 64, 28, 28, 256, 512, 1, 1, 2, "VALID",
        ("uniform", -64, 63), ("uniform", -64, 63), 0.5, 0.004, 0.0, False, False, 2,
        "int8 1x1 projection, N=64 28x28x256 -> 512, stride 2 VALID, BiasAdd only"),
    "bf16_14x14x256": Workload(
        "bf16_14x14x256", "bf16", 32, 14, 14, 256, 256, 3, 3, 1, "SAME",
        ("normal", 1.0), ("normal", 1.0 / 48.0), 0.1, 1.0, 0.0, False, True, 3,
        "bf16 conv+bias+ReLU, N=32 14x14x256, 3x3 stride 1 SAME"),
    "large_i8_28x28x512": Workload(
        "large_i8_28x28x512", "int8", 256, 28, 28, 512, 512, 3, 3, 1, "SAME",
        ("uniform", -128, 127), ("uniform", -128, 127), 1.0, 0.001, 0.25, True, True, 4,
        "int8 N=256 28x28x512, 3x3 stride 1 SAME, side input, ReLU"),
}

ORDER = list(WORKLOADS)

# Further shapes for the paths beyond the five (measured, not the headline):
# transposed convolutions of a decoder / generator, one upsampling by 2.
VARIANT_WORKLOADS = {
    "deconv_bf16_16x16x256_s2": Workload(
        "deconv_bf16_16x16x256_s2", "bf16", 64, 16, 16, 256, 128, 4, 4, 2, "VALID",
        ("normal", 1.0), ("normal", 1.0 / 32.0), 0.1, 1.0, 0.0, False, True, 5,
        "bf16 transposed conv, N=64 16x16x256 -> 32x32x128, 4x4 stride 2 pad 1, bias+ReLU",
        transposed_pads=(1, 1, 1, 1)),
    "deconv_i8_14x14x512_s1": Workload(
        "deconv_i8_14x14x512_s1", "int8", 64, 14, 14, 512, 256, 3, 3, 1, "VALID",
        ("uniform", -128, 127), ("uniform", -128, 127), 1.0, 0.0005, 0.0, False, True, 6,
        "int8 transposed conv, N=64 14x14x512 -> 14x14x256, 3x3 stride 1 pad 1, bias+ReLU",
        transposed_pads=(1, 1, 1, 1)),
}


# The two shapes the page's CPU helper computes as plain matrix products
# ("conv_ops_fused_int8.cc", LaunchFusedConv2DOpCpuInt8Helper): a 1x1 filter
# at stride 1 ([N*H*W][C] x [C][K]) and a filter as large as the input under
# VALID padding ([N][R*S*C] x [R*S*C][K]).
VARIANT_WORKLOADS.update({
    "proj1x1s1_i8_28x28x256": Workload(
        "proj1x1s1_i8_28x28x256", "int8", 64, 28, 28, 256, 512, 1, 1, 1, "VALID",
        ("uniform", -64, 63), ("uniform", -64, 63), 0.5, 0.004, 0.0, False, False, 7,
        "int8 1x1 projection, N=64 28x28x256 -> 512, stride 1 (a matrix product), BiasAdd only"),
    "fullwin_i8_7x7x512": Workload(
        "fullwin_i8_7x7x512", "int8", 32, 7, 7, 512, 1024, 7, 7, 1, "VALID",
        ("uniform", -128, 127), ("uniform", -128, 127), 1.0, 5e-5, 0.0, False, True, 8,
        "int8 full-window VALID, N=32 7x7x512 -> 1x1x1024 (a matrix product), bias+ReLU"),
})


# Deep layers at small batch: few output tiles over long reductions, where
# the plan splits each tile's k-blocks over several CTAs.
VARIANT_WORKLOADS.update({
    "deep_b1_i8_7x7x512": Workload(
        "deep_b1_i8_7x7x512", "int8", 1, 7, 7, 512, 512, 3, 3, 1, "SAME",
        ("uniform", -128, 127), ("uniform", -128, 127), 1.0, 1e-4, 0.0, False, True, 9,
        "int8 batch-one deep layer, N=1 7x7x512 -> 512, 3x3 SAME, bias+ReLU"),
    "deep_b1_i8_14x14x256": Workload(
        "deep_b1_i8_14x14x256", "int8", 1, 14, 14, 256, 256, 3, 3, 1, "SAME",
        ("uniform", -128, 127), ("uniform", -128, 127), 1.0, 1.5e-4, 0.0, False, True, 10,
        "int8 batch-one layer, N=1 14x14x256 -> 256, 3x3 SAME, bias+ReLU"),
    "proj_b8_i8_7x7x2048": Workload(
        "proj_b8_i8_7x7x2048", "int8", 8, 7, 7, 2048, 512, 1, 1, 1, "VALID",
        ("uniform", -128, 127), ("uniform", -128, 127), 1.0, 1.5e-4, 0.0, False, True, 11,
        "int8 1x1 reduction, N=8 7x7x2048 -> 512, bias+ReLU"),
})


def workload(name: str) -> Workload:
    """A workload by name, from either table."""
    return WORKLOADS[name] if name in WORKLOADS else VARIANT_WORKLOADS[name]


def _draw(gen: torch.Generator, shape, dist, dtype: str) -> np.ndarray:
    if dist[0] == "uniform":
        lo, hi = dist[1], dist[2]
        t = torch.randint(lo, hi + 1, tuple(shape), dtype=torch.int8, generator=gen)
        return t.numpy()
    if dist[0] == "normal":
        t = torch.randn(tuple(shape), dtype=torch.float32, generator=gen) * float(dist[1])
        if dtype == "bf16":
            return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        return t.numpy()
    raise ValueError(dist)


def generate(wl: Workload, out_hw: tuple[int, int], batch: int | None = None):
    """Inputs of a workload as numpy arrays.

    Returns dict(x, w, bias, side) with x NHWC, w HWIO, bias [K] float32 and
    side NHWC of the output shape (or None).  int8 tensors are int8 arrays;
    bf16 tensors are uint16 arrays of bf16 bit patterns.  ``batch`` draws
    only the first ``batch`` images' worth of x and side (a bounded sample
    with the same distributions; the draws are not a prefix of the full set).
    """
    P, Q = out_hw
    N = wl.N if batch is None else batch
    gen = torch.Generator(device="cpu")
    gen.manual_seed(wl.seed)
    x = _draw(gen, (N, wl.H, wl.W, wl.C), wl.x_dist, wl.dtype)
    w = _draw(gen, (wl.R, wl.S, wl.C, wl.K), wl.w_dist, wl.dtype)
    bias = (torch.randn((wl.K,), dtype=torch.float32, generator=gen) * wl.bias_std).numpy()
    side = None
    if wl.has_side:
        if wl.dtype == "int8":
            side = _draw(gen, (N, P, Q, wl.K), ("uniform", -128, 127), "int8")
        else:
            side = _draw(gen, (N, P, Q, wl.K), ("normal", 1.0), "bf16")
    return {"x": x, "w": w, "bias": bias, "side": side}


def random_case(seed: int, N, H, W, C, K, R, S, dtype: str, out_hw, with_side: bool,
                x_range=(-128, 127), w_range=(-128, 127), w_std=None, bias_std=1.0):
    """Inputs for a parity sweep case of any shape, same recipe as above."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    if dtype == "int8":
        xd, wd = ("uniform",) + tuple(x_range), ("uniform",) + tuple(w_range)
    else:
        xd = ("normal", 1.0)
        wd = ("normal", w_std if w_std is not None else 1.0 / np.sqrt(R * S * C))
    x = _draw(gen, (N, H, W, C), xd, dtype)
    w = _draw(gen, (R, S, C, K), wd, dtype)
    bias = (torch.randn((K,), dtype=torch.float32, generator=gen) * bias_std).numpy()
    side = None
    if with_side:
        P, Q = out_hw
        sd = ("uniform", -128, 127) if dtype == "int8" else ("normal", 1.0)
        side = _draw(gen, (N, P, Q, K), sd, dtype)
    return {"x": x, "w": w, "bias": bias, "side": side}


def uniform_int8(seed: int, shape) -> np.ndarray:
    """Seeded uniform int8 in [-128, 127] from numpy's PCG64, for inputs of
    billions of elements (the torch CPU generator is too slow there)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(-128, 128, size=shape, dtype=np.int8)
