"""Pins for the oracle's transposed convolution (the forward pass of MXNet's
deconvolution, "cudnn_deconvolution-inl.h": cuDNN backward-data of the
cross-correlation with the op's pad and stride).  No GPU needed."""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_convT.txt")


def _cases():
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            yield json.loads(line)


@pytest.mark.parametrize("case", list(_cases()), ids=lambda c: c["name"])
def test_hand_worked_cases(case):
    x = np.array(case["x"], np.int8)
    w = np.array(case["w"], np.int8)
    got = oracle.convT_acc_i8(x, w, tuple(case["stride"]), tuple(case["pads"]))
    assert np.array_equal(got, np.array(case["out"], np.int32))


ADJ_SHAPES = [
    # N, H, W, C, K, R, S, sh, sw, (pt, pb, pl, pr)
    (2, 5, 4, 3, 4, 3, 3, 1, 1, (1, 1, 1, 1)),
    (1, 4, 6, 2, 5, 3, 2, 2, 2, (1, 0, 0, 1)),      # adj 1 on the bottom: pb = pt - 1
    (2, 3, 3, 4, 2, 4, 4, 3, 2, (2, 1, 1, 2)),
    (1, 6, 5, 5, 3, 2, 3, 2, 1, (0, 0, 2, 2)),
    (1, 3, 4, 2, 2, 3, 3, 2, 2, (1, -1, 1, 0)),      # pb < 0: rows that receive nothing
]


@pytest.mark.parametrize("shape", ADJ_SHAPES)
def test_adjoint_of_the_forward_convolution(shape):
    """<convT(x), z> = <x, F(z)>, exactly, where F is the forward
    cross-correlation with the same stride and pads and the filter's
    input/output channel axes swapped: the transposed convolution is the
    forward convolution's adjoint (its backward-data pass)."""
    N, H, W, C, K, R, S, sh, sw, pads = shape
    pt, pb, pl, pr = pads
    rng = np.random.default_rng(hash(shape) % 2 ** 32)
    x = rng.integers(-128, 128, size=(N, H, W, C)).astype(np.int8)
    w = rng.integers(-128, 128, size=(R, S, C, K)).astype(np.int8)
    out = oracle.convT_acc_i8(x, w, (sh, sw), pads)
    Ho, Wo = out.shape[1:3]
    z = rng.integers(-128, 128, size=(N, Ho, Wo, K)).astype(np.int8)
    wt = np.ascontiguousarray(w.transpose(0, 1, 3, 2))           # [R][S][K][C]
    fz = oracle.conv_acc_i8_explicit(z, wt, sh, sw, pt, pl, H, W)  # [N][H][W][C]
    lhs = int(np.sum(out.astype(np.int64) * z.astype(np.int64)))
    rhs = int(np.sum(x.astype(np.int64) * fz.astype(np.int64)))
    assert lhs == rhs


@pytest.mark.parametrize("shape", [
    # N, H, W, C, K, R, S, stride, pad, output_padding
    (2, 5, 4, 3, 4, 3, 3, 1, 1, 0),
    (1, 4, 6, 2, 5, 3, 3, 2, 1, 1),
    (2, 3, 5, 4, 2, 4, 4, 3, 1, 2),
    (1, 7, 7, 3, 3, 5, 5, 2, 2, 0),
])
def test_matches_torch_conv_transpose2d(shape):
    """The library routine, in float64 on the CPU, for symmetric pads with an
    output adjustment (pt = pad, pb = pad - output_padding)."""
    N, H, W, C, K, R, S, st, pad, op = shape
    rng = np.random.default_rng(sum(shape))
    x = rng.integers(-128, 128, size=(N, H, W, C)).astype(np.int8)
    w = rng.integers(-128, 128, size=(R, S, C, K)).astype(np.int8)
    got = oracle.convT_acc_i8(x, w, st, (pad, pad - op, pad, pad - op))
    ref = torch.nn.functional.conv_transpose2d(
        torch.from_numpy(x.astype(np.float64)).permute(0, 3, 1, 2),
        torch.from_numpy(w.astype(np.float64)).permute(2, 3, 0, 1),   # [C][K][R][S]
        stride=st, padding=pad, output_padding=op).permute(0, 2, 3, 1).numpy()
    assert got.shape == ref.shape
    assert np.array_equal(got, ref.astype(np.int64))


def test_one_by_one_stride_one_is_the_forward_convolution():
    rng = np.random.default_rng(5)
    x = rng.integers(-128, 128, size=(2, 6, 7, 16)).astype(np.int8)
    w = rng.integers(-128, 128, size=(1, 1, 16, 8)).astype(np.int8)
    assert np.array_equal(oracle.convT_acc_i8(x, w, 1, (0, 0, 0, 0)),
                          oracle.conv_acc_i8(x, w, 1, oracle.VALID))


def test_bf16_sums_match_the_int8_sums_on_small_integers():
    """bf16 holds the integers in [-128, 127] exactly and fp64 sums them
    exactly: the two oracles must agree."""
    rng = np.random.default_rng(6)
    x = rng.integers(-128, 128, size=(2, 4, 5, 3)).astype(np.int8)
    w = rng.integers(-128, 128, size=(3, 3, 3, 4)).astype(np.int8)
    to_bits = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    pads = (1, 0, 2, 1)
    a = oracle.convT_acc_i8(x, w, 2, pads)
    b = oracle.convT_acc_bf16_f64(to_bits(x), to_bits(w), 2, pads)
    assert np.array_equal(a.astype(np.float64), b)
