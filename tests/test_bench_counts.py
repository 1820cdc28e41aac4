"""The benchmark's roofline numerators against counts made another way.
bench.ops_counts: the oracle's convolution of an all-ones int8 input with an
all-ones filter gives every output C times the number of its in-bounds
filter taps (for a transposed convolution, C times the number of input
pixel / tap pairs that land on it), so twice the sum of all outputs is the
in-bounds operation count, and the result's shape gives P and Q.  The
nominal count of a transposed convolution is the same sum with no output
cropping (pads 0: every pair lands).  Reduced N, C and K keep each
workload's geometry; both counts are linear in them.  bench.algorithmic_bytes:
the generated tensors' sizes, the output's, and the input pixels that a
brute-force walk over output positions and taps finds read."""
import dataclasses
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import fconv_inputs as FI  # noqa: E402
import oracle  # noqa: E402

NAMES = list(FI.WORKLOADS) + list(FI.VARIANT_WORKLOADS)


@pytest.fixture(scope="module", autouse=True)
def built():
    oracle.build()


@pytest.mark.parametrize("name", NAMES)
def test_ops_counts_match_the_oracle(name):
    wl = dataclasses.replace(FI.workload(name), N=2, C=8, K=3)
    nominal, inbounds, P, Q = bench.ops_counts(wl)
    x = np.ones((wl.N, wl.H, wl.W, wl.C), dtype=np.int8)
    w = np.ones((wl.R, wl.S, wl.C, wl.K), dtype=np.int8)
    if wl.transposed_pads is None:
        pad = oracle.SAME if wl.padding == "SAME" else oracle.VALID
        acc = oracle.conv_acc_i8(x, w, wl.stride, pad)
        assert nominal == 2 * wl.N * P * Q * wl.K * wl.R * wl.S * wl.C
    else:
        acc = oracle.convT_acc_i8(x, w, wl.stride, wl.transposed_pads)
        full = oracle.convT_acc_i8(x, w, wl.stride, (0, 0, 0, 0))
        assert nominal == 2 * int(full.astype(np.int64).sum())
    assert acc.shape == (wl.N, P, Q, wl.K)
    assert inbounds == 2 * int(acc.astype(np.int64).sum())
    assert 0 < inbounds <= nominal


def test_padding_lowers_the_in_bounds_count():
    # a SAME 3x3 layer on a 4x4 image: along each axis the four output
    # positions keep 2, 3, 3 and 2 of their 3 taps (10 pairs), so 10 x 10 of
    # the 16 x 9 (pixel, tap) pairs read the image
    wl = dataclasses.replace(FI.workload("small_i8_16x16x32"), N=1, H=4, W=4, C=1, K=1)
    nominal, inbounds, P, Q = bench.ops_counts(wl)
    assert (P, Q) == (4, 4)
    assert nominal == 2 * 16 * 9
    assert inbounds == 2 * 10 * 10


def _read_extent(size, out, filt, stride, pad):
    # input positions along one axis that some output position reads
    return len({o * stride + t - pad for o in range(out) for t in range(filt)} & set(range(size)))


@pytest.mark.parametrize("name", NAMES)
def test_algorithmic_bytes_match_the_tensors(name):
    """The roofline's byte count against the generated tensors' own sizes,
    the output's, and the input pixels a brute-force walk finds read."""
    wl = dataclasses.replace(FI.workload(name), N=2, C=16, K=8)
    _, _, P, Q = bench.ops_counts(wl)
    t = FI.generate(wl, (P, Q))
    elt = t["x"].itemsize
    if wl.transposed_pads is None:
        pad = oracle.SAME if wl.padding == "SAME" else oracle.VALID
        g = oracle.Geometry(wl.N, wl.H, wl.W, wl.C, wl.K, wl.R, wl.S, wl.stride, wl.stride, pad)
        assert (g.P, g.Q) == (P, Q)
        rows = _read_extent(wl.H, P, wl.R, wl.stride, g.pt)
        cols = _read_extent(wl.W, Q, wl.S, wl.stride, g.pl)
    else:
        rows, cols = wl.H, wl.W   # every input pixel is scattered somewhere
    x_read = wl.N * rows * cols * wl.C * elt
    y = wl.N * P * Q * wl.K * elt
    side = t["side"].nbytes if t["side"] is not None else 0
    assert bench.algorithmic_bytes(wl) == x_read + t["w"].nbytes + side + y + t["bias"].nbytes
