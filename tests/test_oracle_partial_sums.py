"""The oracle's partial-sum bounds (conv_i8_partial_sum_bounds), and what
they show about the int8 workloads.

TensorFlow's CPU path for the fused int8 op ("conv_ops_fused_int8.cc",
LaunchFusedConv2DOpCpuInt8Helper, TempT = float) accumulates the int8
products in fp32; this library (and the oracle) sums them exactly in int32.
The two agree while every value an fp32 summation passes through is an
integer below 2^24.  The bounds are pinned here against a brute-force
enumeration of the patch products, a closed form and a hand case; then they
are evaluated on the four int8 workloads."""
import numpy as np
import pytest

import fconv_inputs as FI
import oracle

PAD = {"SAME": oracle.SAME, "VALID": oracle.VALID}


def brute_force_bounds(x, w, sh, sw, padding):
    """Products of every output's patch in (r, s, c) order from a zero-padded
    copy of the input (padding taps add a zero product, which changes no
    prefix maximum and no sum), then cumulative sums."""
    N, H, W, C = x.shape
    R, S, _, K = w.shape
    P, pt, pb = oracle.out_geometry(H, R, sh, padding)
    Q, pl, pr = oracle.out_geometry(W, S, sw, padding)
    xp = np.pad(x.astype(np.int64), ((0, 0), (pt, pb), (pl, pr), (0, 0)))
    wm = w.astype(np.int64).reshape(R * S * C, K)
    best = [0, 0, 0]
    for n in range(N):
        for p in range(P):
            for q in range(Q):
                patch = xp[n, p * sh:p * sh + R, q * sw:q * sw + S, :].reshape(R * S * C)
                prods = patch[:, None] * wm                 # [RSC][K], patch order
                pre = np.cumsum(prods, axis=0)
                best[0] = max(best[0], int(np.abs(pre[-1]).max()))
                best[1] = max(best[1], int(np.abs(pre).max()))
                best[2] = max(best[2], int(np.abs(prods).sum(axis=0).max()))
    return tuple(best)


CASES = [
    # N, H, W, C, K, R, S, sh, sw, padding
    (2, 5, 6, 3, 4, 3, 3, 1, 1, "SAME"),
    (1, 7, 5, 2, 3, 2, 4, 2, 1, "SAME"),
    (2, 6, 6, 4, 2, 3, 2, 1, 3, "VALID"),
    (1, 3, 3, 5, 5, 1, 1, 2, 2, "VALID"),
    (3, 4, 4, 2, 2, 5, 5, 3, 3, "SAME"),
]


@pytest.mark.parametrize("case", CASES)
def test_bounds_match_brute_force(case):
    N, H, W, C, K, R, S, sh, sw, pad = case
    rng = np.random.default_rng(sum(case[:9]))
    x = rng.integers(-128, 128, size=(N, H, W, C), dtype=np.int8)
    w = rng.integers(-128, 128, size=(R, S, C, K), dtype=np.int8)
    got = oracle.conv_i8_partial_sum_bounds(x, w, (sh, sw), PAD[pad])
    assert got == brute_force_bounds(x, w, sh, sw, PAD[pad])
    # the final sums are the oracle's own convolution
    assert got[0] == int(np.abs(oracle.conv_acc_i8(x, w, (sh, sw), PAD[pad]).astype(np.int64)).max())


def test_constant_inputs_closed_form():
    # x = -7 and w = 9 everywhere: every product is -63, the prefix grows
    # monotonically, so all three bounds are 63 * C * (taps of the fullest window)
    x = np.full((1, 5, 5, 3), -7, np.int8)
    w = np.full((3, 3, 3, 2), 9, np.int8)
    assert oracle.conv_i8_partial_sum_bounds(x, w, 1, oracle.SAME) == (63 * 27,) * 3
    # VALID 3x3 on 5x5 at stride 2: every window is full
    assert oracle.conv_i8_partial_sum_bounds(x, w, 2, oracle.VALID) == (63 * 27,) * 3


def test_prefix_above_the_final_sum():
    # 1x1 over two channels: products 127*127 then 127*(-127); the sum ends at
    # 0 after peaking at 16129, and the sum of magnitudes is 32258
    x = np.array([[[[127, 127]]]], np.int8)
    w = np.array([[[[127], [-127]]]], np.int8)
    assert oracle.conv_i8_partial_sum_bounds(x, w, 1, oracle.VALID) == (0, 16129, 32258)


INT8_WORKLOADS = [n for n, wl in FI.WORKLOADS.items() if wl.dtype == "int8"]


@pytest.mark.parametrize("name", INT8_WORKLOADS)
def test_workload_sums_agree_with_fp32_accumulation(name):
    """On every int8 workload the int32 sums equal what the page's fp32
    accumulation gives: the final sums and every prefix in patch order stay
    below 2^23, so a sequential fp32 sum in that order, or any blocked sum of
    contiguous runs of it, is exact.  Where the sum of |x*w| is below 2^24 as
    well, every summation order is exact."""
    wl = FI.WORKLOADS[name]
    P, _, _ = oracle.out_geometry(wl.H, wl.R, wl.stride, PAD[wl.padding])
    Q, _, _ = oracle.out_geometry(wl.W, wl.S, wl.stride, PAD[wl.padding])
    inp = FI.generate(wl, (P, Q))
    acc_max, prefix_max, abs_max = oracle.conv_i8_partial_sum_bounds(
        inp["x"], inp["w"], wl.stride, PAD[wl.padding])
    assert acc_max <= prefix_max <= abs_max
    assert prefix_max < 2 ** 23, (acc_max, prefix_max, abs_max)
    if name != "large_i8_28x28x512":
        # fewer than 1024 products of magnitude <= 2^14 each (c1: 288 of
        # at most 64; c2: 576; c3: 256 of at most 2^12)
        assert abs_max < 2 ** 24, (acc_max, prefix_max, abs_max)
    print(f"{name}: max|acc| {acc_max}, max|prefix| {prefix_max}, max sum|xw| {abs_max}")
