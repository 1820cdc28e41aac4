"""Pins for the CPU oracle: it is checked here against things other than
itself -- hand-worked values, closed forms, invariants and independent
library routines (torch CPU conv2d in float64, scipy correlate, numpy
matmul).  No GPU needed."""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
PAD = {"SAME": oracle.SAME, "VALID": oracle.VALID}


# --------------------------------------------------------------------------
# geometry
# --------------------------------------------------------------------------
def _geometry_rows():
    rows = []
    with open(os.path.join(GOLDEN, "geometry_cases.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a = line.split()
            rows.append((int(a[0]), int(a[1]), int(a[2]), a[3], int(a[4]), int(a[5]), int(a[6])))
    return rows


@pytest.mark.parametrize("row", _geometry_rows())
def test_geometry_hand_table(row):
    size, filt, stride, pad, out, before, after = row
    if out < 0:
        with pytest.raises(ValueError):
            oracle.out_geometry(size, filt, stride, PAD[pad])
        return
    assert oracle.out_geometry(size, filt, stride, PAD[pad]) == (out, before, after)


@pytest.mark.parametrize("size", range(1, 12))
@pytest.mark.parametrize("filt", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("stride", [1, 2, 3])
def test_geometry_matches_torch_conv_extent(size, filt, stride):
    # torch's conv2d decides the output extent of a padded input by itself;
    # the oracle's pads must give the SAME extent ceil(size/stride) and the
    # VALID extent torch reports for an unpadded input.
    x = torch.zeros(1, 1, 1, size, dtype=torch.float64)
    w = torch.zeros(1, 1, 1, filt, dtype=torch.float64)
    out, before, after = oracle.out_geometry(size, filt, stride, oracle.SAME)
    y = F.conv2d(F.pad(x, (before, after)), w, stride=(1, stride))
    assert y.shape[-1] == out == -(-size // stride)
    assert before <= after <= before + 1
    if filt <= size:
        out_v, b_v, a_v = oracle.out_geometry(size, filt, stride, oracle.VALID)
        assert (b_v, a_v) == (0, 0)
        assert F.conv2d(x, w, stride=(1, stride)).shape[-1] == out_v


# --------------------------------------------------------------------------
# the convolution sum
# --------------------------------------------------------------------------
def _hand_cases():
    cases = []
    with open(os.path.join(GOLDEN, "hand_convs.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            f = [s.strip() for s in line.split("|")]
            N, H, W, C = map(int, f[1].split())
            R, S, K = map(int, f[2].split())
            sh, sw = map(int, f[3].split())
            cases.append((f[0], (N, H, W, C), (R, S, K), (sh, sw), f[4],
                          [int(v) for v in f[5].split()], [int(v) for v in f[6].split()],
                          [int(v) for v in f[7].split()]))
    return cases


@pytest.mark.parametrize("case", _hand_cases(), ids=lambda c: c[0])
def test_conv_hand_worked(case):
    name, (N, H, W, C), (R, S, K), stride, pad, xv, wv, expect = case
    x = np.array(xv, dtype=np.int8).reshape(N, H, W, C)
    w = np.array(wv, dtype=np.int8).reshape(R, S, C, K)
    for fn in (oracle.conv_acc_i8, oracle.conv_acc_i8_im2col):
        acc = fn(x, w, stride, PAD[pad])
        assert acc.ravel().tolist() == expect, (name, fn.__name__)


def _torch_conv_f64(x, w, stride, padding):
    """Library convolution: torch CPU conv2d in float64 on explicitly padded input."""
    N, H, W, C = x.shape
    R, S, _, K = w.shape
    _, pt, pb = oracle.out_geometry(H, R, stride[0], padding)
    _, pl, pr = oracle.out_geometry(W, S, stride[1], padding)
    xt = torch.from_numpy(x.astype(np.float64)).permute(0, 3, 1, 2)
    wt = torch.from_numpy(w.astype(np.float64)).permute(3, 2, 0, 1)
    y = F.conv2d(F.pad(xt, (pl, pr, pt, pb)), wt, stride=stride)
    return y.permute(0, 2, 3, 1).numpy()


def _tiny_cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        N = int(rng.integers(1, 3))
        H, W = int(rng.integers(1, 8)), int(rng.integers(1, 8))
        C, K = int(rng.integers(1, 6)), int(rng.integers(1, 6))
        R, S = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        stride = (int(rng.integers(1, 4)), int(rng.integers(1, 4)))
        pad = oracle.SAME if rng.integers(0, 2) == 0 else oracle.VALID
        if pad == oracle.VALID and (R > H or S > W):
            continue
        x = rng.integers(-128, 128, size=(N, H, W, C)).astype(np.int8)
        w = rng.integers(-128, 128, size=(R, S, C, K)).astype(np.int8)
        out.append((x, w, stride, pad))
    return out


@pytest.mark.parametrize("case", _tiny_cases(120, 1))
def test_conv_matches_torch_conv2d_f64(case):
    x, w, stride, pad = case
    acc = oracle.conv_acc_i8(x, w, stride, pad)
    ref = _torch_conv_f64(x, w, stride, pad)
    assert ref.shape == acc.shape
    assert np.array_equal(acc.astype(np.float64), ref)


@pytest.mark.parametrize("case", _tiny_cases(60, 2))
def test_direct_equals_im2col_gemm(case):
    x, w, stride, pad = case
    assert np.array_equal(oracle.conv_acc_i8(x, w, stride, pad),
                          oracle.conv_acc_i8_im2col(x, w, stride, pad))


def test_conv_matches_scipy_correlate():
    signal = pytest.importorskip("scipy.signal")
    rng = np.random.default_rng(3)
    for _ in range(10):
        H, W, C, K, R, S = 6, 7, 3, 2, 3, 2
        x = rng.integers(-128, 128, size=(1, H, W, C)).astype(np.int8)
        w = rng.integers(-128, 128, size=(R, S, C, K)).astype(np.int8)
        acc = oracle.conv_acc_i8(x, w, 1, oracle.VALID)
        for k in range(K):
            ref = signal.correlate(x[0].astype(np.int64), w[:, :, :, k].astype(np.int64),
                                   mode="valid", method="direct")[:, :, 0]
            assert np.array_equal(acc[0, :, :, k], ref)


def test_1x1_stride1_is_matmul():
    rng = np.random.default_rng(4)
    x = rng.integers(-128, 128, size=(2, 5, 3, 16)).astype(np.int8)
    w = rng.integers(-128, 128, size=(1, 1, 16, 7)).astype(np.int8)
    ref = x.reshape(-1, 16).astype(np.int64) @ w.reshape(16, 7).astype(np.int64)
    for pad in (oracle.SAME, oracle.VALID):
        acc = oracle.conv_acc_i8(x, w, 1, pad)
        assert np.array_equal(acc.reshape(-1, 7), ref)


def test_full_window_valid_is_matmul():
    rng = np.random.default_rng(5)
    x = rng.integers(-128, 128, size=(3, 4, 5, 6)).astype(np.int8)
    w = rng.integers(-128, 128, size=(4, 5, 6, 9)).astype(np.int8)
    ref = x.reshape(3, -1).astype(np.int64) @ w.reshape(-1, 9).astype(np.int64)
    acc = oracle.conv_acc_i8(x, w, 1, oracle.VALID)
    assert acc.shape == (3, 1, 1, 9)
    assert np.array_equal(acc.reshape(3, 9), ref)


def test_ones_count_in_bounds_taps():
    # x = 1, w = 1, 3x3 SAME stride 1 on a 4x4 image: every output equals
    # C times the number of taps inside the image: 4 at the corners, 6 on
    # the edges, 9 inside.
    C, K = 5, 3
    x = np.ones((1, 4, 4, C), np.int8)
    w = np.ones((3, 3, C, K), np.int8)
    taps = np.array([[4, 6, 6, 4], [6, 9, 9, 6], [6, 9, 9, 6], [4, 6, 6, 4]])
    acc = oracle.conv_acc_i8(x, w, 1, oracle.SAME)
    for k in range(K):
        assert np.array_equal(acc[0, :, :, k], C * taps)
    # stride 2, 3x3 SAME on a 4x4 image: total pad 1 -> 0 before, 1 after.
    # Along each axis output 0 covers inputs 0..2 (3 taps) and output 1
    # covers inputs 2..4, of which 2 are inside the image.
    acc2 = oracle.conv_acc_i8(x, w, 2, oracle.SAME)
    taps2 = np.array([[9, 6], [6, 4]])
    assert np.array_equal(acc2[0, :, :, 0], C * taps2)


def test_identity_filter_copies_input():
    rng = np.random.default_rng(6)
    C = 8
    x = rng.integers(-128, 128, size=(2, 5, 6, C)).astype(np.int8)
    w = np.zeros((3, 3, C, C), np.int8)
    for c in range(C):
        w[1, 1, c, c] = 1
    acc = oracle.conv_acc_i8(x, w, 1, oracle.SAME)
    assert np.array_equal(acc, x.astype(np.int32))
    y = oracle.epilogue_i8(acc, np.zeros(C, np.float32), None, 1.0, 0.0, relu=False)
    assert np.array_equal(y, x)


def test_padding_contributes_zero():
    # VALID on an input embedded in a zero border equals SAME on the input.
    rng = np.random.default_rng(7)
    for R, S in [(3, 3), (2, 4), (5, 1)]:
        x = rng.integers(-128, 128, size=(2, 6, 7, 3)).astype(np.int8)
        w = rng.integers(-128, 128, size=(R, S, 3, 4)).astype(np.int8)
        _, pt, pb = oracle.out_geometry(6, R, 1, oracle.SAME)
        _, pl, pr = oracle.out_geometry(7, S, 1, oracle.SAME)
        xp = np.zeros((2, 6 + pt + pb, 7 + pl + pr, 3), np.int8)
        xp[:, pt:pt + 6, pl:pl + 7, :] = x
        assert np.array_equal(oracle.conv_acc_i8(x, w, 1, oracle.SAME),
                              oracle.conv_acc_i8(xp, w, 1, oracle.VALID))


def test_points_match_full():
    rng = np.random.default_rng(8)
    x = rng.integers(-128, 128, size=(3, 9, 8, 16)).astype(np.int8)
    w = rng.integers(-128, 128, size=(3, 3, 16, 32)).astype(np.int8)
    for stride, pad in [(1, oracle.SAME), (2, oracle.SAME), ((2, 1), oracle.VALID)]:
        full = oracle.conv_acc_i8(x, w, stride, pad)
        idx = rng.choice(full.size, size=500, replace=False)
        assert np.array_equal(oracle.conv_acc_i8_points(x, w, idx, stride, pad), full.ravel()[idx])


def test_im2col_patch_order_and_zero_fill():
    # one 2x2x2 image, 2x2 filter, SAME stride 1 (pads 0 before, 1 after):
    # patch of output (0,0) = pixels (0,0),(0,1),(1,0),(1,1) in that order.
    img = np.arange(1, 9, dtype=np.int8).reshape(2, 2, 2)
    col = oracle.im2col(img, 2, 2, (0, 1, 0, 1), (1, 1))
    assert col.shape == (4, 8)
    assert col[0].tolist() == [1, 2, 3, 4, 5, 6, 7, 8]
    assert col[1].tolist() == [3, 4, 0, 0, 7, 8, 0, 0]
    assert col[3].tolist() == [7, 8, 0, 0, 0, 0, 0, 0]


# --------------------------------------------------------------------------
# bf16 fp64 reference
# --------------------------------------------------------------------------
def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_integer_inputs_equal_int_conv():
    rng = np.random.default_rng(9)
    x = rng.integers(-128, 128, size=(2, 5, 5, 8)).astype(np.int8)
    w = rng.integers(-128, 128, size=(3, 3, 8, 4)).astype(np.int8)
    xb, wb = _to_bf16_bits(x), _to_bf16_bits(w)
    assert np.array_equal(oracle.bf16_bits_to_f64(xb), x.astype(np.float64))
    acc = oracle.conv_acc_bf16_f64(xb, wb, 1, oracle.SAME)
    assert np.array_equal(acc, oracle.conv_acc_i8(x, w, 1, oracle.SAME).astype(np.float64))


def test_bf16_matches_torch_conv2d_f64():
    rng = np.random.default_rng(10)
    for stride, pad in [(1, oracle.SAME), (2, oracle.SAME), (1, oracle.VALID)]:
        xb = _to_bf16_bits(rng.standard_normal((2, 7, 6, 16)))
        wb = _to_bf16_bits(rng.standard_normal((3, 3, 16, 8)) / 12)
        acc = oracle.conv_acc_bf16_f64(xb, wb, stride, pad)
        ref = _torch_conv_f64(oracle.bf16_bits_to_f64(xb), oracle.bf16_bits_to_f64(wb),
                              (stride, stride), pad)
        assert np.allclose(acc, ref, rtol=1e-12, atol=1e-12)
        idx = rng.choice(acc.size, size=100, replace=False)
        pts = oracle.conv_acc_bf16_points_f64(xb, wb, idx, stride, pad)
        assert np.allclose(pts, acc.ravel()[idx], rtol=1e-12, atol=1e-12)


def test_epilogue_f64_hand_values():
    acc = np.array([[2.0, -3.0, 0.5]])
    bias = np.array([0.25, 0.5, -1.0], np.float32)
    side = _to_bf16_bits(np.array([[1.0, 2.0, 4.0]]))
    out = oracle.epilogue_f64(acc, bias, side, 0.5, 0.25, relu=False)
    # 2*0.5 + 1*0.25 + 0.25 = 1.5; -3*0.5 + 2*0.25 + 0.5 = -0.5; 0.25 + 1 - 1 = 0.25
    assert out.tolist() == [[1.5, -0.5, 0.25]]
    out = oracle.epilogue_f64(acc, bias, side, 0.5, 0.25, relu=True)
    assert out.tolist() == [[1.5, 0.0, 0.25]]
    out = oracle.epilogue_f64(acc, bias, None, 0.5, 0.25, relu=False)
    assert out.tolist() == [[1.25, -1.0, -0.75]]
