"""CPU oracle for the fused quantized Conv2D forward pass.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA
library never loads it, and it imports nothing from the CUDA library.

The arithmetic lives in ``fconv_oracle.c`` (plain C, built with
``-ffp-contract=off``); this module only builds it, marshals numpy arrays and
composes the steps.  ``exact.py`` holds an exact-rational restatement of the
epilogue used to pin the C epilogue's floating-point rounding.

Definitions followed (page titles as printed on each page):
  * "conv_ops_fused_int8.cc": fused op semantics, BiasActivationOutputKernel
    epilogue and the SAME padding split;
  * "conv_grad_filter_ops.cc": Im2col patch order, zero taps outside the
    image and the output-size formula.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

SAME = 0
VALID = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fconv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["cc", "-std=c11", "-O3", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i32, i64, p = ctypes.c_int, ctypes.c_longlong, ctypes.c_void_p
        f32, f64 = ctypes.c_float, ctypes.c_double
        geo = [i32] * 13  # N H W C K R S sh sw pt pl P Q
        lib.orc_out_geometry.argtypes = [i32, i32, i32, i32, p, p, p]
        lib.orc_out_geometry.restype = i32
        lib.orc_conv_i8_direct.argtypes = [p, p] + geo + [p]
        lib.orc_conv_i8_points.argtypes = [p, p] + geo + [p, i64, p]
        lib.orc_conv_i8_partial_sums.argtypes = [p, p] + geo + [p]
        lib.orc_conv_bf16_direct_f64.argtypes = [p, p] + geo + [p]
        lib.orc_conv_bf16_points_f64.argtypes = [p, p] + geo + [p, i64, p]
        lib.orc_im2col.argtypes = [p, i32] + [i32] * 11 + [p]
        lib.orc_gemm_i8.argtypes = [p, p, i32, i32, i32, p]
        lib.orc_conv_i8_im2col.argtypes = [p, p] + [i32] * 13 + [p, p]
        lib.orc_convT_i8_direct.argtypes = [p, p] + [i32] * 13 + [p]
        lib.orc_convT_bf16_direct_f64.argtypes = [p, p] + [i32] * 13 + [p]
        lib.orc_epilogue_i8.argtypes = [p, i64, i32, p, p, f32, p, f32, i32, f32, f32, p]
        lib.orc_epilogue_f64.argtypes = [p, i64, i32, p, p, f64, p, f64, i32, f64, f64, p]
        lib.orc_num_threads.restype = i32
        for name in ("orc_conv_i8_direct", "orc_conv_i8_points", "orc_conv_i8_partial_sums",
                     "orc_conv_bf16_direct_f64", "orc_conv_bf16_points_f64",
                     "orc_im2col", "orc_gemm_i8", "orc_conv_i8_im2col",
                     "orc_epilogue_i8", "orc_epilogue_f64",
                     "orc_convT_i8_direct", "orc_convT_bf16_direct_f64"):
            getattr(lib, name).restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().orc_num_threads())


def out_geometry(size: int, filt: int, stride: int, padding: int):
    """(out, pad_before, pad_after) along one axis; raises if no output."""
    o, a, b = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = _load().orc_out_geometry(size, filt, stride, padding, ctypes.byref(o),
                                  ctypes.byref(a), ctypes.byref(b))
    if rc != 0:
        raise ValueError(f"no output for in={size} filt={filt} stride={stride} padding={padding}")
    return o.value, a.value, b.value


class Geometry:
    """Shapes and pads of one convolution, from the oracle's own rule."""

    def __init__(self, N, H, W, C, K, R, S, sh, sw, padding):
        self.N, self.H, self.W, self.C, self.K, self.R, self.S = N, H, W, C, K, R, S
        self.sh, self.sw, self.padding = sh, sw, padding
        self.P, self.pt, self.pb = out_geometry(H, R, sh, padding)
        self.Q, self.pl, self.pr = out_geometry(W, S, sw, padding)

    @property
    def out_shape(self):
        return (self.N, self.P, self.Q, self.K)

    def args(self):
        return (self.N, self.H, self.W, self.C, self.K, self.R, self.S, self.sh,
                self.sw, self.pt, self.pl, self.P, self.Q)


def _geom_of(x: np.ndarray, w: np.ndarray, stride, padding) -> Geometry:
    N, H, W, C = x.shape
    R, S, Cw, K = w.shape
    if Cw != C:
        raise ValueError("filter input depth must equal input depth")
    sh, sw = (stride, stride) if np.isscalar(stride) else stride
    return Geometry(N, H, W, C, K, R, S, sh, sw, padding)


def conv_acc_i8(x: np.ndarray, w: np.ndarray, stride=1, padding=SAME) -> np.ndarray:
    """Exact int32 conv sums, direct 7-loop.  x int8 NHWC, w int8 HWIO."""
    x = np.ascontiguousarray(x, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    g = _geom_of(x, w, stride, padding)
    acc = np.empty(g.out_shape, dtype=np.int32)
    _load().orc_conv_i8_direct(_ptr(x), _ptr(w), *g.args(), _ptr(acc))
    return acc


def conv_i8_partial_sum_bounds(x: np.ndarray, w: np.ndarray, stride=1, padding=SAME):
    """How large the int8 convolution's partial sums get (the page's CPU path
    sums in fp32, which is exact while they stay below 2^24).  Returns
    (max |acc|, max |prefix sum| with the products added in (r, s, c) patch
    order, max sum of |x*w|) over all outputs, as Python ints."""
    x = np.ascontiguousarray(x, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    g = _geom_of(x, w, stride, padding)
    if g.R * g.S * g.C >= 2 ** 17:
        raise ValueError("R*S*C must stay below 2^17 (int32 running sums)")
    out = np.zeros(3, dtype=np.int64)
    _load().orc_conv_i8_partial_sums(_ptr(x), _ptr(w), *g.args(), _ptr(out))
    return tuple(int(v) for v in out)


def conv_acc_i8_explicit(x, w, sh, sw, pt, pl, P, Q) -> np.ndarray:
    """The direct int32 conv sums with explicit top/left pads and output
    extents (taps outside the image contribute zero)."""
    x = np.ascontiguousarray(x, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    N, H, W, C = x.shape
    R, S, _, K = w.shape
    acc = np.empty((N, P, Q, K), dtype=np.int32)
    _load().orc_conv_i8_direct(_ptr(x), _ptr(w), N, H, W, C, K, R, S, sh, sw, pt, pl, P, Q,
                               _ptr(acc))
    return acc


def convT_out_size(size: int, filt: int, stride: int, pad_before: int, pad_after: int) -> int:
    """Output extent of the transposed convolution along one axis."""
    return (size - 1) * stride + filt - pad_before - pad_after


def convT_acc_i8(x, w, stride, pads) -> np.ndarray:
    """Exact int32 sums of the transposed convolution (scatter definition).
    pads = (top, bottom, left, right)."""
    x = np.ascontiguousarray(x, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    N, H, W, C = x.shape
    R, S, Cw, K = w.shape
    assert Cw == C
    sh, sw = (stride, stride) if np.isscalar(stride) else stride
    pt, pb, pl, pr = pads
    Ho, Wo = convT_out_size(H, R, sh, pt, pb), convT_out_size(W, S, sw, pl, pr)
    out = np.empty((N, Ho, Wo, K), dtype=np.int32)
    _load().orc_convT_i8_direct(_ptr(x), _ptr(w), N, H, W, C, K, R, S, sh, sw, pt, pl, Ho, Wo,
                                _ptr(out))
    return out


def convT_acc_bf16_f64(x_bits, w_bits, stride, pads) -> np.ndarray:
    """fp64 sums of the transposed convolution on bf16 inputs (bit patterns)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    N, H, W, C = x.shape
    R, S, Cw, K = w.shape
    assert Cw == C
    sh, sw = (stride, stride) if np.isscalar(stride) else stride
    pt, pb, pl, pr = pads
    Ho, Wo = convT_out_size(H, R, sh, pt, pb), convT_out_size(W, S, sw, pl, pr)
    out = np.empty((N, Ho, Wo, K), dtype=np.float64)
    _load().orc_convT_bf16_direct_f64(_ptr(x), _ptr(w), N, H, W, C, K, R, S, sh, sw, pt, pl, Ho,
                                      Wo, _ptr(out))
    return out


def conv_acc_i8_points(x, w, idx: np.ndarray, stride=1, padding=SAME) -> np.ndarray:
    """Exact int32 conv sums at flat NPQK indices ``idx``."""
    x = np.ascontiguousarray(x, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    g = _geom_of(x, w, stride, padding)
    out = np.empty(idx.shape, dtype=np.int32)
    _load().orc_conv_i8_points(_ptr(x), _ptr(w), *g.args(), _ptr(idx), idx.size, _ptr(out))
    return out


def conv_acc_i8_im2col(x: np.ndarray, w: np.ndarray, stride=1, padding=SAME) -> np.ndarray:
    """Exact int32 conv sums by im2col + GEMM (independent second path)."""
    x = np.ascontiguousarray(x, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    g = _geom_of(x, w, stride, padding)
    acc = np.empty(g.out_shape, dtype=np.int32)
    col = np.empty(g.P * g.Q * g.R * g.S * g.C, dtype=np.int8)
    _load().orc_conv_i8_im2col(_ptr(x), _ptr(w), g.N, g.H, g.W, g.C, g.K, g.R, g.S,
                               g.sh, g.sw, g.pt, g.pb, g.pl, g.pr, _ptr(acc), _ptr(col))
    return acc


def im2col(image: np.ndarray, R, S, pads, stride) -> np.ndarray:
    """Patch matrix [P*Q, R*S*C] of one HWC image (any 1/2/4/8-byte dtype)."""
    image = np.ascontiguousarray(image)
    H, W, C = image.shape
    pt, pb, pl, pr = pads
    sh, sw = stride
    P = (H + pt + pb - R) // sh + 1
    Q = (W + pl + pr - S) // sw + 1
    col = np.empty((P * Q, R * S * C), dtype=image.dtype)
    _load().orc_im2col(_ptr(image), image.itemsize, H, W, C, R, S, pt, pl, pb, pr,
                       sh, sw, _ptr(col))
    return col


def gemm_i8(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.int8)
    b = np.ascontiguousarray(b, dtype=np.int8)
    M, Kd = a.shape
    Kd2, N = b.shape
    assert Kd == Kd2
    c = np.empty((M, N), dtype=np.int32)
    _load().orc_gemm_i8(_ptr(a), _ptr(b), M, Kd, N, _ptr(c))
    return c


def conv_acc_bf16_f64(x_bits: np.ndarray, w_bits: np.ndarray, stride=1, padding=SAME) -> np.ndarray:
    """fp64 conv sums of bf16 inputs given as uint16 bit patterns."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    g = _geom_of(x, w, stride, padding)
    acc = np.empty(g.out_shape, dtype=np.float64)
    _load().orc_conv_bf16_direct_f64(_ptr(x), _ptr(w), *g.args(), _ptr(acc))
    return acc


def conv_acc_bf16_points_f64(x_bits, w_bits, idx, stride=1, padding=SAME) -> np.ndarray:
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    g = _geom_of(x, w, stride, padding)
    out = np.empty(idx.shape, dtype=np.float64)
    _load().orc_conv_bf16_points_f64(_ptr(x), _ptr(w), *g.args(), _ptr(idx), idx.size, _ptr(out))
    return out


# activation codes (the C oracle's): none, Relu, leaky Relu (alpha),
# clipped Relu (alpha), clamp to [alpha, beta]
ACT_NONE, ACT_RELU, ACT_LEAKY_RELU, ACT_CLIPPED_RELU, ACT_CLAMP = 0, 1, 2, 3, 4


def _act_code(relu) -> int:
    """`relu` is a bool (BiasAdd / BiasAdd+Relu) or one of the ACT_ codes."""
    if isinstance(relu, (bool, np.bool_)):
        return ACT_RELU if relu else ACT_NONE
    return int(relu)


def _scale_args(conv_scale, K):
    """(scalar, per-channel array or None): conv_scale is a number, or K
    values, one per output channel."""
    if np.ndim(conv_scale) == 0:
        return float(conv_scale), None
    sk = np.ascontiguousarray(conv_scale, dtype=np.float32)
    assert sk.shape == (K,)
    return 0.0, sk


def epilogue_i8(acc: np.ndarray, bias: np.ndarray, side: np.ndarray | None,
                conv_scale, side_scale: float, relu, alpha: float = 0.0,
                beta: float = 0.0) -> np.ndarray:
    """BiasActivationOutputKernel on int32 sums shaped [..., K] -> int8.
    conv_scale: a scalar, or K fp32 values (one per output channel).
    relu: a bool, or an ACT_ code (alpha/beta parametrise the others)."""
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    K = acc.shape[-1]
    bias = np.ascontiguousarray(bias, dtype=np.float32)
    assert bias.shape == (K,)
    if side is not None:
        side = np.ascontiguousarray(side, dtype=np.int8)
        assert side.shape == acc.shape
    cs, sk = _scale_args(conv_scale, K)
    out = np.empty(acc.shape, dtype=np.int8)
    _load().orc_epilogue_i8(_ptr(acc), acc.size // K, K, _ptr(bias), _ptr(side),
                            float(np.float32(cs)), _ptr(sk), float(np.float32(side_scale)),
                            _act_code(relu), float(np.float32(alpha)),
                            float(np.float32(beta)), _ptr(out))
    return out


def epilogue_f64(acc: np.ndarray, bias: np.ndarray, side_bits: np.ndarray | None,
                 conv_scale, side_scale: float, relu, alpha: float = 0.0,
                 beta: float = 0.0) -> np.ndarray:
    """fp64 reference epilogue of the bf16 variant (no output rounding)."""
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    K = acc.shape[-1]
    bias = np.ascontiguousarray(bias, dtype=np.float32)
    if side_bits is not None:
        side_bits = np.ascontiguousarray(side_bits, dtype=np.uint16)
        assert side_bits.shape == acc.shape
    cs, sk = _scale_args(conv_scale, K)
    out = np.empty(acc.shape, dtype=np.float64)
    _load().orc_epilogue_f64(_ptr(acc), acc.size // K, K, _ptr(bias), _ptr(side_bits),
                             cs, _ptr(sk), float(side_scale), _act_code(relu),
                             float(np.float32(alpha)), float(np.float32(beta)), _ptr(out))
    return out


def fused_conv_i8(x, w, bias, side, conv_scale, side_scale, relu, stride=1, padding=SAME):
    """The whole fused op: int8 output and the int32 sums it came from."""
    acc = conv_acc_i8(x, w, stride, padding)
    return epilogue_i8(acc, bias, side, conv_scale, side_scale, relu), acc


def fused_conv_bf16_ref(x_bits, w_bits, bias, side_bits, conv_scale, side_scale, relu,
                        stride=1, padding=SAME):
    """fp64 reference of the bf16 variant (unrounded)."""
    acc = conv_acc_bf16_f64(x_bits, w_bits, stride, padding)
    return epilogue_f64(acc, bias, side_bits, conv_scale, side_scale, relu)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact values of bf16 bit patterns."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)
