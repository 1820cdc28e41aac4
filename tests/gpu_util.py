"""Helpers shared by the GPU tests: move seeded inputs to the device, run
the CUDA path through the C ABI, and compute the oracle's answer."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import quantized_conv2d_gb300 as fc

PAD = {"SAME": oracle.SAME, "VALID": oracle.VALID}


def to_dev(a: np.ndarray | None, dtype: str):
    if a is None:
        return None
    if dtype == "int8" or a.dtype == np.int8:
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bf16_metric(y_bits: np.ndarray, ref: np.ndarray):
    """(max relative error with |ref| floored at 1e-2, mean absolute error)."""
    y = oracle.bf16_bits_to_f64(y_bits)
    err = np.abs(y - ref)
    rel = err / np.maximum(np.abs(ref), 1e-2)
    return float(rel.max(initial=0.0)), float(err.mean()) if err.size else 0.0


BF16_MAX_REL = 2e-2
BF16_MEAN_ABS = 1e-3


def bf16_round(v: np.ndarray) -> np.ndarray:
    """fp64 values rounded once to the nearest bf16 value (8 significant
    bits, ties to even): the best a bf16 output can be."""
    m, e = np.frexp(np.asarray(v, dtype=np.float64))   # m in [0.5, 1)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)     # rint: half to even


class Case:
    """One convolution problem with its inputs (numpy) and scalars."""

    def __init__(self, N, H, W, C, K, R, S, stride, padding, dtype, relu, conv_scale,
                 side_scale, inputs):
        self.N, self.H, self.W, self.C, self.K, self.R, self.S = N, H, W, C, K, R, S
        self.stride = (stride, stride) if isinstance(stride, int) else tuple(stride)
        self.padding, self.dtype, self.relu = padding, dtype, relu
        self.conv_scale, self.side_scale = conv_scale, side_scale
        self.alpha, self.beta = 0.0, 0.0   # activation parameters (relu may be an act code)
        # bf16: inputs drawn so that the outputs have about unit variance
        # (x ~ N(0,1), w ~ N(0, 1/sqrt(R*S*C)), conv_scale 1): the north-star
        # bar of mean |error| <= 1e-3 applies
        self.unit_variance = False
        self.x, self.w, self.bias, self.side = (inputs["x"], inputs["w"], inputs["bias"],
                                                inputs["side"])

    def geometry(self):
        return oracle.Geometry(self.N, self.H, self.W, self.C, self.K, self.R, self.S,
                               self.stride[0], self.stride[1], PAD[self.padding])

    def plan(self, block_n=None, debug=0):
        p = fc.Conv2dPlan(self.N, self.H, self.W, self.C, self.K, self.R, self.S, self.stride,
                          self.padding, self.dtype, self.relu, alpha=self.alpha, beta=self.beta)
        if block_n:
            p.set_tile(block_n)
        if debug:
            fc.fconv_plan_set_debug(p.handle, debug)
            bn, chunk, _ = p.config()
            chunked = chunk * 64 < self.R * self.S * self.C
            if debug & fc.FCONV_DEBUG_GATHER_CPASYNC and chunked and bn > 128:
                p.set_tile(128)   # the cp.async kernel folds chunks in TMEM: BN <= 128
        return p

    # ------------------------------------------------------------ GPU side
    def run_gpu(self, block_n=None, stream=None, debug=0):
        p = self.plan(block_n, debug)
        x, w = to_dev(self.x, self.dtype), to_dev(self.w, self.dtype)
        bias = torch.from_numpy(self.bias).cuda()
        side = to_dev(self.side, self.dtype)
        cs = self.conv_scale
        if np.ndim(cs) > 0:   # one scale per output channel, a device [K] fp32 vector
            cs = torch.from_numpy(np.ascontiguousarray(cs, dtype=np.float32)).cuda()
        y = p.run(x, w, bias, side, cs, self.side_scale, stream=stream)
        p.check(stream)
        out = to_host(y)
        p.close()
        return out

    def accumulators_gpu(self, block_n=None, debug=0):
        p = self.plan(block_n, debug)
        x, w = to_dev(self.x, self.dtype), to_dev(self.w, self.dtype)
        acc = p.accumulators(x, w)
        p.check()
        out = acc.cpu().numpy()
        p.close()
        return out

    # ------------------------------------------------------------ oracle side
    def oracle_acc(self):
        if self.dtype == "int8":
            return oracle.conv_acc_i8(self.x, self.w, self.stride, PAD[self.padding])
        return oracle.conv_acc_bf16_f64(self.x, self.w, self.stride, PAD[self.padding])

    def oracle_out(self, acc=None):
        if acc is None:
            acc = self.oracle_acc()
        if self.dtype == "int8":
            return oracle.epilogue_i8(acc, self.bias, self.side, self.conv_scale,
                                      self.side_scale, self.relu, self.alpha, self.beta)
        return oracle.epilogue_f64(acc, self.bias, self.side, self.conv_scale, self.side_scale,
                                   self.relu, self.alpha, self.beta)

    def check_output(self, got, ref, unit_variance_bar=False):
        """int8: bit-exact.  bf16: max relative error <= 2e-2 (|ref| floored
        at 1e-2), and a mean absolute error bar:
        * ``unit_variance_bar`` (the unit-variance ReLU workload): mean
          |y - ref| <= 1e-3 against the unrounded fp64 reference;
        * the case's ``unit_variance`` (unit-variance data with any
          activation): mean |y - bf16(ref)| <= 1e-3, the error beyond the
          output's own rounding (without a ReLU, the correctly rounded bf16
          values of N(0,1) data are already ~1.1e-3 from the unrounded
          reference on average);
        * else <= 2^-8 * mean|ref|, the most a single bf16 rounding (8
          significant bits) can add on average."""
        assert got.shape == ref.shape
        if self.dtype == "int8":
            bad = np.argwhere(got != ref)
            assert bad.size == 0, f"{len(bad)} int8 mismatches, first at {bad[:5].tolist()}"
        else:
            mx, mean = bf16_metric(got, ref)
            assert mx <= BF16_MAX_REL, (mx, mean)
            if unit_variance_bar:
                assert mean <= BF16_MEAN_ABS, (mx, mean)
            elif self.unit_variance:
                beyond = float(np.abs(oracle.bf16_bits_to_f64(got) - bf16_round(ref)).mean())
                assert beyond <= BF16_MEAN_ABS, (mx, mean, beyond)
            else:
                bar = 2.0 ** -8 * float(np.abs(ref).mean())
                assert mean <= bar, (mx, mean, bar)

    def check_acc(self, got, ref):
        assert got.shape == ref.shape
        if self.dtype == "int8":
            bad = np.argwhere(got != ref)
            assert bad.size == 0, f"{len(bad)} int32 mismatches, first at {bad[:5].tolist()}"
        else:
            # fp32 sums: the tensor core adds 16 exact products per step to
            # the fp32 accumulator, each step rounding (or truncating) by at
            # most ~2 ulps of the largest partial sum, so the error is bounded
            # by (steps + 2) * 2^-22 * sum|x*w| (the sum of |products|,
            # computed in fp64 by the oracle on |x| and |w|).
            err = np.abs(got.astype(np.float64) - ref)
            absx = (self.x & np.uint16(0x7FFF)).astype(np.uint16)
            absw = (self.w & np.uint16(0x7FFF)).astype(np.uint16)
            mag = oracle.conv_acc_bf16_f64(absx, absw, self.stride, PAD[self.padding])
            steps = -(-self.R * self.S * self.C // 16)
            bound = (steps + 2) * 2.0 ** -22 * mag + 1e-30
            worst = float((err / bound).max(initial=0.0))
            assert worst <= 1.0, f"fp32 sums off by {worst:.3g} x the rounding bound" 
