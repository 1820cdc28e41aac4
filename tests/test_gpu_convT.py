"""GPU parity of the transposed convolution (deconvolution forward with the
fused bias and epilogue) against the oracle's scatter definition: int8
bit-exact, bf16 within the usual bar."""
import numpy as np
import pytest
import torch

import fconv_inputs as FI
import oracle
import quantized_conv2d_gb300 as fc
from gpu_util import Case, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_conv2d_gb300 import build
    build.build()
    oracle.build()


class TCase(Case):
    """A Case whose oracle is the transposed convolution."""

    def __init__(self, seed, N, H, W, C, K, R, S, pads, dtype, side, relu, stride=(1, 1)):
        self.pads = pads
        self.tstride = stride
        Ho = oracle.convT_out_size(H, R, stride[0], pads[0], pads[1])
        Wo = oracle.convT_out_size(W, S, stride[1], pads[2], pads[3])
        inputs = FI.random_case(seed, N, H, W, C, K, R, S, dtype, (Ho, Wo), side,
                                bias_std=1.0 if dtype == "int8" else 0.1)
        cs = 40.0 / (np.sqrt(R * S * C) * 5461.0) if dtype == "int8" else 1.0
        super().__init__(N, H, W, C, K, R, S, 1, "VALID", dtype, relu, cs,
                         0.05 if side else 0.0, inputs)
        self.out_hw = (Ho, Wo)
        # bf16: w ~ N(0, 1/sqrt(R*S*C)), so an output of at most R*S*C
        # products has at most unit variance
        self.unit_variance = dtype == "bf16"

    def plan(self, block_n=None, debug=0):
        p = fc.Conv2dPlan(self.N, self.H, self.W, self.C, self.K, self.R, self.S, self.tstride,
                          "VALID", self.dtype, self.relu, transposed_pads=self.pads)
        assert p.out_shape == (self.N,) + self.out_hw + (self.K,)
        if block_n:
            p.set_tile(block_n)
        if debug:
            fc.fconv_plan_set_debug(p.handle, debug)
            bn, chunk, _ = p.config()
            chunked = chunk * 64 < self.R * self.S * self.C
            if debug & fc.FCONV_DEBUG_GATHER_CPASYNC and chunked and bn > 128:
                p.set_tile(128)
        return p

    def oracle_acc(self):
        if self.dtype == "int8":
            return oracle.convT_acc_i8(self.x, self.w, self.tstride, self.pads)
        return oracle.convT_acc_bf16_f64(self.x, self.w, self.tstride, self.pads)

    def check_acc(self, got, ref):
        if self.dtype == "int8":
            return super().check_acc(got, ref)
        # fp32 sums: the bound of the forward case, on the transposed sums of |x|, |w|
        absx = (self.x & np.uint16(0x7FFF)).astype(np.uint16)
        absw = (self.w & np.uint16(0x7FFF)).astype(np.uint16)
        mag = oracle.convT_acc_bf16_f64(absx, absw, self.tstride, self.pads)
        steps = -(-self.R * self.S * self.C // 16)
        err = np.abs(got.astype(np.float64) - ref)
        assert float((err / ((steps + 2) * 2.0 ** -22 * mag + 1e-30)).max(initial=0.0)) <= 1.0


CASES = [
    # N, H, W, C, K, R, S, (pt, pb, pl, pr), dtype, side, relu
    (2, 9, 11, 64, 80, 3, 3, (1, 1, 1, 1), "int8", True, True),      # TMA gather
    (2, 6, 7, 512, 144, 3, 3, (0, 2, 1, 0), "int8", True, False),    # chunked sums, asymmetric
    (3, 5, 8, 48, 32, 5, 3, (2, 0, 1, 2), "int8", False, True),      # cp.async gather
    (8, 16, 16, 256, 256, 4, 4, (1, 2, 1, 2), "int8", True, True),   # 16x16 -> 16x16, 4x4 filter
    (1, 1, 1, 16, 16, 3, 3, (0, 0, 0, 0), "int8", True, False),      # one pixel: the filter itself
    (2, 9, 11, 64, 80, 3, 3, (0, 0, 0, 0), "bf16", True, True),
    (2, 7, 5, 24, 40, 3, 2, (1, 2, 0, 1), "bf16", False, False),     # cp.async gather
]

# strided (upsampling) transposed convolutions: N, H, W, C, K, R, S, stride, pads, dtype, side, relu
STRIDED = [
    (2, 8, 8, 64, 64, 4, 4, (2, 2), (1, 1, 1, 1), "int8", True, True),      # 8x8 -> 16x16
    (2, 7, 9, 64, 48, 3, 3, (2, 2), (1, 0, 1, 0), "int8", True, False),     # adjustment 1
    (1, 5, 6, 48, 32, 5, 3, (3, 2), (2, -2, 0, -1), "int8", False, True),   # cp.async, pb < 0
    (2, 6, 6, 128, 64, 2, 2, (2, 2), (0, 0, 0, 0), "bf16", True, True),     # 2x2/2: no overlap
    (2, 4, 5, 32, 24, 3, 3, (2, 3), (1, 1, 2, 0), "bf16", False, False),
    (2, 6, 7, 64, 32, 3, 3, (2, 2), (2, 2, 2, 2), "int8", True, True),     # phases starting inside
    (2, 5, 5, 32, 32, 2, 2, (3, 3), (0, 0, 0, 0), "int8", True, False),    # stride > filter: zeros inserted
    (2, 5, 6, 16, 16, 1, 1, (2, 2), (0, -1, 0, 0), "bf16", True, True),    # 1x1 upsampling
]


@pytest.mark.parametrize("i,params", list(enumerate(CASES)))
def test_transposed_parity(i, params):
    N, H, W, C, K, R, S, pads, dtype, side, relu = params
    c = TCase(700 + i, N, H, W, C, K, R, S, pads, dtype, side, relu)
    acc_ref = c.oracle_acc()
    c.check_acc(c.accumulators_gpu(), acc_ref)
    ref = c.oracle_out(acc_ref)
    c.check_output(c.run_gpu(), ref)
    if C % 64 == 0:
        c.check_output(c.run_gpu(debug=fc.FCONV_DEBUG_GATHER_CPASYNC), ref)


@pytest.mark.parametrize("i,params", list(enumerate(STRIDED)))
def test_strided_transposed_parity(i, params):
    N, H, W, C, K, R, S, stride, pads, dtype, side, relu = params
    c = TCase(740 + i, N, H, W, C, K, R, S, pads, dtype, side, relu, stride=stride)
    acc_ref = c.oracle_acc()
    c.check_acc(c.accumulators_gpu(), acc_ref)
    ref = c.oracle_out(acc_ref)
    c.check_output(c.run_gpu(), ref)
    if C % 64 == 0:
        c.check_output(c.run_gpu(debug=fc.FCONV_DEBUG_GATHER_CPASYNC), ref)


@pytest.mark.parametrize("stride", [(1, 1), (2, 2)])
def test_transposed_host_buffers(stride):
    c = TCase(720, 6, 8, 8, 64, 32, 3, 3, (1, 1, 1, 1), "int8", True, True, stride=stride)
    p = c.plan()
    fc.fconv_plan_set_host_chunks(p.handle, 3)
    nbytes = fc.fconv_host_workspace_size(p.handle, True)
    dws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    y = np.empty(p.out_shape, np.int8)
    st = torch.cuda.current_stream()
    fc.fconv_run_host(p.handle, c.x.ctypes.data, c.w.ctypes.data, c.bias.ctypes.data,
                      c.side.ctypes.data, c.conv_scale, c.side_scale, y.ctypes.data,
                      dws.data_ptr(), nbytes, st.cuda_stream)
    st.synchronize()
    p.check()
    c.check_output(y, c.oracle_out())
    p.close()


def test_phased_plan_replays_from_a_cuda_graph():
    """A strided transposed plan is several launches (a prep and a conv per
    phase); captured once, it replays on new contents of the same buffers."""
    first = TCase(760, 2, 8, 8, 64, 64, 4, 4, (1, 1, 1, 1), "int8", True, True, stride=(2, 2))
    second = TCase(761, 2, 8, 8, 64, 64, 4, 4, (1, 1, 1, 1), "int8", True, True, stride=(2, 2))
    p = first.plan()
    assert fc.fconv_plan_launch_count(p.handle) == 8
    x, w = to_dev(first.x, "int8"), to_dev(first.w, "int8")
    bias, side = torch.from_numpy(first.bias).cuda(), to_dev(first.side, "int8")
    y = p.new_output()
    p.run(x, w, bias, side, first.conv_scale, first.side_scale, y=y)   # outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        p.run(x, w, bias, side, first.conv_scale, first.side_scale, y=y)
    for c in (second, first):
        x.copy_(to_dev(c.x, "int8"))
        w.copy_(to_dev(c.w, "int8"))
        bias.copy_(torch.from_numpy(c.bias).cuda())
        side.copy_(to_dev(c.side, "int8"))
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        p.check()
        c.check_output(to_host(y), c.oracle_out())
    p.close()


def test_phased_runs_back_to_back_share_the_workspace():
    """A strided transposed plan runs its phases on side streams joined back
    to the caller's stream; runs enqueued back to back (two input sets
    alternating over 8 runs, no synchronisation) all match the oracle, so a
    run's prep does not overwrite the workspace its predecessor's phases
    still read."""
    cases = [TCase(770 + i, 2, 8, 8, 64, 64, 4, 4, (1, 1, 1, 1), "int8", True, True,
                   stride=(2, 2)) for i in range(2)]
    p = cases[0].plan()
    ins = [(to_dev(c.x, "int8"), to_dev(c.w, "int8"), torch.from_numpy(c.bias).cuda(),
            to_dev(c.side, "int8")) for c in cases]
    ys = [p.new_output() for _ in range(8)]
    for i, y in enumerate(ys):
        x, w, bias, side = ins[i % 2]
        p.run(x, w, bias, side, cases[0].conv_scale, cases[0].side_scale, y=y)
    torch.cuda.synchronize()
    p.check()
    refs = [c.oracle_out() for c in cases]
    for i, y in enumerate(ys):
        cases[i % 2].check_output(to_host(y), refs[i % 2])
    p.close()
