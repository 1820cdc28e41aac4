"""fconv_run_no_alloc: the fused run for callers that cannot allocate device
memory (the scratch comes from the library's built-in 32 MiB array).  Its
results must equal the oracle's and fconv_run's on the same inputs, call
after call, although every call reuses the same scratch: plain, split-K and
phased transposed plans.  Collected last on purpose."""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import fconv_inputs as FI  # noqa: E402
import oracle  # noqa: E402
import quantized_conv2d_gb300 as fc  # noqa: E402
from gpu_util import Case, PAD, to_dev, to_host  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_conv2d_gb300 import build
    build.build()
    oracle.build()


def _case(seed, N, H, W, C, K, dtype, side=True, relu=True):
    P, _, _ = oracle.out_geometry(H, 3, 1, oracle.SAME)
    Q, _, _ = oracle.out_geometry(W, 3, 1, oracle.SAME)
    inputs = FI.random_case(seed, N, H, W, C, K, 3, 3, dtype, (P, Q), side,
                            bias_std=1.0 if dtype == "int8" else 0.1)
    return Case(N, H, W, C, K, 3, 3, 1, "SAME", dtype, relu,
                0.002 if dtype == "int8" else 1.0, 0.5 if side else 0.0, inputs)


def _run_both(plan, c):
    x, w = to_dev(c.x, c.dtype), to_dev(c.w, c.dtype)
    bias = torch.from_numpy(c.bias).cuda()
    side = to_dev(c.side, c.dtype)
    stream = torch.cuda.current_stream()
    y_ref = plan.run(x, w, bias, side, c.conv_scale, c.side_scale)
    y_na = plan.new_output()
    fc.fconv_run_no_alloc(plan.handle, x.data_ptr(), w.data_ptr(), bias.data_ptr(),
                          side.data_ptr() if side is not None else None, c.conv_scale,
                          c.side_scale, y_na.data_ptr(), stream.cuda_stream)
    plan.check()
    return to_host(y_ref), to_host(y_na)


@pytest.mark.parametrize("gather", ["im2col", "halo"])
@pytest.mark.parametrize("dtype", ["int8", "bf16"])
def test_no_alloc_matches_fconv_run_twice(dtype, gather):
    # two calls in a row on the same plan, different inputs each time: the
    # second call must not see anything the first left in the scratch (the
    # im2col gather's int8 plan keeps its fp16 input and filter copies there;
    # the halo gather needs no scratch at all)
    first = _case(501, 4, 19, 21, 64, 96, dtype)
    second = _case(502, 4, 19, 21, 64, 96, dtype)
    plan = first.plan()
    fc.fconv_plan_set_gather(plan.handle, fc.FCONV_GATHER_IM2COL if gather == "im2col"
                             else fc.FCONV_GATHER_HALO)
    ws = fc.fconv_workspace_size(plan.handle)
    assert (ws > 0) == (gather == "im2col" and dtype == "int8")
    for c in (first, second):
        y_ref, y_na = _run_both(plan, c)
        c.check_output(y_na, c.oracle_out())
        c.check_output(y_ref, c.oracle_out())
        assert np.array_equal(y_na, y_ref)
    plan.close()


@pytest.mark.parametrize("dtype", ["int8", "bf16"])
def test_no_alloc_split_k_plan(dtype):
    # split-K keeps every unit's partial sums and the per-tile completion
    # counters in the scratch: the counters must start each call at zero
    # although the previous call's units left them there
    first = _case(511, 2, 9, 11, 64, 80, dtype)
    second = _case(512, 2, 9, 11, 64, 80, dtype)
    plan = first.plan()
    fc.fconv_plan_set_tile_shape(plan.handle, 128, 64)
    fc.fconv_plan_set_splits(plan.handle, 3)
    assert fc.fconv_plan_get_splits(plan.handle) == 3
    for c in (first, second, first):
        y_ref, y_na = _run_both(plan, c)
        c.check_output(y_na, c.oracle_out())
        assert np.array_equal(y_na, y_ref)
    plan.close()


def test_no_alloc_strided_transposed_plan():
    # a stride-2 transposed convolution runs as four phases, three of them on
    # the plan's side streams, each with its own packed filter in the scratch
    from test_gpu_convT import TCase
    first = TCase(521, 2, 8, 8, 64, 64, 4, 4, (1, 1, 1, 1), "int8", True, True, stride=(2, 2))
    second = TCase(522, 2, 8, 8, 64, 64, 4, 4, (1, 1, 1, 1), "int8", True, True, stride=(2, 2))
    plan = first.plan()
    assert fc.fconv_plan_launch_count(plan.handle) > 2
    for c in (first, second):
        y_ref, y_na = _run_both(plan, c)
        c.check_output(y_na, c.oracle_out())
        assert np.array_equal(y_na, y_ref)
    plan.close()


def test_no_alloc_rejects_plans_beyond_its_scratch():
    # int8 plans keep an fp16 copy of the input: N=256 56x56x48 needs ~77 MB
    plan = fc.Conv2dPlan(256, 56, 56, 48, 64, 3, 3, 1, "SAME", "int8", True)
    assert plan.ws_bytes > 32 * 2 ** 20
    y = torch.empty(16, dtype=torch.int8, device="cuda")
    with pytest.raises(fc.FconvError) as ei:
        fc.fconv_run_no_alloc(plan.handle, y.data_ptr(), y.data_ptr(), y.data_ptr(), None, 1.0,
                              0.0, y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert ei.value.status == fc.FCONV_ERR_WORKSPACE
    assert "32 MiB" in fc.fconv_last_error()
    plan.close()
