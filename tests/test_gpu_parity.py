"""GPU parity: the CUDA path, called through the C ABI, against the CPU
oracle on the same seeded inputs.  int8 outputs and int32 sums must match
bit for bit; bf16 outputs must meet max relative error <= 2e-2 (|ref|
floored at 1e-2) and mean absolute error <= 1e-3 against the fp64 oracle."""
import numpy as np
import pytest
import torch

import fconv_inputs as FI
import oracle
import quantized_conv2d_gb300 as fc
from gpu_util import Case, PAD, bf16_metric, to_dev, to_host, BF16_MAX_REL, BF16_MEAN_ABS

pytestmark = pytest.mark.gpu

SMALL = ["small_i8_16x16x32", "resnet_i8_56x56x64", "proj1x1s2_i8_28x28x256", "bf16_14x14x256"]


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_conv2d_gb300 import build
    build.build()
    oracle.build()


def workload_case(name, batch=None):
    wl = FI.workload(name)
    g = oracle.Geometry(wl.N, wl.H, wl.W, wl.C, wl.K, wl.R, wl.S, wl.stride, wl.stride,
                        PAD[wl.padding])
    inputs = FI.generate(wl, (g.P, g.Q), batch=batch)
    n = wl.N if batch is None else batch
    return Case(n, wl.H, wl.W, wl.C, wl.K, wl.R, wl.S, wl.stride, wl.padding, wl.dtype,
                wl.relu, wl.conv_scale, wl.side_scale, inputs)


def assert_fp32_exact_range(c, acc_ref):
    """int8: the oracle's int32 sums stay below 2^24, where they equal what
    the page's fp32 accumulation gives (the prefix bounds of every workload
    are checked on the CPU in test_oracle_partial_sums.py)."""
    if c.dtype == "int8":
        assert int(np.abs(acc_ref.astype(np.int64)).max()) < 2 ** 24


@pytest.mark.parametrize("name", SMALL)
def test_workload_full_parity(name):
    c = workload_case(name)
    acc_ref = c.oracle_acc()
    assert_fp32_exact_range(c, acc_ref)
    c.check_acc(c.accumulators_gpu(), acc_ref)
    c.check_output(c.run_gpu(), c.oracle_out(acc_ref), unit_variance_bar=True)


@pytest.mark.parametrize("name", ["proj1x1s1_i8_28x28x256", "fullwin_i8_7x7x512"])
def test_matrix_product_workloads_full_parity(name):
    """The two shapes the page's CPU helper computes as matrix products (a
    1x1 filter at stride 1, a filter covering the whole input under VALID):
    every int8 output and int32 sum against the oracle."""
    c = workload_case(name)
    acc_ref = c.oracle_acc()
    c.check_acc(c.accumulators_gpu(), acc_ref)
    c.check_output(c.run_gpu(), c.oracle_out(acc_ref))


def test_large_workload_full_parity():
    """N=256 28x28x512 3x3 SAME int8 with side input and ReLU, in the plan
    configuration the benchmark runs: every one of the 102,760,448 int8
    outputs and int32 sums against the oracle."""
    c = workload_case("large_i8_28x28x512")
    p = c.plan()
    assert p.config()[0] == 256 and fc.fconv_plan_get_splits(p.handle) == 1
    p.close()
    got = c.run_gpu()
    acc_gpu = c.accumulators_gpu()
    acc_ref = c.oracle_acc()
    assert acc_ref.shape == (256, 28, 28, 512)
    assert_fp32_exact_range(c, acc_ref)
    c.check_acc(acc_gpu, acc_ref)
    del acc_gpu
    ref = c.oracle_out(acc_ref)
    c.check_output(got, ref)
    assert got.size == 102760448


SWEEP = [
    # N, H, W, C, K, R, S, stride, padding, side, relu
    (1, 1, 1, 16, 16, 1, 1, 1, "SAME", False, False),
    (1, 5, 7, 16, 48, 3, 3, 1, "SAME", True, True),
    (2, 9, 11, 48, 80, 3, 3, 2, "SAME", True, False),      # odd sizes, stride 2, odd pads
    (3, 8, 8, 32, 16, 3, 3, 2, "SAME", False, True),       # total pad 1: 0 before, 1 after
    (1, 13, 6, 80, 144, 5, 5, 1, "SAME", True, True),      # K tail over 128 / 64 / 32 tiles
    (2, 2, 3, 16, 32, 3, 3, 1, "SAME", False, False),      # image smaller than the filter
    (2, 10, 10, 64, 64, 3, 3, (1, 2), "SAME", True, True),
    (4, 7, 7, 16, 32, 2, 4, 1, "VALID", False, False),
    (1, 7, 7, 128, 32, 7, 7, 1, "VALID", True, True),      # full-window VALID = matmul
    (5, 6, 6, 256, 256, 1, 1, 1, "SAME", False, False),    # 1x1 stride 1 = matmul
    (3, 17, 15, 32, 96, 3, 3, 3, "SAME", True, False),
    (1, 30, 30, 1024, 32, 3, 3, 1, "SAME", True, True),    # 9216 k-values: 10 chunks
    (2, 12, 12, 512, 272, 3, 3, 1, "SAME", True, True),    # 4608 k-values, K tail
    (7, 9, 9, 16, 16, 1, 1, 2, "VALID", True, False),
    (2, 11, 9, 64, 96, 5, 3, 2, "SAME", True, True),       # R != S, stride 2, odd pads
    (3, 8, 8, 128, 64, 3, 3, 2, "SAME", False, False),     # total pad 1: 0 before, 1 after
    (2, 7, 12, 192, 48, 1, 3, (2, 1), "VALID", True, True),
    (1, 20, 3, 64, 32, 4, 2, 3, "SAME", False, True),      # stride 3, even filters
    (3, 11, 13, 64, 80, 1, 1, (2, 3), "SAME", True, True),  # 1x1 strided: subsampled copy, TMA
    (2, 10, 9, 48, 32, 1, 1, 3, "VALID", True, False),      # 1x1 stride 3: subsampled, cp.async
    (2, 3, 4, 16, 16, 3, 3, 5, "SAME", True, True),         # stride above the image: 1x1 output
    (1, 2, 2, 64, 16, 5, 5, 4, "SAME", True, False),        # 5x5 on 2x2, stride 4: pads 1 and 2
]

# shapes whose channel count lets the kernel gather A with TMA im2col loads
TMA_SHAPES = [i for i, p in enumerate(SWEEP) if p[3] % 64 == 0]


def sweep_case(i, params, dtype):
    N, H, W, C, K, R, S, stride, pad, side, relu = params
    sh, sw = (stride, stride) if isinstance(stride, int) else stride
    P, _, _ = oracle.out_geometry(H, R, sh, PAD[pad])
    Q, _, _ = oracle.out_geometry(W, S, sw, PAD[pad])
    inputs = FI.random_case(1000 + i, N, H, W, C, K, R, S, dtype, (P, Q), side,
                            bias_std=1.0 if dtype == "int8" else 0.1)
    cs = 0.001 if dtype == "int8" else 1.0
    c = Case(N, H, W, C, K, R, S, (sh, sw), pad, dtype, relu, cs, 0.25 if side else 0.0, inputs)
    c.unit_variance = dtype == "bf16"   # x ~ N(0,1), w ~ N(0, 1/sqrt(R*S*C)), scale 1
    return c


@pytest.mark.parametrize("i,params", list(enumerate(SWEEP)))
def test_sweep_int8(i, params):
    c = sweep_case(i, params, "int8")
    acc_ref = c.oracle_acc()
    c.check_acc(c.accumulators_gpu(), acc_ref)
    c.check_output(c.run_gpu(), c.oracle_out(acc_ref))


@pytest.mark.parametrize("i,params", [(i, p) for i, p in enumerate(SWEEP) if p[3] % 8 == 0])
def test_sweep_bf16(i, params):
    c = sweep_case(i, params, "bf16")
    acc_ref = c.oracle_acc()
    c.check_acc(c.accumulators_gpu(), acc_ref)
    c.check_output(c.run_gpu(), c.oracle_out(acc_ref))


@pytest.mark.parametrize("dtype", ["int8", "bf16"])
@pytest.mark.parametrize("i", TMA_SHAPES)
def test_both_gathers_agree(i, dtype):
    """The TMA im2col gather and the cp.async gather give the same sums."""
    c = sweep_case(i, SWEEP[i], dtype)
    acc_ref = c.oracle_acc()
    tma = c.accumulators_gpu()
    cpa = c.accumulators_gpu(debug=fc.FCONV_DEBUG_GATHER_CPASYNC)
    c.check_acc(tma, acc_ref)
    c.check_acc(cpa, acc_ref)
    if dtype == "int8":
        assert np.array_equal(tma, cpa)
    c.check_output(c.run_gpu(debug=fc.FCONV_DEBUG_GATHER_CPASYNC), c.oracle_out(acc_ref))


@pytest.mark.parametrize("dtype", ["int8", "bf16"])
def test_every_tile_gives_the_same_result(dtype):
    c = sweep_case(50, (2, 9, 9, 64, 256, 3, 3, 1, "SAME", True, True), dtype)
    ref = c.oracle_out()
    outs = {}
    for bn in (32, 64, 128, 256):
        try:
            outs[bn] = c.run_gpu(block_n=bn)
        except fc.FconvError as e:
            assert e.status == fc.FCONV_ERR_NOT_SUPPORTED
            continue
        c.check_output(outs[bn], ref)
    assert len(outs) >= 3
    if dtype == "int8":
        first = next(iter(outs.values()))
        for v in outs.values():
            assert np.array_equal(v, first)


# Plans that fill two k-blocks a pipeline stage (unsplit, unchunked 128-pixel
# tiles of <= 128 channels and >= 12 k-blocks; int8 sums are unchunked up to
# 15): (N, H, W, C, K, R, S, stride, pad, side, relu), block_n.  Odd k-block counts end a unit with a stage of one k-block; K not
# a multiple of 64 takes the 2-D filter boxes (128 k-rows deep).
KB2_CASES = [
    ((2, 14, 14, 832, 128, 1, 1, 1, "VALID", False, True), 128),  # 13 k-blocks
    ((3, 9, 7, 768, 96, 1, 1, 1, "VALID", True, False), 128),     # 12 k-blocks, K = 96, ragged M
    ((2, 8, 8, 192, 64, 2, 2, 1, "SAME", True, True), 64),        # BN 64, 2x2 filter, 12 k-blocks
    ((2, 10, 10, 896, 208, 1, 1, 2, "VALID", False, True), 128),  # 14 k-blocks, stride 2, K = 208
]


@pytest.mark.parametrize("dtype", ["int8", "bf16"])
@pytest.mark.parametrize("i", range(len(KB2_CASES)))
def test_two_kblock_stages_agree(i, dtype):
    """Stages of two k-blocks give the oracle's sums and outputs, and (int8)
    the same sums as stages of one k-block."""
    params, bn = KB2_CASES[i]
    c = sweep_case(80 + i, params, dtype)
    p = c.plan(block_n=bn)
    assert fc.fconv_plan_kernel(p.handle) == "tma-im2col-kb2-dual"
    fc.fconv_plan_set_debug(p.handle, fc.FCONV_DEBUG_ONE_KBLOCK_STAGES)
    assert fc.fconv_plan_kernel(p.handle) == "tma-im2col-dual"
    p.close()
    acc_ref = c.oracle_acc()
    two = c.accumulators_gpu(block_n=bn)
    one = c.accumulators_gpu(block_n=bn, debug=fc.FCONV_DEBUG_ONE_KBLOCK_STAGES)
    c.check_acc(two, acc_ref)
    c.check_acc(one, acc_ref)
    if dtype == "int8":
        assert np.array_equal(two, one)
    c.check_output(c.run_gpu(block_n=bn), c.oracle_out(acc_ref))
    c.check_output(c.run_gpu(block_n=bn, debug=fc.FCONV_DEBUG_ONE_KBLOCK_STAGES),
                   c.oracle_out(acc_ref))


# two threads issuing each k-block's MMAs (half the k16 steps each) into two
# accumulators the epilogue adds, against one issuing thread and the oracle
DUAL_CASES = KB2_CASES + [
    ((1, 30, 30, 1024, 32, 3, 3, 1, "SAME", True, True), 128),   # 144 k-blocks (int8: chunked)
    ((2, 12, 12, 512, 272, 3, 3, 1, "SAME", True, True), 128),   # 72 k-blocks, K tail
    ((128, 14, 14, 256, 128, 3, 3, 1, "SAME", True, True), 128), # 196 tiles: CTAs with two
]


@pytest.mark.parametrize("dtype", ["int8", "bf16"])
@pytest.mark.parametrize("i", range(len(DUAL_CASES)))
def test_split_mma_issue_agrees(i, dtype):
    params, bn = DUAL_CASES[i]
    c = sweep_case(1300 + i, params, dtype)
    p = c.plan(block_n=bn)
    assert fc.fconv_plan_kernel(p.handle).endswith("-dual")
    fc.fconv_plan_set_debug(p.handle, fc.FCONV_DEBUG_ONE_MMA_ISSUER)
    assert not fc.fconv_plan_kernel(p.handle).endswith("-dual")
    p.close()
    acc_ref = c.oracle_acc()
    two = c.accumulators_gpu(block_n=bn)
    one = c.accumulators_gpu(block_n=bn, debug=fc.FCONV_DEBUG_ONE_MMA_ISSUER)
    c.check_acc(two, acc_ref)
    c.check_acc(one, acc_ref)
    if dtype == "int8":
        assert np.array_equal(two, one)
    c.check_output(c.run_gpu(block_n=bn), c.oracle_out(acc_ref))


def test_two_kblock_stages_long_bf16():
    """A 36-k-block bf16 layer (the 32x14x14x256 workload's shape on 2
    images): two k-blocks a stage against the oracle."""
    c = sweep_case(90, (2, 14, 14, 256, 256, 3, 3, 1, "SAME", False, True), "bf16")
    p = c.plan(block_n=128)
    assert fc.fconv_plan_kernel(p.handle) == "tma-im2col-kb2-dual"
    p.close()
    acc_ref = c.oracle_acc()
    c.check_acc(c.accumulators_gpu(block_n=128), acc_ref)
    c.check_output(c.run_gpu(block_n=128), c.oracle_out(acc_ref))


@pytest.mark.parametrize("xv,wv", [(127, 127), (-128, -128), (-128, 127), (None, None)])
def test_chunked_sums_are_exact_at_extreme_magnitudes(xv, wv):
    """Sums far beyond 2^24 (up to 9*1024*16384), where a single fp32
    accumulation would round: the int32 folding of exact chunks must give
    the exact sum."""
    N, H, W, C, K = 2, 6, 6, 1024, 32
    rng = np.random.default_rng(7)
    if xv is None:
        x = rng.choice(np.array([-128, 127, 127, 126], np.int8), size=(N, H, W, C))
        w = rng.choice(np.array([-128, 127, -127], np.int8), size=(3, 3, C, K))
    else:
        x = np.full((N, H, W, C), xv, np.int8)
        w = np.full((3, 3, C, K), wv, np.int8)
    inputs = {"x": x, "w": w, "bias": np.zeros(K, np.float32), "side": None}
    c = Case(N, H, W, C, K, 3, 3, 1, "SAME", "int8", False, 1e-7, 0.0, inputs)
    acc_ref = c.oracle_acc()
    assert np.abs(acc_ref).max() > 2 ** 24 or xv is None
    c.check_acc(c.accumulators_gpu(), acc_ref)
    c.check_output(c.run_gpu(), c.oracle_out(acc_ref))


def test_epilogue_rounding_order_cases():
    """Inputs on which any other arrangement of the three fp32 steps changes
    the int8 result (found by exact rational search): each sum is built by a
    1x1 conv over 32 channels, w = (127, ..., 127, 1)."""
    from epilogue_cases import discriminating_groups
    C, K = 32, 16
    groups = discriminating_groups()
    assert groups
    for (cs, ss, bias, relu), rows in groups:
        M = len(rows)
        x = np.zeros((M, 1, 1, C), np.int8)
        for i, (acc, _, _) in enumerate(rows):
            q, r = divmod(acc, 127)
            if r > 63:
                q, r = q + 1, r - 127
            # spread q over 31 channels of weight 127, r on the weight-1 channel
            parts = np.full(31, q // 31, np.int64)
            parts[: q % 31] += 1
            assert np.abs(parts).max() <= 127 and abs(r) <= 127
            x[i, 0, 0, :31] = parts
            x[i, 0, 0, 31] = r
            assert int(x[i, 0, 0, :31].astype(np.int64).sum()) * 127 + int(x[i, 0, 0, 31]) == acc
        w = np.zeros((1, 1, C, K), np.int8)
        w[0, 0, :31, :] = 127
        w[0, 0, 31, :] = 1
        side = None
        if ss != 0.0:
            side = np.zeros((M, 1, 1, K), np.int8)
            for i, (_, s, _) in enumerate(rows):
                side[i] = s
        inputs = {"x": x, "w": w, "bias": np.full(K, bias, np.float32), "side": side}
        c = Case(M, 1, 1, C, K, 1, 1, 1, "SAME", "int8", relu, cs, ss, inputs)
        got = c.run_gpu()
        expect = np.array([r[2] for r in rows], np.int8)
        assert np.array_equal(got[:, 0, 0, :], np.repeat(expect[:, None], K, axis=1)), (cs, ss, bias)
        assert np.array_equal(got, c.oracle_out())


def test_side_stream_and_guard_bytes():
    c = sweep_case(60, (3, 11, 9, 48, 48, 3, 3, 1, "SAME", True, True), "int8")
    p = c.plan()
    x, w = to_dev(c.x, "int8"), to_dev(c.w, "int8")
    bias = torch.from_numpy(c.bias).cuda()
    side = to_dev(c.side, "int8")
    n_out = int(np.prod(p.out_shape))
    guard = torch.full((n_out + 4096,), 0x5A, dtype=torch.int8, device="cuda")
    y = guard[:n_out].view(p.out_shape)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        p.run(x, w, bias, side, c.conv_scale, c.side_scale, y=y, stream=s)
    p.check(s)
    assert torch.all(guard[n_out:] == 0x5A)
    c.check_output(to_host(y), c.oracle_out())
    p.close()


@pytest.mark.parametrize("chunks,splits", [(0, 1), (1, 1), (3, 1), (3, 3)])
@pytest.mark.parametrize("dtype", ["int8", "bf16"])
def test_run_host_buffers(chunks, splits, dtype):
    """fconv_run_host: host buffers in, host buffer out, the batch split into
    pipelined chunks (7 images in 3 chunks leaves a ragged last chunk), with
    and without split-K (each chunk's tiles split over three units)."""
    c = sweep_case(90, (7, 12, 10, 64, 48, 3, 3, 1, "SAME", True, True), dtype)
    p = c.plan()
    fc.fconv_plan_set_host_chunks(p.handle, chunks)
    if splits > 1:
        fc.fconv_plan_set_tile_shape(p.handle, 128, 64)
        fc.fconv_plan_set_splits(p.handle, splits)
    nbytes = fc.fconv_host_workspace_size(p.handle, True)
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    def pinned(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).pin_memory()
        return torch.from_numpy(a).pin_memory()

    xh, wh, bh, sh = pinned(c.x), pinned(c.w), pinned(c.bias), pinned(c.side)
    yh = torch.empty(p.out_shape, dtype=torch.int8 if dtype == "int8" else torch.int16).pin_memory()
    s = torch.cuda.current_stream()
    for _ in range(2):   # twice: the internal streams and events are reused
        yh.zero_()
        fc.fconv_run_host(p.handle, xh.data_ptr(), wh.data_ptr(), bh.data_ptr(), sh.data_ptr(),
                          c.conv_scale, c.side_scale, yh.data_ptr(), dev.data_ptr(), nbytes,
                          s.cuda_stream)
        p.check()
        got = yh.numpy() if dtype == "int8" else yh.numpy().view(np.uint16)
        c.check_output(got, c.oracle_out())
    p.close()


def test_run_host_ramped_chunks():
    """fconv_run_host's automatic chunks on a batch of more than ten waves of
    output tiles: the ramped schedule (short first and last chunks, whole
    waves between) on this GPU's SM count, every output against the oracle."""
    c = sweep_case(91, (64, 28, 28, 32, 256, 3, 3, 1, "SAME", True, True), "int8")
    p = c.plan()
    fc.fconv_plan_set_tile(p.handle, 64)           # 4 channel tiles: 24.5 tiles an image
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sizes = fc.fconv_plan_host_chunk_sizes(p.handle, sms)
    assert sum(sizes) == c.N and len(sizes) > 3 and sizes[0] < sizes[3] > sizes[-1], sizes
    nbytes = fc.fconv_host_workspace_size(p.handle, True)
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    xh, wh = torch.from_numpy(c.x).pin_memory(), torch.from_numpy(c.w).pin_memory()
    bh, sh = torch.from_numpy(c.bias).pin_memory(), torch.from_numpy(c.side).pin_memory()
    yh = torch.empty(p.out_shape, dtype=torch.int8).pin_memory()
    s = torch.cuda.current_stream()
    fc.fconv_run_host(p.handle, xh.data_ptr(), wh.data_ptr(), bh.data_ptr(), sh.data_ptr(),
                      c.conv_scale, c.side_scale, yh.data_ptr(), dev.data_ptr(), nbytes,
                      s.cuda_stream)
    p.check()
    c.check_output(yh.numpy(), c.oracle_out())
    p.close()


@pytest.mark.parametrize("dtype", ["int8", "bf16"])
@pytest.mark.parametrize("C,K,kernel", [(16, 16, "cp-async"), (64, 64, "tma-im2col"),
                                         (64, 256, "tma-im2col"), (64, 128, "tma-im2col-m256"),
                                         (832, 64, "tma-im2col-kb2-dual"), (64, 64, "tma-halo"),
                                         (64, 128, "tma-halo-m256")])
def test_timeout_exit_keeps_context_usable(C, K, kernel, dtype):
    """A producer that never signals 'stage full' makes the MMA issuer's wait
    run out: the kernel must stop, report FCONV_ERR_TIMEOUT, and the next run
    must work -- for the cp.async loaders and the TMA producers (64- and
    256-wide tiles, 256-pixel tiles, stages of two k-blocks, and the halo
    gather's window loaders, whose int8 form waits for its own copy)."""
    if dtype == "bf16" and not kernel.startswith("tma-halo"):
        pytest.skip("the other loaders wait the same way for both dtypes")
    R = 1 if C > 512 else 3   # 832 channels, 1x1: 13 k-blocks, unchunked
    c = sweep_case(70, (1, 8, 8, C, K, R, R, 1, "SAME", False, True), dtype)
    # a fixed tile is unsplit
    p = c.plan(block_n=256 if K == 256 else (64 if C > 512 else None))
    if kernel.startswith("tma-im2col"):
        fc.fconv_plan_set_gather(p.handle, fc.FCONV_GATHER_IM2COL)
    if kernel.startswith("tma-halo"):
        fc.fconv_plan_set_gather(p.handle, fc.FCONV_GATHER_HALO)
    if kernel.endswith("m256"):
        fc.fconv_plan_set_tile_shape(p.handle, 256, 64 if kernel.startswith("tma-halo") else K)
    elif kernel == "tma-halo":
        fc.fconv_plan_set_tile_shape(p.handle, 128, 64)
    assert fc.fconv_plan_kernel(p.handle) == kernel
    fc.fconv_plan_set_timeout_ms(p.handle, 50)
    fc.fconv_plan_set_debug(p.handle, fc.FCONV_DEBUG_DROP_ARRIVE)
    x, w = to_dev(c.x, dtype), to_dev(c.w, dtype)
    bias = torch.from_numpy(c.bias).cuda()
    p.run(x, w, bias, None, c.conv_scale, 0.0)
    with pytest.raises(fc.FconvError) as ei:
        p.check()
    assert ei.value.status == fc.FCONV_ERR_TIMEOUT
    fc.fconv_plan_set_debug(p.handle, 0)
    y = p.run(x, w, bias, None, c.conv_scale, 0.0)
    p.check()
    c.check_output(to_host(y), c.oracle_out())
    p.close()


def test_misaligned_device_pointer_is_rejected():
    c = sweep_case(80, (1, 8, 8, 16, 16, 3, 3, 1, "SAME", False, True), "int8")
    p = c.plan()
    buf = torch.zeros(8 * 8 * 16 + 64, dtype=torch.int8, device="cuda")
    w = to_dev(c.w, "int8")
    bias = torch.from_numpy(c.bias).cuda()
    y = p.new_output()
    with pytest.raises(fc.FconvError) as ei:
        fc.fconv_run(p.handle, buf.data_ptr() + 1, w.data_ptr(), bias.data_ptr(), None, 1.0, 0.0,
                     y.data_ptr(), p.workspace.data_ptr(), p.workspace.numel(),
                     torch.cuda.current_stream().cuda_stream)
    assert ei.value.status == fc.FCONV_ERR_MISALIGNED
    p.close()


# ---------------------------------------------------------------- split-K
# each tile's k-blocks over several CTAs; the last of a tile portion's units
# adds the partial sums (int32 exactly, fp32 in split order) and stores
SPLIT_CASES = [
    ((2, 9, 11, 64, 80, 3, 3, 1, "SAME", True, True), "int8", (128, 64), 3),
    ((2, 9, 11, 64, 80, 3, 3, 1, "SAME", True, False), "int8", (128, 128), 2),   # K tail
    ((2, 12, 12, 512, 272, 3, 3, 1, "SAME", True, True), "int8", (128, 256), 2),  # chunked units
    ((2, 12, 12, 512, 272, 3, 3, 1, "SAME", True, True), "int8", (128, 128), 5),  # one chunk a unit
    ((3, 9, 11, 64, 64, 3, 3, 1, "SAME", True, True), "int8", (128, 64), 4),      # 2 of 3 k-blocks
    ((3, 8, 8, 64, 200, 3, 3, 1, "SAME", True, False), "bf16", (128, 128), 3),
    ((2, 9, 11, 128, 96, 3, 3, 2, "SAME", False, True), "bf16", (128, 64), 4),
]


@pytest.mark.parametrize("i,item", list(enumerate(SPLIT_CASES)))
def test_split_k(i, item):
    params, dtype, shape, splits = item
    c = sweep_case(700 + i, params, dtype)
    acc_ref = c.oracle_acc()
    p = c.plan()
    fc.fconv_plan_set_tile_shape(p.handle, *shape)
    fc.fconv_plan_set_splits(p.handle, splits)
    assert fc.fconv_plan_get_splits(p.handle) > 1
    x, w = to_dev(c.x, dtype), to_dev(c.w, dtype)
    bias = torch.from_numpy(c.bias).cuda()
    side = to_dev(c.side, dtype)
    acc = p.accumulators(x, w)
    y = p.run(x, w, bias, side, c.conv_scale, c.side_scale)
    y2 = p.run(x, w, bias, side, c.conv_scale, c.side_scale)   # counters zeroed again
    p.check()
    c.check_acc(acc.cpu().numpy(), acc_ref)
    c.check_output(to_host(y), c.oracle_out(acc_ref))
    assert torch.equal(y, y2)   # the same sums in the same order


def test_split_k_with_channel_scale_and_graph_replay():
    c = sweep_case(710, (2, 9, 11, 64, 80, 3, 3, 1, "SAME", True, True), "int8")
    c.conv_scale = _channel_scales(710, c.K, "int8")
    p = c.plan()
    fc.fconv_plan_set_splits(p.handle, 3)
    assert fc.fconv_plan_get_splits(p.handle) == 3
    ref = c.oracle_out(c.oracle_acc())
    x, w = to_dev(c.x, "int8"), to_dev(c.w, "int8")
    bias, side = torch.from_numpy(c.bias).cuda(), to_dev(c.side, "int8")
    scale = torch.from_numpy(c.conv_scale).cuda()
    y = p.new_output()
    p.run(x, w, bias, side, scale, c.side_scale, y=y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        p.run(x, w, bias, side, scale, c.side_scale, y=y)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        p.check()
        c.check_output(to_host(y), ref)
    p.close()


def test_split_k_chosen_for_a_batch_one_deep_layer():
    """One image of 7x7x512 -> 512, 3x3: a handful of tiles and 72 k-blocks,
    where the plan splits K on its own."""
    c = sweep_case(720, (1, 7, 7, 512, 512, 3, 3, 1, "SAME", True, True), "int8")
    p = c.plan()
    assert fc.fconv_plan_get_splits(p.handle) > 1
    c.check_output(c.run_gpu(), c.oracle_out(c.oracle_acc()))
    p.close()


# ---------------------------------------------------------------- per-channel scale
# (shape, dtype): TMA gather (C % 64 == 0) and cp.async gather, chunked int8
# sums, K tails past 32/64/128-wide tiles
CHANNEL_SCALE_SHAPES = [
    ((2, 9, 11, 64, 80, 3, 3, 1, "SAME", True, True), "int8"),
    ((2, 9, 11, 48, 144, 3, 3, 2, "SAME", True, False), "int8"),
    ((2, 12, 12, 512, 272, 3, 3, 1, "SAME", True, True), "int8"),
    ((3, 8, 8, 64, 200, 3, 3, 1, "SAME", True, False), "bf16"),
    ((2, 7, 9, 24, 40, 3, 3, 1, "VALID", False, True), "bf16"),
]


def _channel_scales(seed, K, dtype):
    rng = np.random.default_rng(seed)
    if dtype == "int8":
        # a different binade per channel: a wrong channel index moves outputs
        return (2.0 ** rng.integers(-13, -8, size=K) * rng.uniform(1, 2, size=K)).astype(np.float32)
    return rng.uniform(0.25, 4.0, size=K).astype(np.float32)


@pytest.mark.parametrize("i,item", list(enumerate(CHANNEL_SCALE_SHAPES)))
def test_per_channel_conv_scale(i, item):
    params, dtype = item
    c = sweep_case(300 + i, params, dtype)
    c.conv_scale = _channel_scales(300 + i, c.K, dtype)
    c.unit_variance = False   # channel scales up to 4 widen the outputs
    acc_ref = c.oracle_acc()
    c.check_output(c.run_gpu(), c.oracle_out(acc_ref))
    if params[3] % 64 == 0:
        c.check_output(c.run_gpu(debug=fc.FCONV_DEBUG_GATHER_CPASYNC), c.oracle_out(acc_ref))


@pytest.mark.parametrize("dtype", ["int8", "bf16"])
def test_batchnorm_folded_block(dtype):
    """A conv-BN-add-Relu block: batch-norm inference folded on the host
    (fconv_fold_batchnorm) into the per-channel scale and bias, then one fused
    run.  Bit-exact (int8) against the oracle epilogue with the folded
    parameters, and within one output step of the unfused normalisation
    evaluated in double."""
    c = sweep_case(325, (2, 10, 12, 64, 80, 3, 3, 1, "SAME", True, True), dtype)
    rng = np.random.default_rng(325)
    K = c.K
    acc_ref = c.oracle_acc()
    y_conv = acc_ref.astype(np.float64) * np.float32(c.conv_scale) + c.bias.astype(np.float64)
    # the batch's own statistics, and a gamma that spreads the int8 outputs
    mean = y_conv.reshape(-1, K).mean(axis=0).astype(np.float32)
    var = y_conv.reshape(-1, K).var(axis=0).astype(np.float32)
    gamma = rng.uniform(10.0, 40.0, K).astype(np.float32) if dtype == "int8" else \
        rng.uniform(0.5, 2.0, K).astype(np.float32)
    beta = rng.normal(0, 2.0 if dtype == "int8" else 0.5, K).astype(np.float32)
    scale_k, bias_k = fc.fconv_fold_batchnorm(c.conv_scale, gamma, beta, mean, var, 1e-5,
                                              bias=c.bias)
    c.conv_scale, c.bias = scale_k, bias_k
    c.unit_variance = False   # gamma up to 2 widens the outputs
    got = c.run_gpu()
    c.check_output(got, c.oracle_out(acc_ref))
    if dtype == "int8":
        # the unfused block in double: normalise, add the scaled side, Relu, round
        g = gamma.astype(np.float64) / np.sqrt(var.astype(np.float64) + np.float32(1e-5))
        z = g * (y_conv - mean) + beta + c.side.astype(np.float64) * np.float32(c.side_scale)
        want = np.clip(np.rint(np.maximum(z, 0.0)), 0, 127)
        diff = np.abs(got.astype(np.int64) - want.astype(np.int64))
        assert diff.max() <= 1 and (diff == 0).mean() > 0.99


@pytest.mark.parametrize("dtype", ["int8", "bf16"])
def test_equal_channel_scales_equal_the_scalar_run(dtype):
    c = sweep_case(320, (2, 10, 10, 64, 96, 3, 3, 1, "SAME", True, True), dtype)
    scalar = c.run_gpu()
    c.conv_scale = np.full(c.K, c.conv_scale, np.float32)
    assert np.array_equal(c.run_gpu(), scalar)



@pytest.mark.parametrize("dtype", ["int8", "bf16"])
def test_back_to_back_runs_share_the_workspace(dtype):
    """Runs enqueued back to back on one stream reuse the plan's workspace:
    each convolution (launched as a dependent of its prep launch) must read
    its own prep's output, and finish before the next prep overwrites it.
    Two input sets alternate over 16 runs without a synchronisation."""
    params = (2, 10, 10, 64, 96, 3, 3, 1, "SAME", True, True)
    cases = [sweep_case(340, params, dtype), sweep_case(341, params, dtype)]
    p = cases[0].plan()
    ins = [(to_dev(c.x, dtype), to_dev(c.w, dtype), torch.from_numpy(c.bias).cuda(),
            to_dev(c.side, dtype)) for c in cases]
    ys = [p.new_output() for _ in range(16)]
    for i, y in enumerate(ys):
        x, w, bias, side = ins[i % 2]
        p.run(x, w, bias, side, cases[0].conv_scale, cases[0].side_scale, y=y)
    torch.cuda.synchronize()
    p.check()
    refs = [c.oracle_out(c.oracle_acc()) for c in cases]
    for i, y in enumerate(ys):
        cases[i % 2].check_output(to_host(y), refs[i % 2])
    p.close()


def test_run_replays_from_a_cuda_graph():
    """A captured fconv_run replays on new contents of the same buffers."""
    params = (2, 10, 10, 64, 96, 3, 3, 1, "SAME", True, True)
    first, second = sweep_case(330, params, "int8"), sweep_case(331, params, "int8")
    p = first.plan()
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


# ---------------------------------------------------------------- activations
ACT_CASES = [
    # (shape, dtype, act, alpha, beta)
    ((2, 9, 11, 64, 80, 3, 3, 1, "SAME", True, None), "int8", fc.FCONV_ACT_LEAKY_RELU, 0.1, 0.0),
    ((2, 9, 11, 48, 144, 3, 3, 2, "SAME", True, None), "int8", fc.FCONV_ACT_CLIPPED_RELU, 6.0, 0.0),
    ((2, 12, 12, 512, 272, 3, 3, 1, "SAME", True, None), "int8", fc.FCONV_ACT_CLAMP, -20.5, 33.25),
    ((2, 9, 11, 64, 80, 3, 3, 1, "SAME", True, None), "int8", fc.FCONV_ACT_CLIPPED_RELU, 2.5, 0.0),
    ((3, 8, 8, 64, 200, 3, 3, 1, "SAME", True, None), "bf16", fc.FCONV_ACT_LEAKY_RELU, 0.2, 0.0),
    ((3, 8, 8, 64, 200, 3, 3, 1, "SAME", True, None), "bf16", fc.FCONV_ACT_CLIPPED_RELU, 1.5, 0.0),
    ((2, 7, 9, 24, 40, 3, 3, 1, "VALID", False, None), "bf16", fc.FCONV_ACT_CLAMP, -1.25, 2.0),
]


@pytest.mark.parametrize("i,item", list(enumerate(ACT_CASES)))
def test_activation_variants(i, item):
    params, dtype, act, alpha, beta = item
    c = sweep_case(400 + i, params, dtype)
    c.relu, c.alpha, c.beta = act, alpha, beta
    if dtype == "int8":
        # sums of R*S*C products of uniform int8 values have a standard
        # deviation of about sqrt(R*S*C) * 5461: scale them to about +-40,
        # across the activation bounds and inside the int8 range
        c.conv_scale = 40.0 / (np.sqrt(c.R * c.S * c.C) * 5461.0)
        c.side_scale = 0.05
    ref = c.oracle_out()
    c.check_output(c.run_gpu(), ref)
    if params[3] % 64 == 0:
        c.check_output(c.run_gpu(debug=fc.FCONV_DEBUG_GATHER_CPASYNC), ref)


# ---------------------------------------------------------------- maximum sizes
# Tensors of just under 2^31 elements, the plan's limit: the largest input
# (16 x 255 x 255 x 2048 int8, an fp16 copy of 4.3 GB) and the largest output
# (2048 x 32 x 32 x 1008).  Checked on sampled pixels, the last one included.
@pytest.mark.parametrize("shape", [(16, 255, 255, 2048, 32), (2048, 32, 32, 16, 1008)])
def test_maximum_tensor_sizes(shape):
    N, H, W, C, K = shape
    assert max(N * H * W * C, N * H * W * K) < 2 ** 31
    x = FI.uniform_int8(600 + C, (N, H, W, C))
    w = FI.uniform_int8(601 + C, (1, 1, C, K))
    side = FI.uniform_int8(602 + C, (N, H, W, K))
    bias = np.linspace(-3.0, 3.0, K, dtype=np.float32)
    cs = 1.0 / (np.sqrt(C) * 5461.0) * 60.0
    plan = fc.Conv2dPlan(N, H, W, C, K, 1, 1, 1, "VALID", "int8", False)
    y = plan.run(to_dev(x, "int8"), to_dev(w, "int8"), torch.from_numpy(bias).cuda(),
                 to_dev(side, "int8"), cs, 0.125)
    plan.check()
    got = to_host(y).reshape(-1, K)
    del y
    plan.close()
    rng = np.random.default_rng(7)
    M = N * H * W
    pix = np.unique(np.concatenate([rng.choice(M, size=1500, replace=False), [0, M - 1]]))
    idx = (pix[:, None] * K + np.arange(K)[None, :]).ravel()
    acc = oracle.conv_acc_i8_points(x, w, idx, 1, oracle.VALID).reshape(-1, K)
    ref = oracle.epilogue_i8(acc, bias, side.reshape(-1, K)[pix], cs, 0.125, False)
    bad = np.argwhere(got[pix] != ref)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


# ---------------------------------------------------------------- 256-pixel tiles
# two 128-pixel halves sharing each filter tile (TMA gather, 64 or 128
# channels); ragged ends leave the second half partly or wholly past the
# last pixel
M256_CASES = [
    ((2, 9, 11, 64, 64, 3, 3, 1, "SAME", True, True), "int8", 64),       # M = 198
    ((1, 10, 13, 64, 128, 3, 3, 1, "SAME", True, False), "int8", 128),   # M = 130
    ((2, 12, 12, 512, 272, 3, 3, 1, "SAME", True, True), "int8", 128),   # chunked sums, K tail
    ((4, 14, 14, 128, 96, 3, 3, 2, "SAME", False, True), "int8", 64),    # stride 2, K tail
    ((3, 8, 8, 64, 200, 3, 3, 1, "SAME", True, False), "bf16", 128),
    ((2, 9, 11, 64, 64, 3, 3, 1, "SAME", True, True), "bf16", 64),
]


@pytest.mark.parametrize("i,item", list(enumerate(M256_CASES)))
def test_256_pixel_tiles(i, item):
    params, dtype, bn = item
    c = sweep_case(500 + i, params, dtype)
    acc_ref = c.oracle_acc()
    p = c.plan()
    fc.fconv_plan_set_tile_shape(p.handle, 256, bn)
    assert fc.fconv_plan_kernel(p.handle) == "tma-im2col-m256"
    x, w = to_dev(c.x, dtype), to_dev(c.w, dtype)
    bias = torch.from_numpy(c.bias).cuda()
    side = to_dev(c.side, dtype)
    acc = p.accumulators(x, w)
    y = p.run(x, w, bias, side, c.conv_scale, c.side_scale)
    p.check()
    c.check_acc(acc.cpu().numpy(), acc_ref)
    c.check_output(to_host(y), c.oracle_out(acc_ref))
    p.close()



# ---------------------------------------------------------------- batch shards
@pytest.mark.parametrize("dtype", ["int8", "bf16"])
@pytest.mark.parametrize("world", [2, 3])
def test_batch_shards_on_offset_pointers(dtype, world):
    """The batch split of a multi-GPU run, on one GPU: for each rank's images
    [lo, hi) (bench.shard_range) a plan of hi - lo images runs on pointers
    offset into the whole batch's x, side and y; the reassembled y must be the
    unsharded result (int8 bit for bit).  7 images over 2 or 3 ranks leave
    ragged shards whose tiles cross image boundaries."""
    import bench
    c = sweep_case(950, (7, 10, 9, 64, 80, 3, 3, 1, "SAME", True, True), dtype)
    ref = c.oracle_out(c.oracle_acc())
    x, w = to_dev(c.x, dtype), to_dev(c.w, dtype)
    bias = torch.from_numpy(c.bias).cuda()
    side = to_dev(c.side, dtype)
    y = torch.full(ref.shape, 0x55 if dtype == "int8" else 0,
                   dtype=torch.int8 if dtype == "int8" else torch.bfloat16, device="cuda")
    for rank in range(world):
        lo, hi = bench.shard_range(c.N, world, rank)
        p = fc.Conv2dPlan(hi - lo, c.H, c.W, c.C, c.K, c.R, c.S, c.stride, c.padding, dtype,
                          c.relu)
        p.run(x[lo:hi], w, bias, side[lo:hi], c.conv_scale, c.side_scale, y=y[lo:hi])
        p.check()
        p.close()
    c.check_output(to_host(y), ref)


def test_cpasync_debug_hook_leaves_the_plan_tiling():
    """A run forced onto the cp.async gather drops split-K and 256-pixel tiles
    for that launch only: the plan keeps its splits, tile and workspace size."""
    c = sweep_case(960, (2, 9, 11, 64, 80, 3, 3, 1, "SAME", True, True), "int8")
    p = c.plan()
    fc.fconv_plan_set_tile_shape(p.handle, 128, 64)
    fc.fconv_plan_set_splits(p.handle, 3)
    ws = fc.fconv_workspace_size(p.handle)
    fc.fconv_plan_set_debug(p.handle, fc.FCONV_DEBUG_GATHER_CPASYNC)
    x, w = to_dev(c.x, "int8"), to_dev(c.w, "int8")
    bias, side = torch.from_numpy(c.bias).cuda(), to_dev(c.side, "int8")
    y = p.run(x, w, bias, side, c.conv_scale, c.side_scale)
    p.check()
    c.check_output(to_host(y), c.oracle_out())
    assert fc.fconv_plan_get_splits(p.handle) == 3
    assert fc.fconv_workspace_size(p.handle) == ws
    fc.fconv_plan_set_debug(p.handle, 0)
    y = p.run(x, w, bias, side, c.conv_scale, c.side_scale)
    p.check()
    c.check_output(to_host(y), c.oracle_out())
    p.close()


# ---------------------------------------------------------------- in-kernel widening
# int8 activations widened by the convolution kernel (staged int8 tiles,
# converter warps) against the same plans with an fp16 copy of the input:
# identical sums and outputs, both equal to the oracle
WIDEN_CASES = [
    ((2, 9, 11, 64, 80, 3, 3, 1, "SAME", True, True), None),          # K tail, side input
    ((2, 9, 11, 64, 64, 3, 3, 1, "SAME", True, True), (256, 64)),     # 256-pixel tiles
    ((3, 8, 8, 128, 64, 3, 3, 2, "SAME", False, True), None),         # stride 2, odd pads
    ((3, 11, 13, 64, 80, 1, 1, (2, 3), "SAME", True, True), None),    # 1x1 strided
    ((2, 12, 12, 512, 272, 3, 3, 1, "SAME", True, True), (128, 128)), # chunked sums
    ((1, 7, 7, 128, 32, 7, 7, 1, "VALID", True, True), None),         # full window
    ((5, 6, 6, 256, 256, 1, 1, 1, "SAME", False, False), (128, 128)), # 1x1 stride 1
]


@pytest.mark.parametrize("i,item", list(enumerate(WIDEN_CASES)))
def test_in_kernel_widening(i, item):
    params, shape = item
    c = sweep_case(980 + i, params, "int8")
    acc_ref = c.oracle_acc()
    ref = c.oracle_out(acc_ref)
    got = {}
    for mode in (fc.FCONV_WIDEN_IN_KERNEL, fc.FCONV_WIDEN_COPY):
        p = c.plan()
        fc.fconv_plan_set_gather(p.handle, fc.FCONV_GATHER_IM2COL)   # the im2col form widens
        if shape:
            fc.fconv_plan_set_tile_shape(p.handle, *shape)
        fc.fconv_plan_set_splits(p.handle, 1)   # widening runs unsplit
        fc.fconv_plan_set_input_widening(p.handle, mode)
        assert fc.fconv_plan_get_input_widening(p.handle) == (mode == fc.FCONV_WIDEN_IN_KERNEL)
        x, w = to_dev(c.x, "int8"), to_dev(c.w, "int8")
        bias, side = torch.from_numpy(c.bias).cuda(), to_dev(c.side, "int8")
        acc = p.accumulators(x, w)
        y = p.run(x, w, bias, side, c.conv_scale, c.side_scale)
        y2 = p.run(x, w, bias, side, c.conv_scale, c.side_scale)   # the staging ring reused
        p.check()
        c.check_acc(acc.cpu().numpy(), acc_ref)
        c.check_output(to_host(y), ref)
        assert torch.equal(y, y2)
        got[mode] = to_host(y)
        p.close()
    assert np.array_equal(got[fc.FCONV_WIDEN_IN_KERNEL], got[fc.FCONV_WIDEN_COPY])


# ---------------------------------------------------------------- halo gather
# stride-1 layers with 64 input channels: one window copy a tile, the filter
# tile resident, each tap a row shift of the window (virtual pixel rows of
# Q + S - 1 columns).  Against the oracle and against the im2col gather.
HALO_CASES = [
    # params, tile pixels (None: the plan's own height)
    ((2, 9, 11, 64, 80, 3, 3, 1, "SAME", True, True), None),      # K tail, two channel tiles
    ((3, 10, 10, 64, 64, 3, 3, 1, "SAME", True, True), 256),
    ((2, 13, 17, 64, 64, 3, 3, 1, "VALID", False, True), 128),    # no padding
    ((1, 5, 7, 64, 48, 3, 3, 1, "SAME", True, False), None),      # K below the tile
    ((2, 12, 10, 64, 32, 1, 3, 1, "SAME", False, True), None),    # R != S
    ((2, 7, 9, 64, 64, 2, 2, 1, "SAME", True, True), 256),        # even filter: pads 0 / 1
    ((64, 24, 24, 64, 64, 3, 3, 1, "SAME", True, True), None),    # several tiles a CTA
    ((2, 6, 90, 64, 64, 3, 3, 1, "SAME", False, True), 128),      # a 92-pixel-wide window
    ((3, 1, 1, 64, 64, 1, 1, 1, "SAME", True, True), None),       # 1x1 images
    ((2, 4, 40, 64, 128, 3, 3, 1, "SAME", True, True), 256),      # window rows past the image
    ((2, 16, 16, 32, 32, 3, 3, 1, "SAME", True, True), None),     # C = 32 (int8): zero-filled half
    ((3, 9, 11, 32, 80, 3, 3, 1, "VALID", False, True), 256),     # C = 32, two channel tiles
    ((256, 16, 16, 64, 64, 3, 3, 1, "SAME", True, True), 256),    # 512 tiles: 3-4 a CTA
    ((400, 12, 12, 32, 64, 3, 3, 1, "SAME", True, True), 128),    # C = 32, ~5 tiles a CTA
]


@pytest.mark.parametrize("dtype", ["int8", "bf16"])
@pytest.mark.parametrize("i,item", list(enumerate(HALO_CASES)))
def test_halo_gather(i, item, dtype):
    params, pixels = item
    if dtype == "bf16" and params[3] != 64:
        pytest.skip("the halo gather takes 32 input channels for int8 only")
    c = sweep_case(1200 + i, params, dtype)
    acc_ref = c.oracle_acc()
    ref = c.oracle_out(acc_ref)
    p = c.plan()
    fc.fconv_plan_set_gather(p.handle, fc.FCONV_GATHER_HALO)
    if pixels:
        fc.fconv_plan_set_tile_shape(p.handle, pixels, 64)
    kern = fc.fconv_plan_kernel(p.handle)
    assert kern.startswith("tma-halo") and (pixels is None or kern.endswith("m256") == (pixels == 256))
    # one launch, no workspace: an int8 filter is widened inside the kernel too
    assert fc.fconv_plan_launch_count(p.handle) == 1
    assert fc.fconv_workspace_size(p.handle) == 0
    assert fc.fconv_plan_get_input_widening(p.handle) == (dtype == "int8")
    x, w = to_dev(c.x, dtype), to_dev(c.w, dtype)
    bias, side = torch.from_numpy(c.bias).cuda(), to_dev(c.side, dtype)
    acc = p.accumulators(x, w)
    y = p.run(x, w, bias, side, c.conv_scale, c.side_scale)
    y2 = p.run(x, w, bias, side, c.conv_scale, c.side_scale)   # both window buffers reused
    p.check()
    c.check_acc(acc.cpu().numpy(), acc_ref)
    c.check_output(to_host(y), ref)
    assert torch.equal(y, y2)
    halo = to_host(y)
    p.close()
    # the same plan on the im2col gather
    q = c.plan()
    fc.fconv_plan_set_gather(q.handle, fc.FCONV_GATHER_IM2COL)
    assert not fc.fconv_plan_kernel(q.handle).startswith("tma-halo")
    y3 = q.run(x, w, bias, side, c.conv_scale, c.side_scale)
    q.check()
    q.close()
    if dtype == "int8":
        assert np.array_equal(halo, to_host(y3))
    else:
        c.check_output(to_host(y3), ref)
