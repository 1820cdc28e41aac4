"""Host-side checks of the C ABI: the library loads, exports every function
the public header declares, validates arguments and computes the output
geometry -- all without a GPU (no call here reaches a kernel)."""
import ctypes
import os
import re

import pytest

import oracle
import quantized_conv2d_gb300 as fc
from quantized_conv2d_gb300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fconv.h")


@pytest.fixture(scope="module", autouse=True)
def built_library():
    fbuild.build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fconv_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fconv_plan_create", "fconv_run", "fconv_plan_destroy",
                     "fconv_workspace_size", "fconv_plan_output_shape", "fconv_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(fc.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings():
    for code in range(8):
        assert fc.fconv_status_string(code).startswith("FCONV_")


def _err(fn, *args):
    with pytest.raises(fc.FconvError) as ei:
        fn(*args)
    return ei.value.status


@pytest.mark.parametrize("args,status", [
    ((0, 8, 8, 16, 16, 3, 3, 1, 1, 0, 0, 1), fc.FCONV_ERR_INVALID_VALUE),
    ((1, 8, 8, 16, 16, 3, 3, 0, 1, 0, 0, 1), fc.FCONV_ERR_INVALID_VALUE),
    ((1, 8, 8, 16, 16, 3, 3, 1, 1, 7, 0, 1), fc.FCONV_ERR_INVALID_VALUE),
    ((1, 8, 8, 16, 16, 3, 3, 1, 1, 0, 5, 1), fc.FCONV_ERR_INVALID_VALUE),
    ((1, 8, 8, 16, 16, 3, 3, 1, 1, 0, 0, 5), fc.FCONV_ERR_INVALID_VALUE),   # unknown activation
    ((1, 2, 8, 16, 16, 3, 3, 1, 1, 1, 0, 1), fc.FCONV_ERR_INVALID_VALUE),   # VALID, R > H
    ((1, 8, 8, 24, 16, 3, 3, 1, 1, 0, 0, 1), fc.FCONV_ERR_NOT_SUPPORTED),   # int8 C % 16
    ((1, 8, 8, 16, 40, 3, 3, 1, 1, 0, 0, 1), fc.FCONV_ERR_NOT_SUPPORTED),   # int8 K % 16
    ((1, 8, 8, 12, 16, 3, 3, 1, 1, 0, 1, 1), fc.FCONV_ERR_NOT_SUPPORTED),   # bf16 C % 8
    ((4096, 1024, 1024, 64, 16, 1, 1, 1, 1, 0, 0, 1), fc.FCONV_ERR_NOT_SUPPORTED),  # 2^31 elems
])
def test_plan_create_rejects(args, status):
    assert _err(fc.fconv_plan_create, *args) == status
    assert fc.fconv_last_error() != ""


def test_plan_create_accepts_bf16_multiples_of_8():
    h = fc.fconv_plan_create(1, 8, 8, 24, 40, 3, 3, 1, 1, 0, 1, 1)
    assert fc.fconv_plan_output_shape(h) == (1, 8, 8, 40)
    fc.fconv_plan_destroy(h)


def _geometry_rows():
    rows = []
    for line in open(os.path.join(ROOT, "tests", "golden", "geometry_cases.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            a = line.split()
            rows.append((int(a[0]), int(a[1]), int(a[2]), a[3], int(a[4])))
    return rows


@pytest.mark.parametrize("row", _geometry_rows())
def test_plan_geometry_matches_oracle(row):
    size, filt, stride, pad, out = row
    pad_code = 0 if pad == "SAME" else 1
    args = (1, size, 3, 16, 16, filt, 1, stride, 1, pad_code, 0, 1)
    if out < 0:
        assert _err(fc.fconv_plan_create, *args) == fc.FCONV_ERR_INVALID_VALUE
        return
    h = fc.fconv_plan_create(*args)
    try:
        _, P, _, _ = fc.fconv_plan_output_shape(h)
        top, bottom, _, _ = fc.fconv_plan_padding(h)
        assert (P, top, bottom) == oracle.out_geometry(size, filt, stride, pad_code)
    finally:
        fc.fconv_plan_destroy(h)


def test_tile_override_rules():
    # 3x3x512 int8: 72 k-blocks, so the sums are chunked.  C % 64 == 0 lets
    # the kernel gather by TMA, whose epilogue folds the chunks in registers:
    # every tile from 64 to 256 is allowed.
    h = fc.fconv_plan_create(2, 8, 8, 512, 512, 3, 3, 1, 1, 0, 0, 1)
    try:
        bn, chunk, _ = fc.fconv_plan_get_config(h)
        assert chunk == 15
        for t in (64, 128, 256):
            fc.fconv_plan_set_tile(h, t)
            assert fc.fconv_plan_get_config(h)[0] == t
        assert _err(fc.fconv_plan_set_tile, h, 48) == fc.FCONV_ERR_NOT_SUPPORTED
        fc.fconv_plan_set_tile(h, 0)
        assert fc.fconv_plan_get_config(h)[0] == bn
    finally:
        fc.fconv_plan_destroy(h)
    # C = 176: the cp.async gather folds chunks in TMEM, which caps the tile at 128
    h = fc.fconv_plan_create(2, 8, 8, 176, 256, 3, 3, 1, 1, 0, 0, 1)
    try:
        bn, chunk, _ = fc.fconv_plan_get_config(h)
        assert chunk < 25 and bn <= 128
        assert _err(fc.fconv_plan_set_tile, h, 256) == fc.FCONV_ERR_NOT_SUPPORTED
        fc.fconv_plan_set_tile(h, 64)
        # tiles are whole 64-channel filter boxes: no 32-channel tile
        assert _err(fc.fconv_plan_set_tile, h, 32) == fc.FCONV_ERR_NOT_SUPPORTED
    finally:
        fc.fconv_plan_destroy(h)
    # bf16 sums are never chunked: 256 is allowed
    h = fc.fconv_plan_create(2, 8, 8, 512, 512, 3, 3, 1, 1, 0, 1, 1)
    try:
        assert fc.fconv_plan_get_config(h)[1] == 72
        fc.fconv_plan_set_tile(h, 256)
    finally:
        fc.fconv_plan_destroy(h)


def test_exact_chunk_bound():
    # every chunk holds at most 960 k-values: 960 * 128 * 128 < 2^24
    for C, R in [(16, 1), (64, 3), (256, 3), (512, 3), (512, 5), (1024, 3)]:
        h = fc.fconv_plan_create(1, 8, 8, C, 16, R, R, 1, 1, 0, 0, 1)
        try:
            chunk = fc.fconv_plan_get_config(h)[1]
            assert chunk * 64 * 128 * 128 < 2 ** 24
        finally:
            fc.fconv_plan_destroy(h)


def test_run_argument_errors_before_any_launch():
    h = fc.fconv_plan_create(1, 8, 8, 16, 16, 3, 3, 1, 1, 0, 0, 1)
    ws = fc.fconv_workspace_size(h)
    try:
        A = 1 << 20  # an aligned fake address: never dereferenced, every call fails first
        assert _err(fc.fconv_run, None, A, A, A, None, 1.0, 0.0, A, A, ws, None) == fc.FCONV_ERR_INVALID_VALUE
        assert _err(fc.fconv_run, h, None, A, A, None, 1.0, 0.0, A, A, ws, None) == fc.FCONV_ERR_INVALID_VALUE
        assert _err(fc.fconv_run, h, A, A, None, None, 1.0, 0.0, A, A, ws, None) == fc.FCONV_ERR_INVALID_VALUE
        assert _err(fc.fconv_run, h, A + 8, A, A, None, 1.0, 0.0, A, A, ws, None) == fc.FCONV_ERR_MISALIGNED
        assert _err(fc.fconv_run, h, A, A, A, A + 4, 1.0, 0.5, A, A, ws, None) == fc.FCONV_ERR_MISALIGNED
        assert _err(fc.fconv_run, h, A, A, A, None, 1.0, 0.0, A, A, ws - 1, None) == fc.FCONV_ERR_WORKSPACE
        assert _err(fc.fconv_run, h, A, A, A, None, 1.0, 0.0, A, None, ws, None) == fc.FCONV_ERR_WORKSPACE
        assert _err(fc.fconv_run, h, A, A, A, None, 1.0, 0.0, A, A + 16, ws, None) == fc.FCONV_ERR_MISALIGNED
        # per-channel scale: NULL vector, misaligned vector
        assert _err(fc.fconv_run_channel_scale, h, A, A, A, None, None, 0.0, A, A, ws,
                    None) == fc.FCONV_ERR_INVALID_VALUE
        assert _err(fc.fconv_run_channel_scale, h, A, A, A, None, A + 4, 0.0, A, A, ws,
                    None) == fc.FCONV_ERR_MISALIGNED
        assert _err(fc.fconv_plan_set_timeout_ms, h, 0) == fc.FCONV_ERR_INVALID_VALUE
        assert _err(fc.fconv_plan_set_debug, h, 16) == fc.FCONV_ERR_INVALID_VALUE
    finally:
        fc.fconv_plan_destroy(h)


def test_workspace_sizes():
    h = fc.fconv_plan_create(256, 28, 28, 512, 512, 3, 3, 1, 1, 0, 0, 1)
    try:
        # fp16 filter [512][4608] + fp16 copy of the input
        ws = fc.fconv_workspace_size(h)
        assert ws == 512 * 4608 * 2 + 256 * 28 * 28 * 512 * 2
        hw = fc.fconv_host_workspace_size(h, True)
        assert hw >= ws + 3 * 256 * 28 * 28 * 512 + 4608 * 512 + 512 * 4
    finally:
        fc.fconv_plan_destroy(h)
    h = fc.fconv_plan_create(8, 14, 14, 48, 64, 3, 3, 1, 1, 0, 0, 1)
    try:
        # the fp16 filter [3*3*48][64] (no padding of the 432 rows)
        assert fc.fconv_workspace_size(h) == 432 * 64 * 2 + 8 * 14 * 14 * 48 * 2
    finally:
        fc.fconv_plan_destroy(h)
    h = fc.fconv_plan_create(64, 28, 28, 256, 512, 1, 1, 2, 2, 1, 0, 1)
    try:
        # 1x1 stride 2, int8: only the strided pixels are widened ([64][14][14][256])
        assert fc.fconv_plan_get_input_widening(h) == 0
        assert fc.fconv_workspace_size(h) == 512 * 256 * 2 + 64 * 14 * 14 * 256 * 2
        # widened inside the kernel instead: the fp16 filter alone
        fc.fconv_plan_set_input_widening(h, fc.FCONV_WIDEN_IN_KERNEL)
        assert fc.fconv_plan_get_input_widening(h) == 1
        assert fc.fconv_workspace_size(h) == 512 * 256 * 2
        fc.fconv_plan_set_input_widening(h, fc.FCONV_WIDEN_AUTO)
        assert fc.fconv_plan_get_input_widening(h) == 0
    finally:
        fc.fconv_plan_destroy(h)
    h = fc.fconv_plan_create(32, 14, 14, 256, 256, 3, 3, 1, 1, 0, 1, 1)
    try:
        # bf16 forward plans read the input and the filter as they are
        assert fc.fconv_workspace_size(h) == 0
    finally:
        fc.fconv_plan_destroy(h)


def test_binding_and_oracle_are_separate():
    pkg = os.path.join(ROOT, "quantized_conv2d_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in re.sub(r"#.*|//.*", "", text).lower().replace("oracle-free", ""), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            assert "quantized_conv2d_gb300" not in open(os.path.join(ROOT, "oracle", f)).read()


def test_activation_params_validation():
    for act in (fc.FCONV_ACT_LEAKY_RELU, fc.FCONV_ACT_CLIPPED_RELU, fc.FCONV_ACT_CLAMP):
        h = fc.fconv_plan_create(1, 8, 8, 16, 16, 3, 3, 1, 1, 0, 0, act)
        try:
            fc.fconv_plan_set_activation_params(h, 0.5, 2.0)
            assert _err(fc.fconv_plan_set_activation_params, h, float("nan"), 1.0) == \
                fc.FCONV_ERR_INVALID_VALUE
            assert _err(fc.fconv_plan_set_activation_params, h, 1.0, float("inf")) == \
                fc.FCONV_ERR_INVALID_VALUE
            if act == fc.FCONV_ACT_CLIPPED_RELU:
                assert _err(fc.fconv_plan_set_activation_params, h, -1.0, 0.0) == \
                    fc.FCONV_ERR_INVALID_VALUE
            if act == fc.FCONV_ACT_CLAMP:
                assert _err(fc.fconv_plan_set_activation_params, h, 3.0, 2.0) == \
                    fc.FCONV_ERR_INVALID_VALUE
        finally:
            fc.fconv_plan_destroy(h)
    assert _err(fc.fconv_plan_set_activation_params, None, 0.0, 0.0) == fc.FCONV_ERR_INVALID_VALUE


def test_transposed_plan_geometry_and_limits():
    # Ho = (H-1)*s + R - pt - pb
    h = fc.fconv_plan_create_transposed(2, 7, 9, 16, 32, 3, 5, 1, 1, 1, 0, 2, 1, 0, 1)
    try:
        assert fc.fconv_plan_output_shape(h) == (2, 7 - 1 + 3 - 1 - 0, 9 - 1 + 5 - 2 - 1, 32)
        assert fc.fconv_plan_output_shape(h)[1:3] == (
            oracle.convT_out_size(7, 3, 1, 1, 0), oracle.convT_out_size(9, 5, 1, 2, 1))
    finally:
        fc.fconv_plan_destroy(h)
    bad = [
        ((2, 7, 9, 16, 32, 3, 3, 2, 2, 1, 1, 1, 1, 0, 1), None),                        # stride 2
        ((2, 7, 9, 16, 32, 3, 3, 2, 2, 1, 0, 1, 0, 0, 1), None),        # output adjustment 1
        ((2, 7, 9, 16, 32, 3, 3, 2, 2, 1, -1, 1, 0, 0, 1), None),       # pad_bottom 1 - stride
        ((2, 7, 9, 16, 32, 3, 3, 2, 2, 1, -2, 1, 0, 0, 1), fc.FCONV_ERR_NOT_SUPPORTED),
        ((2, 7, 9, 16, 32, 3, 3, 9, 1, 1, 1, 1, 1, 0, 1), fc.FCONV_ERR_NOT_SUPPORTED),  # stride 9
        ((2, 7, 9, 16, 32, 3, 3, 1, 1, 3, 0, 0, 0, 0, 1), fc.FCONV_ERR_NOT_SUPPORTED),  # pad > R-1
        ((2, 7, 9, 16, 32, 3, 3, 1, 1, -1, 0, 0, 0, 0, 1), fc.FCONV_ERR_NOT_SUPPORTED),
        ((2, 1, 1, 16, 32, 1, 1, 1, 1, 0, 0, 0, 0, 0, 1), None),                        # 1x1 output
        ((2, 7, 9, 24, 32, 3, 3, 1, 1, 1, 1, 1, 1, 0, 1), fc.FCONV_ERR_NOT_SUPPORTED),  # int8 C % 16
        ((0, 7, 9, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1, 0, 1), fc.FCONV_ERR_INVALID_VALUE),
    ]
    for args, status in bad:
        if status is None:
            fc.fconv_plan_destroy(fc.fconv_plan_create_transposed(*args))
        else:
            assert _err(fc.fconv_plan_create_transposed, *args) == status


def test_transposed_workspace_layouts():
    # stride 2, 3x3, bf16: four phases (taps 2x2, 2x1, 1x2, 1x1 of 16 channels,
    # each copied as [taps * 16][32]); bf16 reads x as it is
    h = fc.fconv_plan_create_transposed(2, 7, 9, 16, 32, 3, 3, 2, 2, 1, 1, 1, 1, 1, 1)
    try:
        assert fc.fconv_plan_output_shape(h) == (2, 13, 17, 32)
        assert fc.fconv_plan_padding(h) == (1, 1, 1, 1)
        assert fc.fconv_workspace_size(h) == (64 + 32 + 32 + 16) * 32 * 2
    finally:
        fc.fconv_plan_destroy(h)
    # 1x1 filter, stride 2: no phase has more than one tap and some outputs
    # none, so x is copied with zero rows/columns inserted (13 x 17)
    h = fc.fconv_plan_create_transposed(2, 7, 9, 16, 32, 1, 1, 2, 2, 0, 0, 0, 0, 1, 1)
    try:
        assert fc.fconv_plan_output_shape(h) == (2, 13, 17, 32)
        xh = 2 * 13 * 17 * 16 * 2
        assert fc.fconv_workspace_size(h) == 16 * 32 * 2 + (xh + 255) // 256 * 256
    finally:
        fc.fconv_plan_destroy(h)
    # int8, stride 2, 4x4: four phases of 2x2 taps, then one fp16 copy of x
    h = fc.fconv_plan_create_transposed(2, 7, 9, 64, 32, 4, 4, 2, 2, 1, 1, 1, 1, 0, 1)
    try:
        xh = 2 * 7 * 9 * 64 * 2
        assert fc.fconv_workspace_size(h) == 4 * 32 * 256 * 2 + (xh + 255) // 256 * 256
    finally:
        fc.fconv_plan_destroy(h)


def test_launch_counts():
    cases = [
        ((256, 28, 28, 512, 512, 3, 3, 1, 1, 0, 0, 1), 2),     # prep + conv
        ((1, 3, 3, 16, 16, 3, 3, 1, 1, 0, 0, 1), 3),           # 144 int8 inputs: a tail launch
        ((1, 3, 3, 16, 16, 3, 3, 1, 1, 0, 1, 1), 1),           # bf16 reads x and w as they are
    ]
    for args, n in cases:
        h = fc.fconv_plan_create(*args)
        try:
            assert fc.fconv_plan_launch_count(h) == n
        finally:
            fc.fconv_plan_destroy(h)
    # stride 2, 4x4 transposed: four phases, each prep + conv
    h = fc.fconv_plan_create_transposed(2, 8, 8, 64, 32, 4, 4, 2, 2, 1, 1, 1, 1, 0, 1)
    try:
        assert fc.fconv_plan_launch_count(h) == 8
    finally:
        fc.fconv_plan_destroy(h)


def test_256_pixel_tile_rules():
    h = fc.fconv_plan_create(2, 9, 11, 64, 64, 3, 3, 1, 1, 0, 0, 1)
    try:
        fc.fconv_plan_set_tile_shape(h, 256, 64)
        assert fc.fconv_plan_kernel(h) == "tma-im2col-m256"
        assert fc.fconv_plan_get_config(h)[2] == 1          # 198 pixels: one tile
        fc.fconv_plan_set_tile_shape(h, 128, 64)
        assert fc.fconv_plan_get_config(h)[2] == 2
        assert _err(fc.fconv_plan_set_tile_shape, h, 512, 64) == fc.FCONV_ERR_NOT_SUPPORTED
    finally:
        fc.fconv_plan_destroy(h)
    h = fc.fconv_plan_create(1, 8, 8, 64, 256, 3, 3, 1, 1, 0, 0, 1)
    try:   # 2 x 256 columns of accumulators would not fit in tensor memory twice
        assert _err(fc.fconv_plan_set_tile_shape, h, 256, 256) == fc.FCONV_ERR_NOT_SUPPORTED
    finally:
        fc.fconv_plan_destroy(h)
    h = fc.fconv_plan_create(1, 8, 8, 48, 64, 3, 3, 1, 1, 0, 0, 1)
    try:   # C % 64 != 0: the cp.async gather, which has no 256-pixel tiles
        assert _err(fc.fconv_plan_set_tile_shape, h, 256, 64) == fc.FCONV_ERR_NOT_SUPPORTED
    finally:
        fc.fconv_plan_destroy(h)


def test_split_k_rules():
    """Split-K: forward plans on the TMA gather, no empty unit, workspace
    grown by the partial sums and counters, reset by an explicit tile."""
    h = fc.fconv_plan_create(2, 9, 11, 64, 80, 3, 3, 1, 1, 0, 0, 1)   # 9 k-blocks
    try:
        auto = fc.fconv_workspace_size(h)       # the plan's own tile and split
        fc.fconv_plan_set_tile_shape(h, 128, 64)
        base = fc.fconv_workspace_size(h)       # unsplit
        tiles = fc.fconv_plan_get_config(h)[2]
        assert fc.fconv_plan_get_splits(h) == 1
        fc.fconv_plan_set_splits(h, 3)
        assert fc.fconv_plan_get_splits(h) == 3
        part = tiles * 3 * 128 * 64 * 4
        assert fc.fconv_workspace_size(h) >= base + part + tiles * 8 * 4
        for asked, runs in [(4, 3), (5, 5), (8, 5), (9, 5), (2, 2)]:   # 9 k-blocks
            if asked <= 8:
                fc.fconv_plan_set_splits(h, asked)
                assert fc.fconv_plan_get_splits(h) == runs, asked
        assert _err(fc.fconv_plan_set_splits, h, 9) == fc.FCONV_ERR_INVALID_VALUE
        assert _err(fc.fconv_plan_set_splits, h, -1) == fc.FCONV_ERR_INVALID_VALUE
        fc.fconv_plan_set_tile(h, 128)
        assert fc.fconv_plan_get_splits(h) == 1
        fc.fconv_plan_set_splits(h, 0)   # the automatic choice again
        assert fc.fconv_workspace_size(h) == auto
    finally:
        fc.fconv_plan_destroy(h)
    h = fc.fconv_plan_create(2, 9, 11, 64, 64, 3, 3, 1, 1, 0, 0, 1)
    try:   # 256-pixel tiles have no split-K
        fc.fconv_plan_set_tile_shape(h, 256, 64)
        assert _err(fc.fconv_plan_set_splits, h, 2) == fc.FCONV_ERR_NOT_SUPPORTED
    finally:
        fc.fconv_plan_destroy(h)
    h = fc.fconv_plan_create(1, 8, 8, 48, 64, 3, 3, 1, 1, 0, 0, 1)
    try:   # C % 64 != 0: the cp.async gather, which has no split-K
        assert _err(fc.fconv_plan_set_splits, h, 2) == fc.FCONV_ERR_NOT_SUPPORTED
        fc.fconv_plan_set_splits(h, 1)
    finally:
        fc.fconv_plan_destroy(h)
    h = fc.fconv_plan_create_transposed(2, 8, 8, 64, 32, 4, 4, 2, 2, 1, 1, 1, 1, 0, 1)
    try:
        assert _err(fc.fconv_plan_set_splits, h, 2) == fc.FCONV_ERR_NOT_SUPPORTED
    finally:
        fc.fconv_plan_destroy(h)
    # a batch-one deep layer: few tiles, long K, split on its own
    h = fc.fconv_plan_create(1, 7, 7, 512, 512, 3, 3, 1, 1, 0, 0, 1)
    try:
        assert fc.fconv_plan_get_splits(h) > 1
    finally:
        fc.fconv_plan_destroy(h)


@pytest.mark.parametrize("shape,splits", [
    ((1, 16, 16, 32, 32, 3, 3, 1, 0, 0), 1),        # the five benchmark workloads
    ((32, 56, 56, 64, 64, 3, 3, 1, 0, 0), 1),
    ((64, 28, 28, 256, 512, 1, 1, 2, 1, 0), 1),
    ((32, 14, 14, 256, 256, 3, 3, 1, 0, 1), 1),
    ((256, 28, 28, 512, 512, 3, 3, 1, 0, 0), 1),
    ((1, 7, 7, 512, 512, 3, 3, 1, 0, 0), None),      # batch-one deep layers split
    ((1, 14, 14, 256, 256, 3, 3, 1, 0, 0), None),
    ((8, 7, 7, 2048, 512, 1, 1, 1, 0, 0), None),
])
def test_automatic_split_choice(shape, splits):
    N, H, W, C, K, R, S, st, pad, dt = shape
    h = fc.fconv_plan_create(N, H, W, C, K, R, S, st, st, pad, dt, 1)
    try:
        got = fc.fconv_plan_get_splits(h)
        assert got == splits if splits is not None else got > 1
    finally:
        fc.fconv_plan_destroy(h)


@pytest.mark.parametrize("name,block_n,form,splits", [
    ("small_i8_16x16x32", 64, "tma-halo", 1),
    ("resnet_i8_56x56x64", 64, "tma-halo-m256", 1),
    ("proj1x1s2_i8_28x28x256", 128, "tma-im2col", 1),
    ("bf16_14x14x256", 128, "tma-im2col-kb2-dual", 1),
    ("large_i8_28x28x512", 256, "tma-im2col", 1),
    ("proj1x1s1_i8_28x28x256", 128, "tma-im2col", 1),
    ("fullwin_i8_7x7x512", 64, "tma-im2col", 8),
    ("deep_b1_i8_7x7x512", 64, "tma-im2col", 8),
    ("deep_b1_i8_14x14x256", 64, "tma-im2col", 6),
    ("proj_b8_i8_7x7x2048", 64, "tma-im2col", 4),
    ("deconv_bf16_16x16x256_s2", 128, "tma-im2col-m256", 1),
    ("deconv_i8_14x14x512_s1", 256, "tma-im2col", 1),
])
def test_benchmark_workload_plans(name, block_n, form, splits):
    # The automatic tile choice for each benchmark workload: tile width,
    # kernel form (256-pixel tiles, two k-blocks a stage) and split count.
    # A change to the tile cost model shows here before it shows on a GPU.
    import fconv_inputs as FI
    wl = FI.workload(name)
    dt = fc.FCONV_INT8 if wl.dtype == "int8" else fc.FCONV_BF16
    st = wl.stride if isinstance(wl.stride, int) else wl.stride[0]
    if wl.transposed_pads:
        pt, pb, pl, pr = wl.transposed_pads
        h = fc.fconv_plan_create_transposed(wl.N, wl.H, wl.W, wl.C, wl.K, wl.R, wl.S,
                                            st, st, pt, pb, pl, pr, dt, 1)
    else:
        pad = fc.FCONV_SAME if wl.padding == "SAME" else fc.FCONV_VALID
        h = fc.fconv_plan_create(wl.N, wl.H, wl.W, wl.C, wl.K, wl.R, wl.S,
                                 st, st, pad, dt, 1 if wl.relu else 0)
    try:
        assert fc.fconv_plan_get_config(h)[0] == block_n
        assert fc.fconv_plan_kernel(h) == form
        assert fc.fconv_plan_get_splits(h) == splits
    finally:
        fc.fconv_plan_destroy(h)


@pytest.mark.parametrize("shape,sms", [
    ((256, 28, 28, 512, 512, 3, 3, 1), 152), ((128, 28, 28, 512, 512, 3, 3, 1), 152),
    ((124, 28, 28, 512, 512, 3, 3, 1), 152), ((1024, 28, 28, 512, 512, 3, 3, 1), 152),
    ((32, 56, 56, 64, 64, 3, 3, 1), 152), ((7, 12, 10, 64, 48, 3, 3, 1), 152),
    ((256, 28, 28, 512, 512, 3, 3, 1), 8), ((2048, 7, 7, 64, 64, 3, 3, 1), 8),
    ((5000, 4, 4, 16, 16, 1, 1, 1), 8), ((1, 16, 16, 32, 32, 3, 3, 1), 152),
])
def test_host_chunk_sizes_cover_the_batch(shape, sms):
    N, H, W, C, K, R, S, st = shape
    h = fc.fconv_plan_create(N, H, W, C, K, R, S, st, st, fc.FCONV_SAME, fc.FCONV_INT8, 1)
    try:
        sizes = fc.fconv_plan_host_chunk_sizes(h, sms)
        assert sum(sizes) == N and 1 <= len(sizes) <= 16 and min(sizes) >= 1, sizes
    finally:
        fc.fconv_plan_destroy(h)


def _tiles(n, P, Q, K, block_n):
    # 128-pixel output tiles times channel tiles of an n-image slice
    return -(-n * P * Q // 128) * (K // block_n)


def test_host_chunk_ramp_fills_whole_waves():
    """The automatic host chunks of the N=256 28x28x512 int8 layer on 152 SMs:
    a ramp whose W(2)- and W(1)-sized chunks are the most images that fill
    two waves and one wave of 128 x 256 tiles."""
    h = fc.fconv_plan_create(256, 28, 28, 512, 512, 3, 3, 1, 1, fc.FCONV_SAME, fc.FCONV_INT8, 1)
    try:
        assert fc.fconv_plan_get_config(h)[0] == 256
        sizes = fc.fconv_plan_host_chunk_sizes(h, 152)
    finally:
        fc.fconv_plan_destroy(h)
    w = {k: max(n for n in range(1, 257) if _tiles(n, 28, 28, 512, 256) <= k * 152)
         for k in (1, 2, 3)}
    assert (w[1], w[2], w[3]) == (12, 24, 37)
    assert sizes[:3] == [w[1] // 6, w[1] // 2, w[2]]
    assert sizes[-3:] == [w[2], w[1], 2 * w[1] // 3]
    mids = sizes[3:-3]
    assert max(mids) <= w[3] and max(mids) - min(mids) <= 1 and sum(sizes) == 256
    assert sizes == [2, 6, 24, 36, 36, 36, 36, 36, 24, 12, 8]


def test_host_chunk_sizes_fixed_count_and_errors():
    h = fc.fconv_plan_create(7, 12, 10, 64, 48, 3, 3, 1, 1, fc.FCONV_SAME, fc.FCONV_INT8, 1)
    try:
        fc.fconv_plan_set_host_chunks(h, 3)
        assert fc.fconv_plan_host_chunk_sizes(h, 152) == [3, 3, 1]
        fc.fconv_plan_set_host_chunks(h, 0)
        assert fc.fconv_plan_host_chunk_sizes(h, 152) == [7]   # less than a wave: one chunk
        n = ctypes.c_int(0)
        buf = (ctypes.c_int * 1)()
        lib = fc._load()
        assert lib.fconv_plan_host_chunk_sizes(h, 0, buf, 1, ctypes.byref(n)) == \
            fc.FCONV_ERR_INVALID_VALUE
        fc.fconv_plan_set_host_chunks(h, 3)
        assert lib.fconv_plan_host_chunk_sizes(h, 152, buf, 1, ctypes.byref(n)) == \
            fc.FCONV_ERR_INVALID_VALUE
        assert n.value == 3
    finally:
        fc.fconv_plan_destroy(h)


def _plan(shape, dtype=None, stride=1, pad=None):
    N, H, W, C, K, R, S = shape
    return fc.fconv_plan_create(N, H, W, C, K, R, S, stride, stride,
                                fc.FCONV_SAME if pad is None else pad,
                                fc.FCONV_INT8 if dtype is None else dtype, 1)


@pytest.mark.parametrize("shape,dtype,stride,ok", [
    ((2, 20, 20, 64, 64, 3, 3), fc.FCONV_INT8, 1, True),
    ((2, 20, 20, 64, 64, 3, 3), fc.FCONV_BF16, 1, True),
    ((2, 20, 20, 32, 64, 3, 3), fc.FCONV_INT8, 1, True),     # C = 32: int8 only
    ((2, 20, 20, 32, 64, 3, 3), fc.FCONV_BF16, 1, False),
    ((2, 20, 20, 128, 64, 3, 3), fc.FCONV_INT8, 1, False),   # one k-block a tap: C <= 64
    ((2, 20, 20, 64, 64, 3, 3), fc.FCONV_INT8, 2, False),    # stride 1 only
    ((2, 20, 20, 64, 64, 5, 5), fc.FCONV_INT8, 1, False),    # 25 taps: the filter tile is too big
    ((1, 8, 300, 64, 64, 3, 3), fc.FCONV_INT8, 1, False),    # a window wider than the buffers
    ((1, 8, 115, 64, 64, 3, 3), fc.FCONV_INT8, 1, True),     # the widest int8 3x3 window
])
def test_halo_gather_rules(shape, dtype, stride, ok):
    """Which plans the halo gather takes (forward, stride 1, C == 64 or int8
    C == 32, at most 9 taps, windows that fit shared memory), and what it
    changes: one launch, and no workspace for int8 plans."""
    h = _plan(shape, dtype, stride)
    try:
        if not ok:
            assert _err(fc.fconv_plan_set_gather, h, fc.FCONV_GATHER_HALO) == \
                fc.FCONV_ERR_NOT_SUPPORTED
            assert not fc.fconv_plan_kernel(h).startswith("tma-halo")
            return
        fc.fconv_plan_set_gather(h, fc.FCONV_GATHER_HALO)
        assert fc.fconv_plan_kernel(h).startswith("tma-halo")
        assert fc.fconv_plan_launch_count(h) == 1
        assert fc.fconv_workspace_size(h) == 0
        # the im2col gather (or cp.async for C = 32) brings the prep launch back for int8
        fc.fconv_plan_set_gather(h, fc.FCONV_GATHER_IM2COL)
        assert not fc.fconv_plan_kernel(h).startswith("tma-halo")
        if dtype == fc.FCONV_INT8:
            assert fc.fconv_plan_launch_count(h) == 2
            assert fc.fconv_workspace_size(h) > 0
        fc.fconv_plan_set_gather(h, fc.FCONV_GATHER_AUTO)
    finally:
        fc.fconv_plan_destroy(h)


def test_halo_gather_controls():
    h = _plan((4, 28, 28, 64, 64, 3, 3))
    try:
        assert _err(fc.fconv_plan_set_gather, h, 3) == fc.FCONV_ERR_INVALID_VALUE
        fc.fconv_plan_set_gather(h, fc.FCONV_GATHER_HALO)
        # a halo tile of either height; tile widths and split-K leave the gather
        fc.fconv_plan_set_tile_shape(h, 128, 64)
        assert fc.fconv_plan_kernel(h) == "tma-halo"
        fc.fconv_plan_set_tile_shape(h, 256, 64)
        assert fc.fconv_plan_kernel(h) == "tma-halo-m256"
        fc.fconv_plan_set_splits(h, 1)
        assert fc.fconv_plan_kernel(h) == "tma-halo-m256"
        fc.fconv_plan_set_tile(h, 128)
        assert not fc.fconv_plan_kernel(h).startswith("tma-halo")
        fc.fconv_plan_set_gather(h, fc.FCONV_GATHER_HALO)
        assert fc.fconv_plan_kernel(h).startswith("tma-halo")
        # the fp16 input copy moves an int8 plan off the gather
        fc.fconv_plan_set_input_widening(h, fc.FCONV_WIDEN_COPY)
        assert not fc.fconv_plan_kernel(h).startswith("tma-halo")
        assert _err(fc.fconv_plan_set_gather, h, fc.FCONV_GATHER_HALO) == \
            fc.FCONV_ERR_NOT_SUPPORTED
        fc.fconv_plan_set_input_widening(h, fc.FCONV_WIDEN_AUTO)
        fc.fconv_plan_set_gather(h, fc.FCONV_GATHER_HALO)
        assert fc.fconv_plan_kernel(h).startswith("tma-halo")
        # the cp.async test hook runs the general gather, with its copies
        fc.fconv_plan_set_debug(h, fc.FCONV_DEBUG_GATHER_CPASYNC)
        assert fc.fconv_plan_kernel(h) == "cp-async"
        assert fc.fconv_workspace_size(h) > 0
        fc.fconv_plan_set_debug(h, 0)
        assert fc.fconv_workspace_size(h) == 0
    finally:
        fc.fconv_plan_destroy(h)


def test_halo_tiles_cover_whole_output_rows():
    """Halo tiles are floor(128 * m / (Q + S - 1)) whole output rows of one
    image: the tile count is N * ceil(P / rows) (x the channel tiles)."""
    for (N, H, W, K), px in [((3, 56, 56, 64), 256), ((2, 14, 14, 128), 128), ((5, 9, 30, 64), 256)]:
        h = _plan((N, H, W, 64, K, 3, 3))
        try:
            fc.fconv_plan_set_gather(h, fc.FCONV_GATHER_HALO)
            fc.fconv_plan_set_tile_shape(h, px, 64)
            rows = px // (W + 2)
            tiles = N * -(-H // rows) * -(-K // 64)
            assert fc.fconv_plan_get_config(h)[2] == tiles
        finally:
            fc.fconv_plan_destroy(h)


def test_halo_gather_needs_a_cta_per_channel_tile():
    # each CTA keeps one 64-channel tile: more channel tiles than SMs rules
    # the gather out (152 SMs on GB300; 148 where no GPU reports a count)
    h = _plan((1, 8, 8, 64, 64 * 400, 3, 3))
    try:
        assert not fc.fconv_plan_kernel(h).startswith("tma-halo")
        assert _err(fc.fconv_plan_set_gather, h, fc.FCONV_GATHER_HALO) == \
            fc.FCONV_ERR_NOT_SUPPORTED
    finally:
        fc.fconv_plan_destroy(h)
