"""Fused quantized Conv2D forward pass for GB300 (sm_103a).

A thin ctypes binding over the C ABI of ``include/fconv.h``: every function
here has the name of the C function it calls and only marshals arguments
(integers for device/host pointers, floats for scalars, a CUDA stream
handle).  All computation runs in ``libfconv.so``'s CUDA kernels; there is
no CPU fallback, and the first call raises ImportError when the library
is missing.  ``Conv2dPlan`` is a convenience wrapper that takes torch tensors
and passes their ``data_ptr()``.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfconv.so")

FCONV_OK = 0
FCONV_ERR_INVALID_VALUE = 1
FCONV_ERR_NOT_SUPPORTED = 2
FCONV_ERR_MISALIGNED = 3
FCONV_ERR_CUDA = 4
FCONV_ERR_TIMEOUT = 5
FCONV_ERR_INTERNAL = 6
FCONV_ERR_WORKSPACE = 7

FCONV_SAME, FCONV_VALID = 0, 1
FCONV_INT8, FCONV_BF16 = 0, 1
FCONV_ACT_NONE, FCONV_ACT_RELU, FCONV_ACT_LEAKY_RELU, FCONV_ACT_CLIPPED_RELU, FCONV_ACT_CLAMP = (
    0, 1, 2, 3, 4)
FCONV_DEBUG_DROP_ARRIVE = 1
FCONV_DEBUG_GATHER_CPASYNC = 2
FCONV_DEBUG_ONE_KBLOCK_STAGES = 4
FCONV_DEBUG_ONE_MMA_ISSUER = 8
FCONV_WIDEN_AUTO, FCONV_WIDEN_IN_KERNEL, FCONV_WIDEN_COPY = 0, 1, 2
FCONV_GATHER_AUTO, FCONV_GATHER_IM2COL, FCONV_GATHER_HALO = 0, 1, 2


class FconvError(RuntimeError):
    def __init__(self, status: int, func: str, detail: str):
        self.status = status
        super().__init__(f"{func}: {fconv_status_string(status)}: {detail}")


_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -m quantized_conv2d_gb300.build` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    p, i32, u32, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_float,
                            ctypes.c_size_t)
    pp = ctypes.POINTER(ctypes.c_void_p)
    pi = ctypes.POINTER(ctypes.c_int)
    psz = ctypes.POINTER(ctypes.c_size_t)
    sigs = {
        "fconv_plan_create": [pp] + [i32] * 12,
        "fconv_plan_create_transposed": [pp] + [i32] * 15,
        "fconv_plan_destroy": [p],
        "fconv_plan_output_shape": [p, pi, pi, pi, pi],
        "fconv_plan_padding": [p, pi, pi, pi, pi],
        "fconv_workspace_size": [p, psz],
        "fconv_run": [p, p, p, p, p, f32, f32, p, p, sz, p],
        "fconv_run_channel_scale": [p, p, p, p, p, p, f32, p, p, sz, p],
        "fconv_run_accumulators": [p, p, p, p, p, sz, p],
        "fconv_host_workspace_size": [p, i32, psz],
        "fconv_run_host": [p, p, p, p, p, f32, f32, p, p, sz, p],
        "fconv_plan_check": [p, p],
        "fconv_plan_set_tile": [p, i32],
        "fconv_plan_get_config": [p, pi, pi, pi],
        "fconv_plan_set_timeout_ms": [p, u32],
        "fconv_plan_set_debug": [p, i32],
        "fconv_plan_set_stage_events": [p, ctypes.POINTER(ctypes.c_void_p)],
        "fconv_run_no_alloc": [p, p, p, p, p, f32, f32, p, p],
        "fconv_plan_set_host_chunks": [p, i32],
        "fconv_plan_host_chunk_sizes": [p, i32, pi, i32, pi],
        "fconv_plan_set_tile_shape": [p, i32, i32],
        "fconv_plan_launch_count": [p, pi],
        "fconv_plan_set_activation_params": [p, f32, f32],
        "fconv_fold_batchnorm": [i32, f32, p, p, p, p, p, f32, p, p],
        "fconv_plan_set_splits": [p, i32],
        "fconv_plan_get_splits": [p, pi],
        "fconv_plan_set_input_widening": [p, i32],
        "fconv_plan_set_gather": [p, i32],
        "fconv_plan_get_input_widening": [p, pi],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = i32
    lib.fconv_status_string.argtypes = [i32]
    lib.fconv_status_string.restype = ctypes.c_char_p
    lib.fconv_plan_kernel.argtypes = [p]
    lib.fconv_plan_kernel.restype = ctypes.c_char_p
    lib.fconv_last_error.argtypes = []
    lib.fconv_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int, func: str):
    if status != FCONV_OK:
        raise FconvError(status, func, fconv_last_error())


def fconv_status_string(status: int) -> str:
    return _load().fconv_status_string(int(status)).decode()


def fconv_last_error() -> str:
    return _load().fconv_last_error().decode()


def fconv_plan_create(N, H, W, C, K, R, S, stride_h, stride_w, padding, dtype, act) -> int:
    plan = ctypes.c_void_p()
    _check(_load().fconv_plan_create(ctypes.byref(plan), N, H, W, C, K, R, S, stride_h,
                                     stride_w, padding, dtype, act), "fconv_plan_create")
    return plan.value


def fconv_plan_create_transposed(N, H, W, C, K, R, S, stride_h, stride_w, pad_top, pad_bottom,
                                 pad_left, pad_right, dtype, act) -> int:
    plan = ctypes.c_void_p()
    _check(_load().fconv_plan_create_transposed(ctypes.byref(plan), N, H, W, C, K, R, S, stride_h,
                                                stride_w, pad_top, pad_bottom, pad_left,
                                                pad_right, dtype, act),
           "fconv_plan_create_transposed")
    return plan.value


def fconv_plan_destroy(plan: int) -> None:
    _check(_load().fconv_plan_destroy(plan), "fconv_plan_destroy")


def fconv_plan_output_shape(plan: int):
    v = [ctypes.c_int() for _ in range(4)]
    _check(_load().fconv_plan_output_shape(plan, *[ctypes.byref(x) for x in v]),
           "fconv_plan_output_shape")
    return tuple(x.value for x in v)


def fconv_fold_batchnorm(conv_scale: float, gamma, beta, mean, var, eps: float, bias=None):
    """fconv_fold_batchnorm on host fp32 vectors [K]: returns (conv_scale_k,
    bias_k) numpy arrays for fconv_run_channel_scale."""
    import numpy as np
    arrs = [np.ascontiguousarray(a, dtype=np.float32) for a in (gamma, beta, mean, var)]
    K = arrs[0].shape[0]
    if any(a.shape != (K,) for a in arrs):
        raise ValueError("gamma, beta, mean and var must be vectors of one length")
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    if b is not None and b.shape != (K,):
        raise ValueError("bias must have the length of gamma")
    scale_out = np.empty(K, np.float32)
    bias_out = np.empty(K, np.float32)
    ptr = lambda a: None if a is None else a.ctypes.data
    _check(_load().fconv_fold_batchnorm(K, float(conv_scale), ptr(b), *[ptr(a) for a in arrs],
                                        float(eps), ptr(scale_out), ptr(bias_out)),
           "fconv_fold_batchnorm")
    return scale_out, bias_out


def fconv_plan_padding(plan: int):
    v = [ctypes.c_int() for _ in range(4)]
    _check(_load().fconv_plan_padding(plan, *[ctypes.byref(x) for x in v]), "fconv_plan_padding")
    return tuple(x.value for x in v)


def fconv_workspace_size(plan: int) -> int:
    b = ctypes.c_size_t()
    _check(_load().fconv_workspace_size(plan, ctypes.byref(b)), "fconv_workspace_size")
    return b.value


def fconv_run(plan, x, w, bias, side, conv_scale, side_scale, y, workspace, workspace_bytes,
              stream) -> None:
    _check(_load().fconv_run(plan, x, w, bias, side, conv_scale, side_scale, y, workspace,
                             workspace_bytes, stream), "fconv_run")


def fconv_plan_set_activation_params(plan, alpha: float, beta: float) -> None:
    _check(_load().fconv_plan_set_activation_params(plan, alpha, beta),
           "fconv_plan_set_activation_params")


def fconv_run_channel_scale(plan, x, w, bias, side, conv_scale, side_scale, y, workspace,
                            workspace_bytes, stream) -> None:
    """fconv_run with conv_scale a device fp32 [K] pointer (one scale per
    output channel)."""
    _check(_load().fconv_run_channel_scale(plan, x, w, bias, side, conv_scale, side_scale, y,
                                           workspace, workspace_bytes, stream),
           "fconv_run_channel_scale")


def fconv_run_no_alloc(plan, x, w, bias, side, conv_scale, side_scale, y, stream) -> None:
    """fconv_run with scratch from the library's built-in 32 MiB device array,
    for callers that cannot allocate device memory."""
    _check(_load().fconv_run_no_alloc(plan, x, w, bias, side, conv_scale, side_scale, y, stream),
           "fconv_run_no_alloc")


def fconv_run_accumulators(plan, x, w, acc, workspace, workspace_bytes, stream) -> None:
    _check(_load().fconv_run_accumulators(plan, x, w, acc, workspace, workspace_bytes, stream),
           "fconv_run_accumulators")


def fconv_host_workspace_size(plan: int, with_side: bool) -> int:
    b = ctypes.c_size_t()
    _check(_load().fconv_host_workspace_size(plan, int(bool(with_side)), ctypes.byref(b)),
           "fconv_host_workspace_size")
    return b.value


def fconv_run_host(plan, x_host, w_host, bias_host, side_host, conv_scale, side_scale, y_host,
                   device_workspace, workspace_bytes, stream) -> None:
    _check(_load().fconv_run_host(plan, x_host, w_host, bias_host, side_host, conv_scale,
                                  side_scale, y_host, device_workspace, workspace_bytes, stream),
           "fconv_run_host")


def fconv_plan_set_host_chunks(plan, chunks: int) -> None:
    _check(_load().fconv_plan_set_host_chunks(plan, chunks), "fconv_plan_set_host_chunks")


def fconv_plan_host_chunk_sizes(plan, sm_count: int) -> list:
    n = ctypes.c_int(0)
    _check(_load().fconv_plan_host_chunk_sizes(plan, sm_count, None, 0, ctypes.byref(n)),
           "fconv_plan_host_chunk_sizes")
    buf = (ctypes.c_int * max(n.value, 1))()
    _check(_load().fconv_plan_host_chunk_sizes(plan, sm_count, buf, n.value, ctypes.byref(n)),
           "fconv_plan_host_chunk_sizes")
    return list(buf[:n.value])


def fconv_plan_set_tile_shape(plan, pixels: int, channels: int) -> None:
    _check(_load().fconv_plan_set_tile_shape(plan, pixels, channels), "fconv_plan_set_tile_shape")


def fconv_plan_launch_count(plan) -> int:
    n = ctypes.c_int()
    _check(_load().fconv_plan_launch_count(plan, ctypes.byref(n)), "fconv_plan_launch_count")
    return n.value


def fconv_plan_kernel(plan) -> str:
    return _load().fconv_plan_kernel(plan).decode()


def fconv_plan_check(plan, stream) -> None:
    _check(_load().fconv_plan_check(plan, stream), "fconv_plan_check")


def fconv_plan_set_splits(plan, splits: int) -> None:
    _check(_load().fconv_plan_set_splits(plan, splits), "fconv_plan_set_splits")


def fconv_plan_get_splits(plan) -> int:
    v = ctypes.c_int()
    _check(_load().fconv_plan_get_splits(plan, ctypes.byref(v)), "fconv_plan_get_splits")
    return v.value


def fconv_plan_set_input_widening(plan, mode: int) -> None:
    _check(_load().fconv_plan_set_input_widening(plan, mode), "fconv_plan_set_input_widening")


def fconv_plan_set_gather(plan, mode: int) -> None:
    _check(_load().fconv_plan_set_gather(plan, mode), "fconv_plan_set_gather")


def fconv_plan_get_input_widening(plan) -> int:
    v = ctypes.c_int()
    _check(_load().fconv_plan_get_input_widening(plan, ctypes.byref(v)),
           "fconv_plan_get_input_widening")
    return v.value


def fconv_plan_set_tile(plan, block_n: int) -> None:
    _check(_load().fconv_plan_set_tile(plan, block_n), "fconv_plan_set_tile")


def fconv_plan_get_config(plan):
    v = [ctypes.c_int() for _ in range(3)]
    _check(_load().fconv_plan_get_config(plan, *[ctypes.byref(x) for x in v]),
           "fconv_plan_get_config")
    return tuple(x.value for x in v)


def fconv_plan_set_timeout_ms(plan, ms: int) -> None:
    _check(_load().fconv_plan_set_timeout_ms(plan, ms), "fconv_plan_set_timeout_ms")


def fconv_plan_set_debug(plan, flags: int) -> None:
    _check(_load().fconv_plan_set_debug(plan, flags), "fconv_plan_set_debug")


def fconv_plan_set_stage_events(plan, events) -> None:
    """events: four cudaEvent_t handles (ints), or None to disable."""
    arr = None if events is None else (ctypes.c_void_p * 4)(*events)
    _check(_load().fconv_plan_set_stage_events(plan, arr), "fconv_plan_set_stage_events")


# ---------------------------------------------------------------- torch glue
def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream):
    return stream.cuda_stream if stream is not None else None


class Conv2dPlan:
    """One fconv plan plus its device workspace, for torch tensors.

    Shapes: x [N,H,W,C], w [R,S,C,K] (int8 or bfloat16), bias [K] float32,
    side/y [N,P,Q,K] in the output dtype.  ``stride`` is an int or (sh, sw);
    ``padding`` is "SAME" or "VALID"; ``dtype`` is "int8" or "bf16".
    """

    def __init__(self, N, H, W, C, K, R, S, stride=1, padding="SAME", dtype="int8", relu=True,
                 device=None, alpha=0.0, beta=0.0, transposed_pads=None):
        """relu: True/False (BiasAdd+Relu / BiasAdd) or an FCONV_ACT_* code;
        alpha, beta: that activation's parameters.  transposed_pads =
        (top, bottom, left, right) makes a transposed-convolution plan
        (padding is then ignored)."""
        import torch
        sh, sw = (stride, stride) if isinstance(stride, int) else stride
        dt = {"int8": FCONV_INT8, "bf16": FCONV_BF16}[dtype]
        self.dtype = dtype
        if isinstance(relu, bool):
            act = FCONV_ACT_RELU if relu else FCONV_ACT_NONE
        else:
            act = int(relu)
        if transposed_pads is not None:
            self.handle = fconv_plan_create_transposed(N, H, W, C, K, R, S, sh, sw,
                                                       *transposed_pads, dt, act)
        else:
            pad = {"SAME": FCONV_SAME, "VALID": FCONV_VALID}[padding]
            self.handle = fconv_plan_create(N, H, W, C, K, R, S, sh, sw, pad, dt, act)
        if alpha or beta:
            fconv_plan_set_activation_params(self.handle, alpha, beta)
        self.out_shape = fconv_plan_output_shape(self.handle)
        self.ws_bytes = fconv_workspace_size(self.handle)
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8,
                                     device=self.device)

    @property
    def torch_dtype(self):
        import torch
        return torch.int8 if self.dtype == "int8" else torch.bfloat16

    def new_output(self):
        import torch
        return torch.empty(self.out_shape, dtype=self.torch_dtype, device=self.device)

    def _ensure_workspace(self):
        # the scratch a run needs depends on the tile and gather in force
        need = fconv_workspace_size(self.handle)
        if need > self.workspace.numel():
            import torch
            self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        self.ws_bytes = need

    def run(self, x, w, bias, side=None, conv_scale=1.0, side_scale=0.0, y=None, stream=None):
        """conv_scale: a Python float, or a device fp32 tensor of K elements
        (one scale per output channel)."""
        import torch
        self._ensure_workspace()
        if y is None:
            y = self.new_output()
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        if isinstance(conv_scale, torch.Tensor):
            if conv_scale.dtype != torch.float32 or conv_scale.numel() != self.out_shape[3]:
                raise ValueError("a per-channel conv_scale is a float32 tensor of K elements")
            fconv_run_channel_scale(self.handle, _ptr(x), _ptr(w), _ptr(bias), _ptr(side),
                                    _ptr(conv_scale), side_scale, _ptr(y),
                                    _ptr(self.workspace), self.workspace.numel(),
                                    _stream_handle(st))
        else:
            fconv_run(self.handle, _ptr(x), _ptr(w), _ptr(bias), _ptr(side), conv_scale,
                      side_scale, _ptr(y), _ptr(self.workspace), self.workspace.numel(),
                      _stream_handle(st))
        return y

    def accumulators(self, x, w, acc=None, stream=None):
        import torch
        self._ensure_workspace()
        if acc is None:
            dt = torch.int32 if self.dtype == "int8" else torch.float32
            acc = torch.empty(self.out_shape, dtype=dt, device=self.device)
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        fconv_run_accumulators(self.handle, _ptr(x), _ptr(w), _ptr(acc), _ptr(self.workspace),
                               self.workspace.numel(), _stream_handle(st))
        return acc

    def check(self, stream=None):
        import torch
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        fconv_plan_check(self.handle, _stream_handle(st))

    def config(self):
        return fconv_plan_get_config(self.handle)

    def set_tile(self, block_n: int):
        fconv_plan_set_tile(self.handle, block_n)

    def close(self):
        if getattr(self, "handle", None):
            fconv_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
