"""ctypes binding of the C ABI declared in ``include/dlc.h``.

Argument marshalling only: every function here forwards to the function of
the same name in ``libdlc.so``; all computation runs in the library's CUDA
kernels.  Functions that return a status in C raise :class:`DlcError` on a
non-success status; output parameters become return values.

The library must have been built (``deep_learning_convolution_gb300.build``
or ``__graft_entry__.build()``); importing this module without it raises.
There is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import (POINTER, byref, c_char_p, c_double, c_float, c_int, c_int64, c_size_t,
                    c_uint64, c_void_p)

from .build import LIB_PATH

# status codes (dlcStatus_t)
DLC_STATUS_SUCCESS = 0
DLC_STATUS_NOT_INITIALIZED = 1
DLC_STATUS_BAD_PARAM = 2
DLC_STATUS_NOT_SUPPORTED = 3
DLC_STATUS_EXECUTION_FAILED = 4
DLC_STATUS_INTERNAL_ERROR = 5
DLC_STATUS_ALLOC_FAILED = 6

DLC_DATA_FLOAT = 0
DLC_DATA_BFLOAT16 = 1
DLC_DATA_DOUBLE = 2
DLC_TENSOR_NCHW = 0
DLC_TENSOR_NHWC = 1
DLC_MATH_FP32 = 0
DLC_MATH_TF32 = 1
DLC_MATH_BF16 = 2
DLC_MATH_FP64 = 3
DLC_CROSS_CORRELATION = 0
DLC_CONVOLUTION = 1
DLC_ACTIVATION_IDENTITY = 0
DLC_ACTIVATION_RELU = 1
DLC_ACTIVATION_SIGMOID = 2
DLC_ACTIVATION_TANH = 3
DLC_ACTIVATION_CLIPPED_RELU = 4
DLC_POOLING_MAX = 0
DLC_POOLING_AVERAGE_COUNT_INCLUDE_PADDING = 1
DLC_POOLING_AVERAGE_COUNT_EXCLUDE_PADDING = 2
DLC_KERNEL_NONE = 0
DLC_KERNEL_FFMA = 1
DLC_KERNEL_TC_IM2COL = 2
DLC_KERNEL_TC_GATHER = 3
DLC_KERNEL_TC_GATHER_RUNS = 4
DLC_KERNEL_TC_WINDOW = 5
DLC_KERNEL_TC_IM2COL_PAIR = 6
DLC_KERNEL_DIRECT = 7
DLC_KERNEL_TC_WGRAD = 8
DLC_KERNEL_POOL_NHWC = 9
DLC_KERNEL_TC_ROWSTACK = 10
DLC_DEVERR_NONE = 0
DLC_DEVERR_WAIT_TIMEOUT = 1

KERNEL_NAMES = {DLC_KERNEL_NONE: "none", DLC_KERNEL_FFMA: "ffma",
                DLC_KERNEL_TC_IM2COL: "tc_im2col", DLC_KERNEL_TC_GATHER: "tc_gather",
                DLC_KERNEL_TC_GATHER_RUNS: "tc_runs", DLC_KERNEL_TC_WINDOW: "tc_window",
                DLC_KERNEL_TC_IM2COL_PAIR: "tc_im2col_pair", DLC_KERNEL_DIRECT: "direct",
                DLC_KERNEL_TC_WGRAD: "tc_wgrad", DLC_KERNEL_POOL_NHWC: "pool_nhwc",
                DLC_KERNEL_TC_ROWSTACK: "tc_rowstack"}

_h = c_void_p          # opaque handle / descriptor
_ph = POINTER(c_void_p)
_pi = POINTER(c_int)
_pi64 = POINTER(c_int64)
_pf = POINTER(c_float)

# name -> argtypes (all return dlcStatus_t = int unless listed in _RESTYPES)
SIGNATURES = {
    "dlcGetErrorString": [c_int],
    "dlcGetVersion": [_pi],
    "dlcCreate": [_ph],
    "dlcDestroy": [_h],
    "dlcSetStream": [_h, c_void_p],
    "dlcGetStream": [_h, _ph],
    "dlcSynchronize": [_h],
    "dlcGetLastDeviceError": [_h, _pi, _pi],
    "dlcGetLaunchCount": [_h, POINTER(c_uint64)],
    "dlcSetDeterministic": [_h, c_int],
    "dlcGetDeterministic": [_h, _pi],
    "dlcCreateTensorDescriptor": [_ph],
    "dlcDestroyTensorDescriptor": [_h],
    "dlcSetTensor4dDescriptor": [_h, c_int, c_int, c_int, c_int, c_int, c_int],
    "dlcSetTensor4dDescriptorEx": [_h, c_int, c_int, c_int, c_int, c_int,
                                   c_int64, c_int64, c_int64, c_int64],
    "dlcGetTensor4dDescriptor": [_h, _pi, _pi, _pi, _pi, _pi, _pi64, _pi64, _pi64, _pi64],
    "dlcCreateFilterDescriptor": [_ph],
    "dlcDestroyFilterDescriptor": [_h],
    "dlcSetFilter4dDescriptor": [_h, c_int, c_int, c_int, c_int, c_int, c_int],
    "dlcGetFilter4dDescriptor": [_h, _pi, _pi, _pi, _pi, _pi, _pi],
    "dlcCreateConvolutionDescriptor": [_ph],
    "dlcDestroyConvolutionDescriptor": [_h],
    "dlcSetConvolution2dDescriptor": [_h, c_int, c_int, c_int, c_int, c_int, c_int, c_int],
    "dlcSetConvolution2dPadding": [_h, c_int, c_int, c_int, c_int],
    "dlcGetConvolution2dDescriptor": [_h, _pi, _pi, _pi, _pi, _pi, _pi, _pi, _pi, _pi],
    "dlcGetConvolution2dForwardOutputDim": [_h, _h, _h, _pi, _pi, _pi, _pi],
    "dlcGetConvolutionForwardWorkspaceSize": [_h, _h, _h, _h, _h, POINTER(c_size_t)],
    "dlcGetConvolutionForwardKernel": [_h, _h, c_void_p, _h, c_void_p, _h, _h, c_void_p, _pi],
    "dlcConvolutionForward": [_h, _pf, _h, c_void_p, _h, c_void_p, _h, _pf, _h, c_void_p],
    "dlcConvolutionBiasActivationForward": [_h, _pf, _h, c_void_p, _h, c_void_p, _h, _pf,
                                            c_void_p, c_int, _h, c_void_p],
    "dlcSetConvolutionMode": [_h, c_int],
    "dlcGetConvolutionMode": [_h, _pi],
    "dlcConvolutionBackwardData": [_h, _pf, _h, c_void_p, _h, c_void_p, _h, _pf, _h, c_void_p],
    "dlcConvolutionBackwardFilter": [_h, _pf, _h, c_void_p, _h, c_void_p, _h, _pf, _h, c_void_p],
    "dlcGetConvolutionBackwardDataWorkspaceSize": [_h, _h, _h, _h, _h, POINTER(c_size_t)],
    "dlcGetConvolutionBackwardFilterWorkspaceSize": [_h, _h, _h, _h, _h, POINTER(c_size_t)],
    "dlcGetConvolutionBackwardDataKernel": [_h, _h, c_void_p, _h, c_void_p, _h, _h, c_void_p, _pi],
    "dlcGetConvolutionBackwardFilterKernel": [_h, _h, c_void_p, _h, c_void_p, _h, _h, c_void_p,
                                              _pi],
    "dlcCreatePoolingDescriptor": [_ph],
    "dlcDestroyPoolingDescriptor": [_h],
    "dlcSetPooling2dDescriptor": [_h] + [c_int] * 9,
    "dlcGetPooling2dDescriptor": [_h] + [_pi] * 9,
    "dlcGetPooling2dForwardOutputDim": [_h, _h, _pi, _pi, _pi, _pi],
    "dlcPoolingForward": [_h, _h, _pf, _h, c_void_p, _pf, _h, c_void_p],
    "dlcGetPoolingForwardKernel": [_h, _h, _h, c_void_p, _h, c_void_p, _pi],
    "dlcActivationForward": [_h, c_int, c_double, _pf, _h, c_void_p, _pf, _h, c_void_p],
    "dlcDebugWaitTimeoutSelfTest": [_h, c_int],
    "dlcConvolutionForwardNoAlloc": [c_void_p, _pf, _h, c_void_p, _h, c_void_p, _h, _pf, _h,
                                     c_void_p, c_void_p],
}
_RESTYPES = {"dlcGetErrorString": c_char_p}


class DlcError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} failed: {error_string(status)} ({status})")


_lib = None


def library_path() -> str:
    return LIB_PATH


def load_library(path: str = None):
    """Load libdlc.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build the CUDA library first "
                           "(python -m deep_learning_convolution_gb300.build)")
    import torch  # noqa: F401  -- loads the CUDA runtime this library shares
    lib = ctypes.CDLL(p)
    for name, args in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = _RESTYPES.get(name, c_int)
    if path is None:
        _lib = lib
    return lib


def error_string(status: int) -> str:
    try:
        return load_library().dlcGetErrorString(int(status)).decode()
    except Exception:  # pragma: no cover - library not loadable
        return f"status {status}"


def _check(name: str, status: int):
    if status != DLC_STATUS_SUCCESS:
        raise DlcError(name, status)


def _call(name, *args):
    _check(name, getattr(load_library(), name)(*args))


# ---------------------------------------------------------------------------
# same-named wrappers
# ---------------------------------------------------------------------------

def dlcGetErrorString(status: int) -> str:
    return error_string(status)


def dlcGetVersion() -> int:
    v = c_int()
    _call("dlcGetVersion", byref(v))
    return v.value


def dlcCreate():
    h = c_void_p()
    _call("dlcCreate", byref(h))
    return h


def dlcDestroy(handle):
    _call("dlcDestroy", handle)


def dlcSetStream(handle, stream_ptr: int):
    _call("dlcSetStream", handle, c_void_p(stream_ptr or None))


def dlcGetStream(handle) -> int:
    s = c_void_p()
    _call("dlcGetStream", handle, byref(s))
    return s.value or 0


def dlcSynchronize(handle):
    _call("dlcSynchronize", handle)


def dlcGetLastDeviceError(handle):
    code, detail = c_int(), c_int()
    _call("dlcGetLastDeviceError", handle, byref(code), byref(detail))
    return code.value, detail.value


def dlcGetLaunchCount(handle) -> int:
    n = c_uint64()
    _call("dlcGetLaunchCount", handle, byref(n))
    return n.value


def dlcSetDeterministic(handle, deterministic: int):
    _call("dlcSetDeterministic", handle, int(deterministic))


def dlcGetDeterministic(handle) -> int:
    v = c_int()
    _call("dlcGetDeterministic", handle, byref(v))
    return v.value


def dlcCreateTensorDescriptor():
    d = c_void_p()
    _call("dlcCreateTensorDescriptor", byref(d))
    return d


def dlcDestroyTensorDescriptor(d):
    _call("dlcDestroyTensorDescriptor", d)


def dlcSetTensor4dDescriptor(d, fmt, dtype, n, c, h, w):
    _call("dlcSetTensor4dDescriptor", d, fmt, dtype, n, c, h, w)


def dlcSetTensor4dDescriptorEx(d, dtype, n, c, h, w, ns, cs, hs, ws):
    _call("dlcSetTensor4dDescriptorEx", d, dtype, n, c, h, w, ns, cs, hs, ws)


def dlcGetTensor4dDescriptor(d):
    vals = [c_int() for _ in range(5)] + [c_int64() for _ in range(4)]
    _call("dlcGetTensor4dDescriptor", d, *[byref(v) for v in vals])
    return tuple(v.value for v in vals)


def dlcCreateFilterDescriptor():
    d = c_void_p()
    _call("dlcCreateFilterDescriptor", byref(d))
    return d


def dlcDestroyFilterDescriptor(d):
    _call("dlcDestroyFilterDescriptor", d)


def dlcSetFilter4dDescriptor(d, dtype, fmt, k, c, r, s):
    _call("dlcSetFilter4dDescriptor", d, dtype, fmt, k, c, r, s)


def dlcGetFilter4dDescriptor(d):
    vals = [c_int() for _ in range(6)]
    _call("dlcGetFilter4dDescriptor", d, *[byref(v) for v in vals])
    return tuple(v.value for v in vals)


def dlcCreateConvolutionDescriptor():
    d = c_void_p()
    _call("dlcCreateConvolutionDescriptor", byref(d))
    return d


def dlcDestroyConvolutionDescriptor(d):
    _call("dlcDestroyConvolutionDescriptor", d)


def dlcSetConvolution2dDescriptor(d, pad_h, pad_w, u, v, dil_h, dil_w, math):
    _call("dlcSetConvolution2dDescriptor", d, pad_h, pad_w, u, v, dil_h, dil_w, math)


def dlcSetConvolution2dPadding(d, pt, pb, pl, pr):
    _call("dlcSetConvolution2dPadding", d, pt, pb, pl, pr)


def dlcGetConvolution2dDescriptor(d):
    vals = [c_int() for _ in range(9)]
    _call("dlcGetConvolution2dDescriptor", d, *[byref(v) for v in vals])
    return tuple(v.value for v in vals)


def dlcGetConvolution2dForwardOutputDim(conv, x_desc, w_desc):
    vals = [c_int() for _ in range(4)]
    _call("dlcGetConvolution2dForwardOutputDim", conv, x_desc, w_desc, *[byref(v) for v in vals])
    return tuple(v.value for v in vals)


def dlcGetConvolutionForwardWorkspaceSize(handle, x_desc, w_desc, conv, y_desc) -> int:
    b = c_size_t()
    _call("dlcGetConvolutionForwardWorkspaceSize", handle, x_desc, w_desc, conv, y_desc, byref(b))
    return b.value


def dlcGetConvolutionForwardKernel(handle, x_desc, x_ptr, w_desc, w_ptr, conv, y_desc, y_ptr):
    k = c_int()
    _call("dlcGetConvolutionForwardKernel", handle, x_desc, c_void_p(x_ptr or None), w_desc,
          c_void_p(w_ptr or None), conv, y_desc, c_void_p(y_ptr or None), byref(k))
    return k.value


def dlcConvolutionForward(handle, alpha, x_desc, x_ptr, w_desc, w_ptr, conv, beta, y_desc, y_ptr):
    a, b = c_float(alpha), c_float(beta)
    _call("dlcConvolutionForward", handle, byref(a), x_desc, c_void_p(x_ptr), w_desc,
          c_void_p(w_ptr), conv, byref(b), y_desc, c_void_p(y_ptr))


def dlcConvolutionBiasActivationForward(handle, alpha, x_desc, x_ptr, w_desc, w_ptr, conv, beta,
                                        bias_ptr, activation, y_desc, y_ptr):
    a, b = c_float(alpha), c_float(beta)
    _call("dlcConvolutionBiasActivationForward", handle, byref(a), x_desc, c_void_p(x_ptr),
          w_desc, c_void_p(w_ptr), conv, byref(b), c_void_p(bias_ptr or None), activation,
          y_desc, c_void_p(y_ptr))


def dlcDebugWaitTimeoutSelfTest(handle, timeout_us: int):
    _call("dlcDebugWaitTimeoutSelfTest", handle, timeout_us)


def dlcConvolutionForwardNoAlloc(stream_ptr, alpha, x_desc, x_ptr, w_desc, w_ptr, conv, beta,
                                 y_desc, y_ptr, status_ptr=0):
    a, b = c_float(alpha), c_float(beta)
    _call("dlcConvolutionForwardNoAlloc", c_void_p(stream_ptr or None), byref(a), x_desc,
          c_void_p(x_ptr), w_desc, c_void_p(w_ptr), conv, byref(b), y_desc, c_void_p(y_ptr),
          c_void_p(status_ptr or None))


def dlcSetConvolutionMode(conv, mode: int):
    _call("dlcSetConvolutionMode", conv, int(mode))


def dlcGetConvolutionMode(conv) -> int:
    m = c_int()
    _call("dlcGetConvolutionMode", conv, byref(m))
    return m.value


def dlcConvolutionBackwardData(handle, alpha, w_desc, w_ptr, dy_desc, dy_ptr, conv, beta, dx_desc,
                               dx_ptr):
    a, b = c_float(alpha), c_float(beta)
    _call("dlcConvolutionBackwardData", handle, byref(a), w_desc, c_void_p(w_ptr), dy_desc,
          c_void_p(dy_ptr), conv, byref(b), dx_desc, c_void_p(dx_ptr))


def dlcConvolutionBackwardFilter(handle, alpha, x_desc, x_ptr, dy_desc, dy_ptr, conv, beta, dw_desc,
                                 dw_ptr):
    a, b = c_float(alpha), c_float(beta)
    _call("dlcConvolutionBackwardFilter", handle, byref(a), x_desc, c_void_p(x_ptr), dy_desc,
          c_void_p(dy_ptr), conv, byref(b), dw_desc, c_void_p(dw_ptr))


def dlcGetConvolutionBackwardDataWorkspaceSize(handle, w_desc, dy_desc, conv, dx_desc) -> int:
    n = c_size_t()
    _call("dlcGetConvolutionBackwardDataWorkspaceSize", handle, w_desc, dy_desc, conv, dx_desc,
          byref(n))
    return n.value


def dlcGetConvolutionBackwardFilterWorkspaceSize(handle, x_desc, dy_desc, conv, dw_desc) -> int:
    n = c_size_t()
    _call("dlcGetConvolutionBackwardFilterWorkspaceSize", handle, x_desc, dy_desc, conv, dw_desc,
          byref(n))
    return n.value


def dlcGetConvolutionBackwardDataKernel(handle, w_desc, w_ptr, dy_desc, dy_ptr, conv, dx_desc,
                                        dx_ptr) -> int:
    k = c_int()
    _call("dlcGetConvolutionBackwardDataKernel", handle, w_desc, c_void_p(w_ptr or None), dy_desc,
          c_void_p(dy_ptr or None), conv, dx_desc, c_void_p(dx_ptr or None), byref(k))
    return k.value


def dlcGetConvolutionBackwardFilterKernel(handle, x_desc, x_ptr, dy_desc, dy_ptr, conv, dw_desc,
                                          dw_ptr) -> int:
    k = c_int()
    _call("dlcGetConvolutionBackwardFilterKernel", handle, x_desc, c_void_p(x_ptr or None),
          dy_desc, c_void_p(dy_ptr or None), conv, dw_desc, c_void_p(dw_ptr or None), byref(k))
    return k.value


def dlcCreatePoolingDescriptor():
    d = c_void_p()
    _call("dlcCreatePoolingDescriptor", byref(d))
    return d


def dlcDestroyPoolingDescriptor(d):
    _call("dlcDestroyPoolingDescriptor", d)


def dlcSetPooling2dDescriptor(d, mode, r, s, pt, pb, pl, pr, u, v):
    _call("dlcSetPooling2dDescriptor", d, int(mode), int(r), int(s), int(pt), int(pb), int(pl),
          int(pr), int(u), int(v))


def dlcGetPooling2dDescriptor(d):
    vals = [c_int() for _ in range(9)]
    _call("dlcGetPooling2dDescriptor", d, *[byref(v) for v in vals])
    return tuple(v.value for v in vals)


def dlcGetPooling2dForwardOutputDim(d, x_desc):
    n, c, p, q = c_int(), c_int(), c_int(), c_int()
    _call("dlcGetPooling2dForwardOutputDim", d, x_desc, byref(n), byref(c), byref(p), byref(q))
    return n.value, c.value, p.value, q.value


def dlcPoolingForward(handle, pool, alpha, x_desc, x_ptr, beta, y_desc, y_ptr):
    a, b = c_float(alpha), c_float(beta)
    _call("dlcPoolingForward", handle, pool, byref(a), x_desc, c_void_p(x_ptr), byref(b), y_desc,
          c_void_p(y_ptr))


def dlcGetPoolingForwardKernel(handle, pool, x_desc, x_ptr, y_desc, y_ptr) -> int:
    k = c_int()
    _call("dlcGetPoolingForwardKernel", handle, pool, x_desc, c_void_p(x_ptr or None), y_desc,
          c_void_p(y_ptr or None), byref(k))
    return k.value


def dlcActivationForward(handle, mode, coef, alpha, x_desc, x_ptr, beta, y_desc, y_ptr):
    a, b = c_float(alpha), c_float(beta)
    _call("dlcActivationForward", handle, int(mode), c_double(coef), byref(a), x_desc,
          c_void_p(x_ptr), byref(b), y_desc, c_void_p(y_ptr))
