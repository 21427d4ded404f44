"""Python front end of the CPU oracle (``conv_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package's smoke
check and by the benchmark's CPU-baseline leg, never by the product path.
It shares no code with the CUDA library.

``build()`` compiles ``conv_oracle.c`` with gcc into ``oracle/_build`` (no
OpenMP runtime: plain pthreads).  ``conv2d_fprop`` takes numpy arrays in any
layout (strides are read from the arrays) and returns FP64 y and
bound = sum |x*w|.  ``conv2d_dgrad`` and ``conv2d_wgrad`` are the gradients of
that sum with respect to x and w (the backward routines), with point
evaluators for sampled checks.  ``pool2d_fprop`` and ``activation_fprop``
are the pooling and activation primitives.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from typing import Optional, Tuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "conv_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "libconv_oracle.so")

_lib = None
_i64p = ctypes.POINTER(ctypes.c_longlong)
_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False, src: str = SRC, out: str = LIB) -> str:
    """Compile the oracle shared library (idempotent unless ``force``)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, src, "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: Optional[str] = None):
    """Load (building if needed) the oracle library; returns the ctypes handle."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    p = path or build()
    lib = ctypes.CDLL(p)
    lib.oracle_out_extent.restype = ctypes.c_longlong
    lib.oracle_out_extent.argtypes = [ctypes.c_longlong] * 6
    common = [_dp, _i64p, _dp, _i64p]
    ints = [ctypes.c_int] * 15
    lib.oracle_conv2d_fprop.restype = ctypes.c_int
    lib.oracle_conv2d_fprop.argtypes = (common + [_dp, _i64p, _dp] + ints
                                        + [ctypes.c_double, ctypes.c_double, _dp, _dp,
                                           ctypes.c_int, ctypes.c_int])
    lib.oracle_conv2d_fprop_points.restype = ctypes.c_int
    lib.oracle_conv2d_fprop_points.argtypes = (common + [_i64p] + ints
                                               + [ctypes.c_double, ctypes.c_double, _dp, _dp,
                                                  ctypes.c_int, _i64p, ctypes.c_longlong,
                                                  _dp, _dp])
    grad = [_dp, _i64p, _dp, _i64p, _dp, _i64p, _dp] + [ctypes.c_int] * 16
    lib.oracle_conv2d_dgrad.restype = ctypes.c_int
    lib.oracle_conv2d_dgrad.argtypes = grad
    lib.oracle_conv2d_wgrad.restype = ctypes.c_int
    lib.oracle_conv2d_wgrad.argtypes = grad
    lib.oracle_pool2d_fprop.restype = ctypes.c_int
    lib.oracle_pool2d_fprop.argtypes = ([_dp, _i64p, _dp, _i64p] + [ctypes.c_int] * 13
                                        + [ctypes.c_double, ctypes.c_double, _dp])
    lib.oracle_activation_fprop.restype = ctypes.c_int
    lib.oracle_activation_fprop.argtypes = ([_dp, _i64p, _dp, _i64p] + [ctypes.c_int] * 5
                                            + [ctypes.c_double] * 3 + [_dp])
    gpts = ([_dp, _i64p, _dp, _i64p] + [ctypes.c_int] * 15
            + [_i64p, ctypes.c_longlong, _dp, _dp])
    lib.oracle_conv2d_dgrad_points.restype = ctypes.c_int
    lib.oracle_conv2d_dgrad_points.argtypes = gpts
    lib.oracle_conv2d_wgrad_points.restype = ctypes.c_int
    lib.oracle_conv2d_wgrad_points.argtypes = gpts
    if path is None:
        _lib = lib
    return lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _strides(a: np.ndarray) -> np.ndarray:
    return np.array([s // a.itemsize for s in a.strides], dtype=np.int64)


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(_dp)


def out_extent(inp, pad_lo, pad_hi, filt, dil, stride, lib=None) -> int:
    lib = lib or load()
    return int(lib.oracle_out_extent(inp, pad_lo, pad_hi, filt, dil, stride))


def _as_f64_view(a: np.ndarray, name: str) -> np.ndarray:
    if a.dtype != np.float64:
        raise TypeError(f"{name} must be float64 (widen the rounded inputs exactly first)")
    return a


def conv2d_fprop(x: np.ndarray, w: np.ndarray, *, pads=(0, 0, 0, 0), stride=(1, 1),
                 dilation=(1, 1), alpha: float = 1.0, beta: float = 0.0,
                 y_in: Optional[np.ndarray] = None, bias: Optional[np.ndarray] = None,
                 relu: bool = False, nthreads: Optional[int] = None,
                 x_axes: str = "NCHW", w_axes: str = "KCRS", lib=None
                 ) -> Tuple[np.ndarray, np.ndarray]:
    """Forward convolution on FP64 arrays.

    ``x`` is indexed with axes ``x_axes`` (a permutation of "NCHW"), ``w`` with
    ``w_axes`` (a permutation of "KCRS"); any strides are allowed.  ``pads`` is
    (top, bottom, left, right).  Returns (y, bound) as NCHW-shaped FP64 arrays
    [N, K, P, Q].
    """
    lib = lib or load()
    x = _as_f64_view(x, "x")
    w = _as_f64_view(w, "w")
    xs_ax = _strides(x)
    ws_ax = _strides(w)
    dims_x = dict(zip(x_axes, x.shape))
    dims_w = dict(zip(w_axes, w.shape))
    xs = np.array([xs_ax[x_axes.index(a)] for a in "NCHW"], dtype=np.int64)
    ws = np.array([ws_ax[w_axes.index(a)] for a in "KCRS"], dtype=np.int64)
    N, C, H, W = (dims_x[a] for a in "NCHW")
    K, C2, R, S = (dims_w[a] for a in "KCRS")
    if C2 != C:
        raise ValueError("channel mismatch between x and w")
    pt, pb, pl, pr = pads
    u, v = stride
    dh, dw = dilation
    P = out_extent(H, pt, pb, R, dh, u, lib)
    Q = out_extent(W, pl, pr, S, dw, v, lib)
    if P <= 0 or Q <= 0:
        raise ValueError(f"empty output (P={P}, Q={Q})")
    y = np.zeros((N, K, P, Q), dtype=np.float64)
    bound = np.zeros_like(y)
    ys = _strides(y)
    if y_in is not None:
        y_in = np.ascontiguousarray(y_in, dtype=np.float64).reshape(N, K, P, Q)
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float64).reshape(K)
    rc = lib.oracle_conv2d_fprop(
        _ptr(x), xs.ctypes.data_as(_i64p), _ptr(w), ws.ctypes.data_as(_i64p),
        _ptr(y), ys.ctypes.data_as(_i64p), _ptr(bound),
        N, C, H, W, K, R, S, pt, pb, pl, pr, u, v, dh, dw,
        float(alpha), float(beta), _ptr(y_in), _ptr(bias), int(bool(relu)),
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_conv2d_fprop returned {rc}")
    return y, bound


def conv2d_fprop_points(x: np.ndarray, w: np.ndarray, pts: np.ndarray, *, pads=(0, 0, 0, 0),
                        stride=(1, 1), dilation=(1, 1), alpha: float = 1.0, beta: float = 0.0,
                        y_in: Optional[np.ndarray] = None, bias: Optional[np.ndarray] = None,
                        relu: bool = False, x_axes: str = "NCHW", w_axes: str = "KCRS",
                        lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """The oracle at sampled output coordinates ``pts`` (int64 [n,4]: n,k,p,q).
    ``y_in`` (if used) is an [N,K,P,Q]-indexed FP64 array with any
    non-negative strides (a transposed view is read in place).  Returns
    (values, bound)."""
    lib = lib or load()
    x = _as_f64_view(x, "x")
    w = _as_f64_view(w, "w")
    xs_ax = _strides(x)
    ws_ax = _strides(w)
    dims_x = dict(zip(x_axes, x.shape))
    dims_w = dict(zip(w_axes, w.shape))
    xs = np.array([xs_ax[x_axes.index(a)] for a in "NCHW"], dtype=np.int64)
    ws = np.array([ws_ax[w_axes.index(a)] for a in "KCRS"], dtype=np.int64)
    N, C, H, W = (dims_x[a] for a in "NCHW")
    K, _, R, S = (dims_w[a] for a in "KCRS")
    pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 4)
    out = np.zeros(len(pts), dtype=np.float64)
    bnd = np.zeros(len(pts), dtype=np.float64)
    ys = None
    if y_in is not None:
        # any (non-negative) strides: the C side reads y_in through them
        y_in = _as_f64_view(np.asarray(y_in), "y_in")
        if y_in.shape[1] != K or y_in.ndim != 4 or min(y_in.strides) < 0:
            raise ValueError("y_in must be an [N, K, P, Q] view with non-negative strides")
        ys = _strides(y_in)
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float64).reshape(K)
    pt, pb, pl, pr = pads
    rc = lib.oracle_conv2d_fprop_points(
        _ptr(x), xs.ctypes.data_as(_i64p), _ptr(w), ws.ctypes.data_as(_i64p),
        ys.ctypes.data_as(_i64p) if ys is not None else None,
        N, C, H, W, K, R, S, pt, pb, pl, pr, stride[0], stride[1], dilation[0], dilation[1],
        float(alpha), float(beta), _ptr(y_in), _ptr(bias),
        int(bool(relu)), pts.ctypes.data_as(_i64p), len(pts), _ptr(out), _ptr(bnd))
    if rc != 0:
        raise ValueError(f"oracle_conv2d_fprop_points returned {rc}")
    return out, bnd


def conv2d_dgrad(dy: np.ndarray, w: np.ndarray, in_hw: Tuple[int, int], *, pads=(0, 0, 0, 0),
                 stride=(1, 1), dilation=(1, 1), nthreads: Optional[int] = None,
                 lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """Gradient of the forward convolution with respect to x, for an input of
    spatial size ``in_hw`` = (H, W): dy is NCHW-shaped [N, K, P, Q] FP64, w
    KCRS FP64 (any strides).  Returns (dx, bound) as [N, C, H, W] FP64 arrays,
    bound = sum |dy*w| over the products that make each dx."""
    lib = lib or load()
    dy = _as_f64_view(dy, "dy")
    w = _as_f64_view(w, "w")
    N, K, P, Q = dy.shape
    K2, C, R, S = w.shape
    if K2 != K:
        raise ValueError("filter count mismatch between dy and w")
    H, W = in_hw
    pt, pb, pl, pr = pads
    if (out_extent(H, pt, pb, R, dilation[0], stride[0], lib),
            out_extent(W, pl, pr, S, dilation[1], stride[1], lib)) != (P, Q):
        raise ValueError("dy does not have the forward output's extent")
    dx = np.zeros((N, C, H, W), dtype=np.float64)
    bound = np.zeros_like(dx)
    rc = lib.oracle_conv2d_dgrad(
        _ptr(dy), _strides(dy).ctypes.data_as(_i64p), _ptr(w), _strides(w).ctypes.data_as(_i64p),
        _ptr(dx), _strides(dx).ctypes.data_as(_i64p), _ptr(bound),
        N, C, H, W, K, R, S, pt, pb, pl, pr, stride[0], stride[1], dilation[0], dilation[1],
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_conv2d_dgrad returned {rc}")
    return dx, bound


def conv2d_wgrad(x: np.ndarray, dy: np.ndarray, filt_rs: Tuple[int, int], *, pads=(0, 0, 0, 0),
                 stride=(1, 1), dilation=(1, 1), nthreads: Optional[int] = None,
                 lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """Gradient of the forward convolution with respect to w, for filters of
    size ``filt_rs`` = (R, S): x NCHW-shaped [N, C, H, W] FP64, dy [N, K, P, Q]
    FP64 (any strides).  Returns (dw, bound) as [K, C, R, S] FP64 arrays."""
    lib = lib or load()
    x = _as_f64_view(x, "x")
    dy = _as_f64_view(dy, "dy")
    N, C, H, W = x.shape
    N2, K, P, Q = dy.shape
    if N2 != N:
        raise ValueError("batch mismatch between x and dy")
    R, S = filt_rs
    pt, pb, pl, pr = pads
    if (out_extent(H, pt, pb, R, dilation[0], stride[0], lib),
            out_extent(W, pl, pr, S, dilation[1], stride[1], lib)) != (P, Q):
        raise ValueError("dy does not have the forward output's extent")
    dw = np.zeros((K, C, R, S), dtype=np.float64)
    bound = np.zeros_like(dw)
    rc = lib.oracle_conv2d_wgrad(
        _ptr(x), _strides(x).ctypes.data_as(_i64p), _ptr(dy), _strides(dy).ctypes.data_as(_i64p),
        _ptr(dw), _strides(dw).ctypes.data_as(_i64p), _ptr(bound),
        N, C, H, W, K, R, S, pt, pb, pl, pr, stride[0], stride[1], dilation[0], dilation[1],
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_conv2d_wgrad returned {rc}")
    return dw, bound


def conv2d_dgrad_points(dy: np.ndarray, w: np.ndarray, in_hw: Tuple[int, int], pts: np.ndarray,
                        *, pads=(0, 0, 0, 0), stride=(1, 1), dilation=(1, 1),
                        lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """dx of :func:`conv2d_dgrad` at coordinates ``pts`` (int64 [n,4]:
    n,c,h,w).  Returns (values, bound)."""
    lib = lib or load()
    dy = _as_f64_view(dy, "dy")
    w = _as_f64_view(w, "w")
    N, K, P, Q = dy.shape
    _, C, R, S = w.shape
    H, W = in_hw
    pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 4)
    out = np.zeros(len(pts), dtype=np.float64)
    bnd = np.zeros(len(pts), dtype=np.float64)
    pt, pb, pl, pr = pads
    rc = lib.oracle_conv2d_dgrad_points(
        _ptr(dy), _strides(dy).ctypes.data_as(_i64p), _ptr(w), _strides(w).ctypes.data_as(_i64p),
        N, C, H, W, K, R, S, pt, pb, pl, pr, stride[0], stride[1], dilation[0], dilation[1],
        pts.ctypes.data_as(_i64p), len(pts), _ptr(out), _ptr(bnd))
    if rc != 0:
        raise ValueError(f"oracle_conv2d_dgrad_points returned {rc}")
    return out, bnd


def conv2d_wgrad_points(x: np.ndarray, dy: np.ndarray, filt_rs: Tuple[int, int], pts: np.ndarray,
                        *, pads=(0, 0, 0, 0), stride=(1, 1), dilation=(1, 1),
                        lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """dw of :func:`conv2d_wgrad` at coordinates ``pts`` (int64 [n,4]:
    k,c,r,s).  Returns (values, bound)."""
    lib = lib or load()
    x = _as_f64_view(x, "x")
    dy = _as_f64_view(dy, "dy")
    N, C, H, W = x.shape
    _, K, P, Q = dy.shape
    R, S = filt_rs
    pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 4)
    out = np.zeros(len(pts), dtype=np.float64)
    bnd = np.zeros(len(pts), dtype=np.float64)
    pt, pb, pl, pr = pads
    rc = lib.oracle_conv2d_wgrad_points(
        _ptr(x), _strides(x).ctypes.data_as(_i64p), _ptr(dy), _strides(dy).ctypes.data_as(_i64p),
        N, C, H, W, K, R, S, pt, pb, pl, pr, stride[0], stride[1], dilation[0], dilation[1],
        pts.ctypes.data_as(_i64p), len(pts), _ptr(out), _ptr(bnd))
    if rc != 0:
        raise ValueError(f"oracle_conv2d_wgrad_points returned {rc}")
    return out, bnd


POOL_MODES = {"max": 0, "avg_include_pad": 1, "avg_exclude_pad": 2}
ACT_MODES = {"identity": 0, "relu": 1, "sigmoid": 2, "tanh": 3, "clipped_relu": 4}


def pool2d_fprop(x: np.ndarray, window: Tuple[int, int], *, mode: str = "max",
                 pads=(0, 0, 0, 0), stride=(1, 1), alpha: float = 1.0, beta: float = 0.0,
                 y_in: Optional[np.ndarray] = None, lib=None) -> np.ndarray:
    """Pooling forward on an [N,C,H,W]-indexed FP64 array (any strides):
    returns y [N,C,P,Q]; ``pads`` = (top, bottom, left, right), each smaller
    than the window."""
    lib = lib or load()
    x = _as_f64_view(x, "x")
    N, C, H, W = x.shape
    R, S = window
    pt, pb, pl, pr = pads
    P = out_extent(H, pt, pb, R, 1, stride[0], lib)
    Q = out_extent(W, pl, pr, S, 1, stride[1], lib)
    if P <= 0 or Q <= 0:
        raise ValueError("empty pooling output")
    y = np.zeros((N, C, P, Q), dtype=np.float64)
    if y_in is not None:
        y_in = np.ascontiguousarray(y_in, dtype=np.float64).reshape(N, C, P, Q)
    rc = lib.oracle_pool2d_fprop(_ptr(x), _strides(x).ctypes.data_as(_i64p), _ptr(y),
                                 _strides(y).ctypes.data_as(_i64p), N, C, H, W, R, S,
                                 pt, pb, pl, pr, stride[0], stride[1], POOL_MODES[mode],
                                 float(alpha), float(beta), _ptr(y_in))
    if rc != 0:
        raise ValueError(f"oracle_pool2d_fprop returned {rc}")
    return y


def activation_fprop(x: np.ndarray, *, mode: str = "relu", coef: float = 0.0,
                     alpha: float = 1.0, beta: float = 0.0, y_in: Optional[np.ndarray] = None,
                     lib=None) -> np.ndarray:
    """Activation forward y = alpha * f(x) + beta * y_in on an [N,C,H,W]-indexed
    FP64 array (any strides); returns y [N,C,H,W]."""
    lib = lib or load()
    x = _as_f64_view(x, "x")
    N, C, H, W = x.shape
    y = np.zeros((N, C, H, W), dtype=np.float64)
    if y_in is not None:
        y_in = np.ascontiguousarray(y_in, dtype=np.float64).reshape(N, C, H, W)
    rc = lib.oracle_activation_fprop(_ptr(x), _strides(x).ctypes.data_as(_i64p), _ptr(y),
                                     _strides(y).ctypes.data_as(_i64p), N, C, H, W,
                                     ACT_MODES[mode], float(coef), float(alpha), float(beta),
                                     _ptr(y_in))
    if rc != 0:
        raise ValueError(f"oracle_activation_fprop returned {rc}")
    return y


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
