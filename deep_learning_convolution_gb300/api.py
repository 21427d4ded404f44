"""Descriptor marshalling for torch tensors on top of the C ABI.

Only argument marshalling: descriptor values and device pointers are read
from torch tensors and passed to the C functions in :mod:`binding`; the
convolution itself runs in ``libdlc.so``.

Axis strings name the logical meaning of a tensor's dimensions: activations
use a permutation of ``"NCHW"`` (``"NHWC"`` for channels-last storage),
filters ``"KCRS"`` or ``"KRSC"``.  Any torch strides are passed through, so
views (sub-tensors, padded rows) work where the kernel supports them.
"""
from __future__ import annotations

from typing import Optional, Sequence

from . import binding as B

MATH = {"fp32": B.DLC_MATH_FP32, "tf32": B.DLC_MATH_TF32, "bf16": B.DLC_MATH_BF16,
        "fp64": B.DLC_MATH_FP64}
MODE = {"cross_correlation": B.DLC_CROSS_CORRELATION, "convolution": B.DLC_CONVOLUTION}


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return B.DLC_DATA_FLOAT
    if t.dtype == torch.bfloat16:
        return B.DLC_DATA_BFLOAT16
    if t.dtype == torch.float64:
        return B.DLC_DATA_DOUBLE
    raise TypeError(f"unsupported dtype {t.dtype}")


def _logical(t, axes: str, order: str):
    """(sizes, strides) of tensor t in the logical axis order `order`."""
    if sorted(axes) != sorted(order) or t.dim() != 4:
        raise ValueError(f"axes {axes!r} do not describe a 4-D {order} tensor")
    sizes = [t.shape[axes.index(a)] for a in order]
    strides = [t.stride(axes.index(a)) for a in order]
    return sizes, strides


class Handle:
    """Owns a dlcHandle_t bound to the current device; follows torch's
    current stream unless a stream is given."""

    def __init__(self, stream=None):
        import torch
        self.h = B.dlcCreate()
        self.set_stream(stream if stream is not None else torch.cuda.current_stream())

    def set_stream(self, stream):
        B.dlcSetStream(self.h, int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))

    def synchronize(self):
        B.dlcSynchronize(self.h)

    def set_deterministic(self, on: bool = True):
        B.dlcSetDeterministic(self.h, 1 if on else 0)

    def launches(self) -> int:
        return B.dlcGetLaunchCount(self.h)

    def last_device_error(self):
        return B.dlcGetLastDeviceError(self.h)

    def close(self):
        if self.h is not None:
            B.dlcDestroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


class Conv2dForward:
    """Descriptors of one forward-convolution problem built from example
    tensors; calling it launches dlcConvolution(BiasActivation)Forward."""

    def __init__(self, handle: Handle, x, w, y, *, x_axes: str = "NCHW", w_axes: str = "KCRS",
                 y_axes: str = "NCHW", pads: Sequence[int] = (0, 0, 0, 0),
                 stride: Sequence[int] = (1, 1), dilation: Sequence[int] = (1, 1),
                 math: str = "bf16", mode: str = "cross_correlation"):
        self.handle = handle
        self.x_desc = B.dlcCreateTensorDescriptor()
        self.w_desc = B.dlcCreateFilterDescriptor()
        self.y_desc = B.dlcCreateTensorDescriptor()
        self.conv = B.dlcCreateConvolutionDescriptor()
        xs, xst = _logical(x, x_axes, "NCHW")
        B.dlcSetTensor4dDescriptorEx(self.x_desc, _dtype_code(x), *xs, *xst)
        if w_axes == "KCRS":
            fmt = B.DLC_TENSOR_NCHW
        elif w_axes == "KRSC":
            fmt = B.DLC_TENSOR_NHWC
        else:
            raise ValueError("filters must be KCRS or KRSC")
        if not w.is_contiguous():
            raise ValueError("filter tensors must be dense (contiguous)")
        ws, _ = _logical(w, w_axes, "KCRS")
        B.dlcSetFilter4dDescriptor(self.w_desc, _dtype_code(w), fmt, *ws)
        ys, yst = _logical(y, y_axes, "NCHW")
        B.dlcSetTensor4dDescriptorEx(self.y_desc, _dtype_code(y), *ys, *yst)
        B.dlcSetConvolution2dDescriptor(self.conv, 0, 0, int(stride[0]), int(stride[1]),
                                        int(dilation[0]), int(dilation[1]), MATH[math])
        B.dlcSetConvolution2dPadding(self.conv, *[int(p) for p in pads])
        B.dlcSetConvolutionMode(self.conv, MODE[mode])

    def output_dim(self):
        return B.dlcGetConvolution2dForwardOutputDim(self.conv, self.x_desc, self.w_desc)

    def workspace_size(self) -> int:
        return B.dlcGetConvolutionForwardWorkspaceSize(self.handle.h, self.x_desc, self.w_desc,
                                                       self.conv, self.y_desc)

    def kernel(self, x=None, w=None, y=None) -> str:
        k = B.dlcGetConvolutionForwardKernel(
            self.handle.h, self.x_desc, x.data_ptr() if x is not None else 0, self.w_desc,
            w.data_ptr() if w is not None else 0, self.conv, self.y_desc,
            y.data_ptr() if y is not None else 0)
        return B.KERNEL_NAMES[k]

    def __call__(self, x, w, y, alpha: float = 1.0, beta: float = 0.0, bias=None,
                 relu: bool = False):
        if bias is None and not relu:
            B.dlcConvolutionForward(self.handle.h, alpha, self.x_desc, x.data_ptr(), self.w_desc,
                                    w.data_ptr(), self.conv, beta, self.y_desc, y.data_ptr())
        else:
            B.dlcConvolutionBiasActivationForward(
                self.handle.h, alpha, self.x_desc, x.data_ptr(), self.w_desc, w.data_ptr(),
                self.conv, beta, bias.data_ptr() if bias is not None else 0,
                B.DLC_ACTIVATION_RELU if relu else B.DLC_ACTIVATION_IDENTITY, self.y_desc,
                y.data_ptr())
        return y

    def close(self):
        for d, f in ((self.x_desc, B.dlcDestroyTensorDescriptor),
                     (self.y_desc, B.dlcDestroyTensorDescriptor),
                     (self.w_desc, B.dlcDestroyFilterDescriptor),
                     (self.conv, B.dlcDestroyConvolutionDescriptor)):
            if d is not None:
                f(d)
        self.x_desc = self.y_desc = self.w_desc = self.conv = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class _Descriptors:
    """Tensor, filter and convolution descriptors of one problem, in the
    forward problem's terms: activations x [N,C,H,W], filters w [K,C,R,S],
    outputs y [N,K,P,Q] (the backward routines read or write their gradients
    with the same shapes)."""

    def __init__(self, x, w, y, x_axes, w_axes, y_axes, pads, stride, dilation, math, mode):
        self.x_desc = B.dlcCreateTensorDescriptor()
        self.w_desc = B.dlcCreateFilterDescriptor()
        self.y_desc = B.dlcCreateTensorDescriptor()
        self.conv = B.dlcCreateConvolutionDescriptor()
        xs, xst = _logical(x, x_axes, "NCHW")
        B.dlcSetTensor4dDescriptorEx(self.x_desc, _dtype_code(x), *xs, *xst)
        if w_axes not in ("KCRS", "KRSC"):
            raise ValueError("filters must be KCRS or KRSC")
        if not w.is_contiguous():
            raise ValueError("filter tensors must be dense (contiguous)")
        ws, _ = _logical(w, w_axes, "KCRS")
        B.dlcSetFilter4dDescriptor(self.w_desc, _dtype_code(w),
                                   B.DLC_TENSOR_NCHW if w_axes == "KCRS" else B.DLC_TENSOR_NHWC, *ws)
        ys, yst = _logical(y, y_axes, "NCHW")
        B.dlcSetTensor4dDescriptorEx(self.y_desc, _dtype_code(y), *ys, *yst)
        B.dlcSetConvolution2dDescriptor(self.conv, 0, 0, int(stride[0]), int(stride[1]),
                                        int(dilation[0]), int(dilation[1]), MATH[math])
        B.dlcSetConvolution2dPadding(self.conv, *[int(p) for p in pads])
        B.dlcSetConvolutionMode(self.conv, MODE[mode])

    def close(self):
        for d, f in ((self.x_desc, B.dlcDestroyTensorDescriptor),
                     (self.y_desc, B.dlcDestroyTensorDescriptor),
                     (self.w_desc, B.dlcDestroyFilterDescriptor),
                     (self.conv, B.dlcDestroyConvolutionDescriptor)):
            if d is not None:
                f(d)
        self.x_desc = self.y_desc = self.w_desc = self.conv = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Conv2dBackwardData(_Descriptors):
    """dx = alpha * dgrad(w, dy) + beta * dx through dlcConvolutionBackwardData;
    built from example tensors w [K,C,R,S], dy [N,K,P,Q] and dx [N,C,H,W]."""

    def __init__(self, handle: Handle, w, dy, dx, *, w_axes="KCRS", dy_axes="NCHW",
                 dx_axes="NCHW", pads=(0, 0, 0, 0), stride=(1, 1), dilation=(1, 1),
                 math="bf16", mode="cross_correlation"):
        self.handle = handle
        super().__init__(dx, w, dy, dx_axes, w_axes, dy_axes, pads, stride, dilation, math, mode)

    def kernel(self, w=None, dy=None, dx=None) -> str:
        k = B.dlcGetConvolutionBackwardDataKernel(
            self.handle.h, self.w_desc, w.data_ptr() if w is not None else 0, self.y_desc,
            dy.data_ptr() if dy is not None else 0, self.conv, self.x_desc,
            dx.data_ptr() if dx is not None else 0)
        return B.KERNEL_NAMES[k]

    def workspace_size(self) -> int:
        return B.dlcGetConvolutionBackwardDataWorkspaceSize(self.handle.h, self.w_desc, self.y_desc,
                                                            self.conv, self.x_desc)

    def __call__(self, w, dy, dx, alpha: float = 1.0, beta: float = 0.0):
        B.dlcConvolutionBackwardData(self.handle.h, alpha, self.w_desc, w.data_ptr(), self.y_desc,
                                     dy.data_ptr(), self.conv, beta, self.x_desc, dx.data_ptr())
        return dx


class Conv2dBackwardFilter(_Descriptors):
    """dw = alpha * wgrad(x, dy) + beta * dw through dlcConvolutionBackwardFilter;
    built from example tensors x [N,C,H,W], dy [N,K,P,Q] and dw [K,C,R,S]."""

    def __init__(self, handle: Handle, x, dy, dw, *, x_axes="NCHW", dy_axes="NCHW",
                 dw_axes="KCRS", pads=(0, 0, 0, 0), stride=(1, 1), dilation=(1, 1),
                 math="bf16", mode="cross_correlation"):
        self.handle = handle
        super().__init__(x, dw, dy, x_axes, dw_axes, dy_axes, pads, stride, dilation, math, mode)

    def kernel(self, x=None, dy=None, dw=None) -> str:
        k = B.dlcGetConvolutionBackwardFilterKernel(
            self.handle.h, self.x_desc, x.data_ptr() if x is not None else 0, self.y_desc,
            dy.data_ptr() if dy is not None else 0, self.conv, self.w_desc,
            dw.data_ptr() if dw is not None else 0)
        return B.KERNEL_NAMES[k]

    def workspace_size(self) -> int:
        return B.dlcGetConvolutionBackwardFilterWorkspaceSize(self.handle.h, self.x_desc,
                                                              self.y_desc, self.conv, self.w_desc)

    def __call__(self, x, dy, dw, alpha: float = 1.0, beta: float = 0.0):
        B.dlcConvolutionBackwardFilter(self.handle.h, alpha, self.x_desc, x.data_ptr(), self.y_desc,
                                       dy.data_ptr(), self.conv, beta, self.w_desc, dw.data_ptr())
        return dw


POOL_MODES = {"max": B.DLC_POOLING_MAX, "avg_include_pad": B.DLC_POOLING_AVERAGE_COUNT_INCLUDE_PADDING,
              "avg_exclude_pad": B.DLC_POOLING_AVERAGE_COUNT_EXCLUDE_PADDING}
ACT_MODES = {"identity": B.DLC_ACTIVATION_IDENTITY, "relu": B.DLC_ACTIVATION_RELU,
             "sigmoid": B.DLC_ACTIVATION_SIGMOID, "tanh": B.DLC_ACTIVATION_TANH,
             "clipped_relu": B.DLC_ACTIVATION_CLIPPED_RELU}


class Pool2dForward:
    """y = alpha * pool(x) + beta * y through dlcPoolingForward."""

    def __init__(self, handle: Handle, x, y, *, window=(2, 2), mode="max", pads=(0, 0, 0, 0),
                 stride=(2, 2), x_axes="NCHW", y_axes="NCHW"):
        self.handle = handle
        self.pool = B.dlcCreatePoolingDescriptor()
        B.dlcSetPooling2dDescriptor(self.pool, POOL_MODES[mode], window[0], window[1], *pads,
                                    stride[0], stride[1])
        self.x_desc = B.dlcCreateTensorDescriptor()
        self.y_desc = B.dlcCreateTensorDescriptor()
        xs, xst = _logical(x, x_axes, "NCHW")
        B.dlcSetTensor4dDescriptorEx(self.x_desc, _dtype_code(x), *xs, *xst)
        ys, yst = _logical(y, y_axes, "NCHW")
        B.dlcSetTensor4dDescriptorEx(self.y_desc, _dtype_code(y), *ys, *yst)

    def output_dim(self):
        return B.dlcGetPooling2dForwardOutputDim(self.pool, self.x_desc)

    def kernel(self, x=None, y=None) -> str:
        return B.KERNEL_NAMES[B.dlcGetPoolingForwardKernel(
            self.handle.h, self.pool, self.x_desc, x.data_ptr() if x is not None else 0,
            self.y_desc, y.data_ptr() if y is not None else 0)]

    def __call__(self, x, y, alpha: float = 1.0, beta: float = 0.0):
        B.dlcPoolingForward(self.handle.h, self.pool, alpha, self.x_desc, x.data_ptr(), beta,
                            self.y_desc, y.data_ptr())
        return y

    def close(self):
        if self.pool is not None:
            B.dlcDestroyPoolingDescriptor(self.pool)
            B.dlcDestroyTensorDescriptor(self.x_desc)
            B.dlcDestroyTensorDescriptor(self.y_desc)
            self.pool = None


class ActivationForward:
    """y = alpha * f(x) + beta * y through dlcActivationForward (y may be x),
    with the tensor descriptors built once for repeated calls on the same
    shapes and layouts."""

    def __init__(self, handle: Handle, x, y, *, mode="relu", coef=0.0, x_axes="NCHW",
                 y_axes="NCHW"):
        self.handle = handle
        self.mode = ACT_MODES[mode]
        self.coef = float(coef)
        self.x_desc = B.dlcCreateTensorDescriptor()
        self.y_desc = B.dlcCreateTensorDescriptor()
        xs, xst = _logical(x, x_axes, "NCHW")
        B.dlcSetTensor4dDescriptorEx(self.x_desc, _dtype_code(x), *xs, *xst)
        ys, yst = _logical(y, y_axes, "NCHW")
        B.dlcSetTensor4dDescriptorEx(self.y_desc, _dtype_code(y), *ys, *yst)

    def __call__(self, x, y, alpha: float = 1.0, beta: float = 0.0):
        B.dlcActivationForward(self.handle.h, self.mode, self.coef, alpha, self.x_desc, x.data_ptr(),
                               beta, self.y_desc, y.data_ptr())
        return y

    def close(self):
        if self.x_desc is not None:
            B.dlcDestroyTensorDescriptor(self.x_desc)
            B.dlcDestroyTensorDescriptor(self.y_desc)
            self.x_desc = None


def activation_forward(handle: Handle, x, y, *, mode="relu", coef=0.0, alpha=1.0, beta=0.0,
                       x_axes="NCHW", y_axes="NCHW"):
    """y = alpha * f(x) + beta * y through dlcActivationForward (y may be x):
    one call of ActivationForward, its descriptors built and destroyed here."""
    op = ActivationForward(handle, x, y, mode=mode, coef=coef, x_axes=x_axes, y_axes=y_axes)
    try:
        return op(x, y, alpha=alpha, beta=beta)
    finally:
        op.close()


def output_dim(x, w, *, x_axes="NCHW", w_axes="KCRS", pads=(0, 0, 0, 0), stride=(1, 1),
               dilation=(1, 1)):
    """(N, K, P, Q) from the library's descriptor call (no GPU work)."""
    xd = B.dlcCreateTensorDescriptor()
    wd = B.dlcCreateFilterDescriptor()
    cd = B.dlcCreateConvolutionDescriptor()
    try:
        xs, xst = _logical(x, x_axes, "NCHW")
        B.dlcSetTensor4dDescriptorEx(xd, _dtype_code(x), *xs, *xst)
        ws, _ = _logical(w, w_axes, "KCRS")
        B.dlcSetFilter4dDescriptor(wd, _dtype_code(w),
                                   B.DLC_TENSOR_NCHW if w_axes == "KCRS" else B.DLC_TENSOR_NHWC, *ws)
        B.dlcSetConvolution2dDescriptor(cd, 0, 0, int(stride[0]), int(stride[1]),
                                        int(dilation[0]), int(dilation[1]), B.DLC_MATH_FP32)
        B.dlcSetConvolution2dPadding(cd, *[int(p) for p in pads])
        return B.dlcGetConvolution2dForwardOutputDim(cd, xd, wd)
    finally:
        B.dlcDestroyTensorDescriptor(xd)
        B.dlcDestroyFilterDescriptor(wd)
        B.dlcDestroyConvolutionDescriptor(cd)


def layer_axes(layer):
    """(x_axes, w_axes) of a synth.Layer's storage layout."""
    return ("NHWC", "KRSC") if layer.layout == "NHWC" else ("NCHW", "KCRS")


def layer_tensors(layer, x_nchw, w_kcrs, device):
    """Device tensors x and w for a synth.Layer from logical-NCHW / KCRS numpy
    arrays (already rounded), stored in the layer's layout (dense)."""
    import numpy as np
    import torch
    from . import synth
    if layer.dtype == "bf16":
        xb = synth.round_to_bf16_bits(x_nchw).view(np.int16).reshape(x_nchw.shape)
        wb = synth.round_to_bf16_bits(w_kcrs).view(np.int16).reshape(w_kcrs.shape)
        xt = torch.from_numpy(xb).view(torch.bfloat16)
        wt = torch.from_numpy(wb).view(torch.bfloat16)
    else:
        xt = torch.from_numpy(np.ascontiguousarray(x_nchw, dtype=np.float32))
        wt = torch.from_numpy(np.ascontiguousarray(w_kcrs, dtype=np.float32))
    if layer.layout == "NHWC":
        xt = xt.permute(0, 2, 3, 1)
        wt = wt.permute(0, 2, 3, 1)
    return xt.contiguous().to(device), wt.contiguous().to(device)


def layer_problem(handle, layer, xt, wt, y_dtype=None, y_axes=None):
    """A Conv2dForward for a synth.Layer plus its freshly allocated y
    (FP32 by default, in the layer's layout unless y_axes is given)."""
    import torch
    x_axes, w_axes = layer_axes(layer)
    pads = (layer.pad_top, layer.pad_bottom, layer.pad_left, layer.pad_right)
    stride, dil = (layer.u, layer.v), (layer.dil_h, layer.dil_w)
    n, k, p, q = output_dim(xt, wt, x_axes=x_axes, w_axes=w_axes, pads=pads, stride=stride,
                            dilation=dil)
    y_axes = y_axes or x_axes
    shape = [dict(N=n, C=k, H=p, W=q)[a] for a in y_axes]
    y = torch.empty(shape, dtype=y_dtype or torch.float32, device=xt.device)
    conv = Conv2dForward(handle, xt, wt, y, x_axes=x_axes, w_axes=w_axes, y_axes=y_axes,
                         pads=pads, stride=stride, dilation=dil, math=math_of(layer))
    return conv, y


def math_of(layer) -> str:
    return {"bf16": "bf16", "tf32": "tf32", "f32": "fp32"}[layer.dtype]
