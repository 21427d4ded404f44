"""GPU parity of pooling and activation forward against the CPU oracle,
through the C ABI.

Pooling: every mode (max, average counting the padding and not), NHWC
inputs on the vectorised channel kernel (BF16, FP32; a BF16 maximum
compared in stored pairs) and NCHW /
strided inputs on the per-element kernel, FP64 storage, alpha/beta, ragged extents,
asymmetric pads, an AlexNet-sized max pooling (3 x 3, stride 2 over
128 x 55 x 55 x 64 BF16) checked in full.  The maximum is exact (it selects a
stored value); an average of m terms carries FP32 rounding, bounded by
4e-6 * sum|x| / m, and the final alpha/beta combination one rounding of the
result, 1e-6 * (|ref| + |beta * y_old|) (FP64: 1e-14 in place of 1e-6).  A
BF16 output adds 2^-8 |ref|.

Activation: every mode over dense tensors (the flat vector path, including
a tail shorter than one vector and in-place calls) and strided views (the
per-element path).  The GPU evaluates exp and tanh with CUDA's float
functions; the bound 4e-7 * |ref| + 4e-7 covers their few-ulp errors at
these magnitudes.
"""
import numpy as np
import pytest

from deep_learning_convolution_gb300 import synth
from oracle import oracle

from gpu_util import assert_within

pytestmark = pytest.mark.gpu


def _need_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")


def _dev(a, dtype, axes):
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(synth.round_to_bf16_bits(a.astype(np.float32)).view(np.int16)
                             .reshape(a.shape)).view(torch.bfloat16)
    elif dtype == "f64":
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.permute(*["NCHW".index(c) for c in axes]).contiguous().cuda()


def _vals(a, dtype):
    if dtype == "f64":
        return a.astype(np.float64)
    return synth.round_values(a.astype(np.float32), "bf16" if dtype == "bf16" else "f32").astype(np.float64)


def _tdt(dtype):
    import torch
    return {"bf16": torch.bfloat16, "f32": torch.float32, "f64": torch.float64}[dtype]


POOL_CASES = [
    # name, N, C, H, W, window, pads, stride, dtype, axes, y dtype
    ("max_nhwc_bf16", 2, 64, 27, 27, (3, 3), (0, 0, 0, 0), (2, 2), "bf16", "NHWC", "bf16", "pool_nhwc"),
    ("max_nhwc_bf16_pad", 3, 24, 14, 13, (3, 3), (1, 1, 1, 0), (2, 2), "bf16", "NHWC", "f32", "pool_nhwc"),
    ("avginc_nhwc_f32", 2, 12, 11, 10, (2, 3), (1, 0, 2, 1), (2, 1), "f32", "NHWC", "f32", "pool_nhwc"),
    ("avgexc_nhwc_bf16", 2, 40, 9, 12, (3, 2), (2, 1, 0, 1), (1, 2), "bf16", "NHWC", "f32", "pool_nhwc"),
    ("max_nchw_f32", 2, 5, 13, 11, (3, 3), (1, 1, 1, 1), (2, 2), "f32", "NCHW", "f32", "direct"),
    ("avgexc_nchw_bf16", 2, 3, 12, 17, (4, 2), (3, 0, 1, 1), (3, 2), "bf16", "NCHW", "bf16", "direct"),
    ("avginc_nhwc_c3", 2, 3, 10, 10, (2, 2), (1, 1, 1, 1), (2, 2), "bf16", "NHWC", "f32", "direct"),
    ("max_nchw_f64", 2, 4, 9, 9, (3, 2), (1, 1, 1, 0), (2, 2), "f64", "NCHW", "f64", "direct"),
    ("avgexc_nhwc_f64", 1, 6, 8, 9, (3, 3), (1, 1, 1, 1), (1, 1), "f64", "NHWC", "f64", "pool_nhwc"),
    # wide rows, pads above the first output row and below the last
    ("max_nhwc_bf16_wide", 2, 64, 40, 100, (3, 3), (1, 1, 1, 1), (1, 1), "bf16", "NHWC", "bf16",
     "pool_nhwc"),
    ("avginc_nhwc_bf16_wide", 2, 64, 23, 100, (3, 3), (2, 2, 1, 0), (2, 2), "bf16", "NHWC", "f32",
     "pool_nhwc"),
    # 512 FP32 channels: 128 chunks a pixel
    ("max_nhwc_f32_wide", 1, 512, 6, 40, (3, 3), (1, 1, 1, 1), (1, 1), "f32", "NHWC", "f32",
     "pool_nhwc"),
]
MODES = {"max": "max", "avginc": "avg_include_pad", "avgexc": "avg_exclude_pad"}


def run_pool(case, seed, alpha=1.0, beta=0.0, exact=False):
    import torch
    from deep_learning_convolution_gb300 import api
    name, N, C, H, W, win, pads, stride, dt, axes, ydt, kernel = case
    mode = MODES[name.split("_")[0]]
    rng = np.random.default_rng(seed)
    x = _vals(rng.standard_normal((N, C, H, W)), dt)
    xt = _dev(x, dt, axes)
    handle = api.Handle()
    P = (H + pads[0] + pads[1] - win[0]) // stride[0] + 1
    Q = (W + pads[2] + pads[3] - win[1]) // stride[1] + 1
    yshape = [dict(N=N, C=C, H=P, W=Q)[a] for a in axes]
    y = torch.empty(yshape, dtype=_tdt(ydt), device="cuda")
    old = None
    if beta != 0.0:
        old = _vals(rng.uniform(-1, 1, (N, C, P, Q)), ydt)
        y.copy_(torch.from_numpy(old).permute(*["NCHW".index(a) for a in axes]))
    else:
        y.fill_(float("nan"))
    op = api.Pool2dForward(handle, xt, y, window=win, mode=mode, pads=pads, stride=stride,
                           x_axes=axes, y_axes=axes)
    assert op.output_dim() == (N, C, P, Q)
    assert op.kernel(xt, y) == kernel
    op(xt, y, alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    handle.synchronize()
    got = y.permute(*[axes.index(a) for a in "NCHW"]).double().cpu().numpy()
    ref = oracle.pool2d_fprop(x, win, mode=mode, pads=pads, stride=stride, alpha=alpha, beta=beta,
                              y_in=old)
    # rounding scale: the mean of |x| over the window (sum|x| / m), from the oracle
    absmean = oracle.pool2d_fprop(np.abs(x), win, mode="avg_exclude_pad", pads=pads, stride=stride)
    rel = 1e-14 if dt == "f64" else 1e-6
    tol = (0.0 if mode == "max" else rel * abs(alpha) * absmean * 4) + rel * np.abs(ref) + rel * 1e-2
    if old is not None:
        tol = tol + rel * np.abs(beta * old)
    if ydt == "bf16":
        tol = tol + 2.0 ** -8 * np.abs(ref)
    if exact:  # a maximum is one of the stored values: equal to the bit
        assert np.array_equal(got, ref), f"pool {name}: max differs from the oracle's"
    assert_within(got, ref, tol, f"pool {name}")
    op.close()
    handle.close()


@pytest.mark.parametrize("case", POOL_CASES, ids=lambda c: c[0])
def test_pooling(case):
    _need_cuda()
    run_pool(case, 900)
    run_pool(case, 901, alpha=0.5, beta=-1.5)


def test_pooling_alexnet_size_full():
    _need_cuda()
    run_pool(("max_nhwc_bf16_alex", 128, 64, 55, 55, (3, 3), (0, 0, 0, 0), (2, 2), "bf16", "NHWC",
              "bf16", "pool_nhwc"), 902, exact=True)


@pytest.mark.parametrize("case", [c for c in POOL_CASES if c[0].startswith("max") and c[8] == "bf16"],
                         ids=lambda c: c[0])
def test_max_pooling_bf16_exact(case):
    """BF16 max pooling with alpha = 1 and beta = 0 (into BF16 y the maxima
    are written back as stored, into FP32 y widened): equal to the oracle's
    maximum to the bit, padding included."""
    _need_cuda()
    run_pool(case, 903, exact=True)


def test_pooling_rejects_pad_not_smaller_than_window():
    _need_cuda()
    from deep_learning_convolution_gb300 import binding as B
    d = B.dlcCreatePoolingDescriptor()
    with pytest.raises(B.DlcError):
        B.dlcSetPooling2dDescriptor(d, B.DLC_POOLING_MAX, 2, 2, 2, 0, 0, 0, 1, 1)
    B.dlcDestroyPoolingDescriptor(d)


ACT_MODES = ["identity", "relu", "sigmoid", "tanh", "clipped_relu"]


@pytest.mark.parametrize("mode", ACT_MODES)
@pytest.mark.parametrize("dt,shape,axes,ydt", [
    ("bf16", (2, 64, 9, 7), "NHWC", "bf16"),
    ("f32", (3, 5, 7, 11), "NCHW", "f32"),      # 1155 elements: a tail below one vector
    ("bf16", (2, 3, 5, 5), "NCHW", "f32"),
    ("f64", (2, 3, 4, 5), "NCHW", "f64"),
])
def test_activation(mode, dt, shape, axes, ydt):
    import torch
    from deep_learning_convolution_gb300 import api
    _need_cuda()
    rng = np.random.default_rng(950)
    x = _vals(rng.uniform(-6, 6, shape), dt)
    xt = _dev(x, dt, axes)
    handle = api.Handle()
    for alpha, beta in ((1.0, 0.0), (0.5, 0.25)):
        y = torch.empty_like(xt, dtype=_tdt(ydt))
        old = _vals(rng.uniform(-1, 1, shape), ydt)
        y.copy_(torch.from_numpy(old).permute(*["NCHW".index(a) for a in axes]))
        api.activation_forward(handle, xt, y, mode=mode, coef=2.5, alpha=alpha, beta=beta,
                               x_axes=axes, y_axes=axes)
        torch.cuda.synchronize()
        handle.synchronize()
        got = y.permute(*[axes.index(a) for a in "NCHW"]).double().cpu().numpy()
        ref = oracle.activation_fprop(x, mode=mode, coef=2.5, alpha=alpha, beta=beta,
                                      y_in=old if beta else None)
        rel = 1e-14 if dt == "f64" else 4e-7
        tol = rel * np.abs(ref) + rel + (rel * np.abs(beta * old) if beta else 0.0)
        if ydt == "bf16":
            tol = tol + 2.0 ** -8 * np.abs(ref)
        assert_within(got, ref, tol, f"activation {mode} {dt} {axes}")
    # a strided view of x (every other W column) on the per-element path
    xv = _dev(x.repeat(2, axis=3), dt, axes)
    view = xv[..., ::2] if axes == "NCHW" else xv[:, :, ::2, :]
    yv = torch.empty(xt.shape, dtype=_tdt(ydt), device="cuda")
    api.activation_forward(handle, view, yv, mode=mode, coef=2.5, x_axes=axes, y_axes=axes)
    torch.cuda.synchronize()
    got = yv.permute(*[axes.index(a) for a in "NCHW"]).double().cpu().numpy()
    ref = oracle.activation_fprop(x, mode=mode, coef=2.5)
    rel = 1e-14 if dt == "f64" else 4e-7
    tol = rel * np.abs(ref) + rel + (2.0 ** -8 * np.abs(ref) if ydt == "bf16" else 0.0)
    assert_within(got, ref, tol, f"activation {mode} strided view")
    # in place (same tensor, same descriptor)
    if dt == ydt:
        z = xt.clone()
        api.activation_forward(handle, z, z, mode=mode, coef=2.5, x_axes=axes, y_axes=axes)
        torch.cuda.synchronize()
        got = z.permute(*[axes.index(a) for a in "NCHW"]).double().cpu().numpy()
        assert_within(got, ref, tol, f"activation {mode} in place")
    handle.close()


def test_activation_op_reused():
    """One ActivationForward object (descriptors built once) called repeatedly,
    with different alpha / beta and different tensors of the same shape."""
    import torch
    from deep_learning_convolution_gb300 import api
    _need_cuda()
    rng = np.random.default_rng(960)
    shape, axes = (2, 24, 9, 11), "NHWC"
    handle = api.Handle()
    x0 = _vals(rng.uniform(-3, 3, shape), "bf16")
    op = api.ActivationForward(handle, _dev(x0, "bf16", axes), torch.empty((2, 9, 11, 24), device="cuda"),
                               mode="clipped_relu", coef=1.5, x_axes=axes, y_axes=axes)
    try:
        for i, (alpha, beta) in enumerate(((1.0, 0.0), (-0.5, 2.0), (2.0, -1.0))):
            x = _vals(rng.uniform(-3, 3, shape), "bf16")
            xt = _dev(x, "bf16", axes)
            old = _vals(rng.uniform(-1, 1, shape), "f32")
            y = _dev(old, "f32", axes)
            op(xt, y, alpha=alpha, beta=beta)
            torch.cuda.synchronize()
            handle.synchronize()
            got = y.permute(*[axes.index(a) for a in "NCHW"]).double().cpu().numpy()
            ref = oracle.activation_fprop(x, mode="clipped_relu", coef=1.5, alpha=alpha, beta=beta,
                                          y_in=old if beta else None)
            tol = 4e-7 * np.abs(ref) + 4e-7 + (4e-7 * np.abs(beta * old) if beta else 0.0)
            assert_within(got, ref, tol, f"activation op call {i}")
    finally:
        op.close()
        handle.close()
