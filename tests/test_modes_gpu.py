"""Convolution mode (mirrored filter taps) and FP64 math of the forward call,
through the C ABI, against the CPU oracle.

Convolution mode computes y[n,k,p,q] = sum x[...] * w[k,c,R-1-r,S-1-s]: the
oracle runs on the mirrored filters.  Each forward kernel is covered: the
SM-pair kernel (mirrored filter-load coordinates), the window kernel and the
gather kernel (a mirrored strided view of the filters) and the FFMA kernel.
FP64 math runs the direct kernel on DOUBLE storage and must agree with the
FP64 oracle to 1e-12 of sum|x*w|.
"""
import numpy as np
import pytest

from deep_learning_convolution_gb300 import synth
from oracle import oracle

from gpu_util import run_and_check, assert_within

pytestmark = pytest.mark.gpu

L = synth.Layer
P1 = dict(pad_top=1, pad_bottom=1, pad_left=1, pad_right=1)

MODE_CASES = [
    (L("cm_pair_c64_k96_5x3", 2, 64, 17, 15, 96, 5, 3, pad_top=2, pad_bottom=1, pad_left=1,
       pad_right=0), "tc_im2col_pair"),
    (L("cm_window_c3_11x11_s4", 2, 3, 47, 47, 64, 11, 11, pad_top=2, pad_bottom=2, pad_left=2,
       pad_right=2, u=4, v=4), "tc_window"),
    # more than 64 filters: past the row-stack kernel's limit
    (L("cm_gather_tf32_nchw_c32", 2, 32, 13, 11, 72, 3, 5, **P1, dtype="tf32", layout="NCHW"),
     "tc_gather"),
    (L("cm_rowstack_tf32_nchw_c32", 2, 32, 13, 11, 40, 3, 5, **P1, dtype="tf32", layout="NCHW"),
     "tc_rowstack"),
    (L("cm_ffma_nchw", 2, 8, 16, 16, 16, 3, 3, **P1, dtype="f32", layout="NCHW"), "ffma"),
]


@pytest.mark.parametrize("layer,kernel", MODE_CASES, ids=lambda v: getattr(v, "name", v))
def test_convolution_mode(layer, kernel):
    import torch
    from deep_learning_convolution_gb300 import api
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    handle = api.Handle()
    got = run_and_check(handle, layer, 808, mode="convolution", expect_kernel=kernel, full=True)
    # the same call with bias, ReLU and beta
    run_and_check(handle, layer, 809, mode="convolution", expect_kernel=kernel, full=True,
                  alpha=0.5, beta=0.25, with_bias=True, relu=True)
    handle.close()
    assert got == kernel


@pytest.mark.parametrize("y_axes", ["NCHW", "NHWC"])
def test_fp64_forward(y_axes):
    import torch
    from deep_learning_convolution_gb300 import api
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    rng = np.random.default_rng(64)
    N, C, H, W, K, R, S = 2, 5, 13, 11, 7, 3, 4
    pads, stride, dil = (1, 2, 0, 2), (2, 1), (1, 2)
    x = rng.uniform(-1, 1, (N, C, H, W))
    w = rng.uniform(-1, 1, (K, C, R, S))
    ref, bound = oracle.conv2d_fprop(x, w, pads=pads, stride=stride, dilation=dil)
    handle = api.Handle()
    xt = torch.from_numpy(x).cuda()
    wt = torch.from_numpy(w).cuda()
    shape = [dict(N=N, C=K, H=ref.shape[2], W=ref.shape[3])[a] for a in y_axes]
    y = torch.full(shape, float("nan"), dtype=torch.float64, device="cuda")
    conv = api.Conv2dForward(handle, xt, wt, y, y_axes=y_axes, pads=pads, stride=stride,
                             dilation=dil, math="fp64")
    assert conv.kernel(xt, wt, y) == "ffma"
    conv(xt, wt, y)
    torch.cuda.synchronize()
    handle.synchronize()
    got = y.permute(*[y_axes.index(a) for a in "NCHW"]).cpu().numpy()
    assert_within(got, ref, 1e-12 * bound + 1e-300, "fp64 forward")
    # float storage is refused for FP64 math, double storage for the others
    xf = xt.float()
    with pytest.raises(Exception):
        api.Conv2dForward(handle, xf, wt.float(), y, y_axes=y_axes, pads=pads, stride=stride,
                          dilation=dil, math="fp64")(xf, wt.float(), y)
    conv.close()
    handle.close()
