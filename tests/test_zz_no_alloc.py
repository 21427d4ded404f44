"""The allocation-free entry point, dlcConvolutionForwardNoAlloc.

It serves callers that may not allocate memory after start-up (a serving
process that reserves its memory once, a plug-in inside a framework that owns
all device memory): it takes no handle, allocates nothing, and keeps its
scratch (the few-channel kernel's repacked filters, split-tile flags, error
words) in fixed arrays compiled into the library.  These tests call it
through the C ABI twice in a row and check each result element by element
against the CPU oracle, within the parity bound the other GPU tests use; the
cases cover the SM-pair im2col kernel, the TF32 run-gather kernel and the
few-channel window kernel (whose filter image lives in the fixed array), with
beta = 0 and beta != 0.  A separate fresh process checks that, once the first
call has set the device up, a call that reaches a kernel not launched before
allocates no device memory.  The file runs last (its name) and also passes on
its own in a fresh process, where its first call performs the set-up.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from deep_learning_convolution_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

L = synth.Layer

CASES = [
    # 154 output tiles on the SM-pair im2col kernel
    L("noalloc_bf16_c64_k64_70", 4, 64, 70, 70, 64, 3, 3, pad_top=1, pad_bottom=1, pad_left=1,
      pad_right=1),
    # 32 channels, TF32, NCHW: the row-stack kernel (its filter slices in the
    # fixed array)
    L("noalloc_tf32_nchw_c32_k32_99", 2, 32, 99, 99, 32, 3, 3, pad_top=1, pad_bottom=1,
      pad_left=1, pad_right=1, dtype="tf32", layout="NCHW"),
    # a first layer (3 channels, 11x11, stride 4): the window kernel, whose
    # repacked filter image lives in the library's fixed array
    L("noalloc_bf16_c3_11x11_s4", 2, 3, 63, 63, 64, 11, 11, pad_top=2, pad_bottom=2, pad_left=2,
      pad_right=2, u=4, v=4),
]


def _oracle(layer, x, w, y_in=None, beta=0.0):
    from oracle import oracle
    pads = (layer.pad_top, layer.pad_bottom, layer.pad_left, layer.pad_right)
    return oracle.conv2d_fprop(x.astype(np.float64), w.astype(np.float64), pads=pads,
                               stride=(layer.u, layer.v), dilation=(layer.dil_h, layer.dil_w),
                               beta=beta, y_in=y_in)


@pytest.mark.parametrize("beta", [0.0, 0.5], ids=["beta0", "beta0.5"])
@pytest.mark.parametrize("layer", CASES, ids=lambda l: l.name)
def test_no_alloc_matches_oracle_twice(layer, beta):
    import torch
    from deep_learning_convolution_gb300 import api
    from deep_learning_convolution_gb300 import binding as B
    from deep_learning_convolution_gb300 import build as dlc_build

    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    dlc_build.build()
    x, w, _ = synth.make_inputs(layer, 9090)
    xt, wt = api.layer_tensors(layer, x, w, "cuda")
    handle = api.Handle()
    conv, y = api.layer_problem(handle, layer, xt, wt)
    x_axes, _ = api.layer_axes(layer)
    to_nchw = [x_axes.index(a) for a in "NCHW"]
    n, k, p, q = conv.output_dim()
    y_in = None
    if beta != 0.0:
        y_in = np.random.default_rng(77).uniform(-1, 1, size=(n, k, p, q))
    ref, bound = _oracle(layer, x, w, y_in=y_in, beta=beta)
    tol = 1e-5 * bound + 1e-6
    if y_in is not None:
        tol = tol + 1e-6 * np.abs(beta * y_in)

    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    free_before = None
    for call in range(2):
        if call == 1:
            # after the first call's per-device set-up; the second call must
            # take nothing
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
        if y_in is None:
            y.fill_(float("nan"))  # beta == 0: every output must be written
        else:
            y.copy_(torch.from_numpy(y_in.astype(np.float32)).permute(
                *["NCHW".index(a) for a in x_axes]))
        B.dlcConvolutionForwardNoAlloc(stream, 1.0, conv.x_desc, xt.data_ptr(), conv.w_desc,
                                       wt.data_ptr(), conv.conv, beta, conv.y_desc, y.data_ptr(),
                                       status.data_ptr())
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0], f"call {call}: device status {status.tolist()}"
        got = y.permute(*to_nchw).double().cpu().numpy()
        err = np.abs(got - ref)
        assert np.isfinite(got).all(), f"call {call}: unwritten outputs"
        assert (err <= tol).all(), f"call {call}: max err/tol {float((err / tol).max()):.3g}"
    torch.cuda.synchronize()
    # the second call allocated no device memory (allocations come in >= 2 MiB pages)
    assert torch.cuda.mem_get_info()[0] >= free_before - (1 << 20)
    conv.close()
    handle.close()


def test_no_alloc_rejects_fp32_math_and_runs_many_tiles():
    import torch
    from deep_learning_convolution_gb300 import api
    from deep_learning_convolution_gb300 import binding as B
    from oracle import oracle

    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    handle = api.Handle()
    x = torch.zeros(1, 8, 9, 9, device="cuda")
    w = torch.zeros(4, 8, 3, 3, device="cuda")
    y = torch.zeros(1, 4, 7, 7, device="cuda")
    conv = api.Conv2dForward(handle, x, w, y, math="fp32")
    with pytest.raises(B.DlcError) as e:
        B.dlcConvolutionForwardNoAlloc(0, 1.0, conv.x_desc, x.data_ptr(), conv.w_desc,
                                       w.data_ptr(), conv.conv, 0.0, conv.y_desc, y.data_ptr())
    assert e.value.status == B.DLC_STATUS_NOT_SUPPORTED
    conv.close()
    # more output tiles (4097 x 128 pixels) than the fixed array has split-tile
    # flags: runs whole tiles, checked on sampled outputs
    layer = L("noalloc_many_tiles_1x1", 4097, 64, 1, 128, 16, 1, 1)
    xh, wh, _ = synth.make_inputs(layer, 4242)
    xb, wb = api.layer_tensors(layer, xh, wh, "cuda")
    conv, yb = api.layer_problem(handle, layer, xb, wb)
    yb.fill_(float("nan"))
    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        B.dlcConvolutionForwardNoAlloc(0, 1.0, conv.x_desc, xb.data_ptr(), conv.w_desc,
                                       wb.data_ptr(), conv.conv, 0.0, conv.y_desc, yb.data_ptr(),
                                       status.data_ptr())
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0]
    got = yb.permute(0, 3, 1, 2).double().cpu().numpy()
    assert np.isfinite(got).all()
    rng = np.random.default_rng(5)
    pts = np.stack([rng.integers(0, 4097, 4096), rng.integers(0, 16, 4096),
                    np.zeros(4096, np.int64), rng.integers(0, 128, 4096)], axis=1)
    vals, bnd = oracle.conv2d_fprop_points(xh.astype(np.float64), wh.astype(np.float64), pts)
    err = np.abs(got[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]] - vals)
    assert (err <= 1e-5 * bnd + 1e-6).all()
    conv.close()
    handle.close()


def _fresh_process_body():
    """Runs in a fresh process: the first call (pair kernel) sets the device
    up; a later first call of the window kernel must not allocate."""
    import torch
    from deep_learning_convolution_gb300 import api
    from deep_learning_convolution_gb300 import binding as B
    from deep_learning_convolution_gb300 import build as dlc_build
    dlc_build.build()
    torch.cuda.init()
    handle = api.Handle()
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    probs = []
    for layer in (CASES[0], CASES[2]):
        x, w, _ = synth.make_inputs(layer, 31)
        xt, wt = api.layer_tensors(layer, x, w, "cuda")
        conv, y = api.layer_problem(handle, layer, xt, wt)
        probs.append((conv, xt, wt, y))
    torch.cuda.synchronize()
    free = []
    for conv, xt, wt, y in probs:
        B.dlcConvolutionForwardNoAlloc(0, 1.0, conv.x_desc, xt.data_ptr(), conv.w_desc,
                                       wt.data_ptr(), conv.conv, 0.0, conv.y_desc, y.data_ptr(),
                                       status.data_ptr())
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0]
        free.append(torch.cuda.mem_get_info()[0])
    kernels = [c.kernel(xt, wt, y) for c, xt, wt, y in probs]
    assert kernels == ["tc_im2col_pair", "tc_window"], kernels
    # the window kernel's first launch (after the pair kernel's) took no memory
    assert free[1] >= free[0] - (1 << 20), f"free memory fell by {free[0] - free[1]} bytes"
    print("fresh-process no-alloc ok")


def test_no_alloc_later_kernels_allocate_nothing_fresh_process():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    r = subprocess.run([sys.executable, os.path.abspath(__file__)], capture_output=True,
                       text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0 and "fresh-process no-alloc ok" in r.stdout, r.stdout + r.stderr


if __name__ == "__main__":
    _fresh_process_body()
