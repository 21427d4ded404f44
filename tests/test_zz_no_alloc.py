"""The allocation-free entry point, dlcConvolutionForwardNoAlloc.

It serves callers that may not allocate memory after start-up (a serving
process that reserves its memory once, a plug-in inside a framework that owns
all device memory): it takes no handle, allocates nothing, and keeps its
split-tile flags in a fixed array compiled into the library.  This test calls
it through the C ABI twice in a row and checks each result against the
handle-based dlcConvolutionForward on the same inputs, within the parity bound
the other GPU tests use.  It runs last (file name) and also passes on its own
in a fresh process, where its first call performs the per-device set-up.
"""
import numpy as np
import pytest

from deep_learning_convolution_gb300 import synth

pytestmark = pytest.mark.gpu

L = synth.Layer


@pytest.mark.parametrize("layer", [
    # 154 output tiles: at least one per SM, so the stream-K schedule and the
    # library's scratch flags are in use
    L("noalloc_bf16_c64_k64_70", 4, 64, 70, 70, 64, 3, 3, pad_top=1, pad_bottom=1, pad_left=1,
      pad_right=1),
    # 32 channels: more than the window kernel takes, so the stream-K schedule runs
    L("noalloc_tf32_nchw_c32_k32_99", 2, 32, 99, 99, 32, 3, 3, pad_top=1, pad_bottom=1,
      pad_left=1, pad_right=1, dtype="tf32", layout="NCHW"),
], ids=lambda l: l.name)
def test_no_alloc_matches_handle_path_twice(layer):
    import torch
    from deep_learning_convolution_gb300 import api
    from deep_learning_convolution_gb300 import binding as B
    from deep_learning_convolution_gb300 import build as dlc_build
    from oracle import oracle

    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    dlc_build.build()
    x, w, _ = synth.make_inputs(layer, 9090)
    xt, wt = api.layer_tensors(layer, x, w, "cuda")
    handle = api.Handle()
    conv, y_ref = api.layer_problem(handle, layer, xt, wt)
    conv(xt, wt, y_ref)
    torch.cuda.synchronize()
    handle.synchronize()

    pads = (layer.pad_top, layer.pad_bottom, layer.pad_left, layer.pad_right)
    _, bound = oracle.conv2d_fprop(x.astype(np.float64), w.astype(np.float64), pads=pads,
                                   stride=(layer.u, layer.v), dilation=(layer.dil_h, layer.dil_w))
    tol = 1e-5 * bound + 1e-6
    x_axes, _ = api.layer_axes(layer)
    ref = y_ref.permute(*[x_axes.index(a) for a in "NCHW"]).double().cpu().numpy()

    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    y = torch.empty_like(y_ref)
    stream = torch.cuda.current_stream().cuda_stream
    free_before = None
    for call in range(2):
        if call == 1:
            # after the first call's per-device set-up (which maps the module
            # holding the scratch array); the second call must take nothing
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
        y.fill_(float("nan"))
        B.dlcConvolutionForwardNoAlloc(stream, 1.0, conv.x_desc, xt.data_ptr(), conv.w_desc,
                                       wt.data_ptr(), conv.conv, 0.0, conv.y_desc, y.data_ptr(),
                                       status.data_ptr())
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0], f"call {call}: device status {status.tolist()}"
        got = y.permute(*[x_axes.index(a) for a in "NCHW"]).double().cpu().numpy()
        err = np.abs(got - ref)
        assert np.isfinite(got).all(), f"call {call}: unwritten outputs"
        assert (err <= tol).all(), f"call {call}: max err/tol {float((err / tol).max()):.3g}"
    torch.cuda.synchronize()
    # the second call allocated no device memory (allocations come in >= 2 MiB pages)
    assert torch.cuda.mem_get_info()[0] >= free_before - (1 << 20)
    conv.close()
    handle.close()


def test_no_alloc_rejects_fp32_math_and_oversize():
    import torch
    from deep_learning_convolution_gb300 import api
    from deep_learning_convolution_gb300 import binding as B

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
    # more than DLC_NOALLOC_MAX_TILES (4096) output tiles: 1x1, 1 filter tile,
    # N*P*Q = 4097 * 128 pixels
    xb = torch.zeros(4097, 128, 1, 64, dtype=torch.bfloat16, device="cuda")
    wb = torch.zeros(16, 1, 1, 64, dtype=torch.bfloat16, device="cuda")
    yb = torch.zeros(4097, 128, 1, 16, device="cuda")
    conv = api.Conv2dForward(handle, xb, wb, yb, x_axes="NHWC", w_axes="KRSC", y_axes="NHWC",
                             math="bf16")
    with pytest.raises(B.DlcError) as e:
        B.dlcConvolutionForwardNoAlloc(0, 1.0, conv.x_desc, xb.data_ptr(), conv.w_desc,
                                       wb.data_ptr(), conv.conv, 0.0, conv.y_desc, yb.data_ptr())
    assert e.value.status == B.DLC_STATUS_NOT_SUPPORTED
    torch.cuda.synchronize()
    conv.close()
    handle.close()
