"""Back-to-back dependent convolutions on one stream.

The window, filter-pack and pair kernels are launched with programmatic
dependent launch: a grid may start its prologue while the grid before it is
still running, and must not touch global memory until that grid is done.
This test chains layers the way a network does -- layer B reads the output of
layer A, and a later layer A' overwrites the buffer B reads -- with no
synchronisation between the launches, and checks the results bit for bit
against the same chain run with a device synchronisation after every launch
(the kernels are deterministic).  A read of stale input, or a write that
overtakes an earlier reader, changes the bits.
"""
import pytest

pytestmark = pytest.mark.gpu


def _chain(convs, bufs, sync):
    import torch
    conv_a, conv_b, conv_a2 = convs
    x0, x0b, w1, w2, y1, y2 = bufs
    for _ in range(4):
        conv_a(x0, w1, y1)            # A: window kernel, BF16 y1
        if sync:
            torch.cuda.synchronize()
        conv_b(y1, w2, y2)            # B: pair kernel reads y1
        if sync:
            torch.cuda.synchronize()
        conv_a2(x0b, w1, y1)          # A': overwrites y1 while B may be finishing
        if sync:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return y1.clone(), y2.clone()


def test_dependent_layers_match_synchronised_chain():
    import torch
    from deep_learning_convolution_gb300 import api
    from deep_learning_convolution_gb300 import build as dlc_build

    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    dlc_build.build()
    g = torch.Generator(device="cpu").manual_seed(7070)
    n = 24
    dev = "cuda"
    x0 = torch.randn(n, 112, 112, 3, generator=g).to(torch.bfloat16).to(dev)
    x0b = torch.randn(n, 112, 112, 3, generator=g).to(torch.bfloat16).to(dev)
    w1 = (torch.randn(64, 11, 11, 3, generator=g) * 0.05).to(torch.bfloat16).to(dev)
    p = (112 + 4 - 11) // 4 + 1
    y1 = torch.empty(n, p, p, 64, dtype=torch.bfloat16, device=dev)
    w2 = (torch.randn(128, 3, 3, 64, generator=g) * 0.05).to(torch.bfloat16).to(dev)
    y2 = torch.empty(n, p, p, 128, dtype=torch.float32, device=dev)

    handle = api.Handle(torch.cuda.current_stream())
    kw = dict(x_axes="NHWC", w_axes="KRSC", y_axes="NHWC", math="bf16")
    conv_a = api.Conv2dForward(handle, x0, w1, y1, pads=(2, 2, 2, 2), stride=(4, 4), **kw)
    conv_a2 = api.Conv2dForward(handle, x0b, w1, y1, pads=(2, 2, 2, 2), stride=(4, 4), **kw)
    conv_b = api.Conv2dForward(handle, y1, w2, y2, pads=(1, 1, 1, 1), **kw)
    assert conv_a.kernel(x0, w1, y1) == "tc_window"
    assert conv_b.kernel(y1, w2, y2) == "tc_im2col_pair"

    bufs = (x0, x0b, w1, w2, y1, y2)
    ref = _chain((conv_a, conv_b, conv_a2), bufs, sync=True)
    got = _chain((conv_a, conv_b, conv_a2), bufs, sync=False)
    assert torch.isfinite(ref[1]).all()
    assert torch.equal(got[0], ref[0]), "layer A' output differs"
    assert torch.equal(got[1], ref[1]), "layer B read a stale or overwritten input"
    assert handle.last_device_error() == (0, 0)
    for c in (conv_a, conv_b, conv_a2):
        c.close()
    handle.close()
