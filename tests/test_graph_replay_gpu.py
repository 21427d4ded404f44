"""Convolution calls captured in a CUDA graph and replayed, as the benchmark's
timed passes are (seven passes in eight): every replay writes the y the CPU
oracle gives, element by element within the parity bound, and the
benchmark's helpers count the launches a capture holds.  The cases take the
SM-pair im2col kernel on a layer whose tiles all go to the split tail (its
zeroing memset and reduce-add stores are captured too), the few-channel window
kernel (its filter repack is a launch of its own) and the strict-FP32 kernel.
"""
import os
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
    # 1600 output pixels: 7 SM-pair tiles, every one split along the reduction
    # (DLC_TC_PAIR_SPLIT=2: split even where whole tiles would be as fast)
    L("graph_bf16_c64_k128_20", 4, 64, 20, 20, 128, 3, 3, pad_top=1, pad_bottom=1, pad_left=1,
      pad_right=1),
    L("graph_bf16_c3_11x11_s4", 2, 3, 63, 63, 64, 11, 11, pad_top=2, pad_bottom=2, pad_left=2,
      pad_right=2, u=4, v=4),
    L("graph_f32_nchw_c8_k16", 2, 8, 12, 12, 16, 3, 3, pad_top=1, pad_bottom=1, pad_left=1,
      pad_right=1, dtype="f32", layout="NCHW"),
]


def _check(y, x_axes, ref, tol, what):
    got = y.permute(*[x_axes.index(a) for a in "NCHW"]).double().cpu().numpy()
    assert np.isfinite(got).all(), f"{what}: unwritten outputs"
    err = np.abs(got - ref)
    assert (err <= tol).all(), f"{what}: max err/tol {float((err / tol).max()):.3g}"


@pytest.mark.parametrize("layer", CASES, ids=lambda l: l.name)
def test_replayed_passes_match_oracle(layer, monkeypatch):
    import torch
    import bench
    from deep_learning_convolution_gb300 import api
    from deep_learning_convolution_gb300 import build as dlc_build
    from oracle import oracle

    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    monkeypatch.setenv("DLC_TC_PAIR_SPLIT", "2")
    dlc_build.build()
    x, w, _ = synth.make_inputs(layer, 4242)
    ref, bound = oracle.conv2d_fprop(
        x.astype(np.float64), w.astype(np.float64),
        pads=(layer.pad_top, layer.pad_bottom, layer.pad_left, layer.pad_right),
        stride=(layer.u, layer.v), dilation=(layer.dil_h, layer.dil_w))
    tol = 1e-5 * bound + 1e-6
    x_axes, _ = api.layer_axes(layer)

    stream = torch.cuda.Stream()  # the legacy default stream cannot be captured
    with torch.cuda.stream(stream):
        xt, wt = api.layer_tensors(layer, x, w, "cuda")
        handle = api.Handle(stream)
        conv, y = api.layer_problem(handle, layer, xt, wt)
        launchers = [lambda: conv(xt, wt, y)]

        l0 = handle.launches()
        y.fill_(float("nan"))
        conv(xt, wt, y)
        per_pass = handle.launches() - l0
        stream.synchronize()
        _check(y, x_axes, ref, tol, "direct call")

        graph, per_graph = bench.capture_passes(launchers, stream, handle, bench.INST_EVERY - 1)
        assert graph is not None, "capture failed"
        assert per_graph == (bench.INST_EVERY - 1) * per_pass
        for rep in range(2):
            y.fill_(float("nan"))
            graph.replay()
            stream.synchronize()
            _check(y, x_axes, ref, tol, f"replay {rep}")

        # the benchmark's timed steps: two steps of one block of passes each
        flush = torch.empty(1 << 20, dtype=torch.float32, device="cuda")
        total_ms, per, n_inst, replays = bench.time_steps(2, bench.INST_EVERY, launchers, flush,
                                                          stream, graph)
        assert replays == 2 and n_inst == 2
        assert total_ms > 0 and per[0] > 0 and per[0] < total_ms
        stream.synchronize()
        _check(y, x_axes, ref, tol, "after the timed steps")
    handle.synchronize()  # raises if a kernel recorded a device error
    conv.close()
    handle.close()
