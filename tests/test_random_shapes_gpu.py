"""GPU parity on seeded random layer shapes, each checked in full against the
CPU oracle through the C ABI with the library's own kernel choice.

The shapes are drawn from a fixed seed (so every run checks the same cases):
batch 1-3, 1-160 channels, 5-30 pixels a side, 1-200 filters, windows up to
7 x 7, strides 1-3, dilation 1-2, any pads below the dilated window, BF16
NHWC (the tensor-core kernels), TF32 NCHW and NHWC, and strict FP32 NCHW.
The oracle's work per case is bounded (at most 4e7 multiply-adds), so the
set runs in seconds; the bound the comparison uses is the oracle's own
(the same one every parity test uses).
"""
import numpy as np
import pytest

from deep_learning_convolution_gb300 import synth
from gpu_util import run_and_check

pytestmark = pytest.mark.gpu

KINDS = [("bf16", "NHWC")] * 5 + [("tf32", "NCHW"), ("tf32", "NHWC"), ("f32", "NCHW")]
MAX_MACS = 40_000_000


def _draw(rng, i):
    """One random layer whose output is non-empty and whose oracle cost is bounded."""
    dtype, layout = KINDS[int(rng.integers(len(KINDS)))]
    while True:
        N = int(rng.integers(1, 4))
        C = int(rng.choice([1, 3, 8, 16, 24, 32, 40, 64, 72, 96, 128, 136, 160]))
        H, W = int(rng.integers(5, 31)), int(rng.integers(5, 31))
        K = int(rng.choice([1, 8, 16, 24, 32, 48, 64, 96, 100, 128, 130, 192, 200]))
        R, S = int(rng.integers(1, 8)), int(rng.integers(1, 8))
        u, v = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        dh = int(rng.integers(1, 3)) if R > 1 and rng.random() < 0.25 else 1
        dw = int(rng.integers(1, 3)) if S > 1 and rng.random() < 0.25 else 1
        er, es = (R - 1) * dh + 1, (S - 1) * dw + 1
        pads = [int(rng.integers(0, er)), int(rng.integers(0, er)),
                int(rng.integers(0, es)), int(rng.integers(0, es))]
        P = (H + pads[0] + pads[1] - er) // u + 1
        Q = (W + pads[2] + pads[3] - es) // v + 1
        if P < 1 or Q < 1:
            continue
        if N * K * P * Q * C * R * S > MAX_MACS:
            continue
        return synth.Layer(f"rand{i:02d}_{dtype}_{layout}_c{C}_k{K}_{R}x{S}_s{u}x{v}", N, C, H, W, K,
                           R, S, pad_top=pads[0], pad_bottom=pads[1], pad_left=pads[2],
                           pad_right=pads[3], u=u, v=v, dil_h=dh, dil_w=dw, dtype=dtype,
                           layout=layout)


def _cases(n=32, seed=20261203):
    rng = np.random.default_rng(seed)
    return [_draw(rng, i) for i in range(n)]


CASES = _cases()


@pytest.fixture(scope="module")
def handle():
    import torch
    from deep_learning_convolution_gb300 import api
    from deep_learning_convolution_gb300 import build as dlc_build
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    dlc_build.build()
    h = api.Handle()
    yield h
    h.close()


CHOSEN = {}  # case name -> the kernel the library chose


@pytest.mark.parametrize("layer", CASES, ids=lambda l: l.name)
def test_random_shape_parity(handle, layer):
    seed = 5000 + CASES.index(layer)
    CHOSEN[layer.name] = run_and_check(handle, layer, seed, full=True)
    # the epilogue's other branches on the same shape
    run_and_check(handle, layer, seed + 100, full=True, alpha=0.5, beta=-0.75, with_bias=True,
                  relu=True)


def test_random_shapes_reach_the_tensor_core_kernels():
    """The random set is not all fallbacks: it ran the SM-pair kernel and the
    direct FP32 kernel at least (read from the parity runs above)."""
    if len(CHOSEN) < len(CASES):
        pytest.skip("needs every random-shape parity case run first")
    kinds = set(CHOSEN.values())
    print("kernels chosen for the random shapes:", sorted(kinds))
    assert "tc_im2col_pair" in kinds and "ffma" in kinds, sorted(kinds)


# The backward routines on the BF16 NHWC random shapes (the tensor-core data-
# and filter-gradient kernels where they apply, the direct kernels elsewhere),
# against the oracle's dgrad and wgrad in full.
BWD_CASES = [l for l in CASES if l.dtype == "bf16"][:10]


@pytest.mark.parametrize("layer", BWD_CASES, ids=lambda l: l.name)
def test_random_shape_backward(layer):
    from test_backward_gpu import run_dgrad, run_wgrad
    seed = 6000 + BWD_CASES.index(layer)
    run_dgrad(layer, seed, full=True)
    run_wgrad(layer, seed + 1, full=True)
    run_wgrad(layer, seed + 2, full=True, alpha=0.75, beta=0.5)
