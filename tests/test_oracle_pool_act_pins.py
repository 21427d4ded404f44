"""Pins of the oracle's pooling and activation definitions.

Each is checked against something other than itself:
  * max pooling against numpy's sliding-window view of the input padded with
    -inf (a different formulation of "the largest in-image value");
  * average pooling against torch's avg_pool2d in FP64 (an independent
    library), counting the padding (count_include_pad=True) and not
    (False); the asymmetric padding is applied explicitly;
  * a hand-worked 4 x 4 example for every mode;
  * activations against numpy's closed forms and at special values
    (sigmoid(0) = 1/2, tanh(0) = 0, odd symmetry of tanh, sigmoid(x) +
    sigmoid(-x) = 1, the clipped ReLU's ceiling);
  * layout independence (an NHWC-stored input gives the same values);
  * planted mistakes in copies of the oracle, each caught here.
"""
import os
import shutil
import tempfile

import numpy as np
import pytest

from oracle import oracle

CASES = [
    # N, C, H, W, R, S, pads, stride
    (2, 3, 9, 11, 3, 3, (1, 1, 1, 1), (2, 2)),
    (1, 2, 8, 7, 2, 3, (0, 1, 2, 0), (2, 1)),
    (2, 1, 13, 13, 3, 2, (2, 0, 1, 1), (3, 2)),
    (1, 4, 6, 6, 2, 2, (0, 0, 0, 0), (2, 2)),
]


def _sliding_max(x, R, S, pads, stride):
    pt, pb, pl, pr = pads
    xp = np.pad(x, ((0, 0), (0, 0), (pt, pb), (pl, pr)), constant_values=-np.inf)
    win = np.lib.stride_tricks.sliding_window_view(xp, (R, S), axis=(2, 3))
    return win[:, :, ::stride[0], ::stride[1]].max(axis=(-2, -1))


def _torch_avg(x, R, S, pads, stride, include):
    import torch
    import torch.nn.functional as F
    pt, pb, pl, pr = pads
    xt = torch.from_numpy(x)
    if include:
        xp = F.pad(xt, (pl, pr, pt, pb))
        return F.avg_pool2d(xp, (R, S), stride=stride).numpy()
    ones = torch.ones_like(xt)
    s = F.avg_pool2d(F.pad(xt, (pl, pr, pt, pb)), (R, S), stride=stride, divisor_override=1)
    n = F.avg_pool2d(F.pad(ones, (pl, pr, pt, pb)), (R, S), stride=stride, divisor_override=1)
    return (s / n).numpy()


def check_max(lib):
    rng = np.random.default_rng(1)
    for N, C, H, W, R, S, pads, stride in CASES:
        x = rng.uniform(-1, 1, (N, C, H, W))
        y = oracle.pool2d_fprop(x, (R, S), mode="max", pads=pads, stride=stride, lib=lib)
        ref = _sliding_max(x, R, S, pads, stride)
        assert y.shape == ref.shape and np.array_equal(y, ref)


def check_avg(lib):
    rng = np.random.default_rng(2)
    for N, C, H, W, R, S, pads, stride in CASES:
        x = rng.uniform(-1, 1, (N, C, H, W))
        for mode, inc in (("avg_include_pad", True), ("avg_exclude_pad", False)):
            y = oracle.pool2d_fprop(x, (R, S), mode=mode, pads=pads, stride=stride, lib=lib)
            ref = _torch_avg(x, R, S, pads, stride, inc)
            assert y.shape == ref.shape
            np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-15)


def check_hand_worked(lib):
    x = np.arange(16, dtype=np.float64).reshape(1, 1, 4, 4)
    # 2x2 windows, stride 2, no padding: maxima 5, 7, 13, 15; means 2.5, 4.5, 10.5, 12.5
    assert np.array_equal(oracle.pool2d_fprop(x, (2, 2), stride=(2, 2), lib=lib)[0, 0],
                          [[5, 7], [13, 15]])
    assert np.array_equal(oracle.pool2d_fprop(x, (2, 2), mode="avg_include_pad", stride=(2, 2),
                                              lib=lib)[0, 0], [[2.5, 4.5], [10.5, 12.5]])
    # 2x2 windows, stride 2, top/left pad 1: the corner window holds x[0,0] = 0
    # alone (include: 0/4, exclude: 0/1); window (0,1) holds 1, 2 -> 3/4 and 3/2
    inc = oracle.pool2d_fprop(x, (2, 2), mode="avg_include_pad", pads=(1, 0, 1, 0), stride=(2, 2),
                              lib=lib)[0, 0]
    exc = oracle.pool2d_fprop(x, (2, 2), mode="avg_exclude_pad", pads=(1, 0, 1, 0), stride=(2, 2),
                              lib=lib)[0, 0]
    assert inc[0, 0] == 0.0 and inc[0, 1] == 0.75 and exc[0, 1] == 1.5 and exc[1, 1] == 7.5
    # alpha, beta
    y_in = np.full((1, 1, 2, 2), 2.0)
    got = oracle.pool2d_fprop(x, (2, 2), stride=(2, 2), alpha=0.5, beta=-1.0, y_in=y_in, lib=lib)
    assert np.array_equal(got[0, 0], [[0.5, 1.5], [4.5, 5.5]])


def check_activation(lib):
    rng = np.random.default_rng(3)
    x = rng.uniform(-6, 6, (2, 3, 5, 7))
    forms = {"identity": x, "relu": np.maximum(x, 0), "sigmoid": 1 / (1 + np.exp(-x)),
             "tanh": np.tanh(x), "clipped_relu": np.clip(x, 0, 2.5)}
    for mode, ref in forms.items():
        y = oracle.activation_fprop(x, mode=mode, coef=2.5, lib=lib)
        np.testing.assert_allclose(y, ref, rtol=1e-15, atol=1e-15)
    z = np.zeros((1, 1, 1, 1))
    assert oracle.activation_fprop(z, mode="sigmoid", lib=lib)[0, 0, 0, 0] == 0.5
    assert oracle.activation_fprop(z, mode="tanh", lib=lib)[0, 0, 0, 0] == 0.0
    s = oracle.activation_fprop(x, mode="sigmoid", lib=lib) + oracle.activation_fprop(-x, mode="sigmoid", lib=lib)
    np.testing.assert_allclose(s, 1.0, rtol=1e-15)
    t = oracle.activation_fprop(x, mode="tanh", lib=lib) + oracle.activation_fprop(-x, mode="tanh", lib=lib)
    np.testing.assert_allclose(t, 0.0, atol=1e-15)
    y_in = rng.uniform(-1, 1, x.shape)
    y = oracle.activation_fprop(x, mode="relu", alpha=2.0, beta=-0.5, y_in=y_in, lib=lib)
    np.testing.assert_allclose(y, 2 * np.maximum(x, 0) - 0.5 * y_in, rtol=1e-15, atol=1e-15)


def check_layouts(lib):
    rng = np.random.default_rng(4)
    x = rng.uniform(-1, 1, (2, 3, 9, 10))
    nhwc = np.ascontiguousarray(x.transpose(0, 2, 3, 1)).transpose(0, 3, 1, 2)
    for mode in ("max", "avg_exclude_pad"):
        a = oracle.pool2d_fprop(x, (3, 3), mode=mode, pads=(1, 1, 1, 1), stride=(2, 2), lib=lib)
        b = oracle.pool2d_fprop(nhwc, (3, 3), mode=mode, pads=(1, 1, 1, 1), stride=(2, 2), lib=lib)
        assert np.array_equal(a, b)
    assert np.array_equal(oracle.activation_fprop(x, mode="tanh", lib=lib),
                          oracle.activation_fprop(nhwc, mode="tanh", lib=lib))


PIN_BATTERY = (check_max, check_avg, check_hand_worked, check_activation, check_layouts)


@pytest.mark.parametrize("check", PIN_BATTERY, ids=lambda f: f.__name__)
def test_pool_act_pins(check):
    check(oracle.load())


def test_pool_rejects_pad_not_smaller_than_window():
    with pytest.raises(ValueError):
        oracle.pool2d_fprop(np.zeros((1, 1, 5, 5)), (2, 2), pads=(2, 0, 0, 0))


MUTANTS = {
    "pool_max_keeps_first": ("if (first || xv > acc)", "if (first)"),
    "pool_avg_exclude_uses_window": ("acc /= (double)count;", "acc /= (double)(R * S);"),
    "pool_pad_side": ("i64 wi = q * v - pad_left + j;", "i64 wi = q * v - pad_right + j;"),
    "pool_row_stride": ("i64 h = p * u - pad_top + i;", "i64 h = p * v - pad_top + i;"),
    "act_sigmoid_sign": ("return 1.0 / (1.0 + exp(-xv));", "return 1.0 / (1.0 + exp(xv));"),
    "act_clip_ceiling": ("(xv > coef ? coef : xv)", "(xv > coef ? xv : xv)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_pool_act_mistake_is_caught(name):
    old, new = MUTANTS[name]
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, f"mutation anchor missing or ambiguous for {name}"
    os.makedirs(oracle.BUILD_DIR, exist_ok=True)
    tmp = tempfile.mkdtemp(prefix="mutant_", dir=oracle.BUILD_DIR)
    try:
        msrc = os.path.join(tmp, "conv_oracle_mutant.c")
        with open(msrc, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.load(oracle.build(force=True, src=msrc, out=os.path.join(tmp, "libm.so")))
        caught = 0
        for check in PIN_BATTERY:
            try:
                check(lib)
            except (AssertionError, ValueError):
                caught += 1
        assert caught > 0, f"no pin caught the planted mistake {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
