"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each check ties the oracle to something it does not compute itself:
hand-derived worked examples (tests/golden), an independent GEMM-based
convolution (im2col x matmul, the lowering named in the cuDNN page's method
section), library routines (torch conv2d in FP64, scipy correlate2d), closed
forms (1x1 stride-1 = matrix product; a delta filter = a shifted copy),
invariants (linearity, translation equivariance, layout independence) and a
brute-force count of output positions.  The planted-mistake tests compile
mutated copies of the oracle and check that this battery rejects each one.
"""
import json
import os
import shutil
import tempfile

import numpy as np
import pytest

from oracle import oracle
from deep_learning_convolution_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand(rng, *shape):
    return rng.uniform(-1.0, 1.0, size=shape)


# --------------------------------------------------------------------------
# independent references (test-side; none of them calls the oracle)
# --------------------------------------------------------------------------

def window_origins(extent_padded, eff, stride):
    """Brute-force list of window origins inside a padded axis."""
    out = []
    o = 0
    while o + eff - 1 <= extent_padded - 1:
        out.append(o)
        o += stride
    return out


def im2col_matmul(x, w, pads, stride, dil):
    """GEMM-based convolution: explicit column matrix times the filter matrix."""
    N, C, H, W = x.shape
    K, _, R, S = w.shape
    pt, pb, pl, pr = pads
    xp = np.pad(x, ((0, 0), (0, 0), (pt, pb), (pl, pr)))
    oh = window_origins(xp.shape[2], dil[0] * (R - 1) + 1, stride[0])
    ow = window_origins(xp.shape[3], dil[1] * (S - 1) + 1, stride[1])
    rows = np.array(oh)[:, None] + dil[0] * np.arange(R)[None, :]        # [P, R]
    cols = np.array(ow)[:, None] + dil[1] * np.arange(S)[None, :]        # [Q, S]
    # patches[n, c, p, r, q, s]
    patches = xp[:, :, rows[:, :, None, None], cols[None, None, :, :]]
    colmat = patches.transpose(0, 2, 4, 1, 3, 5).reshape(N * len(oh) * len(ow), C * R * S)
    y = colmat @ w.reshape(K, C * R * S).T
    return y.reshape(N, len(oh), len(ow), K).transpose(0, 3, 1, 2)


def torch_conv(x, w, pads, stride, dil):
    import torch
    import torch.nn.functional as F
    pt, pb, pl, pr = pads
    xt = F.pad(torch.from_numpy(x), (pl, pr, pt, pb))
    return F.conv2d(xt, torch.from_numpy(w), stride=stride, dilation=dil).numpy()


def random_case(rng):
    R, S = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    dil = (int(rng.integers(1, 3)), int(rng.integers(1, 3)))
    H = int(rng.integers(dil[0] * (R - 1) + 1, 14))
    W = int(rng.integers(dil[1] * (S - 1) + 1, 14))
    pads = tuple(int(p) for p in rng.integers(0, 3, size=4))
    stride = (int(rng.integers(1, 4)), int(rng.integers(1, 4)))
    N, C, K = int(rng.integers(1, 3)), int(rng.integers(1, 5)), int(rng.integers(1, 5))
    return _rand(rng, N, C, H, W), _rand(rng, K, C, R, S), pads, stride, dil


# --------------------------------------------------------------------------
# the pin battery (also run against planted-mistake builds below)
# --------------------------------------------------------------------------

def check_golden(lib):
    with open(os.path.join(HERE, "golden", "hand_worked.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        x = np.array(case["x"], dtype=np.float64)
        w = np.array(case["w"], dtype=np.float64)
        y_exp = np.array(case["y"], dtype=np.float64)
        if x.ndim == 2:
            x = x[None, None]
            w = w[None, None]
            y_exp = y_exp[None, None]
        else:
            x = x[None]
            y_exp = y_exp[None]
        y, _ = oracle.conv2d_fprop(x, w, pads=tuple(case["pads"]), stride=tuple(case["stride"]),
                                   dilation=tuple(case["dilation"]), lib=lib)
        assert y.shape == y_exp.shape, case["name"]
        assert np.array_equal(y, y_exp), case["name"]


def check_im2col(lib, seed=1, count=25):
    rng = np.random.Generator(np.random.PCG64(seed))
    for _ in range(count):
        x, w, pads, stride, dil = random_case(rng)
        y, _ = oracle.conv2d_fprop(x, w, pads=pads, stride=stride, dilation=dil, lib=lib)
        ref = im2col_matmul(x, w, pads, stride, dil)
        assert y.shape == ref.shape
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def check_torch(lib, seed=2, count=15):
    rng = np.random.Generator(np.random.PCG64(seed))
    for _ in range(count):
        x, w, pads, stride, dil = random_case(rng)
        y, _ = oracle.conv2d_fprop(x, w, pads=pads, stride=stride, dilation=dil, lib=lib)
        ref = torch_conv(x, w, pads, stride, dil)
        assert y.shape == ref.shape
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def check_epilogue(lib, seed=3):
    rng = np.random.Generator(np.random.PCG64(seed))
    x, w = _rand(rng, 2, 3, 9, 8), _rand(rng, 5, 3, 3, 2)
    kw = dict(pads=(1, 0, 2, 1), stride=(2, 1), dilation=(1, 2), lib=lib)
    plain, _ = oracle.conv2d_fprop(x, w, **kw)
    y_in = _rand(rng, *plain.shape)
    bias = _rand(rng, 5)
    alpha, beta = 0.75, -1.25
    y, _ = oracle.conv2d_fprop(x, w, alpha=alpha, beta=beta, y_in=y_in, bias=bias, relu=True, **kw)
    exp = np.maximum(alpha * plain + beta * y_in + bias[None, :, None, None], 0.0)
    np.testing.assert_allclose(y, exp, rtol=1e-14, atol=1e-14)
    assert (y == 0).any() and (y > 0).any()
    y2, _ = oracle.conv2d_fprop(x, w, bias=bias, **kw)
    np.testing.assert_allclose(y2, plain + bias[None, :, None, None], rtol=1e-14, atol=1e-14)


def check_points_epilogue(lib, seed=4):
    """The point evaluator with beta != 0 reads y_in through its own strides:
    compared with the closed form alpha*conv + beta*y_in + bias on a y_in held
    as a transposed (NHWC-stored) view, so a dropped or misapplied stride
    picks up the wrong y_in element."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x, w = _rand(rng, 2, 3, 9, 8), _rand(rng, 4, 3, 3, 2)
    kw = dict(pads=(1, 2, 0, 1), stride=(2, 1), dilation=(1, 1), lib=lib)
    plain, _ = oracle.conv2d_fprop(x, w, **kw)
    y_nhwc = _rand(rng, plain.shape[0], plain.shape[2], plain.shape[3], plain.shape[1])
    y_in = y_nhwc.transpose(0, 3, 1, 2)   # [N,K,P,Q] view, channels innermost in memory
    bias = _rand(rng, 4)
    alpha, beta = -0.5, 1.75
    pts = np.array([[n, k, p, q] for n in range(plain.shape[0]) for k in range(4)
                    for p in range(plain.shape[2]) for q in range(plain.shape[3])])
    v, _ = oracle.conv2d_fprop_points(x, w, pts, alpha=alpha, beta=beta, y_in=y_in, bias=bias,
                                      **kw)
    exp = alpha * plain + beta * y_in + bias[None, :, None, None]
    np.testing.assert_allclose(v, exp.reshape(-1), rtol=1e-14, atol=1e-14)


PIN_BATTERY = (check_golden, check_im2col, check_torch, check_epilogue, check_points_epilogue)


# --------------------------------------------------------------------------
# tests
# --------------------------------------------------------------------------

def test_golden_hand_worked(oracle_lib):
    check_golden(oracle_lib)


def test_matches_im2col_matmul(oracle_lib):
    check_im2col(oracle_lib, count=60)


def test_matches_torch_conv2d_fp64(oracle_lib):
    check_torch(oracle_lib, count=40)


def test_single_channel_matches_scipy_correlate(oracle_lib):
    from scipy.signal import correlate2d
    rng = np.random.Generator(np.random.PCG64(4))
    for pads in ((0, 0, 0, 0), (1, 2, 0, 3)):
        x = _rand(rng, 1, 1, 11, 7)
        w = _rand(rng, 1, 1, 4, 3)
        y, _ = oracle.conv2d_fprop(x, w, pads=pads, lib=oracle_lib)
        pt, pb, pl, pr = pads
        ref = correlate2d(np.pad(x[0, 0], ((pt, pb), (pl, pr))), w[0, 0], mode="valid")
        np.testing.assert_allclose(y[0, 0], ref, rtol=1e-13, atol=1e-13)


def test_one_by_one_is_matmul(oracle_lib):
    rng = np.random.Generator(np.random.PCG64(5))
    x, w = _rand(rng, 3, 7, 5, 6), _rand(rng, 4, 7, 1, 1)
    y, _ = oracle.conv2d_fprop(x, w, lib=oracle_lib)
    ref = np.einsum("kc,nchw->nkhw", w[:, :, 0, 0], x)
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("r0,s0,pads,stride,dil", [
    (0, 0, (0, 0, 0, 0), (1, 1), (1, 1)),
    (2, 1, (1, 2, 3, 0), (2, 3), (1, 1)),
    (1, 2, (2, 2, 1, 1), (1, 2), (2, 1)),
    (3, 0, (3, 0, 0, 2), (3, 1), (2, 2)),
])
def test_delta_filter_is_shifted_copy(oracle_lib, r0, s0, pads, stride, dil):
    rng = np.random.Generator(np.random.PCG64(6))
    C = 3
    x = _rand(rng, 2, C, 12, 13)
    R, S = 4, 3
    w = np.zeros((C, C, R, S))
    for k in range(C):
        w[k, k, r0, s0] = 1.0
    y, _ = oracle.conv2d_fprop(x, w, pads=pads, stride=stride, dilation=dil, lib=oracle_lib)
    pt, pb, pl, pr = pads
    xp = np.pad(x, ((0, 0), (0, 0), (pt, pb), (pl, pr)))
    P, Q = y.shape[2:]
    exp = xp[:, :, r0 * dil[0]: r0 * dil[0] + stride[0] * (P - 1) + 1: stride[0],
             s0 * dil[1]: s0 * dil[1] + stride[1] * (Q - 1) + 1: stride[1]]
    assert np.array_equal(y, exp)  # exp is cut from the zero-padded input


def test_linearity(oracle_lib):
    rng = np.random.Generator(np.random.PCG64(7))
    x1, x2 = _rand(rng, 2, 3, 8, 9), _rand(rng, 2, 3, 8, 9)
    w1, w2 = _rand(rng, 4, 3, 3, 2), _rand(rng, 4, 3, 3, 2)
    kw = dict(pads=(1, 1, 0, 2), stride=(1, 2), dilation=(2, 1), lib=oracle_lib)
    a, b = 1.5, -0.25
    f = lambda x, w: oracle.conv2d_fprop(x, w, **kw)[0]
    np.testing.assert_allclose(f(a * x1 + b * x2, w1), a * f(x1, w1) + b * f(x2, w1), atol=1e-12)
    np.testing.assert_allclose(f(x1, a * w1 + b * w2), a * f(x1, w1) + b * f(x1, w2), atol=1e-12)


def test_translation_equivariance(oracle_lib):
    rng = np.random.Generator(np.random.PCG64(8))
    u, v, i, j = 2, 3, 2, 1
    x = _rand(rng, 1, 2, 20, 22)
    w = _rand(rng, 3, 2, 3, 4)
    kw = dict(stride=(u, v), dilation=(1, 2), lib=oracle_lib)
    y, _ = oracle.conv2d_fprop(x, w, **kw)
    ys, _ = oracle.conv2d_fprop(np.ascontiguousarray(x[:, :, u * i:, v * j:]), w, **kw)
    P2, Q2 = ys.shape[2:]
    assert np.array_equal(ys, y[:, :, i:i + P2, j:j + Q2])


def test_output_extent_matches_enumeration(oracle_lib):
    for H in range(1, 12):
        for R in range(1, 5):
            for dil in (1, 2, 3):
                for stride in (1, 2, 3, 4):
                    for plo, phi in ((0, 0), (1, 0), (0, 2), (2, 3)):
                        n = len(window_origins(H + plo + phi, dil * (R - 1) + 1, stride))
                        assert oracle.out_extent(H, plo, phi, R, dil, stride, oracle_lib) == n


def test_layout_independence(oracle_lib):
    rng = np.random.Generator(np.random.PCG64(9))
    x, w = _rand(rng, 2, 5, 9, 7), _rand(rng, 6, 5, 3, 3)
    kw = dict(pads=(1, 0, 1, 2), stride=(2, 1), lib=oracle_lib)
    y_nchw, b_nchw = oracle.conv2d_fprop(x, w, **kw)
    x_nhwc = np.ascontiguousarray(x.transpose(0, 2, 3, 1))
    w_krsc = np.ascontiguousarray(w.transpose(0, 2, 3, 1))
    y_nhwc, _ = oracle.conv2d_fprop(x_nhwc, w_krsc, x_axes="NHWC", w_axes="KRSC", **kw)
    big = np.zeros((2, 7, 12, 11))
    big[:, 1:6, 2:11, 3:10] = x
    view = big[:, 1:6, 2:11, 3:10]
    y_view, _ = oracle.conv2d_fprop(view, w, **kw)
    assert np.array_equal(y_nchw, y_nhwc)
    assert np.array_equal(y_nchw, y_view)


def test_bound_is_sum_of_abs_products(oracle_lib):
    rng = np.random.Generator(np.random.PCG64(10))
    x, w = _rand(rng, 1, 4, 6, 6), _rand(rng, 3, 4, 3, 3)
    y, bound = oracle.conv2d_fprop(x, w, pads=(1, 1, 1, 1), lib=oracle_lib)
    ref = im2col_matmul(np.abs(x), np.abs(w), (1, 1, 1, 1), (1, 1), (1, 1))
    np.testing.assert_allclose(bound, ref, rtol=1e-12)
    assert (bound >= np.abs(y) - 1e-12).all()


def test_points_beta_reads_strided_y_in(oracle_lib):
    check_points_epilogue(oracle_lib)


def test_points_match_full(oracle_lib):
    rng = np.random.Generator(np.random.PCG64(11))
    x, w = _rand(rng, 2, 3, 10, 9), _rand(rng, 4, 3, 3, 3)
    kw = dict(pads=(1, 2, 0, 1), stride=(2, 2), dilation=(1, 1), lib=oracle_lib)
    y, bnd = oracle.conv2d_fprop(x, w, bias=np.arange(4.0), relu=True, **kw)
    pts = np.array([[n, k, p, q] for n in range(2) for k in range(4)
                    for p in range(y.shape[2]) for q in range(y.shape[3])])
    v, b = oracle.conv2d_fprop_points(x, w, pts, bias=np.arange(4.0), relu=True, **kw)
    assert np.array_equal(v, y.reshape(-1))
    assert np.array_equal(b, bnd.reshape(-1))


def test_threads_do_not_change_result(oracle_lib):
    rng = np.random.Generator(np.random.PCG64(12))
    x, w = _rand(rng, 3, 4, 8, 8), _rand(rng, 5, 4, 3, 3)
    y1, _ = oracle.conv2d_fprop(x, w, pads=(1, 1, 1, 1), nthreads=1, lib=oracle_lib)
    y7, _ = oracle.conv2d_fprop(x, w, pads=(1, 1, 1, 1), nthreads=7, lib=oracle_lib)
    assert np.array_equal(y1, y7)


def test_rounding_helpers_fix_precision():
    """BF16/TF32 input rounding keeps 8/11 significant bits, nearest-even."""
    a = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -3.14159], np.float32)
    b = synth.round_values(a, "bf16")
    assert b[0] == 1.0 and b[1] == 1.0 and b[2] == 1.0 + 2 ** -6 and b[3] == 1.0
    t = synth.round_values(np.array([1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11], np.float32), "tf32")
    assert t[0] == 1.0 and t[1] == 1.0 + 2 ** -9
    r = synth.round_values(np.random.default_rng(0).standard_normal(1000).astype(np.float32), "tf32")
    assert ((r.view(np.uint32) & 0x1FFF) == 0).all()


# --------------------------------------------------------------------------
# planted mistakes: each mutated oracle must fail at least one pin
# --------------------------------------------------------------------------

MUTANTS = {
    "dilation_axes_swapped": ("i64 h = p * pr->u + r * pr->dh - pr->pt;",
                              "i64 h = p * pr->u + r * pr->dw - pr->pt;"),
    "wrong_pad_side": ("i64 h = p * pr->u + r * pr->dh - pr->pt;",
                       "i64 h = p * pr->u + r * pr->dh - pr->pb;"),
    "dropped_channel": ("for (i64 c = 0; c < pr->C; ++c) {", "for (i64 c = 1; c < pr->C; ++c) {"),
    "filter_taps_transposed": ("c * pr->ws[1] + r * pr->ws[2] + s * pr->ws[3]",
                               "c * pr->ws[1] + s * pr->ws[2] + r * pr->ws[3]"),
    "filter_flipped": ("c * pr->ws[1] + r * pr->ws[2] + s * pr->ws[3]",
                       "c * pr->ws[1] + (pr->R - 1 - r) * pr->ws[2] + s * pr->ws[3]"),
    "ceil_output_size": ("return span / stride + 1;", "return (span + stride - 1) / stride + 1;"),
    "bias_sign": ("val += pr->bias[k];", "val -= pr->bias[k];"),
    "relu_inverted": ("if (pr->relu && val < 0.0)", "if (pr->relu && val > 0.0)"),
    "stride_axes_swapped": ("i64 wi = q * pr->v + s * pr->dw - pr->pl;",
                            "i64 wi = q * pr->u + s * pr->dw - pr->pl;"),
    "beta_ignored": ("val += pr->beta * pr->y_in[yoff];", "val += 0.0 * pr->y_in[yoff];"),
    "points_y_in_strides_ignored": ("NULL, ys ? ys : zero_strides, NULL,",
                                    "NULL, zero_strides, NULL,"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    old, new = MUTANTS[name]
    src = open(oracle.SRC).read()
    assert old in src, f"mutation anchor missing for {name}"
    os.makedirs(oracle.BUILD_DIR, exist_ok=True)
    tmp = tempfile.mkdtemp(prefix="mutant_", dir=oracle.BUILD_DIR)  # inside the repo's build dir
    try:
        msrc = os.path.join(tmp, "conv_oracle_mutant.c")
        with open(msrc, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.load(oracle.build(force=True, src=msrc, out=os.path.join(tmp, "libm.so")))
        caught = []
        for check in PIN_BATTERY:
            try:
                check(lib)
            except (AssertionError, ValueError):
                caught.append(check.__name__)
        assert caught, f"planted mistake {name} passed every pin"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
