"""Run-to-run reproducibility and non-finite inputs, through the C ABI.

Reproducibility: the SM-pair kernel splits the last, mostly idle wave of a
launch along the reduction and adds the partial sums into y with FP32 atomic
adds (their order varies).  An AlexNet-layer-4-shaped problem (384 -> 256,
13 x 13, 3 x 3) is run twice in each mode: in the default mode both runs stay
within the parity bound against the oracle; with dlcSetDeterministic(1) the
two runs are bitwise identical (and within the bound).

Non-finite inputs: the definition is a finite sum of products, so one Inf at
input pixel (n0, c0, h0, w0) makes every output whose receptive field holds
that pixel +-Inf (or NaN where the filter tap is zero) and leaves every other
output finite.  The im2col, run-gather and FFMA kernels read exactly each
output's window and must reproduce that classification element by element;
the window kernel (few-channel layers) also multiplies zero filter taps with
the real input pixels that share a packed phase pixel with a window's edge,
so there an output next to such a window may be NaN: only NaN, only in image
n0, only in rows whose window holds h0 and only within one phase pixel of the
Inf's column.  The row-stack kernel multiplies zero taps with the input rows
of its block of 4 output rows and up to 3 columns past a window: only NaN,
only in image n0, only in the blocks of rows that hold a hit row, and only
within 4 columns of the Inf's.
"""
import numpy as np
import pytest

from deep_learning_convolution_gb300 import synth
from oracle import oracle

from gpu_util import layer_kwargs, sample_points, oracle_points_parallel, to_nchw

pytestmark = pytest.mark.gpu

L = synth.Layer
ALEX4 = L("alex4_384x256_13_3x3", 128, 384, 13, 13, 256, 3, 3, pad_top=1, pad_bottom=1,
          pad_left=1, pad_right=1)


def _need_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")


def _run_twice(handle, layer, xt, wt):
    import torch
    from deep_learning_convolution_gb300 import api
    conv, y = api.layer_problem(handle, layer, xt, wt)
    outs = []
    for _ in range(2):
        y.fill_(float("nan"))
        conv(xt, wt, y)
        torch.cuda.synchronize()
        handle.synchronize()
        outs.append(y.clone())
    kernel = conv.kernel(xt, wt, y)
    conv.close()
    return kernel, outs


@pytest.mark.parametrize("deterministic", [0, 1], ids=["default", "deterministic"])
def test_split_tail_reproducibility(deterministic):
    import torch
    from deep_learning_convolution_gb300 import api
    _need_cuda()
    x, w, _ = synth.make_inputs(ALEX4, synth.workload_seed("alexnet", 3))
    xt, wt = api.layer_tensors(ALEX4, x, w, "cuda")
    handle = api.Handle()
    handle.set_deterministic(bool(deterministic))
    kernel, (y1, y2) = _run_twice(handle, ALEX4, xt, wt)
    assert kernel == "tc_im2col_pair"
    if deterministic:
        assert torch.equal(y1.view(torch.int32), y2.view(torch.int32)), "runs differ in their bits"
    rng = np.random.default_rng(11)
    n, k, p, q = ALEX4.N, ALEX4.K, 13, 13
    # every tail row (the split tiles are the last ones) plus a random sample
    pts = sample_points(rng, n, k, p, q, count=32768)
    tail = np.stack(np.meshgrid(np.arange(n - 2, n), np.arange(0, k, 7), np.arange(p),
                                np.arange(q), indexing="ij"), -1).reshape(-1, 4)
    pts = np.unique(np.concatenate([pts, tail]), axis=0)
    vals, bnd = oracle_points_parallel(x.astype(np.float64), w.astype(np.float64), pts,
                                       layer_kwargs(ALEX4))
    tol = 1e-5 * bnd + 1e-6
    for y in (y1, y2):
        got = to_nchw(y, "NHWC")[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
        assert (np.abs(got - vals) <= tol).all()
    handle.close()


NONFINITE_CASES = [
    (L("nf_pair_c64_5x5", 2, 64, 27, 27, 96, 5, 5, pad_top=2, pad_bottom=2, pad_left=2,
       pad_right=2), "tc_im2col_pair"),
    (L("nf_runs_tf32_nchw_c32", 2, 32, 20, 23, 32, 3, 3, pad_top=1, pad_bottom=1, pad_left=1,
       pad_right=1, dtype="tf32", layout="NCHW"), "tc_runs"),
    (L("nf_rowstack_tf32_nchw_c32", 2, 32, 20, 23, 32, 3, 3, pad_top=1, pad_bottom=1, pad_left=1,
       pad_right=1, dtype="tf32", layout="NCHW"), "tc_rowstack"),
    (L("nf_ffma_nchw_c8", 2, 8, 16, 16, 16, 3, 3, pad_top=1, pad_bottom=1, pad_left=1,
       pad_right=1, dtype="f32", layout="NCHW"), "ffma"),
    (L("nf_window_c3_11x11_s4", 2, 3, 67, 67, 64, 11, 11, pad_top=2, pad_bottom=2, pad_left=2,
       pad_right=2, u=4, v=4), "tc_window"),
]


@pytest.mark.parametrize("layer,kernel", NONFINITE_CASES, ids=lambda v: getattr(v, "name", v))
def test_one_inf_in_x(layer, kernel, monkeypatch):
    import torch
    from deep_learning_convolution_gb300 import api
    _need_cuda()
    if kernel == "tc_runs":
        monkeypatch.setenv("DLC_TC_ROWSTACK", "0")
    x, w, _ = synth.make_inputs(layer, 5150)
    n0, c0, h0, w0 = 1, layer.C // 2, layer.H // 2, layer.W // 2 + 1
    x[n0, c0, h0, w0] = np.inf
    xt, wt = api.layer_tensors(layer, x, w, "cuda")
    handle = api.Handle()
    conv, y = api.layer_problem(handle, layer, xt, wt)
    assert conv.kernel(xt, wt, y) == kernel
    y.fill_(0.0)
    conv(xt, wt, y)
    torch.cuda.synchronize()
    handle.synchronize()
    got = to_nchw(y, api.layer_axes(layer)[0])
    with np.errstate(invalid="ignore", over="ignore"):
        ref, bound = oracle.conv2d_fprop(x.astype(np.float64), w.astype(np.float64),
                                         **layer_kwargs(layer))
    hit = ~np.isfinite(ref)
    assert hit[n0].any() and not hit[0].any()
    # outputs whose window holds the Inf: same class as the definition
    assert np.array_equal(np.isnan(got[hit]), np.isnan(ref[hit]))
    assert np.array_equal(np.isposinf(got[hit]), np.isposinf(ref[hit]))
    assert np.array_equal(np.isneginf(got[hit]), np.isneginf(ref[hit]))
    ok = ~hit & np.isfinite(got)
    tol = 1e-5 * bound + 1e-6
    assert (np.abs(got[ok] - ref[ok]) <= tol[ok]).all()
    spurious = ~hit & ~np.isfinite(got)
    if kernel == "tc_rowstack":
        # zero filter taps meet the Inf in the other output rows of its block of
        # 4 and up to 3 columns past a window
        assert np.isnan(got[spurious]).all()
        nn, kk, pp, qq = np.nonzero(spurious)
        assert (nn == n0).all()
        hit_rows = np.unique(np.nonzero(hit[n0])[1])
        assert all(np.abs(hit_rows - p_).min() < 4 and p_ // 4 in hit_rows // 4 for p_ in pp)
        off = w0 - (qq - layer.pad_left)
        assert ((off >= -4) & (off < layer.S + 4)).all()
    elif kernel != "tc_window":
        assert not spurious.any(), f"{int(spurious.sum())} outputs non-finite off the window"
    else:
        assert np.isnan(got[spurious]).all()
        nn, kk, pp, qq = np.nonzero(spurious)
        assert (nn == n0).all()
        rows = [p for p in range(ref.shape[2])
                if 0 <= h0 - (p * layer.u - layer.pad_top) < layer.R * layer.dil_h]
        assert np.isin(pp, rows).all()
        off = w0 - (qq * layer.v - layer.pad_left)   # Inf's column inside the read span
        assert ((off >= -layer.v) & (off < layer.S + 2 * layer.v)).all()
    conv.close()
    handle.close()
