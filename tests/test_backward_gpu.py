"""GPU parity of the backward routines (data and filter gradients) against
the CPU oracle, through the C ABI.

dx = alpha * dgrad(w, dy) + beta * dx and dw = alpha * wgrad(x, dy) + beta * dw
are compared element by element with the oracle's FP64 gradients of the same
rounded inputs under |got - ref| <= 1e-5 * |alpha| * sum|products| + 1e-6
(+ 1e-6 |beta * old| for the beta term, + 2^-8 |ref| for a BF16 output; FP64
math: 1e-12 * sum|products|).  Small shapes are checked in full; the AlexNet
and ResNet-50 layers at full batch on sampled elements plus every border
element of a few images.  Cases cover the tensor-core dgrad (one SM-pair
launch per stride phase, ragged channel counts, filters read transposed and
mirrored), the direct kernels (TF32 NCHW, strict FP32, FP64, dilation), the
convolution mode and phases that no tap reaches (1x1 stride 2).
"""
import concurrent.futures

import numpy as np
import pytest

from deep_learning_convolution_gb300 import synth
from oracle import oracle

from gpu_util import assert_within

pytestmark = pytest.mark.gpu

L = synth.Layer


def _need_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")


def _round(a, dtype):
    return a.astype(np.float64) if dtype == "f64" else synth.round_values(a, dtype)


def _to_dev(a_nchw, dtype, axes, perm_from="NCHW"):
    """numpy [.. logical perm_from ..] -> device tensor stored in `axes` order."""
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(synth.round_to_bf16_bits(a_nchw).view(np.int16).reshape(a_nchw.shape))
        t = t.view(torch.bfloat16)
    elif dtype == "f64":
        t = torch.from_numpy(np.ascontiguousarray(a_nchw, dtype=np.float64))
    else:
        t = torch.from_numpy(np.ascontiguousarray(a_nchw, dtype=np.float32))
    return t.permute(*[perm_from.index(a) for a in axes]).contiguous().cuda()


def _torch_dtype(dtype):
    import torch
    return {"bf16": torch.bfloat16, "f32": torch.float32, "tf32": torch.float32,
            "f64": torch.float64}[dtype]


def _math(dtype):
    return {"bf16": "bf16", "tf32": "tf32", "f32": "fp32", "f64": "fp64"}[dtype]


def _geom(layer):
    P = (layer.H + layer.pad_top + layer.pad_bottom - layer.dil_h * (layer.R - 1) - 1) // layer.u + 1
    Q = (layer.W + layer.pad_left + layer.pad_right - layer.dil_w * (layer.S - 1) - 1) // layer.v + 1
    kw = dict(pads=(layer.pad_top, layer.pad_bottom, layer.pad_left, layer.pad_right),
              stride=(layer.u, layer.v), dilation=(layer.dil_h, layer.dil_w))
    return P, Q, kw


def _inputs(layer, seed):
    """x [N,C,H,W], w [K,C,R,S], dy [N,K,P,Q] rounded to the layer's storage."""
    st = "f32" if layer.dtype == "f64" else layer.dtype
    x, w, _ = synth.make_inputs(L(**{**layer.__dict__, "dtype": st}), seed)
    P, Q, _ = _geom(layer)
    rng = np.random.default_rng(seed + 1)
    dy = _round(rng.standard_normal((layer.N, layer.K, P, Q)).astype(np.float32), st)
    if layer.dtype == "f64":  # full double inputs (not float-representable only)
        x = x.astype(np.float64) + rng.uniform(-1e-9, 1e-9, x.shape)
        w = w.astype(np.float64) + rng.uniform(-1e-9, 1e-9, w.shape)
        dy = dy.astype(np.float64) + rng.uniform(-1e-9, 1e-9, dy.shape)
    return x.astype(np.float64), w.astype(np.float64), dy.astype(np.float64)


def _tol(bound, dtype, out_bf16=False, ref=None, beta=0.0, old=None, alpha=1.0):
    if dtype == "f64":
        return 1e-12 * abs(alpha) * bound + 1e-300
    tol = 1e-5 * abs(alpha) * bound + 1e-6
    if beta != 0.0 and old is not None:
        tol = tol + 1e-6 * np.abs(beta * old)
    if out_bf16 and ref is not None:
        tol = tol + 2.0 ** -8 * np.abs(ref)
    return tol


def _flip(w):
    return np.ascontiguousarray(w[:, :, ::-1, ::-1])


def _parallel_points(fn, pts, threads=16):
    chunks = np.array_split(pts, max(1, min(threads, len(pts) // 512 + 1)))
    with concurrent.futures.ThreadPoolExecutor(len(chunks)) as ex:
        res = list(ex.map(fn, chunks))
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])


def _border_points(rng, A, B, C_, D, count, images=2, chans=6):
    pts = np.stack([rng.integers(0, A, count), rng.integers(0, B, count),
                    rng.integers(0, C_, count), rng.integers(0, D, count)], axis=1)
    extra = []
    for a in range(min(A, images)):
        for b in np.linspace(0, B - 1, min(B, chans)).astype(int):
            for i in range(C_):
                extra += [(a, b, i, 0), (a, b, i, D - 1)]
            for j in range(D):
                extra += [(a, b, 0, j), (a, b, C_ - 1, j)]
    return np.unique(np.concatenate([pts, np.array(extra, np.int64)]), axis=0)


def run_dgrad(layer, seed, *, alpha=1.0, beta=0.0, mode="cross_correlation", out_dtype=None,
              expect=None, full=None, points=32768):
    import torch
    from deep_learning_convolution_gb300 import api
    _need_cuda()
    x, w, dy = _inputs(layer, seed)
    P, Q, kw = _geom(layer)
    nhwc = layer.layout == "NHWC"
    act_axes, w_axes = ("NHWC", "KRSC") if nhwc else ("NCHW", "KCRS")
    st = layer.dtype
    wt = _to_dev(w, st, w_axes, "KCRS")
    dyt = _to_dev(dy, st, act_axes)
    out_dtype = out_dtype or (torch.float64 if st == "f64" else torch.float32)
    shape = [dict(N=layer.N, C=layer.C, H=layer.H, W=layer.W)[a] for a in act_axes]
    dx = torch.empty(shape, dtype=out_dtype, device="cuda")
    old = None
    if beta != 0.0:
        old = np.random.default_rng(seed + 5).uniform(-1, 1, (layer.N, layer.C, layer.H, layer.W))
        if out_dtype == torch.bfloat16:
            old = synth.round_values(old.astype(np.float32), "bf16").astype(np.float64)
        dx.copy_(torch.from_numpy(old).permute(*["NCHW".index(a) for a in act_axes]))
    else:
        dx.fill_(float("nan"))
    handle = api.Handle()
    op = api.Conv2dBackwardData(handle, wt, dyt, dx, w_axes=w_axes, dy_axes=act_axes,
                                dx_axes=act_axes, math=_math(st), mode=mode, **kw)
    kernel = op.kernel(wt, dyt, dx)
    if expect:
        assert kernel == expect, f"{layer.name}: kernel {kernel}, expected {expect}"
    assert op.workspace_size() == 0
    op(wt, dyt, dx, alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    handle.synchronize()
    got = dx.permute(*[act_axes.index(a) for a in "NCHW"]).double().cpu().numpy()
    wref = _flip(w) if mode == "convolution" else w
    if full is None:
        full = layer.N * layer.C * layer.H * layer.W * layer.K * layer.R * layer.S <= 4e8
    if full:
        ref, bound = oracle.conv2d_dgrad(dy, wref, (layer.H, layer.W), **kw)
        ref = alpha * ref + (beta * old if old is not None else 0.0)
        tol = _tol(bound, st, out_dtype == torch.bfloat16, ref, beta, old, alpha)
        assert_within(got, ref, tol, f"dgrad {layer.name} [{kernel}]")
    else:
        pts = _border_points(np.random.default_rng(seed), layer.N, layer.C, layer.H, layer.W, points)
        vals, bnd = _parallel_points(
            lambda c: oracle.conv2d_dgrad_points(dy, wref, (layer.H, layer.W), c, **kw), pts)
        vals = alpha * vals
        o = None
        if old is not None:
            o = old[tuple(pts.T)]
            vals = vals + beta * o
        tol = _tol(bnd, st, out_dtype == torch.bfloat16, vals, beta, o, alpha)
        assert_within(got[tuple(pts.T)], vals, tol, f"dgrad {layer.name} [{kernel}] sampled")
        assert np.isfinite(got).all(), f"{layer.name}: unwritten dx"
    op.close()
    handle.close()
    return kernel


def run_wgrad(layer, seed, *, alpha=1.0, beta=0.0, mode="cross_correlation", expect=None,
              out_dtype=None, full=None, points=16384, deterministic=False):
    import torch
    from deep_learning_convolution_gb300 import api
    _need_cuda()
    x, w, dy = _inputs(layer, seed)
    P, Q, kw = _geom(layer)
    nhwc = layer.layout == "NHWC"
    act_axes, w_axes = ("NHWC", "KRSC") if nhwc else ("NCHW", "KCRS")
    st = layer.dtype
    xt = _to_dev(x, st, act_axes)
    dyt = _to_dev(dy, st, act_axes)
    out_dtype = out_dtype or (torch.float64 if st == "f64" else torch.float32)
    shape = [dict(K=layer.K, C=layer.C, R=layer.R, S=layer.S)[a] for a in w_axes]
    dw = torch.empty(shape, dtype=out_dtype, device="cuda")
    old = None
    if beta != 0.0:
        old = np.random.default_rng(seed + 5).uniform(-1, 1, (layer.K, layer.C, layer.R, layer.S))
        dw.copy_(torch.from_numpy(old).permute(*["KCRS".index(a) for a in w_axes]))
    else:
        dw.fill_(float("nan"))
    handle = api.Handle()
    handle.set_deterministic(deterministic)
    op = api.Conv2dBackwardFilter(handle, xt, dyt, dw, x_axes=act_axes, dy_axes=act_axes,
                                  dw_axes=w_axes, math=_math(st), mode=mode, **kw)
    kernel = op.kernel(xt, dyt, dw)
    if expect:
        assert kernel == expect, f"{layer.name}: kernel {kernel}, expected {expect}"
    assert op.workspace_size() == 0
    op(xt, dyt, dw, alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    handle.synchronize()
    got = dw.permute(*[w_axes.index(a) for a in "KCRS"]).double().cpu().numpy()
    if mode == "convolution":
        got = _flip(got)  # the oracle's cross-correlation gradient, tap-mirrored
        old = _flip(old) if old is not None else None
    if full is None:
        full = layer.N * layer.C * layer.H * layer.W * layer.K * layer.R * layer.S <= 4e8
    if full:
        ref, bound = oracle.conv2d_wgrad(x, dy, (layer.R, layer.S), **kw)
        ref = alpha * ref + (beta * old if old is not None else 0.0)
        tol = _tol(bound, st, out_dtype == torch.bfloat16, ref, beta, old, alpha)
        assert_within(got, ref, tol, f"wgrad {layer.name} [{kernel}]")
    else:
        rng = np.random.default_rng(seed)
        pts = np.unique(np.stack([rng.integers(0, layer.K, points), rng.integers(0, layer.C, points),
                                  rng.integers(0, layer.R, points), rng.integers(0, layer.S, points)],
                                 axis=1), axis=0)
        vals, bnd = _parallel_points(
            lambda c: oracle.conv2d_wgrad_points(x, dy, (layer.R, layer.S), c, **kw), pts)
        vals = alpha * vals
        o = None
        if old is not None:
            o = old[tuple(pts.T)]
            vals = vals + beta * o
        tol = _tol(bnd, st, False, vals, beta, o, alpha)
        assert_within(got[tuple(pts.T)], vals, tol, f"wgrad {layer.name} [{kernel}] sampled")
        assert np.isfinite(got).all(), f"{layer.name}: unwritten dw"
    op.close()
    handle.close()
    return kernel, dw


P1 = dict(pad_top=1, pad_bottom=1, pad_left=1, pad_right=1)

DGRAD_TC = [
    L("dg_3x3_s1_c64_k64", 2, 64, 15, 17, 64, 3, 3, **P1),
    L("dg_3x3_s1_c72_k96", 3, 72, 13, 11, 96, 3, 3, **P1),
    L("dg_5x5_s1_c136_k64_asym", 2, 136, 12, 14, 64, 5, 5, pad_top=2, pad_bottom=1, pad_left=0,
      pad_right=3),
    L("dg_3x3_s2_c64_k128", 2, 64, 16, 15, 128, 3, 3, u=2, v=2, **P1),
    L("dg_1x1_s2_c128_k64", 2, 128, 14, 14, 64, 1, 1, u=2, v=2),
    L("dg_11x11_s4_c64_k64", 2, 64, 35, 35, 64, 11, 11, pad_top=2, pad_bottom=2, pad_left=2,
      pad_right=2, u=4, v=4),
    L("dg_3x3_s1_c256_k384", 2, 256, 9, 9, 384, 3, 3, **P1),
]


@pytest.mark.parametrize("layer", DGRAD_TC, ids=lambda l: l.name)
def test_dgrad_tensor_cores(layer):
    run_dgrad(layer, 700, expect="tc_im2col_pair")


@pytest.mark.parametrize("loaders", ["0", "1", "2"], ids=["one_thread", "a_b_split", "alternate"])
@pytest.mark.parametrize("layer", [DGRAD_TC[i] for i in (1, 3, 6)], ids=lambda l: l.name)
def test_dgrad_load_issue(layer, loaders, monkeypatch):
    """The data gradient with the SM-pair kernel's loads issued by one thread,
    by two (A and B) and by two taking alternate k-blocks (the default for its
    MN-major filters)."""
    monkeypatch.setenv("DLC_TC_PAIR_SPLITLOAD", loaders)
    run_dgrad(layer, 705, expect="tc_im2col_pair")


@pytest.mark.parametrize("layer", [DGRAD_TC[i] for i in (1, 2, 6)], ids=lambda l: l.name)
def test_dgrad_two_kblocks_a_stage(layer, monkeypatch):
    """The data gradient with two k-blocks per pipeline stage (DLC_TC_PAIR_KPS=2)."""
    monkeypatch.setenv("DLC_TC_PAIR_KPS", "2")
    run_dgrad(layer, 707, expect="tc_im2col_pair")


def test_dgrad_alpha_beta_and_bf16_output():
    import torch
    layer = DGRAD_TC[1]
    run_dgrad(layer, 701, alpha=0.5, beta=-1.25, expect="tc_im2col_pair")
    run_dgrad(layer, 702, out_dtype=torch.bfloat16, expect="tc_im2col_pair")
    run_dgrad(DGRAD_TC[3], 703, alpha=2.0, beta=0.5, expect="tc_im2col_pair")


@pytest.mark.parametrize("layer", [DGRAD_TC[0], DGRAD_TC[3], DGRAD_TC[5]], ids=lambda l: l.name)
def test_dgrad_convolution_mode(layer):
    run_dgrad(layer, 704, mode="convolution", expect="tc_im2col_pair")


DGRAD_DIRECT = [
    L("dg_tf32_nchw_c32", 2, 32, 20, 19, 32, 5, 3, pad_top=2, pad_bottom=2, pad_left=1,
      pad_right=1, u=2, v=1, dtype="tf32", layout="NCHW"),
    L("dg_f32_nchw_dil2", 2, 8, 16, 16, 16, 3, 3, pad_top=2, pad_bottom=2, pad_left=2,
      pad_right=2, dil_h=2, dil_w=2, dtype="f32", layout="NCHW"),
    L("dg_bf16_nhwc_dil2", 2, 64, 12, 12, 64, 3, 3, **P1, dil_h=2, dil_w=1),
    L("dg_f64_nchw", 2, 4, 9, 10, 5, 3, 2, pad_top=1, pad_bottom=0, pad_left=1, pad_right=1,
      u=2, v=1, dtype="f64", layout="NCHW"),
]


@pytest.mark.parametrize("layer", DGRAD_DIRECT, ids=lambda l: l.name)
def test_dgrad_direct(layer):
    run_dgrad(layer, 710, expect="direct")
    run_dgrad(layer, 711, mode="convolution", alpha=0.75, beta=0.5, expect="direct")


FULL_SIZE = [
    L("alex2_64x192_27_5x5", 128, 64, 27, 27, 192, 5, 5, pad_top=2, pad_bottom=2, pad_left=2,
      pad_right=2),
    L("alex4_384x256_13_3x3", 128, 384, 13, 13, 256, 3, 3, **P1),
    L("rn_3x3_28_128", 256, 128, 28, 28, 128, 3, 3, **P1, w_dist="he"),
    L("rn_3x3s2_56_128", 256, 128, 56, 56, 128, 3, 3, **P1, u=2, v=2, w_dist="he"),
    L("rn_1x1s2_28_512x1024", 256, 512, 28, 28, 1024, 1, 1, u=2, v=2, w_dist="he"),
]


@pytest.mark.parametrize("layer", FULL_SIZE, ids=lambda l: l.name)
def test_dgrad_full_size_sampled(layer):
    run_dgrad(layer, 720, full=False, expect="tc_im2col_pair")


WGRAD = [
    L("wg_3x3_s1_c64_k64", 2, 64, 15, 17, 64, 3, 3, **P1),
    L("wg_3x3_s2_c72_k96", 3, 72, 13, 11, 96, 3, 3, u=2, v=2, **P1),
    L("wg_tf32_nchw_c32", 2, 32, 20, 19, 32, 5, 3, pad_top=2, pad_bottom=2, pad_left=1,
      pad_right=1, u=2, v=1, dtype="tf32", layout="NCHW"),
    L("wg_f32_dil2", 2, 8, 16, 16, 16, 3, 3, pad_top=2, pad_bottom=2, pad_left=2, pad_right=2,
      dil_h=2, dil_w=2, dtype="f32", layout="NCHW"),
    L("wg_f64_nchw", 2, 4, 9, 10, 5, 3, 2, pad_top=1, pad_bottom=0, pad_left=1, pad_right=1,
      u=2, v=1, dtype="f64", layout="NCHW"),
    L("wg_c3_11x11_s4", 2, 3, 35, 35, 64, 11, 11, pad_top=2, pad_bottom=2, pad_left=2,
      pad_right=2, u=4, v=4),
]


WGRAD_TC = {"wg_3x3_s1_c64_k64", "wg_3x3_s2_c72_k96"}


@pytest.mark.parametrize("layer", WGRAD, ids=lambda l: l.name)
def test_wgrad(layer):
    tc = layer.name in WGRAD_TC
    run_wgrad(layer, 730, expect="tc_wgrad" if tc else "direct")
    run_wgrad(layer, 731, alpha=0.75, beta=0.5, expect="tc_wgrad" if tc else "direct")
    run_wgrad(layer, 732, mode="convolution", alpha=0.75, beta=0.5, expect="direct")


WGRAD_TC_MORE = [
    L("wg_tc_c136_k200_5x5", 2, 136, 12, 14, 200, 5, 5, pad_top=2, pad_bottom=1, pad_left=0,
      pad_right=3),
    L("wg_tc_c384_k256_3x3", 4, 384, 13, 13, 256, 3, 3, **P1),
    L("wg_tc_c64_k64_1x1_s2", 3, 64, 14, 14, 64, 1, 1, u=2, v=2),
    L("wg_tc_c96_k64_11x11_s4", 2, 96, 35, 35, 64, 11, 11, pad_top=2, pad_bottom=2, pad_left=2,
      pad_right=2, u=4, v=4),
]


@pytest.mark.parametrize("pair", ["1", "0"], ids=["sm_pairs", "single_sm"])
@pytest.mark.parametrize("layer", WGRAD_TC_MORE, ids=lambda l: l.name)
def test_wgrad_tensor_cores(layer, pair, monkeypatch):
    """More than 128 filters run on SM pairs (M = 256 per MMA) unless
    DLC_TC_WGRAD_PAIR=0; both agree with the oracle."""
    if pair == "0" and layer.K <= 128:
        pytest.skip("up to 128 filters always run on single SMs")
    monkeypatch.setenv("DLC_TC_WGRAD_PAIR", pair)
    run_wgrad(layer, 734, expect="tc_wgrad")
    run_wgrad(layer, 735, alpha=-0.5, beta=2.0, expect="tc_wgrad", deterministic=True)


# Pairs with at most 128 channels stack two filter taps per unit (one per CTA
# of the pair): odd and even tap counts (the odd one's last unit has a single
# tap), one or two 64-channel blocks, channels short of a block, stride and
# dilation.
WGRAD_STACK = [
    L("wg_stack_c96_k256_5x5", 2, 96, 12, 12, 256, 5, 5, pad_top=2, pad_bottom=2, pad_left=2,
      pad_right=2),
    L("wg_stack_c64_k192_3x3", 3, 64, 11, 9, 192, 3, 3, **P1),
    L("wg_stack_c128_k160_2x3_s2", 2, 128, 13, 15, 160, 2, 3, pad_top=1, pad_bottom=0,
      pad_left=1, pad_right=1, u=2, v=2),
    L("wg_stack_c72_k136_3x3_d2", 2, 72, 14, 13, 136, 3, 3, pad_top=2, pad_bottom=2, pad_left=1,
      pad_right=2, dil_h=2, dil_w=2),
]


@pytest.mark.parametrize("stack", ["1", "0"], ids=["stacked_taps", "one_tap"])
@pytest.mark.parametrize("layer", WGRAD_STACK, ids=lambda l: l.name)
def test_wgrad_stacked_taps(layer, stack, monkeypatch):
    """SM pairs with two taps a unit (the default at <= 128 channels) and with
    one tap a unit (DLC_TC_WGRAD_STACK=0) both agree with the oracle, split
    and deterministic, with alpha and beta."""
    monkeypatch.setenv("DLC_TC_WGRAD_STACK", stack)
    run_wgrad(layer, 736, expect="tc_wgrad")
    run_wgrad(layer, 737, alpha=-0.5, beta=2.0, expect="tc_wgrad", deterministic=True)


def test_wgrad_bf16_output_and_determinism():
    import torch
    layer = WGRAD[0]
    run_wgrad(layer, 732, out_dtype=torch.bfloat16)
    _, a = run_wgrad(layer, 733, deterministic=True)
    _, b = run_wgrad(layer, 733, deterministic=True)
    assert torch.equal(a, b), "deterministic filter gradients differ between runs"


@pytest.mark.parametrize("layer", FULL_SIZE, ids=lambda l: l.name)
def test_wgrad_full_size_sampled(layer):
    run_wgrad(layer, 740, full=False, expect="tc_wgrad")
