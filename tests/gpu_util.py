"""Helpers for the GPU parity tests: run a layer through the C ABI and compare
with the CPU oracle under the bound |y - y_ref| <= 1e-5 * |alpha| * sum|x*w|
+ 1e-6 (plus 1e-6 of the epilogue's |beta*y_in| and |bias| terms, and
2^-8 |y_ref| when y is stored in BF16)."""
from __future__ import annotations

import concurrent.futures

import numpy as np

from deep_learning_convolution_gb300 import api, synth
from oracle import oracle


def to_nchw(y, axes: str) -> np.ndarray:
    return y.permute(*[axes.index(a) for a in "NCHW"]).double().cpu().numpy()


def tolerance(bound, alpha=1.0, beta=0.0, y_in=None, bias_k=None, ref=None, y_bf16=False):
    tol = 1e-5 * abs(alpha) * bound + 1e-6
    if beta != 0.0 and y_in is not None:
        tol = tol + 1e-6 * np.abs(beta * y_in)
    if bias_k is not None:
        tol = tol + 1e-6 * np.abs(bias_k)
    if y_bf16 and ref is not None:
        tol = tol + 2.0 ** -8 * np.abs(ref)
    return tol


def layer_kwargs(layer):
    return dict(pads=(layer.pad_top, layer.pad_bottom, layer.pad_left, layer.pad_right),
                stride=(layer.u, layer.v), dilation=(layer.dil_h, layer.dil_w))


def assert_within(y, ref, tol, what):
    err = np.abs(y - ref)
    bad = ~(err <= tol)  # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.nanargmax(np.where(np.isfinite(err), err / tol, np.inf))
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} outputs outside the bound; first at "
            f"{idx.tolist()}; worst err/tol = {float((err / tol).reshape(-1)[worst]):.3g}; "
            f"y={y.reshape(-1)[worst]!r} ref={ref.reshape(-1)[worst]!r}")


def sample_points(rng, N, K, P, Q, count=65536, border_images=2, border_filters=8):
    """Random outputs plus every border row/column of a few images x filters."""
    pts = np.stack([rng.integers(0, N, count), rng.integers(0, K, count),
                    rng.integers(0, P, count), rng.integers(0, Q, count)], axis=1)
    extra = []
    for n in range(min(N, border_images)):
        for k in np.linspace(0, K - 1, min(K, border_filters)).astype(int):
            for p in range(P):
                extra.append((n, k, p, 0))
                extra.append((n, k, p, Q - 1))
            for q in range(Q):
                extra.append((n, k, 0, q))
                extra.append((n, k, P - 1, q))
    if extra:
        pts = np.concatenate([pts, np.array(extra, dtype=np.int64)])
    return np.unique(pts, axis=0)


def oracle_points_parallel(x64, w64, pts, kw, threads=None, **epi):
    """Point oracle split over host threads (the C call releases the GIL)."""
    threads = threads or oracle.default_threads()
    chunks = np.array_split(pts, max(1, min(threads, len(pts) // 256 + 1)))
    with concurrent.futures.ThreadPoolExecutor(len(chunks)) as ex:
        res = list(ex.map(lambda c: oracle.conv2d_fprop_points(x64, w64, c, **kw, **epi), chunks))
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])


def strided_view(xt, axes: str, kind: str):
    """The same logical tensor stored inside a larger buffer: "chan_pad" pads
    the channel axis, "width_pad" the W axis, "image_pad" each image."""
    import torch
    pad = {"chan_pad": ("C", 8), "width_pad": ("W", 5), "image_pad": ("N", 0)}[kind]
    shape = list(xt.shape)
    if kind == "image_pad":
        big = torch.zeros([shape[0], shape[1] * shape[2] * shape[3] + 40], dtype=xt.dtype,
                          device=xt.device)
        view = big[:, 8:8 + shape[1] * shape[2] * shape[3]].view(shape)
    else:
        ax = axes.index(pad[0])
        shape[ax] += pad[1]
        big = torch.zeros(shape, dtype=xt.dtype, device=xt.device)
        sl = [slice(None)] * 4
        sl[ax] = slice(3 if kind == "width_pad" else 0, (3 if kind == "width_pad" else 0) + xt.shape[ax])
        view = big[tuple(sl)]
    view.copy_(xt)
    return view


def run_and_check(handle, layer, seed, *, batch=None, full=None, alpha=1.0, beta=0.0,
                  with_bias=False, relu=False, y_dtype=None, y_axes=None, expect_kernel=None,
                  guard=True, points=65536, view=None, w_axes=None, mode="cross_correlation"):
    """Runs one layer on the GPU and checks it against the oracle.
    `view` stores x as a strided view (see strided_view); `w_axes` overrides
    the filter layout; `mode` "convolution" mirrors the filter taps (checked
    against the oracle run on the mirrored filters).  Returns the kernel name
    the library chose."""
    import torch
    x, w, bias = synth.make_inputs(layer, seed, batch=batch, with_bias=with_bias)
    xt, wt = api.layer_tensors(layer, x, w, "cuda")
    x_axes, w_axes0 = api.layer_axes(layer)
    if w_axes is not None and w_axes != w_axes0:
        wt = wt.permute(*[w_axes0.index(a) for a in w_axes]).contiguous()
    w_axes = w_axes or w_axes0
    if view is not None:
        xt = strided_view(xt, x_axes, view)
    kw = layer_kwargs(layer)
    n, k, p, q = api.output_dim(xt, wt, x_axes=x_axes, w_axes=w_axes, **kw)
    y_axes = y_axes or x_axes
    y_dtype = y_dtype or torch.float32
    shape = [dict(N=n, C=k, H=p, W=q)[a] for a in y_axes]
    numel = n * k * p * q
    G = 1024 if guard else 0
    buf = torch.empty(numel + 2 * G, dtype=y_dtype, device="cuda")
    buf.fill_(12288.0)  # exactly representable in FP32 and BF16
    # dense y in y_axes order
    y = buf[G:G + numel].view(shape)
    rng = np.random.default_rng(seed + 7)
    y_in = None
    if beta != 0.0:
        y_in_nchw = rng.uniform(-1, 1, size=(n, k, p, q)).astype(np.float32)
        if y_dtype == torch.bfloat16:
            y_in_nchw = synth.round_values(y_in_nchw, "bf16")
        y.copy_(torch.from_numpy(y_in_nchw).permute(*["NCHW".index(a) for a in y_axes]))
        y_in = y_in_nchw.astype(np.float64)
    else:
        y.fill_(float("nan"))  # beta == 0 must overwrite NaN
    bias_t = torch.from_numpy(bias).cuda() if bias is not None else None
    conv = api.Conv2dForward(handle, xt, wt, y, x_axes=x_axes, w_axes=w_axes, y_axes=y_axes,
                             math=api.math_of(layer), mode=mode, **kw)
    kernel = conv.kernel(xt, wt, y)
    if expect_kernel is not None:
        assert kernel == expect_kernel, f"{layer.name}: kernel {kernel}, expected {expect_kernel}"
    conv(xt, wt, y, alpha=alpha, beta=beta, bias=bias_t, relu=relu)
    torch.cuda.synchronize()
    handle.synchronize()
    if G:
        g = torch.cat([buf[:G], buf[G + numel:]]).float().cpu().numpy()
        assert (g == 12288.0).all(), f"{layer.name}: write outside y"
    yn = to_nchw(y, y_axes)
    x64, w64 = x.astype(np.float64), w.astype(np.float64)
    if mode == "convolution":  # the definition with the filter taps mirrored
        w64 = np.ascontiguousarray(w64[:, :, ::-1, ::-1])
    epi = dict(alpha=alpha, beta=beta, relu=relu,
               bias=None if bias is None else bias.astype(np.float64))
    y_bf16 = y_dtype == torch.bfloat16
    if full is None:
        full = n * k * p * q * layer.C * layer.R * layer.S <= 3e8
    if full:
        ref, bound = oracle.conv2d_fprop(x64, w64, y_in=y_in, **kw, **epi)
        tol = tolerance(bound, alpha, beta, y_in, None if bias is None else bias[None, :, None, None],
                        ref, y_bf16)
        assert_within(yn, ref, tol, f"{layer.name} [{kernel}]")
    else:
        pts = sample_points(rng, n, k, p, q, count=points)
        vals, bnd = oracle_points_parallel(x64, w64, pts, kw, y_in=y_in, **epi)
        got = yn[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
        yin_pts = None if y_in is None else y_in[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
        tol = tolerance(bnd, alpha, beta, yin_pts, None if bias is None else bias[pts[:, 1]],
                        vals, y_bf16)
        assert_within(got, vals, tol, f"{layer.name} [{kernel}] sampled")
        # every output was written (no NaN left from the fill)
        assert np.isfinite(yn).all(), f"{layer.name}: unwritten outputs"
    conv.close()
    return kernel
