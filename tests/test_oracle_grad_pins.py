"""Pins of the oracle's backward routines (data and filter gradients).

The gradients are the next rows of the path; their oracle comes first, pinned
to facts outside itself:
  * the adjoint identity with the (separately pinned) forward oracle:
    <conv(x, w), dy> = <x, dgrad(dy, w)> = <w, wgrad(x, dy)>, which holds
    exactly in real arithmetic for every stride, dilation and padding;
  * torch autograd in FP64 on the CPU (an independent library), with the
    asymmetric padding applied to x explicitly;
  * closed forms for 1x1 stride-1 filters (matrix products);
  * a brute-force enumeration of the products behind one dx element;
  * planted mistakes in copies of the oracle, each caught by this battery.
"""
import os
import shutil
import tempfile

import numpy as np
import pytest

from oracle import oracle

CONFIGS = [
    # (N, C, H, W, K, R, S, pads, stride, dilation)
    (2, 3, 9, 11, 4, 3, 2, (1, 0, 2, 1), (2, 1), (1, 2)),
    (1, 2, 13, 7, 3, 5, 3, (2, 2, 1, 1), (1, 2), (2, 1)),
    (2, 4, 8, 8, 5, 1, 1, (0, 0, 0, 0), (1, 1), (1, 1)),
    (1, 3, 12, 15, 2, 4, 4, (0, 3, 3, 0), (3, 2), (1, 1)),
    (3, 1, 10, 10, 2, 3, 3, (1, 1, 1, 1), (2, 2), (2, 2)),
]


def _case(cfg, seed):
    N, C, H, W, K, R, S, pads, stride, dil = cfg
    rng = np.random.default_rng(seed)
    x = rng.uniform(-1, 1, (N, C, H, W))
    w = rng.uniform(-1, 1, (K, C, R, S))
    kw = dict(pads=pads, stride=stride, dilation=dil)
    return x, w, kw, rng


def _adjoint(lib, cfg, seed=3):
    x, w, kw, rng = _case(cfg, seed)
    y, _ = oracle.conv2d_fprop(x, w, lib=lib, **kw)
    dy = rng.uniform(-1, 1, y.shape)
    dx, _ = oracle.conv2d_dgrad(dy, w, x.shape[2:], lib=lib, **kw)
    dw, _ = oracle.conv2d_wgrad(x, dy, w.shape[2:], lib=lib, **kw)
    a = float((y * dy).sum())
    scale = float(np.abs(y * dy).sum()) + 1e-300
    assert abs(float((x * dx).sum()) - a) <= 1e-12 * scale, "dgrad is not the adjoint of fprop"
    assert abs(float((w * dw).sum()) - a) <= 1e-12 * scale, "wgrad is not the adjoint of fprop"


def _torch(lib, cfg, seed=5):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    x, w, kw, rng = _case(cfg, seed)
    pt, pb, pl, pr = kw["pads"]
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    wt = torch.tensor(w, dtype=torch.float64, requires_grad=True)
    yt = F.conv2d(F.pad(xt, (pl, pr, pt, pb)), wt, stride=kw["stride"], dilation=kw["dilation"])
    dy = rng.uniform(-1, 1, tuple(yt.shape))
    yt.backward(torch.tensor(dy, dtype=torch.float64))
    dx, _ = oracle.conv2d_dgrad(dy, w, x.shape[2:], lib=lib, **kw)
    dw, _ = oracle.conv2d_wgrad(x, dy, w.shape[2:], lib=lib, **kw)
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-12, atol=1e-12)


def _one_by_one(lib):
    rng = np.random.default_rng(11)
    x = rng.uniform(-1, 1, (2, 3, 4, 5))
    w = rng.uniform(-1, 1, (6, 3, 1, 1))
    dy = rng.uniform(-1, 1, (2, 6, 4, 5))
    dx, _ = oracle.conv2d_dgrad(dy, w, (4, 5), lib=lib)
    dw, _ = oracle.conv2d_wgrad(x, dy, (1, 1), lib=lib)
    np.testing.assert_allclose(dx, np.einsum("kc,nkhw->nchw", w[:, :, 0, 0], dy), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dw[:, :, 0, 0], np.einsum("nkhw,nchw->kc", dy, x), rtol=1e-13, atol=1e-13)


def _brute_force_element(lib):
    """dx[n,c,h,w] and its bound from an enumeration of every (k,p,q,r,s)."""
    N, C, H, W, K, R, S = 1, 2, 7, 6, 3, 3, 2
    pads, stride, dil = (1, 2, 0, 1), (2, 2), (2, 1)
    rng = np.random.default_rng(13)
    w = rng.uniform(-1, 1, (K, C, R, S))
    P = (H + pads[0] + pads[1] - dil[0] * (R - 1) - 1) // stride[0] + 1
    Q = (W + pads[2] + pads[3] - dil[1] * (S - 1) - 1) // stride[1] + 1
    dy = rng.uniform(-1, 1, (N, K, P, Q))
    dx, bnd = oracle.conv2d_dgrad(dy, w, (H, W), pads=pads, stride=stride, dilation=dil, lib=lib)
    for (c, h, wi) in [(0, 0, 0), (1, 3, 2), (0, 6, 5), (1, 4, 1)]:
        acc = b = 0.0
        for k in range(K):
            for p in range(P):
                for q in range(Q):
                    for r in range(R):
                        for s in range(S):
                            if (p * stride[0] + r * dil[0] - pads[0] == h
                                    and q * stride[1] + s * dil[1] - pads[2] == wi):
                                acc += dy[0, k, p, q] * w[k, c, r, s]
                                b += abs(dy[0, k, p, q] * w[k, c, r, s])
        assert abs(dx[0, c, h, wi] - acc) <= 1e-13 and abs(bnd[0, c, h, wi] - b) <= 1e-13


def _points(lib):
    """The point evaluators give the full (pinned) gradients at every
    coordinate, listed in a shuffled order."""
    for cfg in (CONFIGS[0], CONFIGS[3]):
        x, w, kw, rng = _case(cfg, 17)
        y, _ = oracle.conv2d_fprop(x, w, lib=lib, **kw)
        dy = rng.uniform(-1, 1, y.shape)
        dx, bx = oracle.conv2d_dgrad(dy, w, x.shape[2:], lib=lib, **kw)
        dw, bw = oracle.conv2d_wgrad(x, dy, w.shape[2:], lib=lib, **kw)
        px = rng.permutation(np.argwhere(np.ones(dx.shape, bool)))
        pw = rng.permutation(np.argwhere(np.ones(dw.shape, bool)))
        v, b = oracle.conv2d_dgrad_points(dy, w, x.shape[2:], px, lib=lib, **kw)
        assert np.array_equal(v, dx[tuple(px.T)]) and np.array_equal(b, bx[tuple(px.T)])
        v, b = oracle.conv2d_wgrad_points(x, dy, w.shape[2:], pw, lib=lib, **kw)
        assert np.array_equal(v, dw[tuple(pw.T)]) and np.array_equal(b, bw[tuple(pw.T)])


PIN_BATTERY = [lambda lib, c=c: _adjoint(lib, c) for c in CONFIGS] + \
              [lambda lib, c=c: _torch(lib, c) for c in CONFIGS] + [_one_by_one, _brute_force_element,
                                                                   _points]


@pytest.mark.parametrize("cfg", CONFIGS, ids=lambda c: "x".join(map(str, c[:7])))
def test_gradients_are_the_adjoint_of_fprop(cfg):
    _adjoint(oracle.load(), cfg)


@pytest.mark.parametrize("cfg", CONFIGS, ids=lambda c: "x".join(map(str, c[:7])))
def test_gradients_match_torch_autograd_fp64(cfg):
    _torch(oracle.load(), cfg)


def test_one_by_one_gradients_are_matrix_products():
    _one_by_one(oracle.load())


def test_dgrad_element_matches_enumeration():
    _brute_force_element(oracle.load())


def test_point_evaluators_match_full_gradients():
    _points(oracle.load())


MUTANTS = {
    "points_coordinate_order": ("i64 a = pts[4 * i], c = pts[4 * i + 1],",
                                "i64 c = pts[4 * i], a = pts[4 * i + 1],"),
    "dgrad_stride_divisibility_dropped": ("if (tp < 0 || tp % g->u != 0)", "if (tp < 0)"),
    "dgrad_dilation_ignored": ("i64 tp = h + g->pt - r * g->dh;", "i64 tp = h + g->pt - r;"),
    "dgrad_pad_side": ("i64 tq = wi + g->pl - s * g->dw;", "i64 tq = wi - g->pl - s * g->dw;"),
    "dgrad_last_output_dropped": ("if (p >= g->P)", "if (p >= g->P - 1)"),
    "wgrad_row_pad_sign": ("i64 h = p * g->u + r * g->dh - g->pt;", "i64 h = p * g->u + r * g->dh + g->pt;"),
    "wgrad_batch_dropped": ("for (i64 n = 0; n < g->N; ++n) {", "for (i64 n = 1; n < g->N; ++n) {"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_gradient_mistake_is_caught(name):
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
