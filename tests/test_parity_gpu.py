"""GPU parity of the C-ABI forward convolution against the CPU oracle.

Small problems are checked element by element (several 128-row tiles, ragged
M and K tails); the full workloads are checked on sampled outputs (65536
random plus all border rows and columns of two images x eight filters) in the
launch configuration the benchmark times.  Guard bands around y catch writes
outside the output; y starts as NaN when beta == 0 so unwritten outputs fail.
"""
import numpy as np
import pytest

from deep_learning_convolution_gb300 import synth
from gpu_util import run_and_check
from window_cases import WINDOW_CASES

pytestmark = pytest.mark.gpu

L = synth.Layer


def P(*a):
    return dict(pad_top=a[0], pad_bottom=a[1], pad_left=a[2], pad_right=a[3])


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


# ---------------------------------------------------------------------------
# strict FP32 (FFMA)
# ---------------------------------------------------------------------------

def test_tiny_fp32_config_full(handle):
    layer = synth.WORKLOADS["tiny"][0]
    assert run_and_check(handle, layer, synth.workload_seed("tiny", 0), full=True,
                         expect_kernel="ffma") == "ffma"


def test_fp32_math_on_bf16_storage_nhwc(handle):
    layer = L("ffma_bf16", 2, 6, 9, 11, 5, 3, 2, **P(1, 0, 2, 1), u=2, dil_w=2, dtype="bf16",
              layout="NHWC")
    # FP32 math requested explicitly through a BF16 layer: use the API directly
    import torch
    from deep_learning_convolution_gb300 import api
    x, w, _ = synth.make_inputs(layer, 5)
    xt, wt = api.layer_tensors(layer, x, w, "cuda")
    n, k, p, q = api.output_dim(xt, wt, x_axes="NHWC", w_axes="KRSC", pads=(1, 0, 2, 1),
                                stride=(2, 1), dilation=(1, 2))
    y = torch.full((n, k, p, q), float("nan"), device="cuda")
    conv = api.Conv2dForward(handle, xt, wt, y, x_axes="NHWC", w_axes="KRSC", y_axes="NCHW",
                             pads=(1, 0, 2, 1), stride=(2, 1), dilation=(1, 2), math="fp32")
    assert conv.kernel(xt, wt, y) == "ffma"
    conv(xt, wt, y)
    torch.cuda.synchronize()
    from oracle import oracle
    ref, bound = oracle.conv2d_fprop(x.astype(np.float64), w.astype(np.float64),
                                     pads=(1, 0, 2, 1), stride=(2, 1), dilation=(1, 2))
    assert (np.abs(y.double().cpu().numpy() - ref) <= 1e-5 * bound + 1e-6).all()


# ---------------------------------------------------------------------------
# tensor cores, TMA im2col producer
# ---------------------------------------------------------------------------

IM2COL_CASES = [
    L("bf16_c64_k96_3x3", 2, 64, 17, 17, 96, 3, 3, **P(1, 1, 1, 1)),
    L("bf16_c96_k256_5x5", 2, 96, 14, 14, 256, 5, 5),
    L("bf16_c64_k40_asym_dil_stride", 3, 64, 19, 23, 40, 3, 2, **P(2, 0, 1, 3), u=2, v=1,
      dil_h=2, dil_w=2),
    L("bf16_c128_k384_1x1", 2, 128, 9, 13, 384, 1, 1),
    L("bf16_c64_k64_1x1_s2", 3, 64, 15, 15, 64, 1, 1, u=2, v=2),
    L("bf16_c192_k130_3x3_s3", 2, 192, 16, 21, 130, 3, 3, **P(1, 1, 1, 1), u=3, v=3),
    L("bf16_c64_k16_7x7_s2_p3", 2, 64, 23, 23, 16, 7, 7, **P(3, 3, 3, 3), u=2, v=2),
    L("tf32_c32_k48_3x3_nhwc", 2, 32, 15, 15, 48, 3, 3, **P(1, 1, 1, 1), dtype="tf32"),
    L("tf32_c64_k96_5x3_nhwc", 2, 64, 12, 10, 96, 5, 3, **P(2, 1, 0, 2), u=1, v=2, dtype="tf32"),
]


@pytest.mark.parametrize("layer", IM2COL_CASES, ids=lambda l: l.name)
def test_tc_im2col_parity_full(handle, layer, monkeypatch):
    monkeypatch.setenv("DLC_TC_PAIR", "0")  # the single-SM kernel
    run_and_check(handle, layer, 1000 + IM2COL_CASES.index(layer), full=True,
                  expect_kernel="tc_im2col")


# the same lowering on pairs of SMs (cta_group::2, M = 256 per MMA)
PAIR_CASES = IM2COL_CASES + [
    # more pair tiles than SM pairs (every cluster runs several), two filter tiles
    L("pair_bf16_c64_k512_3x3_many", 24, 64, 28, 28, 512, 3, 3, **P(1, 1, 1, 1)),
    # ragged: the last pair tile's second CTA has no rows at all
    L("pair_bf16_c64_k64_3x3_ragged", 1, 64, 11, 11, 64, 3, 3, **P(1, 1, 1, 1)),
    # a last channel block with one MMA's worth of channels (BF16 72 = 64 + 8,
    # TF32 40 = 32 + 8): the rest of the block is zero fill
    L("pair_bf16_c72_k64_3x3", 2, 72, 13, 13, 64, 3, 3, **P(1, 1, 1, 1)),
    L("pair_tf32_c40_k32_3x3", 2, 40, 12, 12, 32, 3, 3, **P(1, 1, 1, 1), dtype="tf32"),
]


@pytest.mark.parametrize("bn", [None, 64], ids=["bn_auto", "bn64"])
@pytest.mark.parametrize("layer", PAIR_CASES, ids=lambda l: l.name)
def test_tc_im2col_pair_parity_full(handle, layer, bn, monkeypatch):
    """Direct stores of y from the epilogue registers."""
    monkeypatch.setenv("DLC_TC_PAIR_YTMA", "0")
    if bn:
        monkeypatch.setenv("DLC_TC_PAIR_BN", str(bn))
    run_and_check(handle, layer, 1100 + PAIR_CASES.index(layer), full=True,
                  expect_kernel="tc_im2col_pair")


@pytest.mark.parametrize("epi", ["4", "8"], ids=["epi4", "epi8"])
@pytest.mark.parametrize("layer", [PAIR_CASES[i] for i in (0, 1, 2, 5, 8, 9, 10)],
                         ids=lambda l: l.name)
def test_tc_im2col_pair_bulk_stores(handle, layer, epi, monkeypatch):
    """y written through 2-D bulk tensor stores of 32 x 32 blocks (the default),
    by four epilogue warps or eight (two per TMEM lane quarter, alternate
    32-column chunks)."""
    monkeypatch.setenv("DLC_TC_PAIR_EPI", epi)
    run_and_check(handle, layer, 1150 + PAIR_CASES.index(layer), full=True, with_bias=True,
                  relu=True, expect_kernel="tc_im2col_pair")


@pytest.mark.parametrize("split", ["2", "0"], ids=["split_tail", "whole_tiles"])
@pytest.mark.parametrize("layer", [PAIR_CASES[i] for i in (0, 1, 3, 7, 9, 10)],
                         ids=lambda l: l.name)
def test_tc_im2col_pair_split_tail(handle, layer, split, monkeypatch):
    """Plain epilogue: tiles of the last, mostly idle wave are split along the
    reduction and their partial sums added into y by bulk reduce-adds."""
    monkeypatch.setenv("DLC_TC_PAIR_SPLIT", split)
    run_and_check(handle, layer, 1170 + PAIR_CASES.index(layer), full=True, alpha=0.75,
                  expect_kernel="tc_im2col_pair")


@pytest.mark.parametrize("loaders", ["0", "1", "2"], ids=["one_thread", "a_b_split", "alternate"])
@pytest.mark.parametrize("layer", [PAIR_CASES[i] for i in (0, 3, 9)], ids=lambda l: l.name)
def test_tc_im2col_pair_load_issue(handle, layer, loaders, monkeypatch):
    """The SM-pair kernel's loads issued by one thread, by two (A and B), or by
    two taking alternate k-blocks (DLC_TC_PAIR_SPLITLOAD=0/1/2): the same y."""
    monkeypatch.setenv("DLC_TC_PAIR_SPLITLOAD", loaders)
    run_and_check(handle, layer, 1190 + PAIR_CASES.index(layer), full=True, beta=0.5,
                  expect_kernel="tc_im2col_pair")


@pytest.mark.parametrize("kps", ["2"], ids=["two_kblocks_a_stage"])
@pytest.mark.parametrize("layer", [PAIR_CASES[i] for i in (0, 1, 3, 7, 9, 10)],
                         ids=lambda l: l.name)
def test_tc_im2col_pair_two_kblocks_a_stage(handle, layer, kps, monkeypatch):
    """Two k-blocks per pipeline stage (DLC_TC_PAIR_KPS=2), split tail and whole
    tiles alike, with a unit's odd last k-block alone in its stage (the 96-channel
    case: a full and a 64-byte-row block per tap)."""
    monkeypatch.setenv("DLC_TC_PAIR_KPS", kps)
    run_and_check(handle, layer, 1210 + PAIR_CASES.index(layer), full=True, beta=0.5,
                  with_bias=True, expect_kernel="tc_im2col_pair")


# channel counts whose last 64-channel block holds at most 32 channels: that
# block comes in 64-byte rows (32-channel boxes, two MMAs) unless
# DLC_TC_PAIR_MIXED=0
MIXED_CASES = [
    IM2COL_CASES[1],  # 96 = 64 + 32
    L("pair_bf16_c72_k64_3x3_mixed", 2, 72, 13, 13, 64, 3, 3, **P(1, 1, 1, 1)),
    L("pair_bf16_c160_k96_3x3_s2_mixed", 2, 160, 15, 17, 96, 3, 3, **P(1, 1, 1, 1), u=2, v=2),
    L("pair_bf16_c136_k200_5x5_mixed", 2, 136, 12, 14, 200, 5, 5, **P(2, 1, 0, 3)),
]


@pytest.mark.parametrize("mixed", ["1", "0"], ids=["mixed_last_block", "whole_blocks"])
@pytest.mark.parametrize("layer", MIXED_CASES, ids=lambda l: l.name)
def test_tc_im2col_pair_mixed_last_block(handle, layer, mixed, monkeypatch):
    monkeypatch.setenv("DLC_TC_PAIR_MIXED", mixed)
    seed = 1196 + MIXED_CASES.index(layer)
    run_and_check(handle, layer, seed, full=True, expect_kernel="tc_im2col_pair")
    run_and_check(handle, layer, seed + 10, full=True, alpha=0.5, beta=0.25, with_bias=True,
                  relu=True, expect_kernel="tc_im2col_pair")
    run_and_check(handle, layer, seed + 20, full=True, mode="convolution",
                  expect_kernel="tc_im2col_pair")


def test_tc_im2col_pair_epilogue(handle):
    import torch
    layer = IM2COL_CASES[1]
    run_and_check(handle, layer, 1190, full=True, alpha=-0.5, beta=0.75, with_bias=True,
                  relu=True, expect_kernel="tc_im2col_pair")
    run_and_check(handle, layer, 1191, full=True, y_dtype=torch.bfloat16, beta=0.5,
                  with_bias=True, y_axes="NCHW", expect_kernel="tc_im2col_pair")


# ---------------------------------------------------------------------------
# tensor cores, run-gather producer (NHWC + KRSC runs over (s,c); NCHW + KCRS
# runs over s): the C=3 / C=1 first layers and the NCHW speech layers
# ---------------------------------------------------------------------------

RUN_CASES = [
    L("bf16_c3_k64_11x11_s4_nhwc", 2, 3, 35, 35, 64, 11, 11, **P(2, 2, 2, 2), u=4, v=4),
    L("bf16_c3_k96_11x11_s4_nopad", 2, 3, 39, 43, 96, 11, 11, u=4, v=4),
    L("bf16_c16_k48_3x3_nchw", 2, 16, 14, 18, 48, 3, 3, **P(1, 1, 1, 1), layout="NCHW"),
    L("tf32_c1_k32_21x11_speechlike", 2, 1, 50, 70, 32, 21, 11, **P(10, 10, 5, 5), u=2, v=2,
      dtype="tf32", layout="NCHW"),
    L("tf32_c8_k32_7x5_s2x1_nchw", 2, 8, 27, 40, 32, 7, 5, **P(3, 3, 2, 2), u=2, v=1,
      dtype="tf32", layout="NCHW"),
    L("bf16_c5_k40_4x3_dilh2_nhwc", 3, 5, 17, 16, 40, 4, 3, **P(0, 2, 1, 0), dil_h=2, u=1, v=3),
    L("tf32_c3_k300_3x3_nhwc", 2, 3, 20, 21, 300, 3, 3, **P(1, 1, 1, 1), dtype="tf32"),
    L("bf16_c24_k64_5x5_nhwc", 2, 24, 13, 13, 64, 5, 5, **P(2, 2, 2, 2)),
]


@pytest.mark.parametrize("layer", RUN_CASES, ids=lambda l: l.name)
def test_tc_runs_parity_full(handle, layer, monkeypatch):
    # most of these layers take the window or row-stack kernel by default
    monkeypatch.setenv("DLC_TC_WINDOW", "0")
    monkeypatch.setenv("DLC_TC_ROWSTACK", "0")
    run_and_check(handle, layer, 2000 + RUN_CASES.index(layer), full=True,
                  expect_kernel="tc_runs")


# ---------------------------------------------------------------------------
# tensor cores, row-stack kernel: TF32 channel-planar layers with few filters
# and unit horizontal stride; filters stacked over output rows as M
# ---------------------------------------------------------------------------

ROWSTACK_CASES = [
    # speech layer 2 at N = 2 on a narrower input: 21 x 11 filters, stride 2 x 1
    L("rs_speech2_like", 2, 32, 41, 90, 32, 21, 11, **P(10, 10, 5, 5), u=2, dtype="tf32",
      layout="NCHW"),
    # ragged: 17 channels (a partial group), 3x3 filters (one chunk per channel),
    # Q = 29 (not a multiple of 4), P = 9 (a partial block of 4 rows)
    L("rs_c17_k32_3x3", 3, 17, 9, 29, 32, 3, 3, **P(1, 1, 1, 1), dtype="tf32", layout="NCHW"),
    # 48 filters (two rows of 64 per block), 5x13 filters (4 chunks), stride 3
    L("rs_c19_k48_5x13_s3", 2, 19, 20, 41, 48, 5, 13, **P(2, 0, 6, 3), u=3, dtype="tf32",
      layout="NCHW"),
    # 16 filters, 1x1 (a single tap), several images per tile
    L("rs_c21_k16_1x1", 5, 21, 6, 21, 16, 1, 1, dtype="tf32", layout="NCHW"),
    # 64 filters, 7x12 filters, asymmetric pads, Q = 50
    L("rs_c36_k64_7x12", 2, 36, 15, 55, 64, 7, 12, **P(3, 1, 4, 2), dtype="tf32", layout="NCHW"),
    # a single output row and column per image
    L("rs_c24_k32_3x3_tiny", 3, 24, 3, 3, 32, 3, 3, dtype="tf32", layout="NCHW"),
    # horizontal stride 2 (two phases per unit), one channel (four input rows
    # per stage), a speech-layer-1-like 41x11 filter, Q = 35
    L("rs_c1_k32_41x11_s2", 2, 1, 47, 70, 32, 41, 11, **P(20, 20, 5, 5), u=2, v=2, dtype="tf32",
      layout="NCHW"),
    # two channels (two input rows per stage), stride 1x2, odd width
    L("rs_c2_k16_5x7_s1x2", 3, 2, 13, 37, 16, 5, 7, **P(2, 2, 3, 3), v=2, dtype="tf32",
      layout="NCHW"),
    # three channels and one empty slot, 64 filters, stride 2, 3x5
    L("rs_c3_k64_3x5_s2", 2, 3, 17, 30, 64, 3, 5, **P(1, 1, 2, 2), u=2, v=2, dtype="tf32",
      layout="NCHW"),
    # one channel, stride 1, 48 filters, 7x9
    L("rs_c1_k48_7x9", 2, 1, 20, 33, 48, 7, 9, **P(3, 3, 4, 4), dtype="tf32", layout="NCHW"),
]


@pytest.mark.parametrize("layer", ROWSTACK_CASES, ids=lambda l: l.name)
def test_tc_rowstack_parity_full(handle, layer):
    run_and_check(handle, layer, 2700 + ROWSTACK_CASES.index(layer), full=True,
                  expect_kernel="tc_rowstack")


@pytest.mark.parametrize("layer", ROWSTACK_CASES[:2], ids=lambda l: l.name)
def test_tc_rowstack_epilogue_and_modes(handle, layer):
    import torch
    run_and_check(handle, layer, 2750, full=True, alpha=-0.5, beta=1.25, with_bias=True,
                  relu=True, expect_kernel="tc_rowstack")
    run_and_check(handle, layer, 2751, full=True, y_dtype=torch.bfloat16,
                  expect_kernel="tc_rowstack")
    run_and_check(handle, layer, 2752, full=True, y_axes="NHWC", mode="convolution",
                  expect_kernel="tc_rowstack")


# ---------------------------------------------------------------------------
# tensor cores, window kernel: few channels per horizontal stride step; the
# lowered rows are read in place from a ring of packed input rows
# ---------------------------------------------------------------------------



@pytest.fixture
def no_rowstack(monkeypatch):
    """The window kernel's channel-planar TF32 cases would go to the row-stack
    kernel; these tests keep them on the window kernel."""
    monkeypatch.setenv("DLC_TC_ROWSTACK", "0")


@pytest.mark.parametrize("layer", WINDOW_CASES, ids=lambda l: l.name)
def test_tc_window_parity_full(handle, layer, no_rowstack):
    run_and_check(handle, layer, 2300 + WINDOW_CASES.index(layer), full=True,
                  expect_kernel="tc_window")


@pytest.mark.parametrize("layer", [WINDOW_CASES[i] for i in (4, 5, 6, 10, 14, 18)], ids=lambda l: l.name)
def test_tc_window_word_copies(handle, layer, monkeypatch, no_rowstack):
    """Rows that could be bulk-staged, copied word by word instead."""
    monkeypatch.setenv("DLC_TC_WINSTAGE", "0")
    run_and_check(handle, layer, 2360 + WINDOW_CASES.index(layer), full=True,
                  expect_kernel="tc_window")


@pytest.mark.parametrize("layer", [WINDOW_CASES[i] for i in (0, 2, 5, 7, 12, 13, 15, 16, 17, 18)],
                         ids=lambda l: l.name)
def test_tc_window_cta_pairs(handle, layer, monkeypatch, no_rowstack):
    """CTA pairs sharing each MMA over 256 rows (opt-in)."""
    monkeypatch.setenv("DLC_TC_WINPAIR", "1")
    run_and_check(handle, layer, 2370 + WINDOW_CASES.index(layer), full=True,
                  expect_kernel="tc_window")


@pytest.mark.parametrize("y_axes", ["NCHW", "NHWC"])
def test_tc_window_epilogue(handle, y_axes, no_rowstack):
    import torch
    run_and_check(handle, WINDOW_CASES[0], 2390, full=True, y_axes=y_axes, alpha=-0.5,
                  beta=0.75, with_bias=True, relu=True, expect_kernel="tc_window")
    run_and_check(handle, WINDOW_CASES[4], 2391, full=True, y_axes=y_axes,
                  y_dtype=torch.bfloat16, beta=0.5, with_bias=True, expect_kernel="tc_window")


# ---------------------------------------------------------------------------
# tensor cores, element-gather producer (any strides: dilation along W, KCRS
# filters with NHWC activations, channel-padded views)
# ---------------------------------------------------------------------------

GATHER_CASES = [
    L("bf16_c5_k100_3x3_dil", 2, 5, 13, 12, 100, 3, 3, **P(2, 2, 2, 2), dil_h=2, dil_w=2),
    L("tf32_c16_k32_3x3_dilw3_nchw", 2, 16, 15, 19, 32, 3, 3, **P(1, 1, 3, 3), dil_w=3,
      dtype="tf32", layout="NCHW"),
]


@pytest.mark.parametrize("layer", GATHER_CASES, ids=lambda l: l.name)
def test_tc_gather_parity_full(handle, layer):
    run_and_check(handle, layer, 2500 + GATHER_CASES.index(layer), full=True,
                  expect_kernel="tc_gather")


def test_kcrs_filters_with_nhwc_activations_use_gather(handle):
    layer = L("bf16_nhwc_kcrs", 2, 64, 11, 11, 48, 3, 3, **P(1, 1, 1, 1))
    run_and_check(handle, layer, 77, full=True, w_axes="KCRS", expect_kernel="tc_gather")


@pytest.mark.parametrize("layer,view,kernel", [
    (L("bf16_c64_view", 2, 64, 12, 13, 80, 3, 3, **P(1, 1, 1, 1)), "chan_pad", "tc_im2col"),
    (L("bf16_c64_imgpad", 2, 64, 12, 13, 80, 3, 3, **P(1, 1, 1, 1)), "image_pad", "tc_im2col"),
    (L("bf16_c64_view_pair", 2, 64, 12, 13, 80, 3, 3, **P(1, 1, 1, 1)), "chan_pad",
     "tc_im2col_pair"),
    (L("bf16_c64_imgpad_pair", 2, 64, 12, 13, 80, 3, 3, **P(1, 1, 1, 1)), "image_pad",
     "tc_im2col_pair"),
    (L("bf16_c24_view", 2, 24, 12, 13, 48, 3, 3, **P(1, 1, 1, 1)), "chan_pad", "tc_gather"),
    (L("tf32_nchw_wview", 2, 4, 12, 13, 32, 3, 5, **P(1, 1, 2, 2), dtype="tf32",
       layout="NCHW"), "width_pad", "tc_runs"),
    (L("bf16_c24_view_w", 2, 24, 12, 13, 48, 3, 3, **P(1, 1, 1, 1)), "chan_pad", "tc_window"),
    (L("bf16_c3_imgpad_w", 2, 3, 30, 31, 64, 5, 5, **P(2, 2, 2, 2), u=2, v=2), "image_pad",
     "tc_window"),
    (L("tf32_nchw_wview_w", 2, 4, 12, 13, 32, 3, 5, **P(1, 1, 2, 2), dtype="tf32",
       layout="NCHW"), "width_pad", "tc_window"),
    (L("tf32_nchw_c20_wview_rs", 2, 20, 12, 13, 32, 3, 5, **P(1, 1, 2, 2), dtype="tf32",
       layout="NCHW"), "width_pad", "tc_rowstack"),
    (L("tf32_nchw_c20_imgpad_rs", 2, 20, 12, 13, 32, 3, 5, **P(1, 1, 2, 2), dtype="tf32",
       layout="NCHW"), "image_pad", "tc_rowstack"),
], ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_strided_views(handle, layer, view, kernel, monkeypatch):
    if kernel != "tc_window":
        monkeypatch.setenv("DLC_TC_WINDOW", "0")
    if kernel != "tc_rowstack":
        monkeypatch.setenv("DLC_TC_ROWSTACK", "0")
    if kernel == "tc_im2col":
        monkeypatch.setenv("DLC_TC_PAIR", "0")
    run_and_check(handle, layer, 2600, full=True, view=view, expect_kernel=kernel)


# ---------------------------------------------------------------------------
# stream-K schedule (tiles split between two CTAs, partial parked in y)
# ---------------------------------------------------------------------------

SK_CASES = [
    (L("sk_bf16_c64_k64_70", 4, 64, 70, 70, 64, 3, 3, **P(1, 1, 1, 1)), {}),
    (L("sk_bf16_c64_k300_70", 2, 64, 70, 70, 300, 3, 3, **P(1, 1, 1, 1)), {}),
    (L("sk_tf32_nchw_c16_k32_99", 2, 16, 99, 99, 32, 3, 3, **P(1, 1, 1, 1), dtype="tf32",
       layout="NCHW"), {}),
    (L("sk_bf16_c64_k64_70_epi", 4, 64, 70, 70, 64, 3, 3, **P(1, 1, 1, 1)),
     dict(alpha=0.5, with_bias=True, relu=True)),
    (L("sk_bf16_c64_k64_70_ynchw", 4, 64, 70, 70, 64, 3, 3, **P(1, 1, 1, 1)),
     dict(y_axes="NCHW", with_bias=True)),
]


@pytest.mark.parametrize("layer,kw", SK_CASES, ids=lambda v: v.name if hasattr(v, "name") else "")
def test_stream_k_parity_full(handle, layer, kw, monkeypatch):
    monkeypatch.setenv("DLC_TC_STREAMK", "1")
    monkeypatch.setenv("DLC_TC_WINDOW", "0")
    monkeypatch.setenv("DLC_TC_PAIR", "0")
    run_and_check(handle, layer, 2700 + [c[0] for c in SK_CASES].index(layer), full=True, **kw)


def test_stream_k_is_deterministic_and_flags_reset(handle, monkeypatch):
    """Two launches in a row give bit-identical y (fixed summation order; the
    split-tile flags are consumed and zeroed by each launch)."""
    import torch
    from deep_learning_convolution_gb300 import api
    monkeypatch.setenv("DLC_TC_STREAMK", "1")
    monkeypatch.setenv("DLC_TC_PAIR", "0")
    layer = SK_CASES[0][0]
    x, w, _ = synth.make_inputs(layer, 11)
    xt, wt = api.layer_tensors(layer, x, w, "cuda")
    conv, y = api.layer_problem(handle, layer, xt, wt)
    conv(xt, wt, y)
    y1 = y.clone()
    y.fill_(float("nan"))
    conv(xt, wt, y)
    torch.cuda.synchronize()
    handle.synchronize()
    assert torch.equal(y1, y)
    monkeypatch.setenv("DLC_TC_STREAMK", "0")
    conv(xt, wt, y)
    torch.cuda.synchronize()
    # data-parallel schedule sums in another order: equal within the bound only
    assert torch.allclose(y1, y, rtol=1e-5, atol=1e-4)
    conv.close()


# ---------------------------------------------------------------------------
# seeded sweep of small ragged shapes over both precisions and layouts
# ---------------------------------------------------------------------------

SWEEP = synth.random_small_layers(31, 24, dtypes=("bf16", "tf32"), layouts=("NHWC", "NCHW"))


@pytest.mark.parametrize("layer", SWEEP, ids=lambda l: l.name)
def test_random_sweep_parity(handle, layer):
    run_and_check(handle, layer, 3000 + SWEEP.index(layer), full=True)


# ---------------------------------------------------------------------------
# epilogue: alpha, beta * y, bias, ReLU, BF16 output, other y layouts
# ---------------------------------------------------------------------------

EPI_LAYERS = [IM2COL_CASES[0], RUN_CASES[2], RUN_CASES[3], GATHER_CASES[0], WINDOW_CASES[2]]


@pytest.mark.parametrize("layer", EPI_LAYERS, ids=lambda l: l.name)
@pytest.mark.parametrize("alpha,beta,bias,relu", [
    (0.5, 0.0, True, True), (1.0, -0.75, False, False), (-2.0, 1.5, True, True)])
@pytest.mark.parametrize("window", [True, False], ids=["default", "no_window"])
def test_epilogue_parity(handle, layer, alpha, beta, bias, relu, window, monkeypatch):
    if not window:
        monkeypatch.setenv("DLC_TC_WINDOW", "0")
    run_and_check(handle, layer, 4000, full=True, alpha=alpha, beta=beta, with_bias=bias,
                  relu=relu)


@pytest.mark.parametrize("y_axes", ["NCHW", "NHWC", "CNHW"])
def test_output_layouts(handle, y_axes):
    run_and_check(handle, IM2COL_CASES[2], 4100, full=True, y_axes=y_axes)


def test_bf16_output(handle):
    import torch
    run_and_check(handle, IM2COL_CASES[0], 4200, full=True, y_dtype=torch.bfloat16, beta=0.5,
                  with_bias=True)


# ---------------------------------------------------------------------------
# the benchmark workloads at full size, sampled
# ---------------------------------------------------------------------------

FULL = [(wl, j) for wl in ("alexnet", "overfeat", "resnet50", "speech")
        for j in range(len(synth.WORKLOADS[wl]))]


@pytest.mark.parametrize("wl,j", FULL, ids=lambda v: str(v))
def test_full_workload_layer_sampled(handle, wl, j):
    layer = synth.WORKLOADS[wl][j]
    run_and_check(handle, layer, synth.workload_seed(wl, j), full=False)


# ---------------------------------------------------------------------------
# API behaviour on the device
# ---------------------------------------------------------------------------

def test_workspace_is_zero_and_kernel_choice(handle):
    import torch
    from deep_learning_convolution_gb300 import api
    expect = {"alexnet": ["tc_window"] + ["tc_im2col_pair"] * 4,
              "overfeat": ["tc_window"] + ["tc_im2col_pair"] * 4,
              "resnet50": ["tc_im2col_pair"] * len(synth.WORKLOADS["resnet50"]),
              "speech": ["tc_rowstack", "tc_rowstack"], "tiny": ["ffma"]}
    for wl, kinds in expect.items():
        for layer, kind in zip(synth.WORKLOADS[wl], kinds):
            x, w, _ = synth.make_inputs(layer, 1, batch=1)
            xt, wt = api.layer_tensors(layer, x, w, "cuda")
            conv, y = api.layer_problem(handle, layer, xt, wt)
            assert conv.workspace_size() == 0
            assert conv.kernel(xt, wt, y) == kind, layer.name
            conv.close()


def test_launch_count_and_in_place_rejected(handle):
    import torch
    from deep_learning_convolution_gb300 import api, binding as B
    layer = IM2COL_CASES[0]
    x, w, _ = synth.make_inputs(layer, 9)
    xt, wt = api.layer_tensors(layer, x, w, "cuda")
    conv, y = api.layer_problem(handle, layer, xt, wt)
    before = handle.launches()
    conv(xt, wt, y)
    conv(xt, wt, y)
    assert handle.launches() == before + 2
    # y aliasing x is rejected
    big = torch.zeros(max(xt.numel(), y.numel()) * 2, dtype=torch.float32, device="cuda")
    with pytest.raises(B.DlcError) as e:
        B.dlcConvolutionForward(handle.h, 1.0, conv.x_desc, big.data_ptr(), conv.w_desc,
                                wt.data_ptr(), conv.conv, 0.0, conv.y_desc, big.data_ptr())
    assert e.value.status == B.DLC_STATUS_BAD_PARAM
    torch.cuda.synchronize()


def test_math_dtype_mismatch_not_supported(handle):
    import torch
    from deep_learning_convolution_gb300 import api, binding as B
    x = torch.zeros(1, 8, 8, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(16, 3, 3, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(1, 8, 8, 16, device="cuda")
    conv = api.Conv2dForward(handle, x, w, y, x_axes="NHWC", w_axes="KRSC", y_axes="NHWC",
                             pads=(1, 1, 1, 1), math="tf32")
    with pytest.raises(B.DlcError) as e:
        conv(x, w, y)
    assert e.value.status == B.DLC_STATUS_NOT_SUPPORTED


def test_device_wait_timeout_reports_error_and_recovers(handle):
    """A pipeline wait on a barrier nothing completes runs out after 2 ms;
    the kernel records the error (no fault) and the context stays usable."""
    import torch
    from deep_learning_convolution_gb300 import binding as B
    B.dlcDebugWaitTimeoutSelfTest(handle.h, 2000)
    code, detail = handle.last_device_error()
    assert code == B.DLC_DEVERR_WAIT_TIMEOUT and detail == 99
    # cleared; a pending error blocks launches until read
    B.dlcDebugWaitTimeoutSelfTest(handle.h, 1000)
    torch.cuda.synchronize()
    with pytest.raises(B.DlcError) as e:
        handle.synchronize()
    assert e.value.status == B.DLC_STATUS_EXECUTION_FAILED
    handle.synchronize()  # cleared now
    run_and_check(handle, IM2COL_CASES[0], 5000, full=True)
