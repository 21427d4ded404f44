"""Layers the window kernel takes, shared by its GPU parity tests and the CPU
model of its row ring (test_window_ring.py)."""
from deep_learning_convolution_gb300 import synth

L = synth.Layer


def P(*a):
    return dict(pad_top=a[0], pad_bottom=a[1], pad_left=a[2], pad_right=a[3])


WINDOW_CASES = [
    # 24-byte phase pixels (32-byte swizzled strips), 4-byte copies (pl*C*2 = 12),
    # four output rows per tile
    L("win_bf16_c3_k64_11x11_s4_pad2", 2, 3, 67, 67, 64, 11, 11, **P(2, 2, 2, 2), u=4, v=4),
    # no padding: 8-byte copies; K = 96
    L("win_bf16_c3_k96_11x11_s4_nopad", 2, 3, 99, 99, 96, 11, 11, u=4, v=4),
    # 16-byte phase pixels (no swizzle), wide rows: 150 pixels -> two 128-pixel
    # segments per output row; left pad 2 -> 4-byte copies
    L("win_bf16_c3_k64_7x7_s2_wide", 1, 3, 9, 300, 64, 7, 7, **P(3, 3, 2, 4), u=2, v=2),
    # left pad 3: no aligned copy size, element loads throughout
    L("win_bf16_c3_k64_7x7_s2_pad3", 2, 3, 20, 41, 64, 7, 7, **P(3, 3, 3, 3), u=2, v=2),
    # two output rows per tile (Q + A - 1 = 54), odd P: a half-empty last tile
    L("win_bf16_c8_k32_5x5_two_rows", 2, 8, 25, 50, 32, 5, 5, **P(2, 2, 2, 2)),
    # 64-byte phase pixels (64-byte swizzle), TF32 and BF16
    L("win_tf32_c16_k32_3x3", 2, 16, 19, 23, 32, 3, 3, **P(1, 1, 1, 1), dtype="tf32"),
    L("win_bf16_c24_k64_5x5", 2, 24, 13, 13, 64, 5, 5, **P(2, 2, 2, 2)),
    # K not a multiple of 16 or 32; BN = 208; K = 1
    L("win_bf16_c3_k200_5x5_s2", 2, 3, 31, 29, 200, 5, 5, **P(2, 1, 2, 1), u=2, v=2),
    L("win_bf16_c3_k40_3x3", 2, 3, 17, 17, 40, 3, 3, **P(1, 1, 1, 1)),
    L("win_bf16_c1_k1_3x3", 2, 1, 17, 17, 1, 3, 3, **P(1, 1, 1, 1)),
    # vertical stride and dilation, asymmetric pads
    L("win_bf16_c8_k48_3x3_s2x1", 2, 8, 21, 22, 48, 3, 3, **P(0, 2, 1, 0), u=2),
    L("win_bf16_c5_k40_4x3_dilh2_s3", 3, 5, 17, 16, 40, 4, 3, **P(0, 2, 1, 0), dil_h=2, v=3),
    # NCHW activations: C = 1 (contiguous phase pixels), C = 8 (element loads)
    L("win_tf32_c1_k32_21x11_s2_nchw", 2, 1, 50, 70, 32, 21, 11, **P(10, 10, 5, 5), u=2, v=2,
      dtype="tf32", layout="NCHW"),
    L("win_tf32_c8_k32_7x5_s2x1_nchw", 2, 8, 27, 40, 32, 7, 5, **P(3, 3, 2, 2), u=2, v=1,
      dtype="tf32", layout="NCHW"),
    # 1x1 filters, more tiles than SMs
    L("win_bf16_c4_k16_1x1_many", 40, 4, 30, 30, 16, 1, 1),
    # an odd number of tiles (5): the last CTA pair has one tile
    L("win_bf16_c3_k64_11x11_s4_odd_tiles", 1, 3, 75, 67, 64, 11, 11, **P(2, 2, 2, 2), u=4, v=4),
    # a single tile: one CTA, no pair
    L("win_bf16_c3_k32_5x5_one_tile", 1, 3, 9, 9, 32, 5, 5, **P(2, 2, 2, 2)),
    # wide rows of 64-byte phase pixels and 9 filter rows: the ring of 2*kspan
    # slots does not fit beside the filters, so the short ring (kspan + 1
    # slots) runs, where a tile that starts a new image waits for the MMAs of
    # the tile before it
    L("win_bf16_c24_k64_9x3_wide_short_ring", 19, 24, 12, 150, 64, 9, 3, **P(4, 4, 1, 1)),
    # wide rows (one output row per tile) whose input rows are staged by bulk
    # copies: 224 pixels x 3 channels = 1344-byte rows, 7x7 stride 2 (D = 16),
    # left pad 2 so phase pixels start on 4-byte boundaries
    L("win_bf16_c3_k64_7x7_s2_wide_staged", 2, 3, 20, 224, 64, 7, 7, **P(3, 3, 2, 4), u=2, v=2),
    # OverFeat's first layer at N = 8: 1386-byte rows (2 bytes past a word on
    # every other row), staged as the 16-byte-aligned superset and repacked
    # shifted
    L("win_bf16_c3_k96_11x11_s4_ovf_shifted", 8, 3, 231, 231, 96, 11, 11, u=4, v=4),
    # left pad 3 and odd rows on the shifted staging: 3*2*3 = 18 bytes of
    # padding before a phase pixel
    L("win_bf16_c3_k64_7x7_s2_shifted_pad3", 4, 3, 21, 41, 64, 7, 7, **P(3, 3, 3, 3), u=2, v=2),
]
