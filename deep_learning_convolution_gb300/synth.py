"""Seeded synthetic workloads for the convolution forward pass.

This module is the only code shared by the CUDA path's tests/bench and by the
oracle's tests.  It holds layer shapes, value distributions, seeds and the
rounding of inputs to the storage precision (BF16 or TF32) that both sides
then read.  It holds none of the convolution's arithmetic: no output-size
formula, no index mapping, no summation.

Workload recipe (stand-ins for the networks the cuDNN, maxDNN and batch-reduce
GEMM pages benchmark; no dataset or trained weights are used):

* ``tiny``     : N=2, C=8, 16x16, K=16, 3x3, stride 1, pad 1, NCHW, FP32,
                 x and w ~ U[-1, 1].
* ``alexnet``  : N=128, BF16, NHWC, x ~ N(0,1), w ~ N(0, 1/(C*R*S)).
* ``overfeat`` : N=128, BF16, NHWC (first layer has K=96 filters, not a
                 multiple of 64), same distributions as ``alexnet``.
* ``resnet50`` : N=256, BF16, NHWC, He-init weights w ~ N(0, 2/(C*R*S)).
* ``speech``   : N=32, TF32 math on FP32 storage, NCHW, non-square
                 161 (frequency) x 700 (time) input, x ~ N(0,1).

Seeds: workload i uses ``20260000 + i`` and its layer j uses seed + j
(numpy PCG64).  BF16 values are produced in FP32 and rounded to nearest-even;
TF32 values keep 10 mantissa bits, rounded to nearest-even.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Layer:
    """One forward-convolution problem, in the pages' N,C,H,W / K,C,R,S terms."""

    name: str
    N: int
    C: int
    H: int
    W: int
    K: int
    R: int
    S: int
    pad_top: int = 0
    pad_bottom: int = 0
    pad_left: int = 0
    pad_right: int = 0
    u: int = 1            # vertical stride
    v: int = 1            # horizontal stride
    dil_h: int = 1
    dil_w: int = 1
    dtype: str = "bf16"   # storage/math: "f32" (strict FFMA), "tf32", "bf16"
    layout: str = "NHWC"  # activation layout; filters follow it (KRSC / KCRS)
    x_dist: str = "normal"          # "normal" N(0,1) or "uniform" U[-1,1]
    w_dist: str = "fanin"           # "fanin" N(0,1/CRS), "he" N(0,2/CRS), "uniform"

    def direct_flops(self, P: int, Q: int) -> int:
        """2*N*K*P*Q*C*R*S: the direct-convolution FLOP count (maxDNN's
        efficiency definition); P and Q are supplied by the caller."""
        return 2 * self.N * self.K * P * Q * self.C * self.R * self.S


def _pad(p):
    return dict(pad_top=p, pad_bottom=p, pad_left=p, pad_right=p)


def _layers() -> dict:
    tiny = [Layer("tiny_8x16_3x3", 2, 8, 16, 16, 16, 3, 3, **_pad(1), dtype="f32",
                  layout="NCHW", x_dist="uniform", w_dist="uniform")]
    alex = [
        Layer("alex1_3x64_224_11x11s4", 128, 3, 224, 224, 64, 11, 11, **_pad(2), u=4, v=4),
        Layer("alex2_64x192_27_5x5", 128, 64, 27, 27, 192, 5, 5, **_pad(2)),
        Layer("alex3_192x384_13_3x3", 128, 192, 13, 13, 384, 3, 3, **_pad(1)),
        Layer("alex4_384x256_13_3x3", 128, 384, 13, 13, 256, 3, 3, **_pad(1)),
        Layer("alex5_256x256_13_3x3", 128, 256, 13, 13, 256, 3, 3, **_pad(1)),
    ]
    ovf = [
        Layer("ovf1_3x96_231_11x11s4", 128, 3, 231, 231, 96, 11, 11, u=4, v=4),
        Layer("ovf2_96x256_24_5x5", 128, 96, 24, 24, 256, 5, 5),
        Layer("ovf3_256x512_12_3x3", 128, 256, 12, 12, 512, 3, 3, **_pad(1)),
        Layer("ovf4_512x1024_12_3x3", 128, 512, 12, 12, 1024, 3, 3, **_pad(1)),
        Layer("ovf5_1024x1024_12_3x3", 128, 1024, 12, 12, 1024, 3, 3, **_pad(1)),
    ]
    he = dict(w_dist="he")
    rn = []
    for hw, c in ((56, 64), (28, 128), (14, 256), (7, 512)):
        rn.append(Layer(f"rn_1x1_{hw}_{c}", 256, c, hw, hw, c, 1, 1, **he))
        rn.append(Layer(f"rn_3x3_{hw}_{c}", 256, c, hw, hw, c, 3, 3, **_pad(1), **he))
    for hw, c in ((56, 128), (28, 256), (14, 512)):
        rn.append(Layer(f"rn_3x3s2_{hw}_{c}", 256, c, hw, hw, c, 3, 3, **_pad(1), u=2, v=2, **he))
    for hw, c, k in ((56, 256, 512), (28, 512, 1024), (14, 1024, 2048)):
        rn.append(Layer(f"rn_1x1s2_{hw}_{c}x{k}", 256, c, hw, hw, k, 1, 1, u=2, v=2, **he))
    rn.append(Layer("rn_1x1_56_64x256", 256, 64, 56, 56, 256, 1, 1, **he))
    speech = [
        Layer("speech1_1x32_161x700_41x11", 32, 1, 161, 700, 32, 41, 11, pad_top=20,
              pad_bottom=20, pad_left=5, pad_right=5, u=2, v=2, dtype="tf32", layout="NCHW"),
        # layer 2 reads layer 1's output extent (81 x 350)
        Layer("speech2_32x32_81x350_21x11", 32, 32, 81, 350, 32, 21, 11, pad_top=10,
              pad_bottom=10, pad_left=5, pad_right=5, u=2, v=1, dtype="tf32", layout="NCHW"),
    ]
    return {"tiny": tiny, "alexnet": alex, "overfeat": ovf, "resnet50": rn, "speech": speech}


WORKLOADS = _layers()
WORKLOAD_INDEX = {"tiny": 0, "alexnet": 1, "overfeat": 2, "resnet50": 3, "speech": 4}
SEED_BASE = 20260000


def workload_seed(workload: str, layer_index: int) -> int:
    return SEED_BASE + WORKLOAD_INDEX[workload] + layer_index


# ---------------------------------------------------------------------------
# rounding of inputs to the storage precision (input preparation only)
# ---------------------------------------------------------------------------

def round_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """FP32 -> BF16 bit patterns (uint16), round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return (b >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def round_to_tf32(a: np.ndarray) -> np.ndarray:
    """FP32 -> FP32 holding a TF32 value (low 13 mantissa bits zero), nearest even."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0xFFF + ((b >> 13) & 1)) & ~np.uint64(0x1FFF)
    return b.astype(np.uint32).view(np.float32)


def round_values(a: np.ndarray, dtype: str) -> np.ndarray:
    """Return FP32 values exactly representable in ``dtype`` ("f32", "tf32", "bf16")."""
    a = np.asarray(a, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32(round_to_bf16_bits(a)).reshape(a.shape)
    if dtype == "tf32":
        return round_to_tf32(a).reshape(a.shape)
    if dtype == "f32":
        return a
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# generators
# ---------------------------------------------------------------------------

def _draw(rng: np.random.Generator, shape, dist: str, fan_in: int) -> np.ndarray:
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, size=shape).astype(np.float32)
    if dist == "normal":
        return rng.standard_normal(size=shape, dtype=np.float32)
    if dist == "fanin":
        return (rng.standard_normal(size=shape, dtype=np.float32)
                * np.float32(np.sqrt(1.0 / fan_in)))
    if dist == "he":
        return (rng.standard_normal(size=shape, dtype=np.float32)
                * np.float32(np.sqrt(2.0 / fan_in)))
    raise ValueError(dist)


def make_inputs(layer: Layer, seed: int, batch: Optional[int] = None, with_bias: bool = False):
    """Logical-NCHW x [N,C,H,W] and KCRS w [K,C,R,S] as FP32 arrays already
    rounded to the layer's storage precision; optional bias ~ U[-0.1, 0.1]
    (kept in FP32: the epilogue adds it in FP32).

    ``batch`` overrides N (used for bounded samples of a large workload)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n = layer.N if batch is None else batch
    fan_in = layer.C * layer.R * layer.S
    w = _draw(rng, (layer.K, layer.C, layer.R, layer.S), layer.w_dist, fan_in)
    x = _draw(rng, (n, layer.C, layer.H, layer.W), layer.x_dist, fan_in)
    x = round_values(x, layer.dtype)
    w = round_values(w, layer.dtype)
    bias = None
    if with_bias:
        bias = rng.uniform(-0.1, 0.1, size=(layer.K,)).astype(np.float32)
    return x, w, bias


def random_small_layers(seed: int, count: int, dtypes=("bf16",), layouts=("NHWC",)) -> List[Layer]:
    """A seeded sweep of small, ragged shapes (odd C and K, asymmetric pads,
    strides, dilations) for parity tests."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for i in range(count):
        R = int(rng.integers(1, 6))
        S = int(rng.integers(1, 6))
        dh = int(rng.integers(1, 3))
        dw = int(rng.integers(1, 3))
        u = int(rng.integers(1, 4))
        v = int(rng.integers(1, 4))
        H = int(rng.integers(dh * (R - 1) + 1, 24))
        W = int(rng.integers(dw * (S - 1) + 1, 24))
        out.append(Layer(
            f"rand{seed}_{i}", N=int(rng.integers(1, 4)), C=int(rng.choice([1, 3, 5, 8, 16, 24, 64, 72])),
            H=H, W=W, K=int(rng.choice([1, 8, 16, 40, 96, 100, 130])), R=R, S=S,
            pad_top=int(rng.integers(0, 3)), pad_bottom=int(rng.integers(0, 3)),
            pad_left=int(rng.integers(0, 3)), pad_right=int(rng.integers(0, 3)),
            u=u, v=v, dil_h=dh, dil_w=dw,
            dtype=str(rng.choice(list(dtypes))), layout=str(rng.choice(list(layouts))),
            x_dist="uniform", w_dist="uniform"))
    return out
