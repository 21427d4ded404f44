"""Host-side tests of the C ABI (no GPU): the library builds and loads,
exports every function include/dlc.h declares, and its descriptor layer
validates problems and computes output sizes like the oracle's definition."""
import ctypes
import os
import re

import numpy as np
import pytest

from deep_learning_convolution_gb300 import binding as B
from deep_learning_convolution_gb300 import build as dlc_build
from oracle import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dlc_build.build()
    return B.load_library()


def header_functions():
    text = open(os.path.join(ROOT, "include", "dlc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dlc[A-Za-z0-9_]+)\s*\(", text)))


def test_header_functions_are_exported(lib):
    names = header_functions()
    assert len(names) >= 25
    for n in names:
        assert hasattr(lib, n), f"{n} declared in dlc.h but not exported"
    # and the binding covers exactly the header
    assert sorted(B.SIGNATURES) == names


def test_exports_are_c_linkage(lib):
    # C linkage: plain symbol names resolve via dlsym
    for n in header_functions():
        ctypes.cast(getattr(lib, n), ctypes.c_void_p)


def test_version_and_error_strings(lib):
    assert B.dlcGetVersion() == 100
    assert B.dlcGetErrorString(B.DLC_STATUS_BAD_PARAM) == "DLC_STATUS_BAD_PARAM"
    assert B.dlcGetErrorString(99) == "DLC_STATUS_UNKNOWN"


def _descs(n=2, c=8, h=16, w=16, k=16, r=3, s=3, fmt=B.DLC_TENSOR_NCHW, dt=B.DLC_DATA_FLOAT):
    xd = B.dlcCreateTensorDescriptor()
    B.dlcSetTensor4dDescriptor(xd, fmt, dt, n, c, h, w)
    wd = B.dlcCreateFilterDescriptor()
    B.dlcSetFilter4dDescriptor(wd, dt, fmt, k, c, r, s)
    cd = B.dlcCreateConvolutionDescriptor()
    return xd, wd, cd


def test_output_dim_matches_oracle_definition(lib):
    rng = np.random.default_rng(0)
    olib = oracle.load()
    for _ in range(300):
        H, W = int(rng.integers(1, 40)), int(rng.integers(1, 40))
        R, S = int(rng.integers(1, 8)), int(rng.integers(1, 8))
        pads = [int(p) for p in rng.integers(0, 5, size=4)]
        u, v = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        dh, dw = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        xd, wd, cd = _descs(h=H, w=W, r=R, s=S)
        B.dlcSetConvolution2dDescriptor(cd, 0, 0, u, v, dh, dw, B.DLC_MATH_FP32)
        B.dlcSetConvolution2dPadding(cd, *pads)
        P = oracle.out_extent(H, pads[0], pads[1], R, dh, u, olib)
        Q = oracle.out_extent(W, pads[2], pads[3], S, dw, v, olib)
        if P < 1 or Q < 1:
            with pytest.raises(B.DlcError) as e:
                B.dlcGetConvolution2dForwardOutputDim(cd, xd, wd)
            assert e.value.status == B.DLC_STATUS_BAD_PARAM
        else:
            assert B.dlcGetConvolution2dForwardOutputDim(cd, xd, wd) == (2, 16, P, Q)
        for d, f in ((xd, B.dlcDestroyTensorDescriptor), (wd, B.dlcDestroyFilterDescriptor),
                     (cd, B.dlcDestroyConvolutionDescriptor)):
            f(d)


def test_descriptor_round_trip(lib):
    xd = B.dlcCreateTensorDescriptor()
    B.dlcSetTensor4dDescriptor(xd, B.DLC_TENSOR_NHWC, B.DLC_DATA_BFLOAT16, 2, 3, 5, 7)
    assert B.dlcGetTensor4dDescriptor(xd) == (B.DLC_DATA_BFLOAT16, 2, 3, 5, 7, 105, 1, 21, 3)
    B.dlcSetTensor4dDescriptor(xd, B.DLC_TENSOR_NCHW, B.DLC_DATA_FLOAT, 2, 3, 5, 7)
    assert B.dlcGetTensor4dDescriptor(xd) == (B.DLC_DATA_FLOAT, 2, 3, 5, 7, 105, 35, 7, 1)
    wd = B.dlcCreateFilterDescriptor()
    B.dlcSetFilter4dDescriptor(wd, B.DLC_DATA_FLOAT, B.DLC_TENSOR_NHWC, 4, 3, 2, 1)
    assert B.dlcGetFilter4dDescriptor(wd) == (B.DLC_DATA_FLOAT, B.DLC_TENSOR_NHWC, 4, 3, 2, 1)
    cd = B.dlcCreateConvolutionDescriptor()
    B.dlcSetConvolution2dDescriptor(cd, 1, 2, 3, 4, 2, 1, B.DLC_MATH_TF32)
    assert B.dlcGetConvolution2dDescriptor(cd) == (1, 1, 2, 2, 3, 4, 2, 1, B.DLC_MATH_TF32)
    B.dlcSetConvolution2dPadding(cd, 0, 5, 6, 7)
    assert B.dlcGetConvolution2dDescriptor(cd)[:4] == (0, 5, 6, 7)


@pytest.mark.parametrize("call", [
    lambda d: B.dlcSetTensor4dDescriptor(d, B.DLC_TENSOR_NCHW, B.DLC_DATA_FLOAT, 0, 1, 1, 1),
    lambda d: B.dlcSetTensor4dDescriptor(d, 7, B.DLC_DATA_FLOAT, 1, 1, 1, 1),
    lambda d: B.dlcSetTensor4dDescriptor(d, B.DLC_TENSOR_NCHW, 9, 1, 1, 1, 1),
    lambda d: B.dlcSetTensor4dDescriptorEx(d, B.DLC_DATA_FLOAT, 1, 1, 1, 1, -1, 1, 1, 1),
])
def test_bad_tensor_descriptors(lib, call):
    d = B.dlcCreateTensorDescriptor()
    with pytest.raises(B.DlcError) as e:
        call(d)
    assert e.value.status == B.DLC_STATUS_BAD_PARAM
    B.dlcDestroyTensorDescriptor(d)


def test_bad_convolution_descriptors(lib):
    cd = B.dlcCreateConvolutionDescriptor()
    for args in ((-1, 0, 1, 1, 1, 1, 0), (0, 0, 0, 1, 1, 1, 0), (0, 0, 1, 1, 0, 1, 0),
                 (0, 0, 1, 1, 1, 1, 7)):
        with pytest.raises(B.DlcError):
            B.dlcSetConvolution2dDescriptor(cd, *args)
    with pytest.raises(B.DlcError) as e:  # padding before the descriptor was set
        B.dlcSetConvolution2dPadding(cd, 0, 0, 0, 0)
    assert e.value.status == B.DLC_STATUS_NOT_INITIALIZED


def test_channel_mismatch_rejected(lib):
    xd, wd, cd = _descs()
    B.dlcSetFilter4dDescriptor(wd, B.DLC_DATA_FLOAT, B.DLC_TENSOR_NCHW, 16, 9, 3, 3)
    B.dlcSetConvolution2dDescriptor(cd, 1, 1, 1, 1, 1, 1, B.DLC_MATH_FP32)
    with pytest.raises(B.DlcError) as e:
        B.dlcGetConvolution2dForwardOutputDim(cd, xd, wd)
    assert e.value.status == B.DLC_STATUS_BAD_PARAM


def test_null_handle_is_not_initialized(lib):
    st = lib.dlcSynchronize(None)
    assert st == B.DLC_STATUS_NOT_INITIALIZED
    st = lib.dlcConvolutionForward(None, None, None, None, None, None, None, None, None, None)
    assert st == B.DLC_STATUS_NOT_INITIALIZED


def test_product_path_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "deep_learning_convolution_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle", text, re.M), f
                assert "conv_oracle" not in text and "oracle_conv2d" not in text, f
    text = open(os.path.join(ROOT, "include", "dlc.h")).read()
    assert "oracle" not in text.lower()
