/*
 * dlc.h -- C ABI of the GB300 (sm_103a) 2-D convolution library: the forward
 * convolution, its two backward routines, pooling and activation forward.
 *
 * The forward (FPROP) convolution layer is
 *
 *   y[n,k,p,q] = act( alpha * sum_{c,r,s} x[n, c, p*u + r*dh - pad_top, q*v + s*dw - pad_left]
 *                                         * w[k,c,r,s]
 *                     + beta * y[n,k,p,q] + bias[k] )
 *
 * (cross-correlation; x reads as zero outside the image; act is identity or
 * ReLU), with P = floor((H + pad_top + pad_bottom - dh*(R-1) - 1) / u) + 1 and
 * Q likewise along W.
 *
 * Sources on the pages:
 *  - "cuDNN: Efficient Primitives for Deep Learning", method section: a C
 *    language API whose tensors and filters are opaque descriptors with
 *    arbitrary strides and layouts; the caller owns every device buffer and no
 *    auxiliary buffer is used; non-square inputs and asymmetric padding are
 *    supported (findings section).
 *  - "maxDNN: An Efficient Convolution Kernel for Deep Learning with Maxwell
 *    GPUs", method section: each output coordinate is the product of the input
 *    receptive field with the filter weights; efficiency counts only the
 *    direct-convolution FLOPs 2*N*K*P*Q*C*R*S.
 *  - "High-Performance Deep Learning via a Single Building Block", method
 *    section: the kernel is a batch-reduce GEMM, C += sum_i A_i * B_i, here
 *    with i running over the filter taps (r,s) and channel blocks.
 *  - "High Performance Zero-Memory Overhead Direct Convolutions", abstract and
 *    method section: no packing and no extra memory -- the workspace size is
 *    always 0.
 *
 * Conventions (all functions):
 *  - Every function returns a dlcStatus_t.  Pointers to descriptors and
 *    handles are host pointers; x, w, y and bias are device pointers owned by
 *    the caller; alpha and beta are host pointers to float.
 *  - Sizes and strides are in elements, not bytes.
 *  - Calls that launch work are asynchronous on the handle's stream.  Launch
 *    errors are reported by the call itself.  Errors that kernels detect on
 *    the device (a pipeline wait that ran out of time) are recorded in the
 *    handle and reported as DLC_STATUS_EXECUTION_FAILED by the next launching
 *    call on that handle and by dlcSynchronize(), which clears them.
 *  - The library allocates no device memory on any forward or backward call.
 *    dlcCreate allocates one small mapped host word for device error
 *    reports, the split-tile flags and a 2 MiB device buffer where calls of
 *    the few-channel kernels repack the filters before the convolution reads
 *    them (so two calls on one handle must not overlap on the GPU: use one
 *    handle per stream).  This buffer departs from the cuDNN page's "no
 *    auxiliary buffers"; the caller-visible workspace is zero.
 *  - A handle is not thread-safe; use one handle per host thread.
 */
#ifndef DLC_H_
#define DLC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DLC_VERSION 100

typedef enum {
    DLC_STATUS_SUCCESS = 0,
    DLC_STATUS_NOT_INITIALIZED = 1,   /* handle or descriptor not created/set */
    DLC_STATUS_BAD_PARAM = 2,         /* shape, stride, pointer or size error */
    DLC_STATUS_NOT_SUPPORTED = 3,     /* valid request this library does not offer */
    DLC_STATUS_EXECUTION_FAILED = 4,  /* launch failed or a kernel reported an error */
    DLC_STATUS_INTERNAL_ERROR = 5,
    DLC_STATUS_ALLOC_FAILED = 6       /* host allocation failed */
} dlcStatus_t;

/* Storage type of x, w and y.  x and w must share it; y may be FLOAT or
 * BFLOAT16 independently (DOUBLE with DOUBLE inputs).  Bias is always FLOAT. */
typedef enum {
    DLC_DATA_FLOAT = 0,
    DLC_DATA_BFLOAT16 = 1,
    DLC_DATA_DOUBLE = 2
} dlcDataType_t;

/* Layouts.  For activations NCHW / NHWC; for filters NCHW means KCRS and NHWC
 * means KRSC. */
typedef enum {
    DLC_TENSOR_NCHW = 0,
    DLC_TENSOR_NHWC = 1
} dlcTensorFormat_t;

/* Arithmetic.  FP32: FP32 products and sums on CUDA cores (FFMA), FLOAT or
 * BFLOAT16 storage.  TF32: tensor cores, FLOAT storage read as TF32, FP32
 * accumulation.  BF16: tensor cores, BFLOAT16 storage, FP32 accumulation.
 * FP64: double-precision products and sums on CUDA cores (DFMA), DOUBLE
 * storage throughout (the cuDNN page's method section: routines in single and
 * double precision). */
typedef enum {
    DLC_MATH_FP32 = 0,
    DLC_MATH_TF32 = 1,
    DLC_MATH_BF16 = 2,
    DLC_MATH_FP64 = 3
} dlcMathType_t;

/* Filter orientation (cuDNN page, method section).  CROSS_CORRELATION sums
 * x[.., p*u + r*dh - pad_top, ..] * w[k,c,r,s] (the default, the formula at the
 * top of this file); CONVOLUTION mirrors the filter taps, w[k,c,R-1-r,S-1-s]. */
typedef enum {
    DLC_CROSS_CORRELATION = 0,
    DLC_CONVOLUTION = 1
} dlcConvolutionMode_t;

/* Activation functions (cuDNN page, summary and method section).  The fused
 * convolution epilogue takes IDENTITY and RELU; dlcActivationForward takes
 * every mode: f(x) = x, max(0, x), 1 / (1 + e^-x), tanh x, min(max(0, x), coef). */
typedef enum {
    DLC_ACTIVATION_IDENTITY = 0,
    DLC_ACTIVATION_RELU = 1,
    DLC_ACTIVATION_SIGMOID = 2,
    DLC_ACTIVATION_TANH = 3,
    DLC_ACTIVATION_CLIPPED_RELU = 4
} dlcActivationMode_t;

/* Pooling (cuDNN page, summary and method section): the largest value of the
 * window's in-image elements, or their sum divided by the window size (the
 * padding counts as zeros) or by their number (the padding is excluded). */
typedef enum {
    DLC_POOLING_MAX = 0,
    DLC_POOLING_AVERAGE_COUNT_INCLUDE_PADDING = 1,
    DLC_POOLING_AVERAGE_COUNT_EXCLUDE_PADDING = 2
} dlcPoolingMode_t;

/* Which kernel a forward call launches (diagnostic). */
typedef enum {
    DLC_KERNEL_NONE = 0,
    DLC_KERNEL_FFMA = 1,          /* strict FP32 direct convolution, CUDA cores */
    DLC_KERNEL_TC_IM2COL = 2,     /* tcgen05 implicit GEMM, TMA im2col activations */
    DLC_KERNEL_TC_GATHER = 3,     /* tcgen05 implicit GEMM, element-gathered operands */
    DLC_KERNEL_TC_GATHER_RUNS = 4, /* tcgen05 implicit GEMM, operands gathered as contiguous
                                     runs: (s,c) of a filter row for NHWC + KRSC, s of a
                                     (c,r) pair for NCHW + KCRS */
    DLC_KERNEL_TC_WINDOW = 5,     /* tcgen05 implicit GEMM for few channels per stride step
                                     (v*C*element size <= 64 bytes, no horizontal dilation,
                                     K <= 256): lowered rows read in place from packed input
                                     rows in shared memory */
    DLC_KERNEL_TC_IM2COL_PAIR = 6, /* the TC_IM2COL lowering on pairs of SMs (a cluster of two
                                     CTAs shares each MMA of 256 output pixels; each CTA
                                     loads half of the filter tile) */
    DLC_KERNEL_DIRECT = 7,        /* backward routines and pooling: one output element per
                                     thread, CUDA cores, any strides */
    DLC_KERNEL_TC_WGRAD = 8,      /* filter gradient on the tensor cores: pixels as the
                                     reduction, both operands MN-major from TMA */
    DLC_KERNEL_POOL_NHWC = 9,     /* pooling with channels innermost: 16-byte vectors of
                                     channels per thread */
    DLC_KERNEL_TC_ROWSTACK = 10   /* TF32, channel-planar (NCHW) x, unit horizontal stride,
                                     up to 64 filters: filters stacked over output rows as the
                                     MMA's M side, output pixels (per phase q mod 4) as N,
                                     read in place from shifted copies of input rows */
} dlcKernel_t;

/* Device error codes recorded by kernels (dlcGetLastDeviceError). */
typedef enum {
    DLC_DEVERR_NONE = 0,
    DLC_DEVERR_WAIT_TIMEOUT = 1   /* a pipeline barrier wait ran out of time */
} dlcDeviceError_t;

typedef struct dlcContext *dlcHandle_t;
typedef struct dlcTensorStruct *dlcTensorDescriptor_t;
typedef struct dlcFilterStruct *dlcFilterDescriptor_t;
typedef struct dlcConvolutionStruct *dlcConvolutionDescriptor_t;
typedef struct dlcPoolingStruct *dlcPoolingDescriptor_t;

/* ---- library ------------------------------------------------------------ */

/* Human-readable name of a status code; never NULL. */
const char *dlcGetErrorString(dlcStatus_t status);

/* DLC_VERSION of the loaded library, written to *version. */
dlcStatus_t dlcGetVersion(int *version);

/* ---- handle ------------------------------------------------------------- */

/* Creates a handle bound to the current CUDA device and the legacy default
 * stream.  Allocates the host-side context, one mapped host word for
 * device error reports, the split-tile flags and the 2 MiB filter-repacking
 * buffer.  BAD_PARAM if handle is NULL, NOT_SUPPORTED if the
 * device is not compute capability 10.3, EXECUTION_FAILED on a CUDA error.
 * Source: cuDNN page, method section (a C library whose calls take a context
 * created once and bound to a stream). */
dlcStatus_t dlcCreate(dlcHandle_t *handle);

/* Frees the handle (does not synchronize; the caller must ensure no launched
 * work is still pending). */
dlcStatus_t dlcDestroy(dlcHandle_t handle);

/* Sets the stream (a cudaStream_t passed as void*; NULL = legacy default
 * stream) on which later calls launch.  Source: cuDNN page, method section
 * (the library runs on the caller's stream). */
dlcStatus_t dlcSetStream(dlcHandle_t handle, void *stream);
dlcStatus_t dlcGetStream(dlcHandle_t handle, void **stream);

/* Bitwise reproducibility.  By default (0) the SM-pair kernel splits the
 * output tiles of a launch's last, mostly idle wave along the reduction and
 * adds the partial sums into y with FP32 atomic adds, whose order varies from
 * run to run: those outputs can differ in their last bits between runs (each
 * run stays within the same error bound).  With deterministic = 1 every
 * kernel sums each output in a fixed order, so repeated calls give identical
 * bits, at the cost of the idle tail (a few microseconds per launch).
 * BAD_PARAM unless deterministic is 0 or 1.  No counterpart on the pages
 * (they are silent on reproducibility). */
dlcStatus_t dlcSetDeterministic(dlcHandle_t handle, int deterministic);
dlcStatus_t dlcGetDeterministic(dlcHandle_t handle, int *deterministic);

/* Synchronizes the handle's stream.  Returns EXECUTION_FAILED if a kernel
 * recorded a device error since the last call (the error is then cleared).
 * No counterpart on the pages: the bounded-wait failure report. */
dlcStatus_t dlcSynchronize(dlcHandle_t handle);

/* Synchronizes, then writes the last recorded device error code
 * (dlcDeviceError_t) and its detail word (which wait gave up) and clears
 * them. */
dlcStatus_t dlcGetLastDeviceError(dlcHandle_t handle, int *code, int *detail);

/* Number of kernels this handle has launched since creation. */
dlcStatus_t dlcGetLaunchCount(dlcHandle_t handle, uint64_t *count);

/* ---- tensor descriptors (x and y) ---------------------------------------- */

dlcStatus_t dlcCreateTensorDescriptor(dlcTensorDescriptor_t *desc);
dlcStatus_t dlcDestroyTensorDescriptor(dlcTensorDescriptor_t desc);

/* Dense 4-D tensor in NCHW or NHWC order.  All sizes must be >= 1 and the
 * element count must fit in 63 bits.  Source: cuDNN page, method section
 * (opaque tensor descriptors; NCHW and NHWC both supported) and findings
 * section (non-square images). */
dlcStatus_t dlcSetTensor4dDescriptor(dlcTensorDescriptor_t desc, dlcTensorFormat_t format,
                                     dlcDataType_t dtype, int n, int c, int h, int w);

/* 4-D tensor with arbitrary non-negative strides (elements) for the logical
 * axes n, c, h, w: any layout, including sub-tensor views.  Source: cuDNN
 * page, method section (arbitrary strides along each dimension). */
dlcStatus_t dlcSetTensor4dDescriptorEx(dlcTensorDescriptor_t desc, dlcDataType_t dtype,
                                       int n, int c, int h, int w,
                                       int64_t nStride, int64_t cStride,
                                       int64_t hStride, int64_t wStride);

dlcStatus_t dlcGetTensor4dDescriptor(dlcTensorDescriptor_t desc, dlcDataType_t *dtype,
                                     int *n, int *c, int *h, int *w,
                                     int64_t *nStride, int64_t *cStride,
                                     int64_t *hStride, int64_t *wStride);

/* ---- filter descriptors (w) ---------------------------------------------- */

dlcStatus_t dlcCreateFilterDescriptor(dlcFilterDescriptor_t *desc);
dlcStatus_t dlcDestroyFilterDescriptor(dlcFilterDescriptor_t desc);

/* Dense K x C x R x S filter bank; format NCHW = KCRS, NHWC = KRSC.
 * Source: cuDNN page, method section (filter descriptors beside the tensor
 * descriptors; the filter layout follows the data layout). */
dlcStatus_t dlcSetFilter4dDescriptor(dlcFilterDescriptor_t desc, dlcDataType_t dtype,
                                     dlcTensorFormat_t format, int k, int c, int r, int s);

dlcStatus_t dlcGetFilter4dDescriptor(dlcFilterDescriptor_t desc, dlcDataType_t *dtype,
                                     dlcTensorFormat_t *format, int *k, int *c, int *r, int *s);

/* ---- convolution descriptors --------------------------------------------- */

dlcStatus_t dlcCreateConvolutionDescriptor(dlcConvolutionDescriptor_t *desc);
dlcStatus_t dlcDestroyConvolutionDescriptor(dlcConvolutionDescriptor_t desc);

/* Symmetric padding pad_h (top and bottom) and pad_w (left and right),
 * strides u (vertical) and v (horizontal), dilations, arithmetic.  Pads >= 0,
 * strides and dilations >= 1.  Source: cuDNN page, method section (padding
 * and strides of the convolution descriptor); maxDNN page, method section
 * (the arithmetic counted as direct-convolution FLOPs); dilation enters as
 * r*dh, s*dw (the pages are silent: the common convention). */
dlcStatus_t dlcSetConvolution2dDescriptor(dlcConvolutionDescriptor_t desc, int pad_h, int pad_w,
                                          int u, int v, int dilation_h, int dilation_w,
                                          dlcMathType_t math);

/* Asymmetric padding (replaces the symmetric pads).  Source: cuDNN page,
 * findings section (asymmetric padding). */
dlcStatus_t dlcSetConvolution2dPadding(dlcConvolutionDescriptor_t desc, int pad_top,
                                       int pad_bottom, int pad_left, int pad_right);

dlcStatus_t dlcGetConvolution2dDescriptor(dlcConvolutionDescriptor_t desc, int *pad_top,
                                          int *pad_bottom, int *pad_left, int *pad_right,
                                          int *u, int *v, int *dilation_h, int *dilation_w,
                                          dlcMathType_t *math);

/* Filter orientation (default CROSS_CORRELATION).  BAD_PARAM for another
 * value; NOT_INITIALIZED before dlcSetConvolution2dDescriptor.  Source: cuDNN
 * page, method section (both convolution and cross-correlation; CONVOLUTION
 * mirrors the filter taps in both axes). */
dlcStatus_t dlcSetConvolutionMode(dlcConvolutionDescriptor_t desc, dlcConvolutionMode_t mode);
dlcStatus_t dlcGetConvolutionMode(dlcConvolutionDescriptor_t desc, dlcConvolutionMode_t *mode);

/* ---- forward convolution ------------------------------------------------- */

/* Output dimensions N, K, P, Q.  BAD_PARAM if C differs between x and w or
 * if the dilated filter does not fit the padded input (P or Q < 1).  Source:
 * maxDNN page, method section (one output per receptive-field position; a
 * partial last window is dropped: the floor above). */
dlcStatus_t dlcGetConvolution2dForwardOutputDim(dlcConvolutionDescriptor_t conv,
                                                dlcTensorDescriptor_t xDesc,
                                                dlcFilterDescriptor_t wDesc,
                                                int *n, int *k, int *p, int *q);

/* Workspace needed by dlcConvolutionForward: always 0 bytes (zero memory
 * overhead).  Validates the problem like the forward call.  Source:
 * zero-memory-overhead page, abstract; cuDNN page, method section (no
 * auxiliary buffers). */
dlcStatus_t dlcGetConvolutionForwardWorkspaceSize(dlcHandle_t handle,
                                                  dlcTensorDescriptor_t xDesc,
                                                  dlcFilterDescriptor_t wDesc,
                                                  dlcConvolutionDescriptor_t conv,
                                                  dlcTensorDescriptor_t yDesc, size_t *bytes);

/* Kernel a forward call with these descriptors and pointers would launch;
 * x, w and y may be NULL (alignment is then taken as satisfied).  No
 * counterpart on the pages (a diagnostic). */
dlcStatus_t dlcGetConvolutionForwardKernel(dlcHandle_t handle,
                                           dlcTensorDescriptor_t xDesc, const void *x,
                                           dlcFilterDescriptor_t wDesc, const void *w,
                                           dlcConvolutionDescriptor_t conv,
                                           dlcTensorDescriptor_t yDesc, const void *y,
                                           dlcKernel_t *kernel);

/* y = alpha * conv(x, w) + beta * y.
 * x: device, xDesc layout; w: device, wDesc layout; y: device, yDesc layout
 * with dims (N, K, P, Q) and strides that map distinct elements to distinct
 * addresses.  beta == 0 means y is not read (NaN in y is overwritten).
 * y must not overlap x or w (BAD_PARAM).  x and w must share a storage type
 * that matches the math mode: FP32 math takes FLOAT or BFLOAT16, TF32 math
 * takes FLOAT, BF16 math takes BFLOAT16 (else NOT_SUPPORTED).
 * Non-finite inputs: x and w are expected finite.  An Inf or NaN in x reaches
 * every output whose receptive field holds it, as the sum defines; the
 * few-channel kernel (DLC_KERNEL_TC_WINDOW) also multiplies zero filter taps
 * with the input pixels just outside a window that share its packed phase
 * pixel, so there an output beside such a window can read NaN as well (same
 * image, rows whose window holds the pixel, within one stride step plus one
 * phase pixel of its column).  The row-stack kernel (DLC_KERNEL_TC_ROWSTACK)
 * likewise multiplies zero filter taps with input pixels up to 3 columns past
 * a window and with input rows of its block of output rows that a given
 * output row does not read (for one-channel layers also up to 3 input rows
 * past the block's span): there an output of the same image, within that
 * block of rows and within 4 horizontal strides of such a pixel, can read
 * NaN.  Every other kernel reads exactly each window.
 * Sources: maxDNN page, method section (each output is its receptive field
 * times the filter weights); cuDNN page, method section (C API, descriptors
 * with arbitrary strides, caller-owned buffers). */
dlcStatus_t dlcConvolutionForward(dlcHandle_t handle, const float *alpha,
                                  dlcTensorDescriptor_t xDesc, const void *x,
                                  dlcFilterDescriptor_t wDesc, const void *w,
                                  dlcConvolutionDescriptor_t conv, const float *beta,
                                  dlcTensorDescriptor_t yDesc, void *y);

/* y = act(alpha * conv(x, w) + beta * y + bias[k]); bias is a device array of
 * K floats or NULL (no bias).  Otherwise as dlcConvolutionForward.  Source:
 * the layer's epilogue (bias and activation after the sum); cuDNN page,
 * method section (activation functions beside the convolution). */
dlcStatus_t dlcConvolutionBiasActivationForward(dlcHandle_t handle, const float *alpha,
                                                dlcTensorDescriptor_t xDesc, const void *x,
                                                dlcFilterDescriptor_t wDesc, const void *w,
                                                dlcConvolutionDescriptor_t conv,
                                                const float *beta, const float *bias,
                                                dlcActivationMode_t activation,
                                                dlcTensorDescriptor_t yDesc, void *y);

/* ---- backward routines ---------------------------------------------------
 *
 * The cuDNN page's method section: beside the forward convolution the library
 * offers routines for backward propagation.  They are the derivatives of the
 * forward sum (with the descriptor's mode, pads, strides and dilations):
 *
 *   dx[n,c,h,w] = sum of dy[n,k,p,q] * w[k,c,r,s] over k, r, s and the outputs
 *                 (p, q) with p*u + r*dh - pad_top = h, q*v + s*dw - pad_left = w
 *   dw[k,c,r,s] = sum over n, p, q of dy[n,k,p,q] * x[n,c,p*u + r*dh - pad_top,
 *                 q*v + s*dw - pad_left]   (x reads as zero outside the image)
 *
 * (in convolution mode w[k,c,r,s] reads w[k,c,R-1-r,S-1-s] and dw is written
 * mirrored the same way).  The two inputs share a storage type matching the
 * math mode as for the forward call (FP32 math: FLOAT or BFLOAT16; TF32:
 * FLOAT; BF16: BFLOAT16; FP64: DOUBLE); the output is FLOAT or BFLOAT16 (DOUBLE
 * for FP64).  dy's dimensions must be the forward output's (N, K, P, Q).  The
 * output must not overlap an input (BAD_PARAM).  No workspace: the
 * workspace-size queries return 0.  Asynchronous on the handle's stream.
 */

/* dx = alpha * dgrad(w, dy) + beta * dx (beta == 0: dx is not read).
 * dxDesc gives N, C, H, W; wDesc K, C, R, S.  BF16 math with KRSC filters,
 * channels-innermost dy and dx and no dilation runs on the tensor cores (one
 * SM-pair launch per stride phase, filters read transposed); every other
 * combination runs the direct kernel (DLC_KERNEL_DIRECT).  Source: cuDNN
 * page, method section (backward routines); maxDNN page, research questions
 * (the forward techniques carry over to the backward pass). */
dlcStatus_t dlcConvolutionBackwardData(dlcHandle_t handle, const float *alpha,
                                       dlcFilterDescriptor_t wDesc, const void *w,
                                       dlcTensorDescriptor_t dyDesc, const void *dy,
                                       dlcConvolutionDescriptor_t conv, const float *beta,
                                       dlcTensorDescriptor_t dxDesc, void *dx);

/* dw = alpha * wgrad(x, dy) + beta * dw.  dwDesc gives K, C, R, S and the
 * layout of dw (KCRS or KRSC) and its storage type.  A FLOAT or DOUBLE dw may
 * be written by reductions split over CTAs whose partial sums meet in atomic
 * adds (their order varies; see dlcSetDeterministic, which turns the split
 * off).  Source: cuDNN page, method section (backward routines); batch-reduce
 * GEMM page, method section (the same building block, reducing over the
 * output pixels). */
dlcStatus_t dlcConvolutionBackwardFilter(dlcHandle_t handle, const float *alpha,
                                         dlcTensorDescriptor_t xDesc, const void *x,
                                         dlcTensorDescriptor_t dyDesc, const void *dy,
                                         dlcConvolutionDescriptor_t conv, const float *beta,
                                         dlcFilterDescriptor_t dwDesc, void *dw);

dlcStatus_t dlcGetConvolutionBackwardDataWorkspaceSize(dlcHandle_t handle,
                                                       dlcFilterDescriptor_t wDesc,
                                                       dlcTensorDescriptor_t dyDesc,
                                                       dlcConvolutionDescriptor_t conv,
                                                       dlcTensorDescriptor_t dxDesc,
                                                       size_t *bytes);
dlcStatus_t dlcGetConvolutionBackwardFilterWorkspaceSize(dlcHandle_t handle,
                                                         dlcTensorDescriptor_t xDesc,
                                                         dlcTensorDescriptor_t dyDesc,
                                                         dlcConvolutionDescriptor_t conv,
                                                         dlcFilterDescriptor_t dwDesc,
                                                         size_t *bytes);

/* Kernel the backward calls with these descriptors would launch (diagnostic;
 * pointers may be NULL, alignment is then taken as satisfied).  No
 * counterpart on the pages. */
dlcStatus_t dlcGetConvolutionBackwardDataKernel(dlcHandle_t handle, dlcFilterDescriptor_t wDesc,
                                                const void *w, dlcTensorDescriptor_t dyDesc,
                                                const void *dy, dlcConvolutionDescriptor_t conv,
                                                dlcTensorDescriptor_t dxDesc, const void *dx,
                                                dlcKernel_t *kernel);
dlcStatus_t dlcGetConvolutionBackwardFilterKernel(dlcHandle_t handle, dlcTensorDescriptor_t xDesc,
                                                  const void *x, dlcTensorDescriptor_t dyDesc,
                                                  const void *dy, dlcConvolutionDescriptor_t conv,
                                                  dlcFilterDescriptor_t dwDesc, const void *dw,
                                                  dlcKernel_t *kernel);

/* ---- pooling and activation forward ----------------------------------------
 *
 * The cuDNN page's summary and method section: pooling and activation
 * functions beside convolution, with the same tensor descriptors (any
 * strides) and caller-owned device buffers.  x and y may have different
 * layouts; storage FLOAT or BFLOAT16 (independently) or DOUBLE for both.
 * Sums and comparisons run in FP32 (FP64 for DOUBLE).  alpha and beta as for
 * the convolution (beta == 0: y is not read).  Asynchronous on the handle's
 * stream.  x and y must not overlap, except that dlcActivationForward may
 * run in place (x == y with identical descriptors).
 */

dlcStatus_t dlcCreatePoolingDescriptor(dlcPoolingDescriptor_t *desc);
dlcStatus_t dlcDestroyPoolingDescriptor(dlcPoolingDescriptor_t desc);

/* Window R x S, pads (each smaller than the window along its axis, so that
 * no window is empty), strides u, v >= 1.  BAD_PARAM otherwise.  Source:
 * cuDNN page, method section (pooling); the pad rule is this library's
 * reading (the page is silent). */
dlcStatus_t dlcSetPooling2dDescriptor(dlcPoolingDescriptor_t desc, dlcPoolingMode_t mode,
                                      int window_h, int window_w, int pad_top, int pad_bottom,
                                      int pad_left, int pad_right, int u, int v);
dlcStatus_t dlcGetPooling2dDescriptor(dlcPoolingDescriptor_t desc, dlcPoolingMode_t *mode,
                                      int *window_h, int *window_w, int *pad_top,
                                      int *pad_bottom, int *pad_left, int *pad_right, int *u,
                                      int *v);

/* Output dimensions N, C, P, Q (P = floor((H + pad_top + pad_bottom - R) / u) + 1,
 * Q likewise). */
dlcStatus_t dlcGetPooling2dForwardOutputDim(dlcPoolingDescriptor_t desc,
                                            dlcTensorDescriptor_t xDesc, int *n, int *c, int *p,
                                            int *q);

/* y[n,c,p,q] = alpha * POOL(window of x[n,c]) + beta * y[n,c,p,q].
 * POOL: the maximum, or the window sum over R*S (padding counted) or over the
 * in-image elements (padding excluded).  Source: cuDNN page, summary and
 * method section (pooling beside convolution). */
dlcStatus_t dlcPoolingForward(dlcHandle_t handle, dlcPoolingDescriptor_t desc, const float *alpha,
                              dlcTensorDescriptor_t xDesc, const void *x, const float *beta,
                              dlcTensorDescriptor_t yDesc, void *y);

/* Kernel dlcPoolingForward would launch (diagnostic; pointers may be NULL). */
dlcStatus_t dlcGetPoolingForwardKernel(dlcHandle_t handle, dlcPoolingDescriptor_t desc,
                                       dlcTensorDescriptor_t xDesc, const void *x,
                                       dlcTensorDescriptor_t yDesc, const void *y,
                                       dlcKernel_t *kernel);

/* y = alpha * f(x) + beta * y elementwise; x and y of the same dimensions.
 * coef is the ceiling of CLIPPED_RELU (ignored otherwise).  Source: cuDNN
 * page, summary and method section (activation functions; the page names no
 * list: identity, ReLU, sigmoid, tanh and clipped ReLU are this library's
 * reading). */
dlcStatus_t dlcActivationForward(dlcHandle_t handle, dlcActivationMode_t mode, double coef,
                                 const float *alpha, dlcTensorDescriptor_t xDesc, const void *x,
                                 const float *beta, dlcTensorDescriptor_t yDesc, void *y);

/* ---- self test of the device error path ---------------------------------- */

/* Launches one block whose pipeline wait is on a barrier nothing completes,
 * with a limit of timeout_us microseconds (1..1000000).  The kernel records
 * DLC_DEVERR_WAIT_TIMEOUT and returns; no GPU fault is involved.  Used by the
 * tests of the error path.  No counterpart on the pages. */
dlcStatus_t dlcDebugWaitTimeoutSelfTest(dlcHandle_t handle, int timeout_us);

/* ---- forward convolution that allocates nothing ---------------------------
 *
 * No counterpart on the pages: this is a service for callers that may not
 * allocate memory after start-up -- for example a serving process whose
 * memory is reserved once at start-up, or a plug-in inside a framework that
 * owns all device memory through its own allocator.  Such callers cannot
 * create a handle (dlcCreate allocates its error word, split-tile flags and
 * filter-repacking buffer).
 *
 * dlcConvolutionForwardNoAlloc computes y = alpha * conv(x, w) + beta * y like
 * dlcConvolutionForward, with tensor-core math only (TF32 or BF16; FP32 math
 * returns NOT_SUPPORTED), launched on `stream` (a cudaStream_t as void*,
 * NULL = legacy default stream) of the current device.  It allocates no host
 * or device memory and calls no allocating routine.  Besides x, w, y and
 * `status` it uses only fixed scratch arrays compiled into the library
 * (DLC_NOALLOC_MAX_TILES split-tile flags and two error words, and 256 KiB
 * where the few-channel kernel repacks the filters); every GPU that loads the
 * library holds those arrays until the process exits.
 *
 * It launches the same kernels as dlcConvolutionForward would for the
 * problem (each CTA pair or CTA works on whole output tiles or on an
 * independent part of one; no CTA waits on another CTA of the launch, so
 * other work running on the GPU at the same time cannot stall it), with the
 * few-channel kernel's repacked filters in the fixed array.  The
 * DLC_NOALLOC_MAX_TILES flags serve only the opt-in stream-K schedule
 * (environment DLC_TC_STREAMK=1), whose CTAs do wait on one another and need
 * them all resident; problems with more tiles than flags run whole tiles.
 *
 * The first call on a device sets that device up: it looks up the scratch
 * arrays' device addresses and the tensor-map encoders, and loads every
 * kernel of the library into the context (CUDA loads modules lazily, and a
 * module load allocates device memory), so later calls load nothing.  Make
 * that first call before any stream capture.  A device reset
 * (cudaDeviceReset) invalidates the set-up: calls after one are not
 * supported.  Every call reuses the same scratch arrays and clears its flags
 * on `stream` before launching, so calls whose work overlaps on the GPU (other
 * streams, other host threads) race with each other: issue them one at a
 * time.
 *
 * status: NULL, or a device-accessible array of two ints owned by the caller;
 *   the call zeroes it on `stream`, and a kernel that gives up on a pipeline
 *   wait writes dlcDeviceError_t code and detail there.  With NULL such an
 *   error goes to the scratch array and is not reported.
 * Errors: BAD_PARAM / NOT_SUPPORTED as for dlcConvolutionForward, plus the
 * above; EXECUTION_FAILED if the set-up or the launch fails.
 */
#define DLC_NOALLOC_MAX_TILES 4096

dlcStatus_t dlcConvolutionForwardNoAlloc(void *stream, const float *alpha,
                                         dlcTensorDescriptor_t xDesc, const void *x,
                                         dlcFilterDescriptor_t wDesc, const void *w,
                                         dlcConvolutionDescriptor_t conv, const float *beta,
                                         dlcTensorDescriptor_t yDesc, void *y, int *status);

#ifdef __cplusplus
}
#endif

#endif /* DLC_H_ */
