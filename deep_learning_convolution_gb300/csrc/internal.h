// internal.h -- host-side structures shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dlc.h"

struct dlcTensorStruct {
    int set = 0;
    dlcDataType_t dtype = DLC_DATA_FLOAT;
    int n = 0, c = 0, h = 0, w = 0;
    int64_t stride[4] = {0, 0, 0, 0};  // n, c, h, w (elements)
};

struct dlcFilterStruct {
    int set = 0;
    dlcDataType_t dtype = DLC_DATA_FLOAT;
    dlcTensorFormat_t format = DLC_TENSOR_NCHW;
    int k = 0, c = 0, r = 0, s = 0;
};

struct dlcPoolingStruct {
    int set = 0;
    dlcPoolingMode_t mode = DLC_POOLING_MAX;
    int r = 1, s = 1;
    int pad_top = 0, pad_bottom = 0, pad_left = 0, pad_right = 0;
    int u = 1, v = 1;
};

struct dlcConvolutionStruct {
    int set = 0;
    int pad_top = 0, pad_bottom = 0, pad_left = 0, pad_right = 0;
    int u = 1, v = 1, dil_h = 1, dil_w = 1;
    dlcMathType_t math = DLC_MATH_FP32;
    dlcConvolutionMode_t mode = DLC_CROSS_CORRELATION;
};

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*EncodeIm2colFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const int *,
                                   const int *, cuuint32_t, cuuint32_t, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct dlcContext {
    int device = 0;
    int sm_count = 0;
    cudaStream_t stream = nullptr;
    int *h_err = nullptr;   // mapped host words: [0] code, [1] detail
    int *d_err = nullptr;   // device alias of h_err
    uint64_t launches = 0;
    unsigned long long timeout_ns = 2000000000ull;  // pipeline wait limit
    int *sk_flags = nullptr;  // DLC_SK_FLAGS per-tile flags of split tiles (zero between launches)
    void *wpack = nullptr;    // filters repacked for the window and row-stack kernels
    size_t wpack_bytes = 0;   // its size
    int deterministic = 0;    // no split reductions whose partial sums meet in atomic adds
    EncodeTiledFn encode_tiled = nullptr;
    EncodeIm2colFn encode_im2col = nullptr;
};

// Split-tile flags owned by a handle: at most this many tiles per launch use them.
#define DLC_SK_FLAGS 4096
// Device bytes of the window kernel's repacked filter image (at most the
// shared memory of one CTA): the allocation-free entry point's fixed array.
#define DLC_WPACK_BYTES (256 * 1024)
// Device bytes a handle keeps for repacked filters: the window kernel's image
// or the row-stack kernel's filter slices (up to about one filter bank).
#define DLC_HANDLE_WPACK_BYTES (2 * 1024 * 1024)

inline int dlc_dtype_bytes(dlcDataType_t t) {
    return t == DLC_DATA_BFLOAT16 ? 2 : (t == DLC_DATA_DOUBLE ? 8 : 4);
}

// A fully resolved forward problem (validated by the API layer).
struct ConvProblem {
    int N, C, H, W, K, R, S, P, Q;
    int pt, pb, pl, pr, u, v, dh, dw;
    dlcMathType_t math;
    dlcDataType_t xdt;   // storage of x and w
    dlcDataType_t ydt;   // storage of y
    dlcTensorFormat_t wfmt;
    const void *x;
    int64_t xs[4];       // n, c, h, w
    const void *w;
    int64_t ws[4];       // k, c, r, s
    void *y;
    int64_t ys[4];       // n, k, p, q
    const float *bias;
    float alpha, beta;
    int relu;
    // Filter taps read mirrored, w[k, c, R-1-r, S-1-s] (convolution mode, and
    // the data gradient's transposed filters).
    int flip = 0;
    // Filters given transposed: ws[0] is the stride of the output-channel
    // index k and must be 1 (contiguous), ws[1] that of the reduction channel
    // c.  The data gradient's problem reads the forward filters this way.
    int w_mn = 0;
};

// A fully resolved backward problem (validated by the API layer), in the
// forward problem's terms: x [N,C,H,W], w [K,C,R,S], dy [N,K,P,Q].  For the
// data gradient x is the output dx; for the filter gradient w is the output dw.
struct BwdProblem {
    int N, C, H, W, K, R, S, P, Q;
    int pt, pb, pl, pr, u, v, dh, dw;
    dlcMathType_t math;
    dlcDataType_t in_dt;   // storage of the two inputs
    dlcDataType_t out_dt;  // storage of the output
    dlcTensorFormat_t wfmt;
    int flip;              // convolution mode: the forward read w[k,c,R-1-r,S-1-s]
    const void *x;
    int64_t xs[4];         // n, c, h, w
    const void *w;
    int64_t ws[4];         // k, c, r, s
    const void *dy;
    int64_t dys[4];        // n, k, p, q
    double alpha, beta;
};

// Pooling forward (validated): x [N,C,H,W] -> y [N,C,P,Q].
struct PoolProblem {
    int N, C, H, W, R, S, P, Q;
    int pt, pl, u, v, mode;
    dlcDataType_t xdt, ydt;
    const void *x;
    int64_t xs[4];
    void *y;
    int64_t ys[4];
    double alpha, beta;
};

// Activation forward (validated): y = alpha * f(x) + beta * y, both [N,C,H,W].
struct ActProblem {
    int N, C, H, W, mode;
    dlcDataType_t xdt, ydt;
    const void *x;
    int64_t xs[4];
    void *y;
    int64_t ys[4];
    double alpha, beta, coef;
};

// pool_act.cu
dlcKernel_t dlc_pool_variant(const PoolProblem &pp);
dlcStatus_t dlc_launch_pool(dlcContext *ctx, const PoolProblem &pp);
dlcStatus_t dlc_launch_activation(dlcContext *ctx, const ActProblem &ap);

// conv_bwd.cu: data and filter gradients.
dlcKernel_t dlc_dgrad_variant(const dlcContext *ctx, const BwdProblem &bp);
dlcStatus_t dlc_launch_dgrad(dlcContext *ctx, const BwdProblem &bp);
dlcKernel_t dlc_wgrad_variant(const dlcContext *ctx, const BwdProblem &bp);
// conv_wgrad.cu: the filter gradient on the tensor cores (adds into dw).
bool dlc_wgrad_tc_ok(const BwdProblem &bp);
dlcStatus_t dlc_launch_wgrad_tc(dlcContext *ctx, const BwdProblem &bp);
dlcStatus_t dlc_launch_wgrad(dlcContext *ctx, const BwdProblem &bp);

// Kernel launchers (conv_ffma.cu, conv_tc.cu).  They return SUCCESS or an
// error status and count launches in ctx->launches.
dlcStatus_t dlc_launch_ffma(dlcContext *ctx, const ConvProblem &pb);
dlcKernel_t dlc_tc_variant(const dlcContext *ctx, const ConvProblem &pb);
dlcStatus_t dlc_launch_tc(dlcContext *ctx, const ConvProblem &pb, dlcKernel_t variant);
dlcStatus_t dlc_launch_wait_selftest(dlcContext *ctx, unsigned long long timeout_ns);
// conv_window.cu: layers with few channels per horizontal stride step.
bool dlc_window_ok(const ConvProblem &pb);
dlcStatus_t dlc_launch_window(dlcContext *ctx, const ConvProblem &pb);
// conv_pair.cu: the im2col lowering on pairs of SMs (DLC_TC_PAIR=0 turns it off).
bool dlc_pair_enabled(const dlcContext *ctx);
// Launches of the window and pair kernels overlap the tail of the grid before
// them (programmatic dependent launch) unless DLC_PDL=0.
bool dlc_pdl_enabled();
dlcStatus_t dlc_launch_pair(dlcContext *ctx, const ConvProblem &pb);
// conv_tc.cu: conditions of the TMA im2col lowering (single CTA and pairs).
bool dlc_im2col_ok(const ConvProblem &pb);
// Each loads every kernel of its translation unit into the current context
// (CUDA loads modules lazily by default, and a module load allocates device
// memory): the allocation-free entry point calls them at its per-device set-up.
dlcStatus_t dlc_preload_tc();
dlcStatus_t dlc_preload_window();
dlcStatus_t dlc_preload_pair();
dlcStatus_t dlc_preload_rowstack();
// conv_rowstack.cu: TF32 channel-planar layers with few filters and unit
// horizontal stride (filters stacked over output rows as the MMA's M side).
bool dlc_rowstack_ok(const dlcContext *ctx, const ConvProblem &pb);
dlcStatus_t dlc_launch_rowstack(dlcContext *ctx, const ConvProblem &pb);

