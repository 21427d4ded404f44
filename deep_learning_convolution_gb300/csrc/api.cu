// api.cu -- the C ABI: handles, descriptors, validation and kernel dispatch.
//
// Descriptor-based C interface with arbitrary strides and caller-owned device
// buffers, following the cuDNN page's method section; zero workspace
// following the zero-memory-overhead direct convolution page.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "internal.h"

// Scratch of dlcConvolutionForwardNoAlloc: DLC_NOALLOC_MAX_TILES split-tile
// flags (used only by the opt-in stream-K schedule) followed by two error
// words.  Device code never names it; host code passes its device address,
// looked up once per device.
static __device__ __align__(256) int dlc_noalloc_scratch[DLC_NOALLOC_MAX_TILES + 64];
// Its repacked filter image for the window kernel.
static __device__ __align__(256) unsigned char dlc_noalloc_wpack[DLC_WPACK_BYTES];
static_assert(DLC_NOALLOC_MAX_TILES == DLC_SK_FLAGS, "one flag per split-capable tile");

namespace {

int64_t out_extent(int64_t in, int64_t lo, int64_t hi, int64_t filt, int64_t dil, int64_t stride) {
    int64_t eff = dil * (filt - 1) + 1;
    int64_t span = in + lo + hi - eff;
    if (span < 0) return 0;
    return span / stride + 1;
}

size_t elt_size(dlcDataType_t t) { return (size_t)dlc_dtype_bytes(t); }

bool valid_dtype(int t) {
    return t == DLC_DATA_FLOAT || t == DLC_DATA_BFLOAT16 || t == DLC_DATA_DOUBLE;
}

// Storage of the two inputs allowed by a math mode.
bool math_takes(dlcMathType_t m, dlcDataType_t in) {
    switch (m) {
        case DLC_MATH_FP32: return in == DLC_DATA_FLOAT || in == DLC_DATA_BFLOAT16;
        case DLC_MATH_TF32: return in == DLC_DATA_FLOAT;
        case DLC_MATH_BF16: return in == DLC_DATA_BFLOAT16;
        case DLC_MATH_FP64: return in == DLC_DATA_DOUBLE;
    }
    return false;
}

// Storage of the output allowed for given inputs: DOUBLE with DOUBLE, else
// FLOAT or BFLOAT16.
bool out_ok(dlcDataType_t in, dlcDataType_t out) {
    return in == DLC_DATA_DOUBLE ? out == DLC_DATA_DOUBLE : out != DLC_DATA_DOUBLE;
}
bool valid_format(int f) { return f == DLC_TENSOR_NCHW || f == DLC_TENSOR_NHWC; }

// Largest element offset reachable through (extent, stride) pairs.
int64_t max_offset(const int64_t *ext, const int64_t *str, int nd) {
    int64_t m = 0;
    for (int i = 0; i < nd; ++i) m += (ext[i] - 1) * str[i];
    return m;
}

// True if distinct index tuples map to distinct offsets (no self-overlap):
// sorted by stride, each stride must reach past the span of the smaller ones.
bool strides_injective(const int64_t *ext, const int64_t *str, int nd) {
    int idx[4] = {0, 1, 2, 3};
    std::sort(idx, idx + nd, [&](int a, int b) { return str[a] < str[b]; });
    int64_t span = 0;  // max offset of the dims seen so far
    for (int i = 0; i < nd; ++i) {
        int d = idx[i];
        if (ext[d] == 1) continue;
        if (str[d] <= span) return false;
        span += (ext[d] - 1) * str[d];
    }
    return true;
}

bool ranges_overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) {
    return a0 < b1 && b0 < a1;
}

void filter_strides(const dlcFilterStruct *f, int64_t *ws) {
    if (f->format == DLC_TENSOR_NCHW) {  // KCRS
        ws[3] = 1;
        ws[2] = f->s;
        ws[1] = (int64_t)f->r * f->s;
        ws[0] = (int64_t)f->c * f->r * f->s;
    } else {  // KRSC
        ws[1] = 1;
        ws[3] = f->c;
        ws[2] = (int64_t)f->s * f->c;
        ws[0] = (int64_t)f->r * f->s * f->c;
    }
}

// Validates descriptors (and pointers when check_ptrs) and fills `pb`.
dlcStatus_t resolve(dlcTensorDescriptor_t xd, const void *x, dlcFilterDescriptor_t wd,
                    const void *w, dlcConvolutionDescriptor_t cd, dlcTensorDescriptor_t yd,
                    void *y, bool check_ptrs, ConvProblem &pb) {
    if (!xd || !wd || !cd || !yd) return DLC_STATUS_BAD_PARAM;
    if (!xd->set || !wd->set || !cd->set || !yd->set) return DLC_STATUS_NOT_INITIALIZED;
    if (xd->c != wd->c) return DLC_STATUS_BAD_PARAM;
    if (xd->dtype != wd->dtype) return DLC_STATUS_BAD_PARAM;
    int64_t P = out_extent(xd->h, cd->pad_top, cd->pad_bottom, wd->r, cd->dil_h, cd->u);
    int64_t Q = out_extent(xd->w, cd->pad_left, cd->pad_right, wd->s, cd->dil_w, cd->v);
    if (P < 1 || Q < 1 || P > INT32_MAX || Q > INT32_MAX) return DLC_STATUS_BAD_PARAM;
    if (yd->n != xd->n || yd->c != wd->k || yd->h != P || yd->w != Q) return DLC_STATUS_BAD_PARAM;

    if (cd->math < DLC_MATH_FP32 || cd->math > DLC_MATH_FP64) return DLC_STATUS_BAD_PARAM;
    if (!math_takes(cd->math, xd->dtype) || !out_ok(xd->dtype, yd->dtype))
        return DLC_STATUS_NOT_SUPPORTED;

    pb.N = xd->n; pb.C = xd->c; pb.H = xd->h; pb.W = xd->w;
    pb.K = wd->k; pb.R = wd->r; pb.S = wd->s; pb.P = (int)P; pb.Q = (int)Q;
    pb.pt = cd->pad_top; pb.pb = cd->pad_bottom; pb.pl = cd->pad_left; pb.pr = cd->pad_right;
    pb.u = cd->u; pb.v = cd->v; pb.dh = cd->dil_h; pb.dw = cd->dil_w;
    pb.math = cd->math;
    pb.xdt = xd->dtype;
    pb.ydt = yd->dtype;
    pb.wfmt = wd->format;
    for (int i = 0; i < 4; ++i) {
        pb.xs[i] = xd->stride[i];
        pb.ys[i] = yd->stride[i];
    }
    filter_strides(wd, pb.ws);
    pb.x = x; pb.w = w; pb.y = y;
    pb.bias = nullptr; pb.alpha = 1.f; pb.beta = 0.f; pb.relu = 0;
    pb.flip = cd->mode == DLC_CONVOLUTION ? 1 : 0;
    pb.w_mn = 0;

    const int64_t yext[4] = {pb.N, pb.K, pb.P, pb.Q};
    if (!strides_injective(yext, pb.ys, 4)) return DLC_STATUS_BAD_PARAM;
    const int64_t xext[4] = {pb.N, pb.C, pb.H, pb.W};
    const int64_t wext[4] = {pb.K, pb.C, pb.R, pb.S};
    const int64_t xmax = max_offset(xext, pb.xs, 4);
    const int64_t wmax = max_offset(wext, pb.ws, 4);
    const int64_t ymax = max_offset(yext, pb.ys, 4);
    const int64_t lim = (int64_t)1 << 60;
    if (xmax >= lim || wmax >= lim || ymax >= lim) return DLC_STATUS_BAD_PARAM;

    if (check_ptrs) {
        if (!x || !w || !y) return DLC_STATUS_BAD_PARAM;
        const size_t ex = elt_size(pb.xdt), ey = elt_size(pb.ydt);
        if ((uintptr_t)x % ex || (uintptr_t)w % ex || (uintptr_t)y % ey) return DLC_STATUS_BAD_PARAM;
        uintptr_t x0 = (uintptr_t)x, x1 = x0 + (uintptr_t)(xmax + 1) * ex;
        uintptr_t w0 = (uintptr_t)w, w1 = w0 + (uintptr_t)(wmax + 1) * ex;
        uintptr_t y0 = (uintptr_t)y, y1 = y0 + (uintptr_t)(ymax + 1) * ey;
        if (ranges_overlap(x0, x1, y0, y1) || ranges_overlap(w0, w1, y0, y1))
            return DLC_STATUS_BAD_PARAM;
    }
    return DLC_STATUS_SUCCESS;
}

dlcKernel_t pick_kernel(const dlcContext *ctx, const ConvProblem &pb) {
    if (pb.math == DLC_MATH_FP32 || pb.math == DLC_MATH_FP64) return DLC_KERNEL_FFMA;
    return dlc_tc_variant(ctx, pb);
}

// Convolution mode for the kernels that read filters through strides: the
// mirrored taps as a view based at tap (R-1, S-1) with negated tap strides.
// (The SM-pair kernel mirrors its filter-load coordinates instead.)
void mirror_filter_view(ConvProblem &pb) {
    const long long e = dlc_dtype_bytes(pb.xdt);
    pb.w = static_cast<const char *>(pb.w) +
           e * ((long long)(pb.R - 1) * pb.ws[2] + (long long)(pb.S - 1) * pb.ws[3]);
    pb.ws[2] = -pb.ws[2];
    pb.ws[3] = -pb.ws[3];
    pb.flip = 0;
}

// Validates a backward problem.  `xd`/`x` describe the forward input (dx for
// the data gradient), `wd`/`w` the filters (dw for the filter gradient),
// `dyd`/`dy` the forward output's gradient; `out` says which of x (0) or w (1)
// is written.
dlcStatus_t resolve_bwd(dlcTensorDescriptor_t xd, const void *x, dlcFilterDescriptor_t wd,
                        const void *w, dlcConvolutionDescriptor_t cd, dlcTensorDescriptor_t dyd,
                        const void *dy, int out, bool check_ptrs, BwdProblem &bp) {
    if (!xd || !wd || !cd || !dyd) return DLC_STATUS_BAD_PARAM;
    if (!xd->set || !wd->set || !cd->set || !dyd->set) return DLC_STATUS_NOT_INITIALIZED;
    if (xd->c != wd->c) return DLC_STATUS_BAD_PARAM;
    const int64_t P = out_extent(xd->h, cd->pad_top, cd->pad_bottom, wd->r, cd->dil_h, cd->u);
    const int64_t Q = out_extent(xd->w, cd->pad_left, cd->pad_right, wd->s, cd->dil_w, cd->v);
    if (P < 1 || Q < 1 || P > INT32_MAX || Q > INT32_MAX) return DLC_STATUS_BAD_PARAM;
    if (dyd->n != xd->n || dyd->c != wd->k || dyd->h != P || dyd->w != Q) return DLC_STATUS_BAD_PARAM;
    // the two inputs share a storage type; the output's may differ
    const dlcDataType_t in = out == 0 ? wd->dtype : xd->dtype;
    const dlcDataType_t od = out == 0 ? xd->dtype : wd->dtype;
    if (dyd->dtype != in) return DLC_STATUS_BAD_PARAM;
    if (cd->math < DLC_MATH_FP32 || cd->math > DLC_MATH_FP64) return DLC_STATUS_BAD_PARAM;
    if (!math_takes(cd->math, in) || !out_ok(in, od)) return DLC_STATUS_NOT_SUPPORTED;

    bp.N = xd->n; bp.C = xd->c; bp.H = xd->h; bp.W = xd->w;
    bp.K = wd->k; bp.R = wd->r; bp.S = wd->s; bp.P = (int)P; bp.Q = (int)Q;
    bp.pt = cd->pad_top; bp.pb = cd->pad_bottom; bp.pl = cd->pad_left; bp.pr = cd->pad_right;
    bp.u = cd->u; bp.v = cd->v; bp.dh = cd->dil_h; bp.dw = cd->dil_w;
    bp.math = cd->math;
    bp.in_dt = in;
    bp.out_dt = od;
    bp.wfmt = wd->format;
    bp.flip = cd->mode == DLC_CONVOLUTION ? 1 : 0;
    for (int i = 0; i < 4; ++i) {
        bp.xs[i] = xd->stride[i];
        bp.dys[i] = dyd->stride[i];
    }
    filter_strides(wd, bp.ws);
    bp.x = x; bp.w = w; bp.dy = dy;
    bp.alpha = 1.0; bp.beta = 0.0;

    const int64_t xext[4] = {bp.N, bp.C, bp.H, bp.W};
    const int64_t wext[4] = {bp.K, bp.C, bp.R, bp.S};
    const int64_t yext[4] = {bp.N, bp.K, bp.P, bp.Q};
    if (out == 0 && !strides_injective(xext, bp.xs, 4)) return DLC_STATUS_BAD_PARAM;
    const int64_t xmax = max_offset(xext, bp.xs, 4);
    const int64_t wmax = max_offset(wext, bp.ws, 4);
    const int64_t ymax = max_offset(yext, bp.dys, 4);
    const int64_t lim = (int64_t)1 << 60;
    if (xmax >= lim || wmax >= lim || ymax >= lim) return DLC_STATUS_BAD_PARAM;
    if (check_ptrs) {
        if (!x || !w || !dy) return DLC_STATUS_BAD_PARAM;
        const size_t ex = elt_size(xd->dtype), ew = elt_size(wd->dtype), ey = elt_size(in);
        if ((uintptr_t)x % ex || (uintptr_t)w % ew || (uintptr_t)dy % ey) return DLC_STATUS_BAD_PARAM;
        const uintptr_t x0 = (uintptr_t)x, x1 = x0 + (uintptr_t)(xmax + 1) * ex;
        const uintptr_t w0 = (uintptr_t)w, w1 = w0 + (uintptr_t)(wmax + 1) * ew;
        const uintptr_t y0 = (uintptr_t)dy, y1 = y0 + (uintptr_t)(ymax + 1) * ey;
        const bool bad = out == 0 ? (ranges_overlap(x0, x1, w0, w1) || ranges_overlap(x0, x1, y0, y1))
                                  : (ranges_overlap(w0, w1, x0, x1) || ranges_overlap(w0, w1, y0, y1));
        if (bad) return DLC_STATUS_BAD_PARAM;
    }
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t pending_device_error(dlcContext *h) {
    volatile int *e = h->h_err;
    return (e && e[0] != 0) ? DLC_STATUS_EXECUTION_FAILED : DLC_STATUS_SUCCESS;
}

dlcStatus_t forward(dlcHandle_t h, const float *alpha, dlcTensorDescriptor_t xd, const void *x,
                    dlcFilterDescriptor_t wd, const void *w, dlcConvolutionDescriptor_t cd,
                    const float *beta, const float *bias, int relu, dlcTensorDescriptor_t yd,
                    void *y) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!alpha || !beta) return DLC_STATUS_BAD_PARAM;
    ConvProblem pb;
    dlcStatus_t st = resolve(xd, x, wd, w, cd, yd, y, true, pb);
    if (st != DLC_STATUS_SUCCESS) return st;
    if ((uintptr_t)bias % 4) return DLC_STATUS_BAD_PARAM;
    pb.alpha = *alpha;
    pb.beta = *beta;
    pb.bias = bias;
    pb.relu = relu;
    st = pending_device_error(h);
    if (st != DLC_STATUS_SUCCESS) return st;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return DLC_STATUS_BAD_PARAM;
    dlcKernel_t k = pick_kernel(h, pb);
    if (k == DLC_KERNEL_NONE) return DLC_STATUS_NOT_SUPPORTED;
    if (pb.flip && k != DLC_KERNEL_TC_IM2COL_PAIR) mirror_filter_view(pb);
    if (k == DLC_KERNEL_FFMA) return dlc_launch_ffma(h, pb);
    return dlc_launch_tc(h, pb, k);
}

}  // namespace

extern "C" {

const char *dlcGetErrorString(dlcStatus_t s) {
    switch (s) {
        case DLC_STATUS_SUCCESS: return "DLC_STATUS_SUCCESS";
        case DLC_STATUS_NOT_INITIALIZED: return "DLC_STATUS_NOT_INITIALIZED";
        case DLC_STATUS_BAD_PARAM: return "DLC_STATUS_BAD_PARAM";
        case DLC_STATUS_NOT_SUPPORTED: return "DLC_STATUS_NOT_SUPPORTED";
        case DLC_STATUS_EXECUTION_FAILED: return "DLC_STATUS_EXECUTION_FAILED";
        case DLC_STATUS_INTERNAL_ERROR: return "DLC_STATUS_INTERNAL_ERROR";
        case DLC_STATUS_ALLOC_FAILED: return "DLC_STATUS_ALLOC_FAILED";
    }
    return "DLC_STATUS_UNKNOWN";
}

dlcStatus_t dlcGetVersion(int *version) {
    if (!version) return DLC_STATUS_BAD_PARAM;
    *version = DLC_VERSION;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcCreate(dlcHandle_t *handle) {
    if (!handle) return DLC_STATUS_BAD_PARAM;
    *handle = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    if (prop.major != 10 || prop.minor != 3) return DLC_STATUS_NOT_SUPPORTED;
    dlcContext *h = new (std::nothrow) dlcContext();
    if (!h) return DLC_STATUS_ALLOC_FAILED;
    h->device = dev;
    h->sm_count = prop.multiProcessorCount;
    h->wpack_bytes = DLC_HANDLE_WPACK_BYTES;
    if (cudaHostAlloc((void **)&h->h_err, 4 * sizeof(int), cudaHostAllocMapped) != cudaSuccess) {
        delete h;
        return DLC_STATUS_EXECUTION_FAILED;
    }
    std::memset(h->h_err, 0, 4 * sizeof(int));
    if (cudaHostGetDevicePointer((void **)&h->d_err, h->h_err, 0) != cudaSuccess) {
        cudaFreeHost(h->h_err);
        delete h;
        return DLC_STATUS_EXECUTION_FAILED;
    }
    if (cudaMalloc((void **)&h->sk_flags, DLC_SK_FLAGS * sizeof(int)) != cudaSuccess ||
        cudaMemset(h->sk_flags, 0, DLC_SK_FLAGS * sizeof(int)) != cudaSuccess ||
        cudaMalloc(&h->wpack, DLC_HANDLE_WPACK_BYTES) != cudaSuccess) {
        if (h->sk_flags) cudaFree(h->sk_flags);
        if (h->wpack) cudaFree(h->wpack);
        cudaFreeHost(h->h_err);
        delete h;
        return DLC_STATUS_EXECUTION_FAILED;
    }
    cudaDriverEntryPointQueryResult q1, q2;
    void *f1 = nullptr, *f2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f1, 12000, cudaEnableDefault,
                                         &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &f2, 12000, cudaEnableDefault,
                                         &q2) != cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess) {
        cudaFree(h->sk_flags);
        cudaFree(h->wpack);
        cudaFreeHost(h->h_err);
        delete h;
        return DLC_STATUS_EXECUTION_FAILED;
    }
    h->encode_tiled = reinterpret_cast<EncodeTiledFn>(f1);
    h->encode_im2col = reinterpret_cast<EncodeIm2colFn>(f2);
    const char *tmo = std::getenv("DLC_WAIT_TIMEOUT_US");
    if (tmo) {
        long long us = std::atoll(tmo);
        if (us >= 1 && us <= 60000000LL) h->timeout_ns = (unsigned long long)us * 1000ull;
    }
    *handle = h;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcDestroy(dlcHandle_t h) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (h->h_err) cudaFreeHost(h->h_err);
    if (h->sk_flags) cudaFree(h->sk_flags);
    if (h->wpack) cudaFree(h->wpack);
    delete h;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcSetStream(dlcHandle_t h, void *stream) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    h->stream = static_cast<cudaStream_t>(stream);
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetStream(dlcHandle_t h, void **stream) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!stream) return DLC_STATUS_BAD_PARAM;
    *stream = h->stream;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcSetDeterministic(dlcHandle_t h, int deterministic) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (deterministic != 0 && deterministic != 1) return DLC_STATUS_BAD_PARAM;
    h->deterministic = deterministic;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetDeterministic(dlcHandle_t h, int *deterministic) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!deterministic) return DLC_STATUS_BAD_PARAM;
    *deterministic = h->deterministic;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetLastDeviceError(dlcHandle_t h, int *code, int *detail) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!code || !detail) return DLC_STATUS_BAD_PARAM;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    volatile int *e = h->h_err;
    *code = e[0];
    *detail = e[1];
    e[0] = 0;
    e[1] = 0;
    // a kernel that gave up may have left split-tile flags raised
    if (*code != 0 && cudaMemset(h->sk_flags, 0, DLC_SK_FLAGS * sizeof(int)) != cudaSuccess)
        return DLC_STATUS_EXECUTION_FAILED;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcSynchronize(dlcHandle_t h) {
    int code = 0, detail = 0;
    dlcStatus_t st = dlcGetLastDeviceError(h, &code, &detail);
    if (st != DLC_STATUS_SUCCESS) return st;
    return code ? DLC_STATUS_EXECUTION_FAILED : DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetLaunchCount(dlcHandle_t h, uint64_t *count) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!count) return DLC_STATUS_BAD_PARAM;
    *count = h->launches;
    return DLC_STATUS_SUCCESS;
}

// ---- tensor descriptors ----------------------------------------------------
dlcStatus_t dlcCreateTensorDescriptor(dlcTensorDescriptor_t *d) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    *d = new (std::nothrow) dlcTensorStruct();
    return *d ? DLC_STATUS_SUCCESS : DLC_STATUS_ALLOC_FAILED;
}

dlcStatus_t dlcDestroyTensorDescriptor(dlcTensorDescriptor_t d) {
    delete d;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcSetTensor4dDescriptorEx(dlcTensorDescriptor_t d, dlcDataType_t dtype, int n, int c,
                                       int h, int w, int64_t ns, int64_t cs, int64_t hs,
                                       int64_t ws) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    if (!valid_dtype(dtype) || n < 1 || c < 1 || h < 1 || w < 1) return DLC_STATUS_BAD_PARAM;
    if (ns < 0 || cs < 0 || hs < 0 || ws < 0) return DLC_STATUS_BAD_PARAM;
    const int64_t lim = (int64_t)1 << 40;
    if (ns > lim || cs > lim || hs > lim || ws > lim) return DLC_STATUS_BAD_PARAM;
    d->dtype = dtype;
    d->n = n; d->c = c; d->h = h; d->w = w;
    d->stride[0] = ns; d->stride[1] = cs; d->stride[2] = hs; d->stride[3] = ws;
    d->set = 1;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcSetTensor4dDescriptor(dlcTensorDescriptor_t d, dlcTensorFormat_t f,
                                     dlcDataType_t dtype, int n, int c, int h, int w) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    if (!valid_format(f) || n < 1 || c < 1 || h < 1 || w < 1) return DLC_STATUS_BAD_PARAM;
    const int64_t C = c, H = h, W = w;
    if (f == DLC_TENSOR_NCHW)
        return dlcSetTensor4dDescriptorEx(d, dtype, n, c, h, w, C * H * W, H * W, W, 1);
    return dlcSetTensor4dDescriptorEx(d, dtype, n, c, h, w, H * W * C, 1, W * C, C);
}

dlcStatus_t dlcGetTensor4dDescriptor(dlcTensorDescriptor_t d, dlcDataType_t *dtype, int *n,
                                     int *c, int *h, int *w, int64_t *ns, int64_t *cs,
                                     int64_t *hs, int64_t *ws) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    if (!d->set) return DLC_STATUS_NOT_INITIALIZED;
    if (dtype) *dtype = d->dtype;
    if (n) *n = d->n;
    if (c) *c = d->c;
    if (h) *h = d->h;
    if (w) *w = d->w;
    if (ns) *ns = d->stride[0];
    if (cs) *cs = d->stride[1];
    if (hs) *hs = d->stride[2];
    if (ws) *ws = d->stride[3];
    return DLC_STATUS_SUCCESS;
}

// ---- filter descriptors ------------------------------------------------------
dlcStatus_t dlcCreateFilterDescriptor(dlcFilterDescriptor_t *d) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    *d = new (std::nothrow) dlcFilterStruct();
    return *d ? DLC_STATUS_SUCCESS : DLC_STATUS_ALLOC_FAILED;
}

dlcStatus_t dlcDestroyFilterDescriptor(dlcFilterDescriptor_t d) {
    delete d;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcSetFilter4dDescriptor(dlcFilterDescriptor_t d, dlcDataType_t dtype,
                                     dlcTensorFormat_t f, int k, int c, int r, int s) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    if (!valid_dtype(dtype) || !valid_format(f) || k < 1 || c < 1 || r < 1 || s < 1)
        return DLC_STATUS_BAD_PARAM;
    if ((int64_t)k * c * r * s >= ((int64_t)1 << 40)) return DLC_STATUS_BAD_PARAM;
    d->dtype = dtype;
    d->format = f;
    d->k = k; d->c = c; d->r = r; d->s = s;
    d->set = 1;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetFilter4dDescriptor(dlcFilterDescriptor_t d, dlcDataType_t *dtype,
                                     dlcTensorFormat_t *f, int *k, int *c, int *r, int *s) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    if (!d->set) return DLC_STATUS_NOT_INITIALIZED;
    if (dtype) *dtype = d->dtype;
    if (f) *f = d->format;
    if (k) *k = d->k;
    if (c) *c = d->c;
    if (r) *r = d->r;
    if (s) *s = d->s;
    return DLC_STATUS_SUCCESS;
}

// ---- convolution descriptors ---------------------------------------------------
dlcStatus_t dlcCreateConvolutionDescriptor(dlcConvolutionDescriptor_t *d) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    *d = new (std::nothrow) dlcConvolutionStruct();
    return *d ? DLC_STATUS_SUCCESS : DLC_STATUS_ALLOC_FAILED;
}

dlcStatus_t dlcDestroyConvolutionDescriptor(dlcConvolutionDescriptor_t d) {
    delete d;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcSetConvolution2dDescriptor(dlcConvolutionDescriptor_t d, int pad_h, int pad_w,
                                          int u, int v, int dil_h, int dil_w, dlcMathType_t math) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    if (pad_h < 0 || pad_w < 0 || u < 1 || v < 1 || dil_h < 1 || dil_w < 1)
        return DLC_STATUS_BAD_PARAM;
    if (math != DLC_MATH_FP32 && math != DLC_MATH_TF32 && math != DLC_MATH_BF16 &&
        math != DLC_MATH_FP64)
        return DLC_STATUS_BAD_PARAM;
    const int big = 1 << 20;
    if (pad_h > big || pad_w > big || u > big || v > big || dil_h > big || dil_w > big)
        return DLC_STATUS_BAD_PARAM;
    d->pad_top = d->pad_bottom = pad_h;
    d->pad_left = d->pad_right = pad_w;
    d->u = u; d->v = v; d->dil_h = dil_h; d->dil_w = dil_w;
    d->math = math;
    d->set = 1;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcSetConvolution2dPadding(dlcConvolutionDescriptor_t d, int pt, int pb, int pl,
                                       int pr) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    if (!d->set) return DLC_STATUS_NOT_INITIALIZED;
    const int big = 1 << 20;
    if (pt < 0 || pb < 0 || pl < 0 || pr < 0 || pt > big || pb > big || pl > big || pr > big)
        return DLC_STATUS_BAD_PARAM;
    d->pad_top = pt; d->pad_bottom = pb; d->pad_left = pl; d->pad_right = pr;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetConvolution2dDescriptor(dlcConvolutionDescriptor_t d, int *pt, int *pb, int *pl,
                                          int *pr, int *u, int *v, int *dh, int *dw,
                                          dlcMathType_t *math) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    if (!d->set) return DLC_STATUS_NOT_INITIALIZED;
    if (pt) *pt = d->pad_top;
    if (pb) *pb = d->pad_bottom;
    if (pl) *pl = d->pad_left;
    if (pr) *pr = d->pad_right;
    if (u) *u = d->u;
    if (v) *v = d->v;
    if (dh) *dh = d->dil_h;
    if (dw) *dw = d->dil_w;
    if (math) *math = d->math;
    return DLC_STATUS_SUCCESS;
}

// ---- forward ------------------------------------------------------------------
dlcStatus_t dlcGetConvolution2dForwardOutputDim(dlcConvolutionDescriptor_t cd,
                                                dlcTensorDescriptor_t xd, dlcFilterDescriptor_t wd,
                                                int *n, int *k, int *p, int *q) {
    if (!cd || !xd || !wd || !n || !k || !p || !q) return DLC_STATUS_BAD_PARAM;
    if (!cd->set || !xd->set || !wd->set) return DLC_STATUS_NOT_INITIALIZED;
    if (xd->c != wd->c) return DLC_STATUS_BAD_PARAM;
    int64_t P = out_extent(xd->h, cd->pad_top, cd->pad_bottom, wd->r, cd->dil_h, cd->u);
    int64_t Q = out_extent(xd->w, cd->pad_left, cd->pad_right, wd->s, cd->dil_w, cd->v);
    if (P < 1 || Q < 1 || P > INT32_MAX || Q > INT32_MAX) return DLC_STATUS_BAD_PARAM;
    *n = xd->n;
    *k = wd->k;
    *p = (int)P;
    *q = (int)Q;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetConvolutionForwardWorkspaceSize(dlcHandle_t h, dlcTensorDescriptor_t xd,
                                                  dlcFilterDescriptor_t wd,
                                                  dlcConvolutionDescriptor_t cd,
                                                  dlcTensorDescriptor_t yd, size_t *bytes) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!bytes) return DLC_STATUS_BAD_PARAM;
    ConvProblem pb;
    dlcStatus_t st = resolve(xd, nullptr, wd, nullptr, cd, yd, nullptr, false, pb);
    if (st != DLC_STATUS_SUCCESS) return st;
    *bytes = 0;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetConvolutionForwardKernel(dlcHandle_t h, dlcTensorDescriptor_t xd, const void *x,
                                           dlcFilterDescriptor_t wd, const void *w,
                                           dlcConvolutionDescriptor_t cd, dlcTensorDescriptor_t yd,
                                           const void *y, dlcKernel_t *kernel) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!kernel) return DLC_STATUS_BAD_PARAM;
    ConvProblem pb;
    dlcStatus_t st = resolve(xd, x, wd, w, cd, yd, const_cast<void *>(y), false, pb);
    if (st != DLC_STATUS_SUCCESS) return st;
    *kernel = pick_kernel(h, pb);
    return *kernel == DLC_KERNEL_NONE ? DLC_STATUS_NOT_SUPPORTED : DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcConvolutionForward(dlcHandle_t h, const float *alpha, dlcTensorDescriptor_t xd,
                                  const void *x, dlcFilterDescriptor_t wd, const void *w,
                                  dlcConvolutionDescriptor_t cd, const float *beta,
                                  dlcTensorDescriptor_t yd, void *y) {
    return forward(h, alpha, xd, x, wd, w, cd, beta, nullptr, 0, yd, y);
}

dlcStatus_t dlcConvolutionBiasActivationForward(dlcHandle_t h, const float *alpha,
                                                dlcTensorDescriptor_t xd, const void *x,
                                                dlcFilterDescriptor_t wd, const void *w,
                                                dlcConvolutionDescriptor_t cd, const float *beta,
                                                const float *bias, dlcActivationMode_t act,
                                                dlcTensorDescriptor_t yd, void *y) {
    if (act < DLC_ACTIVATION_IDENTITY || act > DLC_ACTIVATION_CLIPPED_RELU) return DLC_STATUS_BAD_PARAM;
    if (act != DLC_ACTIVATION_IDENTITY && act != DLC_ACTIVATION_RELU) return DLC_STATUS_NOT_SUPPORTED;
    return forward(h, alpha, xd, x, wd, w, cd, beta, bias, act == DLC_ACTIVATION_RELU, yd, y);
}

// Per-device set-up of the allocation-free entry point: the scratch array's
// device address (cudaGetSymbolAddress with the device current), every kernel
// of the library loaded into the context, the SM count and the tensor-map
// encoders.  Done by the first call on each device.
namespace {
struct NoAllocDevice {
    int ready = 0;
    int *scratch = nullptr;
    void *wpack = nullptr;
    int sm_count = 0;
    EncodeTiledFn encode_tiled = nullptr;
    EncodeIm2colFn encode_im2col = nullptr;
};
constexpr int kNoAllocMaxDevices = 64;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

dlcStatus_t noalloc_setup(int dev, NoAllocDevice **out) {
    if (dev < 0 || dev >= kNoAllocMaxDevices) return DLC_STATUS_NOT_SUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocDevice &d = g_noalloc_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return DLC_STATUS_EXECUTION_FAILED;
        if (major != 10 || minor != 3) return DLC_STATUS_NOT_SUPPORTED;
        int *ptr = nullptr;
        void *wptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, dlc_noalloc_scratch) != cudaSuccess || !ptr ||
            cudaGetSymbolAddress(&wptr, dlc_noalloc_wpack) != cudaSuccess || !wptr)
            return DLC_STATUS_EXECUTION_FAILED;
        // Load every kernel a later call may launch now: modules are loaded
        // lazily, and a module load allocates device memory.
        if (dlc_preload_tc() != DLC_STATUS_SUCCESS || dlc_preload_window() != DLC_STATUS_SUCCESS ||
            dlc_preload_pair() != DLC_STATUS_SUCCESS || dlc_preload_rowstack() != DLC_STATUS_SUCCESS)
            return DLC_STATUS_EXECUTION_FAILED;
        cudaDriverEntryPointQueryResult q1, q2;
        void *f1 = nullptr, *f2 = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f1, 12000, cudaEnableDefault,
                                             &q1) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &f2, 12000,
                                             cudaEnableDefault, &q2) != cudaSuccess ||
            q2 != cudaDriverEntryPointSuccess)
            return DLC_STATUS_EXECUTION_FAILED;
        d.scratch = ptr;
        d.wpack = wptr;
        d.sm_count = sms;
        d.encode_tiled = reinterpret_cast<EncodeTiledFn>(f1);
        d.encode_im2col = reinterpret_cast<EncodeIm2colFn>(f2);
        d.ready = 1;
    }
    *out = &d;
    return DLC_STATUS_SUCCESS;
}
}  // namespace

dlcStatus_t dlcConvolutionForwardNoAlloc(void *stream, const float *alpha,
                                         dlcTensorDescriptor_t xd, const void *x,
                                         dlcFilterDescriptor_t wd, const void *w,
                                         dlcConvolutionDescriptor_t cd, const float *beta,
                                         dlcTensorDescriptor_t yd, void *y, int *status) {
    if (!alpha || !beta) return DLC_STATUS_BAD_PARAM;
    if ((uintptr_t)status % sizeof(int)) return DLC_STATUS_BAD_PARAM;
    ConvProblem pb;
    dlcStatus_t st = resolve(xd, x, wd, w, cd, yd, y, true, pb);
    if (st != DLC_STATUS_SUCCESS) return st;
    pb.alpha = *alpha;
    pb.beta = *beta;
    if (pb.math == DLC_MATH_FP32) return DLC_STATUS_NOT_SUPPORTED;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    NoAllocDevice *nd = nullptr;
    st = noalloc_setup(dev, &nd);
    if (st != DLC_STATUS_SUCCESS) return st;

    // A context on the stack: no handle, no allocation.
    dlcContext ctx;
    ctx.device = dev;
    ctx.sm_count = nd->sm_count;
    ctx.stream = static_cast<cudaStream_t>(stream);
    ctx.h_err = nullptr;
    ctx.d_err = status ? status : nd->scratch + DLC_NOALLOC_MAX_TILES;
    ctx.sk_flags = nd->scratch;
    ctx.wpack = nd->wpack;
    ctx.wpack_bytes = DLC_WPACK_BYTES;
    ctx.encode_tiled = nd->encode_tiled;
    ctx.encode_im2col = nd->encode_im2col;
    if (pb.math == DLC_MATH_FP64) return DLC_STATUS_NOT_SUPPORTED;
    const dlcKernel_t k = dlc_tc_variant(&ctx, pb);
    if (k == DLC_KERNEL_NONE || k == DLC_KERNEL_FFMA) return DLC_STATUS_NOT_SUPPORTED;
    if (pb.flip && k != DLC_KERNEL_TC_IM2COL_PAIR) mirror_filter_view(pb);
    // the flags and the error words start at zero on every call
    if (cudaMemsetAsync(nd->scratch, 0, (DLC_NOALLOC_MAX_TILES + 2) * sizeof(int), ctx.stream) !=
            cudaSuccess ||
        (status && cudaMemsetAsync(status, 0, 2 * sizeof(int), ctx.stream) != cudaSuccess))
        return DLC_STATUS_EXECUTION_FAILED;
    return dlc_launch_tc(&ctx, pb, k);
}

dlcStatus_t dlcSetConvolutionMode(dlcConvolutionDescriptor_t d, dlcConvolutionMode_t mode) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    if (!d->set) return DLC_STATUS_NOT_INITIALIZED;
    if (mode != DLC_CROSS_CORRELATION && mode != DLC_CONVOLUTION) return DLC_STATUS_BAD_PARAM;
    d->mode = mode;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetConvolutionMode(dlcConvolutionDescriptor_t d, dlcConvolutionMode_t *mode) {
    if (!d || !mode) return DLC_STATUS_BAD_PARAM;
    if (!d->set) return DLC_STATUS_NOT_INITIALIZED;
    *mode = d->mode;
    return DLC_STATUS_SUCCESS;
}

// ---- backward routines -----------------------------------------------------------
dlcStatus_t dlcConvolutionBackwardData(dlcHandle_t h, const float *alpha,
                                       dlcFilterDescriptor_t wd, const void *w,
                                       dlcTensorDescriptor_t dyd, const void *dy,
                                       dlcConvolutionDescriptor_t cd, const float *beta,
                                       dlcTensorDescriptor_t dxd, void *dx) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!alpha || !beta) return DLC_STATUS_BAD_PARAM;
    BwdProblem bp;
    dlcStatus_t st = resolve_bwd(dxd, dx, wd, w, cd, dyd, dy, 0, true, bp);
    if (st != DLC_STATUS_SUCCESS) return st;
    bp.alpha = *alpha;
    bp.beta = *beta;
    st = pending_device_error(h);
    if (st != DLC_STATUS_SUCCESS) return st;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return DLC_STATUS_BAD_PARAM;
    return dlc_launch_dgrad(h, bp);
}

dlcStatus_t dlcConvolutionBackwardFilter(dlcHandle_t h, const float *alpha,
                                         dlcTensorDescriptor_t xd, const void *x,
                                         dlcTensorDescriptor_t dyd, const void *dy,
                                         dlcConvolutionDescriptor_t cd, const float *beta,
                                         dlcFilterDescriptor_t dwd, void *dw) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!alpha || !beta) return DLC_STATUS_BAD_PARAM;
    BwdProblem bp;
    dlcStatus_t st = resolve_bwd(xd, x, dwd, dw, cd, dyd, dy, 1, true, bp);
    if (st != DLC_STATUS_SUCCESS) return st;
    bp.alpha = *alpha;
    bp.beta = *beta;
    st = pending_device_error(h);
    if (st != DLC_STATUS_SUCCESS) return st;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return DLC_STATUS_BAD_PARAM;
    return dlc_launch_wgrad(h, bp);
}

dlcStatus_t dlcGetConvolutionBackwardDataWorkspaceSize(dlcHandle_t h, dlcFilterDescriptor_t wd,
                                                       dlcTensorDescriptor_t dyd,
                                                       dlcConvolutionDescriptor_t cd,
                                                       dlcTensorDescriptor_t dxd, size_t *bytes) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!bytes) return DLC_STATUS_BAD_PARAM;
    BwdProblem bp;
    dlcStatus_t st = resolve_bwd(dxd, nullptr, wd, nullptr, cd, dyd, nullptr, 0, false, bp);
    if (st != DLC_STATUS_SUCCESS) return st;
    *bytes = 0;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetConvolutionBackwardFilterWorkspaceSize(dlcHandle_t h, dlcTensorDescriptor_t xd,
                                                         dlcTensorDescriptor_t dyd,
                                                         dlcConvolutionDescriptor_t cd,
                                                         dlcFilterDescriptor_t dwd, size_t *bytes) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!bytes) return DLC_STATUS_BAD_PARAM;
    BwdProblem bp;
    dlcStatus_t st = resolve_bwd(xd, nullptr, dwd, nullptr, cd, dyd, nullptr, 1, false, bp);
    if (st != DLC_STATUS_SUCCESS) return st;
    *bytes = 0;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetConvolutionBackwardDataKernel(dlcHandle_t h, dlcFilterDescriptor_t wd,
                                                const void *w, dlcTensorDescriptor_t dyd,
                                                const void *dy, dlcConvolutionDescriptor_t cd,
                                                dlcTensorDescriptor_t dxd, const void *dx,
                                                dlcKernel_t *kernel) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!kernel) return DLC_STATUS_BAD_PARAM;
    BwdProblem bp;
    dlcStatus_t st = resolve_bwd(dxd, dx, wd, w, cd, dyd, dy, 0, false, bp);
    if (st != DLC_STATUS_SUCCESS) return st;
    *kernel = dlc_dgrad_variant(h, bp);
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetConvolutionBackwardFilterKernel(dlcHandle_t h, dlcTensorDescriptor_t xd,
                                                  const void *x, dlcTensorDescriptor_t dyd,
                                                  const void *dy, dlcConvolutionDescriptor_t cd,
                                                  dlcFilterDescriptor_t dwd, const void *dw,
                                                  dlcKernel_t *kernel) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!kernel) return DLC_STATUS_BAD_PARAM;
    BwdProblem bp;
    dlcStatus_t st = resolve_bwd(xd, x, dwd, dw, cd, dyd, dy, 1, false, bp);
    if (st != DLC_STATUS_SUCCESS) return st;
    *kernel = dlc_wgrad_variant(h, bp);
    return DLC_STATUS_SUCCESS;
}

// ---- pooling and activation ---------------------------------------------------
dlcStatus_t dlcCreatePoolingDescriptor(dlcPoolingDescriptor_t *d) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    *d = new (std::nothrow) dlcPoolingStruct();
    return *d ? DLC_STATUS_SUCCESS : DLC_STATUS_ALLOC_FAILED;
}

dlcStatus_t dlcDestroyPoolingDescriptor(dlcPoolingDescriptor_t d) {
    delete d;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcSetPooling2dDescriptor(dlcPoolingDescriptor_t d, dlcPoolingMode_t mode, int r, int s,
                                      int pt, int pb, int pl, int pr, int u, int v) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    if (mode != DLC_POOLING_MAX && mode != DLC_POOLING_AVERAGE_COUNT_INCLUDE_PADDING &&
        mode != DLC_POOLING_AVERAGE_COUNT_EXCLUDE_PADDING)
        return DLC_STATUS_BAD_PARAM;
    const int big = 1 << 20;
    if (r < 1 || s < 1 || u < 1 || v < 1 || r > big || s > big || u > big || v > big)
        return DLC_STATUS_BAD_PARAM;
    if (pt < 0 || pb < 0 || pl < 0 || pr < 0 || pt >= r || pb >= r || pl >= s || pr >= s)
        return DLC_STATUS_BAD_PARAM;
    d->mode = mode;
    d->r = r; d->s = s;
    d->pad_top = pt; d->pad_bottom = pb; d->pad_left = pl; d->pad_right = pr;
    d->u = u; d->v = v;
    d->set = 1;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetPooling2dDescriptor(dlcPoolingDescriptor_t d, dlcPoolingMode_t *mode, int *r,
                                      int *s, int *pt, int *pb, int *pl, int *pr, int *u, int *v) {
    if (!d) return DLC_STATUS_BAD_PARAM;
    if (!d->set) return DLC_STATUS_NOT_INITIALIZED;
    if (mode) *mode = d->mode;
    if (r) *r = d->r;
    if (s) *s = d->s;
    if (pt) *pt = d->pad_top;
    if (pb) *pb = d->pad_bottom;
    if (pl) *pl = d->pad_left;
    if (pr) *pr = d->pad_right;
    if (u) *u = d->u;
    if (v) *v = d->v;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcGetPooling2dForwardOutputDim(dlcPoolingDescriptor_t d, dlcTensorDescriptor_t xd,
                                            int *n, int *c, int *p, int *q) {
    if (!d || !xd || !n || !c || !p || !q) return DLC_STATUS_BAD_PARAM;
    if (!d->set || !xd->set) return DLC_STATUS_NOT_INITIALIZED;
    const int64_t P = out_extent(xd->h, d->pad_top, d->pad_bottom, d->r, 1, d->u);
    const int64_t Q = out_extent(xd->w, d->pad_left, d->pad_right, d->s, 1, d->v);
    if (P < 1 || Q < 1 || P > INT32_MAX || Q > INT32_MAX) return DLC_STATUS_BAD_PARAM;
    *n = xd->n; *c = xd->c; *p = (int)P; *q = (int)Q;
    return DLC_STATUS_SUCCESS;
}

namespace {
dlcStatus_t resolve_pool(dlcPoolingDescriptor_t d, dlcTensorDescriptor_t xd, const void *x,
                         dlcTensorDescriptor_t yd, const void *y, bool check_ptrs, PoolProblem &pp) {
    if (!d || !xd || !yd) return DLC_STATUS_BAD_PARAM;
    if (!d->set || !xd->set || !yd->set) return DLC_STATUS_NOT_INITIALIZED;
    int n, c, p, q;
    dlcStatus_t st = dlcGetPooling2dForwardOutputDim(d, xd, &n, &c, &p, &q);
    if (st != DLC_STATUS_SUCCESS) return st;
    if (yd->n != n || yd->c != c || yd->h != p || yd->w != q) return DLC_STATUS_BAD_PARAM;
    if (!out_ok(xd->dtype, yd->dtype)) return DLC_STATUS_NOT_SUPPORTED;
    pp.N = n; pp.C = c; pp.H = xd->h; pp.W = xd->w; pp.R = d->r; pp.S = d->s; pp.P = p; pp.Q = q;
    pp.pt = d->pad_top; pp.pl = d->pad_left; pp.u = d->u; pp.v = d->v; pp.mode = (int)d->mode;
    pp.xdt = xd->dtype; pp.ydt = yd->dtype;
    for (int i = 0; i < 4; ++i) {
        pp.xs[i] = xd->stride[i];
        pp.ys[i] = yd->stride[i];
    }
    pp.x = x; pp.y = const_cast<void *>(y);
    pp.alpha = 1.0; pp.beta = 0.0;
    const int64_t xext[4] = {pp.N, pp.C, pp.H, pp.W}, yext[4] = {pp.N, pp.C, pp.P, pp.Q};
    if (!strides_injective(yext, pp.ys, 4)) return DLC_STATUS_BAD_PARAM;
    const int64_t xmax = max_offset(xext, pp.xs, 4), ymax = max_offset(yext, pp.ys, 4);
    if (xmax >= ((int64_t)1 << 60) || ymax >= ((int64_t)1 << 60)) return DLC_STATUS_BAD_PARAM;
    if (check_ptrs) {
        if (!x || !y) return DLC_STATUS_BAD_PARAM;
        const size_t ex = elt_size(pp.xdt), ey = elt_size(pp.ydt);
        if ((uintptr_t)x % ex || (uintptr_t)y % ey) return DLC_STATUS_BAD_PARAM;
        const uintptr_t x0 = (uintptr_t)x, y0 = (uintptr_t)y;
        if (ranges_overlap(x0, x0 + (uintptr_t)(xmax + 1) * ex, y0, y0 + (uintptr_t)(ymax + 1) * ey))
            return DLC_STATUS_BAD_PARAM;
    }
    return DLC_STATUS_SUCCESS;
}
}  // namespace

dlcStatus_t dlcPoolingForward(dlcHandle_t h, dlcPoolingDescriptor_t d, const float *alpha,
                              dlcTensorDescriptor_t xd, const void *x, const float *beta,
                              dlcTensorDescriptor_t yd, void *y) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!alpha || !beta) return DLC_STATUS_BAD_PARAM;
    PoolProblem pp;
    dlcStatus_t st = resolve_pool(d, xd, x, yd, y, true, pp);
    if (st != DLC_STATUS_SUCCESS) return st;
    pp.alpha = *alpha;
    pp.beta = *beta;
    st = pending_device_error(h);
    if (st != DLC_STATUS_SUCCESS) return st;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return DLC_STATUS_BAD_PARAM;
    return dlc_launch_pool(h, pp);
}

dlcStatus_t dlcGetPoolingForwardKernel(dlcHandle_t h, dlcPoolingDescriptor_t d,
                                       dlcTensorDescriptor_t xd, const void *x,
                                       dlcTensorDescriptor_t yd, const void *y, dlcKernel_t *kernel) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!kernel) return DLC_STATUS_BAD_PARAM;
    PoolProblem pp;
    dlcStatus_t st = resolve_pool(d, xd, x, yd, y, false, pp);
    if (st != DLC_STATUS_SUCCESS) return st;
    *kernel = dlc_pool_variant(pp);
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlcActivationForward(dlcHandle_t h, dlcActivationMode_t mode, double coef,
                                 const float *alpha, dlcTensorDescriptor_t xd, const void *x,
                                 const float *beta, dlcTensorDescriptor_t yd, void *y) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (!alpha || !beta || !xd || !yd) return DLC_STATUS_BAD_PARAM;
    if (!xd->set || !yd->set) return DLC_STATUS_NOT_INITIALIZED;
    if (mode < DLC_ACTIVATION_IDENTITY || mode > DLC_ACTIVATION_CLIPPED_RELU) return DLC_STATUS_BAD_PARAM;
    if (xd->n != yd->n || xd->c != yd->c || xd->h != yd->h || xd->w != yd->w) return DLC_STATUS_BAD_PARAM;
    if (!out_ok(xd->dtype, yd->dtype)) return DLC_STATUS_NOT_SUPPORTED;
    if (!x || !y) return DLC_STATUS_BAD_PARAM;
    ActProblem ap;
    ap.N = xd->n; ap.C = xd->c; ap.H = xd->h; ap.W = xd->w; ap.mode = (int)mode;
    ap.xdt = xd->dtype; ap.ydt = yd->dtype;
    bool same = xd->dtype == yd->dtype;
    for (int i = 0; i < 4; ++i) {
        ap.xs[i] = xd->stride[i];
        ap.ys[i] = yd->stride[i];
        same = same && ap.xs[i] == ap.ys[i];
    }
    const int64_t ext[4] = {ap.N, ap.C, ap.H, ap.W};
    if (!strides_injective(ext, ap.ys, 4)) return DLC_STATUS_BAD_PARAM;
    const int64_t xmax = max_offset(ext, ap.xs, 4), ymax = max_offset(ext, ap.ys, 4);
    if (xmax >= ((int64_t)1 << 60) || ymax >= ((int64_t)1 << 60)) return DLC_STATUS_BAD_PARAM;
    const size_t ex = elt_size(ap.xdt), ey = elt_size(ap.ydt);
    if ((uintptr_t)x % ex || (uintptr_t)y % ey) return DLC_STATUS_BAD_PARAM;
    const bool in_place = x == y && same;
    const uintptr_t x0 = (uintptr_t)x, y0 = (uintptr_t)y;
    if (!in_place &&
        ranges_overlap(x0, x0 + (uintptr_t)(xmax + 1) * ex, y0, y0 + (uintptr_t)(ymax + 1) * ey))
        return DLC_STATUS_BAD_PARAM;
    ap.x = x; ap.y = y;
    ap.alpha = *alpha; ap.beta = *beta; ap.coef = coef;
    dlcStatus_t st = pending_device_error(h);
    if (st != DLC_STATUS_SUCCESS) return st;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return DLC_STATUS_BAD_PARAM;
    return dlc_launch_activation(h, ap);
}

dlcStatus_t dlcDebugWaitTimeoutSelfTest(dlcHandle_t h, int timeout_us) {
    if (!h) return DLC_STATUS_NOT_INITIALIZED;
    if (timeout_us < 1 || timeout_us > 1000000) return DLC_STATUS_BAD_PARAM;
    return dlc_launch_wait_selftest(h, (unsigned long long)timeout_us * 1000ull);
}

}  // extern "C"
