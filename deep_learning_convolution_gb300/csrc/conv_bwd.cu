// conv_bwd.cu -- the backward routines: gradient of the forward convolution
// with respect to its data (dgrad) and to its filters (wgrad).
//
// The cuDNN page's method section lists, beside the forward convolution,
// routines for backward propagation; the maxDNN page's research questions
// carry the forward kernel's techniques over to it.  Both are the plain
// derivatives of the forward sum
//
//   dx[n,c,h,w] = sum over k, r, s and the outputs (p, q) that read input
//                 pixel (h, w) through tap (r, s) (p*u + r*dh - pad_top = h,
//                 q*v + s*dw - pad_left = w) of dy[n,k,p,q] * w[k,c,r,s],
//   dw[k,c,r,s] = sum_{n,p,q} dy[n,k,p,q] * X(n, c, p*u + r*dh - pad_top,
//                                               q*v + s*dw - pad_left),
//
// with dx = alpha * dgrad + beta * dx and dw = alpha * wgrad + beta * dw.
//
// dgrad on the tensor cores is a set of forward problems: splitting dx by the
// phase (h + pad_top) mod u, (w + pad_left) mod v, each phase is a stride-1
// correlation of dy with the filter taps of that phase, mirrored, whose
// output channels are the forward input channels.  The SM-pair kernel runs
// each phase with the filters read transposed (the output channel index c is
// contiguous in KRSC storage, so the filter operand is MN-major) and mirrored
// taps, writing its phase of dx through strides; phases without taps only
// scale dx by beta.  Everything else (other layouts, dilation, FP32 and FP64
// math) takes the direct kernels below, which evaluate the sums above per
// output element.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "internal.h"

namespace {

struct BwdParams {
    int N, C, H, W, K, R, S, P, Q;
    int pt, pl, u, v, dh, dw;
    int flip;
    long long xs[4], ws[4], dys[4];
    const void *x;    // x (wgrad) or dx (dgrad)
    const void *w;    // w (dgrad) or dw (wgrad)
    const void *dy;
    float alpha, beta;
    double alpha_d, beta_d;
    int c_fastest;    // dgrad: enumerate dx with c innermost
    long long red_chunk;  // wgrad: (n, p, q) per split; 0 = no split
};

template <typename T> struct Num;
template <> struct Num<float> {
    using acc = float;
    __device__ static float ld(const float *p, long long o) { return __ldg(p + o); }
    __device__ static void st(float *p, long long o, float v) { p[o] = v; }
};
template <> struct Num<unsigned short> {  // BF16 storage
    using acc = float;
    __device__ static float ld(const unsigned short *p, long long o) {
        return __uint_as_float(static_cast<unsigned int>(__ldg(p + o)) << 16);
    }
    __device__ static void st(unsigned short *p, long long o, float v) {
        __nv_bfloat16 b = __float2bfloat16_rn(v);
        p[o] = *reinterpret_cast<unsigned short *>(&b);
    }
};
template <> struct Num<double> {
    using acc = double;
    __device__ static double ld(const double *p, long long o) { return __ldg(p + o); }
    __device__ static void st(double *p, long long o, double v) { p[o] = v; }
};

template <typename ACC> __device__ __forceinline__ ACC fma_acc(ACC a, ACC b, ACC c);
template <> __device__ __forceinline__ float fma_acc(float a, float b, float c) { return __fmaf_rn(a, b, c); }
template <> __device__ __forceinline__ double fma_acc(double a, double b, double c) { return __fma_rn(a, b, c); }

template <typename ACC> __device__ __forceinline__ ACC alpha_of(const BwdParams &p);
template <> __device__ __forceinline__ float alpha_of<float>(const BwdParams &p) { return p.alpha; }
template <> __device__ __forceinline__ double alpha_of<double>(const BwdParams &p) { return p.alpha_d; }
template <typename ACC> __device__ __forceinline__ ACC beta_of(const BwdParams &p);
template <> __device__ __forceinline__ float beta_of<float>(const BwdParams &p) { return p.beta; }
template <> __device__ __forceinline__ double beta_of<double>(const BwdParams &p) { return p.beta_d; }

// One dx element per thread: the taps (r, s) whose output (p, q) exists, and
// every filter k, in the order r, s, k.
template <typename TI, typename TO>
__global__ void __launch_bounds__(256) dgrad_direct_kernel(const __grid_constant__ BwdParams p) {
    using ACC = typename Num<TI>::acc;
    const TI *dy = static_cast<const TI *>(p.dy);
    const TI *w = static_cast<const TI *>(p.w);
    TO *dx = static_cast<TO *>(const_cast<void *>(p.x));
    const long long total = (long long)p.N * p.C * p.H * p.W;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        int n, c, h, wi;
        long long t = idx;
        if (p.c_fastest) {
            c = (int)(t % p.C); t /= p.C;
            wi = (int)(t % p.W); t /= p.W;
            h = (int)(t % p.H); t /= p.H;
            n = (int)t;
        } else {
            wi = (int)(t % p.W); t /= p.W;
            h = (int)(t % p.H); t /= p.H;
            c = (int)(t % p.C); t /= p.C;
            n = (int)t;
        }
        ACC acc = 0;
        for (int r = 0; r < p.R; ++r) {
            const int th = h + p.pt - r * p.dh;
            if (th < 0 || th % p.u) continue;
            const int op = th / p.u;
            if (op >= p.P) continue;
            const int rr = p.flip ? p.R - 1 - r : r;
            for (int s = 0; s < p.S; ++s) {
                const int tw = wi + p.pl - s * p.dw;
                if (tw < 0 || tw % p.v) continue;
                const int oq = tw / p.v;
                if (oq >= p.Q) continue;
                const int ss = p.flip ? p.S - 1 - s : s;
                const long long dyo = (long long)n * p.dys[0] + (long long)op * p.dys[2] +
                                      (long long)oq * p.dys[3];
                const long long wo = (long long)c * p.ws[1] + (long long)rr * p.ws[2] +
                                     (long long)ss * p.ws[3];
                for (int k = 0; k < p.K; ++k)
                    acc = fma_acc<ACC>(Num<TI>::ld(dy, dyo + (long long)k * p.dys[1]),
                                       Num<TI>::ld(w, wo + (long long)k * p.ws[0]), acc);
            }
        }
        const long long o = (long long)n * p.xs[0] + (long long)c * p.xs[1] + (long long)h * p.xs[2] +
                            (long long)wi * p.xs[3];
        ACC val = alpha_of<ACC>(p) * acc;
        if (beta_of<ACC>(p) != 0) val = fma_acc<ACC>(beta_of<ACC>(p), (ACC)Num<TO>::ld(dx, o), val);
        Num<TO>::st(dx, o, (typename Num<TO>::acc)val);
    }
}

// dw[k,c,r,s] over one chunk of the (n, p, q) reduction per thread.  With a
// split (red_chunk > 0) the chunks' partial sums are added into dw (FP32 or
// FP64 storage, scaled by beta beforehand); otherwise each thread owns its
// element and applies alpha and beta itself.
template <typename TI, typename TO>
__global__ void __launch_bounds__(256) wgrad_direct_kernel(const __grid_constant__ BwdParams p) {
    using ACC = typename Num<TI>::acc;
    const TI *x = static_cast<const TI *>(p.x);
    const TI *dy = static_cast<const TI *>(p.dy);
    TO *dw = static_cast<TO *>(const_cast<void *>(p.w));
    const long long elems = (long long)p.K * p.C * p.R * p.S;
    const long long red = (long long)p.N * p.P * p.Q;
    const long long chunk = p.red_chunk > 0 ? p.red_chunk : red;
    const long long splits = (red + chunk - 1) / chunk;
    const long long total = elems * splits;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long e = idx % elems, sp = idx / elems;
        long long t = e;
        const int c = (int)(t % p.C); t /= p.C;
        const int s = (int)(t % p.S); t /= p.S;
        const int r = (int)(t % p.R); t /= p.R;
        const int k = (int)t;
        const int rr = p.flip ? p.R - 1 - r : r, ss = p.flip ? p.S - 1 - s : s;
        ACC acc = 0;
        const long long j1 = min(red, (sp + 1) * chunk);
        for (long long j = sp * chunk; j < j1; ++j) {
            const int oq = (int)(j % p.Q);
            const long long j2 = j / p.Q;
            const int op = (int)(j2 % p.P), n = (int)(j2 / p.P);
            const int h = op * p.u + rr * p.dh - p.pt;
            const int wi = oq * p.v + ss * p.dw - p.pl;
            if (h < 0 || h >= p.H || wi < 0 || wi >= p.W) continue;
            acc = fma_acc<ACC>(
                Num<TI>::ld(dy, (long long)n * p.dys[0] + (long long)k * p.dys[1] +
                                    (long long)op * p.dys[2] + (long long)oq * p.dys[3]),
                Num<TI>::ld(x, (long long)n * p.xs[0] + (long long)c * p.xs[1] + (long long)h * p.xs[2] +
                                   (long long)wi * p.xs[3]),
                acc);
        }
        const long long o = (long long)k * p.ws[0] + (long long)c * p.ws[1] + (long long)r * p.ws[2] +
                            (long long)s * p.ws[3];
        if (p.red_chunk > 0) {
            if constexpr (sizeof(TO) >= 4) atomicAdd(dw + o, (TO)(alpha_of<ACC>(p) * acc));
        } else {
            ACC val = alpha_of<ACC>(p) * acc;
            if (beta_of<ACC>(p) != 0) val = fma_acc<ACC>(beta_of<ACC>(p), (ACC)Num<TO>::ld(dw, o), val);
            Num<TO>::st(dw, o, (typename Num<TO>::acc)val);
        }
    }
}

// y = beta * y over a strided 4-D view (beta == 0 writes zeros).
template <typename T>
__global__ void __launch_bounds__(256) scale_kernel(T *y, long long d0, long long d1, long long d2,
                                                    long long d3, long long s0, long long s1,
                                                    long long s2, long long s3, double beta) {
    const long long total = d0 * d1 * d2 * d3;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        long long t = idx;
        const long long i3 = t % d3; t /= d3;
        const long long i2 = t % d2; t /= d2;
        const long long i1 = t % d1;
        const long long i0 = t / d1;
        const long long o = i0 * s0 + i1 * s1 + i2 * s2 + i3 * s3;
        using ACC = typename Num<T>::acc;
        Num<T>::st(y, o, beta == 0.0 ? (ACC)0 : (ACC)(beta * (double)Num<T>::ld(y, o)));
    }
}

// y = beta * y over n dense elements (beta != 0).
template <typename T>
__global__ void __launch_bounds__(256) scale_flat_kernel(T *y, long long n, double beta) {
    using ACC = typename Num<T>::acc;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        Num<T>::st(y, i, (ACC)(beta * (double)Num<T>::ld(y, i)));
}

// True if the strides of the 4-D view cover exactly the offsets 0 .. n-1.
bool dense_view(const long long *dims, const int64_t *str) {
    int idx[4] = {0, 1, 2, 3};
    std::sort(idx, idx + 4, [&](int a, int b) { return str[a] < str[b]; });
    long long expect = 1;
    for (int i = 0; i < 4; ++i) {
        const int d = idx[i];
        if (dims[d] == 1) continue;
        if (str[d] != expect) return false;
        expect *= dims[d];
    }
    return true;
}

int grid_for(const dlcContext *ctx, long long total) {
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)ctx->sm_count * 16;
    return (int)std::max(1LL, std::min(blocks, cap));
}

template <typename T>
dlcStatus_t launch_scale(dlcContext *ctx, void *y, const long long *dims, const int64_t *str,
                         double beta) {
    const long long total = dims[0] * dims[1] * dims[2] * dims[3];
    if (total == 0) return DLC_STATUS_SUCCESS;
    if (dense_view(dims, str)) {
        // a dense tensor: zeros by a memset (all-zero bits are +0 in every
        // storage type), other factors in one flat pass without index math
        if (beta == 0.0)
            return cudaMemsetAsync(y, 0, (size_t)total * sizeof(T), ctx->stream) == cudaSuccess
                       ? DLC_STATUS_SUCCESS
                       : DLC_STATUS_EXECUTION_FAILED;
        if (beta == 1.0) return DLC_STATUS_SUCCESS;
        scale_flat_kernel<T><<<grid_for(ctx, total), 256, 0, ctx->stream>>>(static_cast<T *>(y), total, beta);
        if (cudaGetLastError() != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
        ctx->launches += 1;
        return DLC_STATUS_SUCCESS;
    }
    scale_kernel<T><<<grid_for(ctx, total), 256, 0, ctx->stream>>>(
        static_cast<T *>(y), dims[0], dims[1], dims[2], dims[3], str[0], str[1], str[2], str[3], beta);
    if (cudaGetLastError() != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t scale_any(dlcContext *ctx, dlcDataType_t dt, void *y, const long long *dims,
                      const int64_t *str, double beta) {
    if (dt == DLC_DATA_BFLOAT16) return launch_scale<unsigned short>(ctx, y, dims, str, beta);
    if (dt == DLC_DATA_DOUBLE) return launch_scale<double>(ctx, y, dims, str, beta);
    return launch_scale<float>(ctx, y, dims, str, beta);
}

BwdParams params_of(const BwdProblem &bp) {
    BwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.N = bp.N; p.C = bp.C; p.H = bp.H; p.W = bp.W; p.K = bp.K; p.R = bp.R; p.S = bp.S;
    p.P = bp.P; p.Q = bp.Q;
    p.pt = bp.pt; p.pl = bp.pl; p.u = bp.u; p.v = bp.v; p.dh = bp.dh; p.dw = bp.dw;
    p.flip = bp.flip;
    for (int i = 0; i < 4; ++i) {
        p.xs[i] = bp.xs[i];
        p.ws[i] = bp.ws[i];
        p.dys[i] = bp.dys[i];
    }
    p.x = bp.x; p.w = bp.w; p.dy = bp.dy;
    p.alpha = (float)bp.alpha; p.beta = (float)bp.beta;
    p.alpha_d = bp.alpha; p.beta_d = bp.beta;
    return p;
}

template <typename TI, typename TO>
cudaError_t launch_dgrad_direct(const BwdParams &p, int grid, cudaStream_t st) {
    dgrad_direct_kernel<TI, TO><<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t launch_wgrad_direct(const BwdParams &p, int grid, cudaStream_t st) {
    wgrad_direct_kernel<TI, TO><<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

// One phase of the data gradient as a forward problem for the SM-pair
// kernel, or false when that kernel cannot take it.  (ph, pw) is the phase of
// (h + pad_top, w + pad_left) modulo the strides.
bool phase_problem(const BwdProblem &bp, int ph, int pw, ConvProblem &f, bool *empty) {
    *empty = false;
    // taps of this phase: r = ph + u*i, i < Rp (dilation 1)
    const int Rp = ph < bp.R ? (bp.R - ph + bp.u - 1) / bp.u : 0;
    const int Sp = pw < bp.S ? (bp.S - pw + bp.v - 1) / bp.v : 0;
    // first dx row/column of the phase and the count of them
    const int h0 = ((ph - bp.pt) % bp.u + bp.u) % bp.u;
    const int w0 = ((pw - bp.pl) % bp.v + bp.v) % bp.v;
    const int Hp = h0 < bp.H ? (bp.H - h0 + bp.u - 1) / bp.u : 0;
    const int Wp = w0 < bp.W ? (bp.W - w0 + bp.v - 1) / bp.v : 0;
    if (Hp == 0 || Wp == 0) {
        *empty = true;  // no dx elements in this phase
        return true;
    }
    f = ConvProblem();
    f.math = bp.math;
    f.xdt = bp.in_dt;
    f.ydt = bp.out_dt;
    f.wfmt = DLC_TENSOR_NHWC;
    f.N = bp.N;
    f.C = bp.K;           // reduction channels: the filters
    f.H = bp.P;
    f.W = bp.Q;           // dy's extent
    f.K = bp.C;           // output channels: the forward input channels
    f.R = Rp;
    f.S = Sp;
    f.P = Hp;
    f.Q = Wp;
    f.u = f.v = f.dh = f.dw = 1;
    // dx row h0 + u*m reads dy rows a0 + m - i for taps i, a0 = (h0 + pt - ph)/u:
    // a stride-1 correlation over mirrored taps with top pad Rp - 1 - a0
    const int a0 = (h0 + bp.pt - ph) / bp.u, b0 = (w0 + bp.pl - pw) / bp.v;
    f.pt = Rp - 1 - a0;
    f.pl = Sp - 1 - b0;
    f.pb = Hp + Rp - 1 - bp.P - f.pt;
    f.pr = Wp + Sp - 1 - bp.Q - f.pl;
    const long long eo = dlc_dtype_bytes(bp.out_dt);
    f.y = static_cast<char *>(const_cast<void *>(bp.x)) +
          eo * ((long long)h0 * bp.xs[2] + (long long)w0 * bp.xs[3]);
    f.ys[0] = bp.xs[0];
    f.ys[1] = bp.xs[1];
    f.ys[2] = bp.xs[2] * bp.u;
    f.ys[3] = bp.xs[3] * bp.v;
    if (Rp == 0 || Sp == 0) {
        *empty = true;  // no tap reaches these dx elements: dx = beta * dx there
        return true;
    }
    f.x = bp.dy;
    for (int i = 0; i < 4; ++i) f.xs[i] = bp.dys[i];
    // The forward tap r = ph + u*i reads filter row r (cross-correlation) or
    // R-1-r (convolution mode).  The phase problem's tap i' = Rp-1-i then
    // reads filter rows ph + u*(Rp-1-i') -- mirrored taps of a filter view
    // based at row ph -- or R-1-ph-u*(Rp-1) + u*i' -- plain taps of a view
    // based at that row.
    const long long e = dlc_dtype_bytes(bp.in_dt);
    const long long r0 = bp.flip ? bp.R - 1 - ph - (long long)bp.u * (Rp - 1) : ph;
    const long long s0 = bp.flip ? bp.S - 1 - pw - (long long)bp.v * (Sp - 1) : pw;
    f.w = static_cast<const char *>(bp.w) + e * (r0 * bp.ws[2] + s0 * bp.ws[3]);
    f.ws[0] = bp.ws[1];
    f.ws[1] = bp.ws[0];
    f.ws[2] = bp.ws[2] * bp.u;
    f.ws[3] = bp.ws[3] * bp.v;
    f.w_mn = 1;
    f.flip = bp.flip ? 0 : 1;
    f.bias = nullptr;
    f.alpha = (float)bp.alpha;
    f.beta = (float)bp.beta;
    f.relu = 0;
    return dlc_im2col_ok(f) && f.ws[0] == 1;
}

}  // namespace

dlcKernel_t dlc_dgrad_variant(const dlcContext *ctx, const BwdProblem &bp) {
    const bool tc = (bp.math == DLC_MATH_BF16 && bp.in_dt == DLC_DATA_BFLOAT16);
    if (!tc || bp.dh != 1 || bp.dw != 1 || !dlc_pair_enabled(ctx) || bp.wfmt != DLC_TENSOR_NHWC ||
        bp.out_dt == DLC_DATA_DOUBLE)
        return DLC_KERNEL_DIRECT;
    for (int ph = 0; ph < bp.u; ++ph)
        for (int pw = 0; pw < bp.v; ++pw) {
            ConvProblem f;
            bool empty;
            if (!phase_problem(bp, ph, pw, f, &empty)) return DLC_KERNEL_DIRECT;
        }
    return DLC_KERNEL_TC_IM2COL_PAIR;
}

dlcStatus_t dlc_launch_dgrad(dlcContext *ctx, const BwdProblem &bp) {
    if (dlc_dgrad_variant(ctx, bp) == DLC_KERNEL_TC_IM2COL_PAIR) {
        for (int ph = 0; ph < bp.u; ++ph)
            for (int pw = 0; pw < bp.v; ++pw) {
                ConvProblem f;
                bool empty;
                phase_problem(bp, ph, pw, f, &empty);
                if (empty) {
                    if (f.P == 0 || f.Q == 0 || f.y == nullptr) continue;  // no dx elements
                    const long long dims[4] = {bp.N, bp.C, f.P, f.Q};
                    dlcStatus_t st = scale_any(ctx, bp.out_dt, f.y, dims, f.ys, bp.beta);
                    if (st != DLC_STATUS_SUCCESS) return st;
                    continue;
                }
                dlcStatus_t st = dlc_launch_pair(ctx, f);
                if (st != DLC_STATUS_SUCCESS) return st;
            }
        return DLC_STATUS_SUCCESS;
    }
    BwdParams p = params_of(bp);
    p.c_fastest = bp.xs[1] == 1 ? 1 : 0;
    const int grid = grid_for(ctx, (long long)bp.N * bp.C * bp.H * bp.W);
    cudaError_t e;
    const dlcDataType_t ti = bp.in_dt, to = bp.out_dt;
    if (ti == DLC_DATA_DOUBLE && to == DLC_DATA_DOUBLE) e = launch_dgrad_direct<double, double>(p, grid, ctx->stream);
    else if (ti == DLC_DATA_FLOAT && to == DLC_DATA_FLOAT) e = launch_dgrad_direct<float, float>(p, grid, ctx->stream);
    else if (ti == DLC_DATA_FLOAT && to == DLC_DATA_BFLOAT16) e = launch_dgrad_direct<float, unsigned short>(p, grid, ctx->stream);
    else if (ti == DLC_DATA_BFLOAT16 && to == DLC_DATA_FLOAT) e = launch_dgrad_direct<unsigned short, float>(p, grid, ctx->stream);
    else if (ti == DLC_DATA_BFLOAT16 && to == DLC_DATA_BFLOAT16) e = launch_dgrad_direct<unsigned short, unsigned short>(p, grid, ctx->stream);
    else return DLC_STATUS_NOT_SUPPORTED;
    if (e != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}

dlcKernel_t dlc_wgrad_variant(const dlcContext *, const BwdProblem &bp) {
    // the tensor-core kernel writes dw in forward tap order; convolution mode
    // (mirrored taps) takes the direct kernel
    return (!bp.flip && dlc_wgrad_tc_ok(bp)) ? DLC_KERNEL_TC_WGRAD : DLC_KERNEL_DIRECT;
}

dlcStatus_t dlc_launch_wgrad(dlcContext *ctx, const BwdProblem &bp) {
    if (dlc_wgrad_variant(ctx, bp) == DLC_KERNEL_TC_WGRAD) {
        // dw = beta * dw first; the kernel adds alpha times its partial sums
        const long long dims[4] = {bp.K, bp.C, bp.R, bp.S};
        dlcStatus_t st = scale_any(ctx, bp.out_dt, const_cast<void *>(bp.w), dims, bp.ws, bp.beta);
        if (st != DLC_STATUS_SUCCESS) return st;
        return dlc_launch_wgrad_tc(ctx, bp);
    }
    BwdParams p = params_of(bp);
    const long long elems = (long long)bp.K * bp.C * bp.R * bp.S;
    const long long red = (long long)bp.N * bp.P * bp.Q;
    // split the (n, p, q) reduction when the filter alone cannot fill the GPU
    // (FP32 or FP64 dw: the partial sums are added atomically)
    const long long want = (long long)ctx->sm_count * 8 * 256;
    long long splits = 1;
    if (bp.out_dt != DLC_DATA_BFLOAT16 && !ctx->deterministic && elems < want && red > 256)
        splits = std::min((want + elems - 1) / elems, (red + 255) / 256);
    if (splits > 1) {
        p.red_chunk = (red + splits - 1) / splits;
        const long long dims[4] = {bp.K, bp.C, bp.R, bp.S};
        dlcStatus_t st = scale_any(ctx, bp.out_dt, const_cast<void *>(bp.w), dims, bp.ws, bp.beta);
        if (st != DLC_STATUS_SUCCESS) return st;
        splits = (red + p.red_chunk - 1) / p.red_chunk;
    }
    const int grid = grid_for(ctx, elems * splits);
    cudaError_t e;
    const dlcDataType_t ti = bp.in_dt, to = bp.out_dt;
    if (ti == DLC_DATA_DOUBLE && to == DLC_DATA_DOUBLE) e = launch_wgrad_direct<double, double>(p, grid, ctx->stream);
    else if (ti == DLC_DATA_FLOAT && to == DLC_DATA_FLOAT) e = launch_wgrad_direct<float, float>(p, grid, ctx->stream);
    else if (ti == DLC_DATA_FLOAT && to == DLC_DATA_BFLOAT16) e = launch_wgrad_direct<float, unsigned short>(p, grid, ctx->stream);
    else if (ti == DLC_DATA_BFLOAT16 && to == DLC_DATA_FLOAT) e = launch_wgrad_direct<unsigned short, float>(p, grid, ctx->stream);
    else if (ti == DLC_DATA_BFLOAT16 && to == DLC_DATA_BFLOAT16) e = launch_wgrad_direct<unsigned short, unsigned short>(p, grid, ctx->stream);
    else return DLC_STATUS_NOT_SUPPORTED;
    if (e != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}
