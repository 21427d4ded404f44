// conv_ffma.cu -- strict FP32 (and FP64) direct convolution on CUDA cores.
//
// Each thread owns output elements; the receptive-field dot product of the
// maxDNN page's method section is accumulated with fused multiply-adds in
// FP32, in the order c, r, s.  Taps that fall in the padding are skipped
// (x reads as zero there).  No packing and no workspace (zero-memory-overhead
// direct convolution page, method section).  Any strides, any layout, FP32 or
// BF16 storage (BF16 is widened exactly to FP32 before the products).  FP64
// math (DOUBLE storage; the cuDNN page's method section offers double
// precision) runs the same loop with double fused multiply-adds.
#include <cuda_bf16.h>

#include "internal.h"

namespace {

struct FfmaParams {
    int N, C, H, W, K, R, S, P, Q;
    int pt, pl, u, v, dh, dw;
    long long xs[4], ws[4], ys[4];
    const void *x;
    const void *w;
    void *y;
    const float *bias;
    float alpha, beta;
    int relu;
    int k_fastest;  // enumerate outputs with k innermost (y has unit k stride)
};

template <typename T>
__device__ __forceinline__ float load_f32(const T *p, long long off);

template <>
__device__ __forceinline__ float load_f32<float>(const float *p, long long off) {
    return __ldg(p + off);
}

template <>
__device__ __forceinline__ float load_f32<unsigned short>(const unsigned short *p, long long off) {
    return __uint_as_float(static_cast<unsigned int>(__ldg(p + off)) << 16);
}

// FP64 problems: every value, product and sum in double.
__global__ void __launch_bounds__(256) conv_fprop_dfma_kernel(const __grid_constant__ FfmaParams p) {
    const double *x = static_cast<const double *>(p.x);
    const double *w = static_cast<const double *>(p.w);
    double *y = static_cast<double *>(p.y);
    const long long total = (long long)p.N * p.K * p.P * p.Q;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        long long t = idx;
        int n, k, op, oq;
        if (p.k_fastest) {
            k = (int)(t % p.K); t /= p.K;
            oq = (int)(t % p.Q); t /= p.Q;
            op = (int)(t % p.P); t /= p.P;
            n = (int)t;
        } else {
            oq = (int)(t % p.Q); t /= p.Q;
            op = (int)(t % p.P); t /= p.P;
            k = (int)(t % p.K); t /= p.K;
            n = (int)t;
        }
        const double *xn = x + (long long)n * p.xs[0];
        const double *wk = w + (long long)k * p.ws[0];
        double acc = 0.0;
        for (int c = 0; c < p.C; ++c) {
            for (int r = 0; r < p.R; ++r) {
                const int h = op * p.u + r * p.dh - p.pt;
                if (h < 0 || h >= p.H) continue;
                for (int s = 0; s < p.S; ++s) {
                    const int wi = oq * p.v + s * p.dw - p.pl;
                    if (wi < 0 || wi >= p.W) continue;
                    acc = __fma_rn(__ldg(xn + c * p.xs[1] + h * p.xs[2] + wi * p.xs[3]),
                                   __ldg(wk + c * p.ws[1] + r * p.ws[2] + s * p.ws[3]), acc);
                }
            }
        }
        const long long yo = (long long)n * p.ys[0] + (long long)k * p.ys[1] +
                             (long long)op * p.ys[2] + (long long)oq * p.ys[3];
        double val = (double)p.alpha * acc;
        if (p.beta != 0.f) val = __fma_rn((double)p.beta, y[yo], val);
        if (p.bias) val += (double)__ldg(p.bias + k);
        if (p.relu) val = fmax(val, 0.0);
        y[yo] = val;
    }
}

template <typename TI, typename TO>
__global__ void __launch_bounds__(256) conv_fprop_ffma_kernel(const __grid_constant__ FfmaParams p) {
    const TI *x = static_cast<const TI *>(p.x);
    const TI *w = static_cast<const TI *>(p.w);
    TO *y = static_cast<TO *>(p.y);
    const long long total = (long long)p.N * p.K * p.P * p.Q;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        int n, k, op, oq;
        long long t = idx;
        if (p.k_fastest) {
            k = (int)(t % p.K); t /= p.K;
            oq = (int)(t % p.Q); t /= p.Q;
            op = (int)(t % p.P); t /= p.P;
            n = (int)t;
        } else {
            oq = (int)(t % p.Q); t /= p.Q;
            op = (int)(t % p.P); t /= p.P;
            k = (int)(t % p.K); t /= p.K;
            n = (int)t;
        }
        const TI *xn = x + (long long)n * p.xs[0];
        const TI *wk = w + (long long)k * p.ws[0];
        float acc = 0.f;
        for (int c = 0; c < p.C; ++c) {
            for (int r = 0; r < p.R; ++r) {
                const int h = op * p.u + r * p.dh - p.pt;
                if (h < 0 || h >= p.H) continue;
                for (int s = 0; s < p.S; ++s) {
                    const int wi = oq * p.v + s * p.dw - p.pl;
                    if (wi < 0 || wi >= p.W) continue;
                    const float xv = load_f32(xn, c * p.xs[1] + h * p.xs[2] + wi * p.xs[3]);
                    const float wv = load_f32(wk, c * p.ws[1] + r * p.ws[2] + s * p.ws[3]);
                    acc = __fmaf_rn(xv, wv, acc);
                }
            }
        }
        const long long yo = (long long)n * p.ys[0] + (long long)k * p.ys[1] +
                             (long long)op * p.ys[2] + (long long)oq * p.ys[3];
        float val = p.alpha * acc;
        if (p.beta != 0.f) {
            float old;
            if constexpr (sizeof(TO) == 4) old = y[yo];
            else old = __uint_as_float(static_cast<unsigned int>(y[yo]) << 16);
            val = __fmaf_rn(p.beta, old, val);
        }
        if (p.bias) val += __ldg(p.bias + k);
        if (p.relu) val = fmaxf(val, 0.f);
        if constexpr (sizeof(TO) == 4) {
            y[yo] = val;
        } else {
            __nv_bfloat16 b = __float2bfloat16_rn(val);
            y[yo] = *reinterpret_cast<unsigned short *>(&b);
        }
    }
}

template <typename TI, typename TO>
cudaError_t launch(const FfmaParams &fp, int grid, cudaStream_t st) {
    conv_fprop_ffma_kernel<TI, TO><<<grid, 256, 0, st>>>(fp);
    return cudaGetLastError();
}

}  // namespace

dlcStatus_t dlc_launch_ffma(dlcContext *ctx, const ConvProblem &pb) {
    FfmaParams fp;
    fp.N = pb.N; fp.C = pb.C; fp.H = pb.H; fp.W = pb.W; fp.K = pb.K; fp.R = pb.R; fp.S = pb.S;
    fp.P = pb.P; fp.Q = pb.Q;
    fp.pt = pb.pt; fp.pl = pb.pl; fp.u = pb.u; fp.v = pb.v; fp.dh = pb.dh; fp.dw = pb.dw;
    for (int i = 0; i < 4; ++i) {
        fp.xs[i] = pb.xs[i];
        fp.ws[i] = pb.ws[i];
        fp.ys[i] = pb.ys[i];
    }
    fp.x = pb.x; fp.w = pb.w; fp.y = pb.y; fp.bias = pb.bias;
    fp.alpha = pb.alpha; fp.beta = pb.beta; fp.relu = pb.relu;
    fp.k_fastest = (pb.ys[1] == 1) ? 1 : 0;
    const long long total = (long long)pb.N * pb.K * pb.P * pb.Q;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)ctx->sm_count * 16;
    int grid = (int)(blocks < cap ? blocks : cap);
    if (grid < 1) grid = 1;
    cudaError_t e;
    const bool xb = pb.xdt == DLC_DATA_BFLOAT16, yb = pb.ydt == DLC_DATA_BFLOAT16;
    if (pb.xdt == DLC_DATA_DOUBLE) {
        if (pb.ydt != DLC_DATA_DOUBLE) return DLC_STATUS_NOT_SUPPORTED;
        conv_fprop_dfma_kernel<<<grid, 256, 0, ctx->stream>>>(fp);
        e = cudaGetLastError();
    } else if (!xb && !yb) e = launch<float, float>(fp, grid, ctx->stream);
    else if (!xb && yb) e = launch<float, unsigned short>(fp, grid, ctx->stream);
    else if (xb && !yb) e = launch<unsigned short, float>(fp, grid, ctx->stream);
    else e = launch<unsigned short, unsigned short>(fp, grid, ctx->stream);
    if (e != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}
