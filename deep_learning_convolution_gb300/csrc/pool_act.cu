// pool_act.cu -- pooling and activation forward.
//
// The cuDNN page's one-line summary and method section name pooling and
// activation functions as the library's other primitives beside convolution,
// with the same descriptors, arbitrary strides and caller-owned buffers.
//
//   pooling:    y[n,c,p,q] = alpha * POOL_{i<R, j<S, in image} x[n, c, p*u - pad_top + i,
//                                                            q*v - pad_left + j]
//                            + beta * y[n,c,p,q]
//               POOL = maximum, or sum / (R*S) (padding counted), or sum / (number
//               of in-image elements) (padding excluded); every pad is smaller than
//               the window, so no window is empty.
//   activation: y = alpha * f(x) + beta * y, f = identity, max(0,x), 1/(1+e^-x),
//               tanh x or min(max(0,x), coef).
//
// Both are memory-bound: they read x once from DRAM and write y once, so the
// kernels are sized for bandwidth.  With channels innermost (NHWC) each thread
// owns 16 bytes of channels of one output pixel and reads the window's pixels
// as 16-byte vectors (consecutive threads read consecutive bytes; a 3 x 3
// window's nine loads are issued together; a maximum of BF16 compares the
// stored pairs without widening them); dense tensors of one layout run
// the activation as a flat array of 16-byte vectors, four per thread in
// flight, one kernel per function; anything else takes one element per
// thread through the strides.
// Grids are a multiple of the SM count (grid-stride loops).  Sums and
// comparisons are in FP32 (FP64 for DOUBLE storage); BF16 is widened exactly.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "internal.h"

namespace {

template <typename T> struct Io;
template <> struct Io<float> {
    using acc = float;
    __device__ static float ld(const float *p, long long o) { return __ldg(p + o); }
    __device__ static void st(float *p, long long o, float v) { p[o] = v; }
};
template <> struct Io<unsigned short> {
    using acc = float;
    __device__ static float ld(const unsigned short *p, long long o) {
        return __uint_as_float(static_cast<unsigned int>(__ldg(p + o)) << 16);
    }
    __device__ static void st(unsigned short *p, long long o, float v) {
        __nv_bfloat16 b = __float2bfloat16_rn(v);
        p[o] = *reinterpret_cast<unsigned short *>(&b);
    }
};
template <> struct Io<double> {
    using acc = double;
    __device__ static double ld(const double *p, long long o) { return __ldg(p + o); }
    __device__ static void st(double *p, long long o, double v) { p[o] = v; }
};

struct PoolParams {
    int N, C, H, W, R, S, P, Q;
    int pt, pl, u, v, mode;
    int y_vec;  // channels-innermost y whose 16-byte channel chunks are aligned
    int raw_max;  // BF16 max pooling into BF16 y, alpha 1, beta 0: maxima stored as they are
    long long xs[4], ys[4];
    const void *x;
    void *y;
    double alpha, beta;
};

// Widen 16 bytes of x into V accumulators.
template <typename T, typename A, int V>
__device__ __forceinline__ void unpack16(const uint4 &q, A (&out)[V]) {
    if constexpr (sizeof(T) == 2) {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            out[2 * i] = __uint_as_float(w[i] << 16);
            out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else if constexpr (sizeof(T) == 4) {
        out[0] = __uint_as_float(q.x);
        out[1] = __uint_as_float(q.y);
        out[2] = __uint_as_float(q.z);
        out[3] = __uint_as_float(q.w);
    } else {
        out[0] = __hiloint2double((int)q.y, (int)q.x);
        out[1] = __hiloint2double((int)q.w, (int)q.z);
    }
}

// V consecutive results as 32-bit words of TO storage.
template <typename TO, typename A, int V>
__device__ __forceinline__ void pack_words(const A (&v)[V], uint32_t *w) {
    if constexpr (sizeof(TO) == 2) {
#pragma unroll
        for (int i = 0; i < V / 2; ++i) {
            const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn((float)v[2 * i]));
            const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn((float)v[2 * i + 1]));
            w[i] = lo | (hi << 16);
        }
    } else if constexpr (sizeof(TO) == 4) {
#pragma unroll
        for (int i = 0; i < V; ++i) w[i] = __float_as_uint((float)v[i]);
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const double d = (double)v[i];
            w[2 * i] = (uint32_t)__double2loint(d);
            w[2 * i + 1] = (uint32_t)__double2hiint(d);
        }
    }
}

// Stores V results (V * sizeof(TO) = 8, 16 or 32 bytes, address aligned to
// that size or 16) with vector stores.
template <typename TO, typename A, int V>
__device__ __forceinline__ void store_vec(TO *dst, const A (&v)[V]) {
    constexpr int WORDS = V * (int)sizeof(TO) / 4;
    uint32_t w[WORDS];
    pack_words<TO, A, V>(v, w);
    if constexpr (WORDS == 2) {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
    } else {
#pragma unroll
        for (int i = 0; i < WORDS / 4; ++i)
            reinterpret_cast<uint4 *>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
}

// Maximum or sum over a window of 16-byte vectors of channels.  fetch(i, j, q)
// loads tap (i, j) into q and says whether it lies in the image; FIX > 0 (a
// FIX x FIX window) issues every load before the first is used.  The maximum
// of BF16 storage compares the stored pairs in place (max.bf16x2, which like
// fmaxf passes over a NaN operand) and widens only the result: it is one of
// the stored values either way.  Sums are taken in A.  Returns the number of
// in-image taps.
// The BF16 maximum of a window: four pairs of stored values (from -inf when
// no tap is in the image); returns the number of in-image taps.
template <int FIX, typename F>
__device__ __forceinline__ int bf16_max_window(const F &fetch, int R, int S, __nv_bfloat162 (&m)[4]) {
    int count = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) m[k] = __bfloat162bfloat162(__ushort_as_bfloat16((unsigned short)0xff80u));
    auto take = [&](const uint4 &q) {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) m[k] = __hmax2(m[k], *reinterpret_cast<const __nv_bfloat162 *>(&w[k]));
    };
    if constexpr (FIX > 0) {
        uint4 q[FIX * FIX];
        bool in[FIX * FIX];
#pragma unroll
        for (int t = 0; t < FIX * FIX; ++t) in[t] = fetch(t / FIX, t % FIX, q[t]);
#pragma unroll
        for (int t = 0; t < FIX * FIX; ++t)
            if (in[t]) take(q[t]), ++count;
    } else {
        for (int i = 0; i < R; ++i)
            for (int j = 0; j < S; ++j) {
                uint4 q;
                if (fetch(i, j, q)) take(q), ++count;
            }
    }
    return count;
}

template <typename TI, typename A, int V, bool MAX, int FIX, typename F>
__device__ __forceinline__ int pool_window(const F &fetch, int R, int S, A (&acc)[V]) {
    int count = 0;
    if constexpr (MAX && sizeof(TI) == 2) {
        __nv_bfloat162 m[4];
        count = bf16_max_window<FIX>(fetch, R, S, m);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc[2 * k] = __bfloat162float(m[k].x);
            acc[2 * k + 1] = __bfloat162float(m[k].y);
        }
    } else {
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = MAX ? (A)-INFINITY : (A)0;
        auto take = [&](const uint4 &q) {
            A v[V];
            unpack16<TI, A, V>(q, v);
#pragma unroll
            for (int e = 0; e < V; ++e) {
                if constexpr (MAX)
                    acc[e] = sizeof(A) == 8 ? (A)fmax((double)acc[e], (double)v[e]) : (A)fmaxf((float)acc[e], (float)v[e]);
                else
                    acc[e] += v[e];
            }
        };
        if constexpr (FIX > 0) {
            uint4 q[FIX * FIX];
            bool in[FIX * FIX];
#pragma unroll
            for (int t = 0; t < FIX * FIX; ++t) in[t] = fetch(t / FIX, t % FIX, q[t]);
#pragma unroll
            for (int t = 0; t < FIX * FIX; ++t)
                if (in[t]) take(q[t]), ++count;
        } else {
            for (int i = 0; i < R; ++i)
                for (int j = 0; j < S; ++j) {
                    uint4 q;
                    if (fetch(i, j, q)) take(q), ++count;
                }
        }
    }
    return count;
}

// Channels-innermost pooling: one thread per (output pixel, 16-byte chunk of
// channels); C * sizeof(TI) is a multiple of 16 and both bases 16-byte aligned.
// I: the index type of the output enumeration (32-bit when the count fits,
// whose divisions are far cheaper than 64-bit ones).  FIX: 0, or the window
// size when it is FIX x FIX, whose loads are then all issued before the first
// is used.
template <typename TI, typename TO, typename I, int FIX>
__global__ void __launch_bounds__(256) pool_nhwc_kernel(const __grid_constant__ PoolParams p) {
    using A = typename Io<TI>::acc;
    constexpr int V = 16 / (int)sizeof(TI);
    const TI *x = static_cast<const TI *>(p.x);
    TO *y = static_cast<TO *>(p.y);
    const int chunks = p.C / V;
    const I total = (I)((long long)p.N * p.P * p.Q * chunks);
    for (I idx = (I)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (I)gridDim.x * blockDim.x) {
        I t = idx;
        const int ch = (int)(t % chunks); t /= chunks;
        const int oq = (int)(t % p.Q); t /= p.Q;
        const int op = (int)(t % p.P);
        const int n = (int)(t / p.P);
        A acc[V];
        const bool is_max = p.mode == 0;
        const TI *xn = x + (long long)n * p.xs[0] + (long long)ch * V;
        const int h0 = op * p.u - p.pt, w0 = oq * p.v - p.pl;
        auto fetch = [&](int i, int j, uint4 &q) {
            const int h = h0 + i, wi = w0 + j;
            const bool in = h >= 0 && h < p.H && wi >= 0 && wi < p.W;
            q = in ? __ldg(reinterpret_cast<const uint4 *>(xn + (long long)h * p.xs[2] + (long long)wi * p.xs[3]))
                   : make_uint4(0, 0, 0, 0);
            return in;
        };
        if constexpr (sizeof(TI) == 2 && std::is_same<TI, TO>::value) {
            if (p.raw_max) {  // the maxima are stored values: written back without widening
                __nv_bfloat162 m[4];
                bf16_max_window<FIX>(fetch, p.R, p.S, m);
                const long long yr = (long long)n * p.ys[0] + (long long)op * p.ys[2] + (long long)oq * p.ys[3] +
                                     (long long)ch * V;
                *reinterpret_cast<uint4 *>(y + yr) = *reinterpret_cast<const uint4 *>(m);
                continue;
            }
        }
        const int count = is_max ? pool_window<TI, A, V, true, FIX>(fetch, p.R, p.S, acc)
                                 : pool_window<TI, A, V, false, FIX>(fetch, p.R, p.S, acc);
        const A div = p.mode == 1 ? (A)(p.R * p.S) : (A)count;
        const long long yo = (long long)n * p.ys[0] + (long long)op * p.ys[2] + (long long)oq * p.ys[3] +
                             (long long)ch * V;
#pragma unroll
        for (int e = 0; e < V; ++e) {
            acc[e] = (A)p.alpha * (is_max ? acc[e] : acc[e] / div);
            if (p.beta != 0.0) acc[e] += (A)p.beta * (A)Io<TO>::ld(y, yo + e);
        }
        if (p.y_vec) {
            store_vec<TO, A, V>(y + yo, acc);
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e) Io<TO>::st(y, yo + e, acc[e]);
        }
    }
}

// Any layout: one output element per thread, outputs enumerated with the
// unit-stride axis of y innermost.
template <typename TI, typename TO, typename I>
__global__ void __launch_bounds__(256) pool_any_kernel(const __grid_constant__ PoolParams p,
                                                       int c_fastest) {
    using A = typename Io<TI>::acc;
    const TI *x = static_cast<const TI *>(p.x);
    TO *y = static_cast<TO *>(p.y);
    const I total = (I)((long long)p.N * p.C * p.P * p.Q);
    for (I idx = (I)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (I)gridDim.x * blockDim.x) {
        I t = idx;
        int n, c, op, oq;
        if (c_fastest) {
            c = (int)(t % p.C); t /= p.C;
            oq = (int)(t % p.Q); t /= p.Q;
            op = (int)(t % p.P);
            n = (int)(t / p.P);
        } else {
            oq = (int)(t % p.Q); t /= p.Q;
            op = (int)(t % p.P); t /= p.P;
            c = (int)(t % p.C);
            n = (int)(t / p.C);
        }
        const bool is_max = p.mode == 0;
        A acc = is_max ? (A)-INFINITY : (A)0;
        int count = 0;
        const TI *xc = x + (long long)n * p.xs[0] + (long long)c * p.xs[1];
        for (int i = 0; i < p.R; ++i) {
            const int h = op * p.u - p.pt + i;
            if (h < 0 || h >= p.H) continue;
            for (int j = 0; j < p.S; ++j) {
                const int wi = oq * p.v - p.pl + j;
                if (wi < 0 || wi >= p.W) continue;
                const A v = Io<TI>::ld(xc, (long long)h * p.xs[2] + (long long)wi * p.xs[3]);
                acc = is_max ? (v > acc ? v : acc) : acc + v;
                ++count;
            }
        }
        if (!is_max) acc /= p.mode == 1 ? (A)(p.R * p.S) : (A)count;
        const long long yo = (long long)n * p.ys[0] + (long long)c * p.ys[1] + (long long)op * p.ys[2] +
                             (long long)oq * p.ys[3];
        A val = (A)p.alpha * acc;
        if (p.beta != 0.0) val += (A)p.beta * (A)Io<TO>::ld(y, yo);
        Io<TO>::st(y, yo, val);
    }
}

struct ActParams {
    int N, C, H, W, mode;
    long long xs[4], ys[4];
    const void *x;
    void *y;
    double alpha, beta, coef;
};

__device__ __forceinline__ float exp_of(float v) { return expf(v); }
__device__ __forceinline__ double exp_of(double v) { return exp(v); }
__device__ __forceinline__ float tanh_of(float v) { return tanhf(v); }
__device__ __forceinline__ double tanh_of(double v) { return tanh(v); }

template <typename A>
__device__ __forceinline__ A act_fn(int mode, A v, A coef) {
    switch (mode) {
        case 1: return v > (A)0 ? v : (A)0;
        case 2: return (A)1 / ((A)1 + exp_of(-v));
        case 3: return tanh_of(v);
        case 4: return v < (A)0 ? (A)0 : (v > coef ? coef : v);
        default: return v;
    }
}

// Flat path: x and y dense with the same strides (elements 0 .. n-1 of both),
// one kernel per activation MODE.  Each thread loads four 16-byte vectors
// before it uses any.
template <typename TI, typename TO, int MODE>
__global__ void __launch_bounds__(256) act_flat_kernel(const __grid_constant__ ActParams p, long long n) {
    using A = typename Io<TI>::acc;
    constexpr int V = 16 / (int)sizeof(TI);
    constexpr int U = 4;
    const TI *x = static_cast<const TI *>(p.x);
    TO *y = static_cast<TO *>(p.y);
    const long long nv = n / V;
    const A alpha = (A)p.alpha, beta = (A)p.beta, coef = (A)p.coef;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += U * stride) {
        uint4 q[U];
#pragma unroll
        for (int h = 0; h < U; ++h) {
            const long long jv = i + h * stride;
            q[h] = jv < nv ? __ldg(reinterpret_cast<const uint4 *>(x) + jv) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int h = 0; h < U; ++h) {
            const long long jv = i + h * stride;
            if (jv >= nv) break;
            A v[V];
            unpack16<TI, A, V>(q[h], v);
#pragma unroll
            for (int e = 0; e < V; ++e) {
                v[e] = alpha * act_fn<A>(MODE, v[e], coef);
                if (beta != (A)0) v[e] += beta * (A)Io<TO>::ld(y, jv * V + e);
            }
            store_vec<TO, A, V>(y + jv * V, v);
        }
    }
    // the tail of fewer than V elements
    for (long long i = nv * V + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        A val = alpha * act_fn<A>(MODE, (A)Io<TI>::ld(x, i), coef);
        if (beta != (A)0) val += beta * (A)Io<TO>::ld(y, i);
        Io<TO>::st(y, i, val);
    }
}

template <typename TI, typename TO, typename I>
__global__ void __launch_bounds__(256) act_any_kernel(const __grid_constant__ ActParams p) {
    using A = typename Io<TI>::acc;
    const TI *x = static_cast<const TI *>(p.x);
    TO *y = static_cast<TO *>(p.y);
    const I total = (I)((long long)p.N * p.C * p.H * p.W);
    for (I idx = (I)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (I)gridDim.x * blockDim.x) {
        I t = idx;
        const int wi = (int)(t % p.W); t /= p.W;
        const int h = (int)(t % p.H); t /= p.H;
        const int c = (int)(t % p.C);
        const int n = (int)(t / p.C);
        const long long xo = (long long)n * p.xs[0] + (long long)c * p.xs[1] + (long long)h * p.xs[2] +
                             (long long)wi * p.xs[3];
        const long long yo = (long long)n * p.ys[0] + (long long)c * p.ys[1] + (long long)h * p.ys[2] +
                             (long long)wi * p.ys[3];
        A val = (A)p.alpha * act_fn<A>(p.mode, (A)Io<TI>::ld(x, xo), (A)p.coef);
        if (p.beta != 0.0) val += (A)p.beta * (A)Io<TO>::ld(y, yo);
        Io<TO>::st(y, yo, val);
    }
}

int grid_of(const dlcContext *ctx, long long work) {
    const long long blocks = (work + 255) / 256;
    const long long cap = (long long)ctx->sm_count * 8;
    return (int)std::max(1LL, std::min(blocks, cap));
}

template <typename TI, typename TO>
cudaError_t launch_pool(const dlcContext *ctx, const PoolParams &p, bool nhwc) {
    // 32-bit enumeration while the count and the grid-stride step stay below 2^31
    constexpr long long kSmall = 1LL << 30;
    if (nhwc) {
        const long long work = (long long)p.N * p.P * p.Q * (p.C / (16 / (int)sizeof(TI)));
        if (work < kSmall && p.R == 3 && p.S == 3)
            pool_nhwc_kernel<TI, TO, int, 3><<<grid_of(ctx, work), 256, 0, ctx->stream>>>(p);
        else if (work < kSmall)
            pool_nhwc_kernel<TI, TO, int, 0><<<grid_of(ctx, work), 256, 0, ctx->stream>>>(p);
        else
            pool_nhwc_kernel<TI, TO, long long, 0><<<grid_of(ctx, work), 256, 0, ctx->stream>>>(p);
    } else {
        const long long work = (long long)p.N * p.C * p.P * p.Q;
        if (work < kSmall)
            pool_any_kernel<TI, TO, int><<<grid_of(ctx, work), 256, 0, ctx->stream>>>(p, p.ys[1] == 1 ? 1 : 0);
        else
            pool_any_kernel<TI, TO, long long><<<grid_of(ctx, work), 256, 0, ctx->stream>>>(p, p.ys[1] == 1 ? 1 : 0);
    }
    return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t launch_act(const dlcContext *ctx, const ActParams &p, long long flat_n) {
    if (flat_n > 0) {
        const int grid = grid_of(ctx, flat_n / (16 / (long long)sizeof(TI)) + 1);
        switch (p.mode) {
            case 1: act_flat_kernel<TI, TO, 1><<<grid, 256, 0, ctx->stream>>>(p, flat_n); break;
            case 2: act_flat_kernel<TI, TO, 2><<<grid, 256, 0, ctx->stream>>>(p, flat_n); break;
            case 3: act_flat_kernel<TI, TO, 3><<<grid, 256, 0, ctx->stream>>>(p, flat_n); break;
            case 4: act_flat_kernel<TI, TO, 4><<<grid, 256, 0, ctx->stream>>>(p, flat_n); break;
            default: act_flat_kernel<TI, TO, 0><<<grid, 256, 0, ctx->stream>>>(p, flat_n); break;
        }
    } else {
        const long long work = (long long)p.N * p.C * p.H * p.W;
        if (work < (1LL << 30))
            act_any_kernel<TI, TO, int><<<grid_of(ctx, work), 256, 0, ctx->stream>>>(p);
        else
            act_any_kernel<TI, TO, long long><<<grid_of(ctx, work), 256, 0, ctx->stream>>>(p);
    }
    return cudaGetLastError();
}

template <template <typename, typename> class F, typename... Args>
cudaError_t by_types(dlcDataType_t ti, dlcDataType_t to, Args &&...args) {
    if (ti == DLC_DATA_DOUBLE && to == DLC_DATA_DOUBLE) return F<double, double>::run(args...);
    if (ti == DLC_DATA_FLOAT && to == DLC_DATA_FLOAT) return F<float, float>::run(args...);
    if (ti == DLC_DATA_FLOAT && to == DLC_DATA_BFLOAT16) return F<float, unsigned short>::run(args...);
    if (ti == DLC_DATA_BFLOAT16 && to == DLC_DATA_FLOAT) return F<unsigned short, float>::run(args...);
    if (ti == DLC_DATA_BFLOAT16 && to == DLC_DATA_BFLOAT16)
        return F<unsigned short, unsigned short>::run(args...);
    return cudaErrorInvalidValue;
}

template <typename TI, typename TO> struct PoolRun {
    static cudaError_t run(const dlcContext *ctx, const PoolParams &p, bool nhwc) {
        return launch_pool<TI, TO>(ctx, p, nhwc);
    }
};
template <typename TI, typename TO> struct ActRun {
    static cudaError_t run(const dlcContext *ctx, const ActParams &p, long long flat_n) {
        return launch_act<TI, TO>(ctx, p, flat_n);
    }
};

// True if the 4-D (extent, stride) pairs cover exactly the offsets 0 .. n-1.
bool dense(const int *ext, const int64_t *str) {
    int idx[4] = {0, 1, 2, 3};
    std::sort(idx, idx + 4, [&](int a, int b) { return str[a] < str[b]; });
    long long expect = 1;
    for (int i = 0; i < 4; ++i) {
        const int d = idx[i];
        if (ext[d] == 1) continue;
        if (str[d] != expect) return false;
        expect *= ext[d];
    }
    return true;
}

}  // namespace

dlcKernel_t dlc_pool_variant(const PoolProblem &pp) {
    const int e = dlc_dtype_bytes(pp.xdt);
    const bool nhwc = pp.xs[1] == 1 && pp.ys[1] == 1 && (pp.C * e) % 16 == 0 &&
                      (pp.xs[3] * e) % 16 == 0 && (pp.xs[2] * e) % 16 == 0 && (pp.xs[0] * e) % 16 == 0 &&
                      ((uintptr_t)pp.x % 16) == 0;
    return nhwc ? DLC_KERNEL_POOL_NHWC : DLC_KERNEL_DIRECT;
}

dlcStatus_t dlc_launch_pool(dlcContext *ctx, const PoolProblem &pp) {
    PoolParams p;
    std::memset(&p, 0, sizeof(p));
    p.N = pp.N; p.C = pp.C; p.H = pp.H; p.W = pp.W; p.R = pp.R; p.S = pp.S; p.P = pp.P; p.Q = pp.Q;
    p.pt = pp.pt; p.pl = pp.pl; p.u = pp.u; p.v = pp.v; p.mode = pp.mode;
    for (int i = 0; i < 4; ++i) {
        p.xs[i] = pp.xs[i];
        p.ys[i] = pp.ys[i];
    }
    p.x = pp.x; p.y = pp.y; p.alpha = pp.alpha; p.beta = pp.beta;
    const bool nhwc = dlc_pool_variant(pp) == DLC_KERNEL_POOL_NHWC;
    {
        // a chunk of 16 bytes of x channels is 16 / sizeof(x) * sizeof(y) bytes of y
        const int ex = dlc_dtype_bytes(pp.xdt), ey = dlc_dtype_bytes(pp.ydt);
        const long long vb = 16LL / ex * ey, al = std::min(vb, 16LL);
        p.y_vec = nhwc && ((uintptr_t)pp.y % al) == 0 && (pp.ys[0] * ey) % al == 0 &&
                  (pp.ys[2] * ey) % al == 0 && (pp.ys[3] * ey) % al == 0;
        p.raw_max = p.y_vec && pp.mode == 0 && pp.xdt == DLC_DATA_BFLOAT16 && pp.ydt == DLC_DATA_BFLOAT16 &&
                    pp.alpha == 1.0 && pp.beta == 0.0;
    }
    if (by_types<PoolRun>(pp.xdt, pp.ydt, ctx, p, nhwc) != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlc_launch_activation(dlcContext *ctx, const ActProblem &ap) {
    ActParams p;
    std::memset(&p, 0, sizeof(p));
    p.N = ap.N; p.C = ap.C; p.H = ap.H; p.W = ap.W; p.mode = ap.mode;
    for (int i = 0; i < 4; ++i) {
        p.xs[i] = ap.xs[i];
        p.ys[i] = ap.ys[i];
    }
    p.x = ap.x; p.y = ap.y; p.alpha = ap.alpha; p.beta = ap.beta; p.coef = ap.coef;
    const int ext[4] = {ap.N, ap.C, ap.H, ap.W};
    bool same = true;
    for (int i = 0; i < 4; ++i) same = same && ap.xs[i] == ap.ys[i];
    const long long n = (long long)ap.N * ap.C * ap.H * ap.W;
    const long long vb = 16LL / dlc_dtype_bytes(ap.xdt) * dlc_dtype_bytes(ap.ydt);
    const long long flat = (same && dense(ext, ap.xs) && ((uintptr_t)ap.x % 16) == 0 &&
                            ((uintptr_t)ap.y % std::min(vb, 16LL)) == 0) ? n : 0;
    if (by_types<ActRun>(ap.xdt, ap.ydt, ctx, p, flat) != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}
