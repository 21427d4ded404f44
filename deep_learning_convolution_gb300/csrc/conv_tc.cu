// conv_tc.cu -- forward convolution as an implicit batch-reduce GEMM on the
// sm_103a tensor cores (tcgen05), FP32 accumulation in tensor memory.
//
// GEMM view (maxDNN page, method section: an output coordinate is the product
// of its receptive field with the filters): rows M = N*P*Q output pixels,
// columns = K filters, reduction = C*R*S.  The reduction is a batch-reduce
// GEMM (batch-reduce GEMM page, method section): acc[128 x BN] += sum_i A_i *
// B_i^T with i over the filter taps (r,s) and channel blocks, so the im2col
// matrix is never stored (zero-memory-overhead page; cuDNN page, method
// section: no auxiliary buffers).
//
// Roles inside one persistent CTA (one CTA per SM, static tile schedule):
//  * producer -- TMA variant: one thread issues, per (tile, r, s, c-block), an
//    im2col-mode TMA load of 128 pixels x 128 bytes of channels (padding comes
//    from the tensor map's bounding box: out-of-image pixels read as zero) and
//    a tiled TMA load of BN filters x 128 bytes of channels at tap (r,s).
//    Gather variant: four warps (one thread per A row) read x and w with
//    ordinary loads in any layout and write the same swizzled tiles; used for
//    NCHW, channel counts below one 128-byte row (C=1, C=3 first layers),
//    KCRS filters under NHWC, or unaligned views.
//  * MMA issuer -- one thread issues tcgen05.mma (M=128, N=BN, K=32 bytes per
//    instruction) into one of two TMEM accumulators and commits each smem
//    stage back to the producer (double-buffered global->shared staging,
//    maxDNN page, method section).
//  * epilogue -- four warps read the accumulator with tcgen05.ld (one output
//    row per thread), apply alpha, beta*y, bias and ReLU, and store y while
//    the MMA issuer already fills the other accumulator.
//
// Every wait is bounded (ptx.cuh: mbar_wait); a wait that runs out records
// an error word and the CTA unwinds: copies in flight are drained, MMAs are
// committed and waited for, tensor memory is released.
#include <cuda_bf16.h>

#include <cstring>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace {

using namespace dlc;

constexpr int BM = 128;                        // rows (output pixels) per tile
constexpr int ROW_BYTES = 128;                 // one 128-byte swizzle row of the reduction
constexpr int A_STAGE_BYTES = BM * ROW_BYTES;  // 16 KiB
constexpr int MAX_DYN_SMEM = 232448;           // 227 KiB per block (opt-in)
constexpr int BAR_AREA = 256;

struct TcParams {
    int N, C, H, W, K, R, S, P, Q;
    int pt, pl, u, v, dh, dw;
    long long M;  // N*P*Q
    int PQ;
    long long xs[4], ws[4], ys[4];
    const void *x;
    const void *w;
    void *y;
    const float *bias;
    float alpha, beta;
    int relu, y_bf16;
    int BN, stages, num_kb, c_blocks;
    int n_tiles;
    long long num_tiles;
    uint32_t idesc, tmem_cols, acc_stride;  // acc_stride: TMEM column offset of accumulator 1
    int *err;
    unsigned long long timeout_ns;
};

// Drain wait: ignores the abort flag, bounded by the same time limit.
__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity, const TcParams &p) {
    volatile int dummy = 0;
    WaitCtl c{&dummy, p.err, p.timeout_ns};
    return mbar_wait(bar, parity, c, 90);
}

struct TileCoord {
    long long m0;
    int k0;
};

__device__ __forceinline__ TileCoord tile_coord(const TcParams &p, long long tile) {
    TileCoord tc;
    tc.m0 = (tile / p.n_tiles) * BM;
    tc.k0 = (int)(tile % p.n_tiles) * p.BN;
    return tc;
}

// ---------------------------------------------------------------------------
// producer, TMA variant (one thread)
// ---------------------------------------------------------------------------
template <int BK>
__device__ void produce_tma(const TcParams &p, const CUtensorMap *tmA, const CUtensorMap *tmB,
                            uint8_t *smA, uint8_t *smB, uint64_t *full, uint64_t *empty,
                            const WaitCtl &ctl) {
    const int ST = p.stages;
    const uint32_t b_stage = (uint32_t)p.BN * ROW_BYTES;
    const uint32_t tx = A_STAGE_BYTES + b_stage;
    int it = 0;
    bool ok = true;
    for (long long tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const TileCoord tc = tile_coord(p, tile);
        const int n0 = (int)(tc.m0 / p.PQ);
        const int rem = (int)(tc.m0 - (long long)n0 * p.PQ);
        const int p0 = rem / p.Q, q0 = rem - (rem / p.Q) * p.Q;
        const int wc = q0 * p.v - p.pl;  // first window origin of the tile
        const int hc = p0 * p.u - p.pt;
        for (int r = 0; ok && r < p.R; ++r) {
            for (int s = 0; ok && s < p.S; ++s) {
                for (int cb = 0; cb < p.c_blocks; ++cb) {
                    const int stage = it % ST;
                    const uint32_t ph = (uint32_t)(it / ST) & 1u;
                    if (!mbar_wait(&empty[stage], ph ^ 1u, ctl, 1)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], tx);
                    tma_load_im2col_4d(smA + (size_t)stage * A_STAGE_BYTES, tmA, &full[stage],
                                       cb * BK, wc, hc, n0, (uint16_t)(s * p.dw),
                                       (uint16_t)(r * p.dh));
                    tma_load_4d(smB + (size_t)stage * b_stage, tmB, &full[stage], cb * BK, s, r,
                                tc.k0);
                    ++it;
                }
            }
        }
    }
    // Copies still in flight must land before the CTA may exit.
    for (int j = (it > ST ? it - ST : 0); j < it; ++j)
        drain_wait(&full[j % ST], (uint32_t)(j / ST) & 1u, p);
}

// ---------------------------------------------------------------------------
// producer, gather variant (128 threads, thread t writes A row t)
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ uint32_t pack2(T lo, T hi);
template <>
__device__ __forceinline__ uint32_t pack2<uint16_t>(uint16_t lo, uint16_t hi) {
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Walks the flattened reduction index kk = (r*S + s)*C + c of one operand row.
struct RscWalker {
    int r, s, c;
    __device__ __forceinline__ void start(int kk0, int C, int S) {
        c = kk0 % C;
        const int rs = kk0 / C;
        s = rs % S;
        r = rs / S;
    }
    __device__ __forceinline__ void step(int C, int S) {
        if (++c == C) {
            c = 0;
            if (++s == S) {
                s = 0;
                ++r;
            }
        }
    }
};

template <typename T>
__device__ __forceinline__ void store_row_chunk(uint8_t *row, int row_idx, int chunk,
                                                const uint32_t (&w4)[4]) {
    uint8_t *dst = row + ((chunk ^ (row_idx & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(dst)), "r"(w4[0]),
                 "r"(w4[1]), "r"(w4[2]), "r"(w4[3])
                 : "memory");
}

template <typename T>
__device__ void produce_gather(const TcParams &p, uint8_t *smA, uint8_t *smB, uint64_t *full,
                               uint64_t *empty, const WaitCtl &ctl) {
    constexpr int BK = ROW_BYTES / (int)sizeof(T);
    constexpr int PER_WORD = 4 / (int)sizeof(T);
    const int t = threadIdx.x;  // 0..127
    const int ST = p.stages;
    const uint32_t b_stage = (uint32_t)p.BN * ROW_BYTES;
    const T *x = static_cast<const T *>(p.x);
    const T *w = static_cast<const T *>(p.w);
    int it = 0;
    bool ok = true;
    for (long long tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const TileCoord tc = tile_coord(p, tile);
        const long long m = tc.m0 + t;
        const bool valid = m < p.M;
        int n = 0, op = 0, oq = 0;
        if (valid) {
            n = (int)(m / p.PQ);
            const int rem = (int)(m - (long long)n * p.PQ);
            op = rem / p.Q;
            oq = rem - op * p.Q;
        }
        const int h0 = op * p.u - p.pt, w0 = oq * p.v - p.pl;
        const T *xn = x + (long long)n * p.xs[0];
        for (int kb = 0; kb < p.num_kb; ++kb) {
            const int stage = it % ST;
            const uint32_t ph = (uint32_t)(it / ST) & 1u;
            if (!mbar_wait(&empty[stage], ph ^ 1u, ctl, 6)) {
                ok = false;
                break;
            }
            const int kk0 = kb * BK;
            // A row t
            {
                uint8_t *row = smA + (size_t)stage * A_STAGE_BYTES + t * ROW_BYTES;
                RscWalker wk;
                wk.start(kk0, p.C, p.S);
#pragma unroll 1
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t w4[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        T e[PER_WORD];
#pragma unroll
                        for (int j = 0; j < PER_WORD; ++j) {
                            T val = 0;
                            if (valid && wk.r < p.R) {
                                const int h = h0 + wk.r * p.dh, wi = w0 + wk.s * p.dw;
                                if (h >= 0 && h < p.H && wi >= 0 && wi < p.W)
                                    val = xn[wk.c * p.xs[1] + h * p.xs[2] + wi * p.xs[3]];
                            }
                            e[j] = val;
                            wk.step(p.C, p.S);
                        }
                        if constexpr (PER_WORD == 2) w4[q] = pack2<T>(e[0], e[1]);
                        else w4[q] = (uint32_t)e[0];
                    }
                    store_row_chunk<T>(row, t, ch, w4);
                }
            }
            // B rows t, t+128 (filters k0 + row)
            for (int br = t; br < p.BN; br += BM) {
                uint8_t *row = smB + (size_t)stage * b_stage + br * ROW_BYTES;
                const int k = tc.k0 + br;
                const bool kval = k < p.K;
                const T *wk_ptr = w + (long long)(kval ? k : 0) * p.ws[0];
                RscWalker wk;
                wk.start(kk0, p.C, p.S);
#pragma unroll 1
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t w4[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        T e[PER_WORD];
#pragma unroll
                        for (int j = 0; j < PER_WORD; ++j) {
                            T val = 0;
                            if (kval && wk.r < p.R)
                                val = wk_ptr[wk.c * p.ws[1] + wk.r * p.ws[2] + wk.s * p.ws[3]];
                            e[j] = val;
                            wk.step(p.C, p.S);
                        }
                        if constexpr (PER_WORD == 2) w4[q] = pack2<T>(e[0], e[1]);
                        else w4[q] = (uint32_t)e[0];
                    }
                    store_row_chunk<T>(row, br, ch, w4);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&full[stage]);
            ++it;
        }
    }
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread)
// ---------------------------------------------------------------------------
template <bool TF32>
__device__ void issue_mma(const TcParams &p, uint32_t tmem_base, uint8_t *smA, uint8_t *smB,
                          uint64_t *full, uint64_t *empty, uint64_t *tfull, uint64_t *tempty,
                          uint64_t *mma_done, const WaitCtl &ctl) {
    const int ST = p.stages;
    const uint32_t b_stage = (uint32_t)p.BN * ROW_BYTES;
    const uint32_t a0 = smem_u32(smA), b0 = smem_u32(smB);
    int it = 0, t = 0;
    bool ok = true;
    for (long long tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const int buf = t & 1;
        const uint32_t aph = (uint32_t)(t >> 1) & 1u;
        if (!mbar_wait(&tempty[buf], aph ^ 1u, ctl, 3)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)buf * p.acc_stride;
        for (int kb = 0; kb < p.num_kb; ++kb) {
            const int stage = it % ST;
            const uint32_t ph = (uint32_t)(it / ST) & 1u;
            if (!mbar_wait(&full[stage], ph, ctl, 4)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t a_addr = a0 + (uint32_t)stage * A_STAGE_BYTES;
            const uint32_t b_addr = b0 + (uint32_t)stage * b_stage;
#pragma unroll
            for (int k = 0; k < ROW_BYTES / 32; ++k) {
                const uint64_t ad = sw128_kmajor_desc(a_addr + k * 32);
                const uint64_t bd = sw128_kmajor_desc(b_addr + k * 32);
                const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
                if constexpr (TF32) umma_tf32(d_tmem, ad, bd, p.idesc, acc);
                else umma_bf16(d_tmem, ad, bd, p.idesc, acc);
            }
            umma_commit(&empty[stage]);  // stage free once these MMAs are done
            ++it;
        }
        if (!ok) break;
        umma_commit(&tfull[buf]);        // accumulator ready for the epilogue
        ++t;
    }
    // Every MMA issued must complete before tensor memory is released.
    umma_commit(mma_done);
    drain_wait(mma_done, 0, p);
}

// ---------------------------------------------------------------------------
// epilogue (4 warps, one output row per thread)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(unsigned short b) {
    return __uint_as_float((uint32_t)b << 16);
}

__device__ __forceinline__ unsigned short f32_to_bf16_bits(float f) {
    __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<unsigned short *>(&b);
}

__device__ void epilogue(const TcParams &p, uint32_t tmem_base, uint64_t *tfull, uint64_t *tempty,
                         const WaitCtl &ctl) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    const int row = quad * 32 + lane;
    float *yf = static_cast<float *>(p.y);
    unsigned short *yb = static_cast<unsigned short *>(p.y);
    int t = 0;
    for (long long tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
        const int buf = t & 1;
        const uint32_t aph = (uint32_t)(t >> 1) & 1u;
        int okw = 0;
        if (lane == 0) okw = mbar_wait(&tfull[buf], aph, ctl, 5) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) break;
        __syncwarp();
        tc_fence_after_sync();
        const TileCoord tc = tile_coord(p, tile);
        const long long m = tc.m0 + row;
        const bool valid = m < p.M;
        long long ybase = 0;
        if (valid) {
            const int n = (int)(m / p.PQ);
            const int rem = (int)(m - (long long)n * p.PQ);
            const int op = rem / p.Q, oq = rem - (rem / p.Q) * p.Q;
            ybase = (long long)n * p.ys[0] + (long long)op * p.ys[2] + (long long)oq * p.ys[3];
        }
        const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)buf * p.acc_stride;
        for (int c0 = 0; c0 < p.BN; c0 += 16) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(taddr + (uint32_t)c0, v);
            tmem_ld_wait();
            if (!valid) continue;
            const int kbase = tc.k0 + c0;
            const bool full16 = kbase + 16 <= p.K;
            const long long yo0 = ybase + (long long)kbase * p.ys[1];
            float val[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) val[j] = p.alpha * __uint_as_float(v[j]);
            if (p.ys[1] == 1 && !p.y_bf16 && full16 &&
                ((reinterpret_cast<uintptr_t>(yf + yo0) & 15u) == 0)) {
                float4 *dst = reinterpret_cast<float4 *>(yf + yo0);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if (p.beta != 0.f) val[j] = __fmaf_rn(p.beta, yf[yo0 + j], val[j]);
                    if (p.bias) val[j] += __ldg(p.bias + kbase + j);
                    if (p.relu) val[j] = fmaxf(val[j], 0.f);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    dst[j] = make_float4(val[4 * j], val[4 * j + 1], val[4 * j + 2], val[4 * j + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int k = kbase + j;
                    if (k < p.K) {
                        const long long yo = ybase + (long long)k * p.ys[1];
                        float f = val[j];
                        if (p.beta != 0.f)
                            f = __fmaf_rn(p.beta, p.y_bf16 ? bf16_bits_to_f32(yb[yo]) : yf[yo], f);
                        if (p.bias) f += __ldg(p.bias + k);
                        if (p.relu) f = fmaxf(f, 0.f);
                        if (p.y_bf16) yb[yo] = f32_to_bf16_bits(f);
                        else yf[yo] = f;
                    }
                }
            }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        ++t;
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <bool TF32, bool GATHER>
__global__ void __launch_bounds__(GATHER ? 288 : 192, 1)
    conv_fprop_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB) {
    using T = typename std::conditional<TF32, uint32_t, uint16_t>::type;
    constexpr int BK = ROW_BYTES / (int)sizeof(T);
    constexpr int PROD_WARPS = GATHER ? 4 : 1;
    constexpr int MMA_WARP = PROD_WARPS;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int ST = p.stages;
    uint8_t *smA = smem;
    uint8_t *smB = smem + (size_t)ST * A_STAGE_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smB + (size_t)ST * p.BN * ROW_BYTES);
    uint64_t *full = bars;
    uint64_t *empty = bars + ST;
    uint64_t *tfull = bars + 2 * ST;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full[i], GATHER ? 128u : 1u);
            mbar_init(&empty[i], 1u);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1u);
            mbar_init(&tempty[i], 4u);  // one arrival per epilogue warp
        }
        mbar_init(mma_done, 1u);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (!GATHER && warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == MMA_WARP) {
        tmem_alloc(tmem_slot, p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtl ctl{abort_flag, p.err, p.timeout_ns};

    if (warp < PROD_WARPS) {
        if constexpr (GATHER) produce_gather<T>(p, smA, smB, full, empty, ctl);
        else if (lane == 0) produce_tma<BK>(p, &tmA, &tmB, smA, smB, full, empty, ctl);
    } else if (warp == MMA_WARP) {
        if (lane == 0) issue_mma<TF32>(p, tmem_base, smA, smB, full, empty, tfull, tempty, mma_done, ctl);
    } else {
        epilogue(p, tmem_base, tfull, tempty, ctl);
    }
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == MMA_WARP) tmem_dealloc(tmem_base, p.tmem_cols);
}

__global__ void wait_selftest_kernel(int *err, unsigned long long timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1u);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtl ctl{&abort_flag, err, timeout_ns};
    if (threadIdx.x == 0) mbar_wait(&bar, 0u, ctl, 99);  // nothing ever arrives
}

// ---------------------------------------------------------------------------
// host side: variant choice, tile shape, tensor maps, launch
// ---------------------------------------------------------------------------
int elt_bytes(const ConvProblem &pb) { return pb.xdt == DLC_DATA_BFLOAT16 ? 2 : 4; }

bool tc_math_ok(const ConvProblem &pb) {
    return (pb.math == DLC_MATH_BF16 && pb.xdt == DLC_DATA_BFLOAT16) ||
           (pb.math == DLC_MATH_TF32 && pb.xdt == DLC_DATA_FLOAT);
}

bool fits_i32(long long v) { return v >= 0 && v <= 0x7fffffffLL; }

// Conditions for the im2col TMA producer (CUDA driver API limits of
// cuTensorMapEncodeIm2col for a rank-4 tensor; the PTX im2col offsets are
// 16-bit values, kept here within 8 bits like the corners).
bool im2col_ok(const ConvProblem &pb) {
    const long long e = elt_bytes(pb);
    const int BK = ROW_BYTES / (int)e;
    if (pb.xs[1] != 1) return false;                       // channels innermost
    if (pb.wfmt != DLC_TENSOR_NHWC) return false;          // KRSC filters
    if (pb.C < BK || (pb.C * e) % 16) return false;
    if (pb.xs[3] < pb.C || pb.xs[2] < pb.xs[3] * (long long)pb.W ||
        pb.xs[0] < pb.xs[2] * (long long)pb.H)
        return false;                                      // NHWC-ordered (possibly padded) view
    for (int i : {0, 2, 3})
        if ((pb.xs[i] * e) % 16 || pb.xs[i] * e >= (1LL << 40)) return false;
    if (pb.x && ((uintptr_t)pb.x % 16)) return false;
    if (pb.w && ((uintptr_t)pb.w % 16)) return false;
    if (pb.u > 8 || pb.v > 8) return false;
    const long long lo_w = -pb.pl, lo_h = -pb.pt;
    const long long up_w = pb.pr - (long long)pb.dw * (pb.S - 1);
    const long long up_h = pb.pb - (long long)pb.dh * (pb.R - 1);
    for (long long c : {lo_w, lo_h, up_w, up_h})
        if (c < -128 || c > 127) return false;
    if ((long long)pb.dw * (pb.S - 1) > 255 || (long long)pb.dh * (pb.R - 1) > 255) return false;
    if (!fits_i32(pb.N) || !fits_i32(pb.H) || !fits_i32(pb.W)) return false;
    return true;
}

int choose_bn(int K) {
    if (K <= 256) return ((K + 15) / 16) * 16;
    int best = 256;
    long long best_pad = -1;
    for (int bn : {256, 192, 128}) {
        long long pad = (long long)((K + bn - 1) / bn) * bn;
        if (best_pad < 0 || pad < best_pad) {
            best_pad = pad;
            best = bn;
        }
    }
    return best;
}

template <bool TF32, bool GATHER>
cudaError_t launch_kernel(const TcParams &tp, const CUtensorMap &a, const CUtensorMap &b, int grid,
                          size_t smem, cudaStream_t st) {
    auto kern = conv_fprop_tc_kernel<TF32, GATHER>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, GATHER ? 288 : 192, smem, st>>>(tp, a, b);
    return cudaGetLastError();
}

}  // namespace

dlcKernel_t dlc_tc_variant(const dlcContext *, const ConvProblem &pb) {
    if (!tc_math_ok(pb)) return DLC_KERNEL_NONE;
    if (!fits_i32((long long)pb.P * pb.Q)) return DLC_KERNEL_NONE;
    return im2col_ok(pb) ? DLC_KERNEL_TC_IM2COL : DLC_KERNEL_TC_GATHER;
}

dlcStatus_t dlc_launch_tc(dlcContext *ctx, const ConvProblem &pb, dlcKernel_t variant) {
    if (variant != DLC_KERNEL_TC_IM2COL && variant != DLC_KERNEL_TC_GATHER)
        return DLC_STATUS_INTERNAL_ERROR;
    const bool tf32 = pb.math == DLC_MATH_TF32;
    const bool gather = variant == DLC_KERNEL_TC_GATHER;
    const int e = elt_bytes(pb);
    const int BK = ROW_BYTES / e;

    TcParams tp;
    tp.N = pb.N; tp.C = pb.C; tp.H = pb.H; tp.W = pb.W; tp.K = pb.K; tp.R = pb.R; tp.S = pb.S;
    tp.P = pb.P; tp.Q = pb.Q;
    tp.pt = pb.pt; tp.pl = pb.pl; tp.u = pb.u; tp.v = pb.v; tp.dh = pb.dh; tp.dw = pb.dw;
    tp.M = (long long)pb.N * pb.P * pb.Q;
    tp.PQ = pb.P * pb.Q;
    for (int i = 0; i < 4; ++i) {
        tp.xs[i] = pb.xs[i];
        tp.ws[i] = pb.ws[i];
        tp.ys[i] = pb.ys[i];
    }
    tp.x = pb.x; tp.w = pb.w; tp.y = pb.y; tp.bias = pb.bias;
    tp.alpha = pb.alpha; tp.beta = pb.beta; tp.relu = pb.relu;
    tp.y_bf16 = pb.ydt == DLC_DATA_BFLOAT16;
    tp.BN = choose_bn(pb.K);
    const int b_stage = tp.BN * ROW_BYTES;
    int stages = (MAX_DYN_SMEM - 1024 - BAR_AREA) / (A_STAGE_BYTES + b_stage);
    tp.stages = stages > 8 ? 8 : stages;
    tp.c_blocks = (pb.C + BK - 1) / BK;
    if (gather) {
        const long long kg = (long long)pb.R * pb.S * pb.C;
        if (kg > 0x7fffffffLL - BK) return DLC_STATUS_NOT_SUPPORTED;
        tp.num_kb = (int)((kg + BK - 1) / BK);
    } else {
        tp.num_kb = pb.R * pb.S * tp.c_blocks;
    }
    tp.n_tiles = (pb.K + tp.BN - 1) / tp.BN;
    const long long m_tiles = (tp.M + BM - 1) / BM;
    tp.num_tiles = m_tiles * tp.n_tiles;
    const uint32_t fmt = tf32 ? 2u : 1u;  // operand format: BF16 = 1, TF32 = 2
    tp.idesc = (1u << 4)                  // FP32 accumulator
               | (fmt << 7) | (fmt << 10)  // A and B formats
               | ((uint32_t)(tp.BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * tp.BN)) cols <<= 1;
    tp.tmem_cols = cols;
    tp.acc_stride = cols / 2;
    tp.err = ctx->d_err;
    tp.timeout_ns = ctx->timeout_ns;

    CUtensorMap ta, tb;
    std::memset(&ta, 0, sizeof(ta));
    std::memset(&tb, 0, sizeof(tb));
    if (!gather) {
        const CUtensorMapDataType dt =
            tf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const cuuint64_t gdim[4] = {(cuuint64_t)pb.C, (cuuint64_t)pb.W, (cuuint64_t)pb.H,
                                    (cuuint64_t)pb.N};
        const cuuint64_t gstr[3] = {(cuuint64_t)(pb.xs[3] * e), (cuuint64_t)(pb.xs[2] * e),
                                    (cuuint64_t)(pb.xs[0] * e)};
        const int lower[2] = {-pb.pl, -pb.pt};  // W, H
        const int upper[2] = {pb.pr - pb.dw * (pb.S - 1), pb.pb - pb.dh * (pb.R - 1)};
        const cuuint32_t estr[4] = {1, (cuuint32_t)pb.v, (cuuint32_t)pb.u, 1};
        CUresult r = ctx->encode_im2col(&ta, dt, 4, const_cast<void *>(pb.x), gdim, gstr, lower,
                                        upper, (cuuint32_t)BK, (cuuint32_t)BM, estr,
                                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return DLC_STATUS_EXECUTION_FAILED;
        const cuuint64_t wdim[4] = {(cuuint64_t)pb.C, (cuuint64_t)pb.S, (cuuint64_t)pb.R,
                                    (cuuint64_t)pb.K};
        const cuuint64_t wstr[3] = {(cuuint64_t)(pb.ws[3] * e), (cuuint64_t)(pb.ws[2] * e),
                                    (cuuint64_t)(pb.ws[0] * e)};
        const cuuint32_t box[4] = {(cuuint32_t)BK, 1, 1, (cuuint32_t)tp.BN};
        const cuuint32_t ones[4] = {1, 1, 1, 1};
        r = ctx->encode_tiled(&tb, dt, 4, const_cast<void *>(pb.w), wdim, wstr, box, ones,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return DLC_STATUS_EXECUTION_FAILED;
    }

    const size_t smem = 1024 + (size_t)tp.stages * (A_STAGE_BYTES + b_stage) + BAR_AREA;
    long long grid = tp.num_tiles < ctx->sm_count ? tp.num_tiles : ctx->sm_count;
    if (grid < 1) grid = 1;
    cudaError_t err;
    if (tf32) {
        err = gather ? launch_kernel<true, true>(tp, ta, tb, (int)grid, smem, ctx->stream)
                     : launch_kernel<true, false>(tp, ta, tb, (int)grid, smem, ctx->stream);
    } else {
        err = gather ? launch_kernel<false, true>(tp, ta, tb, (int)grid, smem, ctx->stream)
                     : launch_kernel<false, false>(tp, ta, tb, (int)grid, smem, ctx->stream);
    }
    if (err != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlc_launch_wait_selftest(dlcContext *ctx, unsigned long long timeout_ns) {
    wait_selftest_kernel<<<1, 32, 0, ctx->stream>>>(ctx->d_err, timeout_ns);
    if (cudaGetLastError() != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}
