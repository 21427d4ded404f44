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

#include <algorithm>
#include <cstdlib>
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
constexpr int EPI_BUF_BYTES = 32 * 128;            // one warp's 32 rows x 32 FP32 columns
constexpr int EPI_SMEM = 4 * 2 * EPI_BUF_BYTES;     // 4 epilogue warps, double-buffered

enum { MODE_IM2COL = 0, MODE_GATHER = 1, MODE_RUNS = 2 };
constexpr int GATHER_GROUPS = 2;

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
    int y_tma;                      // epilogue stores y through the 2-D tensor map tmY
    int BN, stages, num_kb, c_blocks;
    int n_tiles;
    int b_res;                      // gather modes: all num_kb filter blocks resident in smem
    int run_len, num_runs, cpr;     // run gather: elements per run, runs, 16-byte chunks per run
    int img_tiles;                  // > 0: image-aligned M tiles, this many per image
    int halo;                       // run gather stages each tile's input rows in shared memory
    int halo_bytes;                 // bytes of one halo buffer (two are used)
    int ctab;                       // run gather: per-(k-block, chunk) table in shared memory
    int epc;                        // elements per 16-byte chunk
    int nchw_runs;                  // runs over s of one (c, r) (else over (s, c) of one r)
    long long num_tiles;
    uint32_t idesc, tmem_cols, acc_stride;  // acc_stride: TMEM column offset of accumulator 1
    int sk;                         // stream-K schedule over (tile, k-block) units
    long long sk_units;             // units per CTA (>= num_kb, so a tile has <= 2 parts)
    int *sk_flags;                  // per-tile partial-ready flags (zero between launches)
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
    long long m0;  // first output pixel (flattened n, p, q)
    int k0;        // first filter
    int rows;      // valid rows of the tile (<= BM)
};

// M tiles run over the flattened (n, p, q) pixels, or -- when img_tiles > 0 --
// image by image (img_tiles tiles per image, the last one ragged), so that a
// tile never spans two images.
__device__ __forceinline__ TileCoord tile_coord(const TcParams &p, long long tile) {
    TileCoord tc;
    const long long mt = tile / p.n_tiles;
    tc.k0 = (int)(tile % p.n_tiles) * p.BN;
    if (p.img_tiles > 0) {
        const long long n = mt / p.img_tiles;
        const int t = (int)(mt - n * p.img_tiles);
        tc.m0 = n * p.PQ + (long long)t * BM;
        tc.rows = min(BM, p.PQ - t * BM);
    } else {
        tc.m0 = mt * BM;
        const long long left = p.M - tc.m0;
        tc.rows = left < BM ? (int)left : BM;
    }
    return tc;
}

// One piece of work: k-blocks [kb0, kb1) of one output tile.
struct Seg {
    long long tile;
    int kb0, kb1;
};

// The CTA's sequence of segments.  Data-parallel: whole tiles blockIdx.x,
// blockIdx.x + gridDim.x, ...  Stream-K: the contiguous range of sk_units
// (tile, k-block) units starting at blockIdx.x * sk_units; it may begin with
// the last k-blocks of one tile and end with the first k-blocks of another.
struct WorkIter {
    long long u, u_end;
    __device__ __forceinline__ explicit WorkIter(const TcParams &p) {
        if (p.sk) {
            const long long total = p.num_tiles * p.num_kb;
            u = (long long)blockIdx.x * p.sk_units;
            u_end = u + p.sk_units < total ? u + p.sk_units : total;
        } else {
            u = blockIdx.x;
            u_end = p.num_tiles;
        }
    }
    __device__ __forceinline__ bool next(const TcParams &p, Seg &sg) {
        if (u >= u_end) return false;
        if (p.sk) {
            sg.tile = u / p.num_kb;
            sg.kb0 = (int)(u - sg.tile * p.num_kb);
            const long long left = u_end - u;
            sg.kb1 = (long long)(p.num_kb - sg.kb0) <= left ? p.num_kb : sg.kb0 + (int)left;
            u += sg.kb1 - sg.kb0;
        } else {
            sg.tile = u;
            sg.kb0 = 0;
            sg.kb1 = p.num_kb;
            u += gridDim.x;
        }
        return true;
    }
};

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
    int it = 0, stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    WorkIter wi(p);
    Seg sg;
    while (ok && wi.next(p, sg)) {
        const TileCoord tc = tile_coord(p, sg.tile);
        const int n0 = (int)(tc.m0 / p.PQ);
        const int rem = (int)(tc.m0 - (long long)n0 * p.PQ);
        const int p0 = rem / p.Q, q0 = rem - (rem / p.Q) * p.Q;
        const int wc = q0 * p.v - p.pl;  // first window origin of the tile
        const int hc = p0 * p.u - p.pt;
        // k-block kb = (r*S + s)*c_blocks + cb
        int cb = sg.kb0 % p.c_blocks;
        const int rs = sg.kb0 / p.c_blocks;
        int s = rs % p.S, r = rs / p.S;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
            if (!mbar_wait(&empty[stage], ph ^ 1u, ctl, 1)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(&full[stage], tx);
            tma_load_im2col_4d(smA + (size_t)stage * A_STAGE_BYTES, tmA, &full[stage], cb * BK, wc,
                               hc, n0, (uint16_t)(s * p.dw), (uint16_t)(r * p.dh));
            tma_load_4d(smB + (size_t)stage * b_stage, tmB, &full[stage], cb * BK, s, r, tc.k0);
            ++it;
            if (++stage == ST) {
                stage = 0;
                ph ^= 1u;
            }
            if (++cb == p.c_blocks) {
                cb = 0;
                if (++s == p.S) {
                    s = 0;
                    ++r;
                }
            }
        }
    }
    // Copies still in flight must land before the CTA may exit.
    for (int j = (it > ST ? it - ST : 0); j < it; ++j)
        drain_wait(&full[j % ST], (uint32_t)(j / ST) & 1u, p);
}

// ---------------------------------------------------------------------------
// producers, gather variants (GROUPS x 128 threads; thread t of a group
// writes A row t of the stages its group owns: stage iteration it belongs to
// group it % GROUPS, so GROUPS stages are filled concurrently)
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ uint32_t pack2(T lo, T hi);
template <>
__device__ __forceinline__ uint32_t pack2<uint16_t>(uint16_t lo, uint16_t hi) {
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ void store_chunk(uint8_t *row, int row_idx, int chunk, uint32_t a0,
                                            uint32_t a1, uint32_t a2, uint32_t a3) {
    uint8_t *dst = row + ((chunk ^ (row_idx & 7)) << 4);  // 128-byte swizzle
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(dst)), "r"(a0),
                 "r"(a1), "r"(a2), "r"(a3)
                 : "memory");
}

// Element-gather reduction order: kk = (r*S + s)*C + c, any strides.
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

// One 16-byte chunk (BK/8 elements) of an element-gather operand row.
template <typename T, bool IS_A>
__device__ __forceinline__ void gather_elem_chunk(const TcParams &p, const T *base, bool ok, int h0,
                                                  int w0, int kk0, uint32_t (&o)[4]) {
    constexpr int PER_WORD = 4 / (int)sizeof(T);
    RscWalker wk;
    wk.start(kk0, p.C, p.S);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        T e[PER_WORD];
#pragma unroll
        for (int j = 0; j < PER_WORD; ++j) {
            T val = 0;
            if (ok && wk.r < p.R) {
                if constexpr (IS_A) {
                    const int h = h0 + wk.r * p.dh, wi = w0 + wk.s * p.dw;
                    if (h >= 0 && h < p.H && wi >= 0 && wi < p.W)
                        val = base[wk.c * p.xs[1] + h * p.xs[2] + wi * p.xs[3]];
                } else {
                    val = base[wk.c * p.ws[1] + wk.r * p.ws[2] + wk.s * p.ws[3]];
                }
            }
            e[j] = val;
            wk.step(p.C, p.S);
        }
        if constexpr (PER_WORD == 2) o[q] = pack2<T>(e[0], e[1]);
        else o[q] = (uint32_t)e[0];
    }
}

// Run-gather reduction layout.  A run is a sequence of elements that are
// contiguous in memory -- the (s, c) elements of one filter row r for
// channels-innermost activations with KRSC filters, the s elements of one
// (c, r) pair for width-innermost activations with KCRS filters.  Runs are
// padded to whole 16-byte chunks (cpr chunks each) and packed one after the
// other along the reduction; run index = r, or c*R + r.
struct RunPos {
    int run, cr, c, r;  // run index, chunk within run, and the run's (c, r)
    __device__ __forceinline__ void start(const TcParams &p, int g) {
        run = g / p.cpr;
        cr = g - run * p.cpr;
        if (p.nchw_runs) {
            c = run / p.R;
            r = run - c * p.R;
        } else {
            c = 0;
            r = run;
        }
    }
    __device__ __forceinline__ void step(const TcParams &p) {
        if (++cr == p.cpr) {
            cr = 0;
            ++run;
            if (++r == p.R && p.nchw_runs) {
                r = 0;
                ++c;
            }
        }
    }
};

// Loads the chunk of EPC elements that starts at `src`, of which only chunk
// elements [ja, jb) are requested (0 <= ja < jb <= EPC), as aligned 32-bit
// words into raw[0..4] (one 128-bit load when the whole chunk is requested and
// aligned).  A word is loaded only if it holds a requested element, so nothing
// outside the requested elements' words is touched; *mis is the element
// misalignment of `src` (BF16 only).  `src` itself may lie outside the tensor
// when ja > 0.
template <typename T>
__device__ __forceinline__ void load_chunk_raw(const T *src, int ja, int jb, uint32_t (&raw)[5],
                                               int &mis) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(src);
    constexpr int EPC = 16 / (int)sizeof(T);
    if (ja == 0 && jb == EPC && (a & 15u) == 0) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(a));
        raw[0] = v.x; raw[1] = v.y; raw[2] = v.z; raw[3] = v.w; raw[4] = 0;
        mis = 0;
        return;
    }
    if constexpr (sizeof(T) == 2) {
        mis = (int)((a >> 1) & 1u);
        const uint32_t *wp = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
        // word i holds chunk elements 2i - mis and 2i + 1 - mis
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            const bool need = (2 * i - mis < jb) && (2 * i + 1 - mis >= ja);
            raw[i] = need ? __ldg(wp + i) : 0u;
        }
    } else {
        mis = 0;
        const uint32_t *wp = reinterpret_cast<const uint32_t *>(a);
#pragma unroll
        for (int i = 0; i < 4; ++i) raw[i] = (i >= ja && i < jb) ? __ldg(wp + i) : 0u;
        raw[4] = 0;
    }
}

// Zeroes chunk elements outside [ja, jb).
template <typename T>
__device__ __forceinline__ void mask_chunk(uint32_t (&o)[4], int ja, int jb) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (sizeof(T) == 2) {
            const bool lo_ok = (2 * i >= ja) && (2 * i < jb);
            const bool hi_ok = (2 * i + 1 >= ja) && (2 * i + 1 < jb);
            o[i] &= (lo_ok ? 0x0000FFFFu : 0u) | (hi_ok ? 0xFFFF0000u : 0u);
        } else {
            if (i < ja || i >= jb) o[i] = 0u;
        }
    }
}

// Aligns the raw words of load_chunk_raw and zeroes elements outside [ja, jb).
template <typename T>
__device__ __forceinline__ void combine_chunk(const uint32_t (&raw)[5], int mis, int ja, int jb,
                                              uint32_t (&o)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = mis ? __funnelshift_r(raw[i], raw[i + 1], 16) : raw[i];
    mask_chunk<T>(o, ja, jb);
}

// Fills A row `t` (output pixel m) of reduction block kb from global memory.
// Run elements [e_lo, e_hi) of the row's window lie inside the image along W;
// filter rows outside [0, H) are zero.  Every load of the row is issued
// before the first store.
template <typename T>
__device__ __forceinline__ void fill_a_row_runs(const TcParams &p, uint8_t *row, int t, int kb,
                                                bool valid, const T *xn, int h0, int w0, int e_lo,
                                                int e_hi) {
    constexpr int EPC = 16 / (int)sizeof(T);
    RunPos rp;
    rp.start(p, kb * 8);
    uint32_t raw[8][5];
    int mis[8], jas[8], jbs[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        int ja = 0, jb = 0;
        const T *src = xn;
        if (valid && rp.run < p.num_runs) {
            const int h = h0 + rp.r * p.dh;
            if (h >= 0 && h < p.H) {
                const int e0 = rp.cr * EPC;
                const int lo = max(e0, e_lo), hi = min(e0 + EPC, e_hi);
                if (lo < hi) {
                    ja = lo - e0;
                    jb = hi - e0;
                    src = xn + (long long)h * p.xs[2] +
                          (p.nchw_runs ? (long long)rp.c * p.xs[1] + w0 : (long long)w0 * p.C) + e0;
                }
            }
        }
        jas[j] = ja;
        jbs[j] = jb;
        mis[j] = 0;
        if (ja < jb) {
            load_chunk_raw<T>(src, ja, jb, raw[j], mis[j]);
        } else {
#pragma unroll
            for (int i = 0; i < 5; ++i) raw[j][i] = 0u;
        }
        rp.step(p);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t o[4];
        combine_chunk<T>(raw[j], mis[j], jas[j], jbs[j], o);
        store_chunk(row, t, j, o[0], o[1], o[2], o[3]);
    }
}

__device__ __forceinline__ uint32_t lds32(uint32_t saddr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(saddr));
    return v;
}

// Fills A row `t` of reduction block kb from the tile's halo: input rows
// [hr0, hr0 + hrows) of the tile's image, full width, staged at shared byte
// address `hs` (element (hr0, 0, 0)).  Channels-innermost runs only.  A chunk
// is read as the 32-bit words that cover it (a BF16 chunk starts 0 or 2 bytes
// into a word) and shifted into place; only chunks cut by the image border
// or by the run's end are masked.  The halo buffers are padded so that the
// words around a chunk stay inside this CTA's shared memory.
template <typename T>
__device__ __forceinline__ void fill_a_row_halo(const TcParams &p, uint8_t *row, int t, int kb,
                                                bool valid, uint32_t hs, int hr0, int hrows,
                                                int h0, int w0, int e_lo, int e_hi,
                                                const int4 *ctab) {
    constexpr int EPC = 16 / (int)sizeof(T);
    const int WC = p.W * p.C;
    const int hb = h0 - hr0;                  // halo row of filter row 0
    const int base = hb * WC + w0 * p.C;      // halo element of (filter row 0, s = 0, c = 0)
    const int4 *tb = ctab + kb * 8;
    uint32_t o[8][4];
    // all shared loads of the row first (the stores below are compiler
    // barriers), then the stores
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0u;
        const int4 e = tb[j];  // (filter row r, channel c, element offset e0, in range)
        const int hr = hb + e.x * p.dh;
        if (valid && e.w && (unsigned)hr < (unsigned)hrows) {  // rows off the halo are padding
            const int ja = max(e_lo - e.z, 0), jb = min(e_hi - e.z, EPC);
            if (ja < jb) {
                const int el = base + e.x * p.dh * WC + e.z;  // may be < 0 when ja > 0
                const uint32_t sa = hs + (uint32_t)(el * (int)sizeof(T));
                const uint32_t wa = sa & ~3u;
                if constexpr (sizeof(T) == 2) {
                    uint32_t w[5];
#pragma unroll
                    for (int i = 0; i < 5; ++i) w[i] = lds32(wa + 4 * i);
                    const uint32_t sh = (sa & 2u) * 8u;  // 0 or 16
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[j][i] = __funnelshift_r(w[i], w[i + 1], sh);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[j][i] = lds32(wa + 4 * i);
                }
                if ((ja | (jb - EPC)) != 0) mask_chunk<T>(o[j], ja, jb);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) store_chunk(row, t, j, o[j][0], o[j][1], o[j][2], o[j][3]);
}

// The per-(k-block, chunk) table of the run layout: filter row, channel,
// element offset inside the run, and whether the chunk holds a run at all.
template <int GROUPS>
__device__ void build_chunk_table(const TcParams &p, int4 *tab) {
    constexpr int EPC_BF16 = 8;
    (void)EPC_BF16;
    const int epc = p.epc;
    for (int i = threadIdx.x; i < p.num_kb * 8; i += 128 * GROUPS) {
        RunPos rp;
        rp.start(p, i);
        tab[i] = make_int4(rp.r, rp.c, rp.cr * epc, rp.run < p.num_runs ? 1 : 0);
    }
}

// Copies input rows [hr0, hr0 + hrows) of image n (contiguous bytes) into the
// halo buffer at shared address `dst` with 16-byte cp.async copies of the
// aligned envelope (each copied 16-byte block holds at least one byte of the
// rows); returns the shared address of element (hr0, 0, 0).
template <typename T>
__device__ __forceinline__ uint32_t halo_copy(const TcParams &p, uint32_t dst, int n, int hr0,
                                              int hrows, int tid, int nthr) {
    const uintptr_t src = reinterpret_cast<uintptr_t>(static_cast<const T *>(p.x) +
                                                      (long long)n * p.xs[0] +
                                                      (long long)hr0 * p.xs[2]);
    const uintptr_t a0 = src & ~(uintptr_t)15;
    if (hrows > 0) {
        const uintptr_t a1 = (src + (uintptr_t)hrows * p.xs[2] * sizeof(T) + 15) & ~(uintptr_t)15;
        for (uintptr_t a = a0 + (uintptr_t)tid * 16; a < a1; a += (uintptr_t)nthr * 16)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + (uint32_t)(a - a0)),
                         "l"(a)
                         : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    return dst + (uint32_t)(src - a0);
}

// Input rows of the tile's image that a tile reads: [hr0, hr0 + hrows).
__device__ __forceinline__ void tile_halo_rows(const TcParams &p, const TileCoord &tc, int &n,
                                               int &hr0, int &hrows) {
    n = (int)(tc.m0 / p.PQ);
    const int ml = (int)(tc.m0 - (long long)n * p.PQ);
    const int pa = ml / p.Q, pb = (ml + tc.rows - 1) / p.Q;
    const int lo = max(0, pa * p.u - p.pt);
    const int hi = min(p.H - 1, pb * p.u - p.pt + p.dh * (p.R - 1));
    hr0 = lo;
    hrows = hi >= lo ? hi - lo + 1 : 0;
}

// Fills the BN filter rows of reduction block kb into `dst`; one task per
// (row, 16-byte chunk), spread over `nthr` threads, four tasks per thread at a
// time with all their loads issued first.
template <typename T, int MODE>
__device__ void fill_b_block(const TcParams &p, uint8_t *dst, int kb, int k0, int tid, int nthr) {
    constexpr int EPC = 16 / (int)sizeof(T);
    constexpr int BATCH = 4;
    const T *w = static_cast<const T *>(p.w);
    const int tasks = p.BN * 8;
    for (int base = tid; base < tasks; base += BATCH * nthr) {
        uint32_t o[BATCH][4];
        if constexpr (MODE == MODE_RUNS) {
            uint32_t raw[BATCH][5];
            int mis[BATCH], jbs[BATCH];
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const int task = base + b * nthr;
                const int br = task >> 3, j = task & 7;
                const int k = k0 + br;
                jbs[b] = 0;
                mis[b] = 0;
#pragma unroll
                for (int i = 0; i < 5; ++i) raw[b][i] = 0u;
                if (task < tasks && k < p.K) {
                    RunPos rp;
                    rp.start(p, kb * 8 + j);
                    if (rp.run < p.num_runs) {
                        const int e0 = rp.cr * EPC;
                        jbs[b] = min(EPC, p.run_len - e0);
                        const T *src = w + (long long)k * p.ws[0] + (long long)rp.r * p.ws[2] +
                                       (p.nchw_runs ? (long long)rp.c * p.ws[1] : 0) + e0;
                        load_chunk_raw<T>(src, 0, jbs[b], raw[b], mis[b]);
                    }
                }
            }
#pragma unroll
            for (int b = 0; b < BATCH; ++b) combine_chunk<T>(raw[b], mis[b], 0, jbs[b], o[b]);
        } else {
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const int task = base + b * nthr;
                const int br = task >> 3, j = task & 7;
                const int k = k0 + br;
                o[b][0] = o[b][1] = o[b][2] = o[b][3] = 0u;
                if (task < tasks && k < p.K)
                    gather_elem_chunk<T, false>(p, w + (long long)k * p.ws[0], true, 0, 0,
                                                (kb * 8 + j) * EPC, o[b]);
            }
        }
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
            const int task = base + b * nthr;
            if (task < tasks) {
                const int br = task >> 3, j = task & 7;
                store_chunk(dst + br * ROW_BYTES, br, j, o[b][0], o[b][1], o[b][2], o[b][3]);
            }
        }
    }
}

// Shared byte offset of element (hr0, 0, 0) inside its halo buffer: the copy
// starts at the 16-byte boundary at or below it.
template <typename T>
__device__ __forceinline__ uint32_t halo_align(const TcParams &p, int n, int hr0) {
    const uintptr_t src = reinterpret_cast<uintptr_t>(static_cast<const T *>(p.x) +
                                                      (long long)n * p.xs[0] +
                                                      (long long)hr0 * p.xs[2]);
    return (uint32_t)(src & 15u);
}

// Named barrier of all producer threads (id 2).
template <int GROUPS>
__device__ __forceinline__ void producer_bar() {
    asm volatile("bar.sync 2, %0;" ::"n"(128 * GROUPS) : "memory");
}

template <typename T, int MODE, int GROUPS>
__device__ void produce_gather(const TcParams &p, uint8_t *smA, uint8_t *smB, uint8_t *smH,
                               int4 *ctab, uint64_t *full, uint64_t *empty, uint64_t *bres,
                               const WaitCtl &ctl) {
    constexpr int EPC = 16 / (int)sizeof(T);
    constexpr int BK = ROW_BYTES / (int)sizeof(T);
    const int group = threadIdx.x >> 7;  // producer warps are 0 .. 4*GROUPS-1
    const int t = threadIdx.x & 127;
    const int ST = p.stages;
    const uint32_t b_stage = (uint32_t)p.BN * ROW_BYTES;
    const T *x = static_cast<const T *>(p.x);
    const bool halo = MODE == MODE_RUNS && p.halo;
    const uint32_t hbase = smem_u32(smH);

    if (p.b_res) {  // the whole filter tile stays in shared memory
        for (int kb = 0; kb < p.num_kb; ++kb)
            fill_b_block<T, MODE>(p, smB + (size_t)kb * b_stage, kb, 0, threadIdx.x, 128 * GROUPS);
        fence_proxy_async_smem();
        mbar_arrive(bres);
    }
    if (MODE == MODE_RUNS && p.ctab) {
        build_chunk_table<GROUPS>(p, ctab);
        producer_bar<GROUPS>();
    }
    WorkIter wi(p);
    Seg sg;
    if (halo) {  // prefetch the first tile's input rows
        WorkIter w2 = wi;
        Seg s2;
        if (w2.next(p, s2)) {
            int n, r0, rows;
            tile_halo_rows(p, tile_coord(p, s2.tile), n, r0, rows);
            halo_copy<T>(p, hbase, n, r0, rows, threadIdx.x, 128 * GROUPS);
        }
    }
    int it = 0, seq = 0, stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    // Every producer thread walks every segment (even after an abort) so that
    // the named barriers below are always reached by all of them.
    while (wi.next(p, sg)) {
        const TileCoord tc = tile_coord(p, sg.tile);
        int hn = 0, hr0 = 0, hrows = 0;
        uint32_t hs = 0;
        if (halo) {
            asm volatile("cp.async.wait_all;" ::: "memory");
            producer_bar<GROUPS>();  // this tile's rows landed; the previous tile is done
            tile_halo_rows(p, tc, hn, hr0, hrows);
            hs = hbase + (uint32_t)(seq & 1) * p.halo_bytes + halo_align<T>(p, hn, hr0);
            WorkIter w2 = wi;  // prefetch the next tile into the other buffer
            Seg s2;
            if (w2.next(p, s2)) {
                int n2, r2, rows2;
                tile_halo_rows(p, tile_coord(p, s2.tile), n2, r2, rows2);
                halo_copy<T>(p, hbase + (uint32_t)((seq + 1) & 1) * p.halo_bytes, n2, r2, rows2,
                             threadIdx.x, 128 * GROUPS);
            }
            ++seq;
        }
        const long long m = tc.m0 + t;
        const bool valid = t < tc.rows;
        int n = 0, op = 0, oq = 0;
        if (valid) {
            n = (int)(m / p.PQ);
            const int rem = (int)(m - (long long)n * p.PQ);
            op = rem / p.Q;
            oq = rem - op * p.Q;
        }
        const int h0 = op * p.u - p.pt, w0 = oq * p.v - p.pl;
        const T *xn = x + (long long)n * p.xs[0];
        // run elements whose pixel lies inside the image along W (dw == 1 in run mode)
        const int run_c = p.nchw_runs ? 1 : p.C;
        const int e_lo = max(0, -w0) * run_c;
        const int e_hi = max(0, min(p.S, p.W - w0)) * run_c;  // <= run_len
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
            // iteration `it` uses ring slot `stage` in pass parity `ph`; the
            // groups take iterations in turn
            const int my_stage = stage;
            const uint32_t my_ph = ph;
            const bool mine = (GROUPS == 1) || ((it % GROUPS) == group);
            ++it;
            if (++stage == ST) {
                stage = 0;
                ph ^= 1u;
            }
            if (!mine || !ok) continue;
            if (!mbar_wait(&empty[my_stage], my_ph ^ 1u, ctl, 6)) {
                ok = false;
                continue;
            }
            uint8_t *arow = smA + (size_t)my_stage * A_STAGE_BYTES + t * ROW_BYTES;
            if constexpr (MODE == MODE_RUNS) {
                if (halo)
                    fill_a_row_halo<T>(p, arow, t, kb, valid, hs, hr0, hrows, h0, w0, e_lo, e_hi,
                                       ctab);
                else
                    fill_a_row_runs<T>(p, arow, t, kb, valid, xn, h0, w0, e_lo, e_hi);
            } else {
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {
                    uint32_t o[4];
                    gather_elem_chunk<T, true>(p, xn, valid, h0, w0, kb * BK + j * EPC, o);
                    store_chunk(arow, t, j, o[0], o[1], o[2], o[3]);
                }
            }
            if (!p.b_res)
                fill_b_block<T, MODE>(p, smB + (size_t)my_stage * b_stage, kb, tc.k0, t, 128);
            fence_proxy_async_smem();
            mbar_arrive(&full[my_stage]);
        }
    }
    if (halo) asm volatile("cp.async.wait_all;" ::: "memory");  // no copy may outlive the CTA
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread)
// ---------------------------------------------------------------------------
// The loop body is kept short: the issuing thread shares its scheduler with
// an epilogue warp, and every instruction it spends between MMAs is tensor
// time lost.  Stage/phase advance by increments, shared-memory descriptors by
// adds to their 14-bit address field (16-byte units; 227 KB stays below 2^14).
template <bool TF32>
__device__ void issue_mma(const TcParams &p, uint32_t tmem_base, uint8_t *smA, uint8_t *smB,
                          uint64_t *full, uint64_t *empty, uint64_t *tfull, uint64_t *tempty,
                          uint64_t *mma_done, uint64_t *bres, const WaitCtl &ctl) {
    const int ST = p.stages;
    const uint64_t a_desc0 = sw128_kmajor_desc(smem_u32(smA));
    const uint64_t b_desc0 = sw128_kmajor_desc(smem_u32(smB));
    const uint32_t a_step = A_STAGE_BYTES >> 4;               // per stage
    const uint32_t b_step = ((uint32_t)p.BN * ROW_BYTES) >> 4;  // per stage or resident block
    const uint32_t idesc = p.idesc;
    const bool b_res = p.b_res != 0;
    int stage = 0, t = 0;
    uint32_t phase = 0;
    bool ok = true;
    if (b_res && !mbar_wait(bres, 0u, ctl, 7)) ok = false;
    WorkIter wi(p);
    Seg sg;
    while (ok && wi.next(p, sg)) {
        const int buf = t & 1;
        const uint32_t aph = (uint32_t)(t >> 1) & 1u;
        if (!mbar_wait(&tempty[buf], aph ^ 1u, ctl, 3)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)buf * p.acc_stride;
        uint32_t acc = 0u;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
            if (!mbar_wait(&full[stage], phase, ctl, 4)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint64_t ad = a_desc0 + (uint64_t)((uint32_t)stage * a_step);
            const uint64_t bd = b_desc0 + (uint64_t)((uint32_t)(b_res ? kb : stage) * b_step);
            // four K slices of 32 bytes: +2 in the descriptor's 16-byte address units
            if constexpr (TF32) {
                umma_tf32(d_tmem, ad, bd, idesc, acc);
                umma_tf32(d_tmem, ad + 2, bd + 2, idesc, 1u);
                umma_tf32(d_tmem, ad + 4, bd + 4, idesc, 1u);
                umma_tf32(d_tmem, ad + 6, bd + 6, idesc, 1u);
            } else {
                umma_bf16(d_tmem, ad, bd, idesc, acc);
                umma_bf16(d_tmem, ad + 2, bd + 2, idesc, 1u);
                umma_bf16(d_tmem, ad + 4, bd + 4, idesc, 1u);
                umma_bf16(d_tmem, ad + 6, bd + 6, idesc, 1u);
            }
            umma_commit(&empty[stage]);  // stage free once these MMAs are done
            acc = 1u;
            if (++stage == ST) {
                stage = 0;
                phase ^= 1u;
            }
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

// Writes 16 finished FP32 values (columns 16*half .. 16*half+15 of a 32-column
// group) into row `lane` of a warp's 32 x 128-byte staging buffer, in the
// 128-byte swizzle of the y tensor map (16-byte chunk j of row r at j ^ (r % 8)).
__device__ __forceinline__ void stage_half_row(uint8_t *buf, int lane, int half,
                                               const float (&val)[16]) {
    uint8_t *rowp = buf + lane * 128;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint8_t *dst = rowp + (((half * 4 + j) ^ (lane & 7)) << 4);
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(dst)),
                     "f"(val[4 * j]), "f"(val[4 * j + 1]), "f"(val[4 * j + 2]), "f"(val[4 * j + 3])
                     : "memory");
    }
}

// Named barrier of the four epilogue warps (id 1; the block-wide barrier is 0).
__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Waits (bounded) until another CTA has published the partial sum of a tile.
__device__ bool wait_partial_flag(int *flag, const WaitCtl &ctl) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v != 0) return true;
        if (*ctl.abort_flag) return false;
        if (globaltimer_ns() - t0 > ctl.timeout_ns) {
            *ctl.abort_flag = 1;
            record_error(ctl.err, 1 /* DLC_DEVERR_WAIT_TIMEOUT */, 8);
            return false;
        }
        __nanosleep(128);
    }
}

// DEPTH 16-column TMEM loads are in flight before each wait.
template <int DEPTH>
__device__ void epilogue(const TcParams &p, uint32_t tmem_base, uint64_t *tfull, uint64_t *tempty,
                         uint8_t *epi_smem, const CUtensorMap *tmY, const WaitCtl &ctl) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    const int row = quad * 32 + lane;
    const bool leader = threadIdx.x == blockDim.x - 128;  // first epilogue thread
    float *yf = static_cast<float *>(p.y);
    unsigned short *yb = static_cast<unsigned short *>(p.y);
    uint8_t *my_bufs = epi_smem + quad * 2 * EPI_BUF_BYTES;
    int nbuf = 0;  // staging buffers used so far by this warp
    int t = 0;
    WorkIter wi(p);
    Seg sg;
    while (wi.next(p, sg)) {
        const int buf = t & 1;
        const uint32_t aph = (uint32_t)(t >> 1) & 1u;
        int okw = 0;
        if (lane == 0) okw = mbar_wait(&tfull[buf], aph, ctl, 5) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) break;
        __syncwarp();
        tc_fence_after_sync();
        const TileCoord tc = tile_coord(p, sg.tile);
        // Stream-K: a tile split between two CTAs.  The CTA holding its last
        // k-blocks runs them first and parks the raw FP32 partial sum in y
        // (tail); the CTA holding its first k-blocks runs them last, adds the
        // parked partial and applies the epilogue (head).
        const bool tail = p.sk && sg.kb0 > 0;
        const bool head = p.sk && sg.kb0 == 0 && sg.kb1 < p.num_kb;
        bool have_partial = false;
        if (head) {
            if (leader) {
                int *flag = p.sk_flags + sg.tile;
                if (wait_partial_flag(flag, ctl)) *flag = 0;  // consumed; zero for the next launch
            }
            epilogue_bar();
            have_partial = !*ctl.abort_flag;
        }
        const long long m = tc.m0 + row;
        const bool valid = row < tc.rows;
        long long ybase = 0;
        if (valid) {
            const int n = (int)(m / p.PQ);
            const int rem = (int)(m - (long long)n * p.PQ);
            const int op = rem / p.Q, oq = rem - (rem / p.Q) * p.Q;
            ybase = (long long)n * p.ys[0] + (long long)op * p.ys[2] + (long long)oq * p.ys[3];
        }
        const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)buf * p.acc_stride;
        // bulk stores need this warp's 32 rows to be rows of this tile (an
        // image-aligned tile may end early; rows past M are clipped by the map)
        const bool tma_warp = p.y_tma && !tail && (p.img_tiles == 0 || quad * 32 + 32 <= tc.rows);
        int half = 0;  // which 16-column half of the current 32-column group
        bool stop = false;
        for (int c00 = 0; c00 < p.BN && !stop; c00 += 16 * DEPTH) {
        const int nsub = min(DEPTH, (p.BN - c00) >> 4);
        uint32_t vv[DEPTH][16];
#pragma unroll
        for (int q = 0; q < DEPTH; ++q)
            if (q < nsub) tmem_ld_32x32b_x16(taddr + (uint32_t)(c00 + 16 * q), vv[q]);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < DEPTH; ++q) {
            if (q >= nsub || stop) break;
            uint32_t (&v)[16] = vv[q];
            const int c0 = c00 + 16 * q;
            const int kbase = tc.k0 + c0;
            // 16 consecutive filters of one pixel contiguous and 16-byte aligned in y
            const bool vec16 = valid && p.ys[1] == 1 && kbase + 16 <= p.K &&
                               ((reinterpret_cast<uintptr_t>(yf + ybase + kbase) & 15u) == 0);
            if (tail) {  // park the raw partial sum (FP32 y, any strides)
                if (vec16) {
                    float4 *dst = reinterpret_cast<float4 *>(yf + ybase + kbase);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        __stcg(dst + j, make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                                    __uint_as_float(v[4 * j + 2]),
                                                    __uint_as_float(v[4 * j + 3])));
                } else if (valid) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (kbase + j < p.K)
                            __stcg(yf + ybase + (long long)(kbase + j) * p.ys[1], __uint_as_float(v[j]));
                }
                continue;
            }
            if (have_partial && vec16) {
                const float4 *src = reinterpret_cast<const float4 *>(yf + ybase + kbase);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 f = __ldcg(src + j);
                    v[4 * j] = __float_as_uint(__uint_as_float(v[4 * j]) + f.x);
                    v[4 * j + 1] = __float_as_uint(__uint_as_float(v[4 * j + 1]) + f.y);
                    v[4 * j + 2] = __float_as_uint(__uint_as_float(v[4 * j + 2]) + f.z);
                    v[4 * j + 3] = __float_as_uint(__uint_as_float(v[4 * j + 3]) + f.w);
                }
            } else if (have_partial && valid) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (kbase + j < p.K)
                        v[j] = __float_as_uint(__uint_as_float(v[j]) +
                                               __ldcg(yf + ybase + (long long)(kbase + j) * p.ys[1]));
            }
            if (tma_warp) {
                if (kbase >= p.K) {  // warp-uniform; nothing is pending here
                    stop = true;
                    break;
                }
                float val[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float f = p.alpha * __uint_as_float(v[j]);
                    const int k = kbase + j;
                    if (valid && k < p.K) {
                        if (p.beta != 0.f) f = __fmaf_rn(p.beta, yf[ybase + k], f);
                        if (p.bias) f += __ldg(p.bias + k);
                    }
                    if (p.relu) f = fmaxf(f, 0.f);
                    val[j] = f;
                }
                uint8_t *sb = my_bufs + (nbuf & 1) * EPI_BUF_BYTES;
                if (half == 0 && nbuf >= 2) {  // the store issued from this buffer two groups ago
                    if (lane == 0) bulk_wait_group_read<1>();
                    __syncwarp();
                }
                stage_half_row(sb, lane, half, val);
                if (half == 1 || c0 + 16 >= p.BN || kbase + 16 >= p.K) {  // group complete
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(tmY, sb, kbase - 16 * half, (int)(tc.m0 + quad * 32));
                        bulk_commit_group();
                    }
                    ++nbuf;
                    half = 0;
                } else {
                    half = 1;
                }
                continue;
            }
            if (!valid) continue;
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
        }
        if (tail) {  // publish the partial once every epilogue thread has stored its part
            __threadfence();
            epilogue_bar();
            if (leader)
                asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p.sk_flags + sg.tile), "r"(1)
                             : "memory");
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        ++t;
    }
    // staged stores must finish reading shared memory before the CTA exits (the
    // grid's completion makes their writes visible)
    if (p.y_tma && lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int MODE>
struct KernelShape {
    static constexpr int PROD_WARPS = MODE == MODE_IM2COL ? 1 : 4 * GATHER_GROUPS;
    static constexpr int THREADS = (PROD_WARPS + 5) * 32;  // + MMA warp + 4 epilogue warps
};

template <bool TF32, int MODE>
__global__ void __launch_bounds__(KernelShape<MODE>::THREADS, 1)
    conv_fprop_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmY) {
    using T = typename std::conditional<TF32, uint32_t, uint16_t>::type;
    constexpr int BK = ROW_BYTES / (int)sizeof(T);
    constexpr int PROD_WARPS = KernelShape<MODE>::PROD_WARPS;
    constexpr int MMA_WARP = PROD_WARPS;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int ST = p.stages;
    const int b_blocks = p.b_res ? p.num_kb : ST;
    uint8_t *smA = smem;
    uint8_t *epi_smem = smem + (size_t)ST * A_STAGE_BYTES;  // 1024-aligned staging of y
    uint8_t *smB = epi_smem + (p.y_tma ? EPI_SMEM : 0);
    uint8_t *smH = smB + (size_t)b_blocks * p.BN * ROW_BYTES;  // halo buffers (run gather)
    int4 *ctab = reinterpret_cast<int4 *>(smH + (p.halo ? 2 * (size_t)p.halo_bytes : 0));
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(ctab) +
                                                  (p.ctab ? (size_t)p.num_kb * 8 * 16 : 0));
    uint64_t *full = bars;
    uint64_t *empty = bars + ST;
    uint64_t *tfull = bars + 2 * ST;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint64_t *bres = mma_done + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bres + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full[i], MODE == MODE_IM2COL ? 1u : 128u);
            mbar_init(&empty[i], 1u);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1u);
            mbar_init(&tempty[i], 4u);  // one arrival per epilogue warp
        }
        mbar_init(mma_done, 1u);
        mbar_init(bres, 128u * GATHER_GROUPS);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (MODE == MODE_IM2COL && warp == 0 && lane == 0) {
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
        if constexpr (MODE == MODE_IM2COL) {
            if (lane == 0) produce_tma<BK>(p, &tmA, &tmB, smA, smB, full, empty, ctl);
        } else {
            produce_gather<T, MODE, GATHER_GROUPS>(p, smA, smB, smH, ctab, full, empty, bres, ctl);
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0)
            issue_mma<TF32>(p, tmem_base, smA, smB, full, empty, tfull, tempty, mma_done, bres, ctl);
    } else {
        if (p.y_tma && lane == 0) prefetch_tmap(&tmY);
        // the gather kernels run 13 warps and have fewer registers per thread
        epilogue<MODE == MODE_IM2COL ? 4 : 1>(p, tmem_base, tfull, tempty, epi_smem, &tmY, ctl);
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

// Run gather: channels-innermost activations with densely packed pixels and
// KRSC filters (runs over (s, c) of one filter row), or width-innermost
// activations with KCRS filters (runs over s of one (c, r)); no dilation
// along W so that a run is contiguous.
bool runs_ok(const ConvProblem &pb, int *run_len, int *num_runs, int *nchw) {
    if (pb.dw != 1) return false;
    long long len, runs;
    if (pb.xs[1] == 1 && pb.xs[3] == pb.C && pb.wfmt == DLC_TENSOR_NHWC) {
        len = (long long)pb.S * pb.C;
        runs = pb.R;
        *nchw = 0;
    } else if (pb.xs[3] == 1 && pb.wfmt == DLC_TENSOR_NCHW) {
        len = pb.S;
        runs = (long long)pb.C * pb.R;
        *nchw = 1;
    } else {
        return false;
    }
    if (len > 4096 || runs * (len + 8) > 0x3fffffffLL) return false;
    *run_len = (int)len;
    *num_runs = (int)runs;
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

template <bool TF32, int MODE>
cudaError_t launch_kernel(const TcParams &tp, const CUtensorMap &a, const CUtensorMap &b,
                          const CUtensorMap &y, int grid, size_t smem, cudaStream_t st) {
    auto kern = conv_fprop_tc_kernel<TF32, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, KernelShape<MODE>::THREADS, smem, st>>>(tp, a, b, y);
    return cudaGetLastError();
}

template <bool TF32>
cudaError_t launch_mode(int mode, const TcParams &tp, const CUtensorMap &a, const CUtensorMap &b,
                        const CUtensorMap &y, int grid, size_t smem, cudaStream_t st) {
    if (mode == MODE_IM2COL) return launch_kernel<TF32, MODE_IM2COL>(tp, a, b, y, grid, smem, st);
    if (mode == MODE_RUNS) return launch_kernel<TF32, MODE_RUNS>(tp, a, b, y, grid, smem, st);
    return launch_kernel<TF32, MODE_GATHER>(tp, a, b, y, grid, smem, st);
}

// y as a 2-D [M rows, K columns] tensor for bulk tensor stores: K contiguous,
// every output pixel row at one uniform pitch, 16-byte aligned base and pitch.
bool y_tma_ok(const ConvProblem &pb) {
    const long long e = pb.ydt == DLC_DATA_BFLOAT16 ? 2 : 4;
    if (pb.ys[1] != 1) return false;
    const long long pitch = pb.ys[3];
    if (pitch < pb.K || (pitch * e) % 16 || pitch * e >= (1LL << 40)) return false;
    if (pb.P > 1 && pb.ys[2] != (long long)pb.Q * pitch) return false;
    if (pb.N > 1 && pb.ys[0] != (long long)pb.P * pb.Q * pitch) return false;
    if (pb.y && ((uintptr_t)pb.y % 16)) return false;
    return (long long)pb.N * pb.P * pb.Q <= 0xffffffffLL;
}

}  // namespace

bool dlc_im2col_ok(const ConvProblem &pb) { return tc_math_ok(pb) && im2col_ok(pb); }

dlcKernel_t dlc_tc_variant(const dlcContext *ctx, const ConvProblem &pb) {
    if (!tc_math_ok(pb)) return DLC_KERNEL_NONE;
    if (!fits_i32((long long)pb.P * pb.Q)) return DLC_KERNEL_NONE;
    // Convolution mode (pb.flip): the SM-pair kernel mirrors its filter-load
    // coordinates; the window and gather kernels read a mirrored strided view
    // of the filters; the single-SM im2col and run-gather kernels, whose filter
    // loads assume forward order, are not used.
    if (im2col_ok(pb)) {
        if (dlc_pair_enabled(ctx)) return DLC_KERNEL_TC_IM2COL_PAIR;
        if (!pb.flip) return DLC_KERNEL_TC_IM2COL;
    }
    // channel-planar TF32 layers with few filters: the row-stack kernel's
    // MMAs are 192-256 pixels wide where the window kernel's are 64
    if (dlc_rowstack_ok(ctx, pb)) return DLC_KERNEL_TC_ROWSTACK;
    if (dlc_window_ok(pb)) return DLC_KERNEL_TC_WINDOW;
    int a, b, c;
    if (!pb.flip && runs_ok(pb, &a, &b, &c)) return DLC_KERNEL_TC_GATHER_RUNS;
    return DLC_KERNEL_TC_GATHER;
}

dlcStatus_t dlc_launch_tc(dlcContext *ctx, const ConvProblem &pb, dlcKernel_t variant) {
    if (variant == DLC_KERNEL_TC_WINDOW) return dlc_launch_window(ctx, pb);
    if (variant == DLC_KERNEL_TC_IM2COL_PAIR) return dlc_launch_pair(ctx, pb);
    if (variant == DLC_KERNEL_TC_ROWSTACK) return dlc_launch_rowstack(ctx, pb);
    int mode;
    if (variant == DLC_KERNEL_TC_IM2COL) mode = MODE_IM2COL;
    else if (variant == DLC_KERNEL_TC_GATHER_RUNS) mode = MODE_RUNS;
    else if (variant == DLC_KERNEL_TC_GATHER) mode = MODE_GATHER;
    else return DLC_STATUS_INTERNAL_ERROR;
    const bool tf32 = pb.math == DLC_MATH_TF32;
    const int e = elt_bytes(pb);
    const int BK = ROW_BYTES / e;
    const int EPC = 16 / e;

    TcParams tp;
    std::memset(&tp, 0, sizeof(tp));
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
    // tuning knobs for tile sweeps: DLC_TC_BN (multiple of 16, 16..256), DLC_TC_STAGES (2..8)
    if (const char *ev = std::getenv("DLC_TC_BN")) {
        const int bn = std::atoi(ev);
        if (bn >= 16 && bn <= 256 && bn % 16 == 0) tp.BN = bn;
    }
    tp.c_blocks = (pb.C + BK - 1) / BK;
    if (mode == MODE_IM2COL) {
        tp.num_kb = pb.R * pb.S * tp.c_blocks;
    } else if (mode == MODE_RUNS) {
        if (!runs_ok(pb, &tp.run_len, &tp.num_runs, &tp.nchw_runs)) return DLC_STATUS_INTERNAL_ERROR;
        tp.cpr = (tp.run_len + EPC - 1) / EPC;
        const long long chunks = (long long)tp.num_runs * tp.cpr;
        tp.num_kb = (int)((chunks + 7) / 8);
    } else {
        const long long kg = (long long)pb.R * pb.S * pb.C;
        if (kg > 0x3fffffffLL) return DLC_STATUS_NOT_SUPPORTED;
        tp.num_kb = (int)((kg + BK - 1) / BK);
    }
    tp.n_tiles = (pb.K + tp.BN - 1) / tp.BN;
    // Halo staging (run gather, channels-innermost, dense rows): M tiles are
    // image-aligned and each tile's input rows are staged in shared memory.
    long long halo_rows = 0;
    if (mode == MODE_RUNS && !tp.nchw_runs && pb.xs[2] == (long long)pb.W * pb.C) {
        const int it_img = (tp.PQ + BM - 1) / BM;
        for (int t = 0; t < it_img; ++t) {
            const int ml = t * BM, rows = std::min(BM, tp.PQ - ml);
            const int pa = ml / pb.Q, pbb = (ml + rows - 1) / pb.Q;
            const int lo = std::max(0, pa * pb.u - pb.pt);
            const int hi = std::min(pb.H - 1, pbb * pb.u - pb.pt + pb.dh * (pb.R - 1));
            halo_rows = std::max<long long>(halo_rows, hi >= lo ? hi - lo + 1 : 0);
        }
        const long long hb = ((halo_rows * pb.xs[2] * e + 16 + 127) / 128) * 128 + 128;
        if (hb <= 48 * 1024) {
            tp.halo = 1;
            tp.halo_bytes = (int)hb;
            tp.img_tiles = it_img;
        }
        if (const char *ev = std::getenv("DLC_TC_HALO"))
            if (std::atoi(ev) == 0) tp.halo = 0, tp.halo_bytes = 0, tp.img_tiles = 0;
    }
    tp.epc = EPC;
    tp.ctab = (tp.halo && tp.num_kb * 8 * 16 <= 16 * 1024) ? 1 : 0;
    if (tp.halo && !tp.ctab) tp.halo = 0, tp.halo_bytes = 0, tp.img_tiles = 0;
    const long long m_tiles =
        tp.img_tiles > 0 ? (long long)pb.N * tp.img_tiles : (tp.M + BM - 1) / BM;
    tp.num_tiles = m_tiles * tp.n_tiles;

    // shared memory: A stages plus either B stages or the resident filter
    // tile, plus the epilogue's staging buffers when y is stored by TMA
    // Bulk-tensor stores of y measured slower than direct stores from the
    // epilogue registers (small per-warp boxes), so they are opt-in.
    // FP32 y written through a 2-D [M, K] tensor map: bulk stores of 32-row x
    // 32-column groups from a staging buffer per epilogue warp (DLC_TC_YTMA=0
    // falls back to per-thread vector stores).
    // The im2col kernel's TMA unit is busy with operand loads (bulk stores
    // there measured up to 2.4x slower), so there y goes out through direct
    // vector stores from the epilogue registers.
    const bool y_rows = y_tma_ok(pb) && !tp.y_bf16 && (tp.n_tiles == 1 || tp.BN % 32 == 0);
    tp.y_tma = (y_rows && mode != MODE_IM2COL) ? 1 : 0;
    if (const char *ev = std::getenv("DLC_TC_YTMA")) tp.y_tma = y_rows && std::atoi(ev) != 0;
    const int b_stage = tp.BN * ROW_BYTES;
    const int ctab_bytes = tp.ctab ? tp.num_kb * 8 * 16 : 0;
    const int epi_bytes = tp.y_tma ? EPI_SMEM : 0;
    const int budget = MAX_DYN_SMEM - 1024 - BAR_AREA - epi_bytes -
                       (tp.halo ? 2 * tp.halo_bytes : 0) - ctab_bytes;
    const long long b_all = (long long)tp.num_kb * b_stage;
    tp.b_res = (mode != MODE_IM2COL && tp.n_tiles == 1 && b_all <= 120 * 1024 &&
                budget - b_all >= 4 * A_STAGE_BYTES) ? 1 : 0;
    int stages = tp.b_res ? (int)((budget - b_all) / A_STAGE_BYTES)
                          : budget / (A_STAGE_BYTES + b_stage);
    tp.stages = stages > 8 ? 8 : stages;
    if (const char *ev = std::getenv("DLC_TC_STAGES")) {
        const int st = std::atoi(ev);
        if (st >= 2 && st < tp.stages) tp.stages = st;
    }
    if (tp.stages < 2) return DLC_STATUS_INTERNAL_ERROR;
    const long long b_bytes = tp.b_res ? b_all : (long long)tp.stages * b_stage;

    // Stream-K: equal (tile, k-block) ranges per CTA, at most two parts per
    // tile (units per CTA >= k-blocks per tile because tiles >= CTAs).  The
    // partial is parked in y, so it needs FP32 y and beta == 0.
    long long grid = tp.num_tiles < ctx->sm_count ? tp.num_tiles : ctx->sm_count;
    tp.sk = 0;
    tp.sk_units = 0;
    tp.sk_flags = ctx->sk_flags;
    const bool sk_legal = ctx->sk_flags && pb.beta == 0.f && !tp.y_bf16 &&
                          tp.num_tiles >= ctx->sm_count && tp.num_tiles <= DLC_SK_FLAGS &&
                          tp.num_kb >= 4;
    if (sk_legal) {
        // Measured no faster than whole tiles on the small-image layers (the
        // parked partial costs an extra pass over the split tiles), so the
        // stream-K schedule is opt-in: DLC_TC_STREAMK=1.  Problems with more
        // tiles than there are flags run whole tiles.
        if (const char *ev = std::getenv("DLC_TC_STREAMK")) tp.sk = std::atoi(ev) != 0;
    }
    if (tp.sk) {
        const long long total = tp.num_tiles * tp.num_kb;
        tp.sk_units = (total + ctx->sm_count - 1) / ctx->sm_count;
        grid = (total + tp.sk_units - 1) / tp.sk_units;
    }

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

    CUtensorMap ta, tb, ty;
    std::memset(&ta, 0, sizeof(ta));
    std::memset(&tb, 0, sizeof(tb));
    std::memset(&ty, 0, sizeof(ty));
    if (tp.y_tma) {
        const bool yb16 = pb.ydt == DLC_DATA_BFLOAT16;
        const long long ye = yb16 ? 2 : 4;
        const cuuint64_t ydim[2] = {(cuuint64_t)pb.K, (cuuint64_t)tp.M};
        const cuuint64_t ystr[1] = {(cuuint64_t)(pb.ys[3] * ye)};
        const cuuint32_t ybox[2] = {32, 32};
        const cuuint32_t ones[2] = {1, 1};
        CUresult r = ctx->encode_tiled(
            &ty, yb16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, pb.y,
            ydim, ystr, ybox, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return DLC_STATUS_EXECUTION_FAILED;
    }
    if (mode == MODE_IM2COL) {
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

    const size_t smem = 1024 + (size_t)tp.stages * A_STAGE_BYTES + (size_t)b_bytes +
                        (tp.halo ? 2 * (size_t)tp.halo_bytes : 0) + ctab_bytes + epi_bytes +
                        BAR_AREA;
    if (grid < 1) grid = 1;
    cudaError_t err = tf32 ? launch_mode<true>(mode, tp, ta, tb, ty, (int)grid, smem, ctx->stream)
                           : launch_mode<false>(mode, tp, ta, tb, ty, (int)grid, smem, ctx->stream);
    if (err != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlc_preload_tc() {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, conv_fprop_tc_kernel<false, MODE_IM2COL>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_fprop_tc_kernel<false, MODE_RUNS>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_fprop_tc_kernel<false, MODE_GATHER>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_fprop_tc_kernel<true, MODE_IM2COL>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_fprop_tc_kernel<true, MODE_RUNS>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_fprop_tc_kernel<true, MODE_GATHER>) != cudaSuccess)
        return DLC_STATUS_EXECUTION_FAILED;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlc_launch_wait_selftest(dlcContext *ctx, unsigned long long timeout_ns) {
    wait_selftest_kernel<<<1, 32, 0, ctx->stream>>>(ctx->d_err, timeout_ns);
    if (cudaGetLastError() != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}
