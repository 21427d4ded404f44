// conv_window.cu -- forward convolution of layers with few input channels per
// horizontal stride step (first layers: C = 1..16), on the sm_103a tensor
// cores, with the reduction operand read in place from packed input rows.
//
// Lowering (cuDNN page, method section: tiles of the lowered matrix are formed
// in on-chip memory only; zero-memory-overhead page: no lowered copy in off-chip
// memory).  With horizontal stride v, the v input pixels w = v*P + phi - pl
// (phi < v) of an input row form "phase pixel" P: v*C values packed in
// (phi, c) order into D bytes (16, 32 or 64; zero past v*C).  Output pixel q of
// output row p then reads, for filter row r, phase pixels q .. q+A-1 of input
// row h = p*u + r*dh - pt: A*D contiguous bytes, and the windows of
// consecutive q start D bytes apart.  A K-major tcgen05 operand whose rows are
// D bytes apart -- no swizzle with 16-byte rows and a 16-byte K step between
// core matrices, or the 32-/64-byte swizzle, which the tensor core applies on
// absolute shared-memory address bits -- therefore reads the lowered rows of
// up to 128 consecutive output pixels straight out of one strip of phase
// pixels.  Filter taps are reordered to the same (a, phi, c) order once per CTA
// and stay resident in shared memory.
//
// Tiles: the 128 MMA rows are J output rows of one image (Qs rows each, Qs a
// power of two >= Q+A-1, J = 128/Qs) or, for wide rows (J = 1), 128 consecutive
// pixels of one output row.  Strip r of a tile holds, for output row j, the
// phase pixels of input row (p0+j)*u + r*dh - pt at pixel offset j*Qs; tile
// rows past Q read pixels whose value does not matter and are not stored.
//
// Roles (one persistent CTA per SM): eight producer warps pack the strips of
// the next tile into one of two buffers (batched 4-/8-byte loads; padding and
// the packing tail are zero-filled); one thread issues R*steps MMAs (32 bytes
// of reduction each) per tile into one of two TMEM accumulators; four epilogue
// warps read the accumulator, apply alpha, beta*y, bias and ReLU and store y
// (bulk tensor stores of 32x32 blocks when y is dense FP32).  Every wait is
// bounded and records an error word when it runs out.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace {

using namespace dlc;

constexpr int WBM = 128;                             // MMA rows (output pixels) per tile
constexpr int PROD_THREADS = 256;                    // eight producer warps
constexpr int MMA_WARP = PROD_THREADS / 32;          // warp 8
constexpr int WIN_THREADS = PROD_THREADS + 32 + 128;
constexpr int WIN_MAX_SMEM = 232448;
constexpr int WIN_EPI_BUF = 32 * 128;                // one warp's 32 rows x 32 FP32 columns
constexpr int WIN_EPI_SMEM = 4 * WIN_EPI_BUF;        // 4 epilogue warps, one buffer each
constexpr int WIN_BAR_AREA = 256;

struct WinParams {
    int N, C, H, W, K, R, S, P, Q;
    int pt, u, v, dh;
    int pl;           // left padding: phase pixel P starts at input pixel v*P - pl
    int A;            // phase pixels per window (ceil(S / v))
    int D, d_log2;    // bytes per phase pixel and its log2
    int nb, nbw;      // data bytes (v*C elements) and data words of a phase pixel
    int steps;        // MMAs per filter row (32 bytes of window each)
    int Qs, qs_log2, J, segs, PB;
    int strip_px, strip_bytes;
    int groups;       // warp steps per strip: strip_px / (32 / (D/4)), rounded up
    int row_bytes;    // bytes of one input row (x_word)
    int x_raw;        // input rows are bulk-copied to shared memory, then repacked
    int raw_rows;     // input rows one tile spans: (J-1)*u + (R-1)*dh + 1
    const void *wpack;  // the filter slabs, packed by window_pack_filters
    int b_img_bytes;    // their bytes: R*steps*BN rows of 32
    int num_tiles;
    long long xs[4], ws[4], ys[4];
    const void *x;
    const void *w;
    void *y;
    const float *bias;
    float alpha, beta;
    int relu, y_bf16, y_tma;
    int x_word;       // input rows are contiguous 4-byte-aligned runs, phase pixels
                      // start on 4-byte boundaries
    int BN;
    uint32_t idesc, tmem_cols, acc_stride;
    uint64_t a_hi;    // strip descriptor bits other than the start address
    int *err;
    unsigned long long timeout_ns;
};

struct WinTile {
    int n, p0, q0;
};

__device__ __forceinline__ WinTile win_tile(const WinParams &p, int t) {
    WinTile wt;
    const int rest = t / p.segs;
    const int seg = t - rest * p.segs;
    const int n = rest / p.PB;
    wt.p0 = (rest - n * p.PB) * p.J;
    wt.n = n;
    wt.q0 = seg * WBM;
    return wt;
}

// Element eps of a phase pixel (input pixel w0 + eps/C, channel eps%C) of
// input row (n, h), zero outside the row or past v*C.
template <typename T>
__device__ __forceinline__ T phase_elem(const WinParams &p, long long rowoff, int w0, int eps) {
    const T *x = static_cast<const T *>(p.x);
    const int phi = eps / p.C, c = eps - phi * p.C;
    const int wp = w0 + phi;
    const bool in = eps < p.v * p.C && wp >= 0 && wp < p.W;
    const long long off = in ? rowoff + (long long)c * p.xs[1] + (long long)wp * p.xs[3] : 0;
    return in ? __ldg(x + off) : (T)0;
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

template <typename T>
__device__ __forceinline__ uint32_t pack_word(const T (&e)[4 / sizeof(T)]) {
    if constexpr (sizeof(T) == 2)
        return (uint32_t)e[0] | ((uint32_t)e[1] << 16);
    else
        return (uint32_t)e[0];
}

// The filter taps as MMA B operands: slab (r, st) holds BN rows (filters) of
// the 32 window bytes [32*st, 32*st + 32) of filter row r, in the 32-byte
// swizzled K-major layout (row k at 32*k; its two 16-byte halves exchanged
// where address bit 7 is set).  A thread walks the window of one (k, r) pair
// element by element -- phase pixel a, phase phi, channel c, tap s = v*a+phi --
// and writes it a word at a time, sixteen words' loads in flight before their
// stores.
// Barrier of the eight producer warps (id 2) that also ANDs a predicate.
__device__ __forceinline__ bool producers_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 2, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// The filter taps as MMA B operands, packed by a small kernel launched ahead
// of the convolution into device memory, in the exact shared-memory image the
// convolution then bulk-copies: slab (r, st) holds BN rows (filters) of the
// 32 window bytes [32*st, 32*st + 32) of filter row r, 32-byte swizzled K-major
// (row k at 32*k; its two 16-byte halves exchanged where address bit 7 is set,
// which the image reproduces because the slabs start 256-byte aligned).  One
// thread per 4-byte word.
template <typename T>
__global__ void window_pack_filters(const __grid_constant__ WinParams p, uint32_t *img) {
    constexpr int ESZ = (int)sizeof(T), EPW = 4 / ESZ;
    const int words = p.R * p.steps * p.BN * 8;
    const int wi = blockIdx.x * blockDim.x + threadIdx.x;
    if (wi >= words) return;
    const T *w = static_cast<const T *>(p.w);
    const int row = wi >> 3, wd = wi & 7;
    const int sl = row / p.BN, k = row - sl * p.BN;
    const int r = sl / p.steps, st = sl - r * p.steps;
    T e[EPW];
#pragma unroll
    for (int i = 0; i < EPW; ++i) {
        const int b = 32 * st + 4 * wd + i * ESZ;  // byte of the window
        const int a = b / p.D;
        const int eps = (b - a * p.D) / ESZ;        // element of phase pixel a
        const int phi = eps / p.C, c = eps - phi * p.C;
        const int s = p.v * a + phi;
        const bool in = k < p.K && eps < p.v * p.C && s < p.S;
        e[i] = in ? w[(long long)k * p.ws[0] + (long long)c * p.ws[1] + (long long)r * p.ws[2] +
                      (long long)s * p.ws[3]]
                  : (T)0;
    }
    const uint32_t off = (uint32_t)row * 32u + ((((uint32_t)(wd >> 2)) ^ ((uint32_t)(row >> 2) & 1u)) << 4) +
                         ((uint32_t)(wd & 3) << 2);
    img[off >> 2] = pack_word<T>(e);
}

// Packs the R strips of one tile.  Lane l of a warp owns word l % wpp of strip
// pixel l / wpp of each group of 32/wpp consecutive strip pixels (wpp = D/4
// words per phase pixel), so a warp writes 128 contiguous bytes per step; the
// 16-byte chunk of a word is XORed with address bits 7.. of its pixel (the
// swizzle of D-byte rows; none for D = 16).  When the input row is one
// contiguous, 4-byte-aligned byte run (x_word), a phase pixel's data are
// bytes [(v*P - pl)*C, +v*C) of that run and every word is one 4-byte
// cp.async (zero-filled outside the row and in the padding words; the last
// word of a row may be partial).  Otherwise elements are loaded one by one,
// four steps' loads in flight before their stores.
template <typename T>
__device__ void pack_strips(const WinParams &p, uint32_t sbuf, const WinTile &wt, int warp,
                            int lane) {
    constexpr int ESZ = (int)sizeof(T), EPW = 4 / ESZ;
    constexpr uint32_t NONE = 0xffffffffu;
    const int wpp = p.D >> 2;
    const int dp = lane >> (p.d_log2 - 2), wp = lane & (wpp - 1);
    const int G = 32 / wpp;  // strip pixels per warp step
    const int chmask = (p.D >> 4) - 1;
    const int q_need = p.Q + p.A - 1;
    const int total = p.R * p.groups;
    const char *xb = static_cast<const char *>(p.x);
    // strip pixel -> destination word address, input row and phase pixel
    auto decode = [&](int it, uint32_t &dst, long long &rowoff, int &P) -> bool {
        const int r = it / p.groups;
        const int sig = (it - r * p.groups) * G + dp;
        dst = NONE;
        if (sig >= p.strip_px) return false;
        int j;
        bool ok;
        if (p.J > 1) {
            j = sig >> p.qs_log2;
            P = sig & (p.Qs - 1);
            ok = j < p.J && P < q_need;
        } else {
            j = 0;
            P = wt.q0 + sig;
            ok = true;
        }
        const int pr = wt.p0 + j;
        const int h = pr * p.u + r * p.dh - p.pt;
        ok = ok && pr < p.P && h >= 0 && h < p.H && wp < p.nbw;
        const uint32_t paddr = sbuf + (uint32_t)r * p.strip_bytes + (uint32_t)sig * p.D;
        const int byte = wp * 4;
        dst = paddr + ((((uint32_t)(byte >> 4) ^ ((paddr >> 7) & chmask)) << 4) | (uint32_t)(byte & 15));
        rowoff = (long long)wt.n * p.xs[0] + (long long)h * p.xs[2];
        return ok;
    };
    if (p.x_word) {
        // segments (r, j): J per strip, each Qs strip pixels; the last one of a
        // strip also takes the strip's tail pixels (strip_px is a multiple of G)
        const int nseg = p.R * p.J;
        const int lb = p.pl * p.C * ESZ;  // phase pixel P's data start at byte P*nb - lb
        const uint32_t inner = (uint32_t)(wp * 4);
        const int gnb = G * p.nb;          // row bytes advanced per warp step
#pragma unroll 1
        for (int sg = warp; sg < nseg; sg += PROD_THREADS / 32) {
            const int r = sg / p.J, j = sg - r * p.J;
            const int pix0 = p.J > 1 ? j * p.Qs : 0;
            const int nst = ((j == p.J - 1) ? p.strip_px - pix0 : p.Qs) / G;  // warp steps
            const int pr = wt.p0 + j;
            const int h = pr * p.u + r * p.dh - p.pt;
            const int P0 = (p.J > 1 ? 0 : wt.q0) + dp;
            // steps whose word may hold data: the row exists, the word is a data
            // word, and (J > 1) the pixel is one a valid output row reads
            int st_end = 0;
            if (pr < p.P && h >= 0 && h < p.H && wp < p.nbw)
                st_end = p.J > 1 ? max(0, (q_need - P0 + G - 1) / G) : nst;
            const char *rowp = xb + ((long long)wt.n * p.xs[0] + (long long)(h < 0 ? 0 : h) * p.xs[2]) * ESZ;
            int bt = P0 * p.nb - lb + (int)inner;  // byte of the row this lane copies
            uint32_t paddr = sbuf + (uint32_t)r * p.strip_bytes + (uint32_t)(pix0 + dp) * p.D;
#pragma unroll 4
            for (int st = 0; st < nst; ++st) {
                const bool in = st < st_end && (unsigned)bt < (unsigned)p.row_bytes;
                const uint32_t n = in ? (uint32_t)min(p.row_bytes - bt, 4) : 0u;
                const uint32_t dst = paddr + ((((inner >> 4) ^ ((paddr >> 7) & chmask)) << 4) |
                                              (inner & 15u));
                cp_async_4(dst, in ? rowp + bt : xb, n);
                bt += gnb;
                paddr += 128u;  // G pixels of D bytes
            }
        }
        return;
    }
    constexpr int STEPS = 4;
#pragma unroll 1
    for (int it0 = warp; it0 < total; it0 += STEPS * (PROD_THREADS / 32)) {
        uint32_t dst[STEPS];
        T val[STEPS][EPW];
#pragma unroll
        for (int sidx = 0; sidx < STEPS; ++sidx) {
            const int it = it0 + sidx * (PROD_THREADS / 32);
            long long rowoff = 0;
            int P = 0;
            const bool ok = it < total && decode(it, dst[sidx], rowoff, P);
            if (it >= total) dst[sidx] = NONE;
#pragma unroll
            for (int i = 0; i < EPW; ++i)
                val[sidx][i] = ok ? phase_elem<T>(p, rowoff, P * p.v - p.pl, wp * EPW + i) : (T)0;
        }
#pragma unroll
        for (int sidx = 0; sidx < STEPS; ++sidx)
            if (dst[sidx] != NONE) sts32(dst[sidx], pack_word<T>(val[sidx]));
    }
}

// Repacks the R strips of one tile from its input rows staged in shared
// memory at sR (row i = input row p0*u - pt + i, row_bytes each): the same
// lane-to-word mapping as the word copy, four steps' loads before their
// stores.
__device__ void repack_strips(const WinParams &p, uint32_t sbuf, uint32_t sR, const WinTile &wt,
                              int warp, int lane) {
    const int wpp = p.D >> 2;
    const int dp = lane >> (p.d_log2 - 2), wp = lane & (wpp - 1);
    const int G = 32 / wpp;
    const uint32_t chmask = (uint32_t)(p.D >> 4) - 1u;
    const int q_need = p.Q + p.A - 1;
    const int nseg = p.R * p.J;
    const int lb = p.pl * p.C * (p.nb / (p.v * p.C));  // bytes of pl input pixels
    const uint32_t inner = (uint32_t)(wp * 4);
    const int gnb = G * p.nb;
#pragma unroll 1
    for (int sg = warp; sg < nseg; sg += PROD_THREADS / 32) {
        const int r = sg / p.J, j = sg - r * p.J;
        const int pix0 = p.J > 1 ? j * p.Qs : 0;
        const int nst = ((j == p.J - 1) ? p.strip_px - pix0 : p.Qs) / G;
        const int pr = wt.p0 + j;
        const int h = pr * p.u + r * p.dh - p.pt;
        const int P0 = (p.J > 1 ? 0 : wt.q0) + dp;
        int st_end = 0;
        if (pr < p.P && h >= 0 && h < p.H && wp < p.nbw)
            st_end = p.J > 1 ? max(0, (q_need - P0 + G - 1) / G) : nst;
        const uint32_t rb = sR + (uint32_t)(j * p.u + r * p.dh) * (uint32_t)p.row_bytes;
        int bt = P0 * p.nb - lb + (int)inner;
        uint32_t paddr = sbuf + (uint32_t)r * p.strip_bytes + (uint32_t)(pix0 + dp) * p.D;
        for (int st0 = 0; st0 < nst; st0 += 4) {
            uint32_t v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int st = st0 + k, b = bt + k * gnb;
                v[k] = (st < st_end && (unsigned)b < (unsigned)p.row_bytes) ? lds32(rb + b) : 0u;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t pa = paddr + 128u * k;  // G pixels of D bytes per step
                if (st0 + k < nst)
                    sts32(pa + ((((inner >> 4) ^ ((pa >> 7) & chmask)) << 4) | (inner & 15u)), v[k]);
            }
            bt += 4 * gnb;
            paddr += 512u;
        }
    }
}

// Bulk-copies the input rows of tile wt to sR; completes on rawbar.
__device__ void issue_raw_rows(const WinParams &p, uint32_t sR, const WinTile &wt, uint64_t *rawbar,
                               int esz) {
    const int h0 = wt.p0 * p.u - p.pt;
    int valid = 0;
    for (int i = 0; i < p.raw_rows; ++i)
        valid += (h0 + i >= 0 && h0 + i < p.H) ? 1 : 0;
    mbar_arrive_expect_tx(rawbar, (uint32_t)(valid * p.row_bytes));
    const char *xb = static_cast<const char *>(p.x);
    for (int i = 0; i < p.raw_rows; ++i) {
        const int h = h0 + i;
        if (h < 0 || h >= p.H) continue;
        bulk_load_1d(sR + (uint32_t)i * (uint32_t)p.row_bytes,
                     xb + ((long long)wt.n * p.xs[0] + (long long)h * p.xs[2]) * esz,
                     (uint32_t)p.row_bytes, rawbar);
    }
}

template <typename T>
__device__ void win_produce(const WinParams &p, uint32_t sB, uint32_t sS, uint32_t sR,
                            uint64_t *full, uint64_t *empty, uint64_t *bres, uint64_t *rawbar,
                            const WaitCtl &ctl) {
    constexpr int ESZ = (int)sizeof(T);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t raw_bytes = (uint32_t)p.raw_rows * (uint32_t)p.row_bytes;
    volatile int no_abort = 0;
    const WaitCtl drain{&no_abort, p.err, p.timeout_ns};  // waits for copies in flight
    // The packed filter image: one bulk copy, completing on bres (the MMA
    // issuer waits there).  Input rows of the first tile: staging buffer 0.
    int raw_issued = (p.x_raw && (int)blockIdx.x < p.num_tiles) ? 1 : 0, raw_done = 0;
    if (tid == 0) {
        mbar_arrive_expect_tx(bres, (uint32_t)p.b_img_bytes);
        bulk_load_1d(sB, p.wpack, (uint32_t)p.b_img_bytes, bres);
        if (raw_issued) issue_raw_rows(p, sR, win_tile(p, blockIdx.x), &rawbar[0], ESZ);
    }
    int it = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t ph = (uint32_t)(it >> 1) & 1u;
        const uint32_t sbuf = sS + (uint32_t)(buf * p.R) * p.strip_bytes;
        const WinTile wt = win_tile(p, t);
        bool w_ok = mbar_wait(&empty[buf], ph ^ 1u, ctl, 1);
        if (p.x_raw) {
            // staging buffer `buf` holds this tile's rows (copy number it)
            w_ok = w_ok && mbar_wait(&rawbar[buf], ph, ctl, 11);
            if (!producers_and(w_ok)) break;  // every producer leaves together
            ++raw_done;
            // all producers are past the previous tile, so the other staging
            // buffer is free: fetch the next tile's rows while this one is packed
            if (t + (int)gridDim.x < p.num_tiles) {
                ++raw_issued;
                if (tid == 0) {
                    fence_proxy_async_smem();
                    issue_raw_rows(p, sR + (uint32_t)(buf ^ 1) * raw_bytes,
                                   win_tile(p, t + gridDim.x), &rawbar[buf ^ 1], ESZ);
                }
            }
            repack_strips(p, sbuf, sR + (uint32_t)buf * raw_bytes, wt, warp, lane);
            fence_proxy_async_smem();
            mbar_arrive(&full[buf]);
        } else {
            if (!w_ok) break;
            pack_strips<T>(p, sbuf, wt, warp, lane);
            cp_async_commit_wait_all();
            fence_proxy_async_smem();
            mbar_arrive(&full[buf]);
        }
    }
    cp_async_commit_wait_all();  // nothing may land after the CTA exits
    // after an early exit a bulk copy may still be in flight
    if (tid == 0) {
        if (raw_issued > raw_done)
            mbar_wait(&rawbar[raw_done & 1], (uint32_t)(raw_done >> 1) & 1u, drain, 93);
        mbar_wait(bres, 0u, drain, 94);
    }
}

__device__ __forceinline__ bool win_drain(uint64_t *bar, uint32_t parity, const WinParams &p) {
    volatile int dummy = 0;
    WaitCtl c{&dummy, p.err, p.timeout_ns};
    return mbar_wait(bar, parity, c, 90);
}

template <bool TF32>
__device__ void win_mma(const WinParams &p, uint32_t tmem_base, uint32_t sB, uint32_t sS,
                        uint64_t *full, uint64_t *empty, uint64_t *tfull, uint64_t *tempty,
                        uint64_t *mma_done, uint64_t *bres, const WaitCtl &ctl) {
    // 64-bit descriptors advanced in place: the start address (16-byte units)
    // sits in the low bits and stays below 256 KiB, so the additions never
    // carry into other fields.  B slabs: 32-byte swizzle, 8-row groups 256
    // bytes apart.
    const uint64_t b0 = (uint64_t)((sB >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(256 >> 4) << 32) |
                        (1ull << 46) | (6ull << 29 << 32);
    const uint64_t slab16 = (uint64_t)p.BN * 2u;  // slab bytes / 16
    const uint64_t strip16 = (uint64_t)(p.strip_bytes >> 4);
    const int R = p.R, steps = p.steps;
    const uint32_t idesc = p.idesc;
    bool ok = mbar_wait(bres, 0u, ctl, 7);
    int it = 0;
    for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t ph = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait(&tempty[buf], ph ^ 1u, ctl, 3)) break;
        if (!mbar_wait(&full[buf], ph, ctl, 4)) break;
        tc_fence_after_sync();
        const uint32_t d = tmem_base + (uint32_t)buf * p.acc_stride;
        uint64_t a_row = p.a_hi | (uint64_t)(((sS + (uint32_t)(buf * R) * (uint32_t)p.strip_bytes) >> 4) & 0x3FFFu);
        uint64_t bd = b0;
        uint32_t acc = 0;
        for (int r = 0; r < R; ++r, a_row += strip16) {
            uint64_t ad = a_row;
#pragma unroll 4
            for (int st = 0; st < steps; ++st) {  // 32 bytes of window per MMA
                if constexpr (TF32)
                    umma_tf32_nc(d, ad, bd, idesc, acc);
                else
                    umma_bf16_nc(d, ad, bd, idesc, acc);
                acc = 1;
                ad += 2;
                bd += slab16;
            }
        }
        umma_commit(&empty[buf]);  // strip buffer free once these MMAs are done
        umma_commit(&tfull[buf]);  // accumulator ready for the epilogue
    }
    // Every MMA issued must complete before tensor memory is released.
    umma_commit(mma_done);
    win_drain(mma_done, 0u, p);
}

// Row `lane` of a warp's 32 x 32 FP32 staging block, in the 128-byte swizzle
// the y tensor map uses (16-byte chunk j of row l at chunk j ^ (l % 8)).
__device__ __forceinline__ void win_stage_row(uint8_t *buf, int lane, const float (&val)[32]) {
    const uint32_t rowp = smem_u32(buf) + (uint32_t)lane * 128u;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(rowp + (((uint32_t)j ^ (lane & 7)) << 4)),
                     "f"(val[4 * j]), "f"(val[4 * j + 1]), "f"(val[4 * j + 2]), "f"(val[4 * j + 3])
                     : "memory");
}

__device__ __forceinline__ float win_bf16_to_f32(unsigned short b) {
    return __uint_as_float((uint32_t)b << 16);
}

__device__ __forceinline__ unsigned short win_f32_to_bf16(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// alpha * acc + beta * y + bias, then ReLU, for columns k0 .. k0+31 of one row.
__device__ __noinline__ void win_epi_general(const WinParams &p, bool valid, long long ybase, int k0,
                                             float (&val)[32]) {
    const float *yf = static_cast<const float *>(p.y);
    const unsigned short *yb = static_cast<const unsigned short *>(p.y);
    for (int i = 0; i < 32; ++i) {
        const int k = k0 + i;
        float f = val[i];
        if (valid && k < p.K) {
            const long long yo = ybase + (long long)k * p.ys[1];
            if (p.beta != 0.f) f = __fmaf_rn(p.beta, p.y_bf16 ? win_bf16_to_f32(yb[yo]) : yf[yo], f);
            if (p.bias) f += __ldg(p.bias + k);
        }
        if (p.relu) f = fmaxf(f, 0.f);
        val[i] = f;
    }
}

// Direct stores of columns k0 .. k0+31 of one row (any y layout, FP32 or BF16).
__device__ __noinline__ void win_store_direct(const WinParams &p, long long ybase, int k0,
                                              const float (&val)[32]) {
    float *yf = static_cast<float *>(p.y);
    unsigned short *yb = static_cast<unsigned short *>(p.y);
    const long long yo0 = ybase + (long long)k0 * p.ys[1];
    if (p.ys[1] == 1 && !p.y_bf16 && k0 + 32 <= p.K &&
        ((reinterpret_cast<uintptr_t>(yf + yo0) & 15u) == 0)) {
        float4 *dst = reinterpret_cast<float4 *>(yf + yo0);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(val[4 * i], val[4 * i + 1], val[4 * i + 2], val[4 * i + 3]);
        return;
    }
    for (int i = 0; i < 32; ++i) {
        const int k = k0 + i;
        if (k >= p.K) break;
        const long long yo = ybase + (long long)k * p.ys[1];
        if (p.y_bf16)
            yb[yo] = win_f32_to_bf16(val[i]);
        else
            yf[yo] = val[i];
    }
}

__device__ void win_epilogue(const WinParams &p, uint32_t tmem_base, uint64_t *tfull,
                             uint64_t *tempty, uint8_t *epi_smem, const CUtensorMap *tmY,
                             const WaitCtl &ctl) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    const int row = quad * 32 + lane;
    const bool plain = p.beta == 0.f && p.bias == nullptr && !p.relu;
    uint8_t *my_buf = epi_smem + quad * WIN_EPI_BUF;
    const int kend = min(p.BN, ((p.K + 31) / 32) * 32);
    int nbuf = 0;
    int it = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t ph = (uint32_t)(it >> 1) & 1u;
        int okw = 0;
        if (lane == 0) okw = mbar_wait(&tfull[buf], ph, ctl, 5) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) break;
        __syncwarp();
        tc_fence_after_sync();
        const WinTile wt = win_tile(p, t);
        int j, q, qw;
        if (p.J > 1) {
            j = row >> p.qs_log2;
            q = row & (p.Qs - 1);
            qw = (quad * 32) & (p.Qs - 1);
        } else {
            j = 0;
            q = wt.q0 + row;
            qw = wt.q0 + quad * 32;
        }
        const int pr = wt.p0 + j;
        // the same for the whole warp (Qs >= 32): its output row exists and
        // holds at least one of the warp's pixels
        const bool row_in = pr < p.P && qw < p.Q;
        const bool valid = row_in && q < p.Q;
        const long long ybase =
            (long long)wt.n * p.ys[0] + (long long)pr * p.ys[2] + (long long)q * p.ys[3];
        const uint32_t taddr =
            tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)buf * p.acc_stride;
        if (row_in) {
            for (int c0 = 0; c0 < kend; c0 += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(taddr + (uint32_t)c0, v);
                tmem_ld_wait();
                float val[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) val[i] = p.alpha * __uint_as_float(v[i]);
                if (!plain) {  // through memory: the call takes the row by reference
                    float lv[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) lv[i] = val[i];
                    win_epi_general(p, valid, ybase, c0, lv);
#pragma unroll
                    for (int i = 0; i < 32; ++i) val[i] = lv[i];
                }
                if (p.y_tma) {
                    uint8_t *sb = my_buf;
                    if (nbuf >= 1) {  // the previous store has read the buffer
                        if (lane == 0) bulk_wait_group_read<0>();
                        __syncwarp();
                    }
                    win_stage_row(sb, lane, val);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(tmY, sb, c0, qw, wt.n * p.P + pr);
                        bulk_commit_group();
                    }
                    ++nbuf;
                } else if (valid) {
                    float lv[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) lv[i] = val[i];
                    win_store_direct(p, ybase, c0, lv);
                }
            }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
    }
    // staged stores must finish reading shared memory before the CTA exits
    if (p.y_tma && lane == 0) bulk_wait_group_all();
    __syncwarp();
}

template <bool TF32>
__global__ void __launch_bounds__(WIN_THREADS, 1)
    conv_window_kernel(const __grid_constant__ WinParams p, const __grid_constant__ CUtensorMap tmY) {
    using T = typename std::conditional<TF32, uint32_t, uint16_t>::type;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *epi = smem;  // y staging (1024-aligned)
    uint8_t *bptr = epi + (p.y_tma ? WIN_EPI_SMEM : 0);
    const size_t b_bytes = (((size_t)p.R * p.steps * p.BN * 32) + 1023) & ~(size_t)1023;
    uint8_t *sptr = bptr + b_bytes;
    uint8_t *rptr = sptr + (size_t)2 * p.R * p.strip_bytes;  // staged input rows, 2 buffers
    uint64_t *bars = reinterpret_cast<uint64_t *>(
        rptr + (p.x_raw ? (size_t)2 * p.raw_rows * p.row_bytes : 0));
    uint64_t *full = bars;
    uint64_t *empty = bars + 2;
    uint64_t *tfull = bars + 4;
    uint64_t *tempty = bars + 6;
    uint64_t *mma_done = bars + 8;
    uint64_t *bres = bars + 9;
    uint64_t *rawbar = bars + 10;  // two: one per staging buffer
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 12);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full[i], PROD_THREADS);
            mbar_init(&empty[i], 1u);
            mbar_init(&tfull[i], 1u);
            mbar_init(&tempty[i], 4u);
        }
        mbar_init(mma_done, 1u);
        mbar_init(bres, 1u);
        mbar_init(&rawbar[0], 1u);
        mbar_init(&rawbar[1], 1u);
        *abort_flag = 0;
        fence_mbar_init();
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
    const uint32_t sB = smem_u32(bptr), sS = smem_u32(sptr), sR = smem_u32(rptr);

    if (warp < MMA_WARP) {
        win_produce<T>(p, sB, sS, sR, full, empty, bres, rawbar, ctl);
    } else if (warp == MMA_WARP) {
        if (lane == 0)
            win_mma<TF32>(p, tmem_base, sB, sS, full, empty, tfull, tempty, mma_done, bres, ctl);
    } else {
        if (p.y_tma && lane == 0) prefetch_tmap(&tmY);
        win_epilogue(p, tmem_base, tfull, tempty, epi, &tmY, ctl);
    }
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == MMA_WARP) tmem_dealloc(tmem_base, p.tmem_cols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
bool win_math_ok(const ConvProblem &pb) {
    return (pb.math == DLC_MATH_BF16 && pb.xdt == DLC_DATA_BFLOAT16) ||
           (pb.math == DLC_MATH_TF32 && pb.xdt == DLC_DATA_FLOAT);
}

// Fills everything but pointers, error words and the y decision; false when
// the layer does not fit this kernel.
bool window_plan(const ConvProblem &pb, WinParams *wp, size_t *smem_out) {
    if (!win_math_ok(pb)) return false;
    if (pb.dw != 1 || pb.K > 256 || pb.K < 1) return false;
    if (const char *ev = std::getenv("DLC_TC_WINDOW"))
        if (std::atoi(ev) == 0) return false;
    const int e = pb.xdt == DLC_DATA_BFLOAT16 ? 2 : 4;
    const long long nb = (long long)pb.v * pb.C * e;
    int D;
    if (nb <= 16) D = 16;
    else if (nb <= 32) D = 32;
    else if (nb <= 64) D = 64;
    else return false;
    WinParams p;
    std::memset(&p, 0, sizeof(p));
    p.N = pb.N; p.C = pb.C; p.H = pb.H; p.W = pb.W; p.K = pb.K; p.R = pb.R; p.S = pb.S;
    p.P = pb.P; p.Q = pb.Q;
    p.pt = pb.pt; p.u = pb.u; p.v = pb.v; p.dh = pb.dh;
    p.pl = pb.pl;
    p.A = (pb.S + pb.v - 1) / pb.v;
    p.D = D;
    p.d_log2 = D == 16 ? 4 : (D == 32 ? 5 : 6);
    p.nb = (int)nb;
    p.nbw = (int)((nb + 3) / 4);
    p.steps = (p.A * D + 31) / 32;
    const int need = pb.Q + p.A - 1;
    if (need <= 32) p.Qs = 32;
    else if (need <= 64) p.Qs = 64;
    else p.Qs = 128;
    p.qs_log2 = p.Qs == 32 ? 5 : (p.Qs == 64 ? 6 : 7);
    p.J = WBM / p.Qs;
    p.segs = p.J > 1 ? 1 : (pb.Q + WBM - 1) / WBM;
    p.PB = (pb.P + p.J - 1) / p.J;
    // the last MMA step of a row may read past pixel A-1 (16-byte pixels come
    // in pairs); those pixels carry zero weights but must hold finite data
    p.strip_px = WBM - 1 + (p.steps * 32 + D - 1) / D;
    p.strip_px = ((p.strip_px + 128 / D - 1) / (128 / D)) * (128 / D);  // whole warp steps
    const int span = D == 64 ? 512 : 256;
    p.strip_bytes = ((p.strip_px * D + span - 1) / span) * span;
    const int G = 128 / D;
    p.groups = (p.strip_px + G - 1) / G;
    if ((long long)pb.N * p.PB * p.segs > 0x7fffffffLL) return false;
    p.num_tiles = pb.N * p.PB * p.segs;
    p.BN = ((pb.K + 15) / 16) * 16;
    const long long b_bytes = (((long long)pb.R * p.steps * p.BN * 32) + 1023) & ~1023LL;
    const long long strips = 2LL * pb.R * p.strip_bytes;
    if ((long long)pb.R * p.strip_px * 4 > 0x7fffffffLL) return false;
    long long base = 1024 + b_bytes + strips + WIN_BAR_AREA;
    if (base > WIN_MAX_SMEM) return false;
    // Input rows staged whole by bulk copies: channels-innermost (or C == 1)
    // dense rows whose starts and lengths are 16-byte multiples.
    p.raw_rows = (p.J - 1) * pb.u + (pb.R - 1) * pb.dh + 1;
    const long long rowb = (long long)pb.W * pb.C * e;
    const bool rows_dense = (pb.C == 1 && pb.xs[3] == 1) || (pb.xs[1] == 1 && pb.xs[3] == pb.C);
    if (rows_dense && rowb % 16 == 0 && (pb.xs[0] * e) % 16 == 0 && (pb.xs[2] * e) % 16 == 0 &&
        p.raw_rows * rowb < (1LL << 20) && base + 2 * p.raw_rows * rowb <= WIN_MAX_SMEM &&
        ((long long)pb.pl * pb.C * e) % 4 == 0 && nb % 4 == 0) {
        p.x_raw = 1;
        base += 2 * p.raw_rows * rowb;
    }
    // the packed filter image goes through the handle's repacking buffer
    if ((long long)pb.R * p.steps * p.BN * 32 > DLC_WPACK_BYTES) return false;
    if (wp) *wp = p;
    if (smem_out) *smem_out = (size_t)base;
    return true;
}

// y as a 3-D [N*P rows, Q pixels, K columns] FP32 tensor for bulk stores.
bool win_y_tma_ok(const ConvProblem &pb) {
    if (pb.ydt != DLC_DATA_FLOAT || pb.ys[1] != 1) return false;
    const long long pitch = pb.ys[3];
    if (pitch < pb.K || (pitch * 4) % 16 || (pb.ys[2] * 4) % 16) return false;
    if (pb.ys[2] < (long long)pb.Q * pitch) return false;
    if (pb.N > 1 && pb.ys[0] != (long long)pb.P * pb.ys[2]) return false;
    if (pb.y && ((uintptr_t)pb.y % 16)) return false;
    if (pb.ys[2] * 4 >= (1LL << 40)) return false;
    return (long long)pb.N * pb.P <= 0x7fffffffLL;
}

template <bool TF32>
cudaError_t win_launch(const WinParams &p, const CUtensorMap &ty, int grid, size_t smem,
                       cudaStream_t st) {
    auto kern = conv_window_kernel<TF32>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, WIN_THREADS, smem, st>>>(p, ty);
    return cudaGetLastError();
}

}  // namespace

bool dlc_window_ok(const ConvProblem &pb) { return window_plan(pb, nullptr, nullptr); }

dlcStatus_t dlc_launch_window(dlcContext *ctx, const ConvProblem &pb) {
    WinParams p;
    size_t smem = 0;
    if (!window_plan(pb, &p, &smem)) return DLC_STATUS_INTERNAL_ERROR;
    const bool tf32 = pb.math == DLC_MATH_TF32;
    const int e = tf32 ? 4 : 2;
    for (int i = 0; i < 4; ++i) {
        p.xs[i] = pb.xs[i];
        p.ws[i] = pb.ws[i];
        p.ys[i] = pb.ys[i];
    }
    p.x = pb.x; p.w = pb.w; p.y = pb.y; p.bias = pb.bias;
    p.alpha = pb.alpha; p.beta = pb.beta; p.relu = pb.relu;
    p.y_bf16 = pb.ydt == DLC_DATA_BFLOAT16;
    // an input row as one byte run: W pixels of C channels, channels innermost
    // (or C == 1 with W innermost); phase pixel P's data start at byte
    // (v*P - pl)*C*e of the run
    const bool contiguous = (pb.C == 1 && pb.xs[3] == 1) || (pb.xs[1] == 1 && pb.xs[3] == pb.C);
    p.x_word = (contiguous && p.nb % 4 == 0 && ((uintptr_t)pb.x % 4) == 0 &&
                (pb.xs[0] * e) % 4 == 0 && (pb.xs[2] * e) % 4 == 0 &&
                ((long long)pb.pl * pb.C * e) % 4 == 0 && (long long)pb.W * pb.C * e < (1LL << 30))
                   ? 1 : 0;
    p.row_bytes = (int)((long long)pb.W * pb.C * e);
    if (p.x_raw && ((uintptr_t)pb.x % 16) != 0) p.x_raw = 0;  // smem stays reserved
    // Staging whole rows measured slower than the 4-byte copies (the staging
    // needs a producer-wide barrier per tile), so it is opt-in: DLC_TC_WINRAW=1.
    {
        const char *ev = std::getenv("DLC_TC_WINRAW");
        if (!(ev && std::atoi(ev) != 0)) p.x_raw = 0;
    }
    if (!ctx->wpack) return DLC_STATUS_INTERNAL_ERROR;
    p.wpack = ctx->wpack;
    p.b_img_bytes = p.R * p.steps * p.BN * 32;
    p.y_tma = (win_y_tma_ok(pb) && smem + WIN_EPI_SMEM <= (size_t)WIN_MAX_SMEM) ? 1 : 0;
    if (const char *ev = std::getenv("DLC_TC_YTMA")) p.y_tma = p.y_tma && std::atoi(ev) != 0;
    if (p.y_tma) smem += WIN_EPI_SMEM;

    const uint32_t fmt = tf32 ? 2u : 1u;
    p.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(p.BN >> 3) << 17) |
              ((uint32_t)(WBM >> 4) << 24);
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * p.BN)) cols <<= 1;
    p.tmem_cols = cols;
    p.acc_stride = cols / 2;
    // strips: rows D bytes apart, 8-row groups 8*D apart; 16-byte rows use no
    // swizzle and a 16-byte step between the two K halves of an MMA
    if (p.D == 16)
        p.a_hi = ((uint64_t)(16 >> 4) << 16) | ((uint64_t)(128 >> 4) << 32) | (1ull << 46);
    else if (p.D == 32)
        p.a_hi = (1ull << 16) | ((uint64_t)(256 >> 4) << 32) | (1ull << 46) | (6ull << 61);
    else
        p.a_hi = (1ull << 16) | ((uint64_t)(512 >> 4) << 32) | (1ull << 46) | (4ull << 61);
    p.err = ctx->d_err;
    p.timeout_ns = ctx->timeout_ns;

    CUtensorMap ty;
    std::memset(&ty, 0, sizeof(ty));
    if (p.y_tma) {
        const cuuint64_t ydim[3] = {(cuuint64_t)pb.K, (cuuint64_t)pb.Q,
                                    (cuuint64_t)((long long)pb.N * pb.P)};
        const cuuint64_t ystr[2] = {(cuuint64_t)(pb.ys[3] * 4), (cuuint64_t)(pb.ys[2] * 4)};
        const cuuint32_t ybox[3] = {32, 32, 1};
        const cuuint32_t ones[3] = {1, 1, 1};
        CUresult r = ctx->encode_tiled(&ty, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, pb.y, ydim, ystr,
                                       ybox, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return DLC_STATUS_EXECUTION_FAILED;
    }
    {
        const int words = p.R * p.steps * p.BN * 8;
        const int blocks = (words + 255) / 256;
        if (tf32)
            window_pack_filters<uint32_t><<<blocks, 256, 0, ctx->stream>>>(p, static_cast<uint32_t *>(ctx->wpack));
        else
            window_pack_filters<uint16_t><<<blocks, 256, 0, ctx->stream>>>(p, static_cast<uint32_t *>(ctx->wpack));
        if (cudaGetLastError() != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
        ctx->launches += 1;
    }
    int grid = p.num_tiles < ctx->sm_count ? p.num_tiles : ctx->sm_count;
    if (grid < 1) grid = 1;
    cudaError_t err = tf32 ? win_launch<true>(p, ty, grid, smem, ctx->stream)
                           : win_launch<false>(p, ty, grid, smem, ctx->stream);
    if (err != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}
