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
// up to 128 consecutive output pixels straight out of the packed input row.
// Filter taps are reordered to the same (a, phi, c) order once per call by a
// small kernel (into a device buffer the handle owns) and loaded into every
// CTA's shared memory with one bulk copy, where they stay resident.
//
// Tiles: the 128 MMA rows are J output rows of one image (Qs rows each, Qs a
// power of two covering every pixel a stored output reads, J = 128/Qs) or, for
// wide rows (J = 1), 128 consecutive pixels of one output row; tile rows past
// Q read pixels whose value does not matter and are not stored.
//
// Row ring: the phase-pixel rows live in shared memory once per input row, not
// once per filter row.  Input row h = p0*u - pt + i of a tile (i < rows =
// (J-1)*u + (R-1)*dh + 1) goes to ring slot (h mod u, floor(h/u)): the u phases
// of the vertical stride each hold a ring of RS slots, so input rows h and
// h + u -- what output rows j and j+1 of a tile read for one filter row -- sit
// in adjacent slots, and filter row r reads J consecutive slots as one operand
// (J-1 mirror slots after each ring keep a wrapped run contiguous).  A CTA
// walks consecutive tiles of one image, so each tile adds only the J*u input
// rows its predecessor did not hold.
//
// CTA pairs (opt-in, DLC_TC_WINPAIR=1): a cluster of two CTAs shares
// each MMA over M = 256 rows (one tile per CTA, tcgen05 cta_group::2); each CTA
// fills its own ring, at the same offsets as its peer, and holds half of the
// filters.
//
// Roles (one persistent CTA per SM): eight producer warps write the new rows of
// the next tile into the ring.  Where rows are dense, thread 0 first stages
// them in one of two buffers with bulk copies of their 16-byte-aligned
// supersets (a row may start on any element boundary: the repack shifts it by
// its offset), and the warps repack the staged rows into phase pixels with
// shared-memory loads and 16-byte stores; other layouts take 4-byte
// asynchronous copies or element loads.  Padding words, pixels outside the
// image and rows outside it are zeros.  Warp 0 also writes the tile's MMA
// descriptors (one per MMA) into one of two small tables.  One thread issues
// R*steps MMAs (32 bytes of reduction each) per tile into one of four TMEM
// accumulators (two when four would pass 512 columns); four epilogue warps
// read the accumulator, apply alpha, beta*y, bias and ReLU and store y (bulk
// tensor stores of 32x32 blocks when y is dense FP32).  Every wait is bounded
// and records an error word when it runs out.
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
constexpr int WIN_EPI_SMEM = 4 * WIN_EPI_BUF;        // 4 epilogue warps, one buffer each (x2 when
                                                     // two fit: a store overlaps the next staging)
constexpr int WIN_MAX_ROWS = 224;                  // input rows per tile (ring table)
constexpr int WIN_MAX_MMAS = 256;                  // MMAs per tile (descriptor table)
constexpr int WIN_BARS = 192;                      // barriers, TMEM slot, abort flag
// barriers, then the ring table (one word per tile row) and two descriptor
// tables (one word per MMA): sized per problem, as the largest layers need
// every byte of shared memory
__host__ __device__ constexpr int win_bar_area(int rows, int mmas) {
    return (WIN_BARS + 4 * rows + 8 * mmas + 15) / 16 * 16;
}

struct WinParams {
    int N, C, H, W, K, R, S, P, Q;
    int pt, u, v, dh;
    int pl;           // left padding: phase pixel P starts at input pixel v*P - pl
    int A;            // phase pixels per window (ceil(S / v))
    int D, d_log2;    // bytes per phase pixel and its log2
    int nb, nbw;      // data bytes (v*C elements) and data words of a phase pixel
    int steps;        // MMAs per filter row (32 bytes of window each)
    int px_read;      // phase pixels one output's MMAs read: steps*32/D
    int Qs, qs_log2, J, segs, PB;
    int rows;         // input rows one tile spans: (J-1)*u + (R-1)*dh + 1
    int kb_off;       // floor(-pt/u): ring index of a tile's first row, less p0
    int kspan;        // ring indices floor(h/u) one tile's rows span
    int RS, RSJ;      // ring slots per phase, and with the J-1 mirror slots
    int slot_px, slot_bytes;  // phase pixels and bytes of one ring slot
    int disc_wait;    // RS < 2*kspan: a tile that starts a new run of rows waits
                      // for the MMAs of the tile before it
    int ring_bytes;
    int row_bytes;    // bytes of one input row (x_word)
    int x_stage;      // new input rows arrive by one bulk copy per tile into a stage buffer
    int x_shift;      // rows start on any element boundary: the copy takes the 16-byte
                      // aligned superset of the rows and the repack reads them shifted
    int stage_bytes;  // bytes of one of the two stage buffers: rows * row_bytes (+ 32)
    const void *wpack;  // the filter slabs, packed by window_pack_filters
    int b_img_bytes;    // bytes of one CTA's part: R*steps*(BN/ctas) rows of 32
    int pair;           // launched as CTA pairs (cta_group::2, M = 256 per MMA)
    int num_tiles;      // 128-row tiles
    int num_units;      // per-CTA work units: tiles, or pairs of tiles (pair)
    long long xs[4], ws[4], ys[4];
    const void *x;
    const void *w;
    void *y;
    const float *bias;
    float alpha, beta;
    int relu, y_bf16, y_tma;
    int epi_bufs;     // staging buffers per epilogue warp (1 or 2)
    int x_word;       // input rows are contiguous 4-byte-aligned runs, phase pixels
                      // start on 4-byte boundaries
    int BN;
    uint32_t idesc, tmem_cols, acc_stride;
    int nacc_log2;    // TMEM accumulators: 2 or 4
    uint64_t a_hi;    // ring descriptor bits other than the start address
    int *err;
    unsigned long long timeout_ns;
};

struct WinTile {
    int n, p0, q0;
};

__device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((b - 1 - a) / b); }

// Ring table entry of tile row i (input row p0*u - pt + i): the first slot of
// its phase, (i - pt) mod u times RSJ, in the high half and its ring index
// floor((i - pt)/u) - kb_off in the low half.  Both are independent of p0, so
// both CTAs of a pair place their rows alike.
__device__ __forceinline__ uint32_t ring_entry(const WinParams &p, int i) {
    const int a = i - p.pt;
    const int k = floor_div(a, p.u);
    return ((uint32_t)((a - k * p.u) * p.RSJ) << 16) | (uint32_t)(k - p.kb_off);
}
// Ring slot of a row with table entry e for ring base `base`; pos is its
// position in the phase's ring (below RS).
__device__ __forceinline__ int ring_slot(const WinParams &p, uint32_t e, int base, int &pos) {
    pos = base + (int)(e & 0xffffu);
    if (pos >= p.RS) pos -= p.RS;
    return (int)(e >> 16) + pos;
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

// The filter taps as MMA B operands, packed by a small kernel launched ahead
// of the convolution into device memory, in the exact shared-memory image the
// convolution then bulk-copies (for CTA pairs: two images, each with its half
// of the filters, one per CTA): slab (r, st) holds BN rows (filters) of the
// 32 window bytes [32*st, 32*st + 32) of filter row r, 32-byte swizzled K-major
// (row k at 32*k; its two 16-byte halves exchanged where address bit 7 is set,
// which the image reproduces because the slabs start 256-byte aligned).  One
// thread per 4-byte word.
template <typename T>
__global__ void window_pack_filters(const __grid_constant__ WinParams p, uint32_t *img) {
    constexpr int ESZ = (int)sizeof(T), EPW = 4 / ESZ;
    griddep_wait();  // the previous convolution may still read the image
    griddep_launch_dependents();
    const int words = p.R * p.steps * p.BN * 8;
    const int wi = blockIdx.x * blockDim.x + threadIdx.x;
    if (wi >= words) return;
    const T *w = static_cast<const T *>(p.w);
    const int row = wi >> 3, wd = wi & 7;
    const int sl = row / p.BN, k = row - sl * p.BN;
    const int r = sl / p.steps, st = sl - r * p.steps;
    // a pair's CTA `rank` holds filters [rank*BN/2, (rank+1)*BN/2) of every slab
    const int bnc = p.pair ? p.BN / 2 : p.BN;
    const int rank = k / bnc, row_cta = sl * bnc + (k - rank * bnc);
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
    const uint32_t off = (uint32_t)rank * (uint32_t)p.b_img_bytes + (uint32_t)row_cta * 32u +
                         ((((uint32_t)(wd >> 2)) ^ ((uint32_t)(row_cta >> 2) & 1u)) << 4) +
                         ((uint32_t)(wd & 3) << 2);
    img[off >> 2] = pack_word<T>(e);
}

// Writes input rows i in [i0, rows) of one tile into their ring slots (and
// mirror slots), phase pixels [P0, P0 + need) where need covers every pixel a
// stored output reads (P0 = q0 for wide rows, else 0).  The tile's (row, warp
// step) pairs are split into eight equal ranges, one per producer warp.  Lane
// l owns word l % wpp of pixel l / wpp of each step's 32/wpp consecutive
// pixels (wpp = D/4 words per phase pixel), so a warp writes 128 contiguous
// bytes per step; the 16-byte chunk of a word is XORed with address bits 7..
// of its pixel (the swizzle of D-byte rows; none for D = 16).  When the input
// row is one contiguous, 4-byte-aligned byte run (x_word), a phase pixel's
// data are bytes [(v*P - pl)*C, +v*C) of that run and every word is one
// 4-byte cp.async (zero-filled outside the row, in the padding words and for
// rows outside the image; the last word of a row may be partial).  Otherwise
// elements are loaded one by one, four steps' loads in flight before their
// stores.
template <typename T>
__device__ void pack_rows(const WinParams &p, uint32_t ring, const uint32_t *rtab, const WinTile &wt,
                          int base, int i0, int warp, int lane) {
    constexpr int ESZ = (int)sizeof(T), EPW = 4 / ESZ;
    constexpr int NW = PROD_THREADS / 32;
    const int wpp = p.D >> 2;
    const int dp = lane >> (p.d_log2 - 2), wp = lane & (wpp - 1);
    const int G = 32 / wpp;  // pixels per warp step
    const uint32_t chmask = (uint32_t)(p.D >> 4) - 1u;
    const int P0 = p.J > 1 ? 0 : wt.q0;
    const int need = min(p.slot_px, (p.J > 1 ? p.Q : p.Q - wt.q0) - 1 + p.px_read);
    const int spr = (need + G - 1) / G;  // warp steps per row
    const int total = (p.rows - i0) * spr;
    const int lo = (int)(((long long)total * warp) / NW);
    const int hi = (int)(((long long)total * (warp + 1)) / NW);
    const uint32_t inner = (uint32_t)(wp * 4);
    const uint32_t mdelta = (uint32_t)p.RS * (uint32_t)p.slot_bytes;  // slot -> its mirror
    const char *xb = static_cast<const char *>(p.x);
    const int lb = p.pl * p.C * ESZ;  // phase pixel P's data start at byte P*nb - lb
    int ri = lo / spr, st0 = lo - (lo / spr) * spr;  // the warp's first (row, step)
#pragma unroll 1
    for (int item = lo; item < hi; ++ri, st0 = 0) {
        const int st1 = min(spr, st0 + (hi - item));
        item += st1 - st0;
        const int i = i0 + ri;
        const int h = wt.p0 * p.u - p.pt + i;
        const bool row_ok = h >= 0 && h < p.H;  // rows outside the image are zeros
        int pos;
        const int slot = ring_slot(p, rtab[i], base, pos);
        const bool mirror = pos < p.J - 1;
        uint32_t paddr = ring + (uint32_t)slot * (uint32_t)p.slot_bytes + (uint32_t)(st0 * G + dp) * p.D;
        if (p.x_word) {
            const char *rowp = xb + ((long long)wt.n * p.xs[0] + (long long)(row_ok ? h : 0) * p.xs[2]) * ESZ;
            int bt = (P0 + st0 * G + dp) * p.nb - lb + (int)inner;  // byte of the row this lane copies
            // padding words and rows outside the image copy nothing (zero fill)
            const int lim = (row_ok && wp < p.nbw) ? p.row_bytes : 0;
            const int gnb = G * p.nb;
            // slots start on a swizzle period, so step st's chunk XOR is st & chmask
#pragma unroll 4
            for (int st = st0; st < st1; ++st) {
                const int rem = lim - bt;
                const bool in = bt >= 0 && rem > 0;
                const uint32_t n = in ? (uint32_t)min(rem, 4) : 0u;
                const uint32_t dst = paddr + (inner ^ (((uint32_t)st & chmask) << 4));
                const char *src = in ? rowp + bt : xb;
                cp_async_4(dst, src, n);
                if (mirror) cp_async_4(dst + mdelta, src, n);
                bt += gnb;
                paddr += 128u;
            }
            continue;
        }
        const long long rowoff = (long long)wt.n * p.xs[0] + (long long)(row_ok ? h : 0) * p.xs[2];
        int w0 = (P0 + st0 * G + dp) * p.v - p.pl;  // first input pixel of this lane's phase pixel
        const int eps0 = wp * EPW;
#pragma unroll 1
        for (int st = st0; st < st1; st += 4) {
            T val[4][EPW];
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int e = 0; e < EPW; ++e)
                    val[k][e] = (row_ok && st + k < st1) ? phase_elem<T>(p, rowoff, w0 + k * G * p.v, eps0 + e) : (T)0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (st + k >= st1) break;
                const uint32_t dst = paddr + 128u * k + (inner ^ (((uint32_t)(st + k) & chmask) << 4));
                const uint32_t word = pack_word<T>(val[k]);
                sts32(dst, word);
                if (mirror) sts32(dst + mdelta, word);
            }
            w0 += 4 * G * p.v;
            paddr += 512u;
        }
    }
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts128v(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// The in-image part of a tile's new rows i in [i0, rows): stage rows lo ..
// lo + n - 1 (relative to i0), starting at byte src of x.
__device__ __forceinline__ void stage_span(const WinParams &p, const WinTile &wt, int i0, int esz,
                                           int &lo, int &n, long long &src) {
    const int h0 = wt.p0 * p.u - p.pt + i0;
    lo = max(0, -h0);
    n = max(0, min(p.rows - i0, p.H - h0) - lo);
    src = ((long long)wt.n * p.xs[0] + (long long)(h0 + lo) * p.xs[2]) * esz;
}

// Bulk-copies the new rows of a tile -- tile rows i in [i0, rows), input rows
// p0*u - pt + i -- that lie inside the image into stage buffer `sbuf` (stage
// row i - i0; dense rows are consecutive in x, so one copy), completing on
// `bar`.  With x_shift the rows need not start on 16-byte boundaries: the copy
// takes the 16-byte-aligned superset of their bytes to the buffer's start,
// and stage row i - i0 begins (start mod 16) + (i - i0 - lo) * row_bytes bytes
// in.  A tile past the last one (a pair's missing second tile) copies
// nothing but still completes the barrier's phase.
__device__ void stage_rows(const WinParams &p, uint32_t sbuf, const WinTile &wt, bool valid, int i0,
                           uint64_t *bar, int esz) {
    int lo = 0, n = 0;
    long long src = 0;
    if (valid) stage_span(p, wt, i0, esz, lo, n, src);
    const char *g = static_cast<const char *>(p.x) + src;
    uint32_t bytes = (uint32_t)n * (uint32_t)p.row_bytes;
    uint32_t dst = sbuf + (uint32_t)lo * (uint32_t)p.row_bytes;
    if (p.x_shift && n > 0) {
        const uint32_t shift = (uint32_t)(reinterpret_cast<uintptr_t>(g) & 15u);
        g -= shift;
        bytes = (shift + bytes + 15u) & ~15u;
        dst = sbuf;
    }
    mbar_arrive_expect_tx(bar, n > 0 ? bytes : 0u);
    if (n > 0) bulk_load_1d(dst, g, bytes, bar);
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr);

// Bytes [b, b+4) of a staged row at shared address rb (even; rows of 2-byte
// elements may start 2 bytes past a word), zero outside [0, rowb).
__device__ __forceinline__ uint32_t row_word(uint32_t rb, int b, uint32_t rowb) {
    const uint32_t a = rb + (uint32_t)b;
    if (b >= 0 && (uint32_t)b + 4u <= rowb) {
        if ((a & 3u) == 0) return lds32(a);
        return __funnelshift_r(lds32(a - 2u), lds32(a + 2u), 16);
    }
    const uint32_t lo = (b >= 0 && (uint32_t)b < rowb) ? lds16(a) : 0u;
    const uint32_t hi = (b + 2 >= 0 && (uint32_t)(b + 2) < rowb) ? lds16(a + 2u) : 0u;
    return lo | (hi << 16);
}

// Packs a tile's new rows from the stage buffer into their ring slots (and
// mirror slots), the pixels pack_rows covers.  Lane l builds 16-byte chunk
// l % (D/16) of pixel l / (D/16) of each step's 512/D pixels: up to four
// 4-byte loads from the staged row (zeros outside the row, past the data and
// for rows outside the image) and one 16-byte store, its chunk XORed with
// address bits 7.. (a step spans whole swizzle periods, so the XOR depends on
// the lane only).  Two steps' loads are in flight before their stores.
template <bool SHIFT>
__device__ void repack_rows(const WinParams &p, uint32_t ring, uint32_t sbuf, const uint32_t *rtab,
                            const WinTile &wt, int base, int i0, int warp, int lane) {
    constexpr int NW = PROD_THREADS / 32;
    const int chl = p.d_log2 - 4;  // log2 of 16-byte chunks per phase pixel
    const int kap = lane & ((1 << chl) - 1);
    const int dp = lane >> chl;
    const int G = 32 >> chl;       // pixels per warp step
    const uint32_t chmask = (uint32_t)(p.D >> 4) - 1u;
    const uint32_t cho = (((uint32_t)kap ^ (((uint32_t)(dp * p.D) >> 7) & chmask)) << 4);
    const int P0 = p.J > 1 ? 0 : wt.q0;
    const int need = min(p.slot_px, (p.J > 1 ? p.Q : p.Q - wt.q0) - 1 + p.px_read);
    const int spr = (need + G - 1) / G;
    const int total = (p.rows - i0) * spr;
    const int lo = (int)(((long long)total * warp) / NW);
    const int hi = (int)(((long long)total * (warp + 1)) / NW);
    const int esz = p.nb / (p.v * p.C);
    const int lb = p.pl * p.C * esz;
    const int b0 = kap * 16;                              // first byte of the chunk in its pixel
    const int nwords = max(0, min(4, (p.nb - b0) >> 2));  // data words of the chunk
    const uint32_t rowb = (uint32_t)p.row_bytes;
    const uint32_t mdelta = (uint32_t)p.RS * (uint32_t)p.slot_bytes;
    const int gnb = G * p.nb;
    // x_shift: stage row ri begins at sbuf + adj + ri*rowb (see stage_rows)
    int adj = 0;
    if (SHIFT) {
        int slo, sn;
        long long src;
        stage_span(p, wt, i0, esz, slo, sn, src);
        const int shift = (int)(reinterpret_cast<uintptr_t>(static_cast<const char *>(p.x) + src) & 15u);
        adj = shift - slo * p.row_bytes;
    }
    int ri = lo / spr, st0 = lo - (lo / spr) * spr;  // the warp's first (row, step)
#pragma unroll 1
    for (int item = lo; item < hi; ++ri, st0 = 0) {
        const int st1 = min(spr, st0 + (hi - item));
        item += st1 - st0;
        const int i = i0 + ri;
        const int h = wt.p0 * p.u - p.pt + i;
        const int nw = (h >= 0 && h < p.H) ? nwords : 0;  // rows outside the image are zeros
        int pos;
        const int slot = ring_slot(p, rtab[i], base, pos);
        const bool mirror = pos < p.J - 1;
        const uint32_t rb = sbuf + (uint32_t)(adj + ri * (int)rowb);
        int bt = (P0 + st0 * G + dp) * p.nb - lb + b0;
        uint32_t paddr = ring + (uint32_t)slot * (uint32_t)p.slot_bytes + (uint32_t)(st0 * G + dp) * p.D + cho;
        for (int st = st0; st < st1; st += 2) {
            uint32_t v[2][4];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int b = bt + k * gnb;
#pragma unroll
                for (int w = 0; w < 4; ++w) v[k][w] = 0u;
                if (st + k >= st1) continue;
                if constexpr (SHIFT) {
                    if (nw > 0 && b >= 0 && (uint32_t)b + 4u * (uint32_t)nw <= rowb) {
                        // the chunk's nw data words inside the row: aligned words,
                        // or one more and a 16-bit shift when the row starts 2
                        // bytes past a word (nw is the same for every step of
                        // this lane)
                        const uint32_t a = rb + (uint32_t)b;
                        if ((a & 3u) == 0) {
#pragma unroll
                            for (int w = 0; w < 4; ++w) v[k][w] = w < nw ? lds32(a + 4u * w) : 0u;
                        } else {
                            uint32_t t[5];
#pragma unroll
                            for (int w = 0; w < 5; ++w) t[w] = w <= nw ? lds32(a - 2u + 4u * w) : 0u;
#pragma unroll
                            for (int w = 0; w < 4; ++w) v[k][w] = w < nw ? __funnelshift_r(t[w], t[w + 1], 16) : 0u;
                        }
                    } else {
#pragma unroll
                        for (int w = 0; w < 4; ++w)
                            if (w < nw) v[k][w] = row_word(rb, b + 4 * w, rowb);
                    }
                } else {
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        v[k][w] = (w < nw && (unsigned)(b + 4 * w) < rowb) ? lds32(rb + b + 4 * w) : 0u;
                }
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                // a step may run past the slot's last pixel (wide rows): skip those
                if (st + k >= st1 || (st + k) * G + dp >= p.slot_px) break;
                const uint32_t dst = paddr + 512u * k;
                sts128v(dst, v[k][0], v[k][1], v[k][2], v[k][3]);
                if (mirror) sts128v(dst + mdelta, v[k][0], v[k][1], v[k][2], v[k][3]);
            }
            bt += 2 * gnb;
            paddr += 1024u;
        }
    }
}

// A CTA (or CTA pair) takes the contiguous units [ub, ue); unit u is tile u,
// or for a pair tile u (leader) and tile u + num_units (peer).
template <bool PAIR>
__device__ __forceinline__ void unit_range(const WinParams &p, int &ub, int &ue) {
    const long long c = PAIR ? (long long)cluster_id_x() : (long long)blockIdx.x;
    const long long g = PAIR ? (long long)num_clusters_x() : (long long)gridDim.x;
    ub = (int)((p.num_units * c) / g);
    ue = (int)((p.num_units * (c + 1)) / g);
}
template <bool PAIR>
__device__ __forceinline__ int tile_of(const WinParams &p, int u, uint32_t rank) {
    return (PAIR && rank) ? u + p.num_units : u;
}
// Walks a CTA's units [ub, ue).  Unit u continues unit u-1 when, for every
// CTA of the pair, it holds the next J output rows of the same image and
// segment; its ring base then moves J slots (only the last J*u rows of the
// tile are new), else kspan slots (every row is new).  The walk also keeps
// the coordinates of this CTA's tile (rank 1 of a pair: tile u + num_units),
// so no role divides per tile.  Tile t is image t / (segs*PB), segment
// (t / PB) % segs, output rows (t % PB)*J ..: the row blocks of one (image,
// segment) are consecutive, so a CTA moves down one image J rows at a time.
template <bool PAIR>
struct UnitWalk {
    int pbL, pbP, base;
    int n, seg, valid;  // this CTA's tile: image, segment, exists
    __device__ UnitWalk(const WinParams &p, int ub, uint32_t rank)
        : pbL(ub % p.PB), pbP((ub + p.num_units) % p.PB), base(0) {
        const int t = tile_of<PAIR>(p, ub, rank);
        const int rest = t / p.PB;
        n = rest / p.segs;
        seg = rest - n * p.segs;
        valid = t < p.num_tiles;
        own_rank = (int)rank;
    }
    int own_rank;
    // to unit u = (previous unit) + 1; whether u continues the previous unit
    __device__ __forceinline__ bool next(const WinParams &p, int u) {
        if (++pbL == p.PB) pbL = 0;
        if (++pbP == p.PB) pbP = 0;
        if ((PAIR && own_rank ? pbP : pbL) == 0 && ++seg == p.segs) {
            seg = 0;
            ++n;
        }
        if (PAIR && own_rank) valid = u + p.num_units < p.num_tiles;
        const bool cont = pbL != 0 && (!PAIR || u + p.num_units >= p.num_tiles || pbP != 0);
        base += cont ? p.J : p.kspan;
        if (base >= p.RS) base -= p.RS;
        return cont;
    }
    __device__ __forceinline__ WinTile tile(const WinParams &p) const {
        WinTile wt;
        wt.n = n;
        wt.q0 = seg * WBM;
        wt.p0 = (PAIR && own_rank ? pbP : pbL) * p.J;
        return wt;
    }
};

template <typename T, bool PAIR>
__device__ void win_produce(const WinParams &p, uint32_t rank, uint32_t sB, uint32_t sRing,
                            uint32_t sStage, const uint32_t *rtab, uint32_t *atab, uint64_t *full, uint64_t *empty,
                            uint64_t *bres, uint64_t *bpeer, uint64_t *sfull, const WaitCtl &ctl) {
    constexpr int ESZ = (int)sizeof(T);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t full_l = PAIR ? mapa_shared(smem_u32(full), 0) : smem_u32(full);  // leader's
    volatile int no_abort = 0;
    const WaitCtl drain{&no_abort, p.err, p.timeout_ns};  // waits for copies in flight
    const uint32_t slot16 = (uint32_t)p.slot_bytes >> 4;
    const uint32_t a_lo0 = (uint32_t)p.a_hi + ((sRing >> 4) & 0x3FFFu);  // descriptor low word of slot 0
    int ub, ue;
    unit_range<PAIR>(p, ub, ue);
    // this CTA's part of the packed filter image: one bulk copy on bres
    if (tid == 0) {
        mbar_arrive_expect_tx(bres, (uint32_t)p.b_img_bytes);
        bulk_load_1d(sB, static_cast<const char *>(p.wpack) + (size_t)rank * p.b_img_bytes,
                     (uint32_t)p.b_img_bytes, bres);
    }
    if (PAIR && rank == 1 && tid == 0) {  // the leader's MMAs read this CTA's filters too
        if (mbar_wait(bres, 0u, ctl, 12)) mbar_arrive_cluster(mapa_shared(smem_u32(bpeer), 0));
    }
    // Pixels past `need` and the tail after the last slot are read only by
    // tile rows that are not stored: zero them once so they hold finite data.
    for (uint32_t i = (uint32_t)tid; i < (uint32_t)p.ring_bytes / 16u; i += PROD_THREADS)
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(sRing + 16u * i), "r"(0u) : "memory");
    asm volatile("bar.sync 1, %0;" ::"n"(PROD_THREADS) : "memory");  // producer warps only
    // Staged rows: the rows of unit u + 1 are copied while unit u is packed.
    int staged = 0;  // stage copies issued (thread 0)
    UnitWalk<PAIR> walk(p, ub, rank);
    if (p.x_stage && tid == 0 && ub < ue) {
        stage_rows(p, sStage, walk.tile(p), walk.valid, 0, &sfull[0], ESZ);
        staged = 1;
    }
    int it = 0;
    for (int u = ub; u < ue; ++u, ++it) {
        const bool cont = u > ub && walk.next(p, u);
        const int i0 = cont ? max(0, p.rows - p.J * p.u) : 0;
        const int buf = it & 1;
        const uint32_t ph = (uint32_t)(it >> 1) & 1u;
        bool ok = mbar_wait(&empty[buf], ph ^ 1u, ctl, 1);
        // a short ring: the previous tile's rows must be free before a new run overwrites them
        if (ok && !cont && p.disc_wait && it >= 1)
            ok = mbar_wait(&empty[(it - 1) & 1], (uint32_t)((it - 1) >> 1) & 1u, ctl, 15);
        if (p.x_stage) {
            ok = ok && mbar_wait(&sfull[buf], ph, ctl, 16);
            // every producer is past unit u - 1, whose stage buffer the next
            // copy overwrites; the decision to go on is the same for all
            int stop = (!ok || *ctl.abort_flag) ? 1 : 0;
            asm volatile("{\n\t.reg .pred q, r;\n\tsetp.ne.b32 q, %1, 0;\n\t"
                         "bar.red.or.pred r, 1, %2, q;\n\tselp.b32 %0, 1, 0, r;\n\t}\n"
                         : "=r"(stop) : "r"(stop), "n"(PROD_THREADS) : "memory");
            if (stop) break;
            if (tid == 0 && u + 1 < ue) {
                fence_proxy_async_smem();  // the reads of unit u - 1 before the copy's writes
                UnitWalk<PAIR> nx = walk;
                const bool c1 = nx.next(p, u + 1);
                stage_rows(p, sStage + (uint32_t)((it + 1) & 1) * (uint32_t)p.stage_bytes, nx.tile(p),
                           nx.valid, c1 ? max(0, p.rows - p.J * p.u) : 0, &sfull[(it + 1) & 1], ESZ);
                ++staged;
            }
            if (walk.valid) {
                if (p.x_shift)
                    repack_rows<true>(p, sRing, sStage + (uint32_t)buf * (uint32_t)p.stage_bytes, rtab,
                                      walk.tile(p), walk.base, i0, warp, lane);
                else
                    repack_rows<false>(p, sRing, sStage + (uint32_t)buf * (uint32_t)p.stage_bytes, rtab,
                                       walk.tile(p), walk.base, i0, warp, lane);
            }
        } else {
            if (!ok) break;
            if (walk.valid) pack_rows<T>(p, sRing, rtab, walk.tile(p), walk.base, i0, warp, lane);
        }
        if (warp == 0) {
            // the unit's MMA operands for the MMA warp: MMA (r, st) reads the J
            // slots from tile row r*dh's slot on, 32*st bytes into each window
            uint32_t *tab = atab + buf * p.R * p.steps;
            for (int r = lane; r < p.R; r += 32) {
                int pos;
                const int slot = ring_slot(p, rtab[r * p.dh], walk.base, pos);
                const uint32_t a = a_lo0 + (uint32_t)slot * slot16;  // below 256 KiB
                for (int st = 0; st < p.steps; ++st) tab[r * p.steps + st] = a + 2u * (uint32_t)st;
            }
        }
        cp_async_commit_wait_all();
        fence_proxy_async_smem();
        if (PAIR)
            mbar_arrive_cluster(full_l + 8u * buf);  // every producer thread of both CTAs
        else
            mbar_arrive(&full[buf]);
    }
    cp_async_commit_wait_all();  // nothing may land after the CTA exits
    if (tid == 0) {
        // after an early exit the filter copy and a stage copy may be in flight
        mbar_wait(bres, 0u, drain, 94);
        for (int j = it; j < staged; ++j) mbar_wait(&sfull[j & 1], (uint32_t)(j >> 1) & 1u, drain, 95);
    }
}

__device__ __forceinline__ bool win_drain(uint64_t *bar, uint32_t parity, const WinParams &p) {
    volatile int dummy = 0;
    WaitCtl c{&dummy, p.err, p.timeout_ns};
    return mbar_wait(bar, parity, c, 90);
}

// A wait by lane 0 whose outcome the whole warp takes.
template <bool CLUSTER>
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const WaitCtl &ctl, int code) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0)
        ok = (CLUSTER ? mbar_wait_cluster(bar, parity, ctl, code) : mbar_wait(bar, parity, ctl, code)) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

template <bool TF32, bool PAIR>
__device__ void win_mma(const WinParams &p, uint32_t tmem_base, uint32_t sB, const uint32_t *atab,
                        uint64_t *full, uint64_t *empty,
                        uint64_t *tfull, uint64_t *tempty, uint64_t *mma_done, uint64_t *bres,
                        uint64_t *bpeer, const WaitCtl &ctl) {
    // B slabs: 32-byte swizzle, 8-row groups 256 bytes apart, BN/2 rows per
    // CTA for a pair; the descriptor advances in place (its start address, in
    // 16-byte units, stays below 256 KiB and never carries into other fields).
    const int lane = threadIdx.x & 31;
    const uint64_t b0 = (uint64_t)((sB >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(256 >> 4) << 32) |
                        (1ull << 46) | (6ull << 29 << 32);
    const uint64_t slab16 = (uint64_t)(PAIR ? p.BN / 2 : p.BN) * 2u;  // slab bytes / 16
    const int nm = p.R * p.steps;
    const uint32_t idesc = p.idesc;
    const uint64_t a_hi = p.a_hi & 0xFFFFFFFF00000000ull;
    bool ok = warp_wait<false>(bres, 0u, ctl, 7);
    if (PAIR) ok = ok && warp_wait<true>(bpeer, 0u, ctl, 13);
    int ub, ue;
    unit_range<PAIR>(p, ub, ue);
    // MMAs m0 .. m1-1 of a unit: 32 bytes of window each
    auto issue = [&](uint32_t d, const uint32_t *tab, uint64_t &bd, int m0, int m1) {
#pragma unroll 4
        for (int m = m0; m < m1; ++m) {
            const uint64_t ad = a_hi | tab[m];
            const uint32_t acc = m > 0 ? 1u : 0u;
            if constexpr (PAIR) {
                if constexpr (TF32)
                    umma_tf32_pair(d, ad, bd, idesc, acc);
                else
                    umma_bf16_pair(d, ad, bd, idesc, acc);
            } else {
                if constexpr (TF32)
                    umma_tf32_nc(d, ad, bd, idesc, acc);
                else
                    umma_bf16_nc(d, ad, bd, idesc, acc);
            }
            bd += slab16;
        }
    };
    // (pairs: the other CTA's epilogue and producers arrive remotely)
    auto wait = [&](uint64_t *bar, uint32_t parity, int where) {
        return PAIR ? mbar_wait_cluster(bar, parity, ctl, where) : mbar_wait(bar, parity, ctl, where);
    };
    auto done = [&](uint64_t *bar, uint32_t parity) {
        return PAIR ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity);
    };
    // One lane runs the loop.  While a unit's last MMAs are still queued on
    // the tensor pipe it looks, without waiting, whether the next unit's
    // accumulator and ring rows are ready: if so the next unit's MMAs follow
    // the commits with no wait in between.
    if (lane == 0 && ok) {
        const int head = nm > 4 ? nm - 4 : 0;  // MMAs issued before the look-ahead
        const int amask = (1 << p.nacc_log2) - 1;
        bool ready = false;
        int it = 0;
        for (int u = ub; u < ue; ++u, ++it) {
            const int buf = it & 1;
            const int abuf = it & amask;  // accumulator
            if (!ready) {
                if (!wait(&tempty[abuf], ((uint32_t)(it >> p.nacc_log2) & 1u) ^ 1u, 3)) break;
                if (!wait(&full[buf], (uint32_t)(it >> 1) & 1u, 4)) break;
            }
            tc_fence_after_sync();
            const uint32_t d = tmem_base + (uint32_t)abuf * p.acc_stride;
            const uint32_t *tab = atab + buf * nm;  // written by the producers
            uint64_t bd = b0;
            issue(d, tab, bd, 0, head);
            const int in = it + 1;
            ready = u + 1 < ue && done(&tempty[in & amask], ((uint32_t)(in >> p.nacc_log2) & 1u) ^ 1u) &&
                    done(&full[in & 1], (uint32_t)(in >> 1) & 1u);
            issue(d, tab, bd, head, nm);
            if (PAIR) {
                umma_commit_pair(&empty[buf], 3);  // both CTAs' rings may take new rows
                umma_commit_pair(&tfull[abuf], 3);  // both CTAs' accumulator rows ready
            } else {
                umma_commit(&empty[buf]);
                umma_commit(&tfull[abuf]);
            }
        }
    }
    __syncwarp();
    // Every MMA issued must complete before tensor memory is released.
    if (lane == 0) {
        if (PAIR)
            umma_commit_pair(mma_done, 3);
        else
            umma_commit(mma_done);
    }
    __syncwarp();
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

template <bool PAIR>
__device__ void win_epilogue(const WinParams &p, uint32_t rank, uint32_t tmem_base, uint64_t *tfull,
                             uint64_t *tempty, uint8_t *epi_smem, const CUtensorMap *tmY,
                             const WaitCtl &ctl) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    const int row = quad * 32 + lane;
    const bool plain = p.beta == 0.f && p.bias == nullptr && !p.relu;
    uint8_t *my_buf = epi_smem + quad * p.epi_bufs * WIN_EPI_BUF;
    const int kend = min(p.BN, ((p.K + 31) / 32) * 32);
    const uint32_t tempty_l = PAIR ? mapa_shared(smem_u32(tempty), 0) : smem_u32(tempty);
    int nbuf = 0;
    int it = 0;
    int ub, ue;
    unit_range<PAIR>(p, ub, ue);
    UnitWalk<PAIR> walk(p, ub, rank);
    for (int u = ub; u < ue; ++u, ++it) {
        if (u > ub) walk.next(p, u);
        const int buf = it & ((1 << p.nacc_log2) - 1);  // accumulator
        const uint32_t ph = (uint32_t)(it >> p.nacc_log2) & 1u;
        int okw = 0;
        if (lane == 0) okw = mbar_wait(&tfull[buf], ph, ctl, 5) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) break;
        __syncwarp();
        tc_fence_after_sync();
        const bool have = walk.valid;  // a pair's second tile may not exist
        const WinTile wt = walk.tile(p);
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
        const bool row_in = have && pr < p.P && qw < p.Q;
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
                    uint8_t *sb = my_buf + (p.epi_bufs == 2 ? (nbuf & 1) * WIN_EPI_BUF : 0);
                    // the store that last used this buffer has read it
                    if (nbuf >= p.epi_bufs) {
                        if (lane == 0) {
                            if (p.epi_bufs == 2)
                                bulk_wait_group_read<1>();
                            else
                                bulk_wait_group_read<0>();
                        }
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
        if (lane == 0) {
            if (PAIR)
                mbar_arrive_tmem_free(tempty_l + 8u * buf);  // released on the leader
            else
                mbar_arrive(&tempty[buf]);
        }
    }
    // staged stores must finish reading shared memory before the CTA exits
    if (p.y_tma && lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
}

template <bool TF32, bool PAIR>
__global__ void __launch_bounds__(WIN_THREADS, 1)
    conv_window_kernel(const __grid_constant__ WinParams p, const __grid_constant__ CUtensorMap tmY) {
    using T = typename std::conditional<TF32, uint32_t, uint16_t>::type;
    griddep_launch_dependents();  // the next grid may claim SMs this one leaves
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);  // same offset in both CTAs
    uint8_t *epi = smem;  // y staging (1024-aligned)
    uint8_t *bptr = epi + (p.y_tma ? p.epi_bufs * WIN_EPI_SMEM : 0);
    const size_t b_bytes = ((size_t)p.b_img_bytes + 1023) & ~(size_t)1023;
    uint8_t *ring = bptr + b_bytes;
    uint8_t *stage = ring + p.ring_bytes;  // two stage buffers (x_stage)
    uint64_t *bars = reinterpret_cast<uint64_t *>(stage + (p.x_stage ? 2 * (size_t)p.stage_bytes : 0));
    uint64_t *full = bars;
    uint64_t *empty = bars + 2;
    uint64_t *tfull = bars + 4;   // four: an accumulator is ready
    uint64_t *tempty = bars + 8;  // four: an accumulator is free
    uint64_t *mma_done = bars + 12;
    uint64_t *bres = bars + 13;
    uint64_t *bpeer = bars + 14;
    uint64_t *sfull = bars + 15;  // two: a stage buffer's rows landed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 17);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    uint32_t *rtab = reinterpret_cast<uint32_t *>(bars + 24);  // ring table, one entry per tile row
    uint32_t *atab = rtab + p.rows;  // two tables of a unit's A descriptors, one entry per MMA

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full[i], PAIR ? 2u * PROD_THREADS : PROD_THREADS);  // every producer
            mbar_init(&empty[i], 1u);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&tfull[i], 1u);
            mbar_init(&tempty[i], PAIR ? 8u : 4u);  // the epilogue warps (of both CTAs)
        }
        mbar_init(mma_done, 1u);
        mbar_init(bres, 1u);
        mbar_init(bpeer, 1u);
        mbar_init(&sfull[0], 1u);
        mbar_init(&sfull[1], 1u);
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < p.rows; i += WIN_THREADS) rtab[i] = ring_entry(p, i);
    if (warp == MMA_WARP) {
        if (PAIR) {
            tmem_alloc_pair(tmem_slot, p.tmem_cols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, p.tmem_cols);
            tmem_relinquish();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (PAIR) cluster_sync();  // both CTAs' barriers exist before any remote arrival
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtl ctl{abort_flag, p.err, p.timeout_ns};
    const uint32_t sB = smem_u32(bptr), sRing = smem_u32(ring), sStage = smem_u32(stage);
    griddep_wait();  // no global memory before the grid ahead of this one is done

    if (warp < MMA_WARP) {
        win_produce<T, PAIR>(p, rank, sB, sRing, sStage, rtab, atab, full, empty, bres, bpeer, sfull, ctl);
    } else if (warp == MMA_WARP) {
        if (rank == 0)  // the whole warp runs the issuing loop; one lane issues
            win_mma<TF32, PAIR>(p, tmem_base, sB, atab, full, empty, tfull, tempty, mma_done, bres, bpeer, ctl);
        if (lane == 0) win_drain(mma_done, 0u, p);  // the (leader's) final commit reaches this CTA
    } else {
        if (p.y_tma && lane == 0) prefetch_tmap(&tmY);
        win_epilogue<PAIR>(p, rank, tmem_base, tfull, tempty, epi, &tmY, ctl);
    }
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (PAIR) cluster_sync();  // neither CTA leaves while the pair's MMAs may read it
    tc_fence_after_sync();
    if (warp == MMA_WARP) {
        if (PAIR)
            tmem_dealloc_pair(tmem_base, p.tmem_cols);
        else
            tmem_dealloc(tmem_base, p.tmem_cols);
    }
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
    p.px_read = p.steps * 32 / D;
    // pixels the stored outputs of a row read: Q - 1 + px_read
    const int need = pb.Q - 1 + p.px_read;
    if (need <= 32) p.Qs = 32;
    else if (need <= 64) p.Qs = 64;
    else p.Qs = 128;
    p.qs_log2 = p.Qs == 32 ? 5 : (p.Qs == 64 ? 6 : 7);
    p.J = WBM / p.Qs;
    p.segs = p.J > 1 ? 1 : (pb.Q + WBM - 1) / WBM;
    p.PB = (pb.P + p.J - 1) / p.J;
    // A slot holds the phase pixels of one input row: Qs of them (J > 1; the
    // operand of a filter row runs on into the next slot), or for wide rows
    // the 128 + px_read - 1 a segment reads, in whole warp steps of the
    // 4-byte copies (128/D pixels), padded to the swizzle span.
    const int span = D == 64 ? 512 : 256;
    const int step_px = 128 / D;
    if (p.J > 1) {
        p.slot_px = p.Qs;
        p.slot_bytes = p.Qs * D;
    } else {
        p.slot_px = ((WBM - 1 + p.px_read + step_px - 1) / step_px) * step_px;
        p.slot_bytes = ((p.slot_px * D + span - 1) / span) * span;
    }
    p.rows = (p.J - 1) * pb.u + (pb.R - 1) * pb.dh + 1;
    if (p.rows > WIN_MAX_ROWS || pb.R * p.steps > WIN_MAX_MMAS) return false;
    auto fdiv = [](long long a, long long b) { return a >= 0 ? a / b : -((b - 1 - a) / b); };
    p.kb_off = (int)fdiv(-pb.pt, pb.u);
    p.kspan = (int)(fdiv((long long)p.rows - 1 - pb.pt, pb.u) - p.kb_off + 1);
    if ((long long)pb.N * p.PB * p.segs > 0x7fffffffLL) return false;
    p.num_tiles = pb.N * p.PB * p.segs;
    p.BN = ((pb.K + 15) / 16) * 16;
    // CTA pairs share each MMA (M = 256) and split the filters.  Pairing two
    // SMs' producers measured slower at N = 64, so pairs are opt-in:
    // DLC_TC_WINPAIR=1.
    {
        const char *ev = std::getenv("DLC_TC_WINPAIR");
        p.pair = (p.num_tiles >= 2 && ev && std::atoi(ev) != 0) ? 1 : 0;
    }
    p.num_units = p.pair ? (p.num_tiles + 1) / 2 : p.num_tiles;
    p.b_img_bytes = pb.R * p.steps * (p.pair ? p.BN / 2 : p.BN) * 32;
    const long long b_bytes = ((long long)p.b_img_bytes + 1023) & ~1023LL;
    // Ring: 2*kspan slots per phase let a tile that starts a new run fill
    // slots its predecessor does not read; if that does not fit, kspan + J
    // slots and such a tile first waits for its predecessor's MMAs.  After the
    // last slot: the pixels the operand of a J > 1 tile reads past it.
    const long long tail = ((long long)p.px_read * D + 1023) & ~1023LL;
    auto ring_of = [&](int rs) { return (long long)pb.u * (rs + p.J - 1) * p.slot_bytes + tail; };
    const long long fixed = 1024 + b_bytes + win_bar_area(p.rows, pb.R * p.steps);
    p.RS = 2 * p.kspan;
    p.disc_wait = 0;
    if (fixed + ring_of(p.RS) > WIN_MAX_SMEM) {
        p.RS = p.kspan + p.J;
        p.disc_wait = 1;
    }
    p.RSJ = p.RS + p.J - 1;
    if ((long long)pb.u * p.RSJ >= 65536) return false;  // ring table fields
    const long long ring = ring_of(p.RS);
    if (fixed + ring > WIN_MAX_SMEM) return false;
    p.ring_bytes = (int)ring;
    const long long base = fixed + ring;
    // the packed filter image goes through the handle's repacking buffer
    if ((long long)pb.R * p.steps * p.BN * 32 > DLC_WPACK_BYTES) return false;  // both parts
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
cudaError_t win_launch(const WinParams &p, const CUtensorMap &ty, int sm_count, size_t smem,
                       cudaStream_t st) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = dlc_pdl_enabled() ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.blockDim = dim3(WIN_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!p.pair) {
        auto kern = conv_window_kernel<TF32, false>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(std::max(1, std::min(p.num_units, sm_count)), 1, 1);
        return cudaLaunchKernelEx(&cfg, kern, p, ty);
    }
    auto kern = conv_window_kernel<TF32, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cfg.attrs = attr + 1;  // the occupancy query takes the cluster shape only
    cfg.gridDim = dim3(2 * (sm_count / 2), 1, 1);
    int max_clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&max_clusters, (const void *)kern, &cfg);
    if (e != cudaSuccess) return e;
    if (max_clusters < 1) return cudaErrorLaunchOutOfResources;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(2 * std::min(max_clusters, p.num_units), 1, 1);
    return cudaLaunchKernelEx(&cfg, kern, p, ty);
}

}  // namespace

bool dlc_window_ok(const ConvProblem &pb) { return window_plan(pb, nullptr, nullptr); }

dlcStatus_t dlc_preload_window() {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, window_pack_filters<uint16_t>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, window_pack_filters<uint32_t>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_window_kernel<false, false>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_window_kernel<false, true>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_window_kernel<true, false>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_window_kernel<true, true>) != cudaSuccess)
        return DLC_STATUS_EXECUTION_FAILED;
    return DLC_STATUS_SUCCESS;
}

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
    if (!ctx->wpack) return DLC_STATUS_INTERNAL_ERROR;
    p.wpack = ctx->wpack;
    p.y_tma = (win_y_tma_ok(pb) && smem + WIN_EPI_SMEM <= (size_t)WIN_MAX_SMEM) ? 1 : 0;
    if (const char *ev = std::getenv("DLC_TC_YTMA")) p.y_tma = p.y_tma && std::atoi(ev) != 0;
    const size_t epi1 = p.y_tma ? (size_t)WIN_EPI_SMEM : 0;
    // Staged rows: dense rows whose starts and lengths are 16-byte multiples
    // arrive by one bulk copy per tile (DLC_TC_WINSTAGE=0 keeps the 4-byte copies).
    {
        const long long stage = (long long)p.rows * p.row_bytes;
        const bool dense = pb.xs[2] == (long long)pb.W * pb.xs[3];
        bool on = p.x_word && dense && p.row_bytes % 16 == 0 && ((uintptr_t)pb.x % 16) == 0 &&
                  (pb.xs[0] * e) % 16 == 0 && (pb.xs[2] * e) % 16 == 0 && stage < (1LL << 20) &&
                  smem + 2 * (size_t)stage + epi1 <= (size_t)WIN_MAX_SMEM;
        // rows on any element boundary: stage the 16-byte-aligned superset of a
        // tile's rows (its round-up never passes the end of x, whose size is a
        // multiple of 16 bytes) and read it shifted
        const long long xbytes = ((long long)(pb.N - 1) * pb.xs[0] + (long long)pb.H * pb.xs[2]) * e;
        const long long stage2 = (stage + 32 + 15) / 16 * 16;
        bool shift = !on && contiguous && dense && p.nb % 4 == 0 && ((uintptr_t)pb.x % 16) == 0 &&
                     pb.xs[0] >= (long long)pb.H * pb.xs[2] && xbytes % 16 == 0 && stage2 < (1LL << 20);
        if (shift && smem + 2 * (size_t)stage2 + epi1 > (size_t)WIN_MAX_SMEM && !p.disc_wait) {
            // make room with the short ring (kspan + J slots per phase; a tile
            // that starts a new run of rows waits for its predecessor's MMAs)
            const long long tail = ((long long)p.px_read * p.D + 1023) & ~1023LL;
            const int rs2 = p.kspan + p.J;
            const long long ring2 = (long long)pb.u * (rs2 + p.J - 1) * p.slot_bytes + tail;
            const size_t smem2 = smem - (size_t)p.ring_bytes + (size_t)ring2;
            if (rs2 < p.RS && smem2 + 2 * (size_t)stage2 + epi1 <= (size_t)WIN_MAX_SMEM) {
                p.RS = rs2;
                p.RSJ = rs2 + p.J - 1;
                p.disc_wait = 1;
                p.ring_bytes = (int)ring2;
                smem = smem2;
            }
        }
        shift = shift && smem + 2 * (size_t)stage2 + epi1 <= (size_t)WIN_MAX_SMEM;
        if (const char *ev = std::getenv("DLC_TC_WINSTAGE")) on = on && std::atoi(ev) != 0;
        const bool sh = shift && !(std::getenv("DLC_TC_WINSTAGE") && std::atoi(std::getenv("DLC_TC_WINSTAGE")) == 0);
        p.x_stage = (on || sh) ? 1 : 0;
        p.x_shift = sh ? 1 : 0;
        p.stage_bytes = on ? (int)stage : (sh ? (int)stage2 : 0);
        if (p.x_stage) smem += 2 * (size_t)p.stage_bytes;
    }
    p.epi_bufs = (p.y_tma && smem + 2 * WIN_EPI_SMEM <= (size_t)WIN_MAX_SMEM) ? 2 : 1;
    if (p.y_tma) smem += (size_t)p.epi_bufs * WIN_EPI_SMEM;

    const uint32_t fmt = tf32 ? 2u : 1u;
    p.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(p.BN >> 3) << 17) |
              ((uint32_t)((p.pair ? 2 * WBM : WBM) >> 4) << 24);
    // TMEM: four accumulators when they fit in 512 columns, else two, so the
    // MMAs of the next tiles need not wait for the epilogue
    uint32_t acc = 32;
    while (acc < (uint32_t)p.BN) acc <<= 1;
    p.nacc_log2 = 4 * acc <= 512 ? 2 : 1;
    p.acc_stride = acc;
    p.tmem_cols = acc << p.nacc_log2;
    // ring slots: rows D bytes apart, 8-row groups 8*D apart; 16-byte rows use no
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
        cudaLaunchConfig_t cfg;
        std::memset(&cfg, 0, sizeof(cfg));
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = dlc_pdl_enabled() ? 1 : 0;
        cfg.gridDim = dim3((words + 255) / 256, 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = ctx->stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        uint32_t *img = static_cast<uint32_t *>(ctx->wpack);
        const cudaError_t e = tf32 ? cudaLaunchKernelEx(&cfg, window_pack_filters<uint32_t>, p, img)
                                   : cudaLaunchKernelEx(&cfg, window_pack_filters<uint16_t>, p, img);
        if (e != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
        ctx->launches += 1;
    }
    cudaError_t err = tf32 ? win_launch<true>(p, ty, ctx->sm_count, smem, ctx->stream)
                           : win_launch<false>(p, ty, ctx->sm_count, smem, ctx->stream);
    if (err != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}
