// conv_rowstack.cu -- forward convolution of layers with few filters and
// horizontal stride 1 or 2 on channel-planar (NCHW) activations, TF32 on the
// sm_103a tensor cores, with the filters stacked over output rows as the
// MMA's M side.
//
// With K = 32 filters the usual lowering (output pixels as M, filters as N)
// gives tcgen05 MMAs of N = 32: each operand byte of the pixel side feeds only
// 32 multiply-adds, so shared-memory bandwidth, not the tensor core, would
// bound the layer at a fraction of its peak.  Here the roles turn round (the
// batch-reduce GEMM page, method section: acc += sum_i A_i B_i over a block of
// the reduction; maxDNN page, method section: every output coordinate is its
// receptive field times the filters):
//
//  * M = 128 rows = J output rows (p0 .. p0+J-1) x K_pad filters.  For input
//    row h = p0*u - pad_top + t of a tile (t < T = (J-1)*u + (R-1)*dh + 1), MMA
//    row (j, k) takes filter row r = (t - j*u)/dh of filter k (zero when that
//    is not a whole filter row in [0, R)), so one MMA adds the contribution of
//    input row h to J output rows at once.
//  * N = output pixels.  With 4-byte elements and horizontal stride v, output
//    pixel q = PH*a + b (PH = 4/v phases b, a < ceil(Q/PH)) reads
//    x[v*q + s - pad_left] = x[4a + v*b - pad_left + s], s < S: for a fixed
//    phase the windows of consecutive a start 16 bytes apart in a copy of the
//    input row shifted by v*b - pad_left elements.  Such a copy is a K-major,
//    no-swizzle MMA operand (8-row core matrices of 16-byte rows, the next 4
//    window taps 16 bytes further), read in place -- no lowered row is built.
//    N = NI images x seg_a rows.
//  * K (reduction) = (slot, filter tap s) in chunks of 4 taps (S padded to a
//    multiple of 4).  A stage has 4 slots: 4 channels of input row t, or, for
//    a layer with one channel, 4 consecutive input rows t .. t+3 (the packed
//    filters of slot dt are the filter rows shifted by dt).  An MMA takes two chunks, which may belong to two slots: its
//    leading offset is then the distance between their copies.
//
// A work unit is (NI images, J output rows, two phases): two TMEM
// accumulators of N columns.  For every block of input rows and group of
// channels a stage holds the filter slices (A: one TMA load of the packed
// filter image, 128-byte swizzled K-major with four MMAs' slices per 128-byte
// row, rows j read at R-1-t+j*u by a strided box, out-of-range rows
// zero-filled) and the shifted copies of the 4 slots' input rows for both
// phases and all NI images (B).  One copier warp stages each input row once,
// as a 16-byte-aligned superset, with bulk copies into a ring of three raw
// buffers as far ahead as they are free; eight builder warps repack the raw
// rows into the two phase copies (several warps share a row when a stage has
// fewer rows than warps); one thread of a fifteenth warp loads the filter
// slices.  A stage's full barrier counts the builders' arrivals and the
// loader's, which carries the filter bytes.  Input rows outside the image
// contribute nothing and stages wholly outside are skipped.  Four epilogue
// warps read the accumulators and store y (alpha, beta*y, bias, ReLU)
// through its strides.  Every wait is bounded.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace {

using namespace dlc;

constexpr int RS_M = 128;            // MMA rows
constexpr int RS_CG = 4;             // slots per stage: (channel, input-row offset) pairs
constexpr int RS_BUILD_WARPS = 8;
constexpr int RS_PROD_WARPS = RS_BUILD_WARPS + 1;           // the raw-row copier and the builders
constexpr int RS_MMA_WARP = RS_PROD_WARPS;
constexpr int RS_A_WARP = RS_MMA_WARP + 5;                  // after the four epilogue warps
constexpr int RS_THREADS = (RS_A_WARP + 1) * 32;
constexpr int RS_RAW = 3;            // raw-row buffers
constexpr int RS_MAX_SMEM = 232448;
constexpr int RS_BAR_AREA = 256;     // barriers
constexpr int RS_EPI_WORDS = 32 * 33;  // one epilogue warp's staging buffer
constexpr int RS_EPI_BYTES = 4 * RS_EPI_WORDS * 4;
constexpr int RS_MAX_MPG = 16;       // MMAs per stage and phase
constexpr int RS_MAX_RB = 256;       // row blocks the unit order sorts

struct RsParams {
    int N, C, H, W, K, R, S, P, Q;
    int pt, pl, u, v, dh;
    int PH, passes;        // phases (16 bytes / (4 bytes x v)) and pairs of them: one per unit
    int rps, cps;          // input rows and channels per stage (rps x cps = RS_CG slots; rps 1 or 4)
    int J, K_pad;          // output rows per tile, filters per row block (J*K_pad = 128)
    int T;                 // input rows one tile spans
    int R_img;             // rows of the packed filter image: R + rps - 1
    int cpc;               // 4-tap chunks per channel: ceil(S/4)
    int mpg;               // MMAs per stage and phase: RS_CG*cpc/2
    int groups;            // channel groups: ceil(C/cps)
    int qa;                // pixels per phase and row: ceil(Q/PH)
    int seg_a, NI, Nmma;   // rows per image segment, images per tile, MMA N (multiple of 16)
    int copy_bytes;        // bytes of one shifted row copy (all NI images)
    int b_stage;           // bytes of one stage's B copies: 2 phases x RS_CG slots
    int acols;             // 128-byte A columns per stage: ceil(mpg/4), four MMAs' slices each
    int a_stage;           // bytes of one stage's A: acols x 16 KiB
    int raw_bytes;         // bytes of one staged input row (16-byte-aligned superset)
    int raw_stage;         // bytes of one of the RS_RAW raw-row buffers: RS_CG slots x NI rows
    int stages;
    int row_blocks, img_groups, tiles, units;
    int sorted;                   // row_order holds the row blocks, most input rows first
    unsigned short row_order[RS_MAX_RB];
    uint32_t b_off[RS_MAX_MPG];   // start of MMA i's first chunk within a phase's copies
    uint32_t b_lbo[RS_MAX_MPG];   // bytes from its first to its second chunk
    long long xs[4], ys[4];
    const float *x;
    unsigned long long x_beg16;   // start of x rounded up to 16 bytes: copies start there
    unsigned long long x_end16;   // end of x rounded down to 16 bytes: copies stop there
    void *y;
    const float *bias;
    float alpha, beta;
    int relu, y_bf16;
    uint32_t idesc, tmem_cols;
    int *err;
    unsigned long long timeout_ns;
};

// The kernel's compile-time shape: horizontal stride V (1 or 2: PH = 4/V
// phases, PASSES = PH/2 units per tile), SPLIT builder warps per row pair (1,
// or 2 when a stage has only 4 pairs), RPS input rows per stage (1, or 4 for
// one channel).
template <int V_, int SPLIT_, int RPS_>
struct RsCfg {
    static constexpr int V = V_, SPLIT = SPLIT_, RPS = RPS_;
    static constexpr int PH = 4 / V_, PASSES = 2 / V_;
    static constexpr int CPS = RS_CG / RPS_;  // channels per stage
};

struct RsUnit {
    int g, pb, pass;
};

// Unit u of the CTA walk (CTA b takes u = b, b + G, b + 2G, ..., G CTAs).
// Units are ranked row block by row block, the blocks with the most input
// rows inside the image first, and within a block by image group and pass;
// a CTA's second, fourth, ... whole round takes the ranks in reverse, so the
// light blocks of the last rounds even out the heavy ones of the first.
template <class Cf>
__device__ __forceinline__ RsUnit rs_unit(const RsParams &p, int u) {
    const int G = gridDim.x;
    const int round = u / G;
    int rank = u;
    if ((round & 1) && (round + 1) * G <= p.units) rank = round * G + (G - 1 - (u - round * G));
    RsUnit w;
    const int t = rank / Cf::PASSES;
    w.pass = rank - t * Cf::PASSES;
    const int s = t / p.img_groups;
    w.g = t - s * p.img_groups;
    w.pb = p.sorted ? (int)p.row_order[s] : s;
    return w;
}

// True when one of the rps input rows of the stage at tile row t of row block
// pb lies inside the image.
template <class Cf>
__device__ __forceinline__ bool rs_stage_in(const RsParams &p, int pb, int t) {
    const int h = pb * p.J * p.u - p.pt + t;
    return h + Cf::RPS > 0 && h < p.H;
}

// The stages a CTA walks: its units in order; within a unit the blocks of rps
// input rows t, t+1, ... that reach into the image, and for each the channel
// groups.
template <class Cf>
struct RsWalk {
    int u, t, cg;
    bool valid;
    RsUnit w;  // unit u's coordinates
    __device__ void enter(const RsParams &p) {
        valid = u < p.units;
        if (valid) w = rs_unit<Cf>(p, u);
    }
    __device__ void first(const RsParams &p) {
        u = blockIdx.x;
        t = 0;
        cg = 0;
        enter(p);
        settle(p);
    }
    __device__ void settle(const RsParams &p) {  // skip rows outside the image
        while (valid && !rs_stage_in<Cf>(p, w.pb, t)) {
            if ((t += Cf::RPS) >= p.T) {
                t = 0;
                u += gridDim.x;
                enter(p);
            }
        }
    }
    __device__ void next(const RsParams &p) {
        if (++cg < p.groups) return;
        cg = 0;
        if ((t += Cf::RPS) >= p.T) {
            t = 0;
            u += gridDim.x;
            enter(p);
        }
        settle(p);
    }
};

// Global address of input row (n, c, h) of a stage's (slot, image slot): slot
// sl is channel cg*cps + sl/rps, input row t + sl%rps of the tile.  `in` says
// whether the row exists (inside N, C and the image).
template <class Cf>
__device__ __forceinline__ const float *rs_row_ptr(const RsParams &p, const RsUnit &w, int t, int cg,
                                                   int sl, int ii, bool &in) {
    const int n = w.g * p.NI + ii, c = cg * Cf::CPS + sl / Cf::RPS;
    const int h = w.pb * p.J * p.u - p.pt + t + sl % Cf::RPS;
    // with one row per stage, stages outside the image are skipped whole
    in = n < p.N && c < p.C && (Cf::RPS == 1 || (h >= 0 && h < p.H));
    return p.x + (long long)(in ? n : 0) * p.xs[0] + (long long)(in ? c : 0) * p.xs[1] + (long long)h * p.xs[2];
}

// Bytes of input row (cl, ii) of a stage that its bulk copy moves: the
// 16-byte-aligned superset of the row, clipped to the 16-byte-aligned part
// of x (0 when the row lies in the first or last 16 bytes of x or past C, N).
template <class Cf>
__device__ __forceinline__ uint32_t rs_raw_span(const RsParams &p, const RsUnit &w, const RsWalk<Cf> &st, int cl,
                                                int ii, unsigned long long &beg, unsigned long long &a16) {
    bool in;
    const float *src = rs_row_ptr<Cf>(p, w, st.t, st.cg, cl, ii, in);
    const uintptr_t a = reinterpret_cast<uintptr_t>(src);
    a16 = a & ~15ull;
    beg = a16 > p.x_beg16 ? a16 : p.x_beg16;
    unsigned long long end = (a + 4ull * (unsigned long long)p.W + 15ull) & ~15ull;
    end = end < p.x_end16 ? end : p.x_end16;
    return (in && end > beg) ? (uint32_t)(end - beg) : 0u;
}

// Warp 0: bulk-copies the stage's input rows (RS_CG channels x NI images)
// into raw buffer `rb`, row (cl, ii) at slot (cl*NI + ii)*raw_bytes, one row
// per lane; lane 0 first announces the total bytes on `bar`.
template <class Cf>
__device__ void rs_copy_raw(const RsParams &p, uint32_t rb, const RsWalk<Cf> &st, uint64_t *bar, int lane) {
    const int combos = RS_CG * p.NI;
    unsigned long long beg = 0, a16 = 0;
    uint32_t bytes = 0;
    if (lane < combos) bytes = rs_raw_span(p, st.w, st, lane / p.NI, lane % p.NI, beg, a16);
    uint32_t total = bytes;
    for (int cmb = lane + 32; cmb < combos; cmb += 32) total += rs_raw_span(p, st.w, st, cmb / p.NI, cmb % p.NI, beg, a16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    if (lane == 0) mbar_arrive_expect_tx(bar, total);
    __syncwarp();
    if (bytes)
        bulk_load_1d(rb + (uint32_t)(lane * p.raw_bytes) + (uint32_t)(beg - a16), reinterpret_cast<const void *>(beg),
                     bytes, bar);
    for (int cmb = lane + 32; cmb < combos; cmb += 32) {
        const uint32_t b = rs_raw_span(p, st.w, st, cmb / p.NI, cmb % p.NI, beg, a16);
        if (b)
            bulk_load_1d(rb + (uint32_t)(cmb * p.raw_bytes) + (uint32_t)(beg - a16), reinterpret_cast<const void *>(beg),
                         b, bar);
    }
}

// Rows [0, rows) of the shifted copies of one (slot, image) row, shared by
// `split` warps (rows part*32 + lane + 32*split*i): row a of the copy for
// phase b0 holds elements e0 .. e0+3 of the input row, e0 = 4a + v*b0 - pl,
// and the copy for b0 + 1 elements e0+V .. e0+V+3 (V = v, the horizontal
// stride).  Rows in [fa, fb) find all 4+V in the raw row, at words
// 4*(g0 + a) + O .. + 3 + V (O = the offset within a 16-byte word, the same
// for every row), and take them with 16-byte loads, several rows' loads at a
// time; the others (a few at each end) take each element from the raw row,
// from x (the first and last 16 bytes of x are not staged) or zero (padding,
// past C, N or the image, or past the image segment).
template <int V>
__device__ __forceinline__ void rs_copy_rows(const uint4 *raw4, const uint32_t *raw1, uint4 *dst0, uint4 *dst1,
                                             int rows, int fa, int fb, int g0, int O, int e0_0, int sh, int e_lo,
                                             int avail, int lim, const float *src, int W, int first, int step) {
    constexpr int NV = V == 1 ? 2 : 3;  // 16-byte words a row's 4+V elements can span
    constexpr int U = V == 1 ? 4 : 2;   // rows a lane loads before it stores
    for (int a0 = fa + first; a0 < fb; a0 += step * U) {
        uint4 v[U][NV];
#pragma unroll
        for (int j = 0; j < U; ++j)
            if (a0 + step * j < fb) {
#pragma unroll
                for (int m = 0; m < NV; ++m) v[j][m] = raw4[g0 + a0 + step * j + m];
            }
#pragma unroll
        for (int j = 0; j < U; ++j)
            if (a0 + step * j < fb) {
                uint32_t q[4 * NV];
#pragma unroll
                for (int m = 0; m < NV; ++m) {
                    q[4 * m] = v[j][m].x;
                    q[4 * m + 1] = v[j][m].y;
                    q[4 * m + 2] = v[j][m].z;
                    q[4 * m + 3] = v[j][m].w;
                }
                // words O .. O+3+V: shift down by 2, then by 1 (O is the same
                // for every lane)
                if (O & 2) {
#pragma unroll
                    for (int l = 0; l < 4 * NV - 2; ++l) q[l] = q[l + 2];
                }
                if (O & 1) {
#pragma unroll
                    for (int l = 0; l < 4 * NV - 3; ++l) q[l] = q[l + 1];
                }
                dst0[a0 + step * j] = make_uint4(q[0], q[1], q[2], q[3]);
                dst1[a0 + step * j] = make_uint4(q[V], q[V + 1], q[V + 2], q[V + 3]);
            }
    }
    const int edge = fa + (rows - fb);
    for (int i = first; i < edge; i += step) {
        const int a = i < fa ? i : fb + (i - fa);
        const int e0 = e0_0 + 4 * a;
        uint32_t el[4 + V];
#pragma unroll
        for (int l = 0; l < 4 + V; ++l) {
            const int e = e0 + l;
            el[l] = 0u;
            if (a < lim && e >= 0 && e < W)
                el[l] = (e >= e_lo && e < avail) ? raw1[sh + e] : __float_as_uint(__ldg(src + e));
        }
        dst0[a] = make_uint4(el[0], el[1], el[2], el[3]);
        dst1[a] = make_uint4(el[V], el[V + 1], el[V + 2], el[V + 3]);
    }
}

// A builder warp's (slot, image slot) pair, where its copies go, and which of
// the warps that share the pair it is.
struct RsCombo {
    int sl, ii, rows, part;
    size_t raw_off, dst0_off, dst1_off;  // bytes within a raw buffer / a stage's B
    __device__ void set(const RsParams &p, int cmb, int part_) {
        ii = cmb % p.NI;
        sl = cmb / p.NI;
        part = part_;
        const int r0 = ii * p.seg_a;
        rows = (ii == p.NI - 1 ? p.Nmma + p.cpc - 1 : r0 + p.seg_a) - r0;  // the last copy also feeds the tail
        raw_off = (size_t)cmb * p.raw_bytes;
        dst0_off = (size_t)sl * p.copy_bytes + 16 * (size_t)r0;
        dst1_off = (size_t)(RS_CG + sl) * p.copy_bytes + 16 * (size_t)r0;
    }
};

// The shifted row copies of one stage from its raw rows: for phase slot ph
// (phase b = 2*pass + ph), slot sl and image slot ii, row a of the copy holds
// x[n, c, h, 4a + v*b - pl + l], l < 4 (zero outside the row, past C, N or
// the image); rows past the last image segment (read only for unstored
// outputs) are zeros.  fa_c / fb_c: the fast rows of a row that lies wholly in
// the staged part of x, for this pass.  V: the horizontal stride; SPLIT: the
// warps that share a pair's rows.
template <class Cf>
__device__ __forceinline__ void rs_build_one(const RsParams &p, uint8_t *sb, const uint8_t *rb, const RsWalk<Cf> &st,
                                             const RsCombo &cb, int fa_c, int fb_c, int lane) {
    bool in;
    constexpr int V = Cf::V, SPLIT = Cf::SPLIT;
    const float *src = rs_row_ptr<Cf>(p, st.w, st.t, st.cg, cb.sl, cb.ii, in);
    const uintptr_t ra = reinterpret_cast<uintptr_t>(src);
    const int sh = (int)((ra & 15u) >> 2);  // element e of the row is word sh + e of the slot
    const int e0_0 = 2 * V * st.w.pass - p.pl;  // element of row 0 of the first phase's copy
    int e_lo = 0, avail = p.W, fa = fa_c, fb = fb_c;
    const unsigned long long c_lo = ra & ~15ull, c_hi = (ra + 4ull * p.W + 15ull) & ~15ull;
    if (!in) {
        fa = fb = 0;
    } else if (c_lo < p.x_beg16 || c_hi > p.x_end16) {
        // the first or last row of x: elements [e_lo, avail) are staged, the
        // others come from x
        const unsigned long long cbeg = c_lo > p.x_beg16 ? c_lo : p.x_beg16;
        const unsigned long long cend = c_hi < p.x_end16 ? c_hi : p.x_end16;
        e_lo = cbeg > ra ? (int)((cbeg - ra + 3) / 4) : 0;
        avail = cend > ra ? (int)std::min<unsigned long long>((unsigned long long)p.W, (cend - ra) / 4) : 0;
        const int lo = e_lo - e0_0;  // fast rows: 4a >= lo and 4a <= hi
        const int hi = avail - 4 - V - e0_0;
        fa = lo > 0 ? (lo + 3) / 4 : 0;
        fb = hi >= 0 ? std::min(hi / 4 + 1, p.seg_a) : 0;
        fb = std::max(fb, fa);
    }
    const int wb = sh + e0_0;           // word of element e0_0 in the slot (may be negative)
    const int O = wb & 3, g0 = wb >> 2;  // arithmetic shift: floor
    const int lim = in ? p.seg_a : 0;
    uint4 *dst0 = reinterpret_cast<uint4 *>(sb + cb.dst0_off);
    uint4 *dst1 = reinterpret_cast<uint4 *>(sb + cb.dst1_off);
    const uint4 *raw4 = reinterpret_cast<const uint4 *>(rb + cb.raw_off);
    const uint32_t *raw1 = reinterpret_cast<const uint32_t *>(rb + cb.raw_off);
    const int first = SPLIT == 1 ? lane : cb.part * 32 + lane;
    rs_copy_rows<V>(raw4, raw1, dst0, dst1, cb.rows, fa, fb, g0, O, e0_0, sh, e_lo, avail, lim, src, p.W, first,
                    32 * SPLIT);
}

// One lane's bounded wait, its outcome shared with the warp.
__device__ __forceinline__ bool rs_warp_wait(uint64_t *bar, uint32_t parity, const WaitCtl &ctl, int where,
                                             int lane) {
    int ok = 0;
    if (lane == 0) ok = mbar_wait(bar, parity, ctl, where) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Warp 0 bulk-copies the raw rows of the stages in order, each into one of
// RS_RAW buffers once the builders have freed it.  The builders (warps 1..8)
// build a stage's shifted row copies from its raw rows and arrive on its full
// barrier.
template <class Cf>
__device__ void rs_copy_stages(const RsParams &p, uint32_t sRaw, uint64_t *rawfull, uint64_t *rawempty,
                               const WaitCtl &ctl, int lane) {
    volatile int no_abort = 0;
    const WaitCtl drain{&no_abort, p.err, p.timeout_ns};
    RsWalk<Cf> r;
    r.first(p);
    int kr = 0;
    bool ok = true;
    for (; ok && r.valid; ++kr, r.next(p)) {
        if (kr >= RS_RAW) ok = rs_warp_wait(&rawempty[kr % RS_RAW], (uint32_t)((kr / RS_RAW) - 1) & 1u, ctl, 36, lane);
        if (!ok) break;
        fence_proxy_async_smem();
        rs_copy_raw(p, sRaw + (uint32_t)(kr % RS_RAW) * (uint32_t)p.raw_stage, r, &rawfull[kr % RS_RAW], lane);
    }
    // no copy may land after the CTA exits: wait for each raw buffer's last copy
    if (lane == 0)
        for (int j = kr > RS_RAW ? kr - RS_RAW : 0; j < kr; ++j)
            mbar_wait(&rawfull[j % RS_RAW], (uint32_t)(j / RS_RAW) & 1u, drain, 93);
    __syncwarp();
}

// One thread loads each stage's filter slices once its buffers are free
// (one TMA box: J rows u apart from packed row R-1-t on, the stage's channel
// group's columns); its arrival on the full barrier carries their bytes, so
// the stage cannot complete on the builders' arrivals alone.
template <class Cf>
__device__ void rs_load_filters(const RsParams &p, const CUtensorMap *tmA, uint32_t sA, uint64_t *empty,
                                uint64_t *full, const WaitCtl &ctl) {
    const int ST = p.stages;
    RsWalk<Cf> a;
    a.first(p);
    int stage = 0;
    uint32_t ph = 0;
    for (; a.valid; a.next(p)) {
        if (!mbar_wait(&empty[stage], ph ^ 1u, ctl, 31)) break;
        mbar_arrive_expect_tx(&full[stage], (uint32_t)p.a_stage);
        tma_load_4d_u32(sA + (uint32_t)stage * p.a_stage, tmA, &full[stage], 0, 0, p.R - 1 - a.t, a.cg * p.acols);
        if (++stage == ST) stage = 0, ph ^= 1u;
    }
}

template <class Cf>
__device__ void rs_build(const RsParams &p, uint8_t *sB, const uint8_t *sRaw, uint64_t *full, uint64_t *empty,
                         uint64_t *rawfull, uint64_t *rawempty, const WaitCtl &ctl) {
    const int warp = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
    const int ST = p.stages;
    constexpr int V = Cf::V, SPLIT = Cf::SPLIT;
    const int combos = RS_CG * p.NI;
    // the fast rows of a wholly staged row, per pass (phases 0-1, 2-3)
    int fa_c[2], fb_c[2];
    for (int ps = 0; ps < 2; ++ps) {
        const int e0_0 = 2 * V * ps - p.pl;
        fa_c[ps] = e0_0 < 0 ? (3 - e0_0) / 4 : 0;
        const int hi = p.W - 4 - V - e0_0;
        fb_c[ps] = std::max(hi >= 0 ? std::min(hi / 4 + 1, p.seg_a) : 0, fa_c[ps]);
    }
    // with fewer pairs than warps, SPLIT warps share each pair's rows
    RsCombo mine;  // the warp's pair when there is at most one per warp
    const bool has_mine = warp < combos * SPLIT;
    if (has_mine) mine.set(p, warp / SPLIT, warp % SPLIT);
    int stage = 0;
    uint32_t ph = 0;
    RsWalk<Cf> cur;
    cur.first(p);
    for (int k = 0; cur.valid; ++k) {
        bool ok = mbar_wait(&empty[stage], ph ^ 1u, ctl, 37);
        ok = ok && mbar_wait(&rawfull[k % RS_RAW], (uint32_t)(k / RS_RAW) & 1u, ctl, 32);
        // the decision to go on is the same for every builder
        int stop = (!ok || *ctl.abort_flag) ? 1 : 0;
        asm volatile("{\n\t.reg .pred q, r;\n\tsetp.ne.b32 q, %1, 0;\n\t"
                     "bar.red.or.pred r, 1, %2, q;\n\tselp.b32 %0, 1, 0, r;\n\t}\n"
                     : "=r"(stop) : "r"(stop), "n"(RS_BUILD_WARPS * 32) : "memory");
        if (stop) break;
        uint8_t *sb = sB + (size_t)stage * p.b_stage;
        const uint8_t *rb = sRaw + (size_t)(k % RS_RAW) * p.raw_stage;
        const int ps = cur.w.pass;
        if (has_mine) rs_build_one<Cf>(p, sb, rb, cur, mine, fa_c[ps], fb_c[ps], lane);
        for (int cmb = warp + RS_BUILD_WARPS; cmb < combos; cmb += RS_BUILD_WARPS) {  // SPLIT == 1 here
            RsCombo cb;
            cb.set(p, cmb, 0);
            rs_build_one<Cf>(p, sb, rb, cur, cb, fa_c[ps], fb_c[ps], lane);
        }
        fence_proxy_async_smem();  // the copies, for the tensor core
        mbar_arrive(&full[stage]);
        mbar_arrive(&rawempty[k % RS_RAW]);
        if (++stage == ST) stage = 0, ph ^= 1u;
        cur.next(p);
    }
}

template <class Cf>
__device__ void rs_mma(const RsParams &p, uint32_t tmem_base, uint32_t sA, uint32_t sB, uint64_t *full,
                       uint64_t *empty, uint64_t *tfull, uint64_t *tempty, uint64_t *mma_done,
                       const WaitCtl &ctl) {
    const int ST = p.stages;
    // A: 128-byte swizzled K-major, 128 rows of 128 bytes per column (8-row
    // groups 1024 bytes apart); MMA i reads the 32 bytes at (i % 4) * 32 of
    // column i / 4
    const uint64_t a0 = (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61) |
                        (uint64_t)((sA >> 4) & 0x3FFFu);
    // B: no swizzle, 16-byte rows, 8-row core matrices 128 bytes apart; the
    // leading offset (second chunk) per MMA.  The stage-0 descriptors of a
    // stage's MMAs stay in registers.
    const uint64_t b_hi = ((uint64_t)(128 >> 4) << 32) | (1ull << 46);
    uint64_t bd[2][RS_MAX_MPG];
#pragma unroll
    for (int i = 0; i < RS_MAX_MPG; ++i)
#pragma unroll
        for (int q = 0; q < 2; ++q)
            bd[q][i] = i < p.mpg ? (b_hi |
                                    (uint64_t)(((sB + (uint32_t)(q * RS_CG * p.copy_bytes) + p.b_off[i]) >> 4) & 0x3FFFu) |
                                    ((uint64_t)((p.b_lbo[i] >> 4) & 0x3FFFu) << 16))
                                 : 0ull;
    int stage = 0, it = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x, ++it) {
        const RsUnit w = rs_unit<Cf>(p, u);
        if (!mbar_wait(&tempty[0], (uint32_t)(it & 1) ^ 1u, ctl, 33)) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        uint32_t acc = 0;
        for (int t = 0; ok && t < p.T; t += Cf::RPS) {
            if (!rs_stage_in<Cf>(p, w.pb, t)) continue;
            for (int cg = 0; cg < p.groups; ++cg) {
                if (!mbar_wait(&full[stage], ph, ctl, 34)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                // start fields move by whole stages (addresses below 256 KiB: no carry)
                const uint64_t ao = (uint64_t)(((uint32_t)stage * (uint32_t)p.a_stage) >> 4);
                const uint64_t bo = (uint64_t)(((uint32_t)stage * (uint32_t)p.b_stage) >> 4);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint32_t d = tmem_base + (uint32_t)(q * p.Nmma);
#pragma unroll
                    for (int i = 0; i < RS_MAX_MPG; ++i) {
                        // the unit's first MMA into each accumulator starts it
                        if (i < p.mpg)
                            umma_tf32_nc(d, a0 + ao + (uint64_t)(1024 * (i >> 2) + 2 * (i & 3)), bd[q][i] + bo,
                                         p.idesc, (acc | (uint32_t)i) ? 1u : 0u);
                    }
                }
                acc = 1;
                umma_commit(&empty[stage]);
                if (++stage == ST) stage = 0, ph ^= 1u;
            }
        }
        if (!ok) break;
        umma_commit(&tfull[0]);
    }
    if (!ok) {
        volatile int dummy = 0;
        const WaitCtl brief{&dummy, p.err, 50000000ull};
        for (int j = 0; j < ST; ++j) {
            if (!mbar_wait(&full[stage], ph, brief, 99)) break;
            if (++stage == ST) stage = 0, ph ^= 1u;
        }
    }
    umma_commit(mma_done);
    volatile int dummy = 0;
    const WaitCtl fin{&dummy, p.err, p.timeout_ns};
    mbar_wait(mma_done, 0u, fin, 98);
}

__device__ __forceinline__ float rs_bf16_to_f32(unsigned short b) { return __uint_as_float((uint32_t)b << 16); }

// A warp reads its 32 TMEM lanes -- 32 filters k0 .. k0+31 of one output row
// op, since K_pad >= 32 -- 16 columns of both phases at a time, stages them
// in its 32 x 33-word shared buffer (row r: the 16 columns' two phases
// interleaved) and stores filter by filter: lane i writes column c0 + i/2 of
// phase b0 + i%2, so a warp's store covers consecutive outputs of one row
// (32 at horizontal stride 2, 16 pairs 16 bytes apart at stride 1) instead of
// 32 rows' scattered words.  Column c of a phase's accumulator is pixel
// a = c mod seg_a of image slot c / seg_a, output q = PH*a + b.
template <class Cf>
__device__ void rs_epilogue(const RsParams &p, uint32_t tmem_base, float *ebuf_all, uint64_t *tfull,
                            uint64_t *tempty, const WaitCtl &ctl) {
    // a warp reads the TMEM lanes of its index modulo 4
    const int quad = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
    float *ebuf = ebuf_all + quad * RS_EPI_WORDS;
    const int j = quad * 32 / p.K_pad, k0 = quad * 32 - j * p.K_pad;
    const int rows = std::min(32, p.K - k0);  // filters of this warp that exist
    const bool plain = p.beta == 0.f && !p.bias && !p.relu && !p.y_bf16;
    const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16);
    int it = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++it) {
        const RsUnit w = rs_unit<Cf>(p, u);
        int okw = 0;
        if (lane == 0) okw = mbar_wait(&tfull[0], (uint32_t)(it & 1), ctl, 35) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) break;
        __syncwarp();
        tc_fence_after_sync();
        const int op = w.pb * p.J + j;
        const bool warp_ok = rows > 0 && op < p.P;
        const int b = 2 * w.pass + (lane & 1);
        const long long rowbase = (long long)k0 * p.ys[1] + (long long)op * p.ys[2];
        for (int c0 = 0; c0 < p.Nmma; c0 += 16) {
            uint32_t v0[16], v1[16];
            tmem_ld_32x32b_x16(taddr + (uint32_t)c0, v0);
            tmem_ld_32x32b_x16(taddr + (uint32_t)(p.Nmma + c0), v1);
            tmem_ld_wait();
            if (!warp_ok) continue;
            __syncwarp();  // the previous chunk's rows are read
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                ebuf[lane * 33 + 2 * e] = __uint_as_float(v0[e]);
                ebuf[lane * 33 + 2 * e + 1] = __uint_as_float(v1[e]);
            }
            __syncwarp();
            const int col = c0 + (lane >> 1);
            const int ii = col / p.seg_a, a = col - ii * p.seg_a;
            const int n = w.g * p.NI + ii;
            const bool lane_ok = ii < p.NI && n < p.N && a < p.qa && Cf::PH * a + b < p.Q;
            long long yo = (long long)n * p.ys[0] + (long long)(Cf::PH * a + b) * p.ys[3] + rowbase;
            if (plain) {
                float *yf = static_cast<float *>(p.y);
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    if (lane_ok && r < rows) yf[yo] = p.alpha * ebuf[r * 33 + lane];
                    yo += p.ys[1];
                }
            } else {
                float *yf = static_cast<float *>(p.y);
                unsigned short *yb = static_cast<unsigned short *>(p.y);
#pragma unroll 4
                for (int r = 0; r < 32; ++r) {
                    if (lane_ok && r < rows) {
                        float f = p.alpha * ebuf[r * 33 + lane];
                        if (p.beta != 0.f) f = __fmaf_rn(p.beta, p.y_bf16 ? rs_bf16_to_f32(yb[yo]) : yf[yo], f);
                        if (p.bias) f += __ldg(p.bias + k0 + r);
                        if (p.relu) f = fmaxf(f, 0.f);
                        if (p.y_bf16)
                            yb[yo] = __bfloat16_as_ushort(__float2bfloat16_rn(f));
                        else
                            yf[yo] = f;
                    }
                    yo += p.ys[1];
                }
            }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[0]);
    }
}

template <class Cf>
__global__ void __launch_bounds__(RS_THREADS, 1)
    conv_rowstack_kernel(const __grid_constant__ RsParams p, const __grid_constant__ CUtensorMap tmA) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int ST = p.stages;
    uint8_t *smA = smem;
    uint8_t *smB = smA + (size_t)ST * p.a_stage;
    uint8_t *smRaw = smB + (size_t)ST * p.b_stage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smRaw + RS_RAW * (size_t)p.raw_stage);
    uint64_t *full = bars;
    uint64_t *empty = bars + ST;
    uint64_t *tfull = bars + 2 * ST;
    uint64_t *tempty = tfull + 1;
    uint64_t *mma_done = tempty + 1;
    uint64_t *rawfull = mma_done + 1;       // RS_RAW of them
    uint64_t *rawempty = rawfull + RS_RAW;  // RS_RAW of them
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(rawempty + RS_RAW);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) {
            // every producer thread arrives, the A load adds its bytes
            mbar_init(&full[i], RS_BUILD_WARPS * 32 + 1);  // builders and the issuer
            mbar_init(&empty[i], 1u);
        }
        mbar_init(tfull, 1u);
        mbar_init(tempty, 4u);
        mbar_init(mma_done, 1u);
        for (int i = 0; i < RS_RAW; ++i) {
            mbar_init(&rawfull[i], 1u);                   // the issuer's expect-tx arrival
            mbar_init(&rawempty[i], RS_BUILD_WARPS * 32);  // every builder thread
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == RS_MMA_WARP) {
        tmem_alloc(tmem_slot, p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtl ctl{abort_flag, p.err, p.timeout_ns};
    if (warp == 0) {
        rs_copy_stages<Cf>(p, smem_u32(smRaw), rawfull, rawempty, ctl, lane);
    } else if (warp == RS_A_WARP) {
        if (lane == 0) {
            prefetch_tmap(&tmA);
            rs_load_filters<Cf>(p, &tmA, smem_u32(smA), empty, full, ctl);
        }
    } else if (warp < RS_PROD_WARPS) {
        rs_build<Cf>(p, smB, smRaw, full, empty, rawfull, rawempty, ctl);
    } else if (warp == RS_MMA_WARP) {
        if (lane == 0)
            rs_mma<Cf>(p, tmem_base, smem_u32(smA), smem_u32(smB), full, empty, tfull, tempty, mma_done, ctl);
    } else {
        rs_epilogue<Cf>(p, tmem_base, reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(bars) + RS_BAR_AREA),
                        tfull, tempty, ctl);
    }
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == RS_MMA_WARP) tmem_dealloc(tmem_base, p.tmem_cols);
}

// The filters as MMA A operands, in the order the convolution's TMA box reads
// them: image [m][z][k][32] (m = (channel group, 128-byte column), z <
// R + rps - 1, k < K_pad filters, 32 reduction elements: four MMAs' 8 each).
// Element (MMA i, e) belongs to chunk 2i + e/4 of the stage's (slot, chunk)
// sequence; its slot is channel cg*cps + slot/rps and input-row offset
// dt = slot%rps, and it holds tap s of filter row r = R-1-z + dt, or zero.
// The box of the stage at tile row t reads rows z = R-1-t + j*u for output
// rows j, so slot dt gets filter row t + dt - j*u: the one that input row
// t + dt meets for output row j.  One thread per element.
__global__ void rowstack_pack_filters(const __grid_constant__ RsParams p, const float *w, long long ws0,
                                      long long ws1, long long ws2, long long ws3, float *img) {
    griddep_wait();  // the previous convolution may still read the image
    griddep_launch_dependents();
    const long long total = (long long)p.groups * p.acols * p.R_img * p.K_pad * 32;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int f = (int)(i & 31);
    long long t = i >> 5;
    const int k = (int)(t % p.K_pad);
    t /= p.K_pad;
    const int z = (int)(t % p.R_img);
    const int m = (int)(t / p.R_img);
    const int cg = m / p.acols, col = m - cg * p.acols;
    const int mi = 4 * col + (f >> 3), e = f & 7;  // MMA of the stage, its element
    const int chunk = 2 * mi + (e >> 2);
    const int slot = chunk / p.cpc;
    const int c = cg * p.cps + slot / p.rps;
    const int s = 4 * (chunk % p.cpc) + (e & 3);
    const int r = p.R - 1 - z + slot % p.rps;
    float v = 0.f;
    if (mi < p.mpg && k < p.K && c < p.C && s < p.S && r >= 0 && r < p.R)
        v = __ldg(w + (long long)k * ws0 + (long long)c * ws1 + (long long)r * ws2 + (long long)s * ws3);
    img[i] = v;
}

// Plan: every field but the pointers.  False when the kernel does not take
// the problem.
bool rowstack_plan(const ConvProblem &pb, size_t wpack_bytes, RsParams *out, size_t *smem_out) {
    if (pb.math != DLC_MATH_TF32 || pb.xdt != DLC_DATA_FLOAT) return false;
    if (pb.xs[3] != 1 || (pb.v != 1 && pb.v != 2) || pb.dw != 1 || pb.dh != 1) return false;
    if (pb.K > 64 || pb.S > 4 * 2 * RS_MAX_MPG / RS_CG) return false;
    if (pb.W < 1 || pb.Q < 1) return false;
    // input rows arrive by bulk copies of their 16-byte-aligned supersets,
    // clipped to the 16-byte-aligned part of x
    for (int i = 0; i < 3; ++i)
        if (pb.xs[i] < 0) return false;
    RsParams p;
    std::memset(&p, 0, sizeof(p));
    p.N = pb.N; p.C = pb.C; p.H = pb.H; p.W = pb.W; p.K = pb.K; p.R = pb.R; p.S = pb.S;
    p.P = pb.P; p.Q = pb.Q;
    p.pt = pb.pt; p.pl = pb.pl; p.u = pb.u; p.v = pb.v; p.dh = pb.dh;
    // output pixels q = PH*a + b of phase b start 16 bytes apart in the input
    // row; a unit takes two phases
    p.PH = 4 / pb.v;
    p.passes = p.PH / 2;
    // slots: channels, or for one channel 4 consecutive input rows
    p.rps = pb.C == 1 ? 4 : 1;
    p.cps = RS_CG / p.rps;
    p.K_pad = pb.K <= 32 ? 32 : 64;
    p.J = RS_M / p.K_pad;
    p.T = (p.J - 1) * pb.u + (pb.R - 1) * pb.dh + 1;
    p.R_img = pb.R + p.rps - 1;
    p.cpc = (pb.S + 3) / 4;
    if ((RS_CG * p.cpc) % 2) return false;
    p.mpg = RS_CG * p.cpc / 2;
    if (p.mpg > RS_MAX_MPG) return false;
    p.groups = (pb.C + p.cps - 1) / p.cps;
    p.qa = (pb.Q + p.PH - 1) / p.PH;
    p.seg_a = ((p.qa + p.cpc - 1 + 7) / 8) * 8;
    if (p.seg_a > 256) return false;
    p.NI = std::max(1, std::min(pb.N, 256 / p.seg_a));
    p.Nmma = ((p.NI * p.seg_a + 15) / 16) * 16;
    if (p.Nmma > 256) return false;
    p.copy_bytes = (p.Nmma + p.cpc - 1) * 16;
    p.copy_bytes = ((p.copy_bytes + 127) / 128) * 128;
    p.b_stage = 2 * RS_CG * p.copy_bytes;
    p.acols = (p.mpg + 3) / 4;
    p.a_stage = p.acols * 16384;
    // the 16-byte-aligned superset of a row, and room for the fast repack's
    // reads past the row's last word
    p.raw_bytes = ((pb.W * 4 + 48 + 15) / 16) * 16;
    p.raw_stage = RS_CG * p.NI * p.raw_bytes;
    const int stage = p.a_stage + p.b_stage;
    p.stages = std::min(8, (RS_MAX_SMEM - 1024 - RS_BAR_AREA - RS_EPI_BYTES - RS_RAW * p.raw_stage) / stage);
    if (p.stages < 2) return false;
    // MMA i of a stage takes chunks 2i and 2i+1 of the group's (slot, chunk)
    // sequence; chunk ch of slot ch / cpc sits in that slot's copy
    for (int i = 0; i < p.mpg; ++i) {
        auto addr = [&](int ch) { return (uint32_t)((ch / p.cpc) * p.copy_bytes + 16 * (ch % p.cpc)); };
        p.b_off[i] = addr(2 * i);
        p.b_lbo[i] = addr(2 * i + 1) - addr(2 * i);
    }
    p.row_blocks = (pb.P + p.J - 1) / p.J;
    p.img_groups = (pb.N + p.NI - 1) / p.NI;
    if (p.row_blocks <= RS_MAX_RB) {
        // stages of each row block that reach into the image
        int rows_in[RS_MAX_RB];
        for (int b = 0; b < p.row_blocks; ++b) {
            const int h0 = b * p.J * pb.u - pb.pt;
            rows_in[b] = 0;
            for (int t = 0; t < p.T; t += p.rps) rows_in[b] += (h0 + t + p.rps > 0 && h0 + t < pb.H) ? 1 : 0;
            p.row_order[b] = (unsigned short)b;
        }
        std::stable_sort(p.row_order, p.row_order + p.row_blocks,
                         [&](unsigned short a, unsigned short b) { return rows_in[a] > rows_in[b]; });
        p.sorted = 1;
    }
    const long long tiles = (long long)p.row_blocks * p.img_groups;
    if (tiles * p.passes > 0x7fffffffLL) return false;
    p.tiles = (int)tiles;
    p.units = p.passes * p.tiles;
    const long long img = (long long)p.groups * p.acols * p.R_img * p.K_pad * 128;
    if (img > (long long)wpack_bytes) return false;
    if (p.J * pb.u > 256 || pb.u > 8) return false;  // the filter box's strided rows
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * p.Nmma)) cols <<= 1;
    if (cols > 512) return false;
    p.tmem_cols = cols;
    // TF32 A and B (format 2), FP32 D, both K-major, M = 128
    p.idesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(p.Nmma >> 3) << 17) |
              ((uint32_t)(RS_M >> 4) << 24);
    if (out) *out = p;
    if (smem_out)
        *smem_out = 1024 + (size_t)p.stages * stage + RS_RAW * (size_t)p.raw_stage + RS_BAR_AREA + RS_EPI_BYTES;
    return true;
}

}  // namespace

namespace {

using RsKernel = void (*)(RsParams, CUtensorMap);

// The kernel instance for horizontal stride v, split builder warps and rps
// input rows per stage.
RsKernel rowstack_kernel_for(int v, bool split, int rps) {
    if (v == 1) {
        if (split) return rps == 4 ? conv_rowstack_kernel<RsCfg<1, 2, 4>> : conv_rowstack_kernel<RsCfg<1, 2, 1>>;
        return rps == 4 ? conv_rowstack_kernel<RsCfg<1, 1, 4>> : conv_rowstack_kernel<RsCfg<1, 1, 1>>;
    }
    if (split) return rps == 4 ? conv_rowstack_kernel<RsCfg<2, 2, 4>> : conv_rowstack_kernel<RsCfg<2, 2, 1>>;
    return rps == 4 ? conv_rowstack_kernel<RsCfg<2, 1, 4>> : conv_rowstack_kernel<RsCfg<2, 1, 1>>;
}

}  // namespace

bool dlc_rowstack_ok(const dlcContext *ctx, const ConvProblem &pb) {
    if (const char *ev = std::getenv("DLC_TC_ROWSTACK"))
        if (std::atoi(ev) == 0) return false;
    return rowstack_plan(pb, ctx ? ctx->wpack_bytes : 0, nullptr, nullptr);
}

dlcStatus_t dlc_preload_rowstack() {
    cudaFuncAttributes a;
    for (int v = 1; v <= 2; ++v)
        for (int split = 0; split < 2; ++split)
            for (int rps = 1; rps <= 4; rps += 3)
                if (cudaFuncGetAttributes(&a, rowstack_kernel_for(v, split != 0, rps)) != cudaSuccess)
                    return DLC_STATUS_EXECUTION_FAILED;
    if (cudaFuncGetAttributes(&a, rowstack_pack_filters) != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlc_launch_rowstack(dlcContext *ctx, const ConvProblem &pb) {
    RsParams p;
    size_t smem = 0;
    if (!ctx->wpack || !rowstack_plan(pb, ctx->wpack_bytes, &p, &smem)) return DLC_STATUS_INTERNAL_ERROR;
    for (int i = 0; i < 4; ++i) {
        p.xs[i] = pb.xs[i];
        p.ys[i] = pb.ys[i];
    }
    p.x = static_cast<const float *>(pb.x);
    {
        const long long end = ((long long)(pb.N - 1) * pb.xs[0] + (long long)(pb.C - 1) * pb.xs[1] +
                               (long long)(pb.H - 1) * pb.xs[2] + pb.W) * 4;
        p.x_end16 = ((unsigned long long)(uintptr_t)pb.x + (unsigned long long)end) & ~15ull;
        p.x_beg16 = ((unsigned long long)(uintptr_t)pb.x + 15ull) & ~15ull;
    }
    p.y = pb.y;
    p.bias = pb.bias;
    p.alpha = pb.alpha;
    p.beta = pb.beta;
    p.relu = pb.relu;
    p.y_bf16 = pb.ydt == DLC_DATA_BFLOAT16;
    p.err = ctx->d_err;
    p.timeout_ns = ctx->timeout_ns;

    float *img = static_cast<float *>(ctx->wpack);
    // the packed image as {32 elements, K_pad filters, R rows, columns}; the
    // box takes J rows u apart (element stride u along the rows) and a
    // stage's columns, 128-byte swizzled
    CUtensorMap ta;
    std::memset(&ta, 0, sizeof(ta));
    const int slices = p.groups * p.acols;
    const cuuint64_t dim[4] = {32, (cuuint64_t)p.K_pad, (cuuint64_t)p.R_img, (cuuint64_t)slices};
    const cuuint64_t str[3] = {128, (cuuint64_t)p.K_pad * 128, (cuuint64_t)p.R_img * p.K_pad * 128};
    const cuuint32_t box[4] = {32, (cuuint32_t)p.K_pad, (cuuint32_t)(p.J * pb.u), (cuuint32_t)p.acols};
    const cuuint32_t estr[4] = {1, 1, (cuuint32_t)pb.u, 1};
    if (ctx->encode_tiled(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, img, dim, str, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return DLC_STATUS_EXECUTION_FAILED;
    {
        const long long total = (long long)slices * p.R_img * p.K_pad * 32;
        cudaLaunchConfig_t cfg;
        std::memset(&cfg, 0, sizeof(cfg));
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = dlc_pdl_enabled() ? 1 : 0;
        cfg.gridDim = dim3((unsigned)((total + 255) / 256), 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = ctx->stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, rowstack_pack_filters, p, static_cast<const float *>(pb.w),
                               (long long)pb.ws[0], (long long)pb.ws[1], (long long)pb.ws[2],
                               (long long)pb.ws[3], img) != cudaSuccess)
            return DLC_STATUS_EXECUTION_FAILED;
        ctx->launches += 1;
    }
    // the instance for the horizontal stride and for one or two warps per row
    // pair (a stage has 4 * NI pairs for 8 builder warps)
    const bool split = RS_CG * p.NI < RS_BUILD_WARPS;
    RsKernel kern = rowstack_kernel_for(p.v, split, p.rps);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return DLC_STATUS_EXECUTION_FAILED;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 0;
    cfg.gridDim = dim3((unsigned)std::max(1, std::min(p.units, ctx->sm_count)), 1, 1);
    cfg.blockDim = dim3(RS_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx->stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, p, ta) != cudaSuccess)
        return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}
