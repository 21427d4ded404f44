// conv_rowstack.cu -- forward convolution of layers with few filters and unit
// horizontal stride on channel-planar (NCHW) activations, TF32 on the sm_103a
// tensor cores, with the filters stacked over output rows as the MMA's M side.
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
//  * N = output pixels.  With 4-byte elements, output pixel q = 4a + b (b the
//    phase, a < ceil(Q/4)) reads x[q + s - pad_left], s < S: for a fixed phase
//    b the windows of consecutive a start 16 bytes apart in a copy of the
//    input row shifted by b - pad_left elements.  Such a copy is a K-major,
//    no-swizzle MMA operand (8-row core matrices of 16-byte rows, the next 4
//    window taps 16 bytes further), read in place -- no lowered row is built.
//    N = NI images x seg_a rows.
//  * K (reduction) = (channel, filter tap s) in chunks of 4 taps (S padded to
//    a multiple of 4); an MMA takes two chunks, which may belong to two
//    channels: its leading offset is then the distance between their copies.
//
// A work unit is (NI images, J output rows, two phases): two TMEM
// accumulators of N columns.  For every input row t and group of 4 channels a
// stage holds the filter slices (A: one TMA load of the packed filter image,
// 32-byte swizzled K-major, rows j read at filter row R-1-r = R-1-t+j*u by a
// strided box, out-of-range rows zero-filled) and the shifted copies of the
// 4 channels' input rows for both phases and all NI images (B).  One issuer
// warp stages each input row once, as a 16-byte-aligned superset, with bulk
// copies into a ring of three raw buffers two stages ahead, and loads the
// filter slices; eight builder warps repack the raw rows into the two phase
// copies.  A stage's full barrier counts the builders' arrivals and the
// issuer's, which carries the filter bytes.  Input rows outside the image
// contribute nothing and their stages are skipped.  Four epilogue warps read
// the accumulators and store y (alpha, beta*y, bias, ReLU) through its
// strides.  Every wait is bounded.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace {

using namespace dlc;

constexpr int RS_M = 128;            // MMA rows
constexpr int RS_CG = 4;             // channels per stage
constexpr int RS_PH = 4;             // phases: 16 bytes / 4-byte elements
constexpr int RS_BUILD_WARPS = 8;
constexpr int RS_PROD_WARPS = RS_BUILD_WARPS + 1;           // the copy issuer and the builders
constexpr int RS_THREADS = (RS_PROD_WARPS + 1 + 4) * 32;  // producers, MMA, epilogue
constexpr int RS_RAW = 3;            // raw-row buffers
constexpr int RS_RAW_LAG = 2;        // stages the raw copies run ahead
constexpr int RS_MAX_SMEM = 232448;
constexpr int RS_BAR_AREA = 1024;  // barriers, then the MMA descriptor table
constexpr int RS_MAX_MPG = 16;       // MMAs per stage and phase

struct RsParams {
    int N, C, H, W, K, R, S, P, Q;
    int pt, pl, u, dh;
    int J, K_pad;          // output rows per tile, filters per row block (J*K_pad = 128)
    int T;                 // input rows one tile spans
    int cpc;               // 4-tap chunks per channel: ceil(S/4)
    int mpg;               // MMAs per stage and phase: RS_CG*cpc/2
    int groups;            // channel groups: ceil(C/4)
    int qa;                // pixels per phase and row: ceil(Q/4)
    int seg_a, NI, Nmma;   // rows per image segment, images per tile, MMA N (multiple of 16)
    int copy_bytes;        // bytes of one shifted row copy (all NI images)
    int b_stage;           // bytes of one stage's B copies: 2 phases x 4 channels
    int a_stage;           // bytes of one stage's A slices: mpg x 4 KiB
    int raw_bytes;         // bytes of one staged input row (16-byte-aligned superset)
    int raw_stage;         // bytes of one of the RS_RAW raw-row buffers: 4 channels x NI rows
    int stages;
    int row_blocks, img_groups, tiles, units;
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

struct RsUnit {
    int g, pb, pass;
};

__device__ __forceinline__ RsUnit rs_unit(const RsParams &p, int u) {
    RsUnit w;
    w.pass = u & 1;
    const int t = u >> 1;
    w.pb = t % p.row_blocks;
    w.g = t / p.row_blocks;
    return w;
}

// True when tile row t of row block pb is an input row inside the image.
__device__ __forceinline__ bool rs_row_in(const RsParams &p, int pb, int t) {
    const int h = pb * p.J * p.u - p.pt + t;
    return h >= 0 && h < p.H;
}

// The stages a CTA walks: its units in order; within a unit the input rows t
// inside the image, and for each the channel groups.
struct RsWalk {
    int u, t, cg;
    bool valid;
    __device__ void first(const RsParams &p) {
        u = blockIdx.x;
        t = 0;
        cg = 0;
        valid = u < p.units;
        settle(p);
    }
    __device__ void settle(const RsParams &p) {  // skip rows outside the image
        while (valid && !rs_row_in(p, rs_unit(p, u).pb, t)) {
            if (++t == p.T) {
                t = 0;
                u += gridDim.x;
                valid = u < p.units;
            }
        }
    }
    __device__ void next(const RsParams &p) {
        if (++cg < p.groups) return;
        cg = 0;
        if (++t == p.T) {
            t = 0;
            u += gridDim.x;
            valid = u < p.units;
        }
        settle(p);
    }
};

// Global address of input row (n, c, h) of a stage's (channel slot, image slot).
__device__ __forceinline__ const float *rs_row_ptr(const RsParams &p, const RsUnit &w, int t, int cg,
                                                   int cl, int ii, bool &in) {
    const int n = w.g * p.NI + ii, c = cg * RS_CG + cl;
    const int h = w.pb * p.J * p.u - p.pt + t;
    in = n < p.N && c < p.C;
    return p.x + (long long)(in ? n : 0) * p.xs[0] + (long long)(in ? c : 0) * p.xs[1] + (long long)h * p.xs[2];
}

// Thread 0: bulk-copies the stage's input rows (RS_CG channels x NI images)
// into raw buffer `rb`, each as the 16-byte-aligned superset of its bytes at
// slot (cl*NI + ii)*raw_bytes, completing on `bar`.
__device__ void rs_copy_raw(const RsParams &p, uint32_t rb, const RsWalk &st, uint64_t *bar) {
    uint32_t total = 0;
    const RsUnit w = rs_unit(p, st.u);
    for (int pass = 0; pass < 2; ++pass) {
        if (pass == 1) mbar_arrive_expect_tx(bar, total);
        for (int cl = 0; cl < RS_CG; ++cl)
            for (int ii = 0; ii < p.NI; ++ii) {
                bool in;
                const float *src = rs_row_ptr(p, w, st.t, st.cg, cl, ii, in);
                if (!in) continue;
                const uintptr_t a = reinterpret_cast<uintptr_t>(src);
                const unsigned long long a16 = a & ~15ull;
                const unsigned long long beg = std::max<unsigned long long>(a16, p.x_beg16);
                const unsigned long long end = std::min<unsigned long long>(
                    (a + 4ull * (unsigned long long)p.W + 15ull) & ~15ull, p.x_end16);
                if (end <= beg) continue;  // the row lies in the first or last 16 bytes of x
                const uint32_t bytes = (uint32_t)(end - beg);
                if (pass == 0)
                    total += bytes;
                else
                    bulk_load_1d(rb + (uint32_t)((cl * p.NI + ii) * p.raw_bytes) + (uint32_t)(beg - a16),
                                 reinterpret_cast<const void *>(beg), bytes, bar);
            }
    }
}

// The shifted row copies of one stage from its raw rows: for phase slot ph
// (phase b = 2*pass + ph), channel slot cl and image slot ii, row a of the
// copy holds x[n, c, h, 4a + b - pl + l], l < 4 (zero outside the row, past C
// or N).  Warp w builds the copies of (cl, ii) = w, w + 8, ..., both phases,
// one row per lane and step: the 5 elements both phases' chunks take lie in
// two aligned 16-byte words of the raw row; rows past the last image segment
// (read only for unstored outputs) are zeros.
__device__ void rs_build_b(const RsParams &p, uint32_t sb, uint32_t rb, const RsUnit &w, int t, int cg,
                           int warp, int lane) {
    const int combos = RS_CG * p.NI;
    const int tail = p.Nmma + p.cpc - 1;  // rows the MMAs read per copy
    const int b0 = 2 * w.pass;
    for (int cmb = warp; cmb < combos; cmb += RS_BUILD_WARPS) {
        const int ii = cmb % p.NI;
        const int cl = cmb / p.NI;
        bool in;
        const float *src = rs_row_ptr(p, w, t, cg, cl, ii, in);
        const uintptr_t ra = reinterpret_cast<uintptr_t>(src);
        const uint32_t slot = rb + (uint32_t)((cl * p.NI + ii) * p.raw_bytes);
        const int sh = (int)((ra & 15u) >> 2);  // element e of the row is word sh + e of the slot
        // elements [e_lo, avail) are in the copy (the first and last rows of x
        // may start before or end after it; those elements come from x)
        const unsigned long long cbeg = std::max<unsigned long long>(ra & ~15ull, p.x_beg16);
        const unsigned long long cend = std::min<unsigned long long>((ra + 4ull * p.W + 15ull) & ~15ull, p.x_end16);
        const int e_lo = cbeg > ra ? (int)((cbeg - ra + 3) / 4) : 0;
        const int avail = cend > ra ? (int)std::min<unsigned long long>((unsigned long long)p.W, (cend - ra) / 4) : 0;
        const uint32_t dst0 = sb + (uint32_t)(cl * p.copy_bytes);
        const uint32_t dst1 = sb + (uint32_t)((RS_CG + cl) * p.copy_bytes);
        const int r0 = ii * p.seg_a;
        const int r1 = ii == p.NI - 1 ? tail : r0 + p.seg_a;
        for (int row = r0 + lane; row < r1; row += 32) {
            const int a = row - r0;
            const int e0 = 4 * a + b0 - p.pl;  // phase b0 takes e0 .. e0+3, b0+1 takes e0+1 .. e0+4
            uint32_t el[5] = {0u, 0u, 0u, 0u, 0u};
            if (in && a < p.seg_a) {
                if (e0 >= e_lo && e0 + 4 < avail) {
                    const int wd = sh + e0;
                    const uint32_t base = slot + 16u * (uint32_t)(wd >> 2);
                    uint32_t q[8];
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]) : "r"(base));
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7]) : "r"(base + 16u));
                    const int o = wd & 3;
#pragma unroll
                    for (int l = 0; l < 5; ++l)
                        el[l] = o == 0 ? q[l] : (o == 1 ? q[l + 1] : (o == 2 ? q[l + 2] : q[l + 3]));
                } else {
#pragma unroll
                    for (int l = 0; l < 5; ++l) {
                        const int e = e0 + l;
                        if (e >= e_lo && e < avail)
                            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(el[l]) : "r"(slot + 4u * (uint32_t)(sh + e)));
                        else if (e >= 0 && e < p.W)
                            el[l] = __float_as_uint(__ldg(src + e));
                    }
                }
            }
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst0 + 16u * (uint32_t)row), "r"(el[0]),
                         "r"(el[1]), "r"(el[2]), "r"(el[3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst1 + 16u * (uint32_t)row), "r"(el[1]),
                         "r"(el[2]), "r"(el[3]), "r"(el[4])
                         : "memory");
        }
    }
}

// Warp 0 lane 0 issues the copies: the raw rows of up to stage k + 2 (a ring
// of three raw buffers, each freed by the builders), then the filter slices
// of stage k (one TMA box: J rows u apart from packed row R-1-t on, the
// slices of the stage's channel group).  Warps 1..8 build the stage's shifted
// row copies from its raw rows and arrive on its full barrier (which also
// takes the filter bytes).
__device__ void rs_issue(const RsParams &p, const CUtensorMap *tmA, uint32_t sA, uint32_t sRaw,
                         uint64_t *empty, uint64_t *full, uint64_t *rawfull, uint64_t *rawempty,
                         const WaitCtl &ctl) {
    const int ST = p.stages;
    volatile int no_abort = 0;
    const WaitCtl drain{&no_abort, p.err, p.timeout_ns};
    RsWalk a, r;  // the stage whose filters come next, and whose raw rows come next
    a.first(p);
    r = a;
    int kr = 0, stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int k = 0; ok && a.valid; ++k) {
        // raw rows up to stage k + RS_RAW_LAG, each into a buffer the builders freed
        while (ok && r.valid && kr <= k + RS_RAW_LAG) {
            if (kr >= RS_RAW)
                ok = mbar_wait(&rawempty[kr % RS_RAW], (uint32_t)((kr / RS_RAW) - 1) & 1u, ctl, 36);
            if (!ok) break;
            fence_proxy_async_smem();
            rs_copy_raw(p, sRaw + (uint32_t)(kr % RS_RAW) * (uint32_t)p.raw_stage, r, &rawfull[kr % RS_RAW]);
            ++kr;
            r.next(p);
        }
        if (!ok) break;
        ok = mbar_wait(&empty[stage], ph ^ 1u, ctl, 31);
        if (!ok) break;
        // the issuer's arrival carries the filter bytes, so the stage cannot
        // complete on the builders' arrivals alone
        mbar_arrive_expect_tx(&full[stage], (uint32_t)p.a_stage);
        tma_load_4d_u32(sA + (uint32_t)stage * p.a_stage, tmA, &full[stage], 0, 0, p.R - 1 - a.t,
                        a.cg * p.mpg);
        if (++stage == ST) stage = 0, ph ^= 1u;
        a.next(p);
    }
    // no copy may land after the CTA exits: wait for each raw buffer's last copy
    for (int j = kr > RS_RAW ? kr - RS_RAW : 0; j < kr; ++j)
        mbar_wait(&rawfull[j % RS_RAW], (uint32_t)(j / RS_RAW) & 1u, drain, 93);
}

__device__ void rs_build(const RsParams &p, uint32_t sB, uint32_t sRaw, uint64_t *full, uint64_t *empty,
                         uint64_t *rawfull, uint64_t *rawempty, const WaitCtl &ctl) {
    const int warp = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
    const int ST = p.stages;
    int stage = 0;
    uint32_t ph = 0;
    RsWalk cur;
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
        rs_build_b(p, sB + (uint32_t)stage * p.b_stage, sRaw + (uint32_t)(k % RS_RAW) * (uint32_t)p.raw_stage,
                   rs_unit(p, cur.u), cur.t, cur.cg, warp, lane);
        fence_proxy_async_smem();  // the copies, for the tensor core
        mbar_arrive(&full[stage]);
        mbar_arrive(&rawempty[k % RS_RAW]);
        if (++stage == ST) stage = 0, ph ^= 1u;
        cur.next(p);
    }
}

__device__ void rs_mma(const RsParams &p, uint32_t tmem_base, uint32_t sA, uint32_t sB, uint64_t *full,
                       uint64_t *empty, uint64_t *tfull, uint64_t *tempty, uint64_t *mma_done,
                       volatile uint64_t *dtab, const WaitCtl &ctl) {
    const int ST = p.stages;
    // A: 32-byte swizzled K-major slices of 128 rows x 32 bytes (8-row groups 256 bytes apart)
    const uint64_t a_hi = (1ull << 16) | ((uint64_t)(256 >> 4) << 32) | (1ull << 46) | (6ull << 61);
    // B: no swizzle, 16-byte rows, 8-row core matrices 128 bytes apart; the
    // leading offset (second chunk) per MMA
    const uint64_t b_hi = ((uint64_t)(128 >> 4) << 32) | (1ull << 46);
    // the stage-0 descriptors of every MMA of a stage, in shared memory
    for (int i = 0; i < p.mpg; ++i) {
        dtab[i] = a_hi | (uint64_t)(((sA + 4096u * (uint32_t)i) >> 4) & 0x3FFFu);
        for (int q = 0; q < 2; ++q)
            dtab[RS_MAX_MPG * (1 + q) + i] =
                b_hi | (uint64_t)(((sB + (uint32_t)(q * RS_CG * p.copy_bytes) + p.b_off[i]) >> 4) & 0x3FFFu) |
                ((uint64_t)((p.b_lbo[i] >> 4) & 0x3FFFu) << 16);
    }
    int stage = 0, it = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x, ++it) {
        const RsUnit w = rs_unit(p, u);
        if (!mbar_wait(&tempty[0], (uint32_t)(it & 1) ^ 1u, ctl, 33)) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        uint32_t acc = 0;
        for (int t = 0; ok && t < p.T; ++t) {
            if (!rs_row_in(p, w.pb, t)) continue;
            for (int cg = 0; cg < p.groups; ++cg) {
                if (!mbar_wait(&full[stage], ph, ctl, 34)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                // start fields move by whole stages (addresses below 256 KiB: no carry)
                const uint64_t ao = (uint64_t)(((uint32_t)stage * (uint32_t)p.a_stage) >> 4);
                const uint64_t bo = (uint64_t)(((uint32_t)stage * (uint32_t)p.b_stage) >> 4);
#pragma unroll 1
                for (int q = 0; q < 2; ++q) {
                    const uint32_t d = tmem_base + (uint32_t)(q * p.Nmma);
                    const volatile uint64_t *bt = dtab + RS_MAX_MPG * (1 + q);
#pragma unroll 1
                    for (int i = 0; i < p.mpg; ++i) {
                        // the unit's first MMA into each accumulator starts it
                        umma_tf32_nc(d, dtab[i] + ao, bt[i] + bo, p.idesc, (acc | (uint32_t)i) ? 1u : 0u);
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

__device__ void rs_epilogue(const RsParams &p, uint32_t tmem_base, uint64_t *tfull, uint64_t *tempty,
                            const WaitCtl &ctl) {
    // a warp reads the TMEM lanes of its index modulo 4
    const int quad = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
    const int row = quad * 32 + lane;  // MMA row (j, k)
    const int j = row / p.K_pad, k = row - (row / p.K_pad) * p.K_pad;
    float *yf = static_cast<float *>(p.y);
    unsigned short *yb = static_cast<unsigned short *>(p.y);
    int it = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++it) {
        const RsUnit w = rs_unit(p, u);
        int okw = 0;
        if (lane == 0) okw = mbar_wait(&tfull[0], (uint32_t)(it & 1), ctl, 35) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) break;
        __syncwarp();
        tc_fence_after_sync();
        const int op = w.pb * p.J + j;
        const bool row_ok = k < p.K && op < p.P;
        const float bias = (row_ok && p.bias) ? __ldg(p.bias + k) : 0.f;
        for (int q2 = 0; q2 < 2; ++q2) {
            const int b = 2 * w.pass + q2;
            for (int c0 = 0; c0 < p.Nmma; c0 += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(q2 * p.Nmma + c0), v);
                tmem_ld_wait();
                if (!row_ok) continue;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int col = c0 + e;
                    const int ii = col / p.seg_a, a = col - ii * p.seg_a;
                    const int n = w.g * p.NI + ii;
                    const int oq = 4 * a + b;
                    if (ii >= p.NI || n >= p.N || a >= p.qa || oq >= p.Q) continue;
                    const long long yo = (long long)n * p.ys[0] + (long long)k * p.ys[1] +
                                         (long long)op * p.ys[2] + (long long)oq * p.ys[3];
                    float f = p.alpha * __uint_as_float(v[e]);
                    if (p.beta != 0.f) f = __fmaf_rn(p.beta, p.y_bf16 ? rs_bf16_to_f32(yb[yo]) : yf[yo], f);
                    f += bias;
                    if (p.relu) f = fmaxf(f, 0.f);
                    if (p.y_bf16)
                        yb[yo] = __bfloat16_as_ushort(__float2bfloat16_rn(f));
                    else
                        yf[yo] = f;
                }
            }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[0]);
    }
}

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
    if (warp == RS_PROD_WARPS) {
        tmem_alloc(tmem_slot, p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtl ctl{abort_flag, p.err, p.timeout_ns};
    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tmA);
            rs_issue(p, &tmA, smem_u32(smA), smem_u32(smRaw), empty, full, rawfull, rawempty, ctl);
        }
    } else if (warp < RS_PROD_WARPS) {
        rs_build(p, smem_u32(smB), smem_u32(smRaw), full, empty, rawfull, rawempty, ctl);
    } else if (warp == RS_PROD_WARPS) {
        if (lane == 0)
            rs_mma(p, tmem_base, smem_u32(smA), smem_u32(smB), full, empty, tfull, tempty, mma_done,
                   reinterpret_cast<volatile uint64_t *>(reinterpret_cast<uint8_t *>(bars) + 256), ctl);
    } else {
        rs_epilogue(p, tmem_base, tfull, tempty, ctl);
    }
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == RS_PROD_WARPS) tmem_dealloc(tmem_base, p.tmem_cols);
}

// The filters as MMA A slices, in the order the convolution's TMA box reads
// them: image [m][rr][k][8] (m = MMA slice over (channel group, MMA), rr =
// R-1-r, k < K_pad filters, 8 reduction elements), each element the filter
// tap of its (channel, s) chunk or zero.  One thread per element.
__global__ void rowstack_pack_filters(const __grid_constant__ RsParams p, const float *w, long long ws0,
                                      long long ws1, long long ws2, long long ws3, float *img) {
    griddep_wait();  // the previous convolution may still read the image
    griddep_launch_dependents();
    const long long total = (long long)p.groups * p.mpg * p.R * p.K_pad * 8;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int e = (int)(i & 7);
    long long t = i >> 3;
    const int k = (int)(t % p.K_pad);
    t /= p.K_pad;
    const int rr = (int)(t % p.R);
    const int m = (int)(t / p.R);
    const int cg = m / p.mpg, mi = m - cg * p.mpg;
    const int chunk = 2 * mi + (e >> 2);
    const int c = cg * RS_CG + chunk / p.cpc;
    const int s = 4 * (chunk % p.cpc) + (e & 3);
    const int r = p.R - 1 - rr;
    float v = 0.f;
    if (k < p.K && c < p.C && s < p.S)
        v = __ldg(w + (long long)k * ws0 + (long long)c * ws1 + (long long)r * ws2 + (long long)s * ws3);
    img[i] = v;
}

// Plan: every field but the pointers.  False when the kernel does not take
// the problem.
bool rowstack_plan(const ConvProblem &pb, size_t wpack_bytes, RsParams *out, size_t *smem_out) {
    if (pb.math != DLC_MATH_TF32 || pb.xdt != DLC_DATA_FLOAT) return false;
    if (pb.xs[3] != 1 || pb.v != 1 || pb.dw != 1 || pb.dh != 1) return false;
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
    p.pt = pb.pt; p.pl = pb.pl; p.u = pb.u; p.dh = pb.dh;
    p.K_pad = pb.K <= 32 ? 32 : 64;
    p.J = RS_M / p.K_pad;
    p.T = (p.J - 1) * pb.u + (pb.R - 1) * pb.dh + 1;
    p.cpc = (pb.S + 3) / 4;
    if ((RS_CG * p.cpc) % 2) return false;
    p.mpg = RS_CG * p.cpc / 2;
    if (p.mpg > RS_MAX_MPG) return false;
    p.groups = (pb.C + RS_CG - 1) / RS_CG;
    p.qa = (pb.Q + RS_PH - 1) / RS_PH;
    p.seg_a = ((p.qa + p.cpc - 1 + 7) / 8) * 8;
    if (p.seg_a > 256) return false;
    p.NI = std::max(1, std::min(pb.N, 256 / p.seg_a));
    p.Nmma = ((p.NI * p.seg_a + 15) / 16) * 16;
    if (p.Nmma > 256) return false;
    p.copy_bytes = (p.Nmma + p.cpc - 1) * 16;
    p.copy_bytes = ((p.copy_bytes + 127) / 128) * 128;
    p.b_stage = 2 * RS_CG * p.copy_bytes;
    p.a_stage = p.mpg * 4096;
    p.raw_bytes = ((pb.W * 4 + 15 + 15) / 16) * 16;
    p.raw_stage = RS_CG * p.NI * p.raw_bytes;
    const int stage = p.a_stage + p.b_stage;
    p.stages = std::min(8, (RS_MAX_SMEM - 1024 - RS_BAR_AREA - RS_RAW * p.raw_stage) / stage);
    if (p.stages < 2) return false;
    // MMA i of a stage takes chunks 2i and 2i+1 of the group's (channel, chunk)
    // sequence; chunk ch of channel slot ch / cpc sits in that channel's copy
    for (int i = 0; i < p.mpg; ++i) {
        auto addr = [&](int ch) { return (uint32_t)((ch / p.cpc) * p.copy_bytes + 16 * (ch % p.cpc)); };
        p.b_off[i] = addr(2 * i);
        p.b_lbo[i] = addr(2 * i + 1) - addr(2 * i);
    }
    p.row_blocks = (pb.P + p.J - 1) / p.J;
    p.img_groups = (pb.N + p.NI - 1) / p.NI;
    const long long tiles = (long long)p.row_blocks * p.img_groups;
    if (tiles * 2 > 0x7fffffffLL) return false;
    p.tiles = (int)tiles;
    p.units = 2 * p.tiles;
    const long long img = (long long)p.groups * p.mpg * pb.R * p.K_pad * 32;
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
    if (smem_out) *smem_out = 1024 + (size_t)p.stages * stage + RS_RAW * (size_t)p.raw_stage + RS_BAR_AREA;
    return true;
}

}  // namespace

bool dlc_rowstack_ok(const dlcContext *ctx, const ConvProblem &pb) {
    if (const char *ev = std::getenv("DLC_TC_ROWSTACK"))
        if (std::atoi(ev) == 0) return false;
    return rowstack_plan(pb, ctx ? ctx->wpack_bytes : 0, nullptr, nullptr);
}

dlcStatus_t dlc_preload_rowstack() {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, conv_rowstack_kernel) != cudaSuccess ||
        cudaFuncGetAttributes(&a, rowstack_pack_filters) != cudaSuccess)
        return DLC_STATUS_EXECUTION_FAILED;
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
    // the packed image as {8 elements, K_pad filters, R rows, slices}; the
    // box takes J rows u apart (element stride u along the rows) and a
    // stage's mpg slices, 32-byte swizzled
    CUtensorMap ta;
    std::memset(&ta, 0, sizeof(ta));
    const int slices = p.groups * p.mpg;
    const cuuint64_t dim[4] = {8, (cuuint64_t)p.K_pad, (cuuint64_t)pb.R, (cuuint64_t)slices};
    const cuuint64_t str[3] = {32, (cuuint64_t)p.K_pad * 32, (cuuint64_t)pb.R * p.K_pad * 32};
    const cuuint32_t box[4] = {8, (cuuint32_t)p.K_pad, (cuuint32_t)(p.J * pb.u), (cuuint32_t)p.mpg};
    const cuuint32_t estr[4] = {1, 1, (cuuint32_t)pb.u, 1};
    if (ctx->encode_tiled(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, img, dim, str, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return DLC_STATUS_EXECUTION_FAILED;
    {
        const long long total = (long long)slices * pb.R * p.K_pad * 8;
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
    if (cudaFuncSetAttribute(conv_rowstack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
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
    if (cudaLaunchKernelEx(&cfg, conv_rowstack_kernel, p, ta) != cudaSuccess)
        return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}
