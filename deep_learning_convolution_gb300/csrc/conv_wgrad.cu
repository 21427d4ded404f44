// conv_wgrad.cu -- the filter gradient on the tensor cores.
//
//   dw[k,c,r,s] = alpha * sum_{n,p,q} dy[n,k,p,q] * X(n, c, p*u + r*dh - pad_top,
//                                                       q*v + s*dw - pad_left)
//                 + beta * dw[k,c,r,s]
//
// (the cuDNN page's method section: routines for the backward pass; the
// batch-reduce GEMM page's method section: one GEMM building block, here
// with the output pixels as the reduction).  For each filter tap (r, s) the
// sum is a GEMM D[k, c] += A[k, m] * B[c, m] over the output pixels m = (n, p,
// q): A is dy with its filters contiguous (channels-innermost storage, so an
// MN-major operand), B is the tap's im2col view of x with its channels
// contiguous (also MN-major).  TMA brings both in 128-byte-swizzled blocks of
// 64 pixels: dy through a 2-D [pixels, filters] map, x through the same im2col
// map as the forward kernels (filter-tap offsets, padding from the bounding
// box, strides as traversal steps), so pixel m of A and of B is the same
// output pixel.
//
// A work unit is (128 filters, BN channels, one tap, a range of pixel blocks).
// A pair with at most 128 channels stacks two taps instead: each CTA loads all
// channels of its own tap (2r and 2r + 1 of the unit's tap pair r), so one MMA
// of N = 2 x 64 x ceil(C/64) serves both taps from one dy block, where one tap
// per unit would pad N to 128 channels per tap and load dy once per tap.
// The pixel reduction is split into ranges when the tiles alone cannot fill
// the GPU; every unit adds alpha times its partial sum into dw with bulk
// tensor reduce-adds (dw scaled by beta beforehand), so the split's partial
// sums meet in FP32 atomic adds (a deterministic handle keeps one range per
// tile, whose single add per element has a fixed order).
//
// Roles (one CTA per SM, 6 warps): warp 0 lane 0 issues the TMA loads; warp 1
// lane 0 the tcgen05.mma (M = 128, N = BN, K = 16 per instruction, both
// operands MN-major) into one of two TMEM accumulators; warps 2-5 read the
// accumulator, scale it by alpha, stage 32 x 32 blocks in shared memory and
// reduce-add them into dw.  Every wait is bounded.
//
// With more than 128 filters the CTAs work in pairs (a cluster of two, as the
// forward pair kernel): one MMA of M = 256 filters (128 per CTA, each from its
// own dy block) and N = BN channels, of which each CTA loads half of the x
// block.  Per SM a k-block then moves 16 KiB of dy and BN/2 x 128 bytes of x
// instead of BN x 128: a single CTA at BN = 256 moves 48 KiB per 680 cycles of
// MMAs, more than the SM takes in.  Both CTAs' loads complete on the leader's
// barrier; the leader issues the MMAs and commits to both CTAs' barriers; each
// CTA's epilogue adds its 128 filter rows and releases the accumulator on the
// leader's barrier.
#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace {

using namespace dlc;

constexpr int WG_BM = 128;                 // filters per tile
constexpr int WG_BP = 64;                  // pixels per k-block
constexpr int WG_ATOM = 64 * 128;          // one 128-byte x 64-row swizzled block: 8 KiB
constexpr int WG_A_BYTES = 2 * WG_ATOM;    // 128 filters x 64 pixels (BF16)
constexpr int WG_THREADS = 192;
constexpr int WG_MAX_SMEM = 232448;
constexpr int WG_BAR_AREA = 256;
constexpr int WG_EPI_BUF = 32 * 128;              // 32 filters x 32 FP32 channels
constexpr int WG_EPI_SMEM = 4 * 2 * WG_EPI_BUF;   // 4 epilogue warps, double-buffered

struct WgParams {
    int N, C, H, W, K, R, S, P, Q;
    int pt, pl, u, v, dh, dw;
    long long M;       // N*P*Q pixels
    int PQ;
    int BN, b_atoms, stages;
    int m_tiles, c_tiles, tiles;   // tiles = m_tiles * c_tiles * R * S
    int kblocks;                   // ceil(M / 64)
    int splits, units;             // pixel-block ranges per tile; units = tiles * splits
    int stack;                     // pairs: each CTA's x block is a different tap (below)
    int dn, dp, dq;                // one pixel block (64 pixels) as images, rows, columns
    float alpha;
    uint32_t idesc, tmem_cols, acc_stride;
    int *err;
    unsigned long long timeout_ns;
};

struct WgUnit {
    int kt, ct, rs, kb0, kb1;
};

__device__ __forceinline__ WgUnit wg_unit(const WgParams &p, int u) {
    WgUnit w;
    const int t = u / p.splits, sp = u - (u / p.splits) * p.splits;
    w.kt = t % p.m_tiles;
    const int t2 = t / p.m_tiles;
    w.ct = t2 % p.c_tiles;
    w.rs = t2 / p.c_tiles;
    w.kb0 = (int)((long long)p.kblocks * sp / p.splits);
    w.kb1 = (int)((long long)p.kblocks * (sp + 1) / p.splits);
    return w;
}

// The first work unit of this CTA (or pair) and the step to its next.
template <bool PAIR>
__device__ __forceinline__ int wg_first() { return PAIR ? (int)cluster_id_x() : (int)blockIdx.x; }
template <bool PAIR>
__device__ __forceinline__ int wg_step() { return PAIR ? (int)num_clusters_x() : (int)gridDim.x; }

template <bool PAIR>
__device__ void wg_produce(const WgParams &p, uint32_t rank, const CUtensorMap *tmA, const CUtensorMap *tmB,
                           uint32_t sA, uint32_t sB, uint64_t *full, uint64_t *empty,
                           const WaitCtl &ctl) {
    const int ST = p.stages;
    const uint32_t b_bytes = (uint32_t)p.b_atoms * WG_ATOM;
    // a pair's stage completes on the leader's barrier with both CTAs' bytes
    const uint32_t tx = (PAIR ? 2u : 1u) * (WG_A_BYTES + b_bytes);
    const uint32_t full0 = PAIR ? mapa_shared(smem_u32(full), 0) : 0u;
    int stage = 0;
    uint32_t ph = 0;
    for (int u = wg_first<PAIR>(); u < p.units; u += wg_step<PAIR>()) {
        const WgUnit w = wg_unit(p, u);
        // stacked taps: this CTA's tap of the pair (the last tap again when
        // R*S is odd; the epilogue drops its columns)
        const int tap = p.stack ? min(2 * w.rs + (int)rank, p.R * p.S - 1) : w.rs;
        const int r = tap / p.S, s = tap - (tap / p.S) * p.S;
        const int k0 = w.kt * (PAIR ? 2 * WG_BM : WG_BM) + (int)rank * WG_BM;
        const int c0 = p.stack ? 0 : w.ct * p.BN + (int)rank * (p.b_atoms * 64);
        // the first pixel of the unit's first block; later blocks step by 64
        // pixels without a division
        long long m0 = (long long)w.kb0 * WG_BP;
        int n0 = (int)(m0 / p.PQ);
        int p0, q0;
        {
            const int rem = (int)(m0 - (long long)n0 * p.PQ);
            p0 = rem / p.Q;
            q0 = rem - p0 * p.Q;
        }
        for (int kb = w.kb0; kb < w.kb1; ++kb, m0 += WG_BP) {
            if (!mbar_wait(&empty[stage], ph ^ 1u, ctl, 11)) return;
            if (!PAIR || rank == 0) mbar_arrive_expect_tx(&full[stage], tx);
            const uint32_t a = sA + (uint32_t)stage * WG_A_BYTES;
            const uint32_t b = sB + (uint32_t)stage * b_bytes;
            if constexpr (PAIR) {
                const uint32_t fb = full0 + 8u * (uint32_t)stage;
                tma_load_2d_pair(a, tmA, fb, k0, (int)m0);
                tma_load_2d_pair(a + WG_ATOM, tmA, fb, k0 + 64, (int)m0);
                for (int at = 0; at < p.b_atoms; ++at)
                    tma_load_im2col_4d_pair(b + (uint32_t)at * WG_ATOM, tmB, fb, c0 + at * 64,
                                            q0 * p.v - p.pl, p0 * p.u - p.pt, n0, (uint16_t)(s * p.dw),
                                            (uint16_t)(r * p.dh));
            } else {
                tma_load_2d(a, tmA, &full[stage], k0, (int)m0);
                tma_load_2d(a + WG_ATOM, tmA, &full[stage], k0 + 64, (int)m0);
                for (int at = 0; at < p.b_atoms; ++at)
                    tma_load_im2col_4d(b + (uint32_t)at * WG_ATOM, tmB, &full[stage], c0 + at * 64,
                                       q0 * p.v - p.pl, p0 * p.u - p.pt, n0, (uint16_t)(s * p.dw),
                                       (uint16_t)(r * p.dh));
            }
            q0 += p.dq;
            p0 += p.dp;
            n0 += p.dn;
            if (q0 >= p.Q) q0 -= p.Q, ++p0;
            if (p0 >= p.P) p0 -= p.P, ++n0;
            if (++stage == ST) stage = 0, ph ^= 1u;
        }
    }
}

template <bool PAIR>
__device__ void wg_mma(const WgParams &p, uint32_t tmem_base, uint32_t sA, uint32_t sB,
                       uint64_t *full, uint64_t *empty, uint64_t *tfull, uint64_t *tempty,
                       uint64_t *mma_done, const WaitCtl &ctl) {
    const int ST = p.stages;
    const uint32_t b_bytes = (uint32_t)p.b_atoms * WG_ATOM;
    // both operands MN-major: 128-byte rows of 64 filters / channels per
    // pixel, 8-pixel groups 1024 bytes apart, the next 64 filters / channels
    // one 8 KiB block further; an MMA's 16 pixels are 2048 bytes
    const uint64_t a0 = sw128_mnmajor_desc(sA, WG_ATOM), b0 = sw128_mnmajor_desc(sB, WG_ATOM);
    const uint64_t a_step = WG_A_BYTES >> 4, b_step = b_bytes >> 4;
    int stage = 0, it = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int u = wg_first<PAIR>(); ok && u < p.units; u += wg_step<PAIR>(), ++it) {
        const WgUnit w = wg_unit(p, u);
        const int buf = it & 1;
        const uint32_t aph = (uint32_t)(it >> 1) & 1u;
        // (pairs: both CTAs' epilogues arrive, the other one remotely)
        if (!(PAIR ? mbar_wait_cluster(&tempty[buf], aph ^ 1u, ctl, 13)
                   : mbar_wait(&tempty[buf], aph ^ 1u, ctl, 13))) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        const uint32_t d = tmem_base + (uint32_t)buf * p.acc_stride;
        uint64_t ad = a0 + a_step * stage, bd = b0 + b_step * stage;
        uint32_t acc = 0;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
            if (!mbar_wait(&full[stage], ph, ctl, 14)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
#pragma unroll
            for (int j = 0; j < WG_BP / 16; ++j) {
                if constexpr (PAIR)
                    umma_bf16_pair(d, ad + 128u * j, bd + 128u * j, p.idesc, acc);
                else
                    umma_bf16_nc(d, ad + 128u * j, bd + 128u * j, p.idesc, acc);
                acc = 1;
            }
            if (PAIR)
                umma_commit_pair(&empty[stage], 3);  // both CTAs' slots free once these are done
            else
                umma_commit(&empty[stage]);
            if (++stage == ST) {
                stage = 0;
                ph ^= 1u;
                ad = a0;
                bd = b0;
            } else {
                ad += a_step;
                bd += b_step;
            }
        }
        if (!ok) break;
        if (PAIR)
            umma_commit_pair(&tfull[buf], 3);  // both CTAs' accumulator rows are ready
        else
            umma_commit(&tfull[buf]);
    }
    if (!ok) {
        // loads issued for stages not consumed land on these barriers; wait
        // for them briefly so that no copy outlives the CTA
        volatile int dummy = 0;
        const WaitCtl brief{&dummy, p.err, 50000000ull};
        for (int j = 0; j < ST; ++j) {
            if (!mbar_wait(&full[stage], ph, brief, 97)) break;
            if (++stage == ST) stage = 0, ph ^= 1u;
        }
    }
    // every MMA issued must complete before tensor memory is released (the
    // kernel waits for this commit in both CTAs)
    if (PAIR)
        umma_commit_pair(mma_done, 3);
    else
        umma_commit(mma_done);
}

template <bool PAIR>
__device__ void wg_epilogue(const WgParams &p, uint32_t rank, uint32_t tmem_base, uint64_t *tfull,
                            uint64_t *tempty, uint32_t epi_smem, const CUtensorMap *tmD, const WaitCtl &ctl) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31: filters
    const uint32_t my_bufs = epi_smem + (uint32_t)(quad * 2 * WG_EPI_BUF);
    const uint32_t tempty0 = PAIR ? mapa_shared(smem_u32(tempty), 0) : 0u;  // the leader's barriers
    int nbuf = 0, it = 0;
    for (int u = wg_first<PAIR>(); u < p.units; u += wg_step<PAIR>(), ++it) {
        const WgUnit w = wg_unit(p, u);
        const int buf = it & 1;
        const uint32_t ph = (uint32_t)(it >> 1) & 1u;
        int okw = 0;
        if (lane == 0) okw = mbar_wait(&tfull[buf], ph, ctl, 15) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) break;
        __syncwarp();
        tc_fence_after_sync();
        const int krow = w.kt * (PAIR ? 2 * WG_BM : WG_BM) + (int)rank * WG_BM + quad * 32;
        const int c0 = w.ct * p.BN;
        const int half = p.b_atoms * 64;  // accumulator columns from each CTA's x block
        const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)buf * p.acc_stride;
        for (int cc = 0; cc < p.BN && (p.stack || c0 + cc < p.C); cc += 32) {
            int ch = c0 + cc, tap = w.rs;
            if (p.stack) {  // columns [0, half) are tap 2*rs, [half, BN) tap 2*rs + 1
                const int h = cc >= half ? 1 : 0;
                ch = cc - h * half;
                tap = 2 * w.rs + h;
                if (ch >= p.C || tap >= p.R * p.S) continue;  // warp-uniform
            }
            uint32_t v[32];
            tmem_ld_32x32b_x32(taddr + (uint32_t)cc, v);
            tmem_ld_wait();
            if (krow >= p.K) continue;  // every filter row of this warp is past K
            const uint32_t sb = my_bufs + (uint32_t)(nbuf & 1) * WG_EPI_BUF;
            if (nbuf >= 2) {  // the reduce issued from this buffer two groups ago
                if (lane == 0) bulk_wait_group_read<1>();
                __syncwarp();
            }
            const uint32_t rowp = sb + (uint32_t)lane * 128u;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(rowp + (((uint32_t)j ^ (lane & 7)) << 4)),
                             "f"(p.alpha * __uint_as_float(v[4 * j])), "f"(p.alpha * __uint_as_float(v[4 * j + 1])),
                             "f"(p.alpha * __uint_as_float(v[4 * j + 2])), "f"(p.alpha * __uint_as_float(v[4 * j + 3]))
                             : "memory");
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {  // channels past C and filters past K are not written
                tma_reduce_add_3d_s(tmD, sb, ch, tap, krow);
                bulk_commit_group();
            }
            ++nbuf;
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
            if (PAIR)
                mbar_arrive_tmem_free(tempty0 + 8u * (uint32_t)buf);  // release on the leader
            else
                mbar_arrive(&tempty[buf]);
        }
    }
    if (lane == 0) bulk_wait_group_read<0>();  // shared memory read before exit
    __syncwarp();
}

template <bool PAIR>
__global__ void __launch_bounds__(WG_THREADS, 1)
    conv_wgrad_kernel(const __grid_constant__ WgParams p, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmD) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);  // same offset in both CTAs
    const int ST = p.stages;
    const uint32_t b_bytes = (uint32_t)p.b_atoms * WG_ATOM;
    uint8_t *smA = smem;
    uint8_t *smB = smA + (size_t)ST * WG_A_BYTES;
    uint8_t *epi = smB + (size_t)ST * b_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(epi + WG_EPI_SMEM);
    uint64_t *full = bars;
    uint64_t *empty = bars + ST;
    uint64_t *tfull = bars + 2 * ST;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full[i], 1u);   // the (leader's) expect-tx arrival
            mbar_init(&empty[i], 1u);  // the (leader's) commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1u);
            mbar_init(&tempty[i], PAIR ? 8u : 4u);  // one arrival per epilogue warp (of both CTAs)
        }
        mbar_init(mma_done, 1u);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmD);
    }
    if (warp == 1) {
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
    if (warp == 0) {
        if (lane == 0) wg_produce<PAIR>(p, rank, &tmA, &tmB, smem_u32(smA), smem_u32(smB), full, empty, ctl);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0)
            wg_mma<PAIR>(p, tmem_base, smem_u32(smA), smem_u32(smB), full, empty, tfull, tempty, mma_done,
                         ctl);
        if (lane == 0) {  // the (leader's) final commit reaches this CTA
            volatile int dummy = 0;
            const WaitCtl fin{&dummy, p.err, p.timeout_ns};
            mbar_wait(mma_done, 0u, fin, 98);
        }
    } else {
        wg_epilogue<PAIR>(p, rank, tmem_base, tfull, tempty, smem_u32(epi), &tmD, ctl);
    }
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (PAIR) cluster_sync();  // neither CTA leaves while the pair's MMAs or loads may touch it
    tc_fence_after_sync();
    if (warp == 1) {
        if (PAIR)
            tmem_dealloc_pair(tmem_base, p.tmem_cols);
        else
            tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

// x channels-innermost with 16-byte strides, dy dense channels-innermost
// ([N*P*Q, K] rows at one pitch), dw KRSC FP32, BF16 math, TMA limits.
bool wgrad_tc_ok(const BwdProblem &bp) {
    if (bp.math != DLC_MATH_BF16 || bp.in_dt != DLC_DATA_BFLOAT16 || bp.out_dt != DLC_DATA_FLOAT)
        return false;
    if (bp.wfmt != DLC_TENSOR_NHWC) return false;
    if (bp.C < 64 || bp.C % 8 || bp.K % 8) return false;
    if (bp.xs[1] != 1 || bp.xs[3] < bp.C || bp.xs[2] < bp.xs[3] * (long long)bp.W ||
        bp.xs[0] < bp.xs[2] * (long long)bp.H)
        return false;
    for (int i : {0, 2, 3})
        if ((bp.xs[i] * 2) % 16 || bp.xs[i] * 2 >= (1LL << 40)) return false;
    if (bp.dys[1] != 1 || (bp.dys[3] * 2) % 16 || bp.dys[3] < bp.K) return false;
    if ((bp.P > 1 && bp.dys[2] != (long long)bp.Q * bp.dys[3]) ||
        (bp.N > 1 && bp.dys[0] != (long long)bp.P * bp.Q * bp.dys[3]))
        return false;
    if (bp.x && ((uintptr_t)bp.x % 16)) return false;
    if (bp.dy && ((uintptr_t)bp.dy % 16)) return false;
    if (bp.w && ((uintptr_t)bp.w % 16)) return false;
    if (bp.u > 8 || bp.v > 8) return false;
    const long long lo_w = -bp.pl, lo_h = -bp.pt;
    const long long up_w = bp.pr - (long long)bp.dw * (bp.S - 1);
    const long long up_h = bp.pb - (long long)bp.dh * (bp.R - 1);
    for (long long c : {lo_w, lo_h, up_w, up_h})
        if (c < -128 || c > 127) return false;
    if ((long long)bp.dw * (bp.S - 1) > 255 || (long long)bp.dh * (bp.R - 1) > 255) return false;
    const long long M = (long long)bp.N * bp.P * bp.Q;
    if (M > 0x7fffffffLL - 64) return false;
    if ((long long)bp.R * bp.S * bp.C * 4 >= (1LL << 40)) return false;
    return true;
}

}  // namespace

bool dlc_wgrad_tc_ok(const BwdProblem &bp) { return wgrad_tc_ok(bp); }

dlcStatus_t dlc_launch_wgrad_tc(dlcContext *ctx, const BwdProblem &bp) {
    WgParams p;
    std::memset(&p, 0, sizeof(p));
    p.N = bp.N; p.C = bp.C; p.H = bp.H; p.W = bp.W; p.K = bp.K; p.R = bp.R; p.S = bp.S;
    p.P = bp.P; p.Q = bp.Q;
    p.pt = bp.pt; p.pl = bp.pl; p.u = bp.u; p.v = bp.v; p.dh = bp.dh; p.dw = bp.dw;
    p.M = (long long)bp.N * bp.P * bp.Q;
    p.PQ = bp.P * bp.Q;
    // SM pairs once there are more filters than one CTA's 128 (DLC_TC_WGRAD_PAIR=0: single CTAs)
    const bool pair = bp.K > WG_BM && [] {
        const char *ev = std::getenv("DLC_TC_WGRAD_PAIR");
        return !(ev && std::atoi(ev) == 0);
    }();
    // channels per tile: the multiple of 64 (128 for a pair: each CTA loads
    // whole 64-channel blocks) up to 256 that pads C least (ties to the wider)
    p.BN = pair ? 128 : 64;
    long long best = -1;
    for (int bn : {256, 192, 128, 64}) {
        if (pair && bn % 128) continue;
        const long long pad = (long long)((bp.C + bn - 1) / bn) * bn - bp.C;
        if (best < 0 || pad < best) best = pad, p.BN = bn;
    }
    if (const char *ev = std::getenv("DLC_TC_WGRAD_BN")) {
        const int bn = std::atoi(ev);
        if (bn == 128 || bn == 256 || (!pair && (bn == 64 || bn == 192))) p.BN = bn;
    }
    p.b_atoms = (pair ? p.BN / 2 : p.BN) / 64;  // 64-channel blocks of x a CTA loads
    p.m_tiles = (bp.K + (pair ? 2 : 1) * WG_BM - 1) / ((pair ? 2 : 1) * WG_BM);
    p.c_tiles = (bp.C + p.BN - 1) / p.BN;
    p.tiles = p.m_tiles * p.c_tiles * bp.R * bp.S;
    // a pair with at most 128 channels stacks two taps (DLC_TC_WGRAD_STACK=0: one tap a unit)
    p.stack = pair && bp.C <= 128 && bp.R * bp.S >= 2 && [] {
        const char *ev = std::getenv("DLC_TC_WGRAD_STACK");
        return !(ev && std::atoi(ev) == 0);
    }();
    if (p.stack) {
        p.b_atoms = (bp.C + 63) / 64;
        p.BN = 2 * 64 * p.b_atoms;
        p.c_tiles = 1;
        p.tiles = p.m_tiles * ((bp.R * bp.S + 1) / 2);
    }
    p.kblocks = (int)((p.M + WG_BP - 1) / WG_BP);
    // split the pixel reduction where it shortens the busiest CTA (or pair):
    // s ranges of each tile make rounds(s) = ceil(tiles * s / workers) rounds of
    // units of kblocks / s k-blocks each, and a unit costs about ten k-blocks
    // more (its reduce-add epilogue and pipeline fill); the cheapest s, the
    // fewest ranges among equals, each range at least 16 k-blocks
    int splits = 1;
    if (!ctx->deterministic) {
        const long long workers = pair ? ctx->sm_count / 2 : ctx->sm_count;
        const int smax = std::max(1, std::min(32, p.kblocks / 16));
        double best = -1.0;
        for (int sp = 1; sp <= smax; ++sp) {
            const long long rounds = ((long long)p.tiles * sp + workers - 1) / workers;
            const double cost = (double)rounds * ((double)p.kblocks / sp + 10.0);
            if (best < 0 || cost < best - 1e-9) best = cost, splits = sp;
        }
    }
    p.splits = splits;
    p.dn = (int)(WG_BP / p.PQ);
    p.dp = (int)((WG_BP % p.PQ) / p.Q);
    p.dq = (int)((WG_BP % p.PQ) % p.Q);
    if ((long long)p.tiles * splits > 0x7fffffffLL) return DLC_STATUS_NOT_SUPPORTED;
    p.units = p.tiles * splits;
    p.alpha = (float)bp.alpha;
    const int stage_bytes = WG_A_BYTES + p.b_atoms * WG_ATOM;
    int st = (WG_MAX_SMEM - 1024 - WG_BAR_AREA - WG_EPI_SMEM - stage_bytes) / stage_bytes;
    p.stages = std::min(st, 8);
    if (p.stages < 2) return DLC_STATUS_INTERNAL_ERROR;
    // BF16 A and B, FP32 D, both operands MN-major (transpose bits 15, 16);
    // M = 256 for a pair (128 rows in each CTA)
    p.idesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
              ((uint32_t)(p.BN >> 3) << 17) | ((uint32_t)(((pair ? 2 : 1) * WG_BM) >> 4) << 24);
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * p.BN)) cols <<= 1;
    p.tmem_cols = cols;
    p.acc_stride = cols / 2;
    p.err = ctx->d_err;
    p.timeout_ns = ctx->timeout_ns;

    CUtensorMap ta, tb, td;
    std::memset(&ta, 0, sizeof(ta));
    std::memset(&tb, 0, sizeof(tb));
    std::memset(&td, 0, sizeof(td));
    {  // dy as [M pixels, K filters]
        const cuuint64_t dim[2] = {(cuuint64_t)bp.K, (cuuint64_t)p.M};
        const cuuint64_t str[1] = {(cuuint64_t)(bp.dys[3] * 2)};
        const cuuint32_t box[2] = {64, WG_BP};
        const cuuint32_t ones[2] = {1, 1};
        if (ctx->encode_tiled(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(bp.dy), dim,
                              str, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DLC_STATUS_EXECUTION_FAILED;
    }
    {  // x through im2col: 64 pixels x 64 channels per box
        const cuuint64_t gdim[4] = {(cuuint64_t)bp.C, (cuuint64_t)bp.W, (cuuint64_t)bp.H, (cuuint64_t)bp.N};
        const cuuint64_t gstr[3] = {(cuuint64_t)(bp.xs[3] * 2), (cuuint64_t)(bp.xs[2] * 2),
                                    (cuuint64_t)(bp.xs[0] * 2)};
        const int lower[2] = {-bp.pl, -bp.pt};
        const int upper[2] = {bp.pr - bp.dw * (bp.S - 1), bp.pb - bp.dh * (bp.R - 1)};
        const cuuint32_t estr[4] = {1, (cuuint32_t)bp.v, (cuuint32_t)bp.u, 1};
        if (ctx->encode_im2col(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(bp.x), gdim,
                               gstr, lower, upper, 64, WG_BP, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DLC_STATUS_EXECUTION_FAILED;
    }
    {  // dw KRSC FP32 as {C, R*S, K}: 32 channels x 1 tap x 32 filters per box
        const cuuint64_t dim[3] = {(cuuint64_t)bp.C, (cuuint64_t)(bp.R * bp.S), (cuuint64_t)bp.K};
        const cuuint64_t str[2] = {(cuuint64_t)(bp.ws[3] * 4), (cuuint64_t)(bp.ws[0] * 4)};
        const cuuint32_t box[3] = {32, 1, 32};
        const cuuint32_t ones[3] = {1, 1, 1};
        if (bp.ws[2] != (long long)bp.S * bp.ws[3] || bp.ws[1] != 1) return DLC_STATUS_INTERNAL_ERROR;
        if (ctx->encode_tiled(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(bp.w), dim, str,
                              box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DLC_STATUS_EXECUTION_FAILED;
    }
    const size_t smem = 1024 + (size_t)p.stages * stage_bytes + WG_EPI_SMEM + WG_BAR_AREA;
    auto kern = pair ? conv_wgrad_kernel<true> : conv_wgrad_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DLC_STATUS_EXECUTION_FAILED;
    if (!pair) {
        const int grid = std::max(1, std::min(p.units, ctx->sm_count));
        kern<<<grid, WG_THREADS, smem, ctx->stream>>>(p, ta, tb, td);
    } else {
        // persistent pairs: as many clusters of two as can be resident at once
        cudaLaunchConfig_t cfg;
        std::memset(&cfg, 0, sizeof(cfg));
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(WG_THREADS, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = ctx->stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(2 * (ctx->sm_count / 2), 1, 1);
        int max_clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&max_clusters, (const void *)kern, &cfg) != cudaSuccess ||
            max_clusters < 1)
            return DLC_STATUS_EXECUTION_FAILED;
        cfg.gridDim = dim3(2 * std::max(1, std::min(p.units, max_clusters)), 1, 1);
        if (cudaLaunchKernelEx(&cfg, kern, p, ta, tb, td) != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    }
    if (cudaGetLastError() != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}
