// conv_pair.cu -- the im2col implicit GEMM of conv_tc.cu on pairs of SMs:
// tcgen05.mma with cta_group::2 (M = 256, 128 output pixels per SM).
//
// Same lowering as the single-SM im2col kernel (maxDNN page, method section:
// an output coordinate is its receptive field times the filters; batch-reduce
// GEMM page, method section: acc += sum_i A_i B_i^T over filter taps and
// channel blocks; cuDNN page, method section: the lowered matrix exists only
// as on-chip tiles).  What the pair changes is where the operands come from:
// a cluster of two CTAs shares one MMA of M = 256 rows and N = BN filters.
// Each CTA loads its own 128 rows of A (im2col TMA) and HALF of the BN filter
// rows of B into its own shared memory, so per SM the operand traffic per
// MMA falls from A + B to A + B/2 -- the single-SM kernel's stages are bound by
// that traffic at BN = 192..256.
//
// Roles (per CTA, 7 or 11 warps): warp 0 lane 0 issues the A (im2col) loads
// and arms the stage's barrier, warp 2 lane 0 the B (filter) loads (with
// MN-major filters the two take alternate stages, each issuing both operands)
// -- both CTAs' loads complete on the LEADER's (rank 0) full barrier; warp 1 lane 0 of
// the leader alone issues the MMAs and commits each stage back to the empty
// barriers of both CTAs (multicast); warps 3-6 (or 3-10 for tiles of at most
// four k-blocks, two warps per TMEM lane quarter) of each CTA read their CTA's
// 128 accumulator rows from tensor memory, apply the epilogue and store y,
// then release the accumulator on the leader's barrier (a CTA-scope release:
// no generic memory passes to the MMA thread).  Every wait is
// bounded; both CTAs meet at a cluster barrier before tensor memory is
// released.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace {

using namespace dlc;

constexpr int PBM = 128;                    // output pixels per CTA
constexpr int PROW = 128;                   // bytes of one swizzled reduction row
constexpr int PA_BYTES = PBM * PROW;        // A stage: 16 KiB
constexpr int PAIR_EPI_WARP0 = 3;          // warps 0-2 load and issue; the epilogue follows
constexpr int PAIR_MAX_THREADS = (PAIR_EPI_WARP0 + 8) * 32;
constexpr int PAIR_MAX_SMEM = 232448;
constexpr int PAIR_BAR_AREA = 256;
constexpr int PAIR_EPI_BUF = 32 * 128;             // one warp's 32 rows x 32 FP32 columns
constexpr int PAIR_EPI_SMEM = 4 * 2 * PAIR_EPI_BUF;  // 4 epilogue warps, double-buffered

struct PairParams {
    int N, C, H, W, K, R, S, P, Q;
    int pt, pl, u, v, dh, dw;
    long long M;  // N*P*Q
    int PQ;
    long long ys[4];
    void *y;
    const float *bias;
    float alpha, beta;
    int relu, y_bf16;
    int y_tma;         // y through 2-D bulk tensor stores of 32 x 32 blocks
    int BN;            // filters per pair tile (BN/2 per CTA)
    int stages, num_kb, c_blocks, n_tiles;
    int kps;           // k-blocks per stage (1 or 2): one full wait and one commit per stage
    // B operand: K-major rows of BN/2 filters (b_mn = 0), or MN-major (b_mn =
    // 1): b_atoms boxes of 128 bytes of filters x BK reduction rows each.
    int b_mn, b_atoms, flip;
    int split_load;    // 1: a second warp issues the B loads; 2: two warps take alternate k-blocks
    int epi_parts;     // 1: four epilogue warps; 2: eight, two per TMEM lane quarter
    uint32_t b_stage;  // bytes of one CTA's B stage
    int num_tiles;     // pair tiles: ceil(M / 256) * n_tiles
    // Split tail: tiles [full_tiles, num_tiles) -- the part of the last wave
    // that would leave most pairs idle -- are each split into tail_splits
    // ranges of k-blocks whose partial sums are added into y (zeroed first).
    int full_tiles, tail_splits, num_units;
    uint32_t idesc, tmem_cols, acc_stride;
    int *err;
    unsigned long long timeout_ns;
};

// Work unit u: a whole tile, or one k-block range of a tail tile.
struct PairUnit {
    int tile, kb0, kb1, split;
};

__device__ __forceinline__ PairUnit pair_unit(const PairParams &p, int u) {
    PairUnit w;
    if (u < p.full_tiles) {
        w.tile = u;
        w.kb0 = 0;
        w.kb1 = p.num_kb;
        w.split = 0;
    } else {
        const int v = u - p.full_tiles;
        const int t = v / p.tail_splits, sp = v - t * p.tail_splits;
        w.tile = p.full_tiles + t;
        w.kb0 = (int)((long long)p.num_kb * sp / p.tail_splits);
        w.kb1 = (int)((long long)p.num_kb * (sp + 1) / p.tail_splits);
        w.split = 1;
    }
    return w;
}

__device__ __forceinline__ bool pair_drain(uint64_t *bar, uint32_t parity, const PairParams &p) {
    volatile int dummy = 0;
    WaitCtl c{&dummy, p.err, p.timeout_ns};
    return mbar_wait(bar, parity, c, 95);
}

// PART 0: this thread issues both operands' loads; 1: A (and arms the
// barrier), 2: B only -- two threads of different warps share a stage's loads;
// 3 and 4: both operands of the even / odd stages (counted over all of the
// CTA's units) -- two threads take turns, each stepping through every k-block
// to keep the ring's stage and phase (used with MN-major filters, whose B
// takes one load per 64-filter block).  KPS k-blocks share a stage: its one
// full barrier, armed once for all their bytes, and its one commit.
// MIXED: the last channel block of a tap holds at most 32 channels and comes
// in 64-byte rows (tmA2 / tmB2: 32-channel boxes, 64-byte swizzle) -- half the
// bytes of a full block, for half its MMAs.
template <int BK, int PART, bool MIXED, int KPS>
__device__ void pair_produce(const PairParams &p, uint32_t rank, const CUtensorMap *tmA,
                             const CUtensorMap *tmB, const CUtensorMap *tmA2, const CUtensorMap *tmB2,
                             uint32_t sA, uint32_t sB, uint64_t *full, uint64_t *empty, const WaitCtl &ctl) {
    const int ST = p.stages;
    const uint32_t b_half = p.b_stage;
    const uint32_t tx = 2u * (PA_BYTES + b_half);  // both CTAs' bytes land on the leader's barrier
    const uint32_t tx_h = tx / 2u;                 // a block of 64-byte rows
    const uint32_t atom_bytes = (uint32_t)BK * PROW;  // MN-major: BK rows of 128 bytes
    const uint32_t full0 = mapa_shared(smem_u32(full), 0);  // the leader's full barriers
    const uint32_t a_stage = (uint32_t)KPS * PA_BYTES, b_stage = (uint32_t)KPS * b_half;
    int stage = 0;
    uint32_t ph = 0;
    int gc = 0;  // stages so far (PART 3 / 4 fill the even / odd ones)
    for (int u = (int)cluster_id_x(); u < p.num_units; u += (int)num_clusters_x()) {
        const PairUnit w = pair_unit(p, u);
        const int t = w.tile;
        const long long m0 = (long long)(t / p.n_tiles) * (2 * PBM) + (long long)rank * PBM;
        const int k0 = (t % p.n_tiles) * p.BN + (int)rank * (p.BN / 2);
        const int n0 = (int)(m0 / p.PQ);
        const int rem = (int)(m0 - (long long)n0 * p.PQ);
        const int p0 = rem / p.Q, q0 = rem - (rem / p.Q) * p.Q;
        const int wc = q0 * p.v - p.pl;  // first window origin of this CTA's rows
        const int hc = p0 * p.u - p.pt;
        int cb = w.kb0 % p.c_blocks;
        const int rs0 = w.kb0 / p.c_blocks;
        int s = rs0 % p.S, r = rs0 / p.S;
        int sub = 0;  // k-block `sub` of its stage (KPS = 2: a unit's last stage may hold one)
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
            const bool last = KPS == 1 || sub == 1 || kb + 1 == w.kb1;  // the stage's last k-block
            if (PART < 3 || (gc & 1) == PART - 3) {  // (PART 3 / 4: this thread's stage)
                if (sub == 0) {
                    if (!mbar_wait(&empty[stage], ph ^ 1u, ctl, 1)) return;
                    if (PART != 2 && rank == 0) {  // the stage's bytes, both CTAs
                        uint32_t gtx = (MIXED && cb == p.c_blocks - 1) ? tx_h : tx;
                        if (!last) {
                            const int c2 = cb + 1 == p.c_blocks ? 0 : cb + 1;
                            gtx += (MIXED && c2 == p.c_blocks - 1) ? tx_h : tx;
                        }
                        mbar_arrive_expect_tx(&full[stage], gtx);
                    }
                }
                const bool half = MIXED && cb == p.c_blocks - 1;
                const uint32_t a_dst = sA + (uint32_t)stage * a_stage + (uint32_t)sub * PA_BYTES;
                const uint32_t b_dst = sB + (uint32_t)stage * b_stage + (uint32_t)sub * b_half;
                if (PART != 2)
                    tma_load_im2col_4d_pair(a_dst, half ? tmA2 : tmA, full0 + 8u * stage, cb * BK, wc, hc, n0,
                                            (uint16_t)(s * p.dw), (uint16_t)(r * p.dh));
                const int sc = p.flip ? p.S - 1 - s : s, rc = p.flip ? p.R - 1 - r : r;
                if (PART == 1) {
                } else if (MIXED) {
                    tma_load_4d_pair(b_dst, half ? tmB2 : tmB, full0 + 8u * stage, cb * BK, sc, rc, k0);
                } else if (p.b_mn) {
                    for (int a = 0; a < p.b_atoms; ++a)
                        tma_load_4d_pair(b_dst + (uint32_t)a * atom_bytes, tmB, full0 + 8u * stage, k0 + a * BK,
                                         sc, rc, cb * BK);
                } else {
                    tma_load_4d_pair(b_dst, tmB, full0 + 8u * stage, cb * BK, sc, rc, k0);
                }
            }
            if (last) {
                if (++stage == ST) stage = 0, ph ^= 1u;
                ++gc;
                sub = 0;
            } else {
                sub = 1;
            }
            if (++cb == p.c_blocks) {
                cb = 0;
                if (++s == p.S) s = 0, ++r;
            }
        }
    }
}

template <bool TF32, bool MIXED, int KPS>
__device__ void pair_mma(const PairParams &p, uint32_t tmem_base, uint32_t sA, uint32_t sB,
                         uint64_t *full, uint64_t *empty, uint64_t *tfull, uint64_t *tempty,
                         uint64_t *mma_done, const WaitCtl &ctl) {
    const int ST = p.stages;
    const uint32_t b_half = p.b_stage;
    constexpr int E = TF32 ? 4 : 2;
    constexpr int BK = PROW / E;
    const uint64_t a0 = sw128_kmajor_desc(sA);
    // MN-major B: 8-row groups of K 1024 bytes apart, 128-byte column blocks
    // of filters BK rows apart; one MMA's 32 bytes of K are 32/E rows.
    const uint64_t b0 = p.b_mn ? sw128_mnmajor_desc(sB, (uint32_t)BK * PROW) : sw128_kmajor_desc(sB);
    const uint32_t b_k = p.b_mn ? (32u / E) * PROW / 16u : 2u;
    const uint64_t a_sub = PA_BYTES >> 4, b_sub = b_half >> 4;        // next k-block of a stage
    const uint64_t a_step = a_sub * KPS, b_step = b_sub * KPS;        // next stage
    // a block of 64-byte rows: the same start address, the 64-byte swizzle's
    // stride and layout bits (the XOR of the two descriptors of one address)
    const uint64_t to64 = sw64_kmajor_desc(sA) ^ sw128_kmajor_desc(sA);
    int stage = 0, it = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int u = (int)cluster_id_x(); ok && u < p.num_units; u += (int)num_clusters_x(), ++it) {
        const PairUnit w = pair_unit(p, u);
        const int buf = it & 1;
        const uint32_t aph = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_cluster(&tempty[buf], aph ^ 1u, ctl, 3)) {  // both CTAs' epilogues
            ok = false;
            break;
        }
        tc_fence_after_sync();
        const uint32_t d = tmem_base + (uint32_t)buf * p.acc_stride;
        uint64_t ad = a0 + a_step * stage, bd = b0 + b_step * stage;
        uint32_t acc = 0;
        int cb = MIXED ? w.kb0 % p.c_blocks : 0;
        int sub = 0;  // k-block `sub` of its stage
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
            if (sub == 0) {
                if (!mbar_wait(&full[stage], ph, ctl, 4)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
            }
            const uint64_t as = KPS == 1 ? ad : ad + a_sub * (uint32_t)sub;
            const uint64_t bs = KPS == 1 ? bd : bd + b_sub * (uint32_t)sub;
            if constexpr (MIXED && !TF32) {
                if (cb == p.c_blocks - 1) {  // 32 channels in 64-byte rows: two MMAs
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        umma_bf16_pair(d, (as ^ to64) + 2u * j, (bs ^ to64) + 2u * j, p.idesc, acc);
                        acc = 1;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        umma_bf16_pair(d, as + 2u * j, bs + 2u * j, p.idesc, acc);
                        acc = 1;
                    }
                }
                if (++cb == p.c_blocks) cb = 0;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {  // 32 bytes of the 128-byte row each
                    if constexpr (TF32)
                        umma_tf32_pair(d, as + 2u * j, bs + b_k * j, p.idesc, acc);
                    else
                        umma_bf16_pair(d, as + 2u * j, bs + b_k * j, p.idesc, acc);
                    acc = 1;
                }
            }
            if (KPS == 2 && sub == 0 && kb + 1 < w.kb1) {  // the stage's other k-block follows
                sub = 1;
                continue;
            }
            sub = 0;
            umma_commit_pair(&empty[stage], 3);  // both CTAs' slots free once these are done
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
        umma_commit_pair(&tfull[buf], 3);  // both CTAs' accumulator rows are ready
    }
    if (!ok) {
        // gave up: loads of either CTA issued for stages not consumed land on
        // these barriers; wait for them briefly so no copy outlives the CTAs
        volatile int dummy = 0;
        const WaitCtl brief{&dummy, p.err, 50000000ull};
        for (int j = 0; j < ST; ++j) {
            if (!mbar_wait(&full[stage], ph, brief, 96)) break;
            if (++stage == ST) stage = 0, ph ^= 1u;
        }
    }
    // every MMA issued must complete before the pair releases tensor memory
    umma_commit_pair(mma_done, 3);
}

__device__ __forceinline__ float pair_bf16_to_f32(unsigned short b) {
    return __uint_as_float((uint32_t)b << 16);
}

__device__ __forceinline__ unsigned short pair_f32_to_bf16(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// beta*y + bias and ReLU on alpha*acc, in place: columns k0 .. k0+31 of one pixel.
__device__ __noinline__ void pair_epi_math(const PairParams &p, bool valid, long long ybase, int k0,
                                           float (&val)[32]) {
    const float *yf = static_cast<const float *>(p.y);
    const unsigned short *yb = static_cast<const unsigned short *>(p.y);
    for (int i = 0; i < 32; ++i) {
        const int k = k0 + i;
        float f = val[i];
        if (valid && k < p.K) {
            const long long yo = ybase + (long long)k * p.ys[1];
            if (p.beta != 0.f) f = __fmaf_rn(p.beta, p.y_bf16 ? pair_bf16_to_f32(yb[yo]) : yf[yo], f);
            if (p.bias) f += __ldg(p.bias + k);
        }
        if (p.relu) f = fmaxf(f, 0.f);
        val[i] = f;
    }
}

// alpha*acc + beta*y + bias, ReLU, store: columns k0 .. k0+31 of one output pixel.
__device__ __noinline__ void pair_store_general(const PairParams &p, bool valid, long long ybase,
                                                int k0, float (&val)[32]) {
    float *yf = static_cast<float *>(p.y);
    unsigned short *yb = static_cast<unsigned short *>(p.y);
    if (!valid) return;
    for (int i = 0; i < 32; ++i) {
        const int k = k0 + i;
        if (k >= p.K) break;
        const long long yo = ybase + (long long)k * p.ys[1];
        float f = val[i];
        if (p.beta != 0.f) f = __fmaf_rn(p.beta, p.y_bf16 ? pair_bf16_to_f32(yb[yo]) : yf[yo], f);
        if (p.bias) f += __ldg(p.bias + k);
        if (p.relu) f = fmaxf(f, 0.f);
        if (p.y_bf16)
            yb[yo] = pair_f32_to_bf16(f);
        else
            yf[yo] = f;
    }
}

// Row `lane` of a warp's 32 x 32 FP32 staging block, 128-byte swizzled like
// the y tensor map (16-byte chunk j of row l at chunk j ^ (l % 8)).
__device__ __forceinline__ void pair_stage_row(uint32_t buf, int lane, const float (&val)[32]) {
    const uint32_t rowp = buf + (uint32_t)lane * 128u;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(rowp + (((uint32_t)j ^ (lane & 7)) << 4)),
                     "f"(val[4 * j]), "f"(val[4 * j + 1]), "f"(val[4 * j + 2]), "f"(val[4 * j + 3])
                     : "memory");
}

__device__ void pair_epilogue(const PairParams &p, uint32_t rank, uint32_t tmem_base,
                              uint64_t *tfull, uint64_t *tempty, uint32_t epi_smem,
                              const CUtensorMap *tmY, const WaitCtl &ctl) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a warp reads the TMEM lanes of its warp index mod 4; with eight warps
    // each quarter has two, taking alternate 32-column chunks (part 0, 1)
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    const int part = (warp - PAIR_EPI_WARP0) >> 2;
    const int row = quad * 32 + lane;
    const bool plain = p.beta == 0.f && p.bias == nullptr && !p.relu && !p.y_bf16 && p.ys[1] == 1;
    const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);  // the leader's barriers
    float *yf = static_cast<float *>(p.y);
    const uint32_t my_bufs = epi_smem + (uint32_t)((warp - PAIR_EPI_WARP0) * 2 * PAIR_EPI_BUF);
    int nbuf = 0;
    int it = 0;
    for (int u = (int)cluster_id_x(); u < p.num_units; u += (int)num_clusters_x(), ++it) {
        const PairUnit w = pair_unit(p, u);
        const int t = w.tile;
        const int buf = it & 1;
        const uint32_t ph = (uint32_t)(it >> 1) & 1u;
        // the unit's output rows, worked out before its accumulator is ready
        const long long m = (long long)(t / p.n_tiles) * (2 * PBM) + (long long)rank * PBM + row;
        const int kt = (t % p.n_tiles) * p.BN;
        const bool valid = m < p.M;
        long long ybase = 0;
        if (valid) {
            int n, rem;
            if (p.M <= 0x7fffffffLL) {  // a 32-bit division (the 64-bit one is a long call)
                const uint32_t m32 = (uint32_t)m, pq = (uint32_t)p.PQ;
                n = (int)(m32 / pq);
                rem = (int)(m32 - (uint32_t)n * pq);
            } else {
                n = (int)(m / p.PQ);
                rem = (int)(m - (long long)n * p.PQ);
            }
            const int op = rem / p.Q, oq = rem - op * p.Q;
            ybase = (long long)n * p.ys[0] + (long long)op * p.ys[2] + (long long)oq * p.ys[3];
        }
        int okw = 0;
        if (lane == 0) okw = mbar_wait(&tfull[buf], ph, ctl, 5) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) break;
        __syncwarp();
        tc_fence_after_sync();
        const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)buf * p.acc_stride;
        for (int c0 = 32 * part; c0 < p.BN && kt + c0 < p.K; c0 += 32 * p.epi_parts) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(taddr + (uint32_t)c0, v);
            tmem_ld_wait();
            float val[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) val[i] = p.alpha * __uint_as_float(v[i]);
            const int k0 = kt + c0;
            if (p.y_tma) {
                if (m - lane >= p.M) continue;  // the warp's rows are all past M
                if (!plain) {
                    float lv[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) lv[i] = val[i];
                    pair_epi_math(p, valid, ybase, k0, lv);
#pragma unroll
                    for (int i = 0; i < 32; ++i) val[i] = lv[i];
                }
                const uint32_t sb = my_bufs + (uint32_t)(nbuf & 1) * PAIR_EPI_BUF;
                if (nbuf >= 2) {  // the store issued from this buffer two groups ago
                    if (lane == 0) bulk_wait_group_read<1>();
                    __syncwarp();
                }
                pair_stage_row(sb, lane, val);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {  // rows past M and columns past K are not written
                    if (w.split)  // a partial sum: added into y (zeroed before the launch)
                        tma_reduce_add_2d_s(tmY, sb, k0, (int)(m - lane));
                    else
                        tma_store_2d_s(tmY, sb, k0, (int)(m - lane));
                    bulk_commit_group();
                }
                ++nbuf;
                continue;
            }
            if (plain && valid && k0 + 32 <= p.K &&
                ((reinterpret_cast<uintptr_t>(yf + ybase + k0) & 15u) == 0)) {
                float4 *dst = reinterpret_cast<float4 *>(yf + ybase + k0);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    dst[i] = make_float4(val[4 * i], val[4 * i + 1], val[4 * i + 2], val[4 * i + 3]);
            } else {
                float lv[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) lv[i] = val[i];
                pair_store_general(p, valid, ybase, k0, lv);
            }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_tmem_free(tempty0 + 8u * buf);  // release on the leader
    }
    // staged stores must finish reading shared memory before the CTA exits
    if (p.y_tma && lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
}

template <bool TF32, bool MIXED, int KPS>
__global__ void __launch_bounds__(PAIR_MAX_THREADS, 1)
    conv_pair_kernel(const __grid_constant__ PairParams p, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmY,
                     const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2) {
    constexpr int BK = PROW / (TF32 ? 4 : 2);
    griddep_launch_dependents();  // the next grid may claim SMs this one leaves
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);  // same offset in both CTAs
    const int ST = p.stages;
    const uint32_t b_half = p.b_stage;
    uint8_t *smA = smem;
    uint8_t *smB = smA + (size_t)ST * KPS * PA_BYTES;
    uint8_t *epi = smB + (size_t)ST * KPS * b_half;  // y staging (y_tma), 1024-aligned
    uint64_t *bars = reinterpret_cast<uint64_t *>(epi + (p.y_tma ? p.epi_parts * PAIR_EPI_SMEM : 0));
    uint64_t *full = bars;
    uint64_t *empty = bars + ST;
    uint64_t *tfull = bars + 2 * ST;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full[i], 1u);   // the leader's expect-tx arrival (+ both CTAs' bytes)
            mbar_init(&empty[i], 1u);  // the leader's multicast commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1u);
            mbar_init(&tempty[i], 8u * (uint32_t)p.epi_parts);  // every epilogue warp of both CTAs
        }
        mbar_init(mma_done, 1u);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (MIXED) {
            prefetch_tmap(&tmA2);
            prefetch_tmap(&tmB2);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, p.tmem_cols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any remote arrival
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtl ctl{abort_flag, p.err, p.timeout_ns};
    const uint32_t sA = smem_u32(smA), sB = smem_u32(smB);
    griddep_wait();  // no global memory before the grid ahead of this one is done

    if (warp == 0) {
        if (lane == 0) {
            if (p.split_load == 2)
                pair_produce<BK, 3, MIXED, KPS>(p, rank, &tmA, &tmB, &tmA2, &tmB2, sA, sB, full, empty, ctl);
            else if (p.split_load)
                pair_produce<BK, 1, MIXED, KPS>(p, rank, &tmA, &tmB, &tmA2, &tmB2, sA, sB, full, empty, ctl);
            else
                pair_produce<BK, 0, MIXED, KPS>(p, rank, &tmA, &tmB, &tmA2, &tmB2, sA, sB, full, empty, ctl);
        }
    } else if (warp == 2) {
        if (lane == 0 && p.split_load == 2)
            pair_produce<BK, 4, MIXED, KPS>(p, rank, &tmA, &tmB, &tmA2, &tmB2, sA, sB, full, empty, ctl);
        else if (lane == 0 && p.split_load)
            pair_produce<BK, 2, MIXED, KPS>(p, rank, &tmA, &tmB, &tmA2, &tmB2, sA, sB, full, empty, ctl);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) pair_mma<TF32, MIXED, KPS>(p, tmem_base, sA, sB, full, empty, tfull, tempty, mma_done, ctl);
        // the leader's final commit reaches both CTAs; it also covers every
        // stage the MMAs consumed, i.e. every load of either CTA
        if (lane == 0) pair_drain(mma_done, 0u, p);
    } else {
        if (p.y_tma && lane == 0) prefetch_tmap(&tmY);
        pair_epilogue(p, rank, tmem_base, tfull, tempty, smem_u32(epi), &tmY, ctl);
    }
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // neither CTA leaves while the pair's MMAs or loads may touch it
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc_pair(tmem_base, p.tmem_cols);
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// The pair kernel serves every im2col-eligible problem unless DLC_TC_PAIR=0.
bool dlc_pdl_enabled() {
    static const bool on = [] {
        const char *ev = std::getenv("DLC_PDL");
        return !(ev && std::atoi(ev) == 0);
    }();
    return on;
}

bool dlc_pair_enabled(const dlcContext *) {
    const char *ev = std::getenv("DLC_TC_PAIR");
    return !(ev && std::atoi(ev) == 0);
}

dlcStatus_t dlc_preload_pair() {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, conv_pair_kernel<false, false, 1>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_pair_kernel<false, true, 1>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_pair_kernel<true, false, 1>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_pair_kernel<false, false, 2>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_pair_kernel<false, true, 2>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, conv_pair_kernel<true, false, 2>) != cudaSuccess)
        return DLC_STATUS_EXECUTION_FAILED;
    return DLC_STATUS_SUCCESS;
}

dlcStatus_t dlc_launch_pair(dlcContext *ctx, const ConvProblem &pb) {
    const bool tf32 = pb.math == DLC_MATH_TF32;
    const int e = tf32 ? 4 : 2;
    const int BK = PROW / e;
    PairParams p;
    std::memset(&p, 0, sizeof(p));
    p.N = pb.N; p.C = pb.C; p.H = pb.H; p.W = pb.W; p.K = pb.K; p.R = pb.R; p.S = pb.S;
    p.P = pb.P; p.Q = pb.Q;
    p.pt = pb.pt; p.pl = pb.pl; p.u = pb.u; p.v = pb.v; p.dh = pb.dh; p.dw = pb.dw;
    p.M = (long long)pb.N * pb.P * pb.Q;
    p.PQ = pb.P * pb.Q;
    for (int i = 0; i < 4; ++i) p.ys[i] = pb.ys[i];
    p.y = pb.y; p.bias = pb.bias;
    p.alpha = pb.alpha; p.beta = pb.beta; p.relu = pb.relu;
    p.y_bf16 = pb.ydt == DLC_DATA_BFLOAT16;
    // BN: a multiple of 32 (each CTA holds BN/2 filter rows, whole 16-row groups)
    if (pb.K <= 256) {
        p.BN = ((pb.K + 31) / 32) * 32;
    } else {
        p.BN = 256;
        long long best = -1;
        for (int bn : {256, 192, 128}) {
            const long long pad = (long long)((pb.K + bn - 1) / bn) * bn;
            if (best < 0 || pad < best) best = pad, p.BN = bn;
        }
    }
    if (const char *ev = std::getenv("DLC_TC_PAIR_BN")) {
        const int bn = std::atoi(ev);
        if (bn >= 32 && bn <= 256 && bn % 32 == 0) p.BN = bn;
    }
    p.c_blocks = (pb.C + BK - 1) / BK;
    // the last channel block in 64-byte rows when it holds at most 32
    // channels (BF16, K-major filters; DLC_TC_PAIR_MIXED=0 keeps it whole)
    const bool mixed = !tf32 && !pb.w_mn && pb.C % BK != 0 && pb.C % BK <= BK / 2 && [] {
        const char *ev = std::getenv("DLC_TC_PAIR_MIXED");
        return !(ev && std::atoi(ev) == 0);
    }();
    p.num_kb = pb.R * pb.S * p.c_blocks;
    p.n_tiles = (pb.K + p.BN - 1) / p.BN;
    p.flip = pb.flip;
    p.b_mn = pb.w_mn;
    {
        // the A and B loads from two warps; with MN-major filters (the data
        // gradient: one load per 64-filter block of B) the two warps take
        // alternate k-blocks instead (measured: OverFeat data gradient 1397 ->
        // 1422 TFLOP/s, the forward stacks unchanged)
        const char *ev = std::getenv("DLC_TC_PAIR_SPLITLOAD");
        p.split_load = ev ? std::max(0, std::min(2, std::atoi(ev))) : (p.b_mn ? 2 : 1);
    }
    p.b_atoms = (p.BN / 2 + BK - 1) / BK;
    p.b_stage = p.b_mn ? (uint32_t)(p.b_atoms * BK * PROW) : (uint32_t)(p.BN / 2) * PROW;
    const long long m_pairs = (p.M + 2 * PBM - 1) / (2 * PBM);
    if (m_pairs * p.n_tiles > 0x7fffffffLL) return DLC_STATUS_NOT_SUPPORTED;
    p.num_tiles = (int)(m_pairs * p.n_tiles);
    // y through bulk tensor stores: FP32, K contiguous, uniform pixel pitch
    {
        const bool dense = pb.ydt == DLC_DATA_FLOAT && pb.ys[1] == 1 && pb.ys[3] >= pb.K &&
                           (pb.ys[3] * 4) % 16 == 0 && (pb.P <= 1 || pb.ys[2] == (long long)pb.Q * pb.ys[3]) &&
                           (pb.N <= 1 || pb.ys[0] == (long long)pb.P * pb.Q * pb.ys[3]) &&
                           ((uintptr_t)pb.y % 16) == 0 && p.M <= 0x7fffffffLL;
        const char *ev = std::getenv("DLC_TC_PAIR_YTMA");  // =0 for direct stores
        p.y_tma = (dense && !(ev && std::atoi(ev) == 0)) ? 1 : 0;
    }
    // eight epilogue warps when a tile's few k-blocks take less time than its
    // epilogue (DLC_TC_PAIR_EPI=4 or 8 sets the count)
    p.epi_parts = p.num_kb <= 4 ? 2 : 1;
    if (const char *ev = std::getenv("DLC_TC_PAIR_EPI")) {
        const int e = std::atoi(ev);
        if (e == 4 || e == 8) p.epi_parts = e / 4;
    }
    const int epi_bytes = p.y_tma ? p.epi_parts * PAIR_EPI_SMEM : 0;
    // slack after the barriers: one more half filter tile, so that no operand
    // read of the last stage can leave the CTA's shared memory
    const int slack = (int)p.b_stage;
    const int room = PAIR_MAX_SMEM - 1024 - PAIR_BAR_AREA - slack - epi_bytes;
    // one k-block a stage; DLC_TC_PAIR_KPS=2 puts two in each (one full wait
    // and one commit for eight MMAs, half the stages): measured within noise of
    // one on the bench's layers (4-5 % faster on the 64- and 96-channel-output
    // ones, 1-3 % slower on others), so not the default
    p.kps = 1;
    if (const char *ev = std::getenv("DLC_TC_PAIR_KPS")) {
        const int k = std::atoi(ev);
        if (k == 1 || (k == 2 && room / (2 * (PA_BYTES + (int)p.b_stage)) >= 2)) p.kps = k;
    }
    const int stage_bytes = p.kps * (PA_BYTES + (int)p.b_stage);
    int st = room / stage_bytes;
    p.stages = st > 8 ? 8 : st;
    if (const char *ev = std::getenv("DLC_TC_STAGES")) {
        const int s2 = std::atoi(ev);
        if (s2 >= 2 && s2 < p.stages) p.stages = s2;
    }
    if (p.stages < 2) return DLC_STATUS_INTERNAL_ERROR;
    const uint32_t fmt = tf32 ? 2u : 1u;
    p.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)p.b_mn << 16) |  // B MN-major
              ((uint32_t)(p.BN >> 3) << 17) | ((uint32_t)((2 * PBM) >> 4) << 24);
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * p.BN)) cols <<= 1;
    p.tmem_cols = cols;
    p.acc_stride = cols / 2;
    p.err = ctx->d_err;
    p.timeout_ns = ctx->timeout_ns;

    // tensor maps: x through im2col (128 pixels x BK channels), w tiled with a
    // box of BN/2 filters (one CTA's half)
    CUtensorMap ta, tb;
    std::memset(&ta, 0, sizeof(ta));
    std::memset(&tb, 0, sizeof(tb));
    const CUtensorMapDataType dt =
        tf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t gdim[4] = {(cuuint64_t)pb.C, (cuuint64_t)pb.W, (cuuint64_t)pb.H, (cuuint64_t)pb.N};
    const cuuint64_t gstr[3] = {(cuuint64_t)(pb.xs[3] * e), (cuuint64_t)(pb.xs[2] * e),
                                (cuuint64_t)(pb.xs[0] * e)};
    const int lower[2] = {-pb.pl, -pb.pt};
    const int upper[2] = {pb.pr - pb.dw * (pb.S - 1), pb.pb - pb.dh * (pb.R - 1)};
    const cuuint32_t estr[4] = {1, (cuuint32_t)pb.v, (cuuint32_t)pb.u, 1};
    CUresult r = ctx->encode_im2col(&ta, dt, 4, const_cast<void *>(pb.x), gdim, gstr, lower, upper,
                                    (cuuint32_t)BK, (cuuint32_t)PBM, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return DLC_STATUS_EXECUTION_FAILED;
    // K-major: {C, S, R, K} with a box of BK channels x BN/2 filters; MN-major
    // (transposed filters): {K, S, R, C} with boxes of BK filters x BK channels
    const cuuint64_t wdim[4] = {(cuuint64_t)(p.b_mn ? pb.K : pb.C), (cuuint64_t)pb.S, (cuuint64_t)pb.R,
                                (cuuint64_t)(p.b_mn ? pb.C : pb.K)};
    const cuuint64_t wstr[3] = {(cuuint64_t)(pb.ws[3] * e), (cuuint64_t)(pb.ws[2] * e),
                                (cuuint64_t)(pb.ws[p.b_mn ? 1 : 0] * e)};
    const cuuint32_t box[4] = {(cuuint32_t)BK, 1, 1, (cuuint32_t)(p.b_mn ? BK : p.BN / 2)};
    const cuuint32_t ones[4] = {1, 1, 1, 1};
    r = ctx->encode_tiled(&tb, dt, 4, const_cast<void *>(pb.w), wdim, wstr, box, ones,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return DLC_STATUS_EXECUTION_FAILED;

    // the 32-channel boxes of a mixed last block: 64-byte swizzled rows
    CUtensorMap ta2, tb2;
    std::memset(&ta2, 0, sizeof(ta2));
    std::memset(&tb2, 0, sizeof(tb2));
    if (mixed) {
        if (ctx->encode_im2col(&ta2, dt, 4, const_cast<void *>(pb.x), gdim, gstr, lower, upper,
                               (cuuint32_t)(BK / 2), (cuuint32_t)PBM, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DLC_STATUS_EXECUTION_FAILED;
        const cuuint32_t box2[4] = {(cuuint32_t)(BK / 2), 1, 1, (cuuint32_t)(p.BN / 2)};
        if (ctx->encode_tiled(&tb2, dt, 4, const_cast<void *>(pb.w), wdim, wstr, box2, ones,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DLC_STATUS_EXECUTION_FAILED;
    }
    const size_t smem = 1024 + (size_t)p.stages * stage_bytes + epi_bytes + PAIR_BAR_AREA + slack;
    CUtensorMap ty;
    std::memset(&ty, 0, sizeof(ty));
    if (p.y_tma) {
        const cuuint64_t ydim[2] = {(cuuint64_t)pb.K, (cuuint64_t)p.M};
        const cuuint64_t ystr[1] = {(cuuint64_t)(pb.ys[3] * 4)};
        const cuuint32_t ybox[2] = {32, 32};
        const cuuint32_t yones[2] = {1, 1};
        if (ctx->encode_tiled(&ty, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, pb.y, ydim, ystr, ybox, yones,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DLC_STATUS_EXECUTION_FAILED;
    }
    auto kern = p.kps == 2 ? (tf32 ? conv_pair_kernel<true, false, 2>
                                   : (mixed ? conv_pair_kernel<false, true, 2> : conv_pair_kernel<false, false, 2>))
                           : (tf32 ? conv_pair_kernel<true, false, 1>
                                   : (mixed ? conv_pair_kernel<false, true, 1> : conv_pair_kernel<false, false, 1>));
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DLC_STATUS_EXECUTION_FAILED;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = dlc_pdl_enabled() ? 1 : 0;
    cfg.blockDim = dim3((PAIR_EPI_WARP0 + 4 * p.epi_parts) * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx->stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
    // one pair per two SMs that can hold a cluster at once (persistent pairs)
    int max_clusters = 0;
    cfg.gridDim = dim3(2 * (ctx->sm_count / 2), 1, 1);
    if (cudaOccupancyMaxActiveClusters(&max_clusters, (const void *)kern, &cfg) != cudaSuccess ||
        max_clusters < 1)
        return DLC_STATUS_EXECUTION_FAILED;
    // Split tail: when the last wave would leave at least half the pairs
    // idle, its tiles are split along the reduction over the idle pairs (plain
    // epilogue only: the partial sums are added by bulk reduce-adds into y,
    // zeroed here first).  DLC_TC_PAIR_SPLIT=0 turns it off.
    int clusters = std::min(max_clusters, std::max(1, p.num_tiles));
    p.full_tiles = p.num_tiles;
    p.tail_splits = 1;
    p.num_units = p.num_tiles;
    {
        const char *ev = std::getenv("DLC_TC_PAIR_SPLIT");
        // The tail's partial sums meet in FP32 atomic adds in whatever order
        // they arrive, so its outputs may differ in the last bits from run to
        // run; a deterministic handle keeps whole tiles.
        const bool plain = p.y_tma && pb.beta == 0.f && pb.bias == nullptr && !pb.relu &&
                           !ctx->deterministic;
        const int C = max_clusters;
        const int rem = p.num_tiles % C;
        const int splits = rem > 0 ? std::min(std::min(C / rem, p.num_kb), 16) : 1;
        // worth it when the pieces are shorter than a whole tile by more than
        // about ten k-blocks: a piece's reduce-add epilogue and the zeroing
        // memset between launches cost that much (measured: a 1x1 layer of
        // eight k-blocks a tile ran 17.5 us split, 13.3 us whole; 3x3 layers
        // of 36-72 k-blocks gain 3-8 us).  DLC_TC_PAIR_SPLIT=0: never; =2:
        // whenever the tail leaves clusters idle.
        const int mode = ev ? std::atoi(ev) : 1;
        const bool worth = p.num_kb - (p.num_kb + splits - 1) / splits > 10;
        if (plain && splits >= 2 && mode != 0 && (worth || mode == 2)) {
            p.full_tiles = p.num_tiles - rem;
            p.tail_splits = splits;
            p.num_units = p.full_tiles + rem * splits;
            clusters = C;
            const long long row0 = (long long)(p.full_tiles / p.n_tiles) * (2 * PBM);
            if (row0 < p.M &&
                cudaMemset2DAsync(static_cast<float *>(pb.y) + row0 * pb.ys[3], (size_t)pb.ys[3] * 4, 0,
                                  (size_t)pb.K * 4, (size_t)(p.M - row0), ctx->stream) != cudaSuccess)
                return DLC_STATUS_EXECUTION_FAILED;
        }
    }
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, p, ta, tb, ty, ta2, tb2) != cudaSuccess) return DLC_STATUS_EXECUTION_FAILED;
    ctx->launches += 1;
    return DLC_STATUS_SUCCESS;
}
