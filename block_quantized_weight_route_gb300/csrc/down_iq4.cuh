// Routed-MoE down product on sm_103a: q8_1 H times IQ4_NL weights, per expert.
//
//   y[t, n] = sum_b d_H[t, b] * d_W[e, n, b] * I[t, n, b]
//   I[t, n, b] = sum_{k in block b} q[t, k] * codebook[idx[e, n, k]]      (exact)
//
// ("Run Edge0-145B Q3_K on AMD HIP (Linux, gfx1100)", commit 4cb5224: the
// down product reads IQ4_NL weights against H rounded to q8_1.)
//
// Both operands are small integers, exact in f16, and a 32-element block sum
// stays below 2^24, so one f16 tcgen05.mma pair per 32-K block gives I exactly
// in fp32.  Every block gets its own TMEM accumulator (a ring of 4), which the
// epilogue folds with d_H * d_W in fp32.
//
// Orientation: the MMA's M side is 128 weight rows (output dims n), its N side
// 128 routed tokens of one expert.  Each epilogue thread owns one output dim
// and reads its d_W per block from shared memory; d_H varies along the columns
// and is read (broadcast) from a shared-memory copy of the tile's fp32 d values.
// Both scale tables arrive by 1-D bulk copies once per tile: d_H from the
// per-tile-entry layout the gate/up epilogue writes, d_W as the tile's 128
// contiguous rows of [E][D][F/32].
//
// The H codes are stored by the gate/up epilogue as exact f16 integers, so the
// MMA's token operand comes straight from TMA (128-byte swizzle) with no
// conversion; only the IQ4 indices are expanded (codebook lookup) to f16.
//
//   warp 0: TMA producer (IQ4 codes + f16 H codes per K block, d_H and d_W per tile)
//   warp 2: MMA issuer
//   warps 4 .. 4+EPI_WARPS-1: epilogue (EPI_WARPS/4 per TMEM lane quarter)
//   warps 1, 3 (and with four converters two more after the epilogue, on
//   sub-partitions 0 and 2): IQ4 converters; warp 1 also allocates TMEM.
//   With four converters and the fused combine, the remaining two warps after
//   the epilogue (sub-partitions 1 and 3) add each staged tile into Y.
// A warp's SM sub-partition is its index mod 4, the same as the TMEM lane
// quarter it may read, so every sub-partition holds EPI_WARPS/4 epilogue warps
// and one of the producer, a converter or the MMA issuer.  The producer and
// the MMA issuer run on one lane each.
#pragma once
#include "qgemm.cuh"

namespace qmm {

#ifndef QMM_DOWN_CSTAGES
#define QMM_DOWN_CSTAGES 3
#endif
#ifndef QMM_DOWN_PAIR
#define QMM_DOWN_PAIR 1
#endif
#ifndef QMM_DOWN_CONV4
#define QMM_DOWN_CONV4 2
#endif
template <int EPI_WARPS_, int CONV_WARPS_, int TSTAGES_>
struct DownCfgT {
    static constexpr int BM = 128, BN = 128, BK = 64, UMMA_K = 16, GROUP_K = 32;
    static constexpr int EPI_WARPS = EPI_WARPS_, CONV_WARPS = CONV_WARPS_, EPI_BASE = 4;
    static constexpr int CPW = 128 / (EPI_WARPS_ / 4);        // token columns per epilogue warp
    // TMEM loads of CW columns, NCH per 32-K block (16-column loads when every
    // sub-partition also hosts a converter warp: fewer live registers)
    static constexpr int CW = (EPI_WARPS_ == 16 && CONV_WARPS_ == 4) ? 16 : 32;
    static constexpr int NCH = CPW / CW;
    static constexpr int W2 = EPI_BASE + EPI_WARPS;           // first warp after the epilogue (sub-partition 0)
    // 8 epilogue warps and 4 converters: 16 warps launched at 128 registers a
    // thread, the two epilogue warpgroups raised to 168 (their running sums and
    // two 32-column loads) and the other two lowered to 88 - the shares add up
    // to exactly the launch's 16 x 128
    static constexpr bool REG_SPLIT = (EPI_WARPS_ == 8 && CONV_WARPS_ == 4);
    static constexpr int REGS_LAUNCH = 128, REGS_EPI = 168, REGS_OTHER = 88;
    static_assert(!REG_SPLIT || 8 * REGS_EPI + 8 * REGS_OTHER == 16 * REGS_LAUNCH, "register shares = launch registers");
    static constexpr int THREADS = REG_SPLIT ? 512 : 32 * (CONV_WARPS == 2 ? W2 : W2 + 3);
    static constexpr int CONV_THREADS = 32 * CONV_WARPS;
    static constexpr int MMA_WARP = 2;                        // sub-partition 2; TMEM is allocated by warp 1
    __device__ static int conv_slot(int warp) {
        if (warp == 1) return 0;
        if (warp == 3) return 1;
        if (CONV_WARPS == 4) {
            if (warp == W2) return 2;
            if (warp == W2 + QMM_DOWN_CONV4) return 3;
        }
        return -1;
    }
    static_assert(EPI_WARPS == 8 || EPI_WARPS == 16, "epilogue width");
    static_assert(CONV_WARPS == 2 || CONV_WARPS == 4, "converter count");
    static constexpr int TSTAGES = TSTAGES_, CSTAGES = QMM_DOWN_CSTAGES, SSTAGES = 2, NBUF = 4;
    // PAIR: the accumulators of a 64-K step's two blocks are handed over together
    // (one commit / wait / release per pair instead of per block)
    static constexpr bool PAIR = QMM_DOWN_PAIR != 0;
    static constexpr int NHAND = PAIR ? NBUF / 2 : NBUF;        // hand-off barriers
    static constexpr int TMA_GROUPS = TSTAGES_;   // producer lane pairs (IQ4 codes, H codes)
    static_assert(2 * TMA_GROUPS <= 31, "producer lanes: pairs below lane 31");
    static constexpr int KG_MAX = 32;                         // K <= 1024
    static constexpr int A_RAW_BYTES = BM * 32;               // IQ4 codes: 64 indices per row
    static constexpr int B_BYTES = BN * BK * 2;               // f16 H codes, 128-byte rows
    static constexpr int TSTAGE_BYTES = A_RAW_BYTES + B_BYTES;
    static constexpr int CSTAGE_BYTES = BM * BK * 2;          // expanded IQ4 values
    static constexpr int DH_BYTES = KG_MAX * BN * 4;          // d_H of one tile, [block][token] fp32
    static constexpr int DW_BYTES = BM * KG_MAX * 2;          // d_W of one tile, [row][block] fp16
    static constexpr int SSTAGE_BYTES = DH_BYTES + DW_BYTES;
    // Staged tile outputs: the epilogue leaves a finished tile's y [token][row]
    // fp32 in shared memory and goes on to the next tile; two combine warps (the
    // warps without a role under the register split, 13 and 15) add weight x y into
    // Y[token] with 16-byte reductions (per-slot form: store the rows of Yslot)
    // while the next tile is folded.
    static constexpr bool STAGE_Y = REG_SPLIT;
    static constexpr int YS_BYTES = STAGE_Y ? BN * BM * 4 : 0;
    __device__ static int comb_slot(int warp) {
        if (!STAGE_Y) return -1;
        return warp == W2 + 1 ? 0 : (warp == W2 + 3 ? 1 : -1);
    }
    static_assert(!STAGE_Y || QMM_DOWN_CONV4 == 2, "combine warps: the warps after the epilogue without a converter");
    static constexpr uint32_t IDESC = idesc_kind_f16(BM, BN, false);
    static constexpr int BAR_COUNT = 2 * TSTAGES + 2 * CSTAGES + 2 * SSTAGES + 2 * NBUF + 3;   // (NHAND <= NBUF)
    static constexpr int SMEM_BYTES = 1024 + TSTAGES * TSTAGE_BYTES + CSTAGES * CSTAGE_BYTES +
                                      SSTAGES * SSTAGE_BYTES + YS_BYTES + BAR_COUNT * 8 + 64;
    static_assert(A_RAW_BYTES % 1024 == 0 && TSTAGE_BYTES % 1024 == 0 && CSTAGE_BYTES % 1024 == 0 &&
                      SSTAGE_BYTES % 1024 == 0,
                  "align");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};
// Measured on the 5268-token stage (down with the fused combine): 8 epilogue
// warps (64 token columns each, both TMEM loads of a block issued before one
// wait), 4 converters under the register split, accumulators handed over in
// pairs, the staged combine, 3 TMA and 3 expanded-weight stages: 0.404 ms
// (4 + 2 stages: 0.412; before the staged combine, 5 + 2 stages: 0.506; with 2
// converters and one hand-off per block: 0.530; 16 epilogue warps were slower).
#ifndef QMM_DOWN_EPI_WARPS
#define QMM_DOWN_EPI_WARPS 8
#endif
#ifndef QMM_DOWN_CONV_WARPS
#define QMM_DOWN_CONV_WARPS 4
#endif
#ifndef QMM_DOWN_TSTAGES
#define QMM_DOWN_TSTAGES 3
#endif
using DownCfg = DownCfgT<QMM_DOWN_EPI_WARPS, QMM_DOWN_CONV_WARPS, QMM_DOWN_TSTAGES>;

// 1-D bulk copy global -> shared, completion counted on `bar` (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// p[0..3] += {a, b, c, d} as one 16-byte fp32 reduction in L2 (p 16-byte aligned).
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t saddr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(saddr));
    return v;
}

// p.K = F (reduction), p.N = D (weight rows per expert), p.n_tiles = D / 128,
// p.tiles / num_entries / max_entries: the 128-token tile list of the routing,
// p.dW: IQ4_NL scales [E][D][F/32] fp16, p.dH32: d_H fp32 [entry][F/32][128],
// p.Y: Yslot [T*k][D] fp32 (p.ldy = D).
// tmA: IQ4 codes as [E*D][F/2] bytes, box {32, 128}, 32-byte swizzle.
// tmB: H codes as [T*k][F] f16, box {64, 128}, 128-byte swizzle.
// COMBINE = false: each routed row's outputs are stored to p.Y = Yslot [T*k][D];
// COMBINE = true: the weighted combine is fused in: Y[src[r], n] += wrow[r] * y[r, n]
// into p.Y = Y [T][D] (zeroed beforehand), with fp32 atomic adds (red.global.add),
// so the order of a token's k contributions is not fixed.
template <class C, bool COMBINE>
__global__ void __launch_bounds__(C::THREADS, 1)
    down_iq4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* tstage = smem;
    uint8_t* cstage = tstage + C::TSTAGES * C::TSTAGE_BYTES;
    uint8_t* sstage = cstage + C::CSTAGES * C::CSTAGE_BYTES;
    float* ystage = reinterpret_cast<float*>(sstage + C::SSTAGES * C::SSTAGE_BYTES);   // [token][row], STAGE_Y
    uint64_t* bars = reinterpret_cast<uint64_t*>(sstage + C::SSTAGES * C::SSTAGE_BYTES + C::YS_BYTES);
    uint64_t* full_t = bars;
    uint64_t* empty_t = full_t + C::TSTAGES;
    uint64_t* full_c = empty_t + C::TSTAGES;
    uint64_t* empty_c = full_c + C::CSTAGES;
    uint64_t* full_s = empty_c + C::CSTAGES;
    uint64_t* empty_s = full_s + C::SSTAGES;
    uint64_t* acc_full = empty_s + C::SSTAGES;
    uint64_t* acc_empty = acc_full + C::NHAND;
    uint64_t* drain_bar = acc_empty + C::NHAND;
    uint64_t* y_full = drain_bar + 1;      // a tile's y staged (epilogue warps)
    uint64_t* y_empty = y_full + 1;        // the stage read (combine warps)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(y_empty + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::TSTAGES; ++i) {
            mbar_init(&full_t[i], 1);
            // released by the converters (IQ4 codes read) and the MMA commit (H codes read)
            mbar_init(&empty_t[i], C::CONV_WARPS + 1);
        }
        for (int i = 0; i < C::CSTAGES; ++i) {
            mbar_init(&full_c[i], C::CONV_WARPS);
            mbar_init(&empty_c[i], 1);
        }
        for (int i = 0; i < C::SSTAGES; ++i) {
            mbar_init(&full_s[i], 1);
            mbar_init(&empty_s[i], C::EPI_WARPS);
        }
        for (int i = 0; i < C::NHAND; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], C::EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        mbar_init(y_full, C::EPI_WARPS);
        mbar_init(y_empty, 2);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        if (!p.wmaps) tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int kblocks = p.K / C::BK;
    const int groups = p.K / C::GROUP_K;
    const int entries = min(*p.num_entries, p.max_entries);
    const int num_tiles = entries * p.n_tiles;

    // Roles.  With the register split, each warpgroup runs exactly one setmaxnreg
    // (the epilogue warpgroups the inc, the others the dec), at the top of the
    // code it governs.
    if (warp >= C::EPI_BASE && warp < C::EPI_BASE + C::EPI_WARPS) {
        if constexpr (C::REG_SPLIT) setmaxnreg_inc<C::REGS_EPI>();
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int cq = (warp - C::EPI_BASE) >> 2;              // this warp's block of CPW token columns
        const int r = q * 32 + lane;                            // this thread's weight row in the tile
        const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
        int buf = 0, ss = 0;
        uint32_t bph = 0, sph = 0, yph = 0;
        bool ok = true;
        int4 g4 = (int)blockIdx.x < num_tiles ? p.tiles[blockIdx.x / p.n_tiles] : make_int4(0, 0, 0, 0);
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            const int entry = t / p.n_tiles;
            const int n0 = (t - entry * p.n_tiles) * C::BM;
            const int tn = t + gridDim.x;
            // the next tile's descriptor, loaded while this tile runs
            const int4 g4n = tn < num_tiles ? p.tiles[tn / p.n_tiles] : make_int4(0, 0, 0, 0);
            if (!mbar_wait(&full_s[ss], sph, abort_flag, p.err, DEV_TIMEOUT_ACC)) break;
            const uint32_t sbase = smem_u32(sstage + ss * C::SSTAGE_BYTES);
            const uint32_t dh_base = sbase + cq * C::CPW * 4;
            const uint32_t dw_addr = sbase + C::DH_BYTES + (uint32_t)(r * groups * 2);
            // CPW token columns as f32 pairs (the packed f32x2 FMA path; the
            // compiler keeps each pair in an aligned register pair)
            float2 y[C::CPW / 2];
#pragma unroll
            for (int j = 0; j < C::CPW / 2; ++j) y[j] = make_float2(0.f, 0.f);
            // fold this warp's CPW columns of block g from accumulator buffer b
            auto fold_block = [&](int g, int b, bool release, int hand) {
                const float dwf = __half2float(__ushort_as_half((unsigned short)lds_u16(dw_addr + g * 2)));
                const float2 dw2 = make_float2(dwf, dwf);
                const uint32_t acc = lane_addr + (uint32_t)(b * C::BN + cq * C::CPW);
                // all of this warp's accumulator columns for the block: loads issued
                // together, one wait, the buffer handed back before the fold
                uint32_t v[C::NCH][C::CW];
#pragma unroll
                for (int c = 0; c < C::NCH; ++c) {
                    if constexpr (C::CW == 32) tmem_ld32(acc + c * C::CW, v[c]);
                    else tmem_ld16(acc + c * C::CW, v[c]);
                }
                tmem_ld_wait();
                if (release) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_empty[hand]);
                }
#pragma unroll
                for (int c = 0; c < C::NCH; ++c) {
#pragma unroll
                    for (int j = 0; j < C::CW / 4; ++j) {
                        const uint4 dh = lds128(dh_base + (uint32_t)((g * C::BN + c * C::CW + 4 * j) * 4));
                        const float2 i01 = make_float2(__uint_as_float(v[c][4 * j]), __uint_as_float(v[c][4 * j + 1]));
                        const float2 i23 = make_float2(__uint_as_float(v[c][4 * j + 2]), __uint_as_float(v[c][4 * j + 3]));
                        const float2 d01 = make_float2(__uint_as_float(dh.x), __uint_as_float(dh.y));
                        const float2 d23 = make_float2(__uint_as_float(dh.z), __uint_as_float(dh.w));
                        // y += (I * d_H) * d_W, both products rounded to fp32
                        float2& y01 = y[c * (C::CW / 2) + 2 * j];
                        float2& y23 = y[c * (C::CW / 2) + 2 * j + 1];
                        y01 = __ffma2_rn(__fmul2_rn(i01, d01), dw2, y01);
                        y23 = __ffma2_rn(__fmul2_rn(i23, d23), dw2, y23);
                    }
                }
            };
            for (int g = 0; g < groups; g += (C::PAIR ? 2 : 1)) {
                if (!mbar_wait(&acc_full[buf], bph, abort_flag, p.err, DEV_TIMEOUT_ACC)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if constexpr (C::PAIR) {
                    fold_block(g, 2 * buf, false, buf);
                    fold_block(g + 1, 2 * buf + 1, true, buf);
                } else {
                    fold_block(g, buf, true, buf);
                }
                if (++buf == C::NHAND) {
                    buf = 0;
                    bph ^= 1u;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_s[ss]);
            if (++ss == C::SSTAGES) {
                ss = 0;
                sph ^= 1u;
            }
            if (!ok) break;
            const int tok0 = cq * C::CPW;
            if constexpr (C::STAGE_Y) {
                // this warp's token columns of y into the stage, [token][row]: lanes write
                // 32 consecutive rows (conflict-free); the stage must have been read out
                if (!mbar_wait(y_empty, yph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_ACC)) break;
#pragma unroll
                for (int j = 0; j < C::CPW / 2; ++j) {
                    ystage[(tok0 + 2 * j) * C::BM + r] = y[j].x;
                    ystage[(tok0 + 2 * j + 1) * C::BM + r] = y[j].y;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(y_full);
                yph ^= 1u;
            } else if constexpr (!COMBINE) {
                // Yslot[row, n] for this warp's token columns; lanes write consecutive n
                float* out = static_cast<float*>(p.Y) + (long)g4.y * p.ldy + n0 + r;
#pragma unroll
                for (int j = 0; j < C::CPW / 2; ++j) {
                    if (tok0 + 2 * j < g4.z) out[(long)(tok0 + 2 * j) * p.ldy] = y[j].x;
                    if (tok0 + 2 * j + 1 < g4.z) out[(long)(tok0 + 2 * j + 1) * p.ldy] = y[j].y;
                }
            } else {
                // Y[token, n] += weight * y for this warp's token columns: lane l holds the
                // token and weight of columns l, l+32, ...; each column's pair is broadcast
                // and the 32 lanes add 32 consecutive n (one 128-byte reduction)
                constexpr int NC = C::CPW / 32;
                int tk[NC];
                float wt[NC];
#pragma unroll
                for (int i = 0; i < NC; ++i) {
                    const int c = tok0 + 32 * i + lane;
                    tk[i] = c < g4.z ? __ldg(p.src + g4.y + c) : 0;
                    wt[i] = c < g4.z ? __ldg(p.wrow + g4.y + c) : 0.f;
                }
                float* out = static_cast<float*>(p.Y) + n0 + r;
#pragma unroll
                for (int j = 0; j < C::CPW / 2; ++j) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = 2 * j + h;
                        const int t = __shfl_sync(0xffffffffu, tk[c >> 5], c & 31);
                        const float wc = __shfl_sync(0xffffffffu, wt[c >> 5], c & 31);
                        if (tok0 + c < g4.z) atomicAdd(out + (long)t * p.ldy, wc * (h ? y[j].y : y[j].x));
                    }
                }
            }
            g4 = g4n;
        }
    } else {
        if constexpr (C::REG_SPLIT) setmaxnreg_dec<C::REGS_OTHER>();
        if (warp == 0) {
            // ------------------------------------------------------------ producer (one warp)
            // A thread has one TMA copy executing at a time (~0.8-0.9k cycles each on
            // GB300, whatever the size), so the two copies of stage s come from lanes
            // 2*(s % TMA_GROUPS) and 2*(s % TMA_GROUPS) + 1, and the per-tile scale
            // copies from lane 31: copies of different stages overlap.
            {
                int s = 0, ss = 0;
                uint32_t ph = 0, sph = 0;
                long issued = 0, s_issued = 0;
                bool ok = true;
                const uint32_t dh_bytes = (uint32_t)(groups * C::BN * 4);
                const uint32_t dw_bytes = (uint32_t)(C::BM * groups * 2);
                for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                    const int entry = t / p.n_tiles;
                    const int n0 = (t - entry * p.n_tiles) * C::BM;
                    const int4 g = p.tiles[entry];
                    // the expert's IQ4 codes: its own tensor map (pointer-table form) at rows
                    // n0.., or the kernel parameter over the contiguous [E*D] rows
                    const CUtensorMap* amap = p.wmaps ? p.wmaps + g.x : &tmA;
                    const int arow = (p.wmaps ? 0 : g.x * p.N) + n0;
                    if (p.wmaps) tensormap_acquire(amap);
                    // this tile's d_H and d_W values
                    const bool got_s = mbar_wait(&empty_s[ss], sph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_TMA_EMPTY);
                    if (__any_sync(0xffffffffu, !got_s)) break;
                    if (lane == 31) {
                        uint8_t* sst = sstage + ss * C::SSTAGE_BYTES;
                        const __half* dw = p.dW_tab ? p.dW_tab[g.x] + (long)n0 * groups : p.dW + ((long)g.x * p.N + n0) * groups;
                        mbar_arrive_expect_tx(&full_s[ss], dh_bytes + dw_bytes);
                        bulk_load(sst, p.dH32 + (long)entry * groups * C::BN, dh_bytes, &full_s[ss]);
                        bulk_load(sst + C::DH_BYTES, dw, dw_bytes, &full_s[ss]);
                    }
                    __syncwarp();
                    ++s_issued;
                    if (++ss == C::SSTAGES) {
                        ss = 0;
                        sph ^= 1u;
                    }
                    for (int kb = 0; kb < kblocks; ++kb) {
                        const bool got = mbar_wait(&empty_t[s], ph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_TMA_EMPTY);
                        if (__any_sync(0xffffffffu, !got)) {
                            ok = false;
                            break;
                        }
                        const int l0 = 2 * (s % C::TMA_GROUPS);
                        uint8_t* st = tstage + s * C::TSTAGE_BYTES;
                        if (lane == l0) mbar_arrive_expect_tx(&full_t[s], C::TSTAGE_BYTES);
                        __syncwarp();
                        if (lane == l0)
                            tma_load_2d(st, amap, &full_t[s], kb * 32, arow);
                        else if (lane == l0 + 1)
                            tma_load_2d(st + C::A_RAW_BYTES, &tmB, &full_t[s], kb * C::BK, g.y);
                        __syncwarp();
                        ++issued;
                        if (++s == C::TSTAGES) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                }
                if (lane == 0) {
                    drain_ring(full_t, issued, C::TSTAGES, p.err);
                    drain_ring(full_s, s_issued, C::SSTAGES, p.err);
                }
            }
            __syncwarp();
        } else if (warp == C::MMA_WARP) {
            // ------------------------------------------------------------ MMA issuer (one lane)
            // A single thread runs the whole issue loop: no per-MMA election or warp
            // votes, so each K block costs a few dozen instructions on this warp.
            if (lane == 0) {
                int cs = 0, ts = 0, buf = 0;
                uint32_t cph = 0, bph = 0;
                bool ok = true;
                for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                    for (int kb = 0; kb < kblocks && ok; ++kb) {
                        // expanded weights ready: the converters arrive on full_c only after they saw
                        // the TMA stage (IQ4 codes and H codes) complete, so full_c orders the H
                        // codes of the same stage too
                        if (!mbar_wait(&full_c[cs], cph, abort_flag, p.err, DEV_TIMEOUT_CONV)) {
                            ok = false;
                            break;
                        }
                        // (no tcgen05 fence here: the operands are ordered by the mbarriers and the
                        // writers' proxy fence; a tcgen05 fence per K block would drain the MMA pipe)
                        const uint32_t a_base = smem_u32(cstage + cs * C::CSTAGE_BYTES);
                        const uint32_t b_base = smem_u32(tstage + ts * C::TSTAGE_BYTES) + C::A_RAW_BYTES;
                        if constexpr (C::PAIR) {
                            // the step's two 32-K blocks into the two buffers of hand-off pair buf
                            if (!mbar_wait(&acc_empty[buf], bph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_ACC_EMPTY)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
    #pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const uint32_t dtmem = tmem_base + (uint32_t)((2 * buf + h) * C::BN);
                                const uint32_t off = (uint32_t)(h * C::GROUP_K * 2);
                                tc_mma_f16(dtmem, smem_desc_sw128(a_base + off), smem_desc_sw128(b_base + off), C::IDESC,
                                           0u);
                                tc_mma_f16(dtmem, smem_desc_sw128(a_base + off + 32), smem_desc_sw128(b_base + off + 32),
                                           C::IDESC, 1u);
                            }
                            tc_commit(&acc_full[buf]);
                            if (++buf == C::NHAND) {
                                buf = 0;
                                bph ^= 1u;
                            }
                        } else {
    #pragma unroll
                            for (int h = 0; h < C::BK / C::GROUP_K; ++h) {
                                // one 32-K block: two K=16 MMAs into its own accumulator
                                if (!mbar_wait(&acc_empty[buf], bph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_ACC_EMPTY)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                const uint32_t dtmem = tmem_base + (uint32_t)(buf * C::BN);
                                const uint32_t off = (uint32_t)(h * C::GROUP_K * 2);
                                tc_mma_f16(dtmem, smem_desc_sw128(a_base + off), smem_desc_sw128(b_base + off), C::IDESC,
                                           0u);
                                tc_mma_f16(dtmem, smem_desc_sw128(a_base + off + 32), smem_desc_sw128(b_base + off + 32),
                                           C::IDESC, 1u);
                                tc_commit(&acc_full[buf]);
                                if (++buf == C::NBUF) {
                                    buf = 0;
                                    bph ^= 1u;
                                }
                            }
                        }
                        if (!ok) break;
                        tc_commit(&empty_c[cs]);
                        tc_commit(&empty_t[ts]);
                        if (++cs == C::CSTAGES) {
                            cs = 0;
                            cph ^= 1u;
                        }
                        if (++ts == C::TSTAGES) ts = 0;
                    }
                }
                tc_commit(drain_bar);
                drain_ring(drain_bar, 1, 1, p.err);
            }
            __syncwarp();
        } else if (C::comb_slot(warp) >= 0) {
            // ------------------------------------------------------------ combine warps (staged y)
            // warp cw takes tokens [64 cw, 64 cw + 64) of each tile: Y[token][n0 + 4 lane ..]
            // += weight * y[token][4 lane ..] as one 16-byte reduction per lane and token, or
            // (per-slot form) Yslot[row][n0 + 4 lane ..] = y[token][4 lane ..]
            const int cw = C::comb_slot(warp);
            uint32_t yph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const int entry = t / p.n_tiles;
                const int n0 = (t - entry * p.n_tiles) * C::BM;
                const int4 g4 = p.tiles[entry];
                int tk[2] = {0, 0};
                float wt[2] = {0.f, 0.f};
                if constexpr (COMBINE) {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int c = cw * 64 + 32 * i + lane;
                        tk[i] = c < g4.z ? __ldg(p.src + g4.y + c) : 0;
                        wt[i] = c < g4.z ? __ldg(p.wrow + g4.y + c) : 0.f;
                    }
                }
                if (!mbar_wait(y_full, yph, abort_flag, p.err, DEV_TIMEOUT_ACC)) {
                    ok = false;
                    break;
                }
                float* ybase = static_cast<float*>(p.Y) + n0 + 4 * lane;
                const uint32_t ys = smem_u32(ystage) + (uint32_t)(lane * 16);
                const int ncol = min(64, g4.z - cw * 64);
#pragma unroll 4
                for (int c = 0; c < ncol; ++c) {
                    const uint4 v = lds128(ys + (uint32_t)((cw * 64 + c) * C::BM * 4));
                    if constexpr (COMBINE) {
                        const int tok = __shfl_sync(0xffffffffu, tk[c >> 5], c & 31);
                        const float wc = __shfl_sync(0xffffffffu, wt[c >> 5], c & 31);
                        red_add_v4(ybase + (long)tok * p.ldy, wc * __uint_as_float(v.x), wc * __uint_as_float(v.y),
                                   wc * __uint_as_float(v.z), wc * __uint_as_float(v.w));
                    } else {
                        *reinterpret_cast<uint4*>(ybase + (long)(g4.y + cw * 64 + c) * p.ldy) = v;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(y_empty);
                yph ^= 1u;
            }
        } else if (C::conv_slot(warp) >= 0) {
            // ------------------------------------------------------------ converters (IQ4 indices -> f16)
            const int ct = C::conv_slot(warp) * 32 + lane;
            int ts = 0, cs = 0;
            uint32_t tph = 0, cph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(&full_t[ts], tph, abort_flag, p.err, DEV_TIMEOUT_TMA_FULL) ||
                        !mbar_wait(&empty_c[cs], cph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_CONV_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const uint32_t traw = smem_u32(tstage + ts * C::TSTAGE_BYTES);
                    const uint32_t cbase = smem_u32(cstage + cs * C::CSTAGE_BYTES);
    #pragma unroll
                    for (int rr = ct; rr < C::BM; rr += C::CONV_THREADS) convert_iq4_row(traw, cbase, rr);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&full_c[cs]);
                        mbar_arrive(&empty_t[ts]);
                    }
                    if (++ts == C::TSTAGES) {
                        ts = 0;
                        tph ^= 1u;
                    }
                    if (++cs == C::CSTAGES) {
                        cs = 0;
                        cph ^= 1u;
                    }
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace qmm
