// Dense Q8_0 x q8_1 projection with the output rounded to q8_1 (sm_103a).
//
//   y[m, n] = sum_b d_X[m, b] * d_W[n, b] * I[m, n, b]
//   I[m, n, b] = sum_{k in block b} Xq[m, k] * Wq[n, k]                  (exact)
//   then per 32 consecutive n of a row m: d = max|y|/127, q = round-half-away(y/d),
//   s = d * sum(q)   (the q8_1 rounding of the gate/up epilogue)
//
// ("Run Edge0-145B Q3_K on AMD HIP (Linux, gfx1100)", commit 17c02cd: the D and
// U projections of a latent layer as Q8_0 x q8_1 integer dots, 128 weight rows
// per work item, D re-quantising its products to q8_1 blocks.)
//
// The down product's structure: both operands are integers of magnitude <= 127,
// exact in f16, and a 32-element block sum stays below 2^24, so one f16
// tcgen05.mma pair per 32-K block gives I exactly in an fp32 TMEM accumulator
// (a ring of 4), folded by the epilogue with d_X * d_W in fp32.  The MMA's M side
// is 128 weight rows (output columns n), its N side 128 token rows m: each
// epilogue thread owns one n, and the 32 lanes of a warp hold 32 consecutive n,
// i.e. exactly one q8_1 block of each token row, so the block's max and code sum
// are single warp reductions.
//
// K may be long (thousands): the scales arrive per chunk of 8 blocks (256 K), d_W
// by a TMA box [128 rows][8 blocks] fp16 and d_X by a bulk copy of the chunk's
// [8 blocks][128 rows] fp32 from a per-128-row-tile layout a pre-pass writes.
//
//   warp 0: TMA producer (the weight and activation codes as f16 per K step of
//           64 - both expanded once per call by a pre-pass - and the scale
//           chunks); warp 2: MMA issuer; (with int8 weight codes, build option
//           QMM_Q8_WF16=0: warps 1, 3 expand them per K step);
//   warps 4..11: epilogue (two per TMEM lane quarter, 64 token columns each),
//           accumulators handed over two 32-K blocks at a time;
//   warps 12..15: the q8_1 rounding of each finished tile, which the epilogue
//           leaves in shared memory before it goes on to the next tile.
#include "down_iq4.cuh"

namespace qmm {

// WF16: the weight codes arrive already expanded to f16 (a pre-pass per call,
// like the activations), so the TMA stage holds both MMA operands as loaded and
// there are no converter warps: their f16 subtracts would share the FMA pipes
// with the fold, and their stores shared memory with the MMA.  Measured at
// M=2048, K=5120, N=8064 (whole call, pre-passes included): 0.514 ms against
// 0.540 with the int8 codes expanded per K step in the kernel.
#ifndef QMM_Q8_WF16
#define QMM_Q8_WF16 1
#endif
#ifndef QMM_Q8_TSTAGES
#define QMM_Q8_TSTAGES (QMM_Q8_WF16 ? 4 : 3)
#endif
#ifndef QMM_Q8_CSTAGES
#define QMM_Q8_CSTAGES (QMM_Q8_WF16 ? 0 : 3)
#endif
struct Q8Cfg {
    static constexpr int BM = 128, BN = 128, BK = 64, GROUP_K = 32;
    static constexpr bool WF16 = QMM_Q8_WF16 != 0;
    static constexpr int EPI_WARPS = 8, EPI_BASE = 4, CPW = 64, CONV_WARPS = WF16 ? 0 : 2;
    // 16 warps launched at 128 registers a thread: the two epilogue warpgroups
    // raised to 168 (running sums + two 32-column loads), the other two lowered to
    // 88 - the shares add up to exactly the launch's 16 x 128.  Warps 12..15 round
    // each finished tile, staged in shared memory, to q8_1 while the epilogue
    // folds the next tile.
    static constexpr int THREADS = 512, QUANT_BASE = 12, QUANT_WARPS = 4;
    static constexpr int REGS_LAUNCH = 128, REGS_EPI = 168, REGS_OTHER = 88;
    static_assert(8 * REGS_EPI + 8 * REGS_OTHER == 16 * REGS_LAUNCH, "register shares = launch registers");
    static constexpr int MMA_WARP = 2;
    static constexpr int TSTAGES = QMM_Q8_TSTAGES, CSTAGES = QMM_Q8_CSTAGES, SSTAGES = 2, NBUF = 4;
    // the accumulators of a K step's two 32-K blocks are handed over together (one
    // commit, one wait and one release per pair of TMEM buffers)
    static constexpr int NHAND = NBUF / 2;
    static constexpr int TMA_GROUPS = TSTAGES;
    static constexpr int CHUNK_STEPS = 4;                         // K steps of 64 per scale chunk
    static constexpr int CHUNK_BLOCKS = CHUNK_STEPS * BK / GROUP_K;   // 8 blocks of 32
    static constexpr int A_RAW_BYTES = WF16 ? BM * BK * 2 : BM * BK;   // weight codes: f16 128-byte or int8 64-byte rows
    static constexpr int B_BYTES = BN * BK * 2;                   // f16 activation codes, 128-byte rows
    static constexpr int TSTAGE_BYTES = A_RAW_BYTES + B_BYTES;
    static constexpr int CSTAGE_BYTES = WF16 ? 0 : BM * BK * 2;   // expanded weight codes
    static constexpr int DX_BYTES = CHUNK_BLOCKS * BN * 4;        // [block][token] fp32
    static constexpr int DW_BYTES = BM * CHUNK_BLOCKS * 2;        // [row][block] fp16
    static constexpr int SSTAGE_BYTES = 8192;                     // DX + DW, padded to 1 KB multiples
    static constexpr uint32_t IDESC = idesc_kind_f16(BM, BN, false);
    static constexpr int YS_BYTES = BN * BM * 4;                  // a finished tile, [token][row] fp32
    static constexpr int BAR_COUNT = 2 * TSTAGES + 2 * CSTAGES + 2 * SSTAGES + 2 * NBUF + 3;   // (NHAND <= NBUF)
    static constexpr int SMEM_BYTES = 1024 + TSTAGES * TSTAGE_BYTES + CSTAGES * CSTAGE_BYTES +
                                      SSTAGES * SSTAGE_BYTES + YS_BYTES + BAR_COUNT * 8 + 64;
    static_assert(DX_BYTES + DW_BYTES <= SSTAGE_BYTES, "scale stage");
    static_assert(TSTAGE_BYTES % 1024 == 0 && CSTAGE_BYTES % 1024 == 0 && SSTAGE_BYTES % 1024 == 0, "align");
    static_assert(WF16 == (CSTAGES == 0), "converted stages only with int8 weight codes");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// One row of 64 int8 codes (64-byte-swizzled raw rows: 16-byte chunk c of row r
// at chunk c ^ ((r >> 1) & 3)) to 64 exact f16 values in a 128-byte-swizzled
// K-major tile: x + 128 as the low byte of the f16 1024 + (x + 128), minus 1152.
__device__ __forceinline__ void convert_i8_row(uint32_t raw_tile, uint32_t dst_tile, int r) {
    const int sw = (r >> 1) & 3;
    uint4 v[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = lds128(raw_tile + r * 64 + ((c ^ sw) << 4));
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t words[4] = {v[c].x ^ 0x80808080u, v[c].y ^ 0x80808080u, v[c].z ^ 0x80808080u,
                                   v[c].w ^ 0x80808080u};
        uint32_t o[8];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            o[2 * w] = f16x2_sub(prmt(words[w], 0x64646464u, 0x5140u), kF16x2_1152);
            o[2 * w + 1] = f16x2_sub(prmt(words[w], 0x64646464u, 0x5342u), kF16x2_1152);
        }
        sts128(dst_tile + sw128_off(r, 2 * c), o[0], o[1], o[2], o[3]);
        sts128(dst_tile + sw128_off(r, 2 * c + 1), o[4], o[5], o[6], o[7]);
    }
}

// Parameters beyond GemmParams' (p.N = N output columns, p.K = K, p.tiles /
// num_entries / max_entries: the 128-token-row tiles, p.n_tiles = N / 128,
// p.dH32 = d_X per tile [entry][K/32][128] fp32).
struct Q8Out {
    int8_t* Yq;          // [M][N] q8_1 codes
    __half* Yd;          // [M][N/32]
    __half* Ys;          // [M][N/32]
    float* Y;            // [M][N] fp32 before rounding (optional)
    int M;
};

// tmA: Q8_0 codes [N][K] int8, box {64, 128}, 64-byte swizzle; or (WF16) the same
// codes as f16 values, box {64, 128}, 128-byte swizzle.
// tmB: activation codes [M][K] f16, box {64, 128}, 128-byte swizzle.
// tmW: weight scales [N][K/32] fp16, box {8, 128}, no swizzle.
__global__ void __launch_bounds__(Q8Cfg::THREADS, 1)
    q8_dense_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmW, GemmParams p, Q8Out o) {
    using C = Q8Cfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* tstage = smem;
    uint8_t* cstage = tstage + C::TSTAGES * C::TSTAGE_BYTES;
    uint8_t* sstage = cstage + C::CSTAGES * C::CSTAGE_BYTES;
    float* ystage = reinterpret_cast<float*>(sstage + C::SSTAGES * C::SSTAGE_BYTES);
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
    uint64_t* y_full = drain_bar + 1;      // a finished tile staged (epilogue warps)
    uint64_t* y_empty = y_full + 1;        // the stage read (q8_1 warps)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(y_empty + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::TSTAGES; ++i) {
            mbar_init(&full_t[i], 1);
            mbar_init(&empty_t[i], C::CONV_WARPS + 1);   // converters (codes read, int8 form) + MMA commit
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
        mbar_init(y_empty, C::QUANT_WARPS);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int ksteps = p.K / C::BK;
    const int groups = p.K / C::GROUP_K;
    const int nchunks = ksteps / C::CHUNK_STEPS;
    const int entries = min(*p.num_entries, p.max_entries);
    const int num_tiles = entries * p.n_tiles;

    // Roles.  Each warpgroup runs exactly one setmaxnreg (the epilogue warpgroups
    // the inc, the others the dec), at the top of the code it governs.
    if (warp >= C::EPI_BASE && warp < C::EPI_BASE + C::EPI_WARPS) {
        setmaxnreg_inc<C::REGS_EPI>();
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int cq = (warp - C::EPI_BASE) >> 2;   // this warp's block of 64 token columns
        const int r = q * 32 + lane;                 // this thread's weight row in the tile
        const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
        int buf = 0, ss = 0;
        uint32_t bph = 0, sph = 0, yph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            float2 y[C::CPW / 2];
#pragma unroll
            for (int j = 0; j < C::CPW / 2; ++j) y[j] = make_float2(0.f, 0.f);
            for (int kc = 0; kc < nchunks && ok; ++kc) {
                if (!mbar_wait(&full_s[ss], sph, abort_flag, p.err, DEV_TIMEOUT_ACC)) {
                    ok = false;
                    break;
                }
                const uint32_t sbase = smem_u32(sstage + ss * C::SSTAGE_BYTES);
                const uint32_t dh_base = sbase + cq * C::CPW * 4;
                const uint32_t dw_row = sbase + C::DX_BYTES + r * 16;   // this row's 8 block scales
#pragma unroll 1
                for (int gi = 0; gi < C::CHUNK_BLOCKS; gi += 2) {
                    if (!mbar_wait(&acc_full[buf], bph, abort_flag, p.err, DEV_TIMEOUT_ACC)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        const float dwf = __half2float(__ushort_as_half((unsigned short)lds_u16(dw_row + (gi + h) * 2)));
                        const float2 dw2 = make_float2(dwf, dwf);
                        const uint32_t acc = lane_addr + (uint32_t)((2 * buf + h) * C::BN + cq * C::CPW);
                        uint32_t v[2][32];
                        tmem_ld32(acc, v[0]);
                        tmem_ld32(acc + 32, v[1]);
                        tmem_ld_wait();
                        if (h == 1) {
                            // both blocks of the pair read: the buffers go back
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&acc_empty[buf]);
                        }
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const uint4 dh = lds128(dh_base + (uint32_t)(((gi + h) * C::BN + c * 32 + 4 * j) * 4));
                                const float2 i01 =
                                    make_float2(__uint_as_float(v[c][4 * j]), __uint_as_float(v[c][4 * j + 1]));
                                const float2 i23 =
                                    make_float2(__uint_as_float(v[c][4 * j + 2]), __uint_as_float(v[c][4 * j + 3]));
                                const float2 d01 = make_float2(__uint_as_float(dh.x), __uint_as_float(dh.y));
                                const float2 d23 = make_float2(__uint_as_float(dh.z), __uint_as_float(dh.w));
                                // y += (I * d_X) * d_W, both products rounded to fp32
                                float2& y01 = y[c * 16 + 2 * j];
                                float2& y23 = y[c * 16 + 2 * j + 1];
                                y01 = __ffma2_rn(__fmul2_rn(i01, d01), dw2, y01);
                                y23 = __ffma2_rn(__fmul2_rn(i23, d23), dw2, y23);
                            }
                        }
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
            }
            if (!ok) break;
            // the finished tile into the stage, [token][row] (lanes write 32 consecutive
            // rows: conflict-free), once the q8_1 warps have read the previous one
            if (!mbar_wait(y_empty, yph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_ACC)) break;
            {
                const int tok0 = cq * C::CPW;
#pragma unroll
                for (int j = 0; j < C::CPW / 2; ++j) {
                    ystage[(tok0 + 2 * j) * C::BM + r] = y[j].x;
                    ystage[(tok0 + 2 * j + 1) * C::BM + r] = y[j].y;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(y_full);
            yph ^= 1u;
        }
    } else {
        setmaxnreg_dec<C::REGS_OTHER>();
        if (warp == 0) {
            // ------------------------------------------------------------ producer (one warp)
            // Each copy of a stage comes from its own lane (a thread has one TMA copy
            // executing at a time); scale chunks from lanes 30 and 31.
            int s = 0, ss = 0;
            uint32_t ph = 0, sph = 0;
            long issued = 0, s_issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const int entry = t / p.n_tiles;
                const int n0 = (t - entry * p.n_tiles) * C::BM;
                const int4 g = p.tiles[entry];
                for (int kc = 0; kc < nchunks && ok; ++kc) {
                    const bool got_s = mbar_wait(&empty_s[ss], sph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_TMA_EMPTY);
                    if (__any_sync(0xffffffffu, !got_s)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sst = sstage + ss * C::SSTAGE_BYTES;
                    if (lane == 30) mbar_arrive_expect_tx(&full_s[ss], C::DX_BYTES + C::DW_BYTES);
                    __syncwarp();
                    if (lane == 30)
                        bulk_load(sst, p.dH32 + ((long)entry * groups + kc * C::CHUNK_BLOCKS) * C::BN, C::DX_BYTES,
                                  &full_s[ss]);
                    else if (lane == 31)
                        tma_load_2d(sst + C::DX_BYTES, &tmW, &full_s[ss], kc * C::CHUNK_BLOCKS, n0);
                    __syncwarp();
                    ++s_issued;
                    if (++ss == C::SSTAGES) {
                        ss = 0;
                        sph ^= 1u;
                    }
                    for (int kq = 0; kq < C::CHUNK_STEPS; ++kq) {
                        const int kb = kc * C::CHUNK_STEPS + kq;
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
                            tma_load_2d(st, &tmA, &full_t[s], kb * C::BK, n0);
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
            }
            if (lane == 0) {
                drain_ring(full_t, issued, C::TSTAGES, p.err);
                drain_ring(full_s, s_issued, C::SSTAGES, p.err);
            }
            __syncwarp();
        } else if (warp == C::MMA_WARP) {
            // ------------------------------------------------------------ MMA issuer (one lane)
            if (lane == 0) {
                int cs = 0, ts = 0, buf = 0;
                uint32_t cph = 0, bph = 0, tph = 0;
                bool ok = true;
                for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                    for (int kb = 0; kb < ksteps && ok; ++kb) {
                        // WF16: both operands as loaded (the TMA stage); int8 form: converted
                        // weights ready - the converters arrive on full_c only after they saw the
                        // TMA stage (weight and activation codes) complete
                        if (!(C::WF16 ? mbar_wait(&full_t[ts], tph, abort_flag, p.err, DEV_TIMEOUT_TMA_FULL)
                                      : mbar_wait(&full_c[cs], cph, abort_flag, p.err, DEV_TIMEOUT_CONV))) {
                            ok = false;
                            break;
                        }
                        const uint64_t ad = smem_desc_sw128(C::WF16 ? smem_u32(tstage + ts * C::TSTAGE_BYTES)
                                                                    : smem_u32(cstage + cs * C::CSTAGE_BYTES));
                        const uint64_t bd = smem_desc_sw128(smem_u32(tstage + ts * C::TSTAGE_BYTES) + C::A_RAW_BYTES);
                        // the step's two 32-K blocks, each into its own accumulator: the two
                        // buffers of hand-off pair buf
                        if (!mbar_wait(&acc_empty[buf], bph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_ACC_EMPTY)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int h = 0; h < C::BK / C::GROUP_K; ++h) {
                            const uint32_t dtmem = tmem_base + (uint32_t)((2 * buf + h) * C::BN);
                            // descriptor start addresses in 16-byte units: 64 bytes per 32-K block
                            tc_mma_f16(dtmem, ad + (uint64_t)(h * 4), bd + (uint64_t)(h * 4), C::IDESC, 0u);
                            tc_mma_f16(dtmem, ad + (uint64_t)(h * 4 + 2), bd + (uint64_t)(h * 4 + 2), C::IDESC, 1u);
                        }
                        tc_commit(&acc_full[buf]);
                        if (++buf == C::NHAND) {
                            buf = 0;
                            bph ^= 1u;
                        }
                        if constexpr (!C::WF16) {
                            tc_commit(&empty_c[cs]);
                            if (++cs == C::CSTAGES) {
                                cs = 0;
                                cph ^= 1u;
                            }
                        }
                        tc_commit(&empty_t[ts]);
                        if (++ts == C::TSTAGES) {
                            ts = 0;
                            tph ^= 1u;
                        }
                    }
                }
                tc_commit(drain_bar);
                drain_ring(drain_bar, 1, 1, p.err);
            }
            __syncwarp();
        } else if (!C::WF16 && (warp == 1 || warp == 3)) {
            // ------------------------------------------------------------ converters (int8 -> f16)
            const int ct = (warp == 1 ? 0 : 1) * 32 + lane;
            int ts = 0, cs = 0;
            uint32_t tph = 0, cph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                for (int kb = 0; kb < ksteps; ++kb) {
                    if (!mbar_wait(&full_t[ts], tph, abort_flag, p.err, DEV_TIMEOUT_TMA_FULL) ||
                        !mbar_wait(&empty_c[cs], cph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_CONV_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const uint32_t traw = smem_u32(tstage + ts * C::TSTAGE_BYTES);
                    const uint32_t cbase = smem_u32(cstage + cs * C::CSTAGE_BYTES);
                    convert_i8_row(traw, cbase, ct);
                    convert_i8_row(traw, cbase, ct + 64);
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
        } else if (warp >= C::QUANT_BASE) {
            // ---------------------------------------------------------- q8_1 rounding of the staged tile
            // warp w takes tokens [32 w, 32 w + 32); lane l holds n0 + 4l .. 4l + 3 of a token
            // row, so each block of 32 outputs is 8 lanes: d = max|y|/127, q =
            // round-half-away(y/d) clamped to +-127, s = d * sum q
            const int qw = warp - C::QUANT_BASE;
            uint32_t yph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const int entry = t / p.n_tiles;
                const int n0 = (t - entry * p.n_tiles) * C::BM;
                const int4 g4 = p.tiles[entry];
                if (!mbar_wait(y_full, yph, abort_flag, p.err, DEV_TIMEOUT_ACC)) {
                    ok = false;
                    break;
                }
                const int ncol = n0 + 4 * lane;
                const int nblk = (n0 >> 5) + (lane >> 3);
                const int cend = min(32, g4.z - 32 * qw);
#pragma unroll 2
                for (int c = 0; c < cend; ++c) {
                    const int tok = 32 * qw + c;
                    const uint4 u = lds128(smem_u32(ystage) + (uint32_t)((tok * C::BM + 4 * lane) * 4));
                    const float v[4] = {__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                        __uint_as_float(u.w)};
                    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
                    for (int sh = 1; sh < 8; sh <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
                    float d = 0.f;
                    int qi[4] = {0, 0, 0, 0};
                    if (amax > 0.f) {
                        d = amax / 127.0f;
#pragma unroll
                        for (int i = 0; i < 4; ++i) qi[i] = (int)fminf(fmaxf(roundf(v[i] / d), -127.f), 127.f);
                    }
                    int sum = qi[0] + qi[1] + qi[2] + qi[3];
#pragma unroll
                    for (int sh = 1; sh < 8; sh <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
                    const long m = (long)g4.y + tok;
                    const uint32_t packed = (uint32_t)(qi[0] & 0xFF) | ((uint32_t)(qi[1] & 0xFF) << 8) |
                                            ((uint32_t)(qi[2] & 0xFF) << 16) | ((uint32_t)(qi[3] & 0xFF) << 24);
                    *reinterpret_cast<uint32_t*>(o.Yq + m * p.N + ncol) = packed;
                    if ((lane & 7) == 0) {
                        o.Yd[m * (p.N / 32) + nblk] = __float2half_rn(d);
                        o.Ys[m * (p.N / 32) + nblk] = __float2half_rn(d * (float)sum);
                    }
                    if (o.Y) *reinterpret_cast<uint4*>(o.Y + m * p.N + ncol) = u;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(y_empty);
                yph ^= 1u;
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// Dense 128-row tile list {0, first row, rows, 0} of M rows, and its count.
__global__ void dense_tiles_kernel(int M, int4* tiles, int32_t* num_entries) {
    const int n = (M + 127) / 128;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        tiles[i] = make_int4(0, 128 * i, min(128, M - 128 * i), 0);
    if (blockIdx.x == 0 && threadIdx.x == 0) *num_entries = n;
}

cudaError_t launch_dense_tiles(int M, int4* tiles, int32_t* num_entries, cudaStream_t s) {
    dense_tiles_kernel<<<1, 256, 0, s>>>(M, tiles, num_entries);
    return cudaGetLastError();
}

int smem_q8_dense() { return Q8Cfg::SMEM_BYTES; }
bool q8_weights_f16() { return Q8Cfg::WF16; }

cudaError_t launch_q8_dense(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmW, const GemmParams& p,
                            int8_t* Yq, __half* Yd, __half* Ys, float* Y, int M, int grid, cudaStream_t s) {
    cudaError_t e =
        cudaFuncSetAttribute(q8_dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Q8Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // the warpgroups' register shares add up to 128 a thread: launch only if the
    // kernel is allocated exactly that many (more shares than the pool would leave
    // a setmaxnreg.inc waiting)
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, q8_dense_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != Q8Cfg::REGS_LAUNCH) return cudaErrorInvalidConfiguration;
    Q8Out o{Yq, Yd, Ys, Y, M};
    q8_dense_kernel<<<grid, Q8Cfg::THREADS, Q8Cfg::SMEM_BYTES, s>>>(tmA, tmB, tmW, p, o);
    return cudaGetLastError();
}

}  // namespace qmm
