// Warp-specialised block-quantised GEMM for sm_103a (one CTA per SM, persistent).
//
//   warp 0        : TMA producer (activations tile + raw quantised weight tile)
//   warp 1        : TMEM owner and MMA issuer (one thread issues tcgen05.mma)
//   epilogue warps: read fp32 accumulators from TMEM, scale / fold / quantise, store
//                   (12..15; 4..19 for the FP8 fold over two row sub-tiles)
//   converter warps: turn raw weight codes into the exact 16-bit operand tiles
//                    the tensor core reads, in shared memory; none of them runs on
//                    the MMA issuer's sub-partition (warp id % 4 == 1)
//
// Tile: 128*MSUB rows (tokens) x BN columns (weight rows), K step 64.  The MMA
// is tcgen05.mma.cta_group::1.kind::f16 (M=128, N=BN, K=16), MSUB of them per K
// step (one per 128-row sub-tile), fp32 accumulation in TMEM; or, with the
// operands swapped (FP8 fold, gate/up), one M=128 (weight rows), N=256 (token
// rows) MMA per K step, the accumulator transposed.  Operands are
// K-major in the canonical 128-byte-swizzled layout.  Dense problems whose last
// wave of tiles would leave half the clusters idle split those tiles along K
// (fp32 partials in the caller's workspace, added in split order by
// split_reduce_kernel).
//
// The quantised formats it reads (page titles / sections):
//  - W4: e2m1 codes with one E4M3 scale per 16 K and an fp32 scale2 applied once
//    in the epilogue ("perf: strix-hip BF16 GEMMs via hipBLASLt", commit "f16a
//    twins").  e2m1 x E4M3 is exact in bf16, so the dequantised operand is exact.
//  - FP8 with one fp32 scale per 128x128 block: each 128-K block is accumulated
//    unscaled and folded once with its scale (same page, FP8 block-scaling twin).
//  - routed-MoE gate/up: per expert, X rows of the expert's tokens times its W4
//    gate and up rows; the epilogue applies SwiGLU and rounds H to q8_1 blocks
//    of 32 ("Run Edge0-145B Q3_K on AMD HIP (Linux, gfx1100)", commit 4cb5224).
// The IQ4_NL down product has its own kernel (down_iq4.cuh) built from the
// same pieces.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "qmm_internal.h"

namespace qmm {

// CTA-pair (cta_group::2) GEMMs wherever a launch forms clusters of 2.
#ifndef QMM_PAIR
#define QMM_PAIR 0
#endif

// Short tiles (at most 128 live rows of 256) load half the activation tile.
#ifndef QMM_HALF_A
#define QMM_HALF_A 1
#endif

enum class BMode { W4, FP8 };
enum class Epi { STORE, SWIGLU_Q81, FOLD_FP8 };

template <BMode B_, Epi E_, int BN_, int CONV_WARPS_, int EPI_WARPS_, int TSTAGES_, int CSTAGES_, bool GROUPED_,
          int CLUSTER_N_ = 1, int MSUB_ = 1, bool PAIR_ = false, bool SWAP_ = false>
struct GemmCfg {
    static constexpr BMode B = B_;
    // Operands swapped (FP8 fold, gate/up): the converted weight tile is the
    // MMA's A operand (M = 128 weight rows) and the 256-row activation tile its B
    // operand (N = 256 token rows, or the tile's live rows rounded up to 16), one
    // MMA per K step of 16 instead of one per 128-row sub-tile.  An N = 256 MMA
    // reads 12 KB of shared-memory operands per 128 cycles, two N = 128 MMAs 16 KB,
    // and shared-memory bandwidth (operand reads, converter stores, TMA writes)
    // bounds these kernels.  The accumulator is transposed: TMEM lane = weight
    // row, column = token row.
    static constexpr bool SWAP = SWAP_;
    static_assert(!SWAP_ || (MSUB_ == 2 && !PAIR_ && BN_ == 128 &&
                             ((E_ == Epi::FOLD_FP8 && EPI_WARPS_ == 16) || (E_ == Epi::SWIGLU_Q81 && EPI_WARPS_ == 4))),
                  "swapped operands: FP8 fold or gate/up over 256 x 128 tiles");
    // gate/up, swapped: the converted rows are placed so that TMEM lane quarter q
    // holds gate rows f = 16q .. 16q + 15 (lanes 0..15) and the up rows of the same
    // f (lanes 16..31); SwiGLU pairs lanes l and l + 16, and h passes through a
    // shared stage of 32 tokens x 64 f (two buffers, rows padded to 65 floats) to
    // be rounded to q8_1 along f
    static constexpr bool SWAP_GU = SWAP_ && E_ == Epi::SWIGLU_Q81;
    static constexpr int HS_STRIDE = 65, HS_FLOATS = 32 * HS_STRIDE;
    static constexpr int HS_BYTES = SWAP_GU ? 2 * HS_FLOATS * 4 : 0;
    __device__ static int conv_dst_row(int r) {
        if constexpr (SWAP_GU) {
            const int f = r & 63, up = r >> 6;
            return ((f >> 4) << 5) | (up << 4) | (f & 15);
        } else {
            return r;
        }
    }

    // CTA pair (cta_group::2): the two CTAs of a cluster of 2 compute one
    // 256 x 2*BN tile with M = 256 MMAs issued by the even CTA.  Each CTA holds
    // 128 activation rows and converts BN weight rows (its half of the MMA's N);
    // its TMEM receives its 128 rows x all 2*BN columns.  Every MMA then reads
    // half of each operand from each CTA's shared memory, which halves the
    // shared-memory operand traffic per FLOP against a one-CTA M = 128 MMA.
    static constexpr bool PAIR = PAIR_;
    static_assert(!PAIR || (CLUSTER_N_ == 2 && MSUB_ == 1), "CTA pair: a cluster of 2, one 128-row tile per CTA");
    // accumulator columns per row sub-tile, and rows of the tile a work item covers
    static constexpr int ACC_N = PAIR_ ? 2 * BN_ : BN_;
    static constexpr int TILE_M = PAIR_ ? 256 : 128 * MSUB_;
    // MSUB row blocks of 128 share every converted weight tile: each K step
    // issues MSUB MMAs (one per 128-row sub-tile) against the same B operand,
    // which divides the conversion work per FLOP by MSUB.
    static constexpr int MSUB = MSUB_;
    // CTAs of a cluster work on the same activation rows and consecutive column
    // tiles; each loads 1/CLUSTER_N of the activation tile and multicasts it to
    // all, so the activations cross L2 once per cluster instead of once per CTA.
    static constexpr int CLUSTER_N = CLUSTER_N_;
    static constexpr int A_SLICE_ROWS = PAIR_ ? 128 : 128 * MSUB_ / CLUSTER_N_;
    static constexpr Epi EPI = E_;
    static constexpr bool GROUPED = GROUPED_;
    static constexpr int BM = 128 * MSUB_, BN = BN_, BK = 64, UMMA_K = 16;
    static constexpr int CONV_WARPS = CONV_WARPS_, EPI_WARPS = EPI_WARPS_;
    // 16 warps (20, 24 or 28 for the FP8 fold).  Warp w runs on SM sub-partition w % 4; the MMA issuer (warp 1)
    // must not share its sub-partition with ALU-heavy converter warps, or its
    // mbarrier waits are starved and the tensor pipe idles.
    // WIDE16: a W4 tile with 16 converter warps (the wide 256-row tile, two
    // threads per weight row, or gate/up's 128 rows, four threads per row): 28
    // warps, the epilogue on warps 24..27
    static constexpr bool WIDE16 = (B_ == BMode::W4 && EPI_WARPS_ == 4 && CONV_WARPS_ == 16 && !PAIR_);
    static constexpr int EPI_BASE = WIDE16 ? 24 : ((EPI_WARPS_ == 4) ? 12 : 4);
    // 16 fold warps (FP8 with two row sub-tiles) and 2 converters: 20 warps, five
    // per sub-partition, the converters on warps 2 and 3.
    // 16 fold warps with 4 converters: 24 warps launched at 80 registers a thread,
    // the four fold warpgroups raised to 96 (64 running sums a thread), the other
    // two lowered to 48 - the shares add up to exactly the launch's 24 x 80.
    // With 8 converters (two threads per weight row): 28 warps launched at 72, the
    // fold warpgroups raised to 96 and the other three lowered to 40.
    static constexpr bool REG_SPLIT = (EPI_WARPS_ == 16 && (CONV_WARPS_ == 4 || CONV_WARPS_ == 8)) || WIDE16;
    static constexpr int SPLIT_WARPS = (CONV_WARPS_ == 8 || WIDE16) ? 28 : 24;
    static constexpr int REGS_LAUNCH = (CONV_WARPS_ == 8 || WIDE16) ? 72 : 80;
    static constexpr int REGS_EPI = WIDE16 ? 120 : 96, REGS_OTHER = WIDE16 ? 64 : ((CONV_WARPS_ == 8) ? 40 : 48);
    static_assert(!REG_SPLIT || EPI_WARPS_ * REGS_EPI + (SPLIT_WARPS - EPI_WARPS_) * REGS_OTHER == SPLIT_WARPS * REGS_LAUNCH,
                  "register shares = launch registers");
    static constexpr int THREADS = REG_SPLIT ? 32 * SPLIT_WARPS : ((EPI_WARPS_ == 16) ? 32 * 20 : 512);
    // one CTA per SM: each sub-partition's 16384 registers shared by its warps,
    // in the allocation unit of 8 per thread
    static constexpr int WARPS_PER_SMSP = (THREADS / 32 + 3) / 4;
    static constexpr int MAXNREG_RAW = 16384 / (WARPS_PER_SMSP * 32) / 8 * 8;
    static constexpr int MAXNREG = REG_SPLIT ? REGS_LAUNCH : (MAXNREG_RAW > 255 ? 255 : MAXNREG_RAW);
    // fold epilogue: token columns per warp, and the TMEM load width
    static constexpr int FOLD_CPW = ACC_N / (EPI_WARPS_ >= 8 ? EPI_WARPS_ / 4 : 1);
    static constexpr int FOLD_LDW = (EPI_WARPS_ == 16) ? 16 : 32;
    static constexpr int TSTAGES = TSTAGES_, CSTAGES = CSTAGES_;
    // converted stages handed over per proxy fence (at most CSTAGES / 2, so that
    // the MMA always holds a batch while the converters fill the next)
#ifndef QMM_CONV_BATCH
#define QMM_CONV_BATCH 1
#endif
    static constexpr int CONV_BATCH = (QMM_CONV_BATCH < CSTAGES_ / 2) ? QMM_CONV_BATCH : (CSTAGES_ / 2 > 0 ? CSTAGES_ / 2 : 1);
    // producer lane groups (4 lanes each: activation copy, one or two weight copies)
    static constexpr int TMA_GROUPS = TSTAGES_;
    static_assert(TMA_GROUPS * 4 <= 32, "producer lane groups fit one warp");
    // raw (TMA) stage: bf16 activation tile (read by the MMA in place) + weight codes
    static constexpr int A_RAW_BYTES = BM * BK * 2;
    static constexpr int B_ROW_BYTES = (B_ == BMode::FP8) ? 64 : 32;   // bytes of codes per weight row per k-block
    static constexpr int B_RAW_BYTES = BN * B_ROW_BYTES;
    static constexpr int TSTAGE_BYTES = A_RAW_BYTES + B_RAW_BYTES;
    // converted stage: the bf16 weight tile
    static constexpr int CSTAGE_BYTES = BN * BK * 2;
    // accumulation groups: the whole K, or one per 128-K block (FP8 fold)
    static constexpr bool FOLD = (E_ == Epi::FOLD_FP8);
    static constexpr int GROUP_K = FOLD ? 128 : 0;   // 0: whole K
    static_assert(GROUP_K == 0 || GROUP_K == 2 * BK, "fold groups span two K blocks");
    static constexpr int NBUF = 512 / (ACC_N * MSUB_);
    static constexpr uint32_t IDESC = PAIR_ ? idesc_kind_f16(256, 2 * BN_, true) : idesc_kind_f16(128, BN_, true);
    static_assert(ACC_N <= 256, "MMA N");
    // converter threads per weight row, or weight rows per converter thread
    static constexpr int TPR = (CONV_WARPS_ * 32 >= BN_) ? CONV_WARPS_ * 32 / BN_ : 1;
    static constexpr int RPT = (CONV_WARPS_ * 32 >= BN_) ? 1 : BN_ / (CONV_WARPS_ * 32);
    static constexpr int BAR_COUNT = 2 * TSTAGES + 3 * CSTAGES + 2 * NBUF + 1 + (SWAP_GU ? 2 : 0);
    static constexpr int SMEM_BYTES =
        1024 /*align slack*/ + TSTAGES * TSTAGE_BYTES + CSTAGES * CSTAGE_BYTES + HS_BYTES + BAR_COUNT * 8 + 64;
    static_assert(TSTAGE_BYTES % 1024 == 0 && CSTAGE_BYTES % 1024 == 0, "stage alignment");
    static_assert(BN % 32 == 0 && BN <= 256, "BN");
    static_assert(!FOLD || EPI_WARPS == 8 || EPI_WARPS == 16, "fold epilogue: two or four warps per lane quarter");
    static_assert(!FOLD || FOLD_CPW % 8 == 0, "fold columns per warp: whole 16-byte runs");
    static_assert(GROUPED_ || 128 * MSUB_ * ACC_N <= 65536, "split partial tile at most 256 x 256");
    static_assert(FOLD || EPI_WARPS == 4, "store epilogue uses one warpgroup");
    static_assert(TPR == 1 || TPR == 2 || (TPR == 4 && B_ == BMode::W4), "one, two or (W4) four converter threads per weight row");
    static_assert(CONV_WARPS * 32 * RPT == TPR * BN, "converters cover the weight rows");
    static_assert(RPT == 1 || (RPT == 2 && B_ == BMode::FP8), "two rows per converter thread: FP8 only");
    static_assert(MSUB == 1 || MSUB == 2, "row sub-tiles");
    static_assert(MSUB == 1 || !FOLD || EPI_WARPS == 16, "two-sub-tile folds need 16 fold warps (registers)");
    static_assert(NBUF >= 1, "TMEM columns");
    static_assert(CLUSTER_N == 1 || CLUSTER_N == 2 || CLUSTER_N == 4, "cluster size");
    static_assert((EPI_WARPS == 4 && CONV_WARPS == 8) || (EPI_WARPS == 8 && CONV_WARPS == 4) ||
                      (EPI_WARPS == 16 && (CONV_WARPS == 2 || CONV_WARPS == 4 || CONV_WARPS == 8)) || WIDE16,
                  "warp layout");
    // relay threads of a pair's odd CTA: lane 0 of the MMA warp (slot 0) and of the
    // warps without a role (slots 1, 2: warps 5 and 9 with 4 epilogue warps)
#ifndef QMM_RELAYS
#define QMM_RELAYS 3
#endif
    static constexpr int RELAYS = (PAIR_ && EPI_WARPS_ == 4) ? QMM_RELAYS : 1;
    // a relay waits on a converted stage's barrier only after forwarding the stage
    // RELAYS before it, which completes the barrier's previous phase only if
    // RELAYS <= CSTAGES (a parity wait two phases ahead would pass at once)
    static_assert(RELAYS >= 1 && RELAYS <= 3 && (!PAIR_ || RELAYS <= CSTAGES_), "relay threads");
    __device__ static int relay_slot(int warp) {
        if (warp == 1) return 0;
        if (EPI_WARPS == 4 && RELAYS >= 2 && warp == 5) return 1;
        if (EPI_WARPS == 4 && RELAYS >= 3 && warp == 9) return 2;
        return -1;
    }
    // converter slot of a warp, -1 if it is not a converter:
    //   4 epilogue warps (12..15):  converters on warps 2,3,4,6,7,8,10,11
    //   8 epilogue warps (4..11):   converters on warps 2,3,12,14
    //   16 epilogue warps (4..19):  converters on warps 2,3 (and 20, 23 with four;
    //                               20, 22, 23, 24, 26, 27 with eight)
    __device__ static int conv_slot(int warp) {
        if constexpr (WIDE16) {
            // warps 2..22 not on sub-partition 1: 2,3,4,6,7,8,10,11,12,14,15,16,18,19,20,22
            if (warp < 2 || warp > 22 || (warp & 3) == 1) return -1;
            const int r = warp - 2 - (warp - 1) / 4;   // drop the sub-partition-1 warps below
            return r < 16 ? r : -1;
        }
        if constexpr (EPI_WARPS == 16) {
            if (warp == 2 || warp == 3) return warp - 2;
            if (CONV_WARPS == 4 && warp == 20) return 2;
            if (CONV_WARPS == 4 && warp == 23) return 3;
            // 8 converters: warps 2, 3, 20, 22, 23, 24, 26, 27 (none on sub-partition 1)
            if (CONV_WARPS == 8 && warp >= 20 && warp < 28)
                return (int)((0x87065403u >> (4 * (warp - 20))) & 15u) - 1;   // slot + 1 per warp, one nibble each
            return -1;
        } else {
            // slot + 1 per warp, one nibble each (0: not a converter)
            constexpr unsigned long long tab = (EPI_WARPS == 4) ? 0x870654032100ull : 0x403000000002100ull;
            return (int)((tab >> (4 * warp)) & 15u) - 1;
        }
    }
};

struct TileInfo {
    int expert, row0, rows, n0, entry;
    int kb0, kb1;   // K blocks [kb0, kb1) of this work item
    int split, s;   // dense K split: index of the split tile and of this split, or split = -1
};

// Work item g of a cluster: one block of activation rows and CLUSTER_N
// consecutive column tiles; CTA `crank` of the cluster takes column tile
// ng * CLUSTER_N + crank.  (p.n_tiles is a multiple of CLUSTER_N.)
template <class C>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int g, int crank) {
    TileInfo ti;
    const int n_groups = p.n_tiles / C::CLUSTER_N;
    if constexpr (C::GROUPED) {
        const int entry = g / n_groups, nt = (g - entry * n_groups) * C::CLUSTER_N + crank;
        const int4 e4 = p.tiles[entry];
        ti.expert = e4.x;
        if constexpr (C::PAIR) {
            // the 256-row tile's half held by this CTA of the pair (rows may be 0)
            ti.row0 = e4.y + crank * 128;
            ti.rows = max(0, min(128, e4.z - crank * 128));
            ti.entry = e4.w + crank;
        } else {
            ti.row0 = e4.y;
            ti.rows = e4.z;
            // index of the first 128-row routing entry the tile covers (two per tile when MSUB == 2)
            ti.entry = (C::MSUB == 2) ? e4.w : entry;
        }
        ti.n0 = nt * p.n_step;
        ti.kb0 = 0;
        ti.kb1 = (p.K + C::BK - 1) / C::BK;
        ti.split = -1;
        ti.s = 0;
    } else {
        // items from split_from on: split_S K ranges (whole 4-K-block chunks) per tile
        int tile = g, split = -1, s = 0;
        if (g >= p.split_from) {
            const int j = g - p.split_from;
            split = j / p.split_S;
            s = j - split * p.split_S;
            tile = p.split_from + split;
        }
        const int mt = tile % p.m_tiles, nt = (tile / p.m_tiles) * C::CLUSTER_N + crank;
        ti.expert = 0;
        if constexpr (C::PAIR) {
            ti.row0 = mt * C::TILE_M + crank * 128;
            ti.rows = max(0, min(128, p.M - ti.row0));
        } else {
            ti.row0 = mt * C::BM;
            ti.rows = min(C::BM, p.M - ti.row0);
        }
        ti.n0 = nt * p.n_step;
        ti.entry = mt;
        const int kblocks = (p.K + C::BK - 1) / C::BK;   // K % 64 == 32: a last half block
        if (split >= 0) {
            const int nch = kblocks / 4;
            ti.kb0 = 4 * (s * nch / p.split_S);
            ti.kb1 = 4 * ((s + 1) * nch / p.split_S);
        } else {
            ti.kb0 = 0;
            ti.kb1 = kblocks;
        }
        ti.split = split;
        ti.s = s;
    }
    return ti;
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void sts128(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t saddr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr) : "memory");
    return v;
}

// bf16 value 2^112 in both halves: f16 bits >> 3 read as bf16 are the f16 value
// times 2^-112 (exponent bias 15 vs 127), so this factor restores it exactly.
constexpr uint32_t kBf16x2_2p112 = 0x77807780u;
// f16x2 -> bf16x2 bit patterns whose values are the f16 values times 2^-112,
// valid when the low 3 mantissa bits of both halves are zero (true for every
// e2m1 and E4M3 value).  The shift by 3 lines the 5-bit f16 exponent up with
// the low bits of the bf16 exponent and leaves each sign bit 3 places too low
// (bits 12 / 28, with zeros above); adding 7 times that bit moves it up to bit
// 15 / 31 by carry.
__device__ __forceinline__ uint32_t f16x2_to_bf16x2_2m112(uint32_t h) {
    const uint32_t a = h >> 3;
    return a + (a & 0x10001000u) * 7u;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a), y = *reinterpret_cast<__nv_bfloat162*>(&b);
    __nv_bfloat162 r = __hmul2(x, y);
    return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
    __half2 x = *reinterpret_cast<__half2*>(&a), y = *reinterpret_cast<__half2*>(&b);
    __half2 r = __hsub2(x, y);
    return *reinterpret_cast<uint32_t*>(&r);
}

// E4M3 scale byte -> bf16x2 of (scale * 2^112), exact.
__device__ __forceinline__ uint32_t w4_scale_bf16x2(uint32_t byte) {
    uint32_t h[2];
    cvt_e4m3x4_f16x2(byte & 0xFFu, h);
    const float s = __half2float(__ushort_as_half((unsigned short)(h[0] & 0xFFFFu))) * 5.192296858534828e33f;   // 2^112
    const __nv_bfloat16 b = __float2bfloat16_rn(s);
    const uint32_t u = __bfloat16_as_ushort(b);
    return u | (u << 16);
}

// f16 bits 0x64XX are 1024 + XX; subtracting 1152 leaves XX - 128 (int8 codes
// biased by 128 into exact f16).
constexpr uint32_t kF16x2_1152 = 0x64806480u;
// The f16 bit patterns of the IQ4_NL codebook values (index 0..15: -127 -104 -83
// -65 -49 -35 -22 -10 1 13 25 38 53 69 89 113) as a low-byte and a high-byte
// table, four entries per word: the expansion needs only byte permutes, no f16
// arithmetic on the FMA pipes that the down product's fold uses (measured: the
// down product 2% faster than building value + 128 and subtracting in f16).
constexpr uint32_t kIq4L0 = 0x103080F0u, kIq4L1 = 0x00806020u, kIq4L2 = 0xC0408000u, kIq4L3 = 0x109050A0u;
constexpr uint32_t kIq4H0 = 0xD4D5D6D7u, kIq4H1 = 0xC9CDD0D2u, kIq4H2 = 0x504E4A3Cu, kIq4H3 = 0x57555452u;

// ---------------------------------------------------------------------------
// Row converters: one thread turns one row of raw codes for a 64-wide K block
// into 64 exact 16-bit operand values, written as 8 chunks of 16 bytes into a
// 128-byte-swizzled K-major tile.

// W4: 64 e2m1 codes (32 bytes, 32-byte-swizzled rows) and 4 E4M3 scale bytes;
// raw row r becomes row rd of the operand tile.
__device__ __forceinline__ void convert_w4_row(uint32_t raw_tile, uint32_t dst_tile, int r, int rd, uint32_t sbytes) {
    const int sw = (r >> 2) & 1;
    const uint4 c0 = lds128(raw_tile + r * 32 + ((0 ^ sw) << 4));
    const uint4 c1 = lds128(raw_tile + r * 32 + ((1 ^ sw) << 4));
    uint32_t sc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[i] = w4_scale_bf16x2(sbytes >> (8 * i));
    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        uint32_t h[4], o[4];
        cvt_e2m1x8_f16x2(words[w], h);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = bf16x2_mul(f16x2_to_bf16x2_2m112(h[i]), sc[w >> 1]);
        sts128(dst_tile + sw128_off(rd, w), o[0], o[1], o[2], o[3]);
    }
}

// W4, half a row: the 32 codes of K half h (one 16-byte chunk) and their 2 scales.
__device__ __forceinline__ void convert_w4_half(uint32_t raw_tile, uint32_t dst_tile, int r, int rd, int h, uint32_t sbytes) {
    const int sw = (r >> 2) & 1;
    const uint4 c = lds128(raw_tile + r * 32 + ((h ^ sw) << 4));
    const uint32_t sc0 = w4_scale_bf16x2(sbytes >> (16 * h));
    const uint32_t sc1 = w4_scale_bf16x2(sbytes >> (16 * h + 8));
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t hh[4], o[4];
        cvt_e2m1x8_f16x2(words[w], hh);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = bf16x2_mul(f16x2_to_bf16x2_2m112(hh[i]), (w < 2) ? sc0 : sc1);
        sts128(dst_tile + sw128_off(rd, 4 * h + w), o[0], o[1], o[2], o[3]);
    }
}

// W4, a quarter row: the 16 codes of K quarter qt (8 bytes) and their scale.
__device__ __forceinline__ void convert_w4_quarter(uint32_t raw_tile, uint32_t dst_tile, int r, int rd, int qt,
                                                   uint32_t sbytes) {
    const int sw = (r >> 2) & 1;
    uint32_t c0, c1;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                 : "=r"(c0), "=r"(c1)
                 : "r"(raw_tile + r * 32 + (((qt >> 1) ^ sw) << 4) + (qt & 1) * 8)
                 : "memory");
    const uint32_t sc = w4_scale_bf16x2(sbytes >> (8 * qt));
    const uint32_t words[2] = {c0, c1};
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        uint32_t hh[4], o[4];
        cvt_e2m1x8_f16x2(words[w], hh);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = bf16x2_mul(f16x2_to_bf16x2_2m112(hh[i]), sc);
        sts128(dst_tile + sw128_off(rd, 2 * qt + w), o[0], o[1], o[2], o[3]);
    }
}

// FP8: RPT rows (r0, r0 + rstride, ...) of 64 E4M3 bytes (64-byte-swizzled rows) -> exact bf16.
template <int RPT>
__device__ __forceinline__ void convert_fp8_rows(uint32_t raw_tile, uint32_t dst_tile, int r0, int rstride) {
    // all raw chunks first: the shared loads overlap instead of each waiting on the last store
    uint4 v[RPT][4];
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) {
        const int r = r0 + rr * rstride, sw = (r >> 1) & 3;
#pragma unroll
        for (int c = 0; c < 4; ++c) v[rr][c] = lds128(raw_tile + r * 64 + ((c ^ sw) << 4));
    }
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) {
        const int r = r0 + rr * rstride;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t words[4] = {v[rr][c].x, v[rr][c].y, v[rr][c].z, v[rr][c].w};
            uint32_t o[8];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                uint32_t h[2];
                cvt_e4m3x4_f16x2(words[w], h);
                o[2 * w] = bf16x2_mul(f16x2_to_bf16x2_2m112(h[0]), kBf16x2_2p112);
                o[2 * w + 1] = bf16x2_mul(f16x2_to_bf16x2_2m112(h[1]), kBf16x2_2p112);
            }
            sts128(dst_tile + sw128_off(r, 2 * c), o[0], o[1], o[2], o[3]);
            sts128(dst_tile + sw128_off(r, 2 * c + 1), o[4], o[5], o[6], o[7]);
        }
    }
}

// FP8, half a row: the 32 E4M3 bytes of K half h (two 16-byte chunks).
__device__ __forceinline__ void convert_fp8_half(uint32_t raw_tile, uint32_t dst_tile, int r, int h) {
    const int sw = (r >> 1) & 3;
    uint4 v[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) v[i] = lds128(raw_tile + r * 64 + (((2 * h + i) ^ sw) << 4));
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t words[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        uint32_t o[8];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t hh[2];
            cvt_e4m3x4_f16x2(words[w], hh);
            o[2 * w] = bf16x2_mul(f16x2_to_bf16x2_2m112(hh[0]), kBf16x2_2p112);
            o[2 * w + 1] = bf16x2_mul(f16x2_to_bf16x2_2m112(hh[1]), kBf16x2_2p112);
        }
        const int c = 2 * h + i;
        sts128(dst_tile + sw128_off(r, 2 * c), o[0], o[1], o[2], o[3]);
        sts128(dst_tile + sw128_off(r, 2 * c + 1), o[4], o[5], o[6], o[7]);
    }
}

// IQ4_NL: 64 4-bit indices (32 bytes, 32-byte-swizzled rows) -> exact f16 codebook values.
__device__ __forceinline__ void convert_iq4_row(uint32_t raw_tile, uint32_t dst_tile, int r) {
    const int sw = (r >> 2) & 1;
    const uint4 c0 = lds128(raw_tile + r * 32 + ((0 ^ sw) << 4));
    const uint4 c1 = lds128(raw_tile + r * 32 + ((1 ^ sw) << 4));
    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t x = words[w];
        const uint32_t x4 = x << 4;
        const uint32_t xh = x >> 16;
        // elements 0..3 (low 16 bits) and 4..7 (high 16 bits): table entries 0-7 or
        // 8-15 chosen by bit 3 of each index (a byte mask of it by sign replication)
        const uint32_t ma = prmt(x4, x, 0xD9C8u), mb = prmt(x4, x, 0xFBEAu);
        // low and high bytes of the f16 values, interleaved into f16 pairs
        const uint32_t la = bitselect(prmt(kIq4L0, kIq4L1, x), prmt(kIq4L2, kIq4L3, x & 0x7777u), ma);
        const uint32_t ha = bitselect(prmt(kIq4H0, kIq4H1, x), prmt(kIq4H2, kIq4H3, x & 0x7777u), ma);
        const uint32_t lb = bitselect(prmt(kIq4L0, kIq4L1, xh), prmt(kIq4L2, kIq4L3, xh & 0x7777u), mb);
        const uint32_t hb = bitselect(prmt(kIq4H0, kIq4H1, xh), prmt(kIq4H2, kIq4H3, xh & 0x7777u), mb);
        sts128(dst_tile + sw128_off(r, w), prmt(la, ha, 0x5140u), prmt(la, ha, 0x7362u), prmt(lb, hb, 0x5140u),
               prmt(lb, hb, 0x7362u));
    }
}

// Wait (bounded) for the completion of the `issued` most recent fills of a ring.
__device__ __forceinline__ void drain_ring(uint64_t* full, long issued, int stages, uint32_t* err) {
    const long pending = issued < stages ? issued : stages;
    for (long i = 0; i < pending; ++i) {
        const long idx = issued - 1 - i;
        const int s = (int)(idx % stages);
        const uint32_t par = (uint32_t)((idx / stages) & 1);
        if (mbar_try_wait(&full[s], par)) continue;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&full[s], par)) {
            if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
                atomicCAS(err, 0u, DEV_TIMEOUT_DRAIN);
                break;
            }
        }
    }
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// 32 consecutive outputs of one row, times s2, as fp32 or bf16 (RNE).
__device__ __forceinline__ void store_out32(const GemmParams& p, long grow, int col, const float (&v)[32], float s2) {
    if (p.ydt == 0) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.Y) + grow * p.ldy + col);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(v[4 * j] * s2, v[4 * j + 1] * s2, v[4 * j + 2] * s2, v[4 * j + 3] * s2);
    } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.Y) + grow * p.ldy + col);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                __nv_bfloat162 b = __floats2bfloat162_rn(v[8 * j + 2 * i] * s2, v[8 * j + 2 * i + 1] * s2);
                w[i] = *reinterpret_cast<uint32_t*>(&b);
            }
            dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// K splits of the last wave: out[tile rows, tile columns] = scale x (sum of the
// S partial tiles in split order), one thread per 4 consecutive columns; rows
// and columns outside [M, N) are not written.  Partials as in GemmParams: one
// BM x BN partial per CTA, the CTAs of a cluster on consecutive column tiles,
// or (pair) on the two 128-row halves of a 256-row tile with all BN columns.
static __global__ void __launch_bounds__(256) split_reduce_kernel(GemmParams p, int BM, int BN, int CN, int rem, float scale,
                                                                  bool cta_pair) {
    const long per_tile = (long)BM * (BN / 4);
    const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long)rem * CN * per_tile) return;
    const int pair = (int)(idx / per_tile);                 // split tile x cluster rank
    const int within = (int)(idx - (long)pair * per_tile);
    const int r = within / (BN / 4), c4 = within - r * (BN / 4);
    const int j = pair / CN, crank = pair - j * CN;
    const int tile = p.split_from + j;
    const int mt = tile % p.m_tiles;
    const long grow = cta_pair ? (long)mt * 256 + crank * 128 + r : (long)mt * BM + r;
    const int col =
        cta_pair ? (tile / p.m_tiles) * CN * p.n_step + c4 * 4 : ((tile / p.m_tiles) * CN + crank) * p.n_step + c4 * 4;
    if (grow >= p.M || col >= p.N) return;
    const float4* src = reinterpret_cast<const float4*>(p.split_part + (long)pair * p.split_S * BM * BN + (long)r * BN) + c4;
    const long sstride = (long)BM * BN / 4;
    float4 v = __ldcg(src);
    for (int s = 1; s < p.split_S; ++s) {
        const float4 x = __ldcg(src + s * sstride);
        v.x += x.x;
        v.y += x.y;
        v.z += x.z;
        v.w += x.w;
    }
    if (p.ydt == 0) {
        *reinterpret_cast<float4*>(static_cast<float*>(p.Y) + grow * p.ldy + col) =
            make_float4(v.x * scale, v.y * scale, v.z * scale, v.w * scale);
    } else {
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x * scale, v.y * scale);
        __nv_bfloat162 b = __floats2bfloat162_rn(v.z * scale, v.w * scale);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.Y) + grow * p.ldy + col) =
            make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    }
}

template <class C>
__global__ void __launch_bounds__(C::THREADS) __maxnreg__(C::MAXNREG)
    qgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* tstage = smem;
    uint8_t* cstage = tstage + C::TSTAGES * C::TSTAGE_BYTES;
    float* hstage = reinterpret_cast<float*>(cstage + C::CSTAGES * C::CSTAGE_BYTES);   // gate/up swapped: h
    uint64_t* bars = reinterpret_cast<uint64_t*>(cstage + C::CSTAGES * C::CSTAGE_BYTES + C::HS_BYTES);
    uint64_t* full_t = bars;
    uint64_t* empty_t = full_t + C::TSTAGES;
    uint64_t* full_c = empty_t + C::TSTAGES;
    uint64_t* empty_c = full_c + C::CSTAGES;
    uint64_t* acc_full = empty_c + C::CSTAGES;
    uint64_t* acc_empty = acc_full + C::NBUF;
    uint64_t* drain_bar = acc_empty + C::NBUF;
    uint64_t* conv_done = drain_bar + 1;   // pair, odd CTA: its converters' local hand-off to the relay
    uint64_t* hs_full = conv_done + C::CSTAGES;   // gate/up swapped: h stage buffer written by every epilogue warp
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(hs_full + (C::SWAP_GU ? 2 : 0));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::TSTAGES; ++i) {
            mbar_init(&full_t[i], 1);
            // released by the MMA commit of every CTA of the cluster (each read the multicast
            // tile), or (pair) by the pair's one MMA commit
            mbar_init(&empty_t[i], C::PAIR ? 1 : C::CLUSTER_N);
        }
        // pair: the MMA issuer (even CTA) waits on its own full_c, which its converters
        // arrive on and, once per stage, the odd CTA's relay thread; and on its own
        // acc_empty, which the epilogue warps of both CTAs arrive on
        for (int i = 0; i < C::CSTAGES; ++i) {
            mbar_init(&full_c[i], C::PAIR ? C::CONV_WARPS + 1 : C::CONV_WARPS);
            mbar_init(&empty_c[i], 1);
            mbar_init(&conv_done[i], C::CONV_WARPS);
        }
        for (int i = 0; i < C::NBUF; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], (C::PAIR ? 2 : 1) * C::EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        if constexpr (C::SWAP_GU) {
            mbar_init(&hs_full[0], C::EPI_WARPS);
            mbar_init(&hs_full[1], C::EPI_WARPS);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        if (!p.wmaps) tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        if constexpr (C::PAIR)
            tmem_alloc_pair(tmem_slot, 512);
        else
            tmem_alloc(tmem_slot, 512);
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (C::CLUSTER_N > 1) cluster_sync();   // peers' barriers are initialised before any multicast
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int crank = (C::CLUSTER_N > 1) ? (int)cluster_ctarank() : 0;
    // the pair's MMA issuer and the owner of the barriers both CTAs arrive on
    const bool pair_leader = !C::PAIR || crank == 0;
    const int cid = (C::CLUSTER_N > 1) ? (int)cluster_id_x() : (int)blockIdx.x;
    const int ncl = (C::CLUSTER_N > 1) ? (int)cluster_count_x() : (int)gridDim.x;
    int num_tiles;   // work items (one per cluster step)
    if constexpr (C::GROUPED) {
        const int entries = min(*p.num_entries, p.max_entries);
        num_tiles = entries * (p.n_tiles / C::CLUSTER_N);
    } else {
        const int items = p.m_tiles * (p.n_tiles / C::CLUSTER_N);
        num_tiles = (p.split_S > 1) ? p.split_from + (items - p.split_from) * p.split_S : items;
    }

    // Relay r of the odd CTA of a pair (r < RELAYS): the converted stages with
    // global index i = r (mod RELAYS), each once all of that CTA's converters have
    // handed it over (conv_done), to the even CTA's full_c with a cluster-scope
    // release.  Several relay threads forward consecutive stages concurrently.
    auto relay_stages = [&](int r) {
        long i = 0;
        bool ok = true;
        for (int t = cid; t < num_tiles && ok; t += ncl) {
            const TileInfo ri = decode_tile<C>(p, t, crank);
            for (int kb = ri.kb0; kb < ri.kb1; ++kb, ++i) {
                if (i % C::RELAYS != r) continue;
                const int cs = (int)(i % C::CSTAGES);
                const uint32_t cph = (uint32_t)((i / C::CSTAGES) & 1);
                if (!mbar_wait(&conv_done[cs], cph, abort_flag, p.err, DEV_TIMEOUT_CONV)) {
                    ok = false;
                    break;
                }
                mbar_arrive_cluster(&full_c[cs], 0);
            }
        }
    };

    // Roles.  With the register split, each warpgroup runs exactly one setmaxnreg
    // (the fold warpgroups the inc, the others the dec), at the top of the code it
    // governs.
    if (warp >= C::EPI_BASE && warp < C::EPI_BASE + C::EPI_WARPS) {
        if constexpr (C::REG_SPLIT) setmaxnreg_inc<C::REGS_EPI>();
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                         // TMEM lane quarter of this warp
        const int row = q * 32 + lane;                  // accumulator row = TMEM lane
        const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
        int buf = 0;
        uint32_t bph = 0;
        bool ok = true;
        int hc = 0;   // gate/up swapped: 32-token chunks staged so far (h stage buffer hc & 1)
        // K splits: this CTA's partial tile of split s, [BM][ACC_N] fp32
        constexpr long kTileFloats = (long)C::BM * C::ACC_N;
        auto split_part = [&](const TileInfo& tt, int s_) -> float* {
            return p.split_part + ((long)(tt.split * C::CLUSTER_N + crank) * p.split_S + s_) * kTileFloats;
        };
        for (int t = cid; t < num_tiles && ok; t += ncl) {
            const TileInfo ti = decode_tile<C>(p, t, crank);
            // first output column of the tile's accumulator (pair: the even CTA's weight rows)
            const int n0p = C::PAIR ? ti.n0 - crank * p.n_step : ti.n0;
            if constexpr (!C::FOLD) {
                if (!mbar_wait(&acc_full[buf], bph, abort_flag, p.err, DEV_TIMEOUT_ACC)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if constexpr (C::SWAP_GU) {
                    // SwiGLU over the transposed accumulator, 32 tokens at a time: lane l < 16
                    // holds gate f = 16q + l, lane l + 16 the up row of the same f; the two
                    // swap halves so that each lane forms h for 16 of the 32 tokens
                    const float s2 = p.scale2[ti.expert];
                    const int nch = (ti.rows + 31) >> 5;
                    const uint32_t acc0 = lane_addr + (uint32_t)(buf * C::MSUB * C::ACC_N);
                    const bool hi = lane >= 16;
                    const int fl = 16 * q + (lane & 15);
                    // rounding: warp q takes f block q >> 1 of tokens 16 (q & 1) .. +15, two
                    // lanes (16 f each) per token
                    const int qblk = q >> 1, qtok = (q & 1) * 16 + (lane >> 1), qhalf = lane & 1;
                    const int col = n0p + qblk * 32;
#pragma unroll 1
                    for (int c = 0; c < nch; ++c) {
                        uint32_t r[32];
                        tmem_ld32(acc0 + c * 32, r);
                        tmem_ld_wait();
                        float* hb = hstage + (hc & 1) * C::HS_FLOATS;
                        float* hw = hb + (hi ? 16 : 0) * C::HS_STRIDE + fl;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const uint32_t send = hi ? r[j] : r[16 + j];
                            const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 16);
                            const float gv = __uint_as_float(hi ? recv : r[j]) * s2;
                            const float uv = __uint_as_float(hi ? r[16 + j] : recv) * s2;
                            // silu(g) * u, the same fast intrinsics and cap as the unswapped form
                            hw[j * C::HS_STRIDE] = __fdividef(gv, 1.0f + __expf(fminf(-gv, 80.0f))) * uv;
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&hs_full[hc & 1]);
                        if (!mbar_wait(&hs_full[hc & 1], (uint32_t)((hc >> 1) & 1), abort_flag, p.err, DEV_TIMEOUT_ACC)) {
                            ok = false;
                            break;
                        }
                        const int tok = c * 32 + qtok;
                        const float* hr = hb + qtok * C::HS_STRIDE + qblk * 32 + qhalf * 16;
                        float h[16];
                        float amax = 0.f;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            h[i] = hr[i];
                            amax = fmaxf(amax, fabsf(h[i]));
                        }
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                        uint32_t packed[8];
                        int sum = 0;
                        float d = 0.f;
                        if (amax > 0.f) {
                            d = amax / 127.0f;
                            const float rd = __frcp_rn(d);
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                float v0 = roundf(h[2 * j] * rd), v1 = roundf(h[2 * j + 1] * rd);
                                v0 = fminf(fmaxf(v0, -127.f), 127.f);
                                v1 = fminf(fmaxf(v1, -127.f), 127.f);
                                sum += (int)v0 + (int)v1;
                                const __half2 hv = __floats2half2_rn(v0, v1);
                                packed[j] = *reinterpret_cast<const uint32_t*>(&hv);
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 8; ++j) packed[j] = 0;
                        }
                        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                        if (tok < ti.rows) {
                            const long grow = (long)ti.row0 + tok;
                            uint4* hq = reinterpret_cast<uint4*>(p.Hq + grow * p.F + col + qhalf * 16);
                            hq[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                            hq[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                            if (qhalf == 0) {
                                const long bidx = grow * (p.F / 32) + col / 32;
                                const __half d16 = __float2half_rn(d);
                                p.Hd[bidx] = d16;
                                p.Hs[bidx] = __float2half_rn(d * (float)sum);
                                p.Hd32[((long)(ti.entry + (tok >> 7)) * (p.F / 32) + col / 32) * 128 + (tok & 127)] =
                                    __half2float(d16);
                            }
                        }
                        ++hc;
                    }
                    if (!ok) break;
                }
#pragma unroll 1
                for (int m = 0; m < (C::SWAP_GU ? 0 : C::MSUB); ++m) {
                    if (m * 128 >= ti.rows) break;   // the MMA skipped this sub-tile: nothing to read
                    // row sub-tile m: rows m*128 + lane of this warp's quarter
                    const bool valid = m * 128 + row < ti.rows;
                    const long grow = (long)ti.row0 + m * 128 + row;
                    const uint32_t acc = lane_addr + (uint32_t)(buf * C::MSUB * C::ACC_N + m * C::ACC_N);
                    if constexpr (C::EPI == Epi::STORE) {
    #pragma unroll 1
                        for (int c = 0; c < C::ACC_N / 32; ++c) {
                            uint32_t r[32];
                            tmem_ld32(acc + c * 32, r);
                            tmem_ld_wait();
                            float v[32];
    #pragma unroll
                            for (int jj = 0; jj < 32; ++jj) v[jj] = __uint_as_float(r[jj]);
                            const int col = n0p + c * 32;
                            if (ti.split >= 0) {
                                // K split: the unscaled partial, every row and column of the tile
                                float4* dst = reinterpret_cast<float4*>(split_part(ti, ti.s) +
                                                                        (long)(m * 128 + row) * C::ACC_N + c * 32);
    #pragma unroll
                                for (int jj = 0; jj < 8; ++jj)
                                    dst[jj] = make_float4(v[4 * jj], v[4 * jj + 1], v[4 * jj + 2], v[4 * jj + 3]);
                            } else if (valid && col < p.N) {
                                store_out32(p, grow, col, v, p.scale2_dense);
                            }
                        }
                    } else {   // SWIGLU_Q81: per BN columns (one CTA's weight rows), [0, BN/2) gate, [BN/2, BN) up
                        const float s2 = p.scale2[ti.expert];
    #pragma unroll 1
                        for (int cc = 0; cc < C::ACC_N / 64; ++cc) {
                            const int hh = cc / (C::BN / 64), c = cc - hh * (C::BN / 64);
                            uint32_t g[32], u[32];
                            tmem_ld32(acc + hh * C::BN + c * 32, g);
                            tmem_ld32(acc + hh * C::BN + C::BN / 2 + c * 32, u);
                            tmem_ld_wait();
                            if (valid) {
                                float h[32];
                                float amax = 0.f;
    #pragma unroll
                                for (int j = 0; j < 32; ++j) {
                                    const float gv = __uint_as_float(g[j]) * s2;
                                    const float uv = __uint_as_float(u[j]) * s2;
                                    // silu(g) * u with the fast exponential and division
                                    // intrinsics (a few ulp: this epilogue's arithmetic
                                    // competes for issue slots with the converters and the
                                    // MMA issuer); the exponent is capped so 1 + e stays
                                    // below 2^126, where the fast division is valid
                                    h[j] = __fdividef(gv, 1.0f + __expf(fminf(-gv, 80.0f))) * uv;
                                    amax = fmaxf(amax, fabsf(h[j]));
                                }
                                // the codes are stored as exact f16 integers: the down
                                // product's MMA reads them as its operand without conversion
                                uint32_t packed[16];
                                int sum = 0;
                                float d = 0.f;
                                if (amax > 0.f) {
                                    d = amax / 127.0f;
                                    // h / d as h times the correctly rounded 1/d (within
                                    // 1.5 ulp of the quotient: a code moves only when h/d
                                    // lies that close to a half-integer)
                                    const float rd = __frcp_rn(d);
    #pragma unroll
                                    for (int j = 0; j < 16; ++j) {
                                        float v0 = roundf(h[2 * j] * rd), v1 = roundf(h[2 * j + 1] * rd);
                                        v0 = fminf(fmaxf(v0, -127.f), 127.f);
                                        v1 = fminf(fmaxf(v1, -127.f), 127.f);
                                        sum += (int)v0 + (int)v1;
                                        const __half2 hv = __floats2half2_rn(v0, v1);
                                        packed[j] = *reinterpret_cast<const uint32_t*>(&hv);
                                    }
                                } else {
    #pragma unroll
                                    for (int j = 0; j < 16; ++j) packed[j] = 0;
                                }
                                const int col = n0p + hh * (C::BN / 2) + c * 32;
                                uint4* hq = reinterpret_cast<uint4*>(p.Hq + grow * p.F + col);
    #pragma unroll
                                for (int j = 0; j < 4; ++j)
                                    hq[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
                                const long bidx = grow * (p.F / 32) + col / 32;
                                const __half d16 = __float2half_rn(d);
                                p.Hd[bidx] = d16;
                                p.Hs[bidx] = __float2half_rn(d * (float)sum);
                                // the value the down product uses, fp32, per tile entry [entry][F/32][128 rows]
                                p.Hd32[((long)(ti.entry + m) * (p.F / 32) + col / 32) * 128 + row] = __half2float(d16);
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (C::PAIR)
                        mbar_arrive_cluster(&acc_empty[buf], 0);
                    else
                        mbar_arrive(&acc_empty[buf]);
                }
                if (++buf == C::NBUF) {
                    buf = 0;
                    bph ^= 1u;
                }
            } else if constexpr (C::SWAP) {
                // FP8 fold, operands swapped: this thread's TMEM lane is weight row `row`
                // (output column n0 + row), the accumulator's 256 columns the tile's token
                // rows.  Warp cq of a lane quarter folds token columns [64 cq, 64 cq + 64),
                // skipping the 16-column chunks past the tile's live rows.
                constexpr int CPW = 64, LDW = 16;
                const int cq = (warp - C::EPI_BASE) >> 2;
                const int nld = min(CPW / LDW, max(0, (ti.rows - cq * CPW + LDW - 1) / LDW));
                const int groups = p.K / C::GROUP_K;
                float sum[CPW];
#pragma unroll
                for (int j = 0; j < CPW; ++j) sum[j] = 0.f;
                // the tile's 128 weight rows are one scale block
                const int wblk = n0p / 128;
                const bool wblk_ok = wblk < p.N / 128;
                for (int g = ti.kb0 / 2; g < ti.kb1 / 2; ++g) {
                    const float s = wblk_ok ? __ldg(p.blk_scale + (long)wblk * groups + g) : 0.f;
                    if (!mbar_wait(&acc_full[buf], bph, abort_flag, p.err, DEV_TIMEOUT_ACC)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t acc = lane_addr + (uint32_t)(buf * C::MSUB * C::ACC_N + cq * CPW);
#pragma unroll
                    for (int c = 0; c < CPW / LDW; ++c) {
                        if (c < nld) {
                            uint32_t r[LDW];
                            tmem_ld16(acc + c * LDW, r);
                            tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < LDW; ++j) sum[c * LDW + j] = fmaf(s, __uint_as_float(r[j]), sum[c * LDW + j]);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_empty[buf]);
                    if (++buf == C::NBUF) {
                        buf = 0;
                        bph ^= 1u;
                    }
                }
                if (!ok) break;
                if (ti.split >= 0) {
                    // K split: the partial tile in the same [token row][weight row] layout
                    // as the unswapped form (lanes write 32 consecutive columns)
                    float* dst = split_part(ti, ti.s) + (long)(cq * CPW) * C::ACC_N + row;
#pragma unroll
                    for (int j = 0; j < CPW; ++j) dst[(long)j * C::ACC_N] = sum[j];
                    continue;
                }
                const int col = n0p + row;
                const int nrow = min(CPW, ti.rows - cq * CPW);
                if (col < p.N && nrow > 0) {
                    // Y[token][col]: the 32 lanes store 32 consecutive columns of one row
                    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.Y) + (long)(ti.row0 + cq * CPW) * p.ldy + col;
#pragma unroll
                    for (int j = 0; j < CPW; ++j)
                        if (j < nrow) dst[(long)j * p.ldy] = __float2bfloat16_rn(sum[j]);
                }
            } else {
                // FP8 fold: one accumulator per 128-K block and row sub-tile, folded into
                // registers with its scale; FOLD_CPW token columns per warp
                constexpr int CPW = C::FOLD_CPW, LDW = C::FOLD_LDW;
                const int cq = (warp - C::EPI_BASE) >> 2;      // this warp's block of CPW columns
                const int nsub = min(C::MSUB, (ti.rows + 127) / 128);
                const int groups = p.K / C::GROUP_K;
                float sum[C::MSUB][CPW];
#pragma unroll
                for (int m = 0; m < C::MSUB; ++m)
#pragma unroll
                    for (int j = 0; j < CPW; ++j) sum[m][j] = 0.f;
                // this warp's columns lie in one 128-wide weight block (pair: either CTA's)
                const int wblk = (n0p + cq * CPW) / 128;
                const bool wblk_ok = wblk < p.N / 128;
                for (int g = ti.kb0 / 2; g < ti.kb1 / 2; ++g) {
                    const float s = wblk_ok ? __ldg(p.blk_scale + (long)wblk * groups + g) : 0.f;
                    if (!mbar_wait(&acc_full[buf], bph, abort_flag, p.err, DEV_TIMEOUT_ACC)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int m = 0; m < C::MSUB; ++m) {
                        if (m < nsub) {
                            const uint32_t acc = lane_addr + (uint32_t)(buf * C::MSUB * C::ACC_N + m * C::ACC_N + cq * CPW);
#pragma unroll
                            for (int c = 0; c < CPW / LDW; ++c) {
                                uint32_t r[LDW];
                                if constexpr (LDW == 32) tmem_ld32(acc + c * LDW, r);
                                else tmem_ld16(acc + c * LDW, r);
                                tmem_ld_wait();
#pragma unroll
                                for (int j = 0; j < LDW; ++j)
                                    sum[m][c * LDW + j] = fmaf(s, __uint_as_float(r[j]), sum[m][c * LDW + j]);
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (C::PAIR)
                            mbar_arrive_cluster(&acc_empty[buf], 0);
                        else
                            mbar_arrive(&acc_empty[buf]);
                    }
                    if (++buf == C::NBUF) {
                        buf = 0;
                        bph ^= 1u;
                    }
                }
                if (!ok) break;
                if (ti.split >= 0) {
                    // K split: this split's folded sums, every row of the live sub-tiles;
                    // the split-reduce kernel adds the splits and writes the output
#pragma unroll
                    for (int m = 0; m < C::MSUB; ++m) {
                        if (m < nsub) {
                            float4* dst = reinterpret_cast<float4*>(split_part(ti, ti.s) +
                                                                    (long)(m * 128 + row) * C::ACC_N + cq * CPW);
#pragma unroll
                            for (int j = 0; j < CPW / 4; ++j)
                                dst[j] = make_float4(sum[m][4 * j], sum[m][4 * j + 1], sum[m][4 * j + 2], sum[m][4 * j + 3]);
                        }
                    }
                    continue;
                }
#pragma unroll
                for (int m = 0; m < C::MSUB; ++m) {
                    if (m < nsub && m * 128 + row < ti.rows) {
                        const long grow = (long)ti.row0 + m * 128 + row;
                        const int col = n0p + cq * CPW;
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.Y) + grow * p.ldy + col);
#pragma unroll
                        for (int j = 0; j < CPW / 8; ++j) {
                            uint32_t w[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                __nv_bfloat162 b = __floats2bfloat162_rn(sum[m][8 * j + 2 * i], sum[m][8 * j + 2 * i + 1]);
                                w[i] = *reinterpret_cast<uint32_t*>(&b);
                            }
                            dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            }
        }
    } else {
        if constexpr (C::REG_SPLIT) setmaxnreg_dec<C::REGS_OTHER>();
        if (warp == 0) {
            // ------------------------------------------------------------ producer
            {
                int s = 0;
                uint32_t ph = 0;
                long issued = 0;
                bool ok = true;
                TileInfo ti_next{};
                if (cid < num_tiles) ti_next = decode_tile<C>(p, cid, crank);
                for (int t = cid; t < num_tiles && ok; t += ncl) {
                    const TileInfo ti = ti_next;                 // read one tile ahead
                    if (t + ncl < num_tiles) ti_next = decode_tile<C>(p, t + ncl, crank);
                    // the weight codes' tensor map: the expert's own (pointer-table form), or
                    // the kernel parameter over the contiguous [E][...] array
                    const CUtensorMap* bmap = p.wmaps ? p.wmaps + ti.expert : &tmB;
                    if (p.wmaps) tensormap_acquire(bmap);
                    for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
                        const bool got = mbar_wait(&empty_t[s], ph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_TMA_EMPTY);
                        if (__any_sync(0xffffffffu, !got)) {
                            ok = false;
                            break;
                        }
                        // A thread has one TMA copy executing at a time, so each copy of stage s
                        // comes from its own lane of lane group s % TMA_GROUPS: copies of
                        // different stages and kinds overlap.
                        const int l0 = (s % C::TMA_GROUPS) * 4;
                        uint8_t* st = tstage + s * C::TSTAGE_BYTES;
                        // A tile of at most 128 live rows reads only the first 128-row slice of
                        // the activation tile: the CTA that would load the second slice skips
                        // it, and every CTA of the cluster expects that many bytes less.
                        constexpr bool kHalfA = QMM_HALF_A && !C::PAIR && C::CLUSTER_N == 2 && C::MSUB == 2;
                        const bool half_a = kHalfA && ti.rows <= 128;
                        if (lane == l0)
                            mbar_arrive_expect_tx(&full_t[s], C::TSTAGE_BYTES - (half_a ? C::A_SLICE_ROWS * 128 : 0));
                        __syncwarp();
                        if (lane == l0) {
                            if constexpr (C::PAIR) {
                                // this CTA's 128 rows of the pair's 256-row tile
                                tma_load_2d(st, &tmA, &full_t[s], kb * C::BK, ti.row0);
                            } else if constexpr (C::CLUSTER_N > 1) {
                                // this CTA's slice of the activation tile, written into every CTA of the cluster
                                if (!(half_a && crank == 1))
                                    tma_load_2d_multicast(st + crank * C::A_SLICE_ROWS * 128, &tmA, &full_t[s], kb * C::BK,
                                                      ti.row0 + crank * C::A_SLICE_ROWS,
                                                      (uint16_t)((1u << C::CLUSTER_N) - 1));
                            } else {
                                tma_load_2d(st, &tmA, &full_t[s], kb * C::BK, ti.row0);
                            }
                        } else if (lane == l0 + 1 || lane == l0 + 2) {
                            uint8_t* bdst = st + C::A_RAW_BYTES;
                            const int kx = kb * C::B_ROW_BYTES;
                            if constexpr (C::EPI == Epi::SWIGLU_Q81) {
                                // gate rows n0 .. +BN/2 (lane l0+1), up rows F + n0 .. +BN/2 (lane l0+2) of
                                // the expert's [2F] rows (row e*2F + ... of the contiguous array)
                                const int base = (p.wmaps ? 0 : ti.expert * 2 * p.F) + ti.n0;
                                if (lane == l0 + 1)
                                    tma_load_2d(bdst, bmap, &full_t[s], kx, base);
                                else
                                    tma_load_2d(bdst + (C::BN / 2) * C::B_ROW_BYTES, bmap, &full_t[s], kx, base + p.F);
                            } else if (lane == l0 + 1) {
                                tma_load_2d(bdst, bmap, &full_t[s], kx, (p.wmaps ? 0 : ti.expert * p.N) + ti.n0);
                            }
                        }
                        __syncwarp();
                        ++issued;
                        if (++s == C::TSTAGES) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                }
                // Teardown: every copy issued must have landed before the CTA exits.
                if (lane == 0) drain_ring(full_t, issued, C::TSTAGES, p.err);
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------ MMA issuer (one lane)
            // One thread runs the whole issue loop: the descriptors of a K block are
            // built once and advanced by constants, and there is no election or warp
            // synchronisation between MMAs.  Pair: the even CTA issues for both.
            if (lane == 0 && pair_leader) {
                int ts = 0, cs = 0, buf = 0;
                uint32_t cph = 0, bph = 0;
                bool ok = true;
                // the work item, read one ahead so the descriptor load is off the issue
                // path: its K range, and the sub-tiles holding at least one live row (a
                // tile of <= 128 rows skips the second)
                TileInfo mi_next{};
                if (cid < num_tiles) mi_next = decode_tile<C>(p, cid, crank);
                for (int t = cid; t < num_tiles && ok; t += ncl) {
                    const TileInfo mi = mi_next;
                    if (t + ncl < num_tiles) mi_next = decode_tile<C>(p, t + ncl, crank);
                    const int nsub = (C::MSUB == 2 && mi.rows <= 128) ? 1 : C::MSUB;
                    const uint32_t idesc_swap = idesc_kind_f16(128, min(256, max(16, (mi.rows + 15) & ~15)), true);
                    for (int kb = mi.kb0; kb < mi.kb1; ++kb) {
                        // Only the converted weights are waited on: the converters arrive on
                        // full_c after they saw this stage's TMA copies complete (full_t), so
                        // full_c also orders the activation tile.
                        // (pair: both CTAs' converters arrive here, after their own TMA stage)
                        const bool got_c = C::PAIR ? mbar_wait_cl(&full_c[cs], cph, abort_flag, p.err, DEV_TIMEOUT_CONV)
                                                   : mbar_wait(&full_c[cs], cph, abort_flag, p.err, DEV_TIMEOUT_CONV);
                        if (!got_c) {
                            ok = false;
                            break;
                        }
                        // first / last K block of an accumulation group (the item's K range, or
                        // one 128-K block = two K blocks for the FP8 fold)
                        bool first, last;
                        if constexpr (C::GROUP_K == 128) {
                            first = (kb & 1) == 0;
                            last = (kb & 1) == 1;
                        } else {
                            first = kb == mi.kb0;
                            last = kb == mi.kb1 - 1;
                        }
                        if (first) {
                            const bool got_a =
                                C::PAIR ? mbar_wait_cl(&acc_empty[buf], bph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_ACC_EMPTY)
                                        : mbar_wait(&acc_empty[buf], bph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_ACC_EMPTY);
                            if (!got_a) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        // (no tcgen05 fence per K block: the operands are ordered by the mbarrier
                        // and the writers' proxy fence; such a fence would drain the MMA pipe)
                        // descriptor start addresses are in 16-byte units: +2 per K step of 16
                        // (32 bytes), +1024 per 128-row sub-tile (16 KB)
                        const uint64_t ad = smem_desc_sw128(smem_u32(tstage + ts * C::TSTAGE_BYTES));
                        const uint64_t bd = smem_desc_sw128(smem_u32(cstage + cs * C::CSTAGE_BYTES));
                        const uint32_t dtmem = tmem_base + (uint32_t)(buf * C::MSUB * C::ACC_N);
                        if constexpr (C::PAIR) {
                            // M = 256 over the pair, N = 2 * BN: both CTAs' stages at the same offsets
#pragma unroll
                            for (int kk = 0; kk < C::BK / C::UMMA_K; ++kk)
                                tc_mma_f16_pair(dtmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), C::IDESC,
                                                (first && kk == 0) ? 0u : 1u);
                            if (last) {
                                tc_commit_pair(&acc_full[buf], 3);
                                if (++buf == C::NBUF) {
                                    buf = 0;
                                    bph ^= 1u;
                                }
                            }
                            tc_commit_pair(&empty_c[cs], 3);
                            tc_commit_pair(&empty_t[ts], 3);
                        } else {
                            if constexpr (C::SWAP) {
                                // A: the converted weights (128 rows); B: the activation tile, N = its
                                // live rows rounded up to 16
#pragma unroll
                                for (int kk = 0; kk < C::BK / C::UMMA_K; ++kk)
                                    tc_mma_f16(dtmem, bd + (uint64_t)(kk * 2), ad + (uint64_t)(kk * 2), idesc_swap,
                                               (first && kk == 0) ? 0u : 1u);
                            } else {
#pragma unroll
                                for (int kk = 0; kk < C::BK / C::UMMA_K; ++kk) {
#pragma unroll
                                    for (int m = 0; m < C::MSUB; ++m)
                                        if (m < nsub)
                                            tc_mma_f16(dtmem + (uint32_t)(m * C::BN), ad + (uint64_t)(m * 1024 + kk * 2),
                                                       bd + (uint64_t)(kk * 2), C::IDESC, (first && kk == 0) ? 0u : 1u);
                                }
                            }
                            if (last) {
                                tc_commit(&acc_full[buf]);
                                if (++buf == C::NBUF) {
                                    buf = 0;
                                    bph ^= 1u;
                                }
                            }
                            tc_commit(&empty_c[cs]);
                            if constexpr (C::CLUSTER_N > 1)
                                tc_commit_multicast(&empty_t[ts], (uint16_t)((1u << C::CLUSTER_N) - 1));
                            else
                                tc_commit(&empty_t[ts]);
                        }
                        if (++ts == C::TSTAGES) ts = 0;
                        if (++cs == C::CSTAGES) {
                            cs = 0;
                            cph ^= 1u;
                        }
                    }
                }
                // Teardown: wait until every MMA issued has completed before TMEM is freed.
                if constexpr (C::PAIR)
                    tc_commit_pair(drain_bar, 1);
                else
                    tc_commit(drain_bar);
                drain_ring(drain_bar, 1, 1, p.err);
            }
            if constexpr (C::PAIR) {
                if (lane == 0 && !pair_leader) relay_stages(0);
            }
            __syncwarp();
        } else if (C::conv_slot(warp) >= 0) {
            // ------------------------------------------------------------ converters
            const int ct = C::conv_slot(warp) * 32 + lane;
            const int crow = ct % C::BN;                      // this thread's weight row in every tile
            const int chalf = ct / C::BN;                     // and its K half (TPR == 2) or quarter (4)
            const int cdrow = C::conv_dst_row(crow);          // its row in the operand tile
            int ts = 0, cs = 0;
            uint32_t tph = 0, cph = 0;
            bool ok = true;
            // W4 scales: 16-byte loads covering 4 K blocks, one chunk ahead (K % 256 == 0),
            // else one 4-byte load per K block.
            const bool vec_scales = (p.K % 256) == 0;
            // this thread's weight row of a tile: its E4M3 scale row (K/16 bytes)
            auto scale_row = [&](const TileInfo& tt, bool& in_range) -> const uint8_t* {
                if constexpr (C::EPI == Epi::SWIGLU_Q81) {
                    const int hr = (crow < C::BN / 2) ? (tt.n0 + crow) : (p.F + tt.n0 + crow - C::BN / 2);
                    in_range = true;
                    if (p.wscale_tab) return p.wscale_tab[tt.expert] + (long)hr * (p.K / 16);
                    return p.w_scale + ((long)tt.expert * 2 * p.F + hr) * (p.K / 16);
                } else {
                    in_range = (long)tt.n0 + crow < p.N;
                    return p.w_scale + ((long)tt.n0 + crow) * (p.K / 16);
                }
            };
            // Scale prefetch two 4-K-block chunks ahead, through a cursor that walks
            // this CTA's work items (and each item's K range) in the order they are
            // converted: the next item's descriptor is read one chunk before its first
            // scales are needed, so neither global load (descriptor, then scales) sits
            // on the critical path.
            int pf_t = cid, pf_ch = 0;
            TileInfo pf_ti{};
            if (pf_t < num_tiles) {
                pf_ti = decode_tile<C>(p, pf_t, crank);
                pf_ch = pf_ti.kb0 / 4;
            }
            auto next_chunk = [&]() -> uint4 {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (pf_t < num_tiles) {
                    bool in_range;
                    const uint8_t* srow = scale_row(pf_ti, in_range);
                    if (in_range) v = ldg_nc_v4(srow + pf_ch * 16);
                    if (++pf_ch == pf_ti.kb1 / 4) {
                        pf_t += ncl;
                        if (pf_t < num_tiles) {
                            pf_ti = decode_tile<C>(p, pf_t, crank);
                            pf_ch = pf_ti.kb0 / 4;
                        }
                    }
                }
                return v;
            };
            uint4 sc_cur = make_uint4(0, 0, 0, 0), sc_next = make_uint4(0, 0, 0, 0), sc_next2 = make_uint4(0, 0, 0, 0);
            if constexpr (C::B == BMode::W4) {
                if (vec_scales) {
                    sc_next = next_chunk();
                    sc_next2 = next_chunk();
                }
            }
            // Converted stages are handed to the MMA CONV_BATCH at a time: one proxy
            // fence (and, for a pair, one cluster-scope release) per batch.  Each costs
            // a few hundred cycles of the converter's own time, which would otherwise
            // be paid per K block on the pipeline's critical path.
            int pend = 0, pend_first = 0;
            auto flush = [&]() {
                if (pend == 0) return;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    for (int i = 0, c = pend_first; i < pend; ++i, c = (c + 1 == C::CSTAGES) ? 0 : c + 1) {
                        // (pair, odd CTA: to the relay thread, which forwards the stage to the
                        // even CTA's barrier with a cluster-scope release; a converter's own
                        // cluster-scope release would wait for its scale loads in flight)
                        if (C::PAIR && crank != 0)
                            mbar_arrive(&conv_done[c]);
                        else
                            mbar_arrive(&full_c[c]);
                    }
                }
                pend = 0;
            };
            // one K block: wait for its raw codes and a free converted stage, expand,
            // hand the stage to the MMA (with its batch); false if a wait timed out
            auto convert_step = [&](uint32_t sbytes) -> bool {
                if (!mbar_wait(&full_t[ts], tph, abort_flag, p.err, DEV_TIMEOUT_TMA_FULL) ||
                    !mbar_wait(&empty_c[cs], cph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_CONV_EMPTY))
                    return false;
                const uint32_t braw = smem_u32(tstage + ts * C::TSTAGE_BYTES) + C::A_RAW_BYTES;
                const uint32_t bconv = smem_u32(cstage + cs * C::CSTAGE_BYTES);
                if constexpr (C::B == BMode::W4) {
                    if constexpr (C::TPR == 4)
                        convert_w4_quarter(braw, bconv, crow, cdrow, chalf, sbytes);
                    else if constexpr (C::TPR == 2)
                        convert_w4_half(braw, bconv, crow, cdrow, chalf, sbytes);
                    else
                        convert_w4_row(braw, bconv, crow, cdrow, sbytes);
                } else if constexpr (C::TPR == 2) {
                    convert_fp8_half(braw, bconv, crow, chalf);
                } else {
                    convert_fp8_rows<C::RPT>(braw, bconv, crow, C::BN / C::RPT);
                }
                if (pend++ == 0) pend_first = cs;
                if (pend == C::CONV_BATCH) flush();
                if (++ts == C::TSTAGES) {
                    ts = 0;
                    tph ^= 1u;
                }
                if (++cs == C::CSTAGES) {
                    cs = 0;
                    cph ^= 1u;
                }
                return true;
            };
            for (int t = cid; t < num_tiles && ok; t += ncl) {
                const TileInfo ti = decode_tile<C>(p, t, crank);
                if (C::B == BMode::W4 && vec_scales) {
                    // K % 256 == 0: the item's K range is whole 4-K-block chunks; the chunk's
                    // four scale words are picked at compile time in the unrolled steps
                    for (int ch = ti.kb0 >> 2; ch < (ti.kb1 >> 2) && ok; ++ch) {
                        if constexpr (C::B == BMode::W4) {
                            sc_cur = sc_next;
                            sc_next = sc_next2;
                            sc_next2 = next_chunk();
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t sbytes = (C::B == BMode::W4)
                                                        ? (j == 0 ? sc_cur.x : (j == 1 ? sc_cur.y : (j == 2 ? sc_cur.z : sc_cur.w)))
                                                        : 0u;
                            if (!convert_step(sbytes)) {
                                ok = false;
                                break;
                            }
                        }
                    }
                } else {
                    for (int kb = ti.kb0; kb < ti.kb1 && ok; ++kb) {
                        uint32_t sbytes = 0;
                        if constexpr (C::B == BMode::W4) {
                            bool in_range;
                            const uint8_t* srow = scale_row(ti, in_range);
                            if (!in_range) {
                                sbytes = 0u;
                            } else if ((p.K & 63) == 0) {
                                sbytes = __ldg(reinterpret_cast<const uint32_t*>(srow + kb * 4));
                            } else {
                                // K % 64 == 32: scale rows are not 4-byte aligned, and the last K
                                // block has two scale bytes (its other 32 K are zero-filled codes,
                                // given scale 0 so that no NaN scale byte of the next row enters)
                                const int nsc = p.K / 16;
                                sbytes = 0u;
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    if (kb * 4 + i < nsc) sbytes |= (uint32_t)__ldg(srow + kb * 4 + i) << (8 * i);
                            }
                        }
                        if (!convert_step(sbytes)) ok = false;
                    }
                }
            }
            flush();
        } else if (C::PAIR && C::RELAYS > 1 && C::relay_slot(warp) > 0) {
            if (lane == 0 && !pair_leader) relay_stages(C::relay_slot(warp));
            }
    }

    __syncthreads();
    // No CTA leaves while a peer may still multicast into its shared memory or
    // signal its barriers.
    if constexpr (C::CLUSTER_N > 1) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (C::PAIR)
            tmem_dealloc_pair(tmem_base, 512);
        else
            tmem_dealloc(tmem_base, 512);
    }
}

// ---------------------------------------------------------------------------
// Host-side launch of a GemmCfg instantiation: cluster launch when CLUSTER_N > 1,
// persistent grid of (max co-resident clusters, capped by the work) x CLUSTER_N.
template <class C>
cudaError_t launch_qgemm(const CUtensorMap& tmA, const CUtensorMap& tmB, GemmParams p, int max_items,
                         cudaStream_t s) {
    static_assert(C::SMEM_BYTES <= 232448, "shared memory");
    cudaError_t e = cudaFuncSetAttribute(qgemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if constexpr (C::REG_SPLIT) {
        // the warpgroups' register shares add up to the launch's: launch only if the
        // kernel is allocated exactly that many (more shares than the pool would
        // leave a setmaxnreg.inc waiting)
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, qgemm_kernel<C>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != C::REGS_LAUNCH) return cudaErrorInvalidConfiguration;
    }
    if (C::CLUSTER_N > 1) {
        e = cudaFuncSetAttribute(qgemm_kernel<C>, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
        if (e != cudaSuccess) return e;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    static int max_clusters[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C::CLUSTER_N;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (max_clusters[dev] == 0) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        int n = sms / C::CLUSTER_N;
        if (C::CLUSTER_N > 1) {
            cfg.gridDim = dim3(C::CLUSTER_N * n, 1, 1);
            int q = 0;
            if (cudaOccupancyMaxActiveClusters(&q, qgemm_kernel<C>, &cfg) == cudaSuccess && q > 0) n = q;
        }
        max_clusters[dev] = n;
    }
    int clusters = max_clusters[dev];
    p.split_S = 1;
    if constexpr (!C::GROUPED) {
        // Dense: when the last wave of tiles fills at most half the clusters, split
        // each of its tiles into S K ranges (whole 4-K-block chunks, at least two
        // per split) so that S x as many clusters share it.
        const int items = p.m_tiles * (p.n_tiles / C::CLUSTER_N);
        const int kblocks = p.K / C::BK;
        const int full = items / clusters * clusters, rem = items - full;
        p.split_from = items;
        if (p.split_part && p.K % 256 == 0 && rem > 0 && 2 * rem <= clusters) {
            int S = clusters / rem;
            if (S > 8) S = 8;
            if (S > kblocks / 8) S = kblocks / 8;
            if (S >= 2 && (long)rem * C::CLUSTER_N * S * C::BM * C::ACC_N <= p.split_part_cap) {
                p.split_from = full;
                p.split_S = S;
            }
        }
        max_items = p.split_from + (items - p.split_from) * p.split_S;
    }
    if (max_items > 0 && max_items < clusters) clusters = max_items;
    cfg.gridDim = dim3(C::CLUSTER_N * clusters, 1, 1);
    e = cudaLaunchKernelEx(&cfg, qgemm_kernel<C>, tmA, tmB, p);
    if (e != cudaSuccess) return e;
    if (p.split_S > 1) {
        const int rem = (p.m_tiles * (p.n_tiles / C::CLUSTER_N)) - p.split_from;
        const long threads = (long)rem * C::CLUSTER_N * C::BM * (C::ACC_N / 4);
        const float scale = (C::EPI == Epi::STORE) ? p.scale2_dense : 1.0f;
        split_reduce_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(p, C::BM, C::ACC_N, C::CLUSTER_N, rem, scale,
                                                                             C::PAIR);
    }
    return cudaGetLastError();
}

}  // namespace qmm
