// FP8 (E4M3) weight GEMM with one fp32 scale per 128x128 block: each 128-K block
// is accumulated unscaled in its own TMEM buffer and folded once with its scale.
// Kernel body: qgemm.cuh.
#include "qgemm.cuh"

namespace qmm {

// Two 128-row sub-tiles (256 token rows) share each expanded weight tile, which
// halves the E4M3 -> bf16 conversion per FLOP.  The fold takes 16 epilogue warps
// (64 running sums a thread); 8 converter warps expand the weight tile, two
// threads per weight row (one K half each), and the two sets share the SM's
// registers through a warpgroup register split (fold 96, the rest 40, launched at
// 28 x 72).  Measured at M=2048, K=5120, N=5120: 0.111 ms with 8 converters, 0.120
// with 4 (one thread per row).
#ifndef QMM_FP8_CONV
#define QMM_FP8_CONV 8
#endif
// Operands swapped (weights as the MMA's A, M = 128; the 256 token rows as its B,
// N = 256): one N = 256 MMA per K step of 16.
#ifndef QMM_FP8_SWAP
#define QMM_FP8_SWAP 1
#endif
template <int CN>
using CfgFp8 = GemmCfg<BMode::FP8, Epi::FOLD_FP8, 128, QMM_FP8_CONV, 16, 4, 4, false, CN, 2, false, QMM_FP8_SWAP != 0>;
// CTA pair: 256 x 256 tiles, each CTA 128 token rows and 128 weight rows (one
// 128 x 128 scale block), the fold over its 128 rows x both CTAs' columns.
using CfgFp8Pair = GemmCfg<BMode::FP8, Epi::FOLD_FP8, 128, QMM_FP8_CONV, 16, 5, 4, false, 2, 1, true>;
static_assert(CfgFp8<1>::TILE_M == CfgFp8Pair::TILE_M, "one routing of rows for both forms");

int fp8_tile_rows() { return CfgFp8<1>::TILE_M; }

cudaError_t launch_fp8_blk128(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int cn,
                              cudaStream_t s) {
    const int items = p.m_tiles * (p.n_tiles / cn);
    if (QMM_PAIR && cn == 2) return launch_qgemm<CfgFp8Pair>(tmA, tmB, p, items, s);
    switch (cn) {
        case 4: return launch_qgemm<CfgFp8<4>>(tmA, tmB, p, items, s);
        case 2: return launch_qgemm<CfgFp8<2>>(tmA, tmB, p, items, s);
        default: return launch_qgemm<CfgFp8<1>>(tmA, tmB, p, items, s);
    }
}

}  // namespace qmm
