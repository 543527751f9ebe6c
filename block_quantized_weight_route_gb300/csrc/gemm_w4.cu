// W4 (e2m1 codes, E4M3 per-16 scales, fp32 scale2) GEMMs: the dense prefill
// projection and the routed-MoE gate/up product with its fused SwiGLU + q8_1
// epilogue.  Kernel body: qgemm.cuh.
#include "qgemm.cuh"

namespace qmm {

#ifndef QMM_GU_TSTAGES
#define QMM_GU_TSTAGES 4
#endif
#ifndef QMM_GU_CSTAGES
#define QMM_GU_CSTAGES 3
#endif

// Dense: 256 token rows per tile (two 128-row sub-tiles share each converted
// weight tile), 4 epilogue warps.  Wide: 256 weight rows per tile, which halves
// the conversion per FLOP again; the two 128 x 256 accumulators fill TMEM, so the
// epilogue of one tile is not overlapped with the next tile's MMAs; 16 converter
// warps, two threads per weight row (28 warps under a 120 / 64 register split:
// 0.267 ms at M=2048, K=5120, N=17408 against 0.279 with 8, one thread per row).
// Narrow: 128 weight rows, 8 converter warps, double-buffered accumulators, twice
// the tiles (for problems too small to fill the SMs with wide tiles).
#ifndef QMM_W4W_CONV
#define QMM_W4W_CONV 16
#endif
template <int CN>
using CfgW4DenseWide = GemmCfg<BMode::W4, Epi::STORE, 256, QMM_W4W_CONV, 4, 3, 2, false, CN, 2>;
template <int CN>
using CfgW4Dense = GemmCfg<BMode::W4, Epi::STORE, 128, 8, 4, 4, 3, false, CN, 2>;
// Gate/up: 256 token rows x (64 gate + 64 up) weight rows per tile.
// Operands swapped: the converted 128 weight rows as the MMA's A (M = 128), the
// 256 token rows as its B (N = 256, or a short tile's live rows rounded up to 16).
#ifndef QMM_GU_SWAP
#define QMM_GU_SWAP 1
#endif
// 16 converter warps, four threads per weight row (a quarter row each; 28 warps
// under a 120 / 64 register split): 0.3486 against 0.3499 ms with 8 at T=5268.
#ifndef QMM_GU_CONV
#define QMM_GU_CONV 16
#endif
template <int CN>
using CfgW4GateUp = GemmCfg<BMode::W4, Epi::SWIGLU_Q81, 128, QMM_GU_CONV, 4, QMM_GU_TSTAGES, QMM_GU_CSTAGES, true, CN, 2,
                            false, QMM_GU_SWAP != 0>;
// CTA-pair forms (clusters of 2): 256 token rows x 256 weight rows per pair,
// each CTA 128 token rows and 128 weight rows (gate/up: 64 gate + 64 up).
#ifndef QMM_PAIR_TSTAGES
#define QMM_PAIR_TSTAGES 6
#endif
#ifndef QMM_PAIR_CSTAGES
#define QMM_PAIR_CSTAGES 4
#endif
using CfgW4DensePair = GemmCfg<BMode::W4, Epi::STORE, 128, 8, 4, QMM_PAIR_TSTAGES, QMM_PAIR_CSTAGES, false, 2, 1, true>;
using CfgW4GateUpPair = GemmCfg<BMode::W4, Epi::SWIGLU_Q81, 128, 8, 4, QMM_PAIR_TSTAGES, QMM_PAIR_CSTAGES, true, 2, 1, true>;
static_assert(CfgW4GateUp<1>::TILE_M == CfgW4GateUpPair::TILE_M, "one routing of rows for both forms");

// Wide tiles do a tile's work in about 1.75x the time of a narrow one (measured:
// 0.305 against 0.349 ms at M=2048, K=5120, N=17408), so they win unless their
// coarser waves leave more SMs idle.
TileShape w4_dense_shape(int M, int N, int sms) {
    // CTA pairs: narrow per-CTA tiles (the pair's tile is 256 x 256)
    if (QMM_PAIR && ((N + 127) / 128) % 2 == 0) return TileShape{256, 128};
    const long wide = (long)((M + 255) / 256) * ((N + 255) / 256);
    const long narrow = (long)((M + 255) / 256) * ((N + 127) / 128);
    const long wide_waves = (wide + sms - 1) / sms, narrow_waves = (narrow + sms - 1) / sms;
    return (wide_waves * 7 < narrow_waves * 4) ? TileShape{256, 256} : TileShape{256, 128};
}
TileShape w4_gate_up_shape() { return TileShape{CfgW4GateUp<1>::BM, CfgW4GateUp<1>::BN}; }

// Largest cluster (CTAs sharing one activation tile by multicast) a launch may use.
// Measured on the 5268-token stage: gate/up 0.39 ms with pairs against 0.43 ms with
// clusters of 4 (each stage is released only when every CTA of the cluster has read
// it, so larger clusters wait on their slowest member); the dense GEMMs 2-5% faster.
#ifndef QMM_MAX_CLUSTER
#define QMM_MAX_CLUSTER 2
#endif
int cluster_for(int n_tiles) {
    if (QMM_MAX_CLUSTER >= 4 && n_tiles % 4 == 0) return 4;
    if (QMM_MAX_CLUSTER >= 2 && n_tiles % 2 == 0) return 2;
    return 1;
}
// Gate/up: no clusters.  A multicast activation stage is refilled only once the
// MMAs of both CTAs have read it, which couples the two CTAs' pipelines; each CTA
// loading its own activation tiles was faster (5268-token stage: 0.349 against
// 0.355 ms; 21504 tokens: 1.67 against 1.71 ms).
#ifndef QMM_GU_MAX_CLUSTER
#define QMM_GU_MAX_CLUSTER 1
#endif
int gate_up_cluster(int n_tiles) {
    if (QMM_PAIR) return cluster_for(n_tiles);   // the CTA-pair build: pairs wherever they fit
    if (QMM_GU_MAX_CLUSTER >= 4 && n_tiles % 4 == 0) return 4;
    if (QMM_GU_MAX_CLUSTER >= 2 && n_tiles % 2 == 0) return 2;
    return 1;
}

cudaError_t launch_w4a16_dense(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int cn,
                               cudaStream_t s) {
    const int items = p.m_tiles * (p.n_tiles / cn);
    if (p.n_step == 256) {
        switch (cn) {
            case 4: return launch_qgemm<CfgW4DenseWide<4>>(tmA, tmB, p, items, s);
            case 2: return launch_qgemm<CfgW4DenseWide<2>>(tmA, tmB, p, items, s);
            default: return launch_qgemm<CfgW4DenseWide<1>>(tmA, tmB, p, items, s);
        }
    }
    if (QMM_PAIR && cn == 2) return launch_qgemm<CfgW4DensePair>(tmA, tmB, p, items, s);
    switch (cn) {
        case 4: return launch_qgemm<CfgW4Dense<4>>(tmA, tmB, p, items, s);
        case 2: return launch_qgemm<CfgW4Dense<2>>(tmA, tmB, p, items, s);
        default: return launch_qgemm<CfgW4Dense<1>>(tmA, tmB, p, items, s);
    }
}

cudaError_t launch_w4_gate_up_swiglu(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int cn,
                                     cudaStream_t s) {
    if (QMM_PAIR && cn == 2) return launch_qgemm<CfgW4GateUpPair>(tmA, tmB, p, 0, s);
    switch (cn) {
        case 4: return launch_qgemm<CfgW4GateUp<4>>(tmA, tmB, p, 0, s);
        case 2: return launch_qgemm<CfgW4GateUp<2>>(tmA, tmB, p, 0, s);
        default: return launch_qgemm<CfgW4GateUp<1>>(tmA, tmB, p, 0, s);
    }
}

}  // namespace qmm
