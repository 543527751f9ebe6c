// W4 (e2m1 codes, E4M3 per-16 scales, fp32 scale2) GEMMs: the dense prefill
// projection and the routed-MoE gate/up product with its fused SwiGLU + q8_1
// epilogue.  Kernel body: qgemm.cuh.
#include "qgemm.cuh"

namespace qmm {

// Dense: 256 x 128 tiles (two 128-row sub-tiles share each converted weight
// tile), 8 converter warps (two per weight row), 4 epilogue warps.
template <int CN>
using CfgW4Dense = GemmCfg<BMode::W4, Epi::STORE, 128, 8, 4, 4, 3, false, CN, 2>;
// Gate/up: 256 token rows x (64 gate + 64 up) weight rows per tile.
template <int CN>
#ifndef QMM_GU_TSTAGES
#define QMM_GU_TSTAGES 4
#endif
#ifndef QMM_GU_CSTAGES
#define QMM_GU_CSTAGES 3
#endif
using CfgW4GateUp = GemmCfg<BMode::W4, Epi::SWIGLU_Q81, 128, 8, 4, QMM_GU_TSTAGES, QMM_GU_CSTAGES, true, CN, 2>;

int cluster_for(int n_tiles) { return (n_tiles % 4 == 0) ? 4 : ((n_tiles % 2 == 0) ? 2 : 1); }

cudaError_t launch_w4a16_dense(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int cn,
                               cudaStream_t s) {
    const int items = p.m_tiles * (p.n_tiles / cn);
    switch (cn) {
        case 4: return launch_qgemm<CfgW4Dense<4>>(tmA, tmB, p, items, s);
        case 2: return launch_qgemm<CfgW4Dense<2>>(tmA, tmB, p, items, s);
        default: return launch_qgemm<CfgW4Dense<1>>(tmA, tmB, p, items, s);
    }
}

cudaError_t launch_w4_gate_up_swiglu(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int cn,
                                     cudaStream_t s) {
    switch (cn) {
        case 4: return launch_qgemm<CfgW4GateUp<4>>(tmA, tmB, p, 0, s);
        case 2: return launch_qgemm<CfgW4GateUp<2>>(tmA, tmB, p, 0, s);
        default: return launch_qgemm<CfgW4GateUp<1>>(tmA, tmB, p, 0, s);
    }
}

}  // namespace qmm
