// W4 (e2m1 codes, E4M3 per-16 scales, fp32 scale2) GEMMs: the dense prefill
// projection and the routed-MoE gate/up product with its fused SwiGLU + q8_1
// epilogue.  Kernel body: qgemm.cuh.
#include "qgemm.cuh"

namespace qmm {

// Dense: 128 x 256 tiles, 8 converter warps (one weight row per thread), 4 epilogue warps.
using CfgW4Dense = GemmCfg<BMode::W4, Epi::STORE, 256, 8, 4, 4, 3, false>;
// Gate/up: 128 token rows x (128 gate + 128 up) weight rows per tile.
using CfgW4GateUp = GemmCfg<BMode::W4, Epi::SWIGLU_Q81, 256, 8, 4, 4, 3, true>;

int smem_w4a16_dense() { return CfgW4Dense::SMEM_BYTES; }
int smem_w4_gate_up_swiglu() { return CfgW4GateUp::SMEM_BYTES; }

template <class C>
static cudaError_t launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid,
                          cudaStream_t s) {
    static_assert(C::SMEM_BYTES <= 232448, "shared memory");
    cudaError_t e = cudaFuncSetAttribute(qgemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    qgemm_kernel<C><<<grid, C::THREADS, C::SMEM_BYTES, s>>>(tmA, tmB, p);
    return cudaGetLastError();
}

cudaError_t launch_w4a16_dense(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid,
                               cudaStream_t s) {
    return launch<CfgW4Dense>(tmA, tmB, p, grid, s);
}

cudaError_t launch_w4_gate_up_swiglu(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid,
                                     cudaStream_t s) {
    return launch<CfgW4GateUp>(tmA, tmB, p, grid, s);
}

}  // namespace qmm
