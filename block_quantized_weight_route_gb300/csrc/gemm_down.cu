// Routed-MoE down product: q8_1 H (int8 codes + fp16 d per 32) times IQ4_NL
// weights (4-bit codebook indices + fp16 scale per 32).  Each 32-K block is one
// exact integer dot on the f16 tensor path, folded with d_H * d_W in fp32.
// Kernel body: qgemm.cuh.
#include "qgemm.cuh"

namespace qmm {

using CfgDown = GemmCfg<AMode::I8_CONV, BMode::IQ4, Epi::FOLD_IQ4, 128, 4, 8, 4, 3, true>;

int smem_iq4_down() { return CfgDown::SMEM_BYTES; }

cudaError_t launch_iq4_down(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid,
                            cudaStream_t s) {
    static_assert(CfgDown::SMEM_BYTES <= 232448, "shared memory");
    cudaError_t e =
        cudaFuncSetAttribute(qgemm_kernel<CfgDown>, cudaFuncAttributeMaxDynamicSharedMemorySize, CfgDown::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    qgemm_kernel<CfgDown><<<grid, CfgDown::THREADS, CfgDown::SMEM_BYTES, s>>>(tmA, tmB, p);
    return cudaGetLastError();
}

}  // namespace qmm
