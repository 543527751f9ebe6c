// FP8 (E4M3) weight GEMM with one fp32 scale per 128x128 block: each 128-K block
// is accumulated unscaled in its own TMEM buffer and folded once with its scale.
// Kernel body: qgemm.cuh.
#include "qgemm.cuh"

namespace qmm {

using CfgFp8 = GemmCfg<BMode::FP8, Epi::FOLD_FP8, 128, 4, 8, 4, 4, false>;

int smem_fp8_blk128() { return CfgFp8::SMEM_BYTES; }

cudaError_t launch_fp8_blk128(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid,
                              cudaStream_t s) {
    static_assert(CfgFp8::SMEM_BYTES <= 232448, "shared memory");
    cudaError_t e =
        cudaFuncSetAttribute(qgemm_kernel<CfgFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize, CfgFp8::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    qgemm_kernel<CfgFp8><<<grid, CfgFp8::THREADS, CfgFp8::SMEM_BYTES, s>>>(tmA, tmB, p);
    return cudaGetLastError();
}

}  // namespace qmm
