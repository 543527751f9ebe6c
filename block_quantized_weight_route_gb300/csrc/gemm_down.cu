// Routed-MoE down product (q8_1 H x IQ4_NL weights); kernel body: down_iq4.cuh.
#include "down_iq4.cuh"

namespace qmm {

int smem_iq4_down() { return DownCfg::SMEM_BYTES; }

template <bool COMBINE>
static cudaError_t launch_down(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid,
                               cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(down_iq4_kernel<DownCfg, COMBINE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DownCfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if constexpr (DownCfg::REG_SPLIT) {
        // the warpgroups' register shares add up to 128 a thread: launch only if
        // the kernel is allocated exactly that many (more shares than the pool
        // would leave a setmaxnreg.inc waiting)
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, down_iq4_kernel<DownCfg, COMBINE>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != DownCfg::REGS_LAUNCH) return cudaErrorInvalidConfiguration;
    }
    down_iq4_kernel<DownCfg, COMBINE><<<grid, DownCfg::THREADS, DownCfg::SMEM_BYTES, s>>>(tmA, tmB, p);
    return cudaGetLastError();
}

cudaError_t launch_iq4_down(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid, bool combine,
                            cudaStream_t s) {
    return combine ? launch_down<true>(tmA, tmB, p, grid, s) : launch_down<false>(tmA, tmB, p, grid, s);
}

}  // namespace qmm
