// gemm_instances.cuh -- the four kernel configurations.
#pragma once

#include "gemm_kernel.cuh"
#include "kernels.h"

namespace chord {

// template <BK, code stages, token stages, A stages in TMEM, token tile, accum buffers, gate_up>
template <bool G> using CfgD32 = GemmCfg<256, 6, 4, 3, 32, 2, G>;
template <bool G> using CfgD64 = GemmCfg<256, 6, 3, 3, 64, 2, G>;
template <bool G> using CfgD128 = GemmCfg<256, 4, 2, 2, 128, 2, G>;
template <bool G> using CfgP256 = GemmCfg<128, 4, 2, 4, 256, 1, G>;

template <class C>
cudaError_t launch_gemm_cfg(const CUtensorMap& map, const GemmArgs& a, int grid, cudaStream_t s)
{
    static bool attr_set = false;  // set once per configuration (first launch)
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(w4a16_gemm_kernel<C>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    w4a16_gemm_kernel<C><<<grid, kGemmThreads, C::SMEM_BYTES, s>>>(map, a);
    return cudaGetLastError();
}

}  // namespace chord
