// gemm_instances.cuh -- the kernel configurations and their launchers.
#pragma once

#include "gemm_kernel.cuh"
#include "kernels.h"

namespace chord {

// template <BK, code stages, token stages, A stages in TMEM, token tile, accum buffers, gate_up
//           [, accumulator columns: several weight tiles per unit for a one-stage K]>
template <bool G> using CfgD32 = GemmCfg<256, 6, 4, 3, 32, 2, G>;
template <bool G> using CfgD64 = GemmCfg<256, 6, 3, 3, 64, 2, G>;
// down GEMMs with a one-stage K: four (32) or two (64) weight tiles per
// unit, at the cost of one A stage
using CfgS32 = GemmCfg<256, 6, 4, 2, 32, 2, false, 128>;
using CfgS64 = GemmCfg<256, 6, 3, 2, 64, 2, false, 128>;
template <bool G> using CfgD128 = GemmCfg<256, 4, 2, 2, 128, 2, G>;
template <bool G> using CfgP192 = GemmCfg<128, 4, 3, 2, 192, 2, G>;

template <class C, bool PK>
cudaError_t launch_gemm_cfg(const CUtensorMap& map, const CUtensorMap& smap,
                            const CUtensorMap& bmap, const GemmArgs& a, int grid, cudaStream_t s)
{
    static bool attr_set[64] = {};  // per device, set on the first launch there
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(w4a16_gemm_kernel<C, PK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        attr_set[dev] = true;
    }
    return launch_pdl(w4a16_gemm_kernel<C, PK>, grid, C::THREADS, C::SMEM_BYTES, s, map, smap, bmap, a);
}

// The configurations of each GEMM, plain (PK false) or prepacked weights; each
// form is instantiated in its own translation unit.
template <bool PK>
cudaError_t dispatch_gate_up(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                             const CUtensorMap& bmap, const GemmArgs& a, int grid, cudaStream_t s)
{
    switch (cfg) {
    case kCfgD32: return launch_gemm_cfg<CfgD32<true>, PK>(map, smap, bmap, a, grid, s);
    case kCfgD64: return launch_gemm_cfg<CfgD64<true>, PK>(map, smap, bmap, a, grid, s);
    case kCfgD128: return launch_gemm_cfg<CfgD128<true>, PK>(map, smap, bmap, a, grid, s);
    case kCfgP192: return launch_gemm_cfg<CfgP192<true>, PK>(map, smap, bmap, a, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

template <bool PK>
cudaError_t dispatch_down(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                          const CUtensorMap& bmap, const GemmArgs& a, int grid, cudaStream_t s)
{
    switch (cfg) {
    case kCfgD32: return launch_gemm_cfg<CfgD32<false>, PK>(map, smap, bmap, a, grid, s);
    case kCfgD64: return launch_gemm_cfg<CfgD64<false>, PK>(map, smap, bmap, a, grid, s);
    case kCfgD128: return launch_gemm_cfg<CfgD128<false>, PK>(map, smap, bmap, a, grid, s);
    case kCfgP192: return launch_gemm_cfg<CfgP192<false>, PK>(map, smap, bmap, a, grid, s);
    case kCfgS32: return launch_gemm_cfg<CfgS32, PK>(map, smap, bmap, a, grid, s);
    case kCfgS64: return launch_gemm_cfg<CfgS64, PK>(map, smap, bmap, a, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace chord
