// gemm_gate_up.cu -- gate/up GEMM instances (fused SiLU(gate) * up epilogue).
#include "gemm_instances.cuh"

namespace chord {

cudaError_t launch_gemm_gate_up(int cfg, const CUtensorMap& map, const CUtensorMap& smap, const CUtensorMap& bmap,
                                const GemmArgs& a, int grid, cudaStream_t s)
{
    switch (cfg) {
    case kCfgD32: return launch_gemm_cfg<CfgD32<true>>(map, smap, bmap, a, grid, s);
    case kCfgD64: return launch_gemm_cfg<CfgD64<true>>(map, smap, bmap, a, grid, s);
    case kCfgD128: return launch_gemm_cfg<CfgD128<true>>(map, smap, bmap, a, grid, s);
    case kCfgP192: return launch_gemm_cfg<CfgP192<true>>(map, smap, bmap, a, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

int gemm_cfg_smem_gate_up(int cfg)
{
    switch (cfg) {
    case kCfgD32: return CfgD32<true>::SMEM_BYTES;
    case kCfgD64: return CfgD64<true>::SMEM_BYTES;
    case kCfgD128: return CfgD128<true>::SMEM_BYTES;
    case kCfgP192: return CfgP192<true>::SMEM_BYTES;
    default: return 0;
    }
}

}  // namespace chord
