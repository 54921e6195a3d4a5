// gemm_gate_up.cu -- gate/up GEMM instances (fused SiLU(gate) * up epilogue).
#include "gemm_instances.cuh"

namespace chord {

cudaError_t launch_gemm_gate_up(int cfg, const CUtensorMap& map, const CUtensorMap& smap, const CUtensorMap& bmap,
                                const GemmArgs& a, int grid, cudaStream_t s)
{
    return dispatch_gate_up<false>(cfg, map, smap, bmap, a, grid, s);
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
