// gemm_mxfp4.cu -- both GEMMs' instances for MXFP4 weights (chord_mxfp4_prepack packs).
#include "gemm_instances.cuh"

namespace chord {

cudaError_t launch_gemm_gate_up_mx(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                                   const CUtensorMap& bmap, const GemmArgs& a, int grid,
                                   cudaStream_t s)
{
    return dispatch_gate_up<true, kFmtMxfp4>(cfg, map, smap, bmap, a, grid, s);
}

cudaError_t launch_gemm_down_mx(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                                const CUtensorMap& bmap, const GemmArgs& a, int grid, cudaStream_t s)
{
    return dispatch_down<true, kFmtMxfp4>(cfg, map, smap, bmap, a, grid, s);
}

}  // namespace chord
