// gemm_packed.cu -- both GEMMs' instances for prepacked weights (chord_w4a16_prepack).
#include "gemm_instances.cuh"

namespace chord {

cudaError_t launch_gemm_gate_up_packed(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                                       const CUtensorMap& bmap, const GemmArgs& a, int grid,
                                       cudaStream_t s)
{
    return dispatch_gate_up<true>(cfg, map, smap, bmap, a, grid, s);
}

cudaError_t launch_gemm_down_packed(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                                    const CUtensorMap& bmap, const GemmArgs& a, int grid,
                                    cudaStream_t s)
{
    return dispatch_down<true>(cfg, map, smap, bmap, a, grid, s);
}

}  // namespace chord
