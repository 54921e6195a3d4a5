// gemm_down.cu -- down GEMM instances (per-pair store / token reduction / row store).
#include "gemm_instances.cuh"

namespace chord {

cudaError_t launch_gemm_down(int cfg, const CUtensorMap& map, const CUtensorMap& smap, const CUtensorMap& bmap,
                             const GemmArgs& a, int grid, cudaStream_t s)
{
    return dispatch_down<false>(cfg, map, smap, bmap, a, grid, s);
}

int gemm_cfg_smem_down(int cfg)
{
    switch (cfg) {
    case kCfgD32: return CfgD32<false>::SMEM_BYTES;
    case kCfgD64: return CfgD64<false>::SMEM_BYTES;
    case kCfgD128: return CfgD128<false>::SMEM_BYTES;
    case kCfgP192: return CfgP192<false>::SMEM_BYTES;
    case kCfgS32: return CfgS32::SMEM_BYTES;
    case kCfgS64: return CfgS64::SMEM_BYTES;
    default: return 0;
    }
}

int gemm_cfg_tpu_max_down(int cfg)
{
    switch (cfg) {
    case kCfgS32: return CfgS32::TPU_MAX;
    case kCfgS64: return CfgS64::TPU_MAX;
    default: return 1;
    }
}

int gemm_cfg_bk(int cfg) { return cfg == kCfgP192 ? 128 : 256; }

int gemm_cfg_maxn(int cfg)
{
    switch (cfg) {
    case kCfgD32:
    case kCfgS32: return 32;
    case kCfgD64:
    case kCfgS64: return 64;
    case kCfgD128: return 128;
    case kCfgP192: return 192;
    default: return 0;
    }
}

}  // namespace chord
