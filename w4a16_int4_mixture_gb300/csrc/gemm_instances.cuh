// gemm_instances.cuh -- the kernel configurations and their launchers.
#pragma once

#include "gemm_kernel.cuh"
#include "kernels.h"

namespace chord {

// template <BK, code stages, token stages, A stages in TMEM, token tile, accum buffers, gate_up
//           [, accumulator columns: several weight tiles per unit for a one-stage K]
//           [, K stages per accumulation chain]>
// The gate/up GEMM (K = hidden size, the long reduction) restarts its
// accumulator every kPsDecode / kPsWide / kPsPrefill elements of K and adds
// the partials in fp32.  The 32-token tile has room in tensor memory for a
// third accumulator buffer, so its MMA never waits for a merge; the other
// tiles' MMA waits for each merge, so they take longer chains (measured on
// the Kimi-shaped workloads, K = 7168: chains of 1024 / 1792 / 1792 elements
// bring the gate/up output's rounding flips against an fp64 evaluation to
// 0.9-1.7x the fp32 oracle's rate and cost 6 / 9 / 19 % of the decode /
// skewed / prefill gate/up time; 1792 / 3584 / 3584 cost 4 / 3 / 6 % at 1.7
// / 3.5 / 3x the oracle's rate, and at 3x one unlucky flip took a prefill
// output element to 5x the tolerance against fp64; one chain per unit flips
// 7x as often).
constexpr int kPsDecode = 1024;
constexpr int kPsWide = 1792;
constexpr int kPsPrefill = 1792;
// (three token stages, as many as A stages, so that the two rings share
// their barriers: see FUSED_RINGS)
template <bool G> using CfgD32 = GemmCfg<256, 6, 3, 3, 32, G ? 3 : 2, G, 32, G ? kPsDecode / 256 : 0>;
template <bool G> using CfgD64 = GemmCfg<256, 6, 3, 3, 64, 2, G, 64, G ? kPsWide / 256 : 0>;
// down GEMMs with a one-stage K (token-stationary units): a unit is one
// chunk and a run of weight tiles sharing its token tile, each tile in the
// next of eight (32) or four (64) accumulator buffers, at the cost of one A
// stage
using CfgS32 = GemmCfg<256, 6, 4, 2, 32, 8, false, 32, 0, true>;
using CfgS64 = GemmCfg<256, 6, 3, 2, 64, 4, false, 64, 0, true>;
template <bool G> using CfgD128 = GemmCfg<256, 4, 2, 2, 128, 2, G, 128, G ? kPsWide / 256 : 0>;
template <bool G> using CfgP192 = GemmCfg<128, 4, 3, 2, 192, 2, G, 192, G ? kPsPrefill / 128 : 0>;

template <class C, bool PK, int FMT>
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
        // Before the first launch on a device: the configuration must fit this
        // device as built (its static and dynamic shared memory within the
        // opt-in limit, its register allocation allowing C::THREADS threads);
        // otherwise nothing is launched and the call reports a CUDA error.
        cudaFuncAttributes fa;
        int optin = 0;
        e = cudaFuncGetAttributes(&fa, w4a16_gemm_kernel<C, PK, FMT>);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess)
            return e;
        if (fa.sharedSizeBytes + static_cast<size_t>(C::SMEM_BYTES) > static_cast<size_t>(optin) ||
            fa.maxThreadsPerBlock < C::THREADS)
            return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(w4a16_gemm_kernel<C, PK, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        attr_set[dev] = true;
    }
    return launch_pdl(w4a16_gemm_kernel<C, PK, FMT>, grid, C::THREADS, C::SMEM_BYTES, s, map, smap, bmap,
                      a);
}

// The configurations of each GEMM, plain (PK false) or prepacked weights, INT4
// or MXFP4 (FMT); each form is instantiated in its own translation unit.
template <bool PK, int FMT = kFmtInt4>
cudaError_t dispatch_gate_up(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                             const CUtensorMap& bmap, const GemmArgs& a, int grid, cudaStream_t s)
{
    switch (cfg) {
    case kCfgD32: return launch_gemm_cfg<CfgD32<true>, PK, FMT>(map, smap, bmap, a, grid, s);
    case kCfgD64: return launch_gemm_cfg<CfgD64<true>, PK, FMT>(map, smap, bmap, a, grid, s);
    case kCfgD128: return launch_gemm_cfg<CfgD128<true>, PK, FMT>(map, smap, bmap, a, grid, s);
    case kCfgP192: return launch_gemm_cfg<CfgP192<true>, PK, FMT>(map, smap, bmap, a, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

template <bool PK, int FMT = kFmtInt4>
cudaError_t dispatch_down(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                          const CUtensorMap& bmap, const GemmArgs& a, int grid, cudaStream_t s)
{
    switch (cfg) {
    case kCfgD32: return launch_gemm_cfg<CfgD32<false>, PK, FMT>(map, smap, bmap, a, grid, s);
    case kCfgD64: return launch_gemm_cfg<CfgD64<false>, PK, FMT>(map, smap, bmap, a, grid, s);
    case kCfgD128: return launch_gemm_cfg<CfgD128<false>, PK, FMT>(map, smap, bmap, a, grid, s);
    case kCfgP192: return launch_gemm_cfg<CfgP192<false>, PK, FMT>(map, smap, bmap, a, grid, s);
    case kCfgS32: return launch_gemm_cfg<CfgS32, PK, FMT>(map, smap, bmap, a, grid, s);
    case kCfgS64: return launch_gemm_cfg<CfgS64, PK, FMT>(map, smap, bmap, a, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace chord
