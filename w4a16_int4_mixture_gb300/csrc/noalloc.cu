// noalloc.cu -- moe_align for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand over a workspace: code that runs
// inside an allocator or memory-pool callback, a plugin whose host framework
// owns every device buffer and gives it only inputs and outputs, or an embedded
// runtime that forbids allocation after start-up.  For them this file offers
// the routing alignment with its scratch (the per-tile expert histogram and the
// error word) in a fixed, file-scope device array instead of a workspace.
//
// The array is kScratchInts int32 (4 MiB) and lives on every GPU that loads the
// library until the process exits.  Its device address is looked up with
// cudaGetSymbolAddress (the host-side name of a __device__ array is only a
// stand-in, never a device pointer) on the first call in each CUDA context of
// a device, and looked up again when the device's current context changes (a
// symbol address belongs to the context that loaded the module).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "chord.h"
#include "kernels.h"

namespace chord {
namespace {

constexpr int64_t kScratchInts = 1 << 20;  // 4 MiB of int32
constexpr int64_t kErrInts = 64;           // first 256 bytes: the error word

static __device__ __align__(256) int32_t g_align_scratch[kScratchInts];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

std::mutex g_scratch_mu;
CtxGetCurrentFn g_ctx_get_current = nullptr;
struct ScratchAddr {
    CUcontext ctx;
    int32_t* ptr;
};
ScratchAddr g_scratch[64] = {};

// Device address of the scratch array in the current context of the current
// device (looked up on the first call in that context).
chord_status scratch_on_current_device(int dev, int32_t** out)
{
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_ctx_get_current) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return CHORD_ERR_CUDA;
        g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    }
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
        return CHORD_ERR_CUDA;
    ScratchAddr& a = g_scratch[dev];
    if (a.ptr == nullptr || a.ctx != ctx) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_align_scratch);
        if (e != cudaSuccess || p == nullptr)
            return CHORD_ERR_CUDA;
        a.ctx = ctx;
        a.ptr = static_cast<int32_t*>(p);
    }
    *out = a.ptr;
    return CHORD_OK;
}

}  // namespace
}  // namespace chord

using namespace chord;

extern "C" chord_status chord_moe_align_noalloc(const int32_t* topk_ids, int64_t T, int k,
                                                int E_global, const int32_t* expert_map,
                                                int E_local, int block_m, int32_t* sorted_ids,
                                                int32_t* expert_ids, int32_t* num_tokens_padded,
                                                int64_t capacity, void* stream)
{
    if (T < 0 || k < 1 || k > 32 || E_global < 1 || E_local < 1 || E_local > 1024 || block_m < 1 ||
        block_m > 256)
        return CHORD_ERR_INVALID_ARG;
    if (T * k >= (int64_t(1) << 31))
        return CHORD_ERR_UNSUPPORTED_SHAPE;
    // sizes first: a problem beyond the fixed scratch array is refused before
    // any pointer is looked at
    const int64_t tiles = (T * k + 255) / 256;
    if ((tiles > 0 ? tiles : 1) * E_local > kScratchInts - kErrInts)
        return CHORD_ERR_UNSUPPORTED_SHAPE;
    if (!expert_map && E_local != E_global)
        return CHORD_ERR_INVALID_ARG;
    if (!sorted_ids || !expert_ids || !num_tokens_padded || (T > 0 && !topk_ids))
        return CHORD_ERR_INVALID_ARG;
    if (capacity < chord_moe_align_capacity(T, k, E_local, block_m) || capacity % block_m != 0)
        return CHORD_ERR_CAPACITY;
    DeviceInfo dev;
    chord_status st = device_info(&dev);
    if (st != CHORD_OK)
        return st;
    int32_t* scratch = nullptr;
    if ((st = scratch_on_current_device(dev.device, &scratch)) != CHORD_OK)
        return st;
    AlignArgs a{};
    a.topk_ids = topk_ids;
    a.num_pairs = T * k;
    a.E_global = E_global;
    a.expert_map = expert_map;
    a.E_local = E_local;
    a.block_m = block_m;
    a.sorted_ids = sorted_ids;
    a.expert_ids = expert_ids;
    a.num_tokens_padded = num_tokens_padded;
    a.capacity = capacity;
    // every histogram entry the kernels read is written by this call first, and
    // the scan clears the error word, so nothing left from an earlier call leaks
    a.tile_hist = scratch + kErrInts;
    a.n_tiles = static_cast<int>(tiles);
    a.err = scratch;
    PdlScope pdl(T * k <= kPdlMaxRows);
    return from_cuda(launch_align(a, static_cast<cudaStream_t>(stream)));
}
