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
// library until the process exits.  Its device address is looked up once per
// device with cudaGetSymbolAddress (the host-side name of a __device__ array is
// only a stand-in, never a device pointer).
#include <cuda_runtime.h>

#include <mutex>

#include "chord.h"
#include "kernels.h"

namespace chord {
namespace {

constexpr int64_t kScratchInts = 1 << 20;  // 4 MiB of int32
constexpr int64_t kErrInts = 64;           // first 256 bytes: the error word

static __device__ __align__(256) int32_t g_align_scratch[kScratchInts];

std::mutex g_scratch_mu;
int32_t* g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device (set-up on the
// first call per device).
chord_status scratch_on_current_device(int32_t** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return CHORD_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_align_scratch) != cudaSuccess || p == nullptr)
            return CHORD_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_ptr[dev];
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
    if (!expert_map && E_local != E_global)
        return CHORD_ERR_INVALID_ARG;
    if (T * k >= (int64_t(1) << 31))
        return CHORD_ERR_UNSUPPORTED_SHAPE;
    if (!sorted_ids || !expert_ids || !num_tokens_padded || (T > 0 && !topk_ids))
        return CHORD_ERR_INVALID_ARG;
    if (capacity < chord_moe_align_capacity(T, k, E_local, block_m) || capacity % block_m != 0)
        return CHORD_ERR_CAPACITY;
    const int64_t tiles = (T * k + 255) / 256;
    if ((tiles > 0 ? tiles : 1) * E_local > kScratchInts - kErrInts)
        return CHORD_ERR_UNSUPPORTED_SHAPE;  // beyond the fixed scratch array
    int32_t* scratch = nullptr;
    chord_status st = scratch_on_current_device(&scratch);
    if (st != CHORD_OK)
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
    return launch_align(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? CHORD_OK
                                                                              : CHORD_ERR_CUDA;
}
