// kernels.h -- launch interfaces of the device code (host side of the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "chord_internal.h"

namespace chord {

// Whether launch_pdl asks for programmatic stream serialization on this host
// thread, set per call: on for decode-sized calls (it hides the launch
// gaps: EP8 decode, 512 tokens, 237 -> 233 us), off for large ones (prefill measured 661 ->
// 692 us with it).  The kernels are correct either way: griddepcontrol.wait
// returns at once when the launch was serialized.
inline thread_local bool g_launch_pdl = true;
constexpr int64_t kPdlMaxRows = 4096;  // routed rows up to which a call uses it
struct PdlScope {
    bool prev;
    explicit PdlScope(bool on) : prev(g_launch_pdl) { g_launch_pdl = on; }
    ~PdlScope() { g_launch_pdl = prev; }
};

// Launch with programmatic stream serialization (the kernel waits for its
// predecessor itself, with griddepcontrol.wait, before it touches memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = g_launch_pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// The current device: its index and SM count; CHORD_ERR_NO_DEVICE unless it is
// an sm_103 GPU (api.cu; the attributes are read once per device).
struct DeviceInfo {
    int device = -1;
    int sms = 0;
    bool ok = false;
};
chord_status device_info(DeviceInfo* out);
// CHORD_OK for cudaSuccess, else CHORD_ERR_CUDA.
chord_status from_cuda(cudaError_t e);

struct AlignArgs {
    const int32_t* topk_ids;
    int64_t num_pairs;  // T*k, also the sentinel
    int E_global;
    const int32_t* expert_map;
    int E_local;
    int block_m;
    int32_t* sorted_ids;
    int32_t* expert_ids;
    int32_t* num_tokens_padded;
    int64_t capacity;
    int32_t* tile_hist;  // [n_tiles, E_local] scratch
    int n_tiles;         // ceil(num_pairs / 256)
    int* err;
};

// Router: logits float [T, E] -> topk ids int32 [T, k] and weights float [T, k].
struct RouteArgs {
    const float* logits;
    int64_t T;
    int E;       // <= 1024
    int k;       // <= min(E, 32)
    int renorm;  // weights renormalised over the k chosen
    int32_t* ids;
    float* w;
};

enum Layout : int { kLayoutIndexed = 0, kLayoutContiguous = 1, kLayoutMasked = 2 };

struct PrepArgs {
    int layout;
    // indexed
    const int32_t* expert_ids;
    const int32_t* num_tokens_padded;
    int64_t capacity;
    int block_rows;  // block_m (indexed) or 16 (contiguous)
    // contiguous
    const int32_t* m_indices;
    int64_t M;
    // masked
    const int32_t* masked_m;
    int64_t max_m;
    int E_local;
    // outputs: two chunk lists (gate_up, down) with their token-tile limits
    int maxn[2];
    Chunk* chunks[2];
    int max_chunks;       // entries of each chunk list
    int32_t* num_chunks;  // [2]
    // indexed layout: gather the routed token rows of x into padded-row order
    // (gx_out[r] = x[sorted_ids[r] / topk] for r < num_tokens_padded and a valid
    // pair; sentinel rows are left as they are)
    const uint16_t* gx_src;  // x [T, gx_H]
    uint16_t* gx_out;        // [capacity, gx_H]
    const int32_t* gx_ids;   // sorted_ids
    int gx_topk;
    int64_t gx_pairs;        // T*k, the sentinel
    int gx_H;
    // compacted: only the rows holding a pair, in padded-row order with the
    // padding left out (E_local <= 1024); the gate/up chunk list's brow0
    // points into them
    int gx_compact;
    // per padded row r: {pair p, token p / topk, bits of topk_weights[p], 0},
    // or {-1, 0, 0, 0} for a row with no pair; rows r < meta_rows, or
    // r < num_tokens_padded when meta_rows < 0
    int4* meta_out;
    const int32_t* meta_pair;  // pair id of each padded row (sorted_ids / row_to_pair)
    const float* meta_w;       // topk_weights [T * topk]
    int meta_topk;
    int64_t meta_pairs;
    int64_t meta_rows;
    // masked layout: its valid rows (row e * max_m + r, r < masked_m[e]) copied
    // to mc_out in expert order with no gaps, the gate/up GEMM's token rows
    // (its chunk list's brow0 points there)
    const uint16_t* mc_src;
    uint16_t* mc_out;
    int mc_H;
    // buffers to clear
    int32_t* zero_i32;  // (the K-split piece counters; cleared by block 0)
    int zero_i32_count;
    float* zero_f32;
    int64_t zero_count;
    int32_t* fill_i32;  // set to -1
    int64_t fill_count;
    // prepacked weights: the two packs' headers (gate/up, down) and what each
    // must say; on a mismatch both chunk lists
    // are left empty (the GEMMs compute nothing) and CHORD_DEVERR_PACKED is set
    const uint32_t* pk_hdr[2];
    uint32_t pk_want[2][5];  // {kind, experts at least, N, K, weight format}
    int* err;
};

struct CombineArgs {
    int64_t T;
    int k;
    int H;
    const int32_t* pair_row;
    const float* topk_weights;
    const float* y_pairs;
    uint16_t* out;
};

cudaError_t launch_align(const AlignArgs& a, cudaStream_t s);
// Router, then align of its ids (a.topk_ids == r.ids): one CTA for both up to
// 64 tokens and 512 local experts, else a router kernel and launch_align.
cudaError_t launch_route_align(const RouteArgs& r, const AlignArgs& a, cudaStream_t s);

// chord_w4a16_prepack: header, then every 16-byte piece of every block.
struct PackArgs {
    int kind;               // CHORD_PACK_GATE_UP / CHORD_PACK_DOWN
    const int32_t* q;       // [E, N, K/8]
    const uint16_t* sc;     // INT4: bf16 scales [E, N, K/32]
    int E, N, K;
    uint8_t* out;           // header + E * (N/128) * (K/256) blocks
    int fmt;                // kPackFmtInt4 / kPackFmtMxfp4 (header word kPackFormatWord)
    const uint8_t* sc8;     // MXFP4: E8M0 scale bytes [E, N, K/32], widened to bf16 2^(e-127)
};
cudaError_t launch_prepack(const PackArgs& a, int sms, cudaStream_t s);
cudaError_t launch_prep(const PrepArgs& a, int work_blocks, cudaStream_t s);
// Sets CHORD_DEVERR_SCALE_RANGE when a scale of a[0..na) or b[0..nb) (bf16
// bits) is neither +-0 nor of magnitude in [2^-86, 2^35).
cudaError_t launch_scale_check(const uint16_t* a, int64_t na, const uint16_t* b, int64_t nb,
                               int* err, int sms, cudaStream_t s);
cudaError_t launch_finalize(const float* acc, uint16_t* out, int64_t n, int sms, cudaStream_t s);
cudaError_t launch_combine_pairs(const CombineArgs& a, cudaStream_t s);

// GEMM kernel configurations (token tile, stage depth, pipeline depths)
enum GemmConfig : int {
    kCfgD32 = 0,    // BK 256, token tile <= 32, deep code ring: weight-streaming decode
    kCfgD64 = 1,    // BK 256, token tile <= 64
    kCfgD128 = 2,   // BK 256, token tile <= 128
    kCfgP192 = 3,   // BK 128, token tile <= 192, two accumulators: prefill / short K
    kCfgS32 = 4,    // down only, one-stage K: token tile <= 32, up to 4 weight tiles per unit
    kCfgS64 = 5,    // down only, one-stage K: token tile <= 64, up to 2 weight tiles per unit
    kNumGemmConfigs = 6
};

int gemm_cfg_bk(int cfg);
// Most weight tiles one unit of the down GEMM may hold (one-stage K only).
int gemm_cfg_tpu_max_down(int cfg);
int gemm_cfg_maxn(int cfg);
int gemm_cfg_smem(int cfg, bool gate_up);

// Launch one GEMM (gate_up with fused SiLU*up, or down with its epilogue).
// codes_map / scales_map / b_map: the tensor maps of api.cu's codes_map(),
// scales_map() (read only for BK 256 stages) and rows_map() for this
// configuration's BK and token tile.
cudaError_t launch_gemm(int cfg, bool gate_up, const CUtensorMap& codes_map,
                        const CUtensorMap& scales_map, const CUtensorMap& b_map, const GemmArgs& a,
                        int grid, cudaStream_t s);

}  // namespace chord
