// api.cu -- the C ABI (include/chord.h): argument checks, schedule selection,
// workspace layout, tensor-map memo and the launch sequence of each call.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "chord.h"
#include "kernels.h"

namespace chord {

cudaError_t launch_gemm_gate_up(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                                const CUtensorMap& bmap, const GemmArgs& a, int grid,
                                cudaStream_t s);
cudaError_t launch_gemm_down(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                             const CUtensorMap& bmap, const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_gemm_gate_up_packed(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                                       const CUtensorMap& bmap, const GemmArgs& a, int grid,
                                       cudaStream_t s);
cudaError_t launch_gemm_down_packed(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                                    const CUtensorMap& bmap, const GemmArgs& a, int grid,
                                    cudaStream_t s);
cudaError_t launch_gemm_gate_up_mx(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                                   const CUtensorMap& bmap, const GemmArgs& a, int grid,
                                   cudaStream_t s);
cudaError_t launch_gemm_down_mx(int cfg, const CUtensorMap& map, const CUtensorMap& smap,
                                const CUtensorMap& bmap, const GemmArgs& a, int grid, cudaStream_t s);
int gemm_cfg_smem_gate_up(int cfg);
int gemm_cfg_smem_down(int cfg);

// packed: prepacked weights; mx: MXFP4 packs (always prepacked)
cudaError_t launch_gemm(int cfg, bool gate_up, bool packed, bool mx, const CUtensorMap& map,
                        const CUtensorMap& smap, const CUtensorMap& bmap, const GemmArgs& a,
                        int grid, cudaStream_t s)
{
    if (mx)
        return gate_up ? launch_gemm_gate_up_mx(cfg, map, smap, bmap, a, grid, s)
                       : launch_gemm_down_mx(cfg, map, smap, bmap, a, grid, s);
    if (packed)
        return gate_up ? launch_gemm_gate_up_packed(cfg, map, smap, bmap, a, grid, s)
                       : launch_gemm_down_packed(cfg, map, smap, bmap, a, grid, s);
    return gate_up ? launch_gemm_gate_up(cfg, map, smap, bmap, a, grid, s)
                   : launch_gemm_down(cfg, map, smap, bmap, a, grid, s);
}

int gemm_cfg_smem(int cfg, bool gate_up)
{
    return gate_up ? gemm_cfg_smem_gate_up(cfg) : gemm_cfg_smem_down(cfg);
}

// ---------------------------------------------------------------------------
// device properties
// ---------------------------------------------------------------------------
namespace {
std::mutex g_dev_mu;
DeviceInfo g_dev[64];
}  // namespace

chord_status device_info(DeviceInfo* out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return CHORD_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (d.device != dev) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return CHORD_ERR_NO_DEVICE;
        d.device = dev;
        d.sms = sms;
        d.ok = (major == 10 && minor == 3);
    }
    *out = d;
    return d.ok ? CHORD_OK : CHORD_ERR_NO_DEVICE;
}

chord_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CHORD_OK : CHORD_ERR_CUDA; }

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// tensor maps, memoised by everything that goes into the encoding
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct MapKey {
    const void* ptr;
    int dtype;
    int rank;
    uint64_t dims[4];
    uint64_t strides[3];
    uint32_t box[4];
    int swizzle;
    int device;
    bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};

struct MapEntry {
    MapKey key;
    CUtensorMap map;
    uint64_t stamp;
};

std::mutex g_map_mu;
std::vector<MapEntry> g_maps;
uint64_t g_stamp = 0;

chord_status encode_map(MapKey key, CUtensorMap* out)
{
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (auto& e : g_maps)
        if (e.key == key) {
            e.stamp = ++g_stamp;
            *out = e.map;
            return CHORD_OK;
        }
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return CHORD_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    CUtensorMap m;
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4], es[4] = {1, 1, 1, 1};
    for (int i = 0; i < key.rank; ++i) {
        dims[i] = key.dims[i];
        box[i] = key.box[i];
    }
    for (int i = 0; i + 1 < key.rank; ++i)
        strides[i] = key.strides[i];
    const CUresult r = g_encode(&m, static_cast<CUtensorMapDataType>(key.dtype), key.rank,
                                const_cast<void*>(key.ptr), dims, strides, box, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE,
                                static_cast<CUtensorMapSwizzle>(key.swizzle),
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return CHORD_ERR_CUDA;
    if (g_maps.size() >= 48) {
        size_t victim = 0;
        for (size_t i = 1; i < g_maps.size(); ++i)
            if (g_maps[i].stamp < g_maps[victim].stamp)
                victim = i;
        g_maps.erase(g_maps.begin() + static_cast<long>(victim));
    }
    g_maps.push_back({key, m, ++g_stamp});
    *out = m;
    return CHORD_OK;
}

MapKey blank_key(const void* ptr, int dtype, int rank, int swizzle, int device)
{
    MapKey k;
    std::memset(&k, 0, sizeof k);
    k.ptr = ptr;
    k.dtype = dtype;
    k.rank = rank;
    k.swizzle = swizzle;
    k.device = device;
    return k;
}

// Packed codes of one GEMM: int32 words, rows of K/8, read in halves of 128
// codes (16 words, 64 bytes, 64B swizzle) so that a stage of bk codes lands
// as bk/128 halves of [128 tile rows][64 bytes], the layout the dequant reads
// (and the one chord_w4a16_prepack stores).  gate_up (I > 0): a 4-D map
// {16 words, E*N - I rows, 2 halves I rows apart, K/128 blocks}, box {16, 64,
// 2, bk/128}: gate rows and the matching up rows in one box.  down: 3-D {16,
// rows, K/128}, box {16, 128, bk/128}.
chord_status codes_map(const int32_t* q, int64_t rows, int64_t K, int64_t I, int bk, int device,
                       CUtensorMap* out)
{
    const uint64_t row_bytes = static_cast<uint64_t>(K / 8) * 4;
    if (I > 0) {
        MapKey k = blank_key(q, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, CU_TENSOR_MAP_SWIZZLE_64B, device);
        k.dims[0] = 16;
        k.dims[1] = rows - I;
        k.dims[2] = 2;
        k.dims[3] = K / 128;
        k.strides[0] = row_bytes;
        k.strides[1] = row_bytes * I;
        k.strides[2] = 64;
        k.box[0] = 16;
        k.box[1] = 64;
        k.box[2] = 2;
        k.box[3] = bk / 128;
        return encode_map(k, out);
    }
    MapKey k = blank_key(q, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, CU_TENSOR_MAP_SWIZZLE_64B, device);
    k.dims[0] = 16;
    k.dims[1] = rows;
    k.dims[2] = K / 128;
    k.strides[0] = row_bytes;
    k.strides[1] = 64;
    k.box[0] = 16;
    k.box[1] = 128;
    k.box[2] = bk / 128;
    return encode_map(k, out);
}

// Group-32 scales of one GEMM: bf16 rows of K/32, boxes of 8 columns (16 bytes,
// one BK = 256 stage); the same 3-D gate/up pairing as the codes.
chord_status scales_map(const uint16_t* sc, int64_t rows, int64_t K, int64_t I, int device,
                        CUtensorMap* out)
{
    const uint64_t row_bytes = static_cast<uint64_t>(K / 32) * 2;
    if (I > 0) {
        MapKey k = blank_key(sc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, CU_TENSOR_MAP_SWIZZLE_NONE,
                             device);
        k.dims[0] = K / 32;
        k.dims[1] = rows - I;
        k.dims[2] = 2;
        k.strides[0] = row_bytes;
        k.strides[1] = row_bytes * I;
        k.box[0] = 8;
        k.box[1] = 64;
        k.box[2] = 2;
        return encode_map(k, out);
    }
    MapKey k = blank_key(sc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_NONE, device);
    k.dims[0] = K / 32;
    k.dims[1] = rows;
    k.strides[0] = row_bytes;
    k.box[0] = 8;
    k.box[1] = 128;
    return encode_map(k, out);
}

// Token rows (bf16 [rows, K], padded-row order), 128B swizzle, zero past the
// last row.  Token tiles of at most 64 rows: a 3-D map {64 columns, rows, K/64
// column blocks} with box {64, tile, bk/64}, one box per stage laid out as the
// stage's column blocks one after another.  Larger tiles: 2-D boxes {64, 64}.
chord_status rows_map(const uint16_t* x, int64_t rows, int64_t K, int tile, int bk, int device,
                      CUtensorMap* out)
{
    if (tile <= 64) {
        MapKey k = blank_key(x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, CU_TENSOR_MAP_SWIZZLE_128B,
                             device);
        k.dims[0] = 64;
        k.dims[1] = rows;
        k.dims[2] = K / 64;
        k.strides[0] = static_cast<uint64_t>(K) * 2;
        k.strides[1] = 128;
        k.box[0] = 64;
        k.box[1] = tile;
        k.box[2] = bk / 64;
        return encode_map(k, out);
    }
    MapKey k = blank_key(x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_128B, device);
    k.dims[0] = K;
    k.dims[1] = rows;
    k.strides[0] = static_cast<uint64_t>(K) * 2;
    k.box[0] = 64;
    k.box[1] = 64;
    return encode_map(k, out);
}

// ---------------------------------------------------------------------------
// schedule
// ---------------------------------------------------------------------------
struct Schedule {
    int cfg_gate_up;
    int cfg_down;
    bool reduce;  // fp32 reductions into token rows (else per-pair store + ordered combine)
};

// Token tile by expected routed rows per expert (page: "Kernel optimisation":
// the schedule is chosen from the routed tokens per expert, tok_e; prefill
// switches above 80 rows per expert).  Below the switch the weight-streaming
// decode pipeline with the smallest token tile that holds a typical expert
// (mean + 3 sigma of a Poisson count) in one chunk; above it the deep-N
// prefill tile of 192 tokens (two accumulator buffers, so the epilogue of one
// unit overlaps the MMAs of the next; larger experts split into chunks).
int pick_cfg(double tok_e, int K)
{
    if (K % 256 != 0)
        return kCfgP192;
    if (tok_e >= 80.0)
        return kCfgP192;
    const double hi = tok_e + 3.0 * std::sqrt(tok_e > 0 ? tok_e : 0.0);
    if (hi <= 32.0)
        return kCfgD32;
    if (hi <= 64.0)
        return kCfgD64;
    return kCfgD128;
}

// The reduction form keeps the fp32 token accumulators [T, H] L2-resident;
// beyond that size the per-pair store + ordered combine moves fewer bytes.
constexpr double kReduceMaxBytes = 96.0 * 1024 * 1024;

Schedule pick_schedule(double tok_e, int64_t T, int H, int I, int flags)
{
    Schedule s;
    s.cfg_gate_up = pick_cfg(tok_e, H);
    s.cfg_down = pick_cfg(tok_e, I);
    s.reduce = !(flags & CHORD_FLAG_DETERMINISTIC) &&
               static_cast<double>(T) * H * 4.0 <= kReduceMaxBytes;
    return s;
}

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
struct Workspace {
    size_t off_hdr = 0;  // int err; int num_chunks[2]
    size_t off_chunks[2] = {0, 0};
    size_t off_xs = 0;   // indexed: bf16 [capacity, H], token rows in padded-row order
    size_t off_meta = 0; // with tokens: int4 [h_rows] {pair, token, weight bits, 0} per row
    size_t off_h = 0;
    size_t off_acc = 0;       // reduce: float [T, H]; store: float [T*k, H]
    size_t off_pair_row = 0;  // store: int32 [T*k]
    size_t off_split_cnt = 0;   // int32 [2][kSplitSlots]: K-split piece counters per GEMM
    size_t off_split_part = 0;  // fp32 [2][kSplitSlots][split_maxn][128]: K-split partial sums per GEMM
    int split_maxn = 0;
    size_t total = 0;
    int64_t max_chunks = 0;
};

Workspace layout_ws(int64_t max_chunks, int64_t h_rows, int I, int64_t T, int k, int H, bool reduce,
                    bool with_tokens, int64_t xs_rows, int split_maxn)
{
    Workspace w;
    size_t o = 0;
    w.off_hdr = o;
    o += kAlign;
    w.off_split_cnt = o;
    o = align_up(o + 2 * kSplitSlots * sizeof(int32_t), kAlign);
    w.off_split_part = o;
    w.split_maxn = split_maxn;
    // (one region per GEMM: the down GEMM may start while the gate/up GEMM ends)
    o = align_up(o + 2 * static_cast<size_t>(kSplitSlots) * split_maxn * 128 * sizeof(float), kAlign);
    w.max_chunks = max_chunks;
    for (int L = 0; L < 2; ++L) {
        w.off_chunks[L] = o;
        o = align_up(o + static_cast<size_t>(max_chunks) * sizeof(Chunk), kAlign);
    }
    w.off_xs = o;
    o = align_up(o + static_cast<size_t>(xs_rows) * H * 2, kAlign);
    w.off_h = o;
    o = align_up(o + static_cast<size_t>(h_rows) * I * 2, kAlign);
    if (with_tokens) {
        w.off_meta = o;
        o = align_up(o + static_cast<size_t>(h_rows) * 16, kAlign);
        w.off_acc = o;
        if (reduce) {
            o = align_up(o + static_cast<size_t>(T) * H * 4, kAlign);
        } else {
            o = align_up(o + static_cast<size_t>(T) * k * H * 4, kAlign);
            w.off_pair_row = o;
            o = align_up(o + static_cast<size_t>(T) * k * 4, kAlign);
        }
    }
    w.total = o;
    return w;
}

int64_t indexed_max_chunks(int E_local, int64_t capacity) { return E_local + capacity / 16 + 2; }

// Token tile that sizes the K-split slots: the larger of the two GEMMs'
// tiles, or (grouped calls, whose schedule the size query does not fix) the
// largest tile of any configuration.
int split_maxn_of(const Schedule& sc)
{
    const int a = gemm_cfg_maxn(sc.cfg_gate_up), b = gemm_cfg_maxn(sc.cfg_down);
    return a > b ? a : b;
}
// Masked layout: its valid rows are copied (by prep) to a gap-free block for
// the gate/up GEMM, whose token tiles would otherwise read the rows past each
// expert's count (max_m apart, so mostly never touched before) into every box.
bool masked_compacts(int mode, int E_local) { return mode == CHORD_GROUPED_MASKED && E_local <= 1024; }

int split_maxn_any()
{
    int m = 0;
    for (int c = 0; c < kNumGemmConfigs; ++c)
        m = gemm_cfg_maxn(c) > m ? gemm_cfg_maxn(c) : m;
    return m;
}

int64_t grouped_max_chunks(int mode, int64_t M, int E_local, int64_t max_m)
{
    return mode == CHORD_GROUPED_MASKED ? E_local * ((max_m + 15) / 16) + 2 : M / 16 + 2;
}

// ---------------------------------------------------------------------------
// stage timing
// ---------------------------------------------------------------------------
std::mutex g_prof_mu;
bool g_prof_on = false;
struct ProfCall {
    cudaEvent_t ev[5];
};
std::vector<ProfCall> g_prof;

bool stream_capturing(cudaStream_t s)
{
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess)
        return true;
    return st != cudaStreamCaptureStatusNone;
}

struct StageMarks {
    ProfCall call{};
    bool on = false;
    cudaStream_t s = nullptr;
    void begin(cudaStream_t st)
    {
        s = st;
        std::lock_guard<std::mutex> lk(g_prof_mu);
        if (!g_prof_on || stream_capturing(st))
            return;
        for (auto& e : call.ev)
            if (cudaEventCreate(&e) != cudaSuccess)
                return;
        on = true;
        cudaEventRecord(call.ev[0], s);
    }
    void mark(int i)
    {
        if (on)
            cudaEventRecord(call.ev[i], s);
    }
    void end()
    {
        if (!on)
            return;
        std::lock_guard<std::mutex> lk(g_prof_mu);
        g_prof.push_back(call);
    }
};

chord_status check_ws(void* ws, size_t bytes, size_t need)
{
    if (need > 0 && (ws == nullptr || bytes < need))
        return CHORD_ERR_WORKSPACE;
    if (ws && (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0)
        return CHORD_ERR_WORKSPACE;
    return CHORD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Worker blocks of the prep kernel.  Its 1024-thread blocks fit one per SM
// and every loop in it strides over the grid, so block 0 (the chunk lists)
// and 2 x SMs - 1 workers make two whole waves.  (Measured per call, CUDA
// graph replays: against up to 2 x SMs workers, which left one block for a
// third wave, TP8 T=2048 483.7 -> 473.1 us; one wave, SMs - 1 workers, gave
// 471.1 us there but slowed the small calls, skewed decode 249.3 -> 250.5 us.)
int prep_workers(int sms) { return 2 * sms - 1; }

chord_status read_error_word(void* ws, cudaStream_t s, int* bits, bool clear)
{
    int v = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return CHORD_ERR_CUDA;
    if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return CHORD_ERR_CUDA;
    if (clear && v != 0 && cudaMemset(ws, 0, sizeof(int)) != cudaSuccess)
        return CHORD_ERR_CUDA;
    if (bits)
        *bits = v;
    if (v & CHORD_DEVERR_TIMEOUT)
        return CHORD_ERR_TIMEOUT;
    if (v & CHORD_DEVERR_ROUTING)
        return CHORD_ERR_ROUTING;
    if (v & CHORD_DEVERR_CAPACITY)
        return CHORD_ERR_CAPACITY;
    if (v & CHORD_DEVERR_SCALE_RANGE)
        return CHORD_ERR_SCALE_RANGE;
    if (v & CHORD_DEVERR_PACKED)
        return CHORD_ERR_PACKED;
    return CHORD_OK;
}

// The prep kernel checks the packs' headers against the call (gate/up: kind
// GATE_UP, N = 2I, K = H; down: kind DOWN, N = H, K = I; E >= E_local).
void set_pack_check(PrepArgs& pa, bool packed, bool mx, const int32_t* w13_q, const int32_t* w2_q,
                    int E_local, int H, int I)
{
    pa.pk_hdr[0] = packed ? reinterpret_cast<const uint32_t*>(w13_q) : nullptr;
    pa.pk_hdr[1] = packed ? reinterpret_cast<const uint32_t*>(w2_q) : nullptr;
    const uint32_t fmt = mx ? kPackFmtMxfp4 : kPackFmtInt4;
    const uint32_t want[2][5] = {
        {CHORD_PACK_GATE_UP, static_cast<uint32_t>(E_local), 2u * static_cast<uint32_t>(I),
         static_cast<uint32_t>(H), fmt},
        {CHORD_PACK_DOWN, static_cast<uint32_t>(E_local), static_cast<uint32_t>(H),
         static_cast<uint32_t>(I), fmt}};
    std::memcpy(pa.pk_want, want, sizeof want);
}

// Scales are separate arrays, or (prepacked) inside the packs and NULL here.
bool scales_given(bool packed, const uint16_t* w13_s, const uint16_t* w2_s)
{
    return packed ? (w13_s == nullptr && w2_s == nullptr) : (w13_s != nullptr && w2_s != nullptr);
}

chord_status check_shape(int H, int I, int E_local, int k)
{
    if (H <= 0 || I <= 0 || E_local <= 0 || k <= 0)
        return CHORD_ERR_INVALID_ARG;
    // (a K of 128 mod 256, hidden or intermediate, runs the 128-deep stages)
    if (H % 128 != 0 || I % 128 != 0 || k > 32)
        return CHORD_ERR_UNSUPPORTED_SHAPE;
    return CHORD_OK;
}

// The two GEMMs of one layer call, given a prepared chunk list.
struct LayerIO {
    const uint16_t* src;  // token rows in padded-row order: gathered x, or a
    int64_t src_rows;
    const int32_t* pair_of_row;
    int k;
    int64_t num_pairs;
    int H, I, E_local;
    const int32_t *w13_q, *w2_q;
    const uint16_t *w13_s, *w2_s;
    const float* topk_weights;
    const int4* row_meta;
    int64_t h_rows;
    uint16_t* h_out;  // caller-provided intermediate, or null (workspace)
    uint16_t* rows_out;
    int down_epi;
    int flags;
    double tok_e;  // expected rows per local expert
    bool h_zero_unpaired;  // h rows without a pair are written as zeros (indexed layout)
    bool packed;           // w13_q / w2_q are chord_w4a16_prepack / chord_mxfp4_prepack outputs
    bool mx;               // MXFP4 packs
};

// Weight tiles per unit of the down GEMM: with a one-stage K (I = BK) each
// unit is short, and its fixed costs (waits, commits, the token tile) are
// shared by a run of tiles of one chunk in a token-stationary configuration,
// which loads the chunk's token tile once per run.  The run is the longest
// (of 7, 4, 2 tiles, dividing the tile count) that still deals every SM six
// units or more (the units are dealt with a stride of the grid, so fewer,
// longer units leave more of the last round idle).  Measured on the TP8 down
// GEMM (H = 7168: 56 tiles): runs of 7 against 14 took 179.9 -> 176.0 us at
// 2048 tokens and 88.1 -> 86.7 us at 128; runs of 8 took 182.1 and 87.7 us,
// runs of 4 182.3 and 90.2 us;
// a rule of twelve units per SM instead of six took 16 tokens from 34.7 to
// 36.9 us.  Returns the tiles per unit and sets *cfg to the configuration
// that runs them.
int pick_tpu(int* cfg, int K, int n_tiles, int E_local, double tok_e, int sms)
{
    const int s_cfg = *cfg == kCfgD32 ? kCfgS32 : *cfg == kCfgD64 ? kCfgS64 : -1;
    if (s_cfg < 0 || K != gemm_cfg_bk(s_cfg))
        return 1;
    const double chunks = E_local * (1.0 - std::exp(-(tok_e > 0 ? tok_e : 0.0)));
    static const int runs[] = {7, 4, 2};
    for (int r : runs)
        if (r <= gemm_cfg_tpu_max_down(s_cfg) && n_tiles % r == 0 &&
            chunks * n_tiles / r >= 6.0 * sms) {
            *cfg = s_cfg;
            return r;
        }
    *cfg = s_cfg;  // one tile per unit, still with the deeper accumulator ring
    return 1;
}

chord_status run_gemms(const LayerIO& io, const Schedule& sc, const Workspace& w, uint8_t* ws,
                       int* err, int32_t* pair_row, float* acc, const DeviceInfo& dev,
                       cudaStream_t s, StageMarks& marks)
{
    uint16_t* h = io.h_out ? io.h_out : reinterpret_cast<uint16_t*>(ws + w.off_h);
    CUtensorMap map13, map2, smap13, smap2, bmap13, bmap2;
    const int bk13 = gemm_cfg_bk(sc.cfg_gate_up), bk2 = gemm_cfg_bk(sc.cfg_down);
    const int64_t rows13 = static_cast<int64_t>(io.E_local) * 2 * io.I;
    const int64_t rows2 = static_cast<int64_t>(io.E_local) * io.H;
    chord_status st = CHORD_OK;
    if (io.packed) {
        // (prepacked weights are read with plain bulk copies: no weight maps)
        std::memset(&map13, 0, sizeof map13);
        map2 = smap13 = smap2 = map13;
    } else {
        st = codes_map(io.w13_q, rows13, io.H, io.I, bk13, dev.device, &map13);
        if (st == CHORD_OK)
            st = codes_map(io.w2_q, rows2, io.I, 0, bk2, dev.device, &map2);
        // scales by TMA only for BK 256 stages; the kernel ignores the map otherwise
        smap13 = map13;
        smap2 = map2;
        if (st == CHORD_OK && bk13 == 256)
            st = scales_map(io.w13_s, rows13, io.H, io.I, dev.device, &smap13);
        if (st == CHORD_OK && bk2 == 256)
            st = scales_map(io.w2_s, rows2, io.I, 0, dev.device, &smap2);
    }
    // (a call with no rows has no chunks, so no tile is ever read through these
    // maps; one row keeps the encoding valid)
    if (st == CHORD_OK)
        st = rows_map(io.src, io.src_rows > 0 ? io.src_rows : 1, io.H,
                      gemm_cfg_maxn(sc.cfg_gate_up), bk13, dev.device, &bmap13);
    if (st == CHORD_OK)
        st = rows_map(h, io.h_rows > 0 ? io.h_rows : 1, io.I, gemm_cfg_maxn(sc.cfg_down), bk2,
                      dev.device, &bmap2);
    if (st != CHORD_OK)
        return st;
    int32_t* num_chunks = reinterpret_cast<int32_t*>(ws + w.off_hdr) + 1;

    GemmArgs g{};
    g.topk = io.k;
    g.num_pairs = static_cast<int>(io.num_pairs);
    g.K = io.H;
    g.N = 2 * io.I;
    g.I = io.I;
    g.n_tiles = io.I / 64;
    g.tpu = 1;
    g.scales = io.w13_s;
    if (io.packed)
        g.pk = reinterpret_cast<const uint8_t*>(io.w13_q) + kPackHeaderBytes;
    g.chunks = reinterpret_cast<const Chunk*>(ws + w.off_chunks[0]);
    g.num_chunks = num_chunks;
    g.epi = 0;
    g.h_out = h;
    g.ld_h = io.I;
    g.pair_row = pair_row;
    g.pair_of_row = io.pair_of_row;
    g.row_meta = io.row_meta;
    g.err = err;
    g.h_zero_unpaired = io.h_zero_unpaired ? 1 : 0;
    // K-split slots: as many as the workspace holds for this token tile, at
    // most one per CTA
    // (not for the prefill tile: summing pieces of up to 192 columns costs its
    // last round more than the split saves, 215 -> 220 us on the prefill down)
    const bool split = !(io.flags & CHORD_FLAG_NO_SPLIT_K);
    auto slots_for = [&](int cfg) {
        const int n = kSplitSlots * w.split_maxn / gemm_cfg_maxn(cfg);
        return (split && gemm_cfg_bk(cfg) == 256) ? (n < dev.sms ? n : dev.sms) : 0;
    };
    int32_t* split_cnt = reinterpret_cast<int32_t*>(ws + w.off_split_cnt);
    g.split_part = reinterpret_cast<float*>(ws + w.off_split_part);
    g.split_cnt = split_cnt;
    g.split_slots = slots_for(sc.cfg_gate_up);
    marks.mark(1);
    g.test_skip_arrive = (io.flags & CHORD_FLAG_TEST_SKIP_ARRIVE) ? 1 : 0;
    if (launch_gemm(sc.cfg_gate_up, true, io.packed, io.mx, map13, smap13, bmap13, g, dev.sms, s) !=
        cudaSuccess)
        return CHORD_ERR_CUDA;
    marks.mark(2);

    GemmArgs d = g;
    d.test_skip_arrive = 0;
    d.K = io.I;
    d.N = io.H;
    d.n_tiles = io.H / 128;
    int cfg_down = sc.cfg_down;
    d.tpu = pick_tpu(&cfg_down, io.I, d.n_tiles, io.E_local, io.tok_e, dev.sms);
    d.scales = io.w2_s;
    d.pk = io.packed ? reinterpret_cast<const uint8_t*>(io.w2_q) + kPackHeaderBytes : nullptr;
    d.chunks = reinterpret_cast<const Chunk*>(ws + w.off_chunks[1]);
    d.num_chunks = num_chunks + 1;
    d.epi = io.down_epi;
    d.h_out = nullptr;
    d.pair_row = nullptr;
    d.y_pairs = (io.down_epi & kEpiStorePair) ? acc : nullptr;
    d.out_acc = (io.down_epi & kEpiReduceTok) ? acc : nullptr;
    d.rows_out = io.rows_out;
    d.split_cnt = split_cnt + kSplitSlots;
    d.split_part = g.split_part + static_cast<size_t>(kSplitSlots) * w.split_maxn * 128;
    d.split_slots = slots_for(sc.cfg_down);
    if (launch_gemm(cfg_down, false, io.packed, io.mx, map2, smap2, bmap2, d, dev.sms, s) != cudaSuccess)
        return CHORD_ERR_CUDA;
    marks.mark(3);
    return CHORD_OK;
}

chord_status prepack_common(int kind, const int32_t* w_q, const void* w_s, int fmt, int E, int N,
                            int K, void* packed, size_t packed_bytes, void* stream)
{
    if ((kind != CHORD_PACK_GATE_UP && kind != CHORD_PACK_DOWN) || E < 1 || N < 1 || K < 1)
        return CHORD_ERR_INVALID_ARG;
    if (N % 128 != 0 || K % 128 != 0)
        return CHORD_ERR_UNSUPPORTED_SHAPE;
    if (!w_q || !w_s || !packed || !aligned16(w_q) || !aligned16(w_s) || !aligned16(packed))
        return CHORD_ERR_INVALID_ARG;
    if (packed_bytes < chord_w4a16_prepack_size(kind, E, N, K))
        return CHORD_ERR_INVALID_ARG;
    DeviceInfo dev;
    chord_status st = device_info(&dev);
    if (st != CHORD_OK)
        return st;
    PackArgs a{};
    a.kind = kind;
    a.q = w_q;
    a.E = E;
    a.N = N;
    a.K = K;
    a.out = static_cast<uint8_t*>(packed);
    a.fmt = fmt;
    if (fmt == static_cast<int>(kPackFmtMxfp4))
        a.sc8 = static_cast<const uint8_t*>(w_s);
    else
        a.sc = static_cast<const uint16_t*>(w_s);
    return from_cuda(launch_prepack(a, dev.sms, static_cast<cudaStream_t>(stream)));
}

}  // namespace
}  // namespace chord

using namespace chord;

extern "C" {

const char* chord_status_string(int status)
{
    switch (status) {
    case CHORD_OK: return "ok";
    case CHORD_ERR_INVALID_ARG: return "invalid argument";
    case CHORD_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case CHORD_ERR_CAPACITY: return "routing capacity too small";
    case CHORD_ERR_LAYOUT_MODE: return "layout mode mismatch";
    case CHORD_ERR_CUDA: return "CUDA error";
    case CHORD_ERR_TIMEOUT: return "device wait timed out";
    case CHORD_ERR_ROUTING: return "invalid routing data";
    case CHORD_ERR_SCALE_RANGE: return "scale outside the supported range";
    case CHORD_ERR_PACKED: return "packed weights do not match the call";
    case CHORD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case CHORD_ERR_NO_DEVICE: return "no sm_103a device current";
    default: return "unknown status";
    }
}

int chord_version(void) { return 100; }

int64_t chord_moe_align_capacity(int64_t T, int k, int E_local, int block_m)
{
    if (block_m <= 0 || T < 0 || k <= 0 || E_local <= 0)
        return -1;
    const int64_t worst = T * k + static_cast<int64_t>(E_local) * (block_m - 1);
    return (worst + block_m - 1) / block_m * block_m;
}

int chord_select_block_m(int64_t, int, int, int, int, int) { return 16; }

int chord_describe_schedule(int64_t T, int k, int E_global, int E_local, int H, int I, int flags,
                            char* buf, size_t buf_len)
{
    const double tok_e = E_global > 0 ? static_cast<double>(T) * k / E_global : 0.0;
    const Schedule s = pick_schedule(tok_e, T, H, I, flags);
    static const char* names[] = {"decode-tile32", "decode-tile64", "decode-tile128",
                                  "prefill-tile192", "short-k-tile32", "short-k-tile64"};
    // the down GEMM's weight tiles per unit depend on the SM count: with a
    // device, the configuration and run a call on it would launch
    int cfg_down = s.cfg_down;
    int tpu = 0;
    DeviceInfo dev;
    if (H % 128 == 0 && device_info(&dev) == CHORD_OK)
        tpu = pick_tpu(&cfg_down, I, H / 128, E_local, tok_e, dev.sms);
    char run[32] = "";
    if (tpu > 1)
        snprintf(run, sizeof run, "x%d-tiles-per-unit", tpu);
    char tmp[256];
    const int n = snprintf(tmp, sizeof tmp,
                           "tok_e=%.2f gate_up=%s(BK%d) down=%s%s(BK%d) combine=%s block_m=16 "
                           "E_local=%d",
                           tok_e, names[s.cfg_gate_up], gemm_cfg_bk(s.cfg_gate_up),
                           names[cfg_down], run, gemm_cfg_bk(cfg_down),
                           s.reduce ? "fp32-reduce" : "ordered-pairs", E_local);
    if (buf && buf_len) {
        strncpy(buf, tmp, buf_len - 1);
        buf[buf_len - 1] = 0;
    }
    return n;
}

size_t chord_moe_align_workspace_size(int64_t T, int k, int E_local)
{
    const int64_t pairs = T * k;
    const int64_t tiles = (pairs + 255) / 256;
    return align_up(kAlign + static_cast<size_t>(tiles > 0 ? tiles : 1) * E_local * 4, kAlign);
}

size_t chord_w4a16_moe_workspace_size(int64_t T, int k, int E_global, int E_local, int H, int I,
                                      int block_m, int64_t capacity, int flags)
{
    if (T < 0 || k <= 0 || E_local <= 0 || H <= 0 || I <= 0 || block_m <= 0 || capacity < 0)
        return 0;
    const double tok_e = E_global > 0 ? static_cast<double>(T) * k / E_global : 0.0;
    const Schedule s = pick_schedule(tok_e, T, H, I, flags);
    return layout_ws(indexed_max_chunks(E_local, capacity), capacity, I, T, k, H, s.reduce, true,
                     capacity, split_maxn_of(s))
        .total;
}

size_t chord_w4a16_grouped_workspace_size(int mode, int64_t M, int H, int I, int E_local, int64_t T,
                                          int k, int with_tokens, int expected_m)
{
    (void)expected_m;
    if (M < 0 || H <= 0 || I <= 0 || E_local <= 0)
        return 0;
    const int64_t max_m = mode == CHORD_GROUPED_MASKED ? M / E_local : 0;
    return layout_ws(grouped_max_chunks(mode, M, E_local, max_m), M, I, T, k, H, true,
                     with_tokens != 0, masked_compacts(mode, E_local) ? M : 0, split_maxn_any())
        .total;
}

chord_status chord_moe_align(const int32_t* topk_ids, int64_t T, int k, int E_global,
                             const int32_t* expert_map, int E_local, int block_m,
                             int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_tokens_padded,
                             int64_t capacity, void* workspace, size_t workspace_bytes, void* stream)
{
    if (T < 0 || k < 1 || k > 32 || E_global < 1 || E_local < 1 || E_local > 1024 || block_m < 1 ||
        block_m > 256)
        return CHORD_ERR_INVALID_ARG;
    if (!expert_map && E_local != E_global)
        return CHORD_ERR_INVALID_ARG;
    if (T * k >= (int64_t(1) << 31))
        return CHORD_ERR_UNSUPPORTED_SHAPE;
    if (capacity < chord_moe_align_capacity(T, k, E_local, block_m) || capacity % block_m != 0)
        return CHORD_ERR_CAPACITY;
    if (!sorted_ids || !expert_ids || !num_tokens_padded || (T > 0 && !topk_ids))
        return CHORD_ERR_INVALID_ARG;
    chord_status st =
        check_ws(workspace, workspace_bytes, chord_moe_align_workspace_size(T, k, E_local));
    if (st != CHORD_OK)
        return st;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != CHORD_OK)
        return st;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
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
    a.tile_hist = reinterpret_cast<int32_t*>(ws + kAlign);
    a.n_tiles = static_cast<int>((T * k + 255) / 256);
    a.err = reinterpret_cast<int*>(ws);
    PdlScope pdl(T * k <= kPdlMaxRows);
    return from_cuda(launch_align(a, static_cast<cudaStream_t>(stream)));
}

chord_status chord_moe_route_align(const float* logits, int64_t T, int E_global, int k,
                                   int renormalize, const int32_t* expert_map, int E_local,
                                   int block_m, int32_t* topk_ids, float* topk_weights,
                                   int32_t* sorted_ids, int32_t* expert_ids,
                                   int32_t* num_tokens_padded, int64_t capacity, void* workspace,
                                   size_t workspace_bytes, void* stream)
{
    if (T < 0 || k < 1 || k > 32 || E_global < 1 || k > E_global || E_local < 1 ||
        E_local > 1024 || block_m < 1 || block_m > 256)
        return CHORD_ERR_INVALID_ARG;
    if (E_global > 1024)
        return CHORD_ERR_UNSUPPORTED_SHAPE;
    if (!expert_map && E_local != E_global)
        return CHORD_ERR_INVALID_ARG;
    if (T * k >= (int64_t(1) << 31) || T * E_global >= (int64_t(1) << 40))
        return CHORD_ERR_UNSUPPORTED_SHAPE;
    if (!sorted_ids || !expert_ids || !num_tokens_padded ||
        (T > 0 && (!logits || !topk_ids || !topk_weights)))
        return CHORD_ERR_INVALID_ARG;
    if (capacity < chord_moe_align_capacity(T, k, E_local, block_m) || capacity % block_m != 0)
        return CHORD_ERR_CAPACITY;
    chord_status st =
        check_ws(workspace, workspace_bytes, chord_moe_align_workspace_size(T, k, E_local));
    if (st != CHORD_OK)
        return st;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != CHORD_OK)
        return st;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    RouteArgs r{};
    r.logits = logits;
    r.T = T;
    r.E = E_global;
    r.k = k;
    r.renorm = renormalize ? 1 : 0;
    r.ids = topk_ids;
    r.w = topk_weights;
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
    a.tile_hist = reinterpret_cast<int32_t*>(ws + kAlign);
    a.n_tiles = static_cast<int>((T * k + 255) / 256);
    a.err = reinterpret_cast<int*>(ws);
    PdlScope pdl(T * k <= kPdlMaxRows);
    return from_cuda(launch_route_align(r, a, static_cast<cudaStream_t>(stream)));
}

size_t chord_w4a16_prepack_size(int kind, int E, int N, int K)
{
    if ((kind != CHORD_PACK_GATE_UP && kind != CHORD_PACK_DOWN) || E < 1 || N < 128 || K < 128 ||
        N % 128 != 0 || K % 128 != 0)
        return 0;
    return kPackHeaderBytes + static_cast<size_t>(E) * (N / 128) * pack_kblocks(K) * kPackBlockBytes;
}


chord_status chord_mxfp4_prepack(int kind, const int32_t* w_q, const uint8_t* w_e8m0, int E, int N,
                                 int K, void* packed, size_t packed_bytes, void* stream)
{
    return prepack_common(kind, w_q, w_e8m0, static_cast<int>(kPackFmtMxfp4), E, N, K, packed,
                          packed_bytes, stream);
}

chord_status chord_w4a16_prepack(int kind, const int32_t* w_q, const uint16_t* w_s, int E, int N,
                                 int K, void* packed, size_t packed_bytes, void* stream)
{
    return prepack_common(kind, w_q, w_s, static_cast<int>(kPackFmtInt4), E, N, K, packed,
                          packed_bytes, stream);
}

chord_status chord_w4a16_moe_indexed(const uint16_t* x, int64_t T, int H, int I, int E_global,
                                     int E_local, int k, const int32_t* w13_q,
                                     const uint16_t* w13_s, const int32_t* w2_q,
                                     const uint16_t* w2_s, const float* topk_weights,
                                     const int32_t* sorted_ids, const int32_t* expert_ids,
                                     const int32_t* num_tokens_padded, int64_t capacity,
                                     int block_m, void* workspace, size_t workspace_bytes,
                                     uint16_t* out, uint16_t* h_out, int flags, void* stream)
{
    chord_status st = check_shape(H, I, E_local, k);
    if (st != CHORD_OK)
        return st;
    if (T < 0 || E_global < 1 || block_m < 1 || block_m > 256 || (flags & ~63))
        return CHORD_ERR_INVALID_ARG;
    const bool packed = (flags & CHORD_FLAG_PREPACKED) != 0;
    const bool mx = (flags & CHORD_FLAG_MXFP4) != 0;
    if (mx && !packed)
        return CHORD_ERR_INVALID_ARG;
    if (T * k >= (int64_t(1) << 31))
        return CHORD_ERR_UNSUPPORTED_SHAPE;
    if (T == 0)
        return CHORD_OK;
    // (every size check comes before the pointers are looked at)
    if (capacity < chord_moe_align_capacity(T, k, E_local, block_m) || capacity % block_m != 0)
        return CHORD_ERR_CAPACITY;
    if (!x || !w13_q || !w2_q || !topk_weights || !sorted_ids || !expert_ids ||
        !num_tokens_padded || !out || !scales_given(packed, w13_s, w2_s))
        return CHORD_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w13_q) || !aligned16(w13_s) || !aligned16(w2_q) ||
        !aligned16(w2_s) || !aligned16(out) || (h_out && !aligned16(h_out)))
        return CHORD_ERR_INVALID_ARG;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != CHORD_OK)
        return st;
    const double tok_e = static_cast<double>(T) * k / E_global;
    const Schedule sc = pick_schedule(tok_e, T, H, I, flags);
    const Workspace w = layout_ws(indexed_max_chunks(E_local, capacity), capacity, I, T, k, H,
                                  sc.reduce, true, capacity, split_maxn_of(sc));
    if ((st = check_ws(workspace, workspace_bytes, w.total)) != CHORD_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* err = reinterpret_cast<int*>(ws + w.off_hdr);
    float* acc = reinterpret_cast<float*>(ws + w.off_acc);
    int32_t* pair_row = sc.reduce ? nullptr : reinterpret_cast<int32_t*>(ws + w.off_pair_row);

    PdlScope pdl(T * k <= kPdlMaxRows);
    StageMarks marks;
    marks.begin(s);
    PrepArgs pa{};
    pa.layout = kLayoutIndexed;
    pa.expert_ids = expert_ids;
    pa.num_tokens_padded = num_tokens_padded;
    pa.capacity = capacity;
    pa.block_rows = block_m;
    pa.E_local = E_local;
    pa.maxn[0] = gemm_cfg_maxn(sc.cfg_gate_up);
    pa.maxn[1] = gemm_cfg_maxn(sc.cfg_down);
    pa.chunks[0] = reinterpret_cast<Chunk*>(ws + w.off_chunks[0]);
    pa.chunks[1] = reinterpret_cast<Chunk*>(ws + w.off_chunks[1]);
    pa.max_chunks = static_cast<int>(w.max_chunks);
    pa.num_chunks = err + 1;
    pa.zero_i32 = reinterpret_cast<int32_t*>(ws + w.off_split_cnt);
    pa.zero_i32_count = 2 * kSplitSlots;
    if (sc.reduce) {
        pa.zero_f32 = acc;
        pa.zero_count = T * H;
    } else {
        pa.fill_i32 = pair_row;
        pa.fill_count = T * k;
    }
    uint16_t* xs = reinterpret_cast<uint16_t*>(ws + w.off_xs);
    int4* meta = reinterpret_cast<int4*>(ws + w.off_meta);
    pa.meta_out = meta;
    pa.meta_pair = sorted_ids;
    pa.meta_w = topk_weights;
    pa.meta_topk = k;
    pa.meta_pairs = T * k;
    pa.meta_rows = -1;
    pa.gx_src = x;
    pa.gx_out = xs;
    // compact the gathered rows when the layout's padding rows (about
    // (block_m - 1) / 2 per touched expert) would otherwise put more than
    // 16 MB of never-written rows into the token boxes (below that, the
    // compaction scans cost prep more than the GEMM gains)
    {
        const double touched = E_local * (1.0 - std::exp(-tok_e));
        const double pad_bytes = touched * (block_m - 1) * 0.5 * H * 2.0;
        pa.gx_compact = (E_local <= 1024 && pad_bytes >= 16.0 * 1024 * 1024) ? 1 : 0;
    }
    pa.gx_ids = sorted_ids;
    pa.gx_topk = k;
    pa.gx_pairs = T * k;
    pa.gx_H = H;
    pa.err = err;
    set_pack_check(pa, packed, mx, w13_q, w2_q, E_local, H, I);
    const int work_blocks = prep_workers(dev.sms);
    if (launch_prep(pa, work_blocks, s) != cudaSuccess)
        return CHORD_ERR_CUDA;
    // (prepacked weights: the pack recorded its scales' range; the GEMMs report it)
    if ((flags & CHORD_FLAG_VALIDATE) && !packed &&
        launch_scale_check(w13_s, static_cast<int64_t>(E_local) * 2 * I * (H / 32), w2_s,
                           static_cast<int64_t>(E_local) * H * (I / 32), err, dev.sms, s) !=
            cudaSuccess)
        return CHORD_ERR_CUDA;

    LayerIO io{};
    io.src = xs;
    io.src_rows = capacity;
    io.pair_of_row = sorted_ids;
    io.row_meta = meta;
    io.k = k;
    io.num_pairs = T * k;
    io.H = H;
    io.I = I;
    io.E_local = E_local;
    io.w13_q = w13_q;
    io.w13_s = w13_s;
    io.w2_q = w2_q;
    io.w2_s = w2_s;
    io.topk_weights = topk_weights;
    io.h_rows = capacity;
    io.h_out = h_out;
    io.down_epi = sc.reduce ? kEpiReduceTok : kEpiStorePair;
    io.flags = flags;
    io.packed = packed;
    io.mx = mx;
    io.tok_e = tok_e;
    io.h_zero_unpaired = true;
    if ((st = run_gemms(io, sc, w, ws, err, pair_row, acc, dev, s, marks)) != CHORD_OK)
        return st;

    cudaError_t e;
    if (sc.reduce) {
        e = launch_finalize(acc, out, T * H, dev.sms, s);
    } else {
        const CombineArgs ca{T, k, H, pair_row, topk_weights, acc, out};
        e = launch_combine_pairs(ca, s);
    }
    if (e != cudaSuccess)
        return CHORD_ERR_CUDA;
    marks.mark(4);
    marks.end();
    if (flags & CHORD_FLAG_VALIDATE)
        return read_error_word(ws + w.off_hdr, s, nullptr, false);
    return CHORD_OK;
}

chord_status chord_w4a16_moe_grouped(int mode, const uint16_t* a, int64_t M, int H, int I,
                                     int E_local, const int32_t* m_indices,
                                     const int32_t* masked_m, int64_t max_m, int expected_m,
                                     const int32_t* w13_q, const uint16_t* w13_s,
                                     const int32_t* w2_q, const uint16_t* w2_s,
                                     const int32_t* row_to_pair, const float* topk_weights,
                                     int64_t T, int k, void* workspace, size_t workspace_bytes,
                                     uint16_t* out_rows, uint16_t* out_tokens, uint16_t* h_out,
                                     int flags, void* stream)
{
    const bool with_tokens = out_tokens != nullptr;
    chord_status st = check_shape(H, I, E_local, with_tokens ? k : 1);
    if (st != CHORD_OK)
        return st;
    if (M < 0 || (flags & ~63))
        return CHORD_ERR_INVALID_ARG;
    const bool packed = (flags & CHORD_FLAG_PREPACKED) != 0;
    const bool mx = (flags & CHORD_FLAG_MXFP4) != 0;
    if (mx && !packed)
        return CHORD_ERR_INVALID_ARG;
    if (mode == CHORD_GROUPED_CONTIGUOUS) {
        if (masked_m != nullptr || (M > 0 && m_indices == nullptr))
            return CHORD_ERR_LAYOUT_MODE;
        if (M % 16 != 0)
            return CHORD_ERR_UNSUPPORTED_SHAPE;
    } else if (mode == CHORD_GROUPED_MASKED) {
        if (m_indices != nullptr || masked_m == nullptr)
            return CHORD_ERR_LAYOUT_MODE;
        if (max_m < 1 || expected_m < 1 || M != E_local * max_m)
            return CHORD_ERR_INVALID_ARG;
    } else {
        return CHORD_ERR_LAYOUT_MODE;
    }
    if (M >= (int64_t(1) << 31))
        return CHORD_ERR_UNSUPPORTED_SHAPE;
    if (with_tokens) {
        if (!row_to_pair || !topk_weights || T < 0 || k < 1 || T * k >= (int64_t(1) << 31))
            return CHORD_ERR_INVALID_ARG;
    }
    if (M == 0 && !with_tokens)
        return CHORD_OK;
    if (!a || !w13_q || !w2_q || !out_rows || !scales_given(packed, w13_s, w2_s))
        return CHORD_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(w13_q) || !aligned16(w13_s) || !aligned16(w2_q) ||
        !aligned16(w2_s) || !aligned16(out_rows) || (out_tokens && !aligned16(out_tokens)) ||
        (h_out && !aligned16(h_out)))
        return CHORD_ERR_INVALID_ARG;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != CHORD_OK)
        return st;
    const double tok_e = mode == CHORD_GROUPED_MASKED ? static_cast<double>(expected_m)
                                                      : static_cast<double>(M) / E_local;
    Schedule sc = pick_schedule(tok_e, T, H, I, 0);
    sc.reduce = true;
    const bool compact = masked_compacts(mode, E_local);
    const Workspace w = layout_ws(grouped_max_chunks(mode, M, E_local, max_m), M, I, T, k, H, true,
                                  with_tokens, compact ? M : 0, split_maxn_any());
    if ((st = check_ws(workspace, workspace_bytes, w.total)) != CHORD_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* err = reinterpret_cast<int*>(ws + w.off_hdr);
    float* acc = with_tokens ? reinterpret_cast<float*>(ws + w.off_acc) : nullptr;

    PdlScope pdl((with_tokens ? T * k : M) <= kPdlMaxRows);
    StageMarks marks;
    marks.begin(s);
    PrepArgs pa{};
    pa.layout = mode == CHORD_GROUPED_MASKED ? kLayoutMasked : kLayoutContiguous;
    pa.block_rows = 16;
    pa.m_indices = m_indices;
    pa.M = M;
    pa.masked_m = masked_m;
    pa.max_m = max_m;
    pa.E_local = E_local;
    pa.maxn[0] = gemm_cfg_maxn(sc.cfg_gate_up);
    pa.maxn[1] = gemm_cfg_maxn(sc.cfg_down);
    pa.chunks[0] = reinterpret_cast<Chunk*>(ws + w.off_chunks[0]);
    pa.chunks[1] = reinterpret_cast<Chunk*>(ws + w.off_chunks[1]);
    pa.max_chunks = static_cast<int>(w.max_chunks);
    pa.num_chunks = err + 1;
    pa.zero_i32 = reinterpret_cast<int32_t*>(ws + w.off_split_cnt);
    pa.zero_i32_count = 2 * kSplitSlots;
    if (with_tokens) {
        pa.zero_f32 = acc;
        pa.zero_count = T * H;
        pa.meta_out = reinterpret_cast<int4*>(ws + w.off_meta);
        pa.meta_pair = row_to_pair;
        pa.meta_w = topk_weights;
        pa.meta_topk = k;
        pa.meta_pairs = T * k;
        pa.meta_rows = M;
    }
    uint16_t* xs = compact ? reinterpret_cast<uint16_t*>(ws + w.off_xs) : nullptr;
    if (compact) {
        pa.mc_src = a;
        pa.mc_out = xs;
        pa.mc_H = H;
    }
    pa.err = err;
    set_pack_check(pa, packed, mx, w13_q, w2_q, E_local, H, I);
    // (the row records and the compacted rows come from the worker blocks)
    const int work_blocks = (with_tokens || compact) ? prep_workers(dev.sms) : 0;
    if (launch_prep(pa, work_blocks, s) != cudaSuccess)
        return CHORD_ERR_CUDA;
    // (prepacked weights: the pack recorded its scales' range; the GEMMs report it)
    if ((flags & CHORD_FLAG_VALIDATE) && !packed &&
        launch_scale_check(w13_s, static_cast<int64_t>(E_local) * 2 * I * (H / 32), w2_s,
                           static_cast<int64_t>(E_local) * H * (I / 32), err, dev.sms, s) !=
            cudaSuccess)
        return CHORD_ERR_CUDA;

    LayerIO io{};
    io.src = compact ? xs : a;
    io.src_rows = M;
    io.row_meta = with_tokens ? reinterpret_cast<const int4*>(ws + w.off_meta) : nullptr;
    io.pair_of_row = with_tokens ? row_to_pair : nullptr;
    io.k = with_tokens ? k : 1;
    io.num_pairs = with_tokens ? T * k : 0;
    io.H = H;
    io.I = I;
    io.E_local = E_local;
    io.w13_q = w13_q;
    io.w13_s = w13_s;
    io.w2_q = w2_q;
    io.w2_s = w2_s;
    io.topk_weights = topk_weights;
    io.h_rows = M;
    io.h_out = h_out;
    io.rows_out = out_rows;
    io.down_epi = kEpiStoreRows | (with_tokens ? kEpiReduceTok : 0);
    io.flags = flags;
    io.packed = packed;
    io.mx = mx;
    io.tok_e = tok_e;
    if ((st = run_gemms(io, sc, w, ws, err, nullptr, acc, dev, s, marks)) != CHORD_OK)
        return st;
    if (with_tokens && launch_finalize(acc, out_tokens, T * H, dev.sms, s) != cudaSuccess)
        return CHORD_ERR_CUDA;
    marks.mark(4);
    marks.end();
    if (flags & CHORD_FLAG_VALIDATE)
        return read_error_word(ws + w.off_hdr, s, nullptr, false);
    return CHORD_OK;
}

chord_status chord_get_device_error(void* workspace, int* error_bits, int clear, void* stream)
{
    if (!workspace)
        return CHORD_ERR_INVALID_ARG;
    return read_error_word(workspace, static_cast<cudaStream_t>(stream), error_bits, clear != 0);
}

chord_status chord_stage_timing_enable(int enable)
{
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_on = enable != 0;
    for (auto& c : g_prof)
        for (auto& e : c.ev)
            cudaEventDestroy(e);
    g_prof.clear();
    return CHORD_OK;
}

chord_status chord_stage_timing_read(float* ms_per_stage, int* calls)
{
    std::lock_guard<std::mutex> lk(g_prof_mu);
    float sum[4] = {0, 0, 0, 0};
    for (auto& c : g_prof) {
        if (cudaEventSynchronize(c.ev[4]) != cudaSuccess)
            return CHORD_ERR_CUDA;
        for (int i = 0; i < 4; ++i) {
            float ms = 0;
            if (cudaEventElapsedTime(&ms, c.ev[i], c.ev[i + 1]) != cudaSuccess)
                return CHORD_ERR_CUDA;
            sum[i] += ms;
        }
    }
    if (ms_per_stage)
        for (int i = 0; i < 4; ++i)
            ms_per_stage[i] = sum[i];
    if (calls)
        *calls = static_cast<int>(g_prof.size());
    return CHORD_OK;
}

}  // extern "C"
