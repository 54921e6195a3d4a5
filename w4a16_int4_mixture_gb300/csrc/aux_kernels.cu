// aux_kernels.cu -- routing alignment, per-call preparation and the top-k combine.
//
// moe_align (page: "Two kernel families" / "vLLM integration": the indexed
// family consumes moe_align_block_size's sorted_ids / expert_ids /
// num_tokens_padded; Fig. 3: the padding lives in the index as a sentinel).
// Deterministic, three launches, no atomics on the output positions:
//   1. align_hist:    per 256-pair tile, a histogram of local experts;
//   2. align_scan:    one CTA: padded segment offsets, ntp, expert_ids, per-tile
//                     bases, sentinel fill of sorted_ids;
//   3. align_scatter: per tile, the stable rank of each pair among the pairs of
//                     its expert (warp match + per-warp counts) -> sorted_ids.
#include <cuda_runtime.h>

#include "device.cuh"
#include "kernels.h"

namespace chord {

constexpr int kAlignTile = 256;

__device__ __forceinline__ int local_expert_of(int32_t gid, int E_global, const int32_t* expert_map,
                                               int E_local, int* err)
{
    if (gid < 0 || gid >= E_global) {
        raise_error(err, CHORD_DEVERR_ROUTING);
        return -1;
    }
    const int l = expert_map ? expert_map[gid] : gid;
    return (l >= 0 && l < E_local) ? l : -1;
}

__global__ void __launch_bounds__(kAlignTile) align_hist_kernel(AlignArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ int cnt[];  // [E_local]
    for (int e = threadIdx.x; e < a.E_local; e += blockDim.x)
        cnt[e] = 0;
    __syncthreads();
    const int64_t p = static_cast<int64_t>(blockIdx.x) * kAlignTile + threadIdx.x;
    if (p < a.num_pairs) {
        const int l = local_expert_of(a.topk_ids[p], a.E_global, a.expert_map, a.E_local, nullptr);
        if (l >= 0)
            atomicAdd(&cnt[l], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < a.E_local; e += blockDim.x)
        a.tile_hist[static_cast<int64_t>(blockIdx.x) * a.E_local + e] = cnt[e];
}

// block-wide exclusive scan of one int per thread (blockDim.x a multiple of 32)
__device__ int block_exclusive_scan(int v, int* total)
{
    __shared__ int warp_sums[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < static_cast<int>(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        warp_sums[lane] = w;  // inclusive
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
    *total = warp_sums[(blockDim.x >> 5) - 1];
    __syncthreads();
    return before;
}

// One CTA.  Each local expert (E_local <= 1024) gets tpe threads (a power of
// two, tpe * E_local <= 1024), thread j of expert e taking a contiguous range
// of tiles; threads j * E_local + e are adjacent in e, so every load of the
// per-tile histogram is coalesced.  Pass 1 sums each range, pass 2 rewrites
// the histogram in place as the first padded row of each (tile, expert).
__global__ void __launch_bounds__(1024) align_scan_kernel(AlignArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int part[1024];
    __shared__ int offs[1024];
    const int sentinel = static_cast<int>(a.num_pairs);
    const int bm = a.block_m;
    const int E = a.E_local;
    // this call's error word starts clear (the scatter reports bad ids after us)
    if (threadIdx.x == 0)
        *a.err = 0;
    // sentinel everywhere first; the scatter overwrites the real entries
    for (int64_t i = threadIdx.x; i < a.capacity; i += blockDim.x)
        a.sorted_ids[i] = sentinel;
    int tpe = 1;
    while (tpe < 32 && 2 * tpe * E <= static_cast<int>(blockDim.x))
        tpe *= 2;
    const bool act = static_cast<int>(threadIdx.x) < tpe * E;
    const int e = act ? static_cast<int>(threadIdx.x) % E : 0;
    const int j = act ? static_cast<int>(threadIdx.x) / E : 0;
    const int n_tiles = a.n_tiles;
    const int per = (n_tiles + tpe - 1) / tpe;
    const int t0 = j * per;
    const int t1 = t0 + per < n_tiles ? t0 + per : n_tiles;
    int32_t* h = a.tile_hist;
    int sum = 0;
    if (act) {
#pragma unroll 8
        for (int t = t0; t < t1; ++t)
            sum += h[static_cast<int64_t>(t) * E + e];
    }
    part[threadIdx.x] = sum;
    __syncthreads();
    int before = 0, count = 0;
    if (act)
        for (int jj = 0; jj < tpe; ++jj) {
            const int v = part[jj * E + e];
            before += jj < j ? v : 0;
            count += v;
        }
    // padded rows per expert, scanned over the threads j = 0 (threads 0 .. E-1, in expert order)
    const int padded = (act && j == 0) ? (count + bm - 1) / bm * bm : 0;
    int ntp;
    const int off = block_exclusive_scan(padded, &ntp);
    if (act && j == 0)
        offs[e] = off;
    __syncthreads();
    if (act) {
        int run = offs[e] + before;
#pragma unroll 8
        for (int t = t0; t < t1; ++t) {
            const int64_t i = static_cast<int64_t>(t) * E + e;
            const int c = h[i];
            h[i] = run;
            run += c;
        }
    }
    if (act && j == 0 && off + padded <= a.capacity)
        for (int b = off / bm; b < (off + padded) / bm; ++b)
            a.expert_ids[b] = e;
    if (ntp > a.capacity && threadIdx.x == 0)
        raise_error(a.err, CHORD_DEVERR_CAPACITY);
    const int64_t nblocks = a.capacity / bm;
    for (int64_t b = ntp / bm + threadIdx.x; b < nblocks; b += blockDim.x)
        a.expert_ids[b] = -1;
    if (threadIdx.x == 0)
        a.num_tokens_padded[0] = ntp <= a.capacity ? ntp : 0;
}

__global__ void __launch_bounds__(kAlignTile) align_scatter_kernel(AlignArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ int wcnt[];  // [kAlignTile/32][E_local]
    constexpr int W = kAlignTile / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < W * a.E_local; i += blockDim.x)
        wcnt[i] = 0;
    __syncthreads();
    const int64_t p = static_cast<int64_t>(blockIdx.x) * kAlignTile + threadIdx.x;
    int l = -1;
    if (p < a.num_pairs)
        l = local_expert_of(a.topk_ids[p], a.E_global, a.expert_map, a.E_local, a.err);
    // pairs of the same expert inside this warp, and my rank among them
    const unsigned peers = __match_any_sync(0xffffffffu, l);
    const unsigned lower = peers & ((1u << lane) - 1u);
    const int rank_in_warp = __popc(lower);
    if (l >= 0 && lower == 0)
        wcnt[warp * a.E_local + l] = __popc(peers);
    __syncthreads();
    if (l >= 0) {
        int rank = rank_in_warp;
        for (int w = 0; w < warp; ++w)
            rank += wcnt[w * a.E_local + l];
        const int64_t pos = a.tile_hist[static_cast<int64_t>(blockIdx.x) * a.E_local + l] + rank;
        if (pos < a.capacity)
            a.sorted_ids[pos] = static_cast<int32_t>(p);
    }
}

// The whole align in one CTA for routing batches of up to 4096 pairs (the
// three kernels above cost three launches and a single-CTA scan in between).
// The sentinel goes over the whole capacity first (coalesced; the pairs
// overwrite their rows after the barriers).  Warp w takes a contiguous range
// of pairs and ranks them in rounds of 32 on its own: warp match for the
// pairs of one expert inside a round, plus a per-warp running count of each
// expert in shared memory.  One block barrier, then each expert's counts are
// scanned over the warps (so warp w's pairs of expert e come after those of
// warps 0 .. w-1), the padded segments over the experts, and every pair lands
// at segment base + warp prefix + rank.  Same output as the three kernels,
// bit for bit.  (With more pairs one CTA's scattered row writes cost more
// than the three kernels: at 16384 pairs over 384 experts, 31 against 12 us.)
constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallMaxPairs = 4096;
constexpr int kSmallMaxExperts = 512;

// The one-CTA align (called by every thread of a 1024-thread block), for at
// most R rounds of 32 pairs per warp (R * kSmallThreads pairs).
template <int R>
__device__ void align_small_run(const AlignArgs& a)
{
    // pairs of each expert in each warp's range (a running count while the
    // warp ranks its pairs), then the pairs of that expert in earlier warps;
    // both are at most kSmallMaxPairs
    __shared__ short wcnt[kSmallWarps][kSmallMaxExperts];
    __shared__ int base[kSmallMaxExperts];  // first padded row of each expert
    const int E = a.E_local;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int npairs = static_cast<int>(a.num_pairs);
    const int sentinel = npairs;
    const int bm = a.block_m;
    const int64_t cap = a.capacity;
    if (threadIdx.x == 0)
        *a.err = 0;
    for (int i = threadIdx.x; i < kSmallWarps * kSmallMaxExperts / 2; i += blockDim.x)
        reinterpret_cast<int*>(&wcnt[0][0])[i] = 0;
    // pairs per warp: a multiple of 32, at most 32 R
    const int per_warp = (npairs + kSmallThreads - 1) / kSmallThreads * 32;
    const int rounds = per_warp / 32;
    const int p0 = warp * per_warp + lane;
    // per round: the pair's id, then its local expert (-1: none), then the
    // expert and the pair's rank among this warp's pairs of it (l << 16 | rank;
    // both below 2^9), or -1.  The loads go out before the barrier; a bad id
    // is reported after it, once the error word has been cleared.
    int rec[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
        rec[r] = (r < rounds && p0 + 32 * r < npairs) ? a.topk_ids[p0 + 32 * r] : -1;
    for (int64_t i = threadIdx.x; i < cap; i += blockDim.x)
        a.sorted_ids[i] = sentinel;
    bool bad = false;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const bool have = r < rounds && p0 + 32 * r < npairs;
        bad |= have && (rec[r] < 0 || rec[r] >= a.E_global);
        rec[r] = have ? local_expert_of(rec[r], a.E_global, a.expert_map, E, nullptr) : -1;
    }
    __syncthreads();
    if (bad)
        raise_error(a.err, CHORD_DEVERR_ROUTING);
    const unsigned below = (1u << lane) - 1u;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (r < rounds) {
            const int l = rec[r];
            const unsigned peers = __match_any_sync(0xffffffffu, l);
            const int before = l >= 0 ? wcnt[warp][l] : 0;
            __syncwarp();
            if (l >= 0) {
                rec[r] = (l << 16) | (before + __popc(peers & below));
                if ((peers & below) == 0)
                    wcnt[warp][l] = static_cast<short>(before + __popc(peers));
            }
            __syncwarp();
        }
    }
    __syncthreads();
    // per expert: the warp counts become the counts of earlier warps (the
    // loads eight at a time ahead of the stores)
    const int e = threadIdx.x;
    int total = 0;
    if (e < E) {
#pragma unroll
        for (int h = 0; h < kSmallWarps; h += 8) {
            int c[8];
#pragma unroll
            for (int w = 0; w < 8; ++w)
                c[w] = wcnt[h + w][e];
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                wcnt[h + w][e] = static_cast<short>(total);
                total += c[w];
            }
        }
    }
    const int padded = e < E ? (total + bm - 1) / bm * bm : 0;
    int ntp;
    const int off = block_exclusive_scan(padded, &ntp);
    if (e < E) {
        base[e] = off;
        if (off + padded <= cap)
            for (int b = off / bm; b < (off + padded) / bm; ++b)
                a.expert_ids[b] = e;
    }
    if (ntp > cap && threadIdx.x == 0)
        raise_error(a.err, CHORD_DEVERR_CAPACITY);
    const int64_t nblocks = cap / bm;
    for (int64_t b = ntp / bm + threadIdx.x; b < nblocks; b += blockDim.x)
        a.expert_ids[b] = -1;
    if (threadIdx.x == 0)
        a.num_tokens_padded[0] = ntp <= cap ? ntp : 0;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (r < rounds && rec[r] >= 0) {
            const int l = rec[r] >> 16;
            const int64_t pos = static_cast<int64_t>(base[l]) + wcnt[warp][l] + (rec[r] & 0xffff);
            if (pos < cap)
                a.sorted_ids[pos] = p0 + 32 * r;
        }
    }
}

__global__ void __launch_bounds__(kSmallThreads) align_small_kernel(AlignArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    align_small_run<kSmallMaxPairs / kSmallThreads>(a);
}

// ---------------------------------------------------------------------------
// router: per token the k largest logits (ties to the lower expert id), in
// descending order, each weighted by its softmax probability over all experts,
// renormalised over the k when asked.  One warp per token: lane l holds logits
// l, l + 32, ...; k rounds of a warp argmax over (logit, lower id).
// ---------------------------------------------------------------------------
// NI logits per lane: E <= 32 * NI (NI = 4, 8, 16 or 32).
template <int NI>
__device__ void route_token_warp(const RouteArgs& r, int64_t t, int lane)
{
    const int E = r.E;
    const float* row = r.logits + t * E;
    float v[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? row[e] : -INFINITY;
    }
    uint32_t taken = 0u;  // bit i: logit lane + 32 i already chosen
    float top = 0.f;      // the largest logit (the first one chosen)
    int my_id = -1;       // lane j keeps the j-th choice
    float my_v = 0.f;
    for (int j = 0; j < r.k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && (bi == 0x7fffffff || v[i] > bv)) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane)
            taken |= 1u << (bi >> 5);
        if (j == 0)
            top = bv;
        if (lane == j) {
            my_id = bi;
            my_v = bv;
        }
    }
    // denominators: over the chosen k, or over every expert
    float den = 0.f;
    if (r.renorm) {
        den = lane < r.k ? expf(my_v - top) : 0.f;
    } else {
#pragma unroll
        for (int i = 0; i < NI; ++i)
            if (lane + 32 * i < E)
                den += expf(v[i] - top);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        den += __shfl_xor_sync(0xffffffffu, den, o);
    if (lane < r.k) {
        r.ids[t * r.k + lane] = my_id;
        r.w[t * r.k + lane] = expf(my_v - top) / den;
    }
}

template <int NI>
__global__ void __launch_bounds__(256) route_topk_kernel(RouteArgs r)
{
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t t = warp; t < r.T; t += nwarps)
        route_token_warp<NI>(r, t, lane);
}

// Router and align in one CTA (up to 64 tokens and 512 local experts): the 32 warps route the tokens into topk_ids / topk_weights, then
// the block aligns them.
constexpr int kRouteFusedMaxT = 64;

template <int NI>
__global__ void __launch_bounds__(kSmallThreads) route_align_small_kernel(RouteArgs r, AlignArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t t = warp; t < r.T; t += kSmallThreads / 32)
        route_token_warp<NI>(r, t, lane);
    __syncthreads();  // (the block's writes of topk_ids are visible to it)
    align_small_run<kRouteFusedMaxT * 32 / kSmallThreads>(a);
}

template <int NI>
cudaError_t launch_route_align_ni(const RouteArgs& r, const AlignArgs& a, cudaStream_t s)
{
    // (k <= 32: at most kRouteFusedMaxT * 32 pairs, the rounds the fused kernel takes)
    if (r.T <= kRouteFusedMaxT && a.num_pairs <= kRouteFusedMaxT * 32 && a.E_local <= kSmallMaxExperts)
        return launch_pdl(route_align_small_kernel<NI>, 1, kSmallThreads, 0, s, r, a);
    if (r.T > 0) {
        int64_t blocks = (r.T + 7) / 8;  // 8 warps per block, a token each
        if (blocks > 65535)
            blocks = 65535;
        cudaError_t e = launch_pdl(route_topk_kernel<NI>, static_cast<int>(blocks), 256, 0, s, r);
        if (e != cudaSuccess)
            return e;
    }
    return launch_align(a, s);
}

cudaError_t launch_route_align(const RouteArgs& r, const AlignArgs& a, cudaStream_t s)
{
    if (r.E <= 128)
        return launch_route_align_ni<4>(r, a, s);
    if (r.E <= 256)
        return launch_route_align_ni<8>(r, a, s);
    if (r.E <= 512)
        return launch_route_align_ni<16>(r, a, s);
    return launch_route_align_ni<32>(r, a, s);
}

cudaError_t launch_align(const AlignArgs& a, cudaStream_t s)
{
    if (a.num_pairs <= kSmallMaxPairs && a.E_local <= kSmallMaxExperts) {
        return launch_pdl(align_small_kernel, 1, kSmallThreads, 0, s, a);
    }
    const int tiles = a.n_tiles;
    if (tiles > 0) {
        cudaError_t e = launch_pdl(align_hist_kernel, tiles, kAlignTile, a.E_local * sizeof(int), s, a);
        if (e != cudaSuccess)
            return e;
    }
    cudaError_t e = launch_pdl(align_scan_kernel, 1, 1024, 0, s, a);
    if (e != cudaSuccess || tiles == 0)
        return e;
    return launch_pdl(align_scatter_kernel, tiles, kAlignTile, (kAlignTile / 32) * a.E_local * sizeof(int), s, a);
}

// ---------------------------------------------------------------------------
// per-call preparation: chunk lists for the GEMMs, zeroed / initialised buffers
// and (indexed layout) the routed token rows gathered into padded-row order
// ---------------------------------------------------------------------------
__device__ __forceinline__ int chunks_for(int rows, int maxn) { return (rows + maxn - 1) / maxn; }

// Splits a segment of `rows` rows starting at row0 into chunks of at most maxn
// rows (balanced, each but the last a multiple of 16).  False when the list
// would overflow (only reachable with a malformed layout).
__device__ bool emit_chunks(Chunk* out, int slot, int row0, int rows, int expert, int maxn,
                            int max_chunks, int* err, int brow_base)
{
    const int n = chunks_for(rows, maxn);
    if (slot + n > max_chunks) {
        raise_error(err, CHORD_DEVERR_ROUTING);
        return false;
    }
    int cs = (rows + n - 1) / n;
    cs = (cs + 15) & ~15;
    if (cs > maxn)
        cs = maxn;
    for (int c = 0, r = 0; c < n; ++c, r += cs) {
        Chunk ch;
        ch.row0 = row0 + r;
        ch.nrows = min(cs, rows - r);
        ch.expert = expert;
        ch.brow0 = brow_base + r;
        out[slot + c] = ch;
    }
    return true;
}

// expert of block b (block_m rows indexed, 16 rows contiguous): -1 for padding
// or an invalid id, -2 outside [0, nblocks)
__device__ __forceinline__ int block_expert(const PrepArgs& a, int b, int nblocks)
{
    if (b < 0 || b >= nblocks)
        return -2;
    if (a.layout == kLayoutIndexed) {
        const int e = a.expert_ids[b];
        if (e < 0 || e >= a.E_local) {
            raise_error(a.err, CHORD_DEVERR_ROUTING);
            return -1;
        }
        return e;
    }
    const int e = a.m_indices[static_cast<int64_t>(b) * a.block_rows];
    return (e >= 0 && e < a.E_local) ? e : -1;
}

// Indexed layout, compacted token rows: the rows of each expert's segment
// that hold a pair come first (the layout pads each segment at its end), so
// padded row r of expert e holds compacted row coff[e] + (r - seg[e]), where
// seg[e] is the segment's first row and coff[e] the pairs of the experts
// before it.  Needs E_local <= blockDim.x; every thread of the block calls it.
struct CompactIdx {
    int* seg;   // [E_local] first padded row, or -1
    int* coff;  // [E_local] first compacted row
    int total;  // compacted rows
};
// 16-byte global load / store under an L2 cache policy (createpolicy)
__device__ __forceinline__ uint4 ld16_hint(const uint4* p, uint64_t policy)
{
    uint4 v;
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}
__device__ __forceinline__ void st16_hint(uint4* p, uint4 v, uint64_t policy)
{
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
                 : "memory");
}

__device__ CompactIdx indexed_compaction(const PrepArgs& a)
{
    __shared__ int s_seg[1024];
    __shared__ int s_end[1024];
    __shared__ int s_coff[1024];
    const int E = a.E_local;
    const int bm = a.block_rows;
    const int ntp = a.num_tokens_padded[0];
    const int nblocks = (ntp >= 0 && ntp <= a.capacity) ? ntp / bm : 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        s_seg[e] = -1;
        s_end[e] = -1;
    }
    __syncthreads();
    for (int b = threadIdx.x; b < nblocks; b += blockDim.x) {
        const int e = a.expert_ids[b];
        if (e < 0 || e >= E)
            continue;
        const int prev = b > 0 ? a.expert_ids[b - 1] : -1;
        const int next = b + 1 < nblocks ? a.expert_ids[b + 1] : -1;
        if (prev != e)
            s_seg[e] = b * bm;
        if (next != e) {
            int v = 0;  // rows of the segment's last block that hold a pair
            const int32_t* ids = a.gx_ids + static_cast<int64_t>(b) * bm;
            for (int i0 = 0; i0 < bm; i0 += 16) {
                int p[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    p[i] = i0 + i < bm ? ids[i0 + i] : -1;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v += (p[i] >= 0 && p[i] < a.gx_pairs) ? 1 : 0;
            }
            s_end[e] = b * bm + v;
        }
    }
    __syncthreads();
    const int e = threadIdx.x;
    int cnt = 0;
    if (e < E && s_seg[e] >= 0 && s_end[e] >= s_seg[e])
        cnt = s_end[e] - s_seg[e];
    int total;
    const int off = block_exclusive_scan(cnt, &total);
    if (e < E)
        s_coff[e] = off;
    __syncthreads();
    return CompactIdx{s_seg, s_coff, total};
}

__device__ __forceinline__ int end_block_of(int b, int rows, int bm) { return b + rows / bm; }

__device__ void build_chunk_lists(const PrepArgs& a)
{
    __shared__ int s_off[2];
    __shared__ int s_bad;
    if (threadIdx.x == 0) {
        s_off[0] = 0;
        s_off[1] = 0;
        s_bad = 0;
        *a.err = 0;  // this call's error word starts clear
    }
    __syncthreads();
    if (a.layout == kLayoutMasked) {
        __shared__ int s_roff;  // compacted rows of the experts before this slice
        if (threadIdx.x == 0)
            s_roff = 0;
        __syncthreads();
        for (int e0 = 0; e0 < a.E_local; e0 += blockDim.x) {
            const int e = e0 + threadIdx.x;
            int rows = 0;
            if (e < a.E_local) {
                rows = a.masked_m[e];
                if (rows < 0 || rows > a.max_m) {
                    raise_error(a.err, CHORD_DEVERR_ROUTING);
                    rows = rows < 0 ? 0 : static_cast<int>(a.max_m);
                }
            }
            int rtotal;
            const int roff = s_roff + block_exclusive_scan(rows, &rtotal);
            for (int L = 0; L < 2; ++L) {
                const int n = rows > 0 ? chunks_for(rows, a.maxn[L]) : 0;
                int total;
                const int off = s_off[L] + block_exclusive_scan(n, &total);
                const int row0 = static_cast<int>(e * a.max_m);
                const int brow = (L == 0 && a.mc_out != nullptr) ? roff : row0;
                if (n > 0 && !emit_chunks(a.chunks[L], off, row0, rows, e, a.maxn[L], a.max_chunks,
                                          a.err, brow))
                    s_bad = 1;
                __syncthreads();
                if (threadIdx.x == 0)
                    s_off[L] += total;
                __syncthreads();
            }
            if (threadIdx.x == 0)
                s_roff += rtotal;
            __syncthreads();
        }
    } else {
        int nblocks;
        if (a.layout == kLayoutIndexed) {
            const int ntp = a.num_tokens_padded[0];
            nblocks = (ntp >= 0 && ntp <= a.capacity) ? ntp / a.block_rows : 0;
        } else {
            nblocks = static_cast<int>(a.M / a.block_rows);
        }
        // compacted token rows of the gate/up GEMM (indexed layout): each run's
        // paired rows counted from its last block, scanned like the chunks
        const bool compact = a.layout == kLayoutIndexed && a.gx_compact;
        __shared__ int s_roff;
        if (threadIdx.x == 0)
            s_roff = 0;
        // the experts of this tile of blocks (plus one on each side) in shared
        // memory, read with one coalesced pass; a run that leaves the staged
        // tile continues with direct reads
        __shared__ int s_e[1024 + 2];
        const int staged = static_cast<int>(blockDim.x) + 2;
        for (int b0 = 0; b0 < nblocks; b0 += blockDim.x) {
            for (int i = threadIdx.x; i < staged; i += blockDim.x)
                s_e[i] = block_expert(a, b0 - 1 + i, nblocks);
            __syncthreads();
            const int b = b0 + threadIdx.x;
            int rows = 0, e = -1;
            if (b < nblocks) {
                e = s_e[threadIdx.x + 1];
                if (e >= 0 && s_e[threadIdx.x] != e) {
                    int end = b + 1;
                    int li = threadIdx.x + 2;
                    while (end < nblocks && li < staged && s_e[li] == e) {
                        ++end;
                        ++li;
                    }
                    if (li == staged)
                        while (end < nblocks && block_expert(a, end, nblocks) == e)
                            ++end;
                    rows = (end - b) * a.block_rows;
                }
            }
            int paired = 0;
            if (compact && rows > 0) {
                const int bm = a.block_rows;
                const int32_t* ids = a.gx_ids + static_cast<int64_t>(end_block_of(b, rows, bm) - 1) * bm;
                int v = 0;
                for (int i0 = 0; i0 < bm; i0 += 16) {
                    int p[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        p[i] = i0 + i < bm ? ids[i0 + i] : -1;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        v += (p[i] >= 0 && p[i] < a.gx_pairs) ? 1 : 0;
                }
                paired = rows - bm + v;
            }
            int rtotal = 0;
            const int roff = compact ? s_roff + block_exclusive_scan(paired, &rtotal) : 0;
            for (int L = 0; L < 2; ++L) {
                const int n = rows > 0 ? chunks_for(rows, a.maxn[L]) : 0;
                int total;
                const int off = s_off[L] + block_exclusive_scan(n, &total);
                const int brow = (L == 0 && compact) ? roff : b * a.block_rows;
                if (n > 0 && !emit_chunks(a.chunks[L], off, b * a.block_rows, rows, e, a.maxn[L],
                                          a.max_chunks, a.err, brow))
                    s_bad = 1;
                __syncthreads();
                if (threadIdx.x == 0)
                    s_off[L] += total;
                __syncthreads();
            }
            if (compact) {
                if (threadIdx.x == 0)
                    s_roff += rtotal;
                __syncthreads();
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // prepacked weights whose header does not describe this call: no GEMM
        // unit may read them
        bool pk_bad = false;
        for (int g = 0; g < 2; ++g) {
            const uint32_t* h = a.pk_hdr[g];
            if (h == nullptr)
                continue;
            const uint32_t* w = a.pk_want[g];
            if (h[0] != kPackMagic || h[1] != 1u || h[2] != w[0] || h[3] < w[1] || h[4] != w[2] ||
                h[5] != w[3] || h[6] != static_cast<uint32_t>(kPackBlockBytes) ||
                h[kPackFormatWord] != w[4])
                pk_bad = true;
            else if (h[7] & 1u)
                raise_error(a.err, CHORD_DEVERR_SCALE_RANGE);
        }
        if (pk_bad)
            raise_error(a.err, CHORD_DEVERR_PACKED);
        // a malformed layout that overflows the list runs nothing rather than
        // reading entries this call did not write
        a.num_chunks[0] = (s_bad || pk_bad) ? 0 : s_off[0];
        a.num_chunks[1] = (s_bad || pk_bad) ? 0 : s_off[1];
    }
}

__global__ void __launch_bounds__(1024) prep_kernel(PrepArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i < a.zero_i32_count; i += blockDim.x)
            a.zero_i32[i] = 0;
        build_chunk_lists(a);
        return;
    }
    const int64_t tid = static_cast<int64_t>(blockIdx.x - 1) * blockDim.x + threadIdx.x;
    const int64_t nth = static_cast<int64_t>(gridDim.x - 1) * blockDim.x;
    if (a.mc_out != nullptr) {
        // the experts' first compacted rows (the same scan as the chunk lists),
        // then 128 threads per compacted row
        __shared__ int s_mcoff[1025];
        const int E = a.E_local;  // <= 1024 (the host compacts only then)
        int rows = 0;
        if (static_cast<int>(threadIdx.x) < E) {
            rows = a.masked_m[threadIdx.x];
            rows = rows < 0 ? 0 : (rows > a.max_m ? static_cast<int>(a.max_m) : rows);
        }
        int total;
        const int off = block_exclusive_scan(rows, &total);
        if (static_cast<int>(threadIdx.x) < E)
            s_mcoff[threadIdx.x] = off;
        if (threadIdx.x == 0)
            s_mcoff[E] = total;
        __syncthreads();
        constexpr int kGroup = 128;
        const int gl = static_cast<int>(tid % kGroup);
        const int64_t ngrp = nth / kGroup;
        const int n16 = a.mc_H / 8;
        for (int64_t i = tid / kGroup; i < total; i += ngrp) {
            // expert of compacted row i: the last e with s_mcoff[e] <= i
            int lo = 0, hi = E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_mcoff[mid] <= i)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            const int64_t srow = static_cast<int64_t>(lo) * a.max_m + (i - s_mcoff[lo]);
            const uint4* src = reinterpret_cast<const uint4*>(a.mc_src + srow * a.mc_H);
            uint4* dst = reinterpret_cast<uint4*>(a.mc_out + i * a.mc_H);
            for (int c0 = gl; c0 < n16; c0 += 8 * kGroup) {
                uint4 v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int c = c0 + j * kGroup;
                    v[j] = c < n16 ? src[c] : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int c = c0 + j * kGroup;
                    if (c < n16)
                        dst[c] = v[j];
                }
            }
        }
    }
    if (a.zero_f32 != nullptr) {
        float4* z = reinterpret_cast<float4*>(a.zero_f32);
        const int64_t n4 = a.zero_count / 4;
        for (int64_t i = tid; i < n4; i += nth)
            z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int64_t i = n4 * 4 + tid; i < a.zero_count; i += nth)
            a.zero_f32[i] = 0.f;
    }
    if (a.fill_i32 != nullptr)
        for (int64_t i = tid; i < a.fill_count; i += nth)
            a.fill_i32[i] = -1;
    if (a.meta_out != nullptr && a.gx_out == nullptr) {
        // (with a gather, the gather loop below writes the records)
        int64_t rows = a.meta_rows;
        if (rows < 0) {
            const int ntp = a.num_tokens_padded[0];
            rows = (ntp >= 0 && ntp <= a.capacity) ? ntp : 0;
        }
        for (int64_t r = tid; r < rows; r += nth) {
            const int p = a.meta_pair[r];
            int4 m = make_int4(-1, 0, 0, 0);
            if (p >= 0 && p < a.meta_pairs)
                m = make_int4(p, p / a.meta_topk, __float_as_int(a.meta_w[p]), 0);
            a.meta_out[r] = m;
        }
    }
    if (a.gx_out != nullptr) {
        // 128 threads per padded row, up to 8 16-byte loads in flight per
        // thread before the stores.  Rows with no pair (the block padding of
        // the layout) are not written: they only feed MMA columns that no
        // output reads, and the gate/up epilogue writes zeros for their h rows.
        // Compacted: row r of expert e goes to coff[e] + (r - seg[e]), so no
        // token box reads a padding row; then the row records come from a
        // loop of their own (one thread per padded row) and the copies walk
        // the compacted rows, so no copy group waits on a padding row.
        constexpr int kGroup = 128;
        const int gl = static_cast<int>(tid % kGroup);
        const int64_t ngrp = nth / kGroup;
        const int ntp = a.num_tokens_padded[0];
        const int64_t rows = (ntp >= 0 && ntp <= a.capacity) ? ntp : 0;
        const int n16 = a.gx_H / 8;
        // Each token row is copied once per local slot (up to k times), far
        // apart in the walk: the source rows are read with an L2 evict-last
        // policy and the gathered rows written evict-first, so that the copies
        // stream through L2 without pushing x out of it (measured at TP8
        // T=2048, k = 8: without the policies 22 % of the copy's L2 reads hit).
        const uint64_t keep = policy_evict_last();
        const uint64_t pass = policy_evict_first();
        auto copy_row = [&](int p, int64_t drow) {
            const uint4* src = reinterpret_cast<const uint4*>(a.gx_src + static_cast<int64_t>(p / a.gx_topk) * a.gx_H);
            uint4* dst = reinterpret_cast<uint4*>(a.gx_out + drow * a.gx_H);
            for (int c0 = gl; c0 < n16; c0 += 8 * kGroup) {
                uint4 v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int c = c0 + j * kGroup;
                    v[j] = c < n16 ? ld16_hint(src + c, keep) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int c = c0 + j * kGroup;
                    if (c < n16)
                        st16_hint(dst + c, v[j], pass);
                }
            }
        };
        if (a.gx_compact) {
            const CompactIdx cx = indexed_compaction(a);
            if (a.meta_out != nullptr)
                for (int64_t r = tid; r < rows; r += nth) {
                    const int p = a.gx_ids[r];
                    const bool valid = p >= 0 && p < a.gx_pairs;
                    a.meta_out[r] = valid ? make_int4(p, p / a.gx_topk, __float_as_int(a.meta_w[p]), 0)
                                          : make_int4(-1, 0, 0, 0);
                }
            const int E = a.E_local;
            for (int64_t cc = tid / kGroup; cc < cx.total; cc += ngrp) {
                const int64_t c = cx.total - 1 - cc;  // (last to first, as below)
                // expert of compacted row c: the last e with a segment and coff[e] <= c
                int lo = 0, hi = E - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (cx.coff[mid] <= c)
                        lo = mid;
                    else
                        hi = mid - 1;
                }
                while (lo > 0 && cx.seg[lo] < 0)
                    --lo;  // (experts without rows share the offset of the next one)
                if (cx.seg[lo] < 0)
                    continue;
                const int64_t r = cx.seg[lo] + (c - cx.coff[lo]);
                if (r >= rows)
                    continue;
                const int p = a.gx_ids[r];
                if (p >= 0 && p < a.gx_pairs)
                    copy_row(p, c);
            }
            return;
        }
        // (rows are copied last to first: the gate/up GEMM starts on the first
        // experts' rows, which are then the ones most recently written and
        // still in L2)
        for (int64_t rr = tid / kGroup; rr < rows; rr += ngrp) {
            const int64_t r = rows - 1 - rr;
            const int p = a.gx_ids[r];
            const bool valid = p >= 0 && p < a.gx_pairs;  // sentinel rows become zeros
            if (gl == 0 && a.meta_out != nullptr)
                a.meta_out[r] = valid ? make_int4(p, p / a.gx_topk, __float_as_int(a.meta_w[p]), 0)
                                      : make_int4(-1, 0, 0, 0);
            if (valid)
                copy_row(p, r);
        }
    }
}

// CHORD_FLAG_VALIDATE: every scale is +-0 or has magnitude in [2^-86, 2^35)
// (bf16 exponent field 41..161), the range in which the GEMMs' scaled weights
// are exact; anything else sets CHORD_DEVERR_SCALE_RANGE.
__device__ __forceinline__ bool scale_in_range(uint32_t bits16)
{
    const uint32_t mag = bits16 & 0x7FFFu;
    const uint32_t e = mag >> 7;
    return mag == 0 || (e >= 41 && e <= 161);
}

__global__ void scale_range_kernel(const uint16_t* __restrict__ a, int64_t na,
                                   const uint16_t* __restrict__ b, int64_t nb, int* err)
{
    pdl_launch_dependents();
    pdl_wait();
    bool ok = true;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < na + nb;
         i += stride) {
        const uint32_t v = i < na ? a[i] : b[i - na];
        ok = ok && scale_in_range(v);
    }
    if (!ok)
        raise_error(err, CHORD_DEVERR_SCALE_RANGE);
}

cudaError_t launch_scale_check(const uint16_t* a, int64_t na, const uint16_t* b, int64_t nb,
                               int* err, int sms, cudaStream_t s)
{
    if (na + nb <= 0)
        return cudaSuccess;
    return launch_pdl(scale_range_kernel, 4 * sms, 256, 0, s, a, na, b, nb, err);
}

// ---------------------------------------------------------------------------
// offline prepack (format in chord.h)
// ---------------------------------------------------------------------------
__global__ void pack_header_kernel(PackArgs a)
{
    uint32_t* hd = reinterpret_cast<uint32_t*>(a.out);
    const int i = threadIdx.x;  // 64 threads: the 64 header words
    uint32_t v = 0;
    if (i == 0)
        v = kPackMagic;
    else if (i == 1)
        v = 1;
    else if (i == 2)
        v = static_cast<uint32_t>(a.kind);
    else if (i == 3)
        v = static_cast<uint32_t>(a.E);
    else if (i == 4)
        v = static_cast<uint32_t>(a.N);
    else if (i == 5)
        v = static_cast<uint32_t>(a.K);
    else if (i == 6)
        v = kPackBlockBytes;
    else if (i == kPackFormatWord)
        v = static_cast<uint32_t>(a.fmt);
    hd[i] = v;  // word 7 (flags) starts at 0
}

// One thread per 16-byte piece of the output: pieces 0..1023 of a block are
// codes (half h = j / 512, tile row r, stored position pos of the row's four
// pieces, holding source piece pos ^ ((r >> 1) & 3)), 1024..1151 the rows'
// scales.  Consecutive threads write consecutive pieces.
__global__ void __launch_bounds__(256) pack_kernel(PackArgs a)
{
    const int tiles = a.N / 128;
    const int kbs = pack_kblocks(a.K);  // the last block is half past K when K % 256 == 128
    const int64_t words_per_row = a.K / 8;
    const int64_t scales_per_row = a.K / 32;
    const int64_t total = static_cast<int64_t>(a.E) * tiles * kbs * 1152;
    uint8_t* blocks = a.out + kPackHeaderBytes;
    uint32_t* flags = reinterpret_cast<uint32_t*>(a.out) + 7;
    bool ok = true;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = i / 1152;
        const int j = static_cast<int>(i - b * 1152);
        const int kb = static_cast<int>(b % kbs);
        const int t = static_cast<int>((b / kbs) % tiles);
        const int64_t e = b / (static_cast<int64_t>(kbs) * tiles);
        const int r = j < 1024 ? (j >> 2) & 127 : j - 1024;
        const int row = a.kind == CHORD_PACK_GATE_UP ? (r < 64 ? 64 * t + r : a.N / 2 + 64 * t + r - 64)
                                                     : 128 * t + r;
        const int64_t grow = e * a.N + row;
        // the second half of the last block lies past K when K % 256 == 128: zeros
        const bool tail = kb == kbs - 1 && (a.K & 255) != 0;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (j < 1024) {
            const int h = j >> 9;
            const int c = (j & 3) ^ ((r >> 1) & 3);
            if (!(tail && h == 1))
                v = *reinterpret_cast<const uint4*>(a.q + grow * words_per_row + kb * 32 + h * 16 + c * 4);
        } else if (a.fmt == static_cast<int>(kPackFmtMxfp4)) {
            // E8M0 byte e -> the bf16 value 2^(e - 127): exponent field e for
            // 1 <= e <= 254, the subnormal 0x0040 for e = 0, NaN for e = 255.
            // (4-byte reads: a row of K / 32 scale bytes is a multiple of 4.)
            const uint32_t* src8 = reinterpret_cast<const uint32_t*>(a.sc8 + grow * scales_per_row + kb * 8);
            const uint32_t b8[2] = {src8[0], tail ? 0u : src8[1]};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t src = b8[q >> 1];
                uint32_t h[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint32_t e = (src >> (16 * (q & 1) + 8 * u)) & 0xFFu;
                    h[u] = e == 0u ? 0x0040u : (e == 255u ? 0x7FC0u : e << 7);
                }
                o[q] = h[0] | (h[1] << 16);
            }
            v = make_uint4(o[0], o[1], tail ? 0u : o[2], tail ? 0u : o[3]);
        } else {
            // (8-byte reads: a row of K / 32 bf16 scales is a multiple of 8 bytes)
            const uint2* src = reinterpret_cast<const uint2*>(a.sc + grow * scales_per_row + kb * 8);
            const uint2 lo = src[0];
            const uint2 hi = tail ? make_uint2(0u, 0u) : src[1];
            v = make_uint4(lo.x, lo.y, hi.x, hi.y);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
                ok = ok && scale_in_range(w[q] & 0xFFFFu) && scale_in_range(w[q] >> 16);
        }
        *reinterpret_cast<uint4*>(blocks + b * kPackBlockBytes + static_cast<int64_t>(j) * 16) = v;
    }
    if (!ok)
        atomicOr(flags, 1u);
}

cudaError_t launch_prepack(const PackArgs& a, int sms, cudaStream_t s)
{
    pack_header_kernel<<<1, 64, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    pack_kernel<<<8 * sms, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_prep(const PrepArgs& a, int work_blocks, cudaStream_t s)
{
    return launch_pdl(prep_kernel, 1 + work_blocks, 1024, 0, s, a);
}

// ---------------------------------------------------------------------------
// combine
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

// out[i] = bf16(acc[i]) for the fp32 token accumulators of the reduction form.
// (four 8-element groups per thread and step, all loads before the stores)
constexpr int kFinUnroll = 4;

__global__ void finalize_kernel(const float* __restrict__ acc, uint16_t* __restrict__ out, int64_t n)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t n8 = n / 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const float4* a4 = reinterpret_cast<const float4*>(acc);
    uint4* o4 = reinterpret_cast<uint4*>(out);
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n8;
         i0 += kFinUnroll * stride) {
        float4 a[kFinUnroll], b[kFinUnroll];
#pragma unroll
        for (int u = 0; u < kFinUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < n8) {
                a[u] = a4[2 * i];
                b[u] = a4[2 * i + 1];
            }
        }
#pragma unroll
        for (int u = 0; u < kFinUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < n8) {
                uint4 o;
                o.x = pack_bf16x2(a[u].x, a[u].y);
                o.y = pack_bf16x2(a[u].z, a[u].w);
                o.z = pack_bf16x2(b[u].x, b[u].y);
                o.w = pack_bf16x2(b[u].z, b[u].w);
                o4[i] = o;
            }
        }
    }
    for (int64_t i = n8 * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride)
        out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[i]));
}

// Ordered top-k combine of per-pair fp32 outputs.  One block per token
// (grid-stride): the token's local slots are compacted once into shared memory
// in ascending slot order, then each thread produces 8 output columns as
// sum_j w_j * y_j over those slots in that order, so the result is
// bit-identical run to run.  A token with no local slot gets zeros.
constexpr int kCombineThreads = 128;
constexpr int kCombineGroups = 4;  // 8-column groups per thread in flight

__global__ void __launch_bounds__(kCombineThreads) combine_pairs_kernel(CombineArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int64_t s_pair[32];
    __shared__ float s_w[32];
    __shared__ int s_n;
    const int H8 = a.H / 8;
    for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        if (threadIdx.x < 32) {
            const int j = threadIdx.x;
            const int64_t p = t * a.k + j;
            const bool valid = j < a.k && a.pair_row[p] >= 0;
            const uint32_t m = __ballot_sync(0xffffffffu, valid);
            if (valid) {
                const int idx = __popc(m & ((1u << j) - 1u));
                s_pair[idx] = p;
                s_w[idx] = a.topk_weights[p];
            }
            if (j == 0)
                s_n = __popc(m);
        }
        __syncthreads();
        const int n = s_n;
        // kCombineGroups column groups per thread at a time, each slot's loads
        // for all of them issued together (a token has about one local slot at
        // EP8 prefill: one group's two loads per thread kept too few bytes in
        // flight); the sum per column is still over the slots in ascending order
        for (int c0 = threadIdx.x; c0 < H8; c0 += kCombineGroups * blockDim.x) {
            float acc[kCombineGroups][8];
#pragma unroll
            for (int u = 0; u < kCombineGroups; ++u)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[u][e] = 0.f;
            for (int i = 0; i < n; ++i) {
                const float4* y = reinterpret_cast<const float4*>(a.y_pairs + s_pair[i] * a.H);
                const float w = s_w[i];
                float4 y0[kCombineGroups], y1[kCombineGroups];
#pragma unroll
                for (int u = 0; u < kCombineGroups; ++u) {
                    const int c = c0 + u * blockDim.x;
                    if (c < H8) {
                        y0[u] = y[2 * c];
                        y1[u] = y[2 * c + 1];
                    }
                }
#pragma unroll
                for (int u = 0; u < kCombineGroups; ++u) {
                    if (c0 + u * blockDim.x < H8) {
                        acc[u][0] += w * y0[u].x;
                        acc[u][1] += w * y0[u].y;
                        acc[u][2] += w * y0[u].z;
                        acc[u][3] += w * y0[u].w;
                        acc[u][4] += w * y1[u].x;
                        acc[u][5] += w * y1[u].y;
                        acc[u][6] += w * y1[u].z;
                        acc[u][7] += w * y1[u].w;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kCombineGroups; ++u) {
                const int c = c0 + u * blockDim.x;
                if (c < H8) {
                    uint4 o;
                    o.x = pack_bf16x2(acc[u][0], acc[u][1]);
                    o.y = pack_bf16x2(acc[u][2], acc[u][3]);
                    o.z = pack_bf16x2(acc[u][4], acc[u][5]);
                    o.w = pack_bf16x2(acc[u][6], acc[u][7]);
                    reinterpret_cast<uint4*>(a.out + t * a.H)[c] = o;
                }
            }
        }
        __syncthreads();
    }
}

cudaError_t launch_finalize(const float* acc, uint16_t* out, int64_t n, int sms, cudaStream_t s)
{
    if (n <= 0)
        return cudaSuccess;
    int64_t blocks = (n / 8 + 256 * kFinUnroll - 1) / (256 * kFinUnroll);
    if (blocks < 1)
        blocks = 1;
    if (blocks > 4LL * sms)
        blocks = 4LL * sms;
    return launch_pdl(finalize_kernel, static_cast<int>(blocks), 256, 0, s, acc, out, n);
}

// The same combine for fewer tokens: a block takes one token's slots over
// kCombineThreads x G column groups (several blocks per token), and each
// thread issues the loads of G groups x S slots together before it sums them
// in ascending slot order (the same operations, in the same order, as
// combine_pairs_kernel).  With one block per token, a token's eight slots cost
// eight dependent round trips per column group: 12 us at one token.
template <int G, int S>
__global__ void __launch_bounds__(kCombineThreads) combine_pairs_split_kernel(CombineArgs a, int splits)
{
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int64_t s_pair[32];
    __shared__ float s_w[32];
    __shared__ int s_n;
    const int H8 = a.H / 8;
    const int64_t items = a.T * splits;
    for (int64_t b = blockIdx.x; b < items; b += gridDim.x) {
        const int64_t t = b / splits;
        const int c0 = static_cast<int>(b % splits) * kCombineThreads * G + threadIdx.x;
        if (threadIdx.x < 32) {
            const int j = threadIdx.x;
            const int64_t p = t * a.k + j;
            const bool valid = j < a.k && a.pair_row[p] >= 0;
            const uint32_t m = __ballot_sync(0xffffffffu, valid);
            if (valid) {
                const int idx = __popc(m & ((1u << j) - 1u));
                s_pair[idx] = p;
                s_w[idx] = a.topk_weights[p];
            }
            if (j == 0)
                s_n = __popc(m);
        }
        __syncthreads();
        const int n = s_n;
        float acc[G][8];
#pragma unroll
        for (int u = 0; u < G; ++u)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[u][e] = 0.f;
        for (int i0 = 0; i0 < n; i0 += S) {
            float4 y0[G][S], y1[G][S];
#pragma unroll
            for (int v = 0; v < S; ++v) {
                if (i0 + v < n) {
                    const float4* y = reinterpret_cast<const float4*>(a.y_pairs + s_pair[i0 + v] * a.H);
#pragma unroll
                    for (int u = 0; u < G; ++u) {
                        const int c = c0 + u * kCombineThreads;
                        if (c < H8) {
                            y0[u][v] = y[2 * c];
                            y1[u][v] = y[2 * c + 1];
                        }
                    }
                }
            }
#pragma unroll
            for (int v = 0; v < S; ++v) {
                if (i0 + v < n) {
                    const float w = s_w[i0 + v];
#pragma unroll
                    for (int u = 0; u < G; ++u) {
                        if (c0 + u * kCombineThreads < H8) {
                            acc[u][0] += w * y0[u][v].x;
                            acc[u][1] += w * y0[u][v].y;
                            acc[u][2] += w * y0[u][v].z;
                            acc[u][3] += w * y0[u][v].w;
                            acc[u][4] += w * y1[u][v].x;
                            acc[u][5] += w * y1[u][v].y;
                            acc[u][6] += w * y1[u][v].z;
                            acc[u][7] += w * y1[u][v].w;
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < G; ++u) {
            const int c = c0 + u * kCombineThreads;
            if (c < H8) {
                uint4 o;
                o.x = pack_bf16x2(acc[u][0], acc[u][1]);
                o.y = pack_bf16x2(acc[u][2], acc[u][3]);
                o.z = pack_bf16x2(acc[u][4], acc[u][5]);
                o.w = pack_bf16x2(acc[u][6], acc[u][7]);
                reinterpret_cast<uint4*>(a.out + t * a.H)[c] = o;
            }
        }
        __syncthreads();
    }
}

template <int G, int S>
static cudaError_t launch_combine_split(const CombineArgs& a, cudaStream_t s)
{
    const int splits = (a.H / 8 + kCombineThreads * G - 1) / (kCombineThreads * G);
    const int64_t items = a.T * splits;
    const int64_t blocks = items < 65535 ? items : 65535;
    return launch_pdl(combine_pairs_split_kernel<G, S>, static_cast<unsigned>(blocks), kCombineThreads, 0, s,
                      a, splits);
}

cudaError_t launch_combine_pairs(const CombineArgs& a, cudaStream_t s)
{
    if (a.T <= 0)
        return cudaSuccess;
    // one group per thread and eight slots in flight for a few tokens (many
    // slots each at TP8); four groups and two slots up to 2048 tokens; one
    // block per token beyond
    if (a.T <= 256)
        return launch_combine_split<1, 8>(a, s);
    if (a.T <= 2048)
        return launch_combine_split<4, 2>(a, s);
    const int64_t blocks = a.T < 65535 ? a.T : 65535;
    return launch_pdl(combine_pairs_kernel, static_cast<unsigned>(blocks), kCombineThreads, 0, s, a);
}

}  // namespace chord
