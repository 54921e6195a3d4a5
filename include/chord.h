/*
 * chord.h -- C ABI of the GB300 (sm_103a) W4A16 INT4 Mixture-of-Experts library.
 *
 * The operation (page: "vLLM x Novita AI: Chord W4A16 INT4 MoE kernels for
 * Kimi K2.x", novita.ai; sections TL;DR, "Two kernel families", "vLLM
 * integration", "Kernel optimisation", Fig. 3):
 *   BF16 activations x unsigned INT4 weight codes with one BF16 scale per 32
 *   input channels, dequantised as w = (q - 8) * scale (subtract, then scale,
 *   one bf16 rounding).  Per routed (token, slot) pair of a local expert e:
 *     g = W13_e[0:I] x,  u = W13_e[I:2I] x          (gate/up GEMM, fp32 accum)
 *     h = bf16(silu(g) * u)                          (fused epilogue)
 *     y = W2_e h                                     (down GEMM, fp32 accum)
 *   and per token: out = bf16(sum over its local slots of weight * y).
 *
 * Storage conventions shared by every entry point:
 *   bf16 values are passed as uint16_t bit patterns;
 *   weight codes: int32 words, 8 codes per word along K, element c = 8w+i in
 *     bits [4i, 4i+4) (low nibble first); W13 codes [E_local, 2I, H/8] (rows
 *     0..I-1 gate, I..2I-1 up), W2 codes [E_local, H, I/8];
 *   scales: bf16 [E_local, 2I, H/32] and [E_local, H, I/32]; every scale is
 *     +-0 or has magnitude in [2^-86, 2^35) (about 1.3e-26 to 3.4e10).  The
 *     kernels form each weight as bf16((q - 8) * scale * 2^-40) with one
 *     rounding and scale the fp32 accumulators by 2^40; inside this range
 *     that equals bf16((q - 8) * scale) exactly.  With
 *     CHORD_FLAG_VALIDATE the layer calls check every scale and return
 *     CHORD_ERR_SCALE_RANGE (device error bit CHORD_DEVERR_SCALE_RANGE);
 *     without it an out-of-range scale gives an inexact weight, not an error.
 *   all matrices row-major and densely packed.
 *
 * Ownership and execution:
 *   every pointer argument marked "device" must point to device memory that the
 *   caller allocated and keeps alive until the work on `stream` completes;
 *   `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Calls enqueue work on the stream and return without waiting,
 *   except where CHORD_FLAG_VALIDATE is set.  No call allocates device memory:
 *   scratch lives in a caller-provided workspace whose size the *_workspace_size
 *   queries return.  Without CHORD_FLAG_VALIDATE no call copies anything back
 *   to the host, so a sequence of calls can be captured in a CUDA graph.
 *
 * Errors: each call returns a chord_status.  Argument, shape and capacity
 * checks happen on the host before anything is launched; nothing is launched
 * when they fail.  Faults the device detects (a routing id out of range, a
 * bounded wait that expired) set bits in a device error word inside the
 * workspace; chord_get_device_error() reads it.  There is no CPU fallback and
 * no silent alternative path: an unsupported case is an error.
 */
#ifndef CHORD_W4A16_H
#define CHORD_W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CHORD_OK = 0,
    CHORD_ERR_INVALID_ARG = -1,       /* null pointer, negative size, bad flag or mode */
    CHORD_ERR_UNSUPPORTED_SHAPE = -2, /* a size the kernels do not handle (see each call) */
    CHORD_ERR_CAPACITY = -3,          /* routing buffers smaller than the required capacity */
    CHORD_ERR_LAYOUT_MODE = -4,       /* grouped mode / layout combination not allowed */
    CHORD_ERR_CUDA = -5,              /* a CUDA runtime call or launch failed */
    CHORD_ERR_TIMEOUT = -6,           /* a device-side bounded wait expired (validate / query) */
    CHORD_ERR_ROUTING = -7,           /* device found invalid routing data (validate / query) */
    CHORD_ERR_WORKSPACE = -8,         /* workspace missing, misaligned or too small */
    CHORD_ERR_NO_DEVICE = -9,         /* no sm_103a device is current */
    CHORD_ERR_SCALE_RANGE = -10,      /* a scale outside the supported range (validate / query) */
    CHORD_ERR_PACKED = -11            /* packed weights that do not match the call (validate / query) */
} chord_status;

/* grouped layouts (page: "grouped SM90 kernels", Fig. 3) */
#define CHORD_GROUPED_CONTIGUOUS 0
#define CHORD_GROUPED_MASKED 1

/* flags */
#define CHORD_FLAG_VALIDATE 1      /* synchronise the stream after the call and turn the
                                      device error word into the status (not capturable) */
#define CHORD_FLAG_DETERMINISTIC 2 /* per-pair fp32 down outputs + ordered combine instead of
                                      fp32 reductions into the token rows.  Without it the
                                      indexed call (for outputs of up to 96 MB of fp32 token
                                      rows) and the grouped call's token output add the pairs
                                      of a token in the order their reductions reach memory,
                                      which changes from run to run: the result is within
                                      the tolerance but not bit-reproducible.  With it the
                                      indexed output is bit-identical run to run. */

#define CHORD_FLAG_TEST_SKIP_ARRIVE 4 /* test hook: the gate/up GEMM drops one mbarrier arrival
                                         (first K stage, CTA 0), so that a bounded device wait
                                         expires; the call's outputs are then undefined and, with
                                         CHORD_FLAG_VALIDATE, it returns CHORD_ERR_TIMEOUT.  Exists
                                         to show that an expired wait ends the kernel cleanly. */
#define CHORD_FLAG_NO_SPLIT_K 8 /* keep every work unit whole: no K-split of the last, partly
                                   filled round of units (see chord_w4a16_moe_indexed) */
#define CHORD_FLAG_PREPACKED 16 /* the layer calls' w13_q / w2_q are chord_w4a16_prepack
                                   outputs (kinds CHORD_PACK_GATE_UP / CHORD_PACK_DOWN) and
                                   w13_s / w2_s are NULL (the scales live in the packs) */
#define CHORD_FLAG_MXFP4 32     /* with CHORD_FLAG_PREPACKED: the packs are chord_mxfp4_prepack
                                   outputs (MXFP4 weights); without it CHORD_ERR_INVALID_ARG */

/* bits of the device error word */
#define CHORD_DEVERR_TIMEOUT 1
#define CHORD_DEVERR_ROUTING 2
#define CHORD_DEVERR_CAPACITY 4
#define CHORD_DEVERR_SCALE_RANGE 8
#define CHORD_DEVERR_PACKED 16

/* Human-readable name of a status. */
const char* chord_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int chord_version(void);

/* ------------------------------------------------------------------------- */
/* Host-side queries (pure functions of their arguments)                      */
/* ------------------------------------------------------------------------- */

/* Capacity of the aligned routing buffers (page: "vLLM integration": the
 * moe_align_block_size buffers are over-allocated): the worst case of
 * sum_e ceil(c_e / block_m) * block_m over any routing of T*k pairs, i.e.
 * T*k + E_local*(block_m-1) rounded up to a multiple of block_m.
 * sorted_ids has `capacity` entries, expert_ids capacity/block_m.
 * Returns -1 for non-positive block_m or negative sizes. */
int64_t chord_moe_align_capacity(int64_t T, int k, int E_local, int block_m);

/* Padding granularity to use for the indexed path (page: "Kernel optimisation",
 * block-M selection by routed tokens per expert).  Here the token tile of the
 * tensor-core MMA is chosen per expert segment at run time, so block_m only
 * sets padding; it is 16, the MMA's N granularity, for every shape. */
int chord_select_block_m(int64_t T, int k, int E_global, int E_local, int H, int I);

/* Writes a one-line description of the schedule the indexed path picks for a
 * shape (token tile, pipeline, combine form) into buf; returns its length.
 * With a CUDA device current, the down GEMM's configuration is the one a call
 * on that device launches (a one-stage K takes the token-stationary tile and
 * a run of weight tiles per unit, chosen by the SM count); without one it is
 * the token tile alone. */
int chord_describe_schedule(int64_t T, int k, int E_global, int E_local, int H, int I, int flags,
                            char* buf, size_t buf_len);

/* Workspace bytes for chord_moe_align. */
size_t chord_moe_align_workspace_size(int64_t T, int k, int E_local);

/* Workspace bytes for chord_w4a16_moe_indexed with these sizes and flags. */
size_t chord_w4a16_moe_workspace_size(int64_t T, int k, int E_global, int E_local, int H, int I,
                                      int block_m, int64_t capacity, int flags);

/* Workspace bytes for chord_w4a16_moe_grouped. M = rows of the grouped input
 * (contiguous: m; masked: E_local*max_m); T, k only matter with out_tokens. */
size_t chord_w4a16_grouped_workspace_size(int mode, int64_t M, int H, int I, int E_local,
                                          int64_t T, int k, int with_tokens, int expected_m);

/* ------------------------------------------------------------------------- */
/* moe_align: routing -> indexed layout                                       */
/* ------------------------------------------------------------------------- */
/*
 * Groups the (token, slot) pairs routed to local experts by expert (page:
 * "Two kernel families": the indexed family consumes vLLM's sorted_ids /
 * expert_ids / num_tokens_padded; Fig. 3: activations are not padded, the
 * padding lives in the index as a sentinel).  Result, fully defined over the
 * whole capacity so that it compares bit-exactly:
 *   experts in ascending local id; inside an expert the pair ids p = t*k + j in
 *   ascending order; each expert padded to a multiple of block_m with the
 *   sentinel T*k; experts without pairs get no block; sorted_ids[ntp..cap) =
 *   T*k and expert_ids[ntp/block_m..cap/block_m) = -1, where ntp =
 *   *num_tokens_padded = sum_e ceil(c_e/block_m)*block_m.
 *
 *   topk_ids     device int32 [T, k]   global expert ids
 *   expert_map   device int32 [E_global] or NULL; local id of each global id,
 *                -1 for experts held elsewhere (NULL: identity, E_local ==
 *                E_global).  Pairs whose expert is not local are dropped; an id
 *                outside [0, E_global) is dropped and sets CHORD_DEVERR_ROUTING.
 *   sorted_ids   device int32 [capacity]         (output)
 *   expert_ids   device int32 [capacity/block_m] (output)
 *   num_tokens_padded device int32 [1]           (output)
 *   capacity     entries of sorted_ids; must be >= chord_moe_align_capacity().
 *   workspace    device, >= chord_moe_align_workspace_size() bytes, 256-aligned.
 * Limits: 1 <= k <= 32, 1 <= E_local <= 1024, 1 <= block_m <= 256,
 *   T*k < 2^31.  T = 0 is allowed (everything becomes padding/tail).
 */
chord_status chord_moe_align(const int32_t* topk_ids, int64_t T, int k, int E_global,
                             const int32_t* expert_map, int E_local, int block_m,
                             int32_t* sorted_ids, int32_t* expert_ids,
                             int32_t* num_tokens_padded, int64_t capacity, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * chord_moe_align without a workspace.  The page has no counterpart: this is
 * for callers that cannot allocate device memory or pass a workspace (code
 * running inside an allocator or memory-pool callback, a plugin whose host owns
 * every device buffer and hands over only inputs and outputs, a runtime that
 * forbids allocation once started).  Same arguments, result and limits as
 * chord_moe_align, minus the workspace; it allocates nothing.
 *
 * Its scratch (a per-256-pair-tile expert histogram and an error word) is a
 * fixed 4 MiB device array inside the library, present on every GPU that
 * loads it until the process exits.  Limit: ceil(T*k/256) * E_local must not
 * exceed 1048512 (T*k up to 261888 pairs at the largest E_local of 1024, or
 * up to about 5.5 million pairs at 48 local experts); larger problems return
 * CHORD_ERR_UNSUPPORTED_SHAPE (checked before any pointer is looked at).  The
 * first call in a CUDA context of a device looks up the array's device address
 * (cudaGetSymbolAddress), and does so again when the device's current context
 * has changed since (a symbol address belongs to one context), so make the
 * first call after a context is created before capturing a stream in it.  All calls share
 * the array: calls whose work overlaps on the GPU (different streams, or
 * different host threads) race and must not be issued; each call rewrites all
 * the scratch it reads.  Routing errors are recorded in the array and are not
 * reported back.
 */
chord_status chord_moe_align_noalloc(const int32_t* topk_ids, int64_t T, int k, int E_global,
                                     const int32_t* expert_map, int E_local, int block_m,
                                     int32_t* sorted_ids, int32_t* expert_ids,
                                     int32_t* num_tokens_padded, int64_t capacity, void* stream);

/* ------------------------------------------------------------------------- */
/* router + moe_align in one call                                             */
/* ------------------------------------------------------------------------- */
/*
 * The router step before the layer, then chord_moe_align of its result, with
 * no host round trip (graph capturable).  Per token t (page: "vLLM
 * integration": top-k routing over the router's softmax):
 *   topk_ids[t, 0..k)     the k largest logits[t, :] in descending order, ties
 *                         to the lower expert id (global ids);
 *   topk_weights[t, j]    softmax probability of expert topk_ids[t, j] over all
 *                         E_global logits, renormalised to sum 1 over the k
 *                         chosen when renormalize != 0 (fp32; exp and the sums
 *                         in fp32, within a few ulp of the fp64 value);
 * then sorted_ids / expert_ids / num_tokens_padded exactly as chord_moe_align
 * on those ids.  Up to 64 tokens (and 512 local experts) both steps
 * run in one CTA (one launch), else as a router kernel and the align kernels.
 *
 *   logits       device float [T, E_global], finite
 *   E_global     1..1024;  k in [1, min(32, E_global)]
 *   topk_ids     device int32 [T, k] (output)
 *   topk_weights device float [T, k] (output)
 *   the other arguments as chord_moe_align; workspace >=
 *   chord_moe_align_workspace_size(T, k, E_local) bytes.
 */
chord_status chord_moe_route_align(const float* logits, int64_t T, int E_global, int k,
                                   int renormalize, const int32_t* expert_map, int E_local,
                                   int block_m, int32_t* topk_ids, float* topk_weights,
                                   int32_t* sorted_ids, int32_t* expert_ids,
                                   int32_t* num_tokens_padded, int64_t capacity, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------- */
/* offline weight prepack                                                     */
/* ------------------------------------------------------------------------- */
/*
 * Rewrites one GEMM's codes and scales into the order the GEMM kernels hold
 * them in shared memory, so that each K stage of a weight tile is one
 * contiguous block read with plain bulk copies (page: "Kernel optimisation /
 * grouped SM90 kernels": the grouped weights are prepacked offline into a
 * kernel layout, and the packing mode is recorded in the prepared weight and
 * checked when the kernel runs).  Done once per weight, like loading it.
 *
 * kind CHORD_PACK_GATE_UP: w_q [E, N = 2I, K/8], w_s [E, 2I, K/32]; tile t
 *   (0 <= t < I/64) has rows 64t .. 64t+63 (gate) then I+64t .. I+64t+63 (up).
 * kind CHORD_PACK_DOWN: w_q [E, N, K/8], w_s [E, N, K/32]; tile t has rows
 *   128t .. 128t+127.
 * Sizes: K % 128 == 0 and N % 128 == 0 (else CHORD_ERR_UNSUPPORTED_SHAPE).  A
 * tile has KB = ceil(K / 256) blocks; when K % 256 == 128 the second half of
 * its last block (codes and scales) is zero, and the GEMMs, which then run
 * 128-deep K stages, never read it.
 *
 * Format (version 1), little-endian:
 *   bytes [0, 256): header of 64 uint32: [0] magic 0x4B504843 ("CHPK"),
 *     [1] version 1, [2] kind, [3] E, [4] N, [5] K, [6] block bytes 18432,
 *     [7] flags (bit 0: some scale outside the range of the header comment),
 *     [8] weight format (0 INT4; 1 MXFP4, chord_mxfp4_prepack), the rest 0.
 *   then blocks of 18432 bytes, block b = (e * (N/128) + t) * KB + j for
 *   expert e, tile t and K block j (codes 256j .. 256j+255):
 *     [0, 16384) codes: half h (codes 256j + 128h ..) at 8192 h; in it, tile
 *       row r at 64 r; the row's four 16-byte pieces (32 codes each, one scale
 *       group, in the word order of the source) with piece c stored at
 *       position c ^ ((r >> 1) & 3);
 *     [16384, 18432) scales: tile row r at 16 r, its 8 bf16 scales of groups
 *       8j .. 8j+7.
 * Total bytes: chord_w4a16_prepack_size() = 256 + E * (N/128) * KB * 18432
 * (the same as codes + scales, plus the header, when K % 256 == 0).
 *
 *   w_q, w_s   device, as above (read only)
 *   packed     device, >= packed_bytes, 16-byte aligned; written entirely.
 *              The layer calls read a pack through its header alone: it must
 *              stay whole (chord_w4a16_prepack_size bytes) while in use.
 * Asynchronous on `stream`; two kernels; graph capturable.
 */
#define CHORD_PACK_GATE_UP 1
#define CHORD_PACK_DOWN 2
size_t chord_w4a16_prepack_size(int kind, int E, int N, int K);  /* 0 for bad arguments */
chord_status chord_w4a16_prepack(int kind, const int32_t* w_q, const uint16_t* w_s, int E, int N,
                                 int K, void* packed, size_t packed_bytes, void* stream);

/*
 * MXFP4 weights (page: vLLM Kimi K3 production support, news.ainew.jp, "MXFP4
 * MoE": MoE weights in MXFP4; the OCP Microscaling FP4 format that name
 * refers to): each 4-bit code is an FP4 E2M1 number (bit 3 sign, bits 2-1 an
 * exponent with bias 1, bit 0 a mantissa bit; exponent 0 is subnormal, so the
 * sixteen codes are +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}), and each group of 32
 * input channels shares one E8M0 scale byte e meaning 2^(e - 127) (e = 255:
 * NaN).  The weight is w = bf16(e2m1(q) * 2^(e - 127)): exact for every code
 * and byte unless it overflows bf16 (then +-inf, as bf16 rounding gives).  The
 * activation (SiLU(gate) * up), the combine and everything else are those of
 * the INT4 layer.
 *
 * chord_mxfp4_prepack packs such weights for the layer calls: the codes are
 * stored like INT4 codes (8 per int32 word, low nibble first, [E, N, K/8]),
 * w_e8m0 holds the scale bytes [E, N, K/32] (device, 16-byte aligned), and the
 * output is a pack of the chord_w4a16_prepack format and size whose scale rows
 * hold each byte widened to the bf16 value 2^(e - 127) (0x0040 for e = 0, NaN
 * 0x7FC0 for e = 255), with header word 8 (weight format) = 1 (INT4 packs: 0).
 * The layer calls take MXFP4 packs with CHORD_FLAG_PREPACKED | CHORD_FLAG_MXFP4
 * and check the format word with the rest of the header.
 */
chord_status chord_mxfp4_prepack(int kind, const int32_t* w_q, const uint8_t* w_e8m0, int E, int N,
                                 int K, void* packed, size_t packed_bytes, void* stream);

/* ------------------------------------------------------------------------- */
/* the MoE layer on the indexed layout                                        */
/* ------------------------------------------------------------------------- */
/*
 * out[T, H] = the layer above, reading the pairs from the aligned layout
 * (page: "Two kernel families": the indexed path; "vLLM integration": the
 * over-allocated buffers are consumed without reading counts back to the
 * host, so the call is CUDA-graph capturable).
 *
 *   x            device bf16 [T, H]
 *   E_global     experts the router chose from; with T*k it gives the expected
 *                rows per local expert that steers the schedule (must match the
 *                value given to chord_w4a16_moe_workspace_size)
 *   w13_q, w13_s, w2_q, w2_s  device weights as in the header comment; with
 *                CHORD_FLAG_PREPACKED, w13_q / w2_q are chord_w4a16_prepack
 *                outputs (kinds GATE_UP with N = 2I, K = H, and DOWN with N = H,
 *                K = I, E >= E_local) and w13_s / w2_s are NULL.  The call
 *                checks both headers on the device before the GEMMs run; on a
 *                mismatch the GEMMs compute nothing (no output is valid) and
 *                CHORD_DEVERR_PACKED is set (CHORD_ERR_PACKED with
 *                CHORD_FLAG_VALIDATE); a pack whose flags record an
 *                out-of-range scale sets CHORD_DEVERR_SCALE_RANGE
 *   topk_weights device float [T, k]; weight of pair p = t*k+j is topk_weights[p]
 *   sorted_ids, expert_ids, num_tokens_padded  device, the chord_moe_align
 *                layout (any producer of the same layout works)
 *   capacity, block_m  the sizes the layout was built with
 *   workspace    device, >= chord_w4a16_moe_workspace_size() bytes, 256-aligned
 *   out          device bf16 [T, H] (output; every element written)
 *   h_out        device bf16 [capacity, I] or NULL: when given, the gate/up
 *                stage writes its output h = bf16(silu(g) * u) here (rows
 *                < num_tokens_padded; sentinel rows get 0) instead of into the
 *                workspace, so a caller can inspect or reuse it
 *   flags        CHORD_FLAG_* ; CHORD_FLAG_DETERMINISTIC gives run-to-run
 *                bit-identical outputs (slots summed in a fixed order); the
 *                default fp32 reductions are not bit-reproducible run to run
 * Limits (CHORD_ERR_UNSUPPORTED_SHAPE otherwise): H % 128 == 0, I % 128 == 0,
 *   1 <= k <= 32, E_local >= 1, T*k < 2^31, block_m in [1, 256].
 * Work schedule of both GEMMs: one CTA per SM takes (chunk of rows, weight
 *   tile) units in turn.  When the last round of units would leave at least
 *   half of the SMs idle (decode token tiles, K stages of 256), each of its
 *   units is cut along K into pieces of two
 *   or more K stages, one per otherwise idle SM; every piece leaves its fp32
 *   partial sum in the workspace and the last piece of a unit to finish adds
 *   the pieces in piece order (a fixed order: results stay bit-identical from
 *   run to run) and runs the unit's epilogue.  CHORD_FLAG_NO_SPLIT_K turns
 *   this off.
 */
chord_status chord_w4a16_moe_indexed(const uint16_t* x, int64_t T, int H, int I, int E_global,
                                     int E_local, int k, const int32_t* w13_q,
                                     const uint16_t* w13_s, const int32_t* w2_q,
                                     const uint16_t* w2_s, const float* topk_weights,
                                     const int32_t* sorted_ids, const int32_t* expert_ids,
                                     const int32_t* num_tokens_padded, int64_t capacity,
                                     int block_m, void* workspace, size_t workspace_bytes,
                                     uint16_t* out, uint16_t* h_out, int flags, void* stream);

/* ------------------------------------------------------------------------- */
/* the MoE layer on a grouped layout                                          */
/* ------------------------------------------------------------------------- */
/*
 * Same expert MLP on the grouped layouts (page: "grouped SM90 kernels",
 * Fig. 3, and the grouped operator entry points contiguous(a2, w, m_indices)
 * / masked(a3, w, masked_m, expected_m)).
 *
 * mode CHORD_GROUPED_CONTIGUOUS: a is [M, H]; row r belongs to expert
 *   m_indices[r], or is padding when m_indices[r] < 0.  Each expert's rows are
 *   contiguous and start on a multiple of 16 rows (the page pads each expert
 *   to 128); M % 16 == 0.  masked_m must be NULL.
 * mode CHORD_GROUPED_MASKED: a is [E_local, max_m, H] (M = E_local*max_m);
 *   rows e*max_m + i with i < masked_m[e] are valid, the rest are never read.
 *   expected_m (> 0) is the host-side launch hint (expected valid rows per
 *   expert); masked_m (device int32 [E_local]) is authoritative.  m_indices
 *   must be NULL.
 *
 *   out_rows     device bf16 [M, H]: bf16(y) for every valid row.  Rows that
 *                are padding (contiguous) or past masked_m (masked) carry no
 *                result; consumers ignore them, as on the page.
 *   row_to_pair, topk_weights, out_tokens: optional token combine.  When
 *                out_tokens is not NULL, row_to_pair (device int32 [M], pair id
 *                t*k+j of each valid row or -1) and topk_weights (device float
 *                [T, k]) are required and out_tokens (device bf16 [T, H]) gets
 *                the same combine as the indexed layer.
 *   h_out        device bf16 [M, I] or NULL: the gate/up output of every row
 *                the call computes (as for the indexed call).
 *   w13_q, w13_s, w2_q, w2_s  as for the indexed call, CHORD_FLAG_PREPACKED
 *                included.
 * Limits as for the indexed call, plus max_m >= 1.
 */
chord_status chord_w4a16_moe_grouped(int mode, const uint16_t* a, int64_t M, int H, int I,
                                     int E_local, const int32_t* m_indices,
                                     const int32_t* masked_m, int64_t max_m, int expected_m,
                                     const int32_t* w13_q, const uint16_t* w13_s,
                                     const int32_t* w2_q, const uint16_t* w2_s,
                                     const int32_t* row_to_pair, const float* topk_weights,
                                     int64_t T, int k, void* workspace, size_t workspace_bytes,
                                     uint16_t* out_rows, uint16_t* out_tokens, uint16_t* h_out,
                                     int flags, void* stream);

/* ------------------------------------------------------------------------- */
/* device error word                                                          */
/* ------------------------------------------------------------------------- */
/* Synchronises `stream`, copies the error word of `workspace` (of a layer or
 * align call) to *error_bits, clears it when `clear` is non-zero, and returns
 * CHORD_ERR_TIMEOUT / CHORD_ERR_ROUTING / CHORD_ERR_CAPACITY /
 * CHORD_ERR_SCALE_RANGE / CHORD_ERR_PACKED for the first bit set, else
 * CHORD_OK.  Not capturable. */
chord_status chord_get_device_error(void* workspace, int* error_bits, int clear, void* stream);

/* ------------------------------------------------------------------------- */
/* stage timing (profiling aid)                                               */
/* ------------------------------------------------------------------------- */
/* When enabled, each indexed / grouped layer call records CUDA events around
 * its stages (prepare, gate_up, down, combine) on its stream.  read() waits for
 * the recorded events and returns the summed milliseconds per stage over all
 * calls since enable, and the number of calls.  Stage events are skipped while
 * a stream is being captured. */
chord_status chord_stage_timing_enable(int enable);
chord_status chord_stage_timing_read(float* ms_per_stage /* [4] */, int* calls);

#ifdef __cplusplus
}
#endif

#endif /* CHORD_W4A16_H */
