// chord_internal.h -- definitions shared by the host side and the kernels.
#pragma once

#include <stdint.h>

#include "chord.h"

namespace chord {

// One run of padded rows that share an expert, at most one MMA token tile long.
struct Chunk {
    int32_t row0;    // first padded row
    int32_t nrows;   // rows in this chunk (the token tile is nrows rounded up to 16)
    int32_t expert;  // local expert
    int32_t brow0;   // first row of the chunk in the GEMM's token-row source: row0, except
                     // that the masked layout's gate/up reads its rows compacted
};

// Down-GEMM epilogue forms (bit set).
enum Epilogue : int {
    kEpiStorePair = 1,   // y_pairs[p, n] = y (fp32) for the pair of each row
    kEpiReduceTok = 2,   // out_acc[t, n] += w_p * y (fp32 reductions)
    kEpiStoreRows = 4,   // rows_out[r, n] = bf16(y)
};

struct GemmArgs {
    // B operand: the token rows of each chunk are contiguous in the tensor map
    // passed next to the codes map (x gathered into padded-row order, a, or h)
    int topk;
    int num_pairs;            // T*k, the sentinel
    // problem
    int K;                    // reduction length
    int N;                    // rows of one expert's weight
    int I;                    // intermediate size (gate_up: up rows start at I)
    int n_tiles;              // output tiles per chunk
    int tpu;                  // tiles per work unit (n_tiles % tpu == 0; > 1 only when K is one stage)
    const uint16_t* scales;   // [E, N, K/32]
    // prepacked weights (chord_w4a16_prepack; its header was checked by the
    // prep kernel), or null: the codes and scales of K block j of tile t of
    // expert e are block (e * n_tiles + t) * (K/256) + j of pk, in the
    // shared-memory order of a code / scale stage
    const uint8_t* pk;
    const Chunk* chunks;
    const int32_t* num_chunks;
    // epilogue
    int epi;
    uint16_t* h_out;          // gate_up: [rows, I]
    int64_t ld_h;
    int32_t* pair_row;        // gate_up: pair -> padded row (ordered combine), or null
    float* y_pairs;           // down: [T*k, N]
    float* out_acc;           // down: [T, N]
    uint16_t* rows_out;       // down: [rows, N]
    const int32_t* pair_of_row;  // pair id t*k+j of each padded row (or -1 / sentinel)
    int h_zero_unpaired;         // gate_up: rows whose pair_of_row is not a pair get h = 0
    const int4* row_meta;        // down: {pair, token, weight bits, 0} per padded row
    int* err;
    int test_skip_arrive;  // CHORD_FLAG_TEST_SKIP_ARRIVE (gate_up only)
    // K-split of the last, partly filled round of units (0 slots: never split)
    float* split_part;     // [split_slots][MAXN columns][128 rows] fp32 partial sums
    int32_t* split_cnt;    // [split_slots] finished pieces per split unit, zero on entry
    int split_slots;
};

// Partial-sum slots of the K-split per GEMM (at least the SM count of the part).
constexpr int kSplitSlots = 160;
// Fewest K stages in one piece of a split unit.
constexpr int kSplitMinStages = 2;

// prepacked weights (format in chord.h, chord_w4a16_prepack)
constexpr uint32_t kPackMagic = 0x4B504843u;  // "CHPK"
constexpr int kPackHeaderBytes = 256;
constexpr int kPackCodeBytes = 16384;          // one 256-deep K block of a 128-row tile
constexpr int kPackBlockBytes = kPackCodeBytes + 2048;
constexpr int kPackFormatWord = 8;             // header word: weight format of the pack
// 256-deep K blocks of one pack tile (K % 128 == 0; a 128 tail is half a block)
__host__ __device__ constexpr int pack_kblocks(int K) { return (K + 255) / 256; }
constexpr uint32_t kPackFmtInt4 = 0;           // chord_w4a16_prepack
constexpr uint32_t kPackFmtMxfp4 = 1;          // chord_mxfp4_prepack

constexpr int kGemmThreads = 512;  // 16 warps (the GEMM configurations may add a warp group)

}  // namespace chord
