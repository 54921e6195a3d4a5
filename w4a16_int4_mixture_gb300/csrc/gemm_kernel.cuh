// gemm_kernel.cuh -- the W4A16 expert GEMM for sm_103a (tcgen05 + TMEM + TMA).
//
// One persistent CTA per SM takes work units (chunk of padded rows that share an
// expert) x (128-row tile of that expert's weight), dealt to the CTAs with a
// stride of the grid.  Per unit it computes
//   D[128 weight rows, ntok tokens] = W_tile[128, K] * X_rows[ntok, K]^T
// with the dequantised weights as the MMA's M operand (held in tensor memory)
// and the routed tokens as its N operand (in shared memory).  This is the
// Blackwell form of the swap-AB decode schedule of the Chord page ("Kernel
// optimisation / H200 and Blackwell indexed decode": dequantised weights take
// the MMA-M operand), used here for every token count.
//
// Roles (16 warps; 20 with three dequant warps per quadrant or a second
// epilogue group):
//   warp 0      code producer: packed 4-bit codes of each K stage into a ring, one
//               TMA box (gate and up halves as one 4-D box), L2 evict-first,
//               and the group-32 scales (a TMA box, or cp.async for BK 128);
//               for prepacked weights one or two plain bulk copies of the
//               stage's contiguous block instead.
//   warp 1      token producer: the chunk's activation rows, contiguous in the
//               B tensor map, as 128B-swizzled K-major TMA tiles (one 3-D box
//               per stage for token tiles of up to 64 rows; the rows past the
//               chunk only feed discarded columns).  With as many token stages
//               as A stages the two rings share their barriers (FUSED_RINGS).
//   warp 2      MMA issuer (the whole warp walks the schedule; elect.sync picks
//               the issuing lane) and TMEM owner.
//   warp 3      idle.
//   warps 4-7   epilogue: TMEM -> registers; gate_up: SiLU(gate)*up -> bf16 h;
//               down: per-pair fp32 store, fp32 reductions into token rows,
//               or bf16 row store.
//   warps 8-15  dequant, two warps per TMEM lane quadrant (three, warps 8-19,
//               in the configurations with three A stages and one epilogue
//               group: the decode tiles of both GEMMs), taking K stages in
//               order from a shared counter: codes + scales from shared memory
//               -> w = bf16((q - 8) * s), one rounding of the exact product as
//               in the page's order (exact q - 8, then the scale multiply),
//               held as w * 2^-40 (undone on the fp32 accumulators); MXFP4
//               codes: w = bf16(e2m1(q) * 2^(e - 127)) by an exact placement
//               and one multiply (see dequant_word_mx) -> tcgen05.st into the
//               A-operand stage in TMEM.
//   warps 16-19 (token-stationary down configurations) a second epilogue group
//               taking every other tile.
// Every wait is bounded (2 s); on expiry the CTA records CHORD_DEVERR_TIMEOUT,
// every role leaves its loop, in-flight tensor-core work is drained and TMEM
// is freed.
#pragma once

#include "device.cuh"

namespace chord {

template <int BK_, int KS_, int BS_, int AS_, int MAXN_, int ACCB_, bool GATE_UP_, int ACCW_ = MAXN_,
          int PS_ = 0, bool TS_ = false>
struct GemmCfg {
    static constexpr int BK = BK_;        // K elements per stage
    static constexpr int KS = KS_;        // code/scale stages in shared memory
    static constexpr int BS = BS_;        // token stages in shared memory
    static constexpr int AS = AS_;        // A-operand stages in TMEM
    static constexpr int MAXN = MAXN_;    // largest token tile
    static constexpr int ACCB = ACCB_;    // accumulator buffers in TMEM
    // columns of one accumulator buffer: ACCW / MAXN weight tiles of a unit
    // (one-stage K: several tiles share the unit's token tile)
    static constexpr int ACCW = ACCW_;
    // token-stationary units (down GEMM, one K stage): a unit is one chunk and
    // a run of weight tiles; its token tile is loaded once, and each tile is
    // accumulated in the next of the ACCB buffers and drained on its own
    static constexpr bool TS = TS_;
    static constexpr int TPU_MAX = TS ? 64 : ACCW / MAXN;
    static constexpr bool GATE_UP = GATE_UP_;
    // K stages per accumulation chain (0: a unit's whole K range in one chain).
    // The tensor core's fp32 accumulation loses accuracy as one chain grows
    // (measured against an fp64 evaluation: over K = 7168 in one chain the
    // gate/up output's bf16 rounding differs from the exact one about 7x as
    // often as for a sequential fp32 sum).  With PS > 0 the MMA starts a fresh
    // accumulator every PS stages, alternating between the accumulator
    // buffers, and the epilogue adds each finished partial into the next one
    // (fp32, round to nearest, in order) before the unit's epilogue runs on
    // the last.
    static constexpr int PS = PS_;

    // codes of a stage: BK/128 halves of [128 tile rows][64 bytes], 64B swizzle
    static constexpr int CODE_STAGE = 128 * (BK / 2);
    static constexpr int SCALE_ROW = BK / 16;               // bytes of scales per weight row
    static constexpr int SCALE_STAGE = 128 * SCALE_ROW;
    static constexpr int B_KBLK = BK / 64;                  // 128B swizzle atoms along K
    static constexpr int B_REGION = MAXN * 128;             // one atom column of the tile
    static constexpr int B_BOX_ROWS = MAXN < 64 ? MAXN : 64; // rows per token TMA box
    // token tile of a stage as one 3-D TMA box {64 columns, MAXN rows, BK/64
    // column blocks} when it fits one box of rows; else 2-D boxes of 64 rows
    static constexpr bool B_3D = MAXN <= 64;
    // the stage's scales as a TMA box (16-byte rows) when BK = 256; cp.async
    // (8-byte rows) when BK = 128
    static constexpr bool SCALES_TMA = BK == 256;
    // One tile per unit and as many token stages as A stages: stage g uses A
    // slot and token slot g % AS, so the two rings share their barriers.  The
    // token tile's TMA completes on the A stage's full barrier (the four
    // dequant arrivals plus the token producer's expect_tx arrival) and the
    // A stage's empty barrier frees the token slot too: the MMA warp, the
    // critical role of the decode tiles (measured), waits and commits once
    // per stage instead of twice.
    static constexpr bool FUSED_RINGS = !TS && ACCW == MAXN && AS == BS;
    static constexpr int B_STAGE = B_KBLK * B_REGION;
    static constexpr int HS_BYTES = GATE_UP ? MAXN * 128 : 0;  // 64 channels of bf16 per row
    static constexpr int META_BYTES = 0;  // (column records live in registers)
    // token-stationary down units (a one-stage K, where every tile's
    // epilogue is short and the epilogue is the critical role): a second group
    // of four epilogue warps (warps 16-19) takes every other tile, each group
    // owning every other accumulator buffer
    static constexpr int EPI_GROUPS = (!GATE_UP && MAXN <= 64 && TS) ? 2 : 1;
    // dequant warps per TMEM lane quadrant.  Each holds one claimed K stage,
    // so up to DQW stages are in dequant at once; their A slots (and code
    // slots) must be distinct phases of the rings, hence DQW <= AS and KS.
    // Three when there are three A stages and one epilogue group: the dequant
    // is the bound of the weight-streaming tiles (measured 145.6 -> 141.1 us
    // for the EP8 decode gate/up); a CTA of 640 threads has no registers for
    // a sixth warp group.
    static constexpr int DQW = (AS >= 3 && EPI_GROUPS == 1) ? 3 : 2;
    // (a split dequant, every warp of a quadrant taking every stage and in it
    // every DQW-th scale group, cut one stage's latency but ran the EP8 decode
    // gate/up at 188 us against 145: whole stages per warp, in turn, it is)
    static constexpr int EPI1_WARP = 8 + 4 * DQW;  // first warp of the second epilogue group
    static constexpr int THREADS = 32 * EPI1_WARP + 128 * (EPI_GROUPS - 1);
    // down: per epilogue warp a 16-column x 32-row fp32 tile to transpose the
    // accumulator so each lane owns four consecutive output rows of a column
    // (a direct epilogue without the tile, lane l reducing output channel l of
    // its quadrant one token column at a time, took the TP8 2048-token down
    // GEMM from 182 to 401 us: four times the reductions, each coalesced)
    static constexpr int EPIT_BYTES = GATE_UP ? 0 : EPI_GROUPS * 4 * 16 * 32 * 4;
    // (bulk reductions of the tile's token columns through the copy engine,
    // 128 bytes each, took the same GEMM to 281 us: vector reductions by every
    // lane are the fastest of the three forms measured)

    static constexpr int OFF_CODES = 0;
    static constexpr int OFF_B = OFF_CODES + KS * CODE_STAGE;
    static constexpr int OFF_SCALES = OFF_B + BS * B_STAGE;
    static constexpr int OFF_HS = OFF_SCALES + KS * SCALE_STAGE;
    static constexpr int OFF_META = OFF_HS + HS_BYTES;
    static constexpr int OFF_EPIT = OFF_META + META_BYTES;
    static constexpr int OFF_BARS = OFF_EPIT + EPIT_BYTES;
    // rings, then one rendezvous per epilogue group and the drain barrier
    static constexpr int NBARS = 2 * KS + 2 * AS + 2 * BS + 2 * ACCB + 3;
    static constexpr int OFF_MISC = OFF_BARS + NBARS * 8;
    // misc: TMEM base, abort flag, a split-unit verdict per epilogue group,
    // 4 per-quadrant stage counters
    static constexpr int SMEM_BYTES = OFF_MISC + 32 + 1024;  // + alignment slack

    static constexpr int A_COLS = BK / 2;                   // TMEM columns per A stage
    static constexpr int D_COL0 = AS * A_COLS;
    static constexpr int TMEM_COLS = 512;

    // producers and epilogue wait with the spin loop out of line (smaller hot
    // code; measured faster for the BK 256 decode tiles, slower for the
    // prefill tile, whose producers wake on every one of its short stages)
    static constexpr bool COLD_WAITS = BK == 256;

    static_assert(BK == 128 || BK == 256, "stage depth");
    static_assert(MAXN % 16 == 0 && MAXN >= 16 && MAXN <= 256, "token tile");
    static_assert(D_COL0 + ACCB * ACCW <= TMEM_COLS, "tensor memory budget");
    static_assert(ACCW % MAXN == 0 && (TPU_MAX == 1 || (!GATE_UP && BK == 256)), "tiles per unit");
    static_assert(!TS || (ACCW == MAXN && PS == 0), "token-stationary: one tile per accumulator buffer");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(SMEM_BYTES > 116 * 1024, "one CTA per SM keeps the 512-column TMEM alloc safe");
    static_assert(OFF_B % 1024 == 0 && B_REGION % 1024 == 0, "swizzle atoms need 1024B alignment");
    static_assert(MAXN % B_BOX_ROWS == 0 && (B_BOX_ROWS * 128) % 1024 == 0, "token boxes");
    static_assert(ACCB % EPI_GROUPS == 0, "each epilogue group owns whole accumulator buffers");
    static_assert(DQW <= AS && DQW <= KS, "stages in dequant at once fit the A and code rings");
    static_assert(THREADS <= 640, "register budget of one CTA per SM");
    static_assert(PS == 0 || (EPI_GROUPS == 1 && TPU_MAX == 1 && ACCB >= 2),
                  "partial accumulation: one epilogue group walks every partial of a unit");
    static_assert(CODE_STAGE % 1024 == 0, "TMA destinations");
};

// Byte offset in a code stage of piece g (codes 32g .. 32g+31 of the stage,
// one scale group, 16 bytes) of tile row r: halves of 128 codes, each 128
// rows x 64 bytes with the 64-byte swizzle (piece c of a half at position
// c ^ ((r >> 1) & 3)).  The TMA writes this layout and chord_w4a16_prepack
// stores it.  The 32 rows a warp reads at once fall on distinct banks for
// every 8 rows.
__device__ __forceinline__ int code_piece_offset(int g, int r)
{
    return (g >> 2) * 8192 + r * 64 + (((g & 3) ^ ((r >> 1) & 3)) << 4);
}

// bf16x2 helpers (single rounding each, round to nearest even)
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// generic-mode byte permute: selector bit 3 of a byte replicates the sign bit
// of the selected byte (0x00 for the code bytes here, which are 0..15)
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// The weights enter the MMA as w' = bf16((q - 8) * s * 2^-40); the epilogue
// multiplies the fp32 accumulators by 2^40 (exact).  For +-0 scales and
// |s| in [2^-86, 2^35) every step below is exact up to the one rounding and
// (q - 8) * s * 2^-40 stays a normal bf16, so w' * 2^40 = bf16((q - 8) * s):
// the page's value, one rounding of the exact product.  (2^-40 keeps the
// products w' * x far above the fp32 subnormal range for any realistic scale
// and activation.)
constexpr float kWeightRescale = 1099511627776.0f;  // 2^40

// Per scale group: the fma constants from the bf16x2 scale pair s2 = (s, s):
// A = (s * 2^93, s * 2^89) (for the low / high element of a pair, whose codes
// arrive scaled by 2^-133 / 2^-129) and B = -8 s * 2^-40 = -s * 2^-37; both are
// power-of-two multiples of s, so exact inside the scale range.
struct ScalePair {
    uint32_t a;
    uint32_t b;
};
__device__ __forceinline__ ScalePair scale_pair(uint32_t s2)
{
    return {bf16x2_mul(s2, 0x6C006E00u) /* (2^93, 2^89) */,
            bf16x2_mul(s2, 0xAD00AD00u) /* -2^-37 */};
}

// Dequantise one word of 8 codes (element i in bits 4i..4i+3) into 4 bf16x2
// columns (elements (0,1) .. (6,7)) of w' (see above).
//   lo / hi: w & 0x0F0F0F0F / w & 0xF0F0F0F0: byte j holds q_2j / 16 q_2j+1;
//   prmt:    bytes (q_2j, 0, 16 q_2j+1, 0) as two bf16 bit patterns: q_2j *
//            2^-133 and q_2j+1 * 2^-129 (subnormal, or for 16 q >= 128 the
//            first normal binade, which continues the subnormal spacing); the
//            zero bytes replicate the sign bit of a lo byte (always 0);
//   fma:     q * 2^-133 * (s * 2^93) + (-s * 2^-37) = (q - 8) * s * 2^-40
//            (likewise for the high element): the product and the sum are
//            exact before the one rounding.
__device__ __forceinline__ void dequant_word(uint32_t w, ScalePair sp, uint32_t* o)
{
    const uint32_t lo = w & 0x0F0F0F0Fu;
    const uint32_t hi = w & 0xF0F0F0F0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t sel = static_cast<uint32_t>(j | ((8 | j) << 4) | ((4 + j) << 8) | ((8 | j) << 12));
        o[j] = bf16x2_fma(prmt(lo, hi, sel), sp.a, sp.b);
    }
}

// Weight formats of the kernel (a template parameter: see PK below for why not
// a run-time switch).
constexpr int kFmtInt4 = 0;   // unsigned codes q, bf16 scales s: w = bf16((q - 8) * s)
constexpr int kFmtMxfp4 = 1;  // FP4 E2M1 codes, one E8M0 scale byte per 32 inputs:
                              // w = bf16(e2m1(q) * 2^(e - 127)); the pack holds the
                              // scale widened to the bf16 value 2^(e - 127)

// MXFP4 (vLLM Kimi K3 production support page, "MXFP4 MoE"; OCP Microscaling
// FP4): a code is sign (bit 3), two exponent bits with bias 1 (bits 2-1) and one
// mantissa bit (bit 0); exponent 0 is subnormal (m * 0.5).  Placing the three
// magnitude bits at bf16 bits 8-6 (the exponent's two low bits and the
// mantissa's top bit) and the sign at bit 15 gives the bf16 number
// e2m1(q) * 2^-126 exactly: a bf16 exponent field 1..3 reads (1 + m/2) *
// 2^(e - 127), and field 0 is a bf16 subnormal m/2 * 2^-126, which continues
// the spacing the same way E2M1's subnormal does.
//   lo / hi: w & 0x0F0F0F0F / (w >> 4) & 0x0F0F0F0F, byte j holding code 2j /
//            code 2j+1;
//   prmt:    x = code 2j in bits 0-3 and code 2j+1 in bits 16-19 (the other
//            bytes zero: sign replication of a byte below 0x80);
//   place:   x * 0x1040 = (x << 6) + (x << 12): the two copies of each code
//            do not overlap (bits 6-9 and 12-15 of each half), and the mask
//            keeps the first copy's magnitude (bits 6-8 / 22-24) and the
//            second copy's sign (bit 15 / 31).
__device__ __forceinline__ uint32_t mx_place_pair(uint32_t lo, uint32_t hi, int j)
{
    const uint32_t sel = static_cast<uint32_t>(j | (8 << 4) | ((4 + j) << 8) | (8 << 12));
    return (prmt(lo, hi, sel) * 0x1040u) & 0x81C081C0u;
}
// Every scale byte e <= 128: one exact product with m = (2^(e-1), 2^(e-1)),
// e2m1(q) * 2^-126 * 2^(e-1) = e2m1(q) * 2^(e-127) (two significant bits, so
// the one rounding is exact unless the value overflows bf16, as in the
// definition's rounding).
__device__ __forceinline__ void dequant_word_mx(uint32_t w, uint32_t m, uint32_t* o)
{
    const uint32_t lo = w & 0x0F0F0F0Fu;
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        o[j] = bf16x2_mul(mx_place_pair(lo, hi, j), m);
}
// Any scale byte: 2^(e-1) leaves bf16 above e = 128, so the factor is split:
// e2m1(q) * 2^-126 * 2^127 = 2 e2m1(q) (exact), then * 2^(e-128) (m2, also a
// bf16 value for every e): the same single effective rounding.
__device__ __forceinline__ void dequant_word_mx2(uint32_t w, uint32_t m2, uint32_t* o)
{
    const uint32_t lo = w & 0x0F0F0F0Fu;
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        o[j] = bf16x2_mul(bf16x2_mul(mx_place_pair(lo, hi, j), 0x7F007F00u /* 2^127 */), m2);
}

// One work item of a GEMM CTA: a whole unit, or one K piece of a split unit.
struct WorkItem {
    int unit;   // chunk * units_per_chunk + tile group
    int k0;     // K stages [k0, k1)
    int k1;
    int piece;  // -1 for a whole unit, else the piece index
    int tail;   // split units: index of the unit among the split ones
};

// PK: the weights are prepacked (chord_w4a16_prepack) and arrive by plain bulk
// copies.  A template parameter, not a run-time switch: with both load paths
// in one kernel the plain path ran 23 % slower (EP8 decode gate/up 139.5 ->
// 171 us) although the branch was never taken.
// FMT: the weight format (kFmtInt4 / kFmtMxfp4; MXFP4 weights come prepacked).
template <class C, bool PK, int FMT>
__global__ void __launch_bounds__(C::THREADS, 1)
    w4a16_gemm_kernel(const __grid_constant__ CUtensorMap codes_map,
                      const __grid_constant__ CUtensorMap scales_map,
                      const __grid_constant__ CUtensorMap b_map, const GemmArgs args)
{
    static_assert(FMT == kFmtInt4 || (FMT == kFmtMxfp4 && PK), "MXFP4 weights are read from packs");
    // the INT4 dequant forms w * 2^-40 (undone here on the fp32 accumulators);
    // the MXFP4 dequant forms w itself
    constexpr float kRescale = FMT == kFmtInt4 ? kWeightRescale : 1.0f;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw_u32);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if constexpr (!C::GATE_UP)
        pdl_launch_dependents();

    // barriers
    const uint32_t bar0 = sbase + C::OFF_BARS;
    auto codes_full = [&](int s) { return bar0 + 8u * s; };
    auto codes_empty = [&](int s) { return bar0 + 8u * (C::KS + s); };
    auto a_full = [&](int s) { return bar0 + 8u * (2 * C::KS + s); };
    auto a_empty = [&](int s) { return bar0 + 8u * (2 * C::KS + C::AS + s); };
    auto b_full = [&](int s) { return bar0 + 8u * (2 * C::KS + 2 * C::AS + s); };
    auto b_empty = [&](int s) { return bar0 + 8u * (2 * C::KS + 2 * C::AS + C::BS + s); };
    auto d_full = [&](int s) { return bar0 + 8u * (2 * C::KS + 2 * C::AS + 2 * C::BS + s); };
    auto d_empty = [&](int s) {
        return bar0 + 8u * (2 * C::KS + 2 * C::AS + 2 * C::BS + C::ACCB + s);
    };
    const uint32_t epi_bar0 = bar0 + 8u * (C::NBARS - 3);  // + 8 * epilogue group
    const uint32_t drain_bar = bar0 + 8u * (C::NBARS - 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* split_last = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);  // [2]
    int* stage_ctr = reinterpret_cast<int*>(smem + C::OFF_MISC + 16);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::KS; ++s) {
            // expect_tx arrive (+ 32 cp.async arrivals when scales come by cp.async)
            mbar_init(codes_full(s), C::SCALES_TMA ? 1 : 1 + 32);
            mbar_init(codes_empty(s), 4);      // the 4 warps of one dequant group
        }
        for (int s = 0; s < C::AS; ++s) {
            // the 4 dequant warps (+ the token tile's expect_tx arrival when fused)
            mbar_init(a_full(s), C::FUSED_RINGS ? 5 : 4);
            mbar_init(a_empty(s), 1);          // tcgen05.commit
        }
        for (int s = 0; s < C::BS; ++s) {
            mbar_init(b_full(s), 1);           // expect_tx arrive
            mbar_init(b_empty(s), 1);
        }
        for (int s = 0; s < C::ACCB; ++s) {
            mbar_init(d_full(s), 1);
            mbar_init(d_empty(s), 4);          // 4 epilogue warps
        }
        mbar_init(epi_bar0, 4);                // epilogue group rendezvous
        mbar_init(epi_bar0 + 8u, 4);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        for (int qq = 0; qq < 4; ++qq)
            stage_ctr[qq] = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0 && !PK) {
        prefetch_tensormap(&codes_map);
        if constexpr (C::SCALES_TMA)
            prefetch_tensormap(&scales_map);
    }
    if (warp == 1 && lane == 0)
        prefetch_tensormap(&b_map);
    if (warp == 2)
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Barriers and tensor memory are set up while the previous kernel ends.
    // gate_up reads prep's outputs everywhere, so it waits here, and only then
    // lets the down GEMM be scheduled; the down GEMM, whose chunk lists, row
    // records and weights are ready by then, waits only where it reads h (the
    // token producer): on an SM the gate/up tail has freed it already streams
    // and dequantises weights.
    if constexpr (C::GATE_UP) {
        pdl_wait();
        pdl_launch_dependents();
    }

    const int n_tiles = args.n_tiles;
    const int KT = args.K / C::BK;
    // weight tiles per unit (1, or up to TPU_MAX for a one-stage K): a unit
    // covers tiles nt0 .. nt0 + tpu - 1 of one chunk, K stage by K stage, each
    // tile into its own MAXN columns of the accumulator
    const int tpu = C::TPU_MAX == 1 ? 1 : args.tpu;
    const int units_per_chunk = n_tiles / tpu;
    int issued_stages = 0;  // code / token producers: K stages whose copies were issued
    // Units are dealt to CTAs with a stride of the grid, so at any time the
    // CTAs work on neighbouring units: a few chunks, whose token tiles stay hot
    // in L2 across the CTAs that share them.  Each role loads the descriptor of
    // a unit two units ahead (one unit of a short-K GEMM is shorter than a
    // global load).
    const int total_units = args.num_chunks[0] * units_per_chunk;
    auto chunk_of = [&](int u) -> Chunk {
        return u < total_units ? args.chunks[u / units_per_chunk] : Chunk{};
    };
    // The work items are those units, except that when the last round of
    // units (rem = units mod grid) would leave at least half of the CTAs idle,
    // each of its units is cut along K into split_p pieces of at least
    // kSplitMinStages stages, items split_base + t * split_p + j (piece j of
    // tail unit t), one per CTA.  Every role derives the same schedule.
    int split_base = total_units;
    int split_p = 1;
    {
        const int grid = static_cast<int>(gridDim.x);
        const int rem = total_units % grid;
        const int slots = args.split_slots < grid ? args.split_slots : grid;
        if (rem > 0 && slots >= 2 * rem && tpu == 1) {
            int p = slots / rem;
            if (p > KT / kSplitMinStages)
                p = KT / kSplitMinStages;
            if (p >= 2) {
                split_base = total_units - rem;
                split_p = p;
            }
        }
    }
    const int total_items = split_base + (total_units - split_base) * split_p;
    auto item_of = [&](int v) -> WorkItem {
        WorkItem it;
        if (v < split_base) {
            it.unit = v;
            it.k0 = 0;
            it.k1 = KT;
            it.piece = -1;
            it.tail = 0;
        } else {
            const int r = v - split_base;
            it.tail = r / split_p;
            it.piece = r - it.tail * split_p;
            it.unit = split_base + it.tail;
            it.k0 = it.piece * KT / split_p;
            it.k1 = (it.piece + 1) * KT / split_p;
        }
        return it;
    };
    auto chunk_of_item = [&](int v) -> Chunk { return chunk_of(item_of(v).unit); };
    int* err = args.err;
    // waits off the critical path (producers, epilogue)
    auto wait_side = [&](uint32_t bar, uint32_t parity) -> bool {
        if constexpr (C::COLD_WAITS)
            return mbar_wait_cold(bar, parity, abort_flag, err);
        else
            return mbar_wait(bar, parity, abort_flag, err);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        const uint64_t pol = policy_evict_first();
        int g = 0;
        bool ok = true;
        Chunk next = chunk_of_item(blockIdx.x);
        Chunk next2 = chunk_of_item(blockIdx.x + gridDim.x);
        for (int v = blockIdx.x; v < total_items && ok; v += gridDim.x) {
            const WorkItem it = item_of(v);
            const Chunk ch = next;
            next = next2;
            next2 = chunk_of_item(v + 2 * gridDim.x);
            const int nt0 = (it.unit % units_per_chunk) * tpu;
            const int e = ch.expert;
            // K stage by K stage, the unit's tiles in turn
            for (int ks = it.k0, nt = nt0; ks < it.k1 && ok; ++g) {
                // first weight row of the tile: gate_up takes rows [row0, row0 + 64)
                // (gate) and the same 64 rows I further on (up) as one 3-D box
                const int row0 = C::GATE_UP ? e * args.N + nt * 64 : e * args.N + nt * 128;
                const int s = g % C::KS;
                if (!wait_side(codes_empty(s), ((g / C::KS) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                const uint32_t dst = sbase + C::OFF_CODES + s * C::CODE_STAGE;
                const uint32_t sdst = sbase + C::OFF_SCALES + s * C::SCALE_STAGE;
                // prepacked: the stage's block (BK 256), or half h of it (BK 128)
                const uint8_t* pblk = nullptr;
                if constexpr (PK)
                    pblk = args.pk + ((static_cast<int64_t>(e) * n_tiles + nt) * pack_kblocks(args.K) +
                                      ks / (256 / C::BK)) *
                                         kPackBlockBytes;
                const int ph = C::BK == 256 ? 0 : (ks & 1);
                if (PK && lane == 0) {
                    mbar_arrive_expect_tx(codes_full(s),
                                          C::CODE_STAGE + (C::SCALES_TMA ? C::SCALE_STAGE : 0));
                    bulk_load(dst, pblk + ph * 8192, C::CODE_STAGE, codes_full(s), pol);
                    if constexpr (C::SCALES_TMA)
                        bulk_load(sdst, pblk + kPackCodeBytes, C::SCALE_STAGE, codes_full(s), pol);
                } else if (!PK && lane == 0) {
                    mbar_arrive_expect_tx(codes_full(s),
                                          C::CODE_STAGE + (C::SCALES_TMA ? C::SCALE_STAGE : 0));
                    const int kb = ks * (C::BK / 128);
                    if constexpr (C::GATE_UP)
                        tma_load_4d(dst, &codes_map, 0, row0, 0, kb, codes_full(s), pol);
                    else
                        tma_load_3d(dst, &codes_map, 0, row0, kb, codes_full(s), pol);
                    if constexpr (C::SCALES_TMA) {
                        if constexpr (C::GATE_UP)
                            tma_load_3d(sdst, &scales_map, ks * (C::BK / 32), row0, 0, codes_full(s), pol);
                        else
                            tma_load_2d(sdst, &scales_map, ks * (C::BK / 32), row0, codes_full(s), pol);
                    }
                }
                if constexpr (!C::SCALES_TMA) {
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr) {
                        const int r = lane + 32 * rr;
                        const int grow = C::GATE_UP ? row0 + (r < 64 ? r : args.I + r - 64) : row0 + r;
                        const void* src =
                            PK  ? static_cast<const void*>(pblk + kPackCodeBytes + r * 16 + ph * 8)
                                : static_cast<const void*>(args.scales +
                                                           static_cast<int64_t>(grow) * (args.K / 32) +
                                                           ks * (C::BK / 32));
                        cp_async_8(sdst + r * C::SCALE_ROW, src);
                    }
                    cp_async_arrive_noinc(codes_full(s));
                }
                __syncwarp();
                if (++nt == nt0 + tpu) {
                    nt = nt0;
                    ++ks;
                }
            }
        }
        issued_stages = g;
    } else if (warp == 1) {
        // ----------------------------------------------------------- token producer
        if constexpr (!C::GATE_UP)
            pdl_wait();
        const uint64_t pol = policy_evict_last();
        int g = 0;
        bool ok = true;
        Chunk next = chunk_of_item(blockIdx.x);
        Chunk next2 = chunk_of_item(blockIdx.x + gridDim.x);
        for (int v = blockIdx.x; v < total_items && ok; v += gridDim.x) {
            const WorkItem it = item_of(v);
            const int row0 = next.brow0;  // (token rows: compacted for the masked gate/up)
            // boxes of B_BOX_ROWS rows, as many as the token tile needs
            const int nbox = ((next.nrows + 15) / 16 * 16 + C::B_BOX_ROWS - 1) / C::B_BOX_ROWS;
            next = next2;
            next2 = chunk_of_item(v + 2 * gridDim.x);
            for (int ks = it.k0; ks < it.k1; ++ks, ++g) {
                const int s = g % C::BS;
                const uint32_t fbar = C::FUSED_RINGS ? a_full(s) : b_full(s);
                if (!wait_side(C::FUSED_RINGS ? a_empty(s) : b_empty(s), ((g / C::BS) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t dst = sbase + C::OFF_B + s * C::B_STAGE;
                    if constexpr (C::B_3D) {
                        mbar_arrive_expect_tx(fbar, C::B_STAGE);
                        tma_load_3d(dst, &b_map, 0, row0, ks * (C::BK / 64), fbar, pol);
                    } else {
                        mbar_arrive_expect_tx(fbar, C::B_KBLK * nbox * C::B_BOX_ROWS * 128);
#pragma unroll
                        for (int kb = 0; kb < C::B_KBLK; ++kb)
                            for (int ib = 0; ib < nbox; ++ib)
                                tma_load_2d(dst + kb * C::B_REGION + ib * (C::B_BOX_ROWS * 128), &b_map,
                                            ks * C::BK + kb * 64, row0 + ib * C::B_BOX_ROWS, fbar, pol);
                    }
                }
                __syncwarp();
            }
        }
        issued_stages = g;
    } else if (warp == 2) {
        // ------------------------------------------------------------- MMA issuer
        // The whole warp walks the schedule (so every operand stays warp-uniform)
        // and elect.sync picks the lane that issues each MMA and commit.
        int ga = 0;  // A stages (one per K stage and tile)
        int gb = 0;  // token stages (one per K stage)
        int pc = 0;  // accumulation chains (one per unit, or one per PS stages)
        int issued = 0;
        bool ok = true;
        Chunk next = chunk_of_item(blockIdx.x);
        Chunk next2 = chunk_of_item(blockIdx.x + gridDim.x);
        for (int v = blockIdx.x; v < total_items && ok; v += gridDim.x) {
            const WorkItem it = item_of(v);
            const Chunk ch = next;
            next = next2;
            next2 = chunk_of_item(v + 2 * gridDim.x);
            const int ntok16 = (ch.nrows + 15) & ~15;
            const uint32_t idesc = idesc_bf16_f32(128, ntok16);
            if constexpr (C::TS) {
                // one K stage (the host picks these configurations only for K =
                // BK): the unit's token stage, then each tile into the next buffer
                const int sb = gb % C::BS;
                if (!__all_sync(0xffffffffu, mbar_wait(b_full(sb), (gb / C::BS) & 1, abort_flag, err))) {
                    ok = false;
                    break;
                }
                const uint64_t bdesc = smem_desc_sw128(sbase + C::OFF_B + sb * C::B_STAGE);
                for (int t = 0; t < tpu; ++t, ++ga, ++pc) {
                    const int acc = pc % C::ACCB;
                    const int sa = ga % C::AS;
                    const bool got = mbar_wait(d_empty(acc), ((pc / C::ACCB) & 1) ^ 1, abort_flag, err) &&
                                     mbar_wait(a_full(sa), (ga / C::AS) & 1, abort_flag, err);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    mma_stage16<C::B_REGION / 16>(tmem + C::D_COL0 + acc * C::ACCW, tmem + sa * C::A_COLS,
                                                  bdesc, idesc, 0u);
                    issued = 1;
                    mma_commit_elect(a_empty(sa));
                    mma_commit_elect(d_full(acc));
                }
                if (!ok)
                    break;
                mma_commit_elect(b_empty(sb));
                ++gb;
                continue;
            }
          for (int g0 = it.k0, g1; g0 < it.k1 && ok; g0 = g1, ++pc) {
            g1 = (C::PS > 0 && g0 + C::PS < it.k1) ? g0 + C::PS : it.k1;
            const int acc = pc % C::ACCB;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(d_empty(acc), ((pc / C::ACCB) & 1) ^ 1, abort_flag, err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + C::D_COL0 + acc * C::ACCW;
            for (int ks = g0; ks < g1 && ok; ++ks, ++gb) {
                const int sb = gb % C::BS;
                const uint64_t bdesc = smem_desc_sw128(sbase + C::OFF_B + sb * C::B_STAGE);
                const uint32_t accum = ks != g0 ? 1u : 0u;
                if constexpr (C::TPU_MAX == 1) {
                    const int sa = ga % C::AS;
                    const bool got = mbar_wait(a_full(sa), (ga / C::AS) & 1, abort_flag, err) &&
                                     (C::FUSED_RINGS || mbar_wait(b_full(sb), (gb / C::BS) & 1, abort_flag, err));
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = tmem + sa * C::A_COLS;
                    if constexpr (C::BK == 256)
                        mma_stage16<C::B_REGION / 16>(d_tmem, a_base, bdesc, idesc, accum);
                    else
                        mma_stage8<C::B_REGION / 16>(d_tmem, a_base, bdesc, idesc, accum);
                    issued = 1;
                    mma_commit_elect(a_empty(sa));
                    ++ga;
                } else {
                    if (!__all_sync(0xffffffffu, mbar_wait(b_full(sb), (gb / C::BS) & 1, abort_flag, err))) {
                        ok = false;
                        break;
                    }
                    for (int t = 0; t < tpu; ++t, ++ga) {
                        const int sa = ga % C::AS;
                        if (!__all_sync(0xffffffffu, mbar_wait(a_full(sa), (ga / C::AS) & 1, abort_flag, err))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_base = tmem + sa * C::A_COLS;
                        mma_stage16<C::B_REGION / 16>(d_tmem + t * C::MAXN, a_base, bdesc, idesc, accum);
                        issued = 1;
                        mma_commit_elect(a_empty(sa));
                    }
                }
                if (ok && !C::FUSED_RINGS)
                    mma_commit_elect(b_empty(sb));
            }
            if (!ok)
                break;
            mma_commit_elect(d_full(acc));
          }
        }
        if (!ok && issued) {
            // drain tensor-core work in flight before TMEM is released
            mma_commit_elect(drain_bar);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else if ((warp >= 4 && warp < 8) || warp >= C::EPI1_WARP) {
        // --------------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int egrp = warp >= C::EPI1_WARP ? 1 : 0;  // epilogue group: units i with i % EPI_GROUPS == egrp
        const int et = threadIdx.x - (egrp ? 32 * C::EPI1_WARP : 128);  // 0..127 inside the epilogue group
        int esync = 0;
        const uint32_t epi_bar = epi_bar0 + 8u * egrp;
        // the four warps of the group meet here (bounded, unlike bar.sync)
        auto epi_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(epi_bar);
            const bool r = wait_side(epi_bar, esync & 1);
            ++esync;
            return r;
        };
        // down: the pair, token and weight of each column come from the
        // per-row records prep wrote.  Every epilogue warp holds the unit's
        // records itself (lane l: columns l, l + 32, ...) and takes them by
        // warp shuffle, so the down path needs no cross-warp rendezvous.  The
        // records of the next unit are loaded one unit ahead (their chunk
        // descriptor two ahead), so no unit waits on a global load.
        const bool per_pair = !C::GATE_UP && (args.epi & (kEpiStorePair | kEpiReduceTok)) != 0;
        constexpr int MPT = C::MAXN / 32;  // record columns per lane
        int4 meta_next[MPT];
        auto load_meta = [&](const Chunk& c_, int4* dst) {
#pragma unroll
            for (int k = 0; k < MPT; ++k) {
                const int col = lane + 32 * k;
                dst[k] = (per_pair && col < c_.nrows) ? args.row_meta[c_.row0 + col]
                                                      : make_int4(-1, 0, 0, 0);
            }
        };
        constexpr int EG = C::EPI_GROUPS;
        // the epilogue groups take every EG-th unit, or (token-stationary
        // units) every unit and in it every EG-th tile
        constexpr int US = C::TS ? 1 : EG;
        const int ev0 = C::TS ? 0 : egrp;
        // accumulation chains taken (PS > 0: several per unit; TS: one per tile,
        // counted over both groups)
        int i = ev0;
        Chunk c_cur = chunk_of_item(blockIdx.x + ev0 * gridDim.x);
        Chunk c_nxt = chunk_of_item(blockIdx.x + (ev0 + US) * gridDim.x);
        load_meta(c_cur, meta_next);
        constexpr int kSlotFloats = 128 * C::MAXN;
        // down: the epilogue of one accumulator buffer holding weight tiles
        // nt0u .. nt0u + tpuu - 1 of chunk ch (tpuu > 1: consecutive column
        // ranges of the buffer); it goes back to the MMA after its last read
        auto down_blocks = [&](const Chunk& ch, int nt0u, int tpuu, uint32_t dbase, int acc,
                               const int4* meta_cur) {
            const int ntok = ch.nrows;
            const int ntok16 = (ntok + 15) & ~15;
            // Each 32-row x 16-column block goes through a shared tile so that
            // lane l owns rows 4 (l % 8) .. +3 of columns l / 8 + {0, 4, 8, 12}:
            // 16-byte stores and vector reductions instead of one 4-byte
            // access per lane and column.
            const int N = args.N;
            float* tile = reinterpret_cast<float*>(smem + C::OFF_EPIT) + (egrp * 4 + q) * 16 * 32;
            const int m4 = (lane & 7) * 4;
            const int cg = lane >> 3;
            // one 16-column block of tile t: accumulator columns -> shared tile
            // -> per-pair stores / token reductions / row stores
            auto block = [&](int t, int c0, int4 mrec) {
                const int nq = (nt0u + t) * 128 + q * 32;
                uint32_t v[16];
                tmem_ld_x16(dbase + t * C::MAXN + c0, v);
                tmem_wait_ld();
                if (t == tpuu - 1 && c0 + 16 >= ntok16) {
                    // last block read: the accumulator goes back to the MMA
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(d_empty(acc));
                }
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    tile[j * 32 + lane] = __uint_as_float(v[j]) * kRescale;
                __syncwarp();
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    const int j = cg + 4 * ii;
                    const int c = c0 + j;
                    const int src = c & 31;
                    const int p = __shfl_sync(0xffffffffu, mrec.x, src);
                    const int tok = __shfl_sync(0xffffffffu, mrec.y, src);
                    const float w = __int_as_float(__shfl_sync(0xffffffffu, mrec.z, src));
                    if (c >= ntok)
                        continue;
                    const float4 y = *reinterpret_cast<const float4*>(tile + j * 32 + m4);
                    if (args.epi & kEpiStoreRows) {
                        uint2 o;
                        o.x = bf16x2_pack_rn(y.x, y.y);
                        o.y = bf16x2_pack_rn(y.z, y.w);
                        *reinterpret_cast<uint2*>(args.rows_out + static_cast<int64_t>(ch.row0 + c) * N + nq +
                                                  m4) = o;
                    }
                    if (per_pair && p >= 0) {
                        if (args.epi & kEpiStorePair)
                            *reinterpret_cast<float4*>(args.y_pairs + static_cast<int64_t>(p) * N + nq + m4) = y;
                        if (args.epi & kEpiReduceTok)
                            red_add_v4_f32(args.out_acc + static_cast<int64_t>(tok) * N + nq + m4, w * y.x,
                                           w * y.y, w * y.z, w * y.w);
                    }
                }
                __syncwarp();  // the tile is rewritten by the next block
            };
            if constexpr (C::COLD_WAITS) {
                // (rolled loops for the BK 256 tiles: their epilogue runs once
                // per short unit, and its code competes for the instruction
                // cache with every other role's)
#pragma unroll 1
                for (int t = 0; t < tpuu; ++t) {
#pragma unroll 1
                    for (int c0 = 0; c0 < ntok16; c0 += 16) {
                        // columns c0 .. c0 + 15 sit in one lane group: records meta_cur[c0 / 32]
                        int4 mrec = meta_cur[0];
#pragma unroll
                        for (int k = 1; k < MPT; ++k)
                            if (c0 >= 32 * k)
                                mrec = meta_cur[k];
                        block(t, c0, mrec);
                    }
                }
            } else {
                // (the prefill tile's long units: unrolled over the token tile)
#pragma unroll
                for (int c0 = 0; c0 < C::MAXN; c0 += 16) {
                    if (c0 >= ntok16)
                        break;
                    block(0, c0, meta_cur[c0 / 32]);
                }
            }
        };
        for (int v = blockIdx.x + ev0 * gridDim.x; v < total_items;
             v += US * gridDim.x, i += C::TS ? 0 : EG) {
            const WorkItem it = item_of(v);
            const Chunk ch = c_cur;
            int4 meta_cur[MPT];
#pragma unroll
            for (int k = 0; k < MPT; ++k)
                meta_cur[k] = meta_next[k];
            load_meta(c_nxt, meta_next);
            const Chunk c_nn = chunk_of_item(v + 2 * US * gridDim.x);
            const int nt0 = (it.unit % units_per_chunk) * tpu;
            const int ntok = ch.nrows;
            const int ntok16 = (ntok + 15) & ~15;
            c_cur = c_nxt;
            c_nxt = c_nn;
            if constexpr (C::TS) {
                // one K stage; tile t of the unit is accumulation chain i, in
                // buffer i % ACCB, drained by group i % EG
                bool okt = true;
                for (int t = 0; t < tpu; ++t, ++i) {
                    if (i % EG != egrp)
                        continue;
                    const int acct = i % C::ACCB;
                    if (!wait_side(d_full(acct), (i / C::ACCB) & 1)) {
                        okt = false;
                        break;
                    }
                    tc_fence_after();
                    down_blocks(ch, nt0 + t, 1,
                                tmem + (static_cast<uint32_t>(q * 32) << 16) + C::D_COL0 + acct * C::ACCW,
                                acct, meta_cur);
                }
                if (!okt)
                    break;
                continue;
            }
            int acc = i % C::ACCB;
            if (!wait_side(d_full(acc), (i / C::ACCB) & 1))
                break;
            tc_fence_after();
            if constexpr (C::PS > 0) {
                // add each finished partial into the next one; the last holds the sum
                bool okp = true;
                for (int g0 = it.k0 + C::PS; g0 < it.k1; g0 += C::PS) {
                    const int nacc = (i + 1) % C::ACCB;
                    if (!wait_side(d_full(nacc), ((i + 1) / C::ACCB) & 1)) {
                        okp = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16) + C::D_COL0;
                    const uint32_t src = lane_base + acc * C::ACCW;
                    const uint32_t dst = lane_base + nacc * C::ACCW;
                    // 16 columns per load wait: two 16-column pairs per wait
                    // (64 registers) made every gate/up instance spill, and the
                    // spill-free form ran faster where chains are long (prefill
                    // gate/up 406 -> 400 us, TP8 T=2048 205 -> 201 us)
                    for (int c0 = 0; c0 < ntok16; c0 += 16) {
                        uint32_t a0[16], b0[16];
                        tmem_ld_x16(src + c0, a0);
                        tmem_ld_x16(dst + c0, b0);
                        tmem_wait_ld();
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            b0[jj] = __float_as_uint(__uint_as_float(a0[jj]) + __uint_as_float(b0[jj]));
                        tmem_st_x16(dst + c0, b0);
                    }
                    tmem_wait_st();
                    // the earlier partial's buffer goes back to the MMA
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(d_empty(acc));
                    ++i;
                    acc = nacc;
                }
                if (!okp)
                    break;
            }
            const uint32_t dbase =
                tmem + (static_cast<uint32_t>(q * 32) << 16) + C::D_COL0 + acc * C::ACCW;
            // A piece of a split unit: the accumulator goes to the piece's slot
            // (column-major, so a warp stores 128 contiguous bytes per column).
            // The last piece of the unit to get here adds the unit's slots in
            // piece order back into its accumulator and runs the epilogue below
            // on it; the other pieces hand their accumulator back to the MMA.
            if (it.piece >= 0) {
                const float* slots = args.split_part + static_cast<int64_t>(it.tail * split_p) * kSlotFloats +
                                     q * 32 + lane;
                float* mine = args.split_part + static_cast<int64_t>(it.tail * split_p + it.piece) * kSlotFloats +
                              q * 32 + lane;
                for (int c0 = 0; c0 < ntok16; c0 += 16) {
                    uint32_t vv[16];
                    tmem_ld_x16(dbase + c0, vv);
                    tmem_wait_ld();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        __stcg(mine + (c0 + jj) * 128, __uint_as_float(vv[jj]));
                }
                __threadfence();  // the slot is visible before the count says so
                if (!epi_sync())
                    break;
                if (et == 0) {
                    const int before = atomicAdd(args.split_cnt + it.tail, 1);
                    __threadfence();  // the other pieces' slots are read after their counts
                    split_last[egrp] = before == split_p - 1;
                }
                if (!epi_sync())
                    break;
                if (!split_last[egrp]) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(d_empty(acc));
                    continue;
                }
                for (int c0 = 0; c0 < ntok16; c0 += 16) {
                    float sum[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        sum[jj] = __ldcg(slots + (c0 + jj) * 128);
                    for (int j = 1; j < split_p; ++j) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            sum[jj] += __ldcg(slots + static_cast<int64_t>(j) * kSlotFloats + (c0 + jj) * 128);
                    }
                    uint32_t vv[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        vv[jj] = __float_as_uint(sum[jj]);
                    tmem_st_x16(dbase + c0, vv);
                }
                tmem_wait_st();
            }
            if constexpr (C::GATE_UP) {
                // lanes (l, l^8): gate and up of channel 16q + 8(l>>4) + (l&7)
                __nv_bfloat16* hs = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_HS);
                const int chl = 16 * q + 8 * (lane >> 4) + (lane & 7);
                const bool is_gate = (lane & 15) < 8;
                for (int c0 = 0; c0 < ntok16; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld_x16(dbase + c0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const float mine = __uint_as_float(v[jj]) * kRescale;
                        const float other = __shfl_xor_sync(0xffffffffu, mine, 8);
                        if (is_gate) {
                            // fast exp / divide: a few fp32 ulp, far below the bf16 rounding of h
                            const float silu = __fdividef(mine, 1.0f + __expf(-mine));
                            hs[(c0 + jj) * 64 + chl] = __float2bfloat16_rn(silu * other);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(d_empty(acc));
                if (!epi_sync())
                    break;
                const int64_t col0 = static_cast<int64_t>(nt0) * 64;
                // 16 rows per pass of the 128 threads (8 x 16 bytes per row).  An
                // unpaired row's token row was never written, so its h is whatever
                // the MMA made of it: it is stored as zeros.  Every pair record of
                // the thread's rows is loaded before the first store, so the pass
                // waits for one global load, not one per row.
                constexpr int kPasses = C::MAXN / 16;
                bool keep[kPasses];
#pragma unroll
                for (int ps = 0; ps < kPasses; ++ps) {
                    const int c = (et >> 3) + 16 * ps;
                    keep[ps] = true;
                    if (args.h_zero_unpaired && c < ntok) {
                        const int p = args.pair_of_row[ch.row0 + c];
                        keep[ps] = p >= 0 && p < args.num_pairs;
                    }
                }
                const int part = et & 7;
#pragma unroll
                for (int ps = 0; ps < kPasses; ++ps) {
                    const int c = (et >> 3) + 16 * ps;
                    if (c < ntok) {
                        uint4 val = *reinterpret_cast<const uint4*>(hs + c * 64 + part * 8);
                        if (!keep[ps])
                            val = make_uint4(0u, 0u, 0u, 0u);
                        *reinterpret_cast<uint4*>(args.h_out + static_cast<int64_t>(ch.row0 + c) * args.ld_h +
                                                  col0 + part * 8) = val;
                    }
                }
                if (args.pair_row != nullptr && nt0 == 0) {
                    for (int c = et; c < ntok; c += 128) {
                        const int p = args.pair_of_row[ch.row0 + c];
                        if (p >= 0 && p < args.num_pairs)
                            args.pair_row[p] = ch.row0 + c;
                    }
                }
                if (!epi_sync())
                    break;
            } else {
                down_blocks(ch, nt0, tpu, dbase, acc, meta_cur);
            }
        }
    } else if (warp >= 8) {
        // ---------------------------------------------------------------- dequant
        // The DQW warps of each TMEM lane quadrant (warps q+8, q+12 [, q+16])
        // take K stages in order from a shared counter, each the next one not
        // yet taken, so none waits for another's turn.
        const int q = warp & 3;
        int srow;
        if constexpr (C::GATE_UP)
            srow = (((lane & 15) >= 8) ? 64 : 0) + 16 * q + 8 * (lane >> 4) + (lane & 7);
        else
            srow = q * 32 + lane;
        const uint32_t tlane = static_cast<uint32_t>(q * 32) << 16;
        int total_stages = 0;
        for (int v = blockIdx.x; v < total_items; v += gridDim.x) {
            const WorkItem it = item_of(v);
            total_stages += (it.k1 - it.k0) * tpu;
        }
        bool ok = true;
        for (;;) {
            {
                int g = 0;
                if (lane == 0)
                    g = atomicAdd(&stage_ctr[q], 1);
                g = __shfl_sync(0xffffffffu, g, 0);
                if (g >= total_stages)
                    break;
                const int s = g % C::KS;
                if (!mbar_wait(codes_full(s), (g / C::KS) & 1, abort_flag, err)) {
                    ok = false;
                    break;
                }
                const uint8_t* cstage = smem + C::OFF_CODES + s * C::CODE_STAGE;
                uint32_t sc[C::BK / 64];  // two bf16 scales per 32-bit word
                {
                    const uint8_t* sp = smem + C::OFF_SCALES + s * C::SCALE_STAGE + srow * C::SCALE_ROW;
                    if constexpr (C::BK == 256) {
                        const uint4 v = *reinterpret_cast<const uint4*>(sp);
                        sc[0] = v.x;
                        sc[1] = v.y;
                        sc[2] = v.z;
                        sc[3] = v.w;
                    } else {
                        const uint2 v = *reinterpret_cast<const uint2*>(sp);
                        sc[0] = v.x;
                        sc[1] = v.y;
                    }
                }
                const int sa = g % C::AS;
                if (!mbar_wait(a_empty(sa), ((g / C::AS) & 1) ^ 1, abort_flag, err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // One scale group per step: 32 elements = one 16-byte chunk of codes =
                // 16 TMEM columns.  Codes are read from shared memory group by group
                // (not all up front) so the stores of one group overlap the
                // arithmetic of the next without running out of registers.
                if constexpr (FMT == kFmtInt4) {
#pragma unroll
                    for (int grp = 0; grp < C::BK / 32; ++grp) {
                        const uint4 v = *reinterpret_cast<const uint4*>(cstage + code_piece_offset(grp, srow));
                        const ScalePair sp =
                            scale_pair(__byte_perm(sc[grp >> 1], 0, (grp & 1) ? 0x3232 : 0x1010));
                        uint32_t o[16];
                        dequant_word(v.x, sp, &o[0]);
                        dequant_word(v.y, sp, &o[4]);
                        dequant_word(v.z, sp, &o[8]);
                        dequant_word(v.w, sp, &o[12]);
                        tmem_st_x16(tmem + tlane + sa * C::A_COLS + grp * 16, o);
                    }
                } else {
                    // the widened scales are 2^(e-127) (or NaN for e = 255): a scale
                    // byte above 128 is a bf16 value above 2 (bits above 0x4000)
                    bool big = false;
#pragma unroll
                    for (int i = 0; i < C::BK / 64; ++i)
                        big = big || (sc[i] & 0x7FFFu) > 0x4000u || ((sc[i] >> 16) & 0x7FFFu) > 0x4000u;
                    if (!__any_sync(0xffffffffu, big)) {
#pragma unroll
                        for (int grp = 0; grp < C::BK / 32; ++grp) {
                            const uint4 v = *reinterpret_cast<const uint4*>(cstage + code_piece_offset(grp, srow));
                            // (2^(e-127), 2^(e-127)) * 2^126 = 2^(e-1), exact
                            const uint32_t m = bf16x2_mul(
                                __byte_perm(sc[grp >> 1], 0, (grp & 1) ? 0x3232 : 0x1010), 0x7E807E80u);
                            uint32_t o[16];
                            dequant_word_mx(v.x, m, &o[0]);
                            dequant_word_mx(v.y, m, &o[4]);
                            dequant_word_mx(v.z, m, &o[8]);
                            dequant_word_mx(v.w, m, &o[12]);
                            tmem_st_x16(tmem + tlane + sa * C::A_COLS + grp * 16, o);
                        }
                    } else {
#pragma unroll
                        for (int grp = 0; grp < C::BK / 32; ++grp) {
                            const uint4 v = *reinterpret_cast<const uint4*>(cstage + code_piece_offset(grp, srow));
                            // 2^(e-127) * 2^-1 = 2^(e-128), exact (a subnormal for e = 0)
                            const uint32_t m2 = bf16x2_mul(
                                __byte_perm(sc[grp >> 1], 0, (grp & 1) ? 0x3232 : 0x1010), 0x3F003F00u);
                            uint32_t o[16];
                            dequant_word_mx2(v.x, m2, &o[0]);
                            dequant_word_mx2(v.y, m2, &o[4]);
                            dequant_word_mx2(v.z, m2, &o[8]);
                            dequant_word_mx2(v.w, m2, &o[12]);
                            tmem_st_x16(tmem + tlane + sa * C::A_COLS + grp * 16, o);
                        }
                    }
                }
                // The next TMA into this code stage writes through the async proxy;
                // order these generic-proxy reads before it (without the fence a
                // few lanes intermittently read the following stage's codes).
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(codes_empty(s));
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                // (test hook: one arrival dropped so that the MMA's bounded wait expires)
                const bool drop = args.test_skip_arrive && blockIdx.x == 0 && q == 0 && g == 0;
                if (lane == 0 && !drop)
                    mbar_arrive(a_full(sa));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // An aborted CTA may leave copies it issued but nobody consumed: the
        // producers wait (bounded) for the last stages they issued to land, so
        // the CTA does not end while the TMA engine still writes its shared
        // memory.
        if (warp == 0 || warp == 1) {
            const int depth = warp == 0 ? C::KS : C::BS;
            if (lane == 0)
                for (int gg = issued_stages > depth ? issued_stages - depth : 0; gg < issued_stages; ++gg)
                    mbar_drain(warp == 0 ? codes_full(gg % C::KS)
                                         : (C::FUSED_RINGS ? a_full(gg % C::AS) : b_full(gg % C::BS)),
                               (gg / depth) & 1);
            asm volatile("cp.async.wait_all;" ::: "memory");
            __syncwarp();
        }
    }
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace chord
