/*
 * oracle.c -- plain, slow CPU oracle of the W4A16 INT4 Mixture-of-Experts
 * expert computation.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, __graft_entry__.smoke() and the
 * CPU-baseline / reference legs of bench.py load this library.  The CUDA path
 * never calls it and shares no code with it.
 *
 * What it follows (page: "vLLM x Novita AI: Chord W4A16 INT4 MoE kernels for
 * Kimi K2.x", novita.ai):
 *   - TL;DR: BF16 activations, INT4 weights, group-32 scales.
 *   - "vLLM integration": the uint4 / group-32 / BF16-scale schema; routing
 *     consumed as moe_align_block_size buffers (sorted_ids / expert_ids /
 *     num_tokens_padded), over-allocated.
 *   - "Kernel optimisation / H200 and Blackwell indexed decode": dequant is
 *     subtract-then-scale, w = (q - 8) * scale, keeping the unfused BF16
 *     rounding order.
 *   - "Kernel optimisation / grouped SM90 kernels" and Fig. 3: indexed layout
 *     (padding lives in the index as a sentinel), contiguous layout (rows per
 *     expert padded to 128 with m_indices = -1 on padding), masked layout
 *     (fixed row budget per expert, masked_m valid counts, flat output).
 *   - "Measurement": gate_up and down are the two GEMM calls of a layer.
 * The expert MLP itself (gate/up GEMM, SiLU(gate) * up, down GEMM, top-k
 * weighted sum per token) is the standard MoE layer the page accelerates.
 *
 * Readings where the page is silent (each is one choice, applied everywhere):
 *   R1 codes: 8 per int32 along K, element c = 8w+i in bits [4i, 4i+4).
 *   R2 zero point fixed at 8; no per-group zero.
 *   R3 dequant: W = RNE_bf16( float(q-8) * float(s) ), one rounding (the
 *      product of a 4-bit integer and an 8-bit significand is exact in fp32).
 *   R4 scale groups: 32 consecutive input channels, scales [E, N, K/32].
 *   R5 fused gate/up: rows 0..I-1 are gate, rows I..2I-1 are up.
 *   R6 FP32 accumulation in ascending input channel; products of two bf16
 *      values are exact in fp32.
 *   R7 g and u are not rounded before SiLU; h = RNE_bf16(silu(g) * u),
 *      silu(v) = v / (1 + exp(-v)) in fp32.
 *   R8 per-pair down output y kept in fp32.
 *   R9 router weights applied in the combine, after down, in fp32, summed in
 *      ascending slot order over the local slots; out = RNE_bf16(sum), 0 when
 *      the token has no local slot.
 *   R10 align: experts in ascending local id, pairs p = t*k + j ascending
 *      inside an expert, each expert padded to a multiple of block_m with the
 *      sentinel T*k, empty experts get no block, sorted_ids tail = sentinel,
 *      expert_ids tail = -1.
 *   R11 pairs routed to a non-local expert (expert_map = -1) are dropped.
 *   R14 router (the step before align; the tiny workload's routing rule): per token
 *      the k largest logits, ties to the lower expert id, in descending order;
 *      weight of a selected expert = its softmax probability over all
 *      E_global experts, renormalised over the k selected when asked.
 * MXFP4 weights (the variant on the vLLM Kimi K3 page, "MXFP4 MoE"; the
 * element and scale encodings are those of the OCP Microscaling formats the
 * name refers to): with oracle_set_weight_format(1) every code is an FP4
 * E2M1 number (bit 3 sign, bits 2..1 exponent with bias 1, bit 0 mantissa;
 * exponent 0 is subnormal, m * 2^-1) and every group of 32 input channels
 * shares one E8M0 scale byte s (2^(s - 127), s = 255 is NaN), stored uint8
 * [E, N, K/32] in place of the bf16 scales.  W = RNE_bf16(e2m1(q) * 2^(s-127)),
 * which is exact unless it overflows bf16.  The page names a "SiTU"
 * activation for this variant without defining it; the MLP here keeps
 * SiLU(gate) * up (R7).
 * Prepack (the storage order of chord_w4a16_prepack, stated in the library's
 * header chord.h; an offline rearrangement that the pages' grouped kernels
 * also make, "Kernel optimisation / grouped SM90 kernels"): no arithmetic,
 * only where each code and scale goes, written out here loop by loop.
 *
 * Every function below is pinned by the CPU tests (closed forms, exhaustive
 * dequant against exact rational rounding, brute-force fp64 evaluation,
 * routing invariants, cross-layout agreement); none is "parity unpinned".
 *
 * Built with -O2 -ffp-contract=off so that every a*b+c stays two roundings
 * exactly as written.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------- */
/* test-only planted mistakes: 0 = none.  The tests set one at a time and     */
/* check that some pin fails; nothing else sets this.                         */
/* ------------------------------------------------------------------------- */
enum {
    MUT_NONE = 0,
    MUT_NIBBLE_HIGH_FIRST = 1, /* R1 violated: element c in bits [28-4i, 32-4i) */
    MUT_GATE_UP_SWAPPED = 2,   /* R5 violated */
    MUT_DEQUANT_FMA = 3,       /* R3 violated: (128+q)*s - bf16(136*s), the folded form */
    MUT_SCALE_GROUP = 4,       /* R4 violated: the next group's scale */
    MUT_ZERO_SIGN = 5,         /* (8 - q) instead of (q - 8) */
    MUT_DROP_WEIGHT = 6,       /* R9 violated: router weight ignored */
    MUT_DROP_LAST_SLOT = 7,    /* combine stops one slot early */
    MUT_ALIGN_DESCENDING = 8,  /* R10 violated: pairs descending inside an expert */
    MUT_SILU_SIGN = 9,         /* silu(v) = v / (1 + exp(v)) */
    MUT_DOWN_TRANSPOSED = 10,  /* down weight read as [I, H] */
    MUT_ALIGN_NO_PAD = 11,     /* segments not padded to block_m */
    MUT_CODE_OFFSET = 12,      /* reads the code of element c+1 */
    MUT_ROUTE_TIE_HIGH = 13,   /* R14 violated: equal logits go to the higher id */
    MUT_ROUTE_NO_RENORM = 14,  /* R14 violated: weights not renormalised */
    MUT_PACK_NO_SWIZZLE = 15,  /* prepack: pieces stored unpermuted */
    MUT_PACK_TILE_ROWS = 16,   /* prepack: gate/up tiles as 128 consecutive rows */
    MUT_MX_SCALE_BIAS = 17,    /* MXFP4: scale 2^(s - 128) instead of 2^(s - 127) */
    MUT_MX_NO_SUBNORMAL = 18,  /* MXFP4: exponent field 0 read as a normal number */
};
static int g_mutation = 0;
void oracle_set_mutation(int m) { g_mutation = m; }
int oracle_get_mutation(void) { return g_mutation; }

/* ------------------------------------------------------------------------- */
/* bf16 <-> fp32                                                             */
/* ------------------------------------------------------------------------- */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest-even of an fp32 value to bf16.  NaN stays NaN (quiet). */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

static float rbf(float f) { return oracle_bf16_to_f32(oracle_f32_to_bf16(f)); }

/* silu(v) = v / (1 + exp(-v)) in fp32 (R7). */
float oracle_silu(float v)
{
    if (g_mutation == MUT_SILU_SIGN)
        return v / (1.0f + expf(v));
    return v / (1.0f + expf(-v));
}

/* ------------------------------------------------------------------------- */
/* threads: a plain parallel-for over independent items                     */
/* ------------------------------------------------------------------------- */
static int g_threads = 0;
void oracle_set_threads(int n) { g_threads = n; }
int oracle_num_threads(void)
{
    if (g_threads > 0)
        return g_threads;
    const char* env = getenv("ORACLE_THREADS");
    if (env && atoi(env) > 0)
        return atoi(env);
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

typedef void (*range_fn)(void* ctx, int64_t begin, int64_t end);
typedef struct {
    range_fn fn;
    void* ctx;
    int64_t begin, end;
} range_job;

static void* range_trampoline(void* p)
{
    range_job* j = (range_job*)p;
    j->fn(j->ctx, j->begin, j->end);
    return NULL;
}

static void parallel_for(int64_t n, range_fn fn, void* ctx)
{
    int nt = oracle_num_threads();
    if (nt > 256)
        nt = 256;
    if (n <= 0)
        return;
    if (nt <= 1 || n == 1) {
        fn(ctx, 0, n);
        return;
    }
    if (nt > n)
        nt = (int)n;
    pthread_t th[256];
    range_job jobs[256];
    int started[256];
    for (int i = 0; i < nt; ++i) {
        jobs[i].fn = fn;
        jobs[i].ctx = ctx;
        jobs[i].begin = n * i / nt;
        jobs[i].end = n * (i + 1) / nt;
        started[i] = pthread_create(&th[i], NULL, range_trampoline, &jobs[i]) == 0;
        if (!started[i])
            fn(ctx, jobs[i].begin, jobs[i].end);
    }
    for (int i = 0; i < nt; ++i)
        if (started[i])
            pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------------- */
/* weights: unpack (R1) and dequantise (R2, R3, R4)                          */
/* ------------------------------------------------------------------------- */
/* 0: INT4 codes with bf16 scales; 1: MXFP4 (E2M1 codes, E8M0 scale bytes) */
static int g_wfmt = 0;
void oracle_set_weight_format(int f) { g_wfmt = f; }
int oracle_get_weight_format(void) { return g_wfmt; }

/* The scale array advanced by idx scales of the current format. */
static const uint16_t* scales_at(const uint16_t* base, int64_t idx)
{
    if (g_wfmt == 1)
        return (const uint16_t*)(const void*)((const uint8_t*)(const void*)base + idx);
    return base + idx;
}

/* FP4 E2M1 value of a 4-bit code (exact in double). */
double oracle_e2m1(int q)
{
    const int sign = (q >> 3) & 1;
    const int ex = (q >> 1) & 3;
    const int man = q & 1;
    double v;
    if (ex == 0 && g_mutation != MUT_MX_NO_SUBNORMAL)
        v = 0.5 * man;                               /* subnormal: m * 2^(1 - bias) / 2 */
    else
        v = ldexp(1.0 + 0.5 * man, ex - 1);          /* (1 + m/2) * 2^(e - bias) */
    return sign ? -v : v;
}

/* E8M0 scale byte -> 2^(s - 127); s = 255 is NaN. */
double oracle_e8m0(int s)
{
    if (s == 255)
        return NAN;
    return ldexp(1.0, s - (g_mutation == MUT_MX_SCALE_BIAS ? 128 : 127));
}

/* 4-bit code of element (n, c) of a [N, K] weight stored as [N, K/8] words. */
int oracle_code(const int32_t* wq, int64_t K, int64_t n, int64_t c)
{
    if (g_mutation == MUT_CODE_OFFSET)
        c = (c + 1) % K;
    uint32_t w = (uint32_t)wq[n * (K / 8) + c / 8];
    int i = (int)(c % 8);
    if (g_mutation == MUT_NIBBLE_HIGH_FIRST)
        i = 7 - i;
    return (int)((w >> (4 * i)) & 0xFu);
}

/* Index of the scale of element (n, c): scales stored [N, K/32]. */
static int64_t scale_index(int64_t K, int64_t n, int64_t c)
{
    int64_t g = c / 32;
    if (g_mutation == MUT_SCALE_GROUP)
        g = (g + 1) % (K / 32);
    return n * (K / 32) + g;
}

static float scale_of(const uint16_t* ws, int64_t K, int64_t n, int64_t c)
{
    return oracle_bf16_to_f32(ws[scale_index(K, n, c)]);
}

/* W[n, c] = RNE_bf16( float(q - 8) * float(s) ): one rounding.  (MXFP4:
 * RNE_bf16( e2m1(q) * 2^(s - 127) ), the product formed in double.) */
float oracle_dequant_one(const int32_t* wq, const uint16_t* ws, int64_t K, int64_t n, int64_t c)
{
    int q = oracle_code(wq, K, n, c);
    if (g_wfmt == 1) {
        const uint8_t* sb = (const uint8_t*)(const void*)ws;
        return rbf((float)(oracle_e2m1(q) * oracle_e8m0(sb[scale_index(K, n, c)])));
    }
    float s = scale_of(ws, K, n, c);
    if (g_mutation == MUT_DEQUANT_FMA) /* magic-number form folded into one multiply-add */
        return rbf((float)(128 + q) * s - rbf(136.0f * s));
    float d = (g_mutation == MUT_ZERO_SIGN) ? (float)(8 - q) : (float)(q - 8);
    return rbf(d * s);
}

typedef struct {
    const int32_t* wq;
    const uint16_t* ws;
    int64_t K;
    float* out;
} dequant_ctx;

static void dequant_rows(void* p, int64_t b, int64_t e)
{
    dequant_ctx* c = (dequant_ctx*)p;
    for (int64_t n = b; n < e; ++n)
        for (int64_t k = 0; k < c->K; ++k)
            c->out[n * c->K + k] = oracle_dequant_one(c->wq, c->ws, c->K, n, k);
}

/* Dequantise a whole [N, K] weight to fp32 values (each one a bf16 value). */
void oracle_dequant(const int32_t* wq, const uint16_t* ws, int64_t N, int64_t K, float* out)
{
    dequant_ctx c = {wq, ws, K, out};
    parallel_for(N, dequant_rows, &c);
}

/* ------------------------------------------------------------------------- */
/* align (R10, R11)                                                          */
/* ------------------------------------------------------------------------- */
/*
 * Router (R14).  logits float [T, E]; writes ids int32 [T, k] (descending
 * logit, ties to the lower id) and w float [T, k]:
 *   w_j = exp(l_j - m) / D,  m = max_e l_e,
 *   D = sum over the k selected of exp(l - m) when renorm, else over all E
 * (the softmax probability, renormalised over the selected experts or not),
 * evaluated in fp64 and rounded to fp32.  Returns -1 on bad sizes.
 */
int oracle_route_topk(const float* logits, int64_t T, int64_t E, int64_t k, int renorm,
                      int32_t* ids, float* w)
{
    if (k < 1 || k > E || E < 1)
        return -1;
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    if (!taken)
        return -1;
    const int do_renorm = renorm && g_mutation != MUT_ROUTE_NO_RENORM;
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        memset(taken, 0, (size_t)E);
        for (int64_t j = 0; j < k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                if (best < 0 || l[e] > l[best] ||
                    (g_mutation == MUT_ROUTE_TIE_HIGH && l[e] == l[best]))
                    best = e;
            }
            taken[best] = 1;
            ids[t * k + j] = (int32_t)best;
        }
        double m = l[0];
        for (int64_t e = 1; e < E; ++e)
            if (l[e] > m)
                m = l[e];
        double denom = 0.0;
        if (do_renorm)
            for (int64_t j = 0; j < k; ++j)
                denom += exp((double)l[ids[t * k + j]] - m);
        else
            for (int64_t e = 0; e < E; ++e)
                denom += exp((double)l[e] - m);
        for (int64_t j = 0; j < k; ++j)
            w[t * k + j] = (float)(exp((double)l[ids[t * k + j]] - m) / denom);
    }
    free(taken);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* prepack                                                                    */
/* ------------------------------------------------------------------------- */
/* weight row held at row r (0..127) of tile t */
static int64_t pack_tile_row(int kind, int64_t N, int64_t t, int64_t r)
{
    if (kind == 1 && g_mutation != MUT_PACK_TILE_ROWS) /* gate/up: 64 gate rows, then 64 up */
        return r < 64 ? 64 * t + r : N / 2 + 64 * t + (r - 64);
    return 128 * t + r;
}

/* one bf16 scale is +-0 or of magnitude in [2^-86, 2^35): exponent field 41..161 */
static int pack_scale_ok(uint16_t s)
{
    const unsigned mag = s & 0x7fffu;
    const unsigned ex = mag >> 7;
    return mag == 0 || (ex >= 41 && ex <= 161);
}

/*
 * kind 1 (gate/up) or 2 (down); w_q int32 [E, N, K/8], w_s bf16 bits
 * [E, N, K/32]; out has 256 + E*(N/128)*(K/256)*18432 bytes.  Header words:
 * magic 0x4B504843, version 1, kind, E, N, K, 18432, flags (bit 0: a scale
 * out of range), zeros.  Block (e, t, j), in that order: for tile row r and
 * K half h, the row's four 16-byte pieces of codes 256j + 128h + 32c .. +31
 * go to offset 8192h + 64r + 16(c ^ ((r >> 1) & 3)); the row's scales of
 * groups 8j .. 8j+7 go to 16384 + 16r.  Returns -1 on bad sizes.
 */
int oracle_prepack(int kind, const int32_t* w_q, const uint16_t* w_s, int64_t E, int64_t N,
                   int64_t K, uint8_t* out)
{
    if ((kind != 1 && kind != 2) || E < 1 || N % 128 != 0 || K % 128 != 0 || N < 128 || K < 128)
        return -1;
    /* a tile has ceil(K / 256) blocks; when K % 256 == 128 the second half of
       the last one (codes and scales) stays zero */
    const int64_t tiles = N / 128, kbs = (K + 255) / 256;
    uint32_t hdr[64];
    memset(hdr, 0, sizeof hdr);
    hdr[0] = 0x4B504843u;
    hdr[1] = 1;
    hdr[2] = (uint32_t)kind;
    hdr[3] = (uint32_t)E;
    hdr[4] = (uint32_t)N;
    hdr[5] = (uint32_t)K;
    hdr[6] = 18432;
    uint8_t* blk = out + 256;
    memset(blk, 0, (size_t)(E * tiles * kbs) * 18432);
    for (int64_t e = 0; e < E; ++e)
        for (int64_t t = 0; t < tiles; ++t)
            for (int64_t j = 0; j < kbs; ++j, blk += 18432) {
                /* halves of this block inside K: 2, or 1 for the tail block */
                const int64_t halves = (256 * j + 256 <= K) ? 2 : 1;
                for (int64_t r = 0; r < 128; ++r) {
                    const int64_t row = e * N + pack_tile_row(kind, N, t, r);
                    for (int64_t h = 0; h < halves; ++h)
                        for (int64_t c = 0; c < 4; ++c) {
                            const int64_t pos =
                                g_mutation == MUT_PACK_NO_SWIZZLE ? c : (c ^ ((r >> 1) & 3));
                            memcpy(blk + 8192 * h + 64 * r + 16 * pos,
                                   w_q + row * (K / 8) + 32 * j + 16 * h + 4 * c, 16);
                        }
                    const uint16_t* sc = w_s + row * (K / 32) + 8 * j;
                    memcpy(blk + 16384 + 16 * r, sc, (size_t)(8 * halves));
                    for (int g = 0; g < 4 * halves; ++g)
                        if (!pack_scale_ok(sc[g]))
                            hdr[7] |= 1u;
                }
            }
    memcpy(out, hdr, sizeof hdr);
    return 0;
}

int64_t oracle_align_capacity(int64_t T, int64_t k, int64_t E_local, int64_t block_m)
{
    if (block_m <= 0)
        return -1;
    int64_t worst = T * k + E_local * (block_m - 1);
    return (worst + block_m - 1) / block_m * block_m;
}

/* local expert of a global id, -1 when not local or out of range */
static int64_t local_of(int32_t gid, int64_t E_global, const int32_t* expert_map, int64_t E_local)
{
    if (gid < 0 || gid >= E_global)
        return -1;
    int64_t l = expert_map ? expert_map[gid] : gid;
    if (l < 0 || l >= E_local)
        return -1;
    return l;
}

/*
 * Group the local (token, slot) pairs by expert.  Returns 0, or -1 when the
 * capacity is too small.  Outputs:
 *   sorted_ids[capacity]        pair ids, sentinel T*k on padding and tail
 *   expert_ids[capacity/block_m] expert of each block, -1 on the tail
 *   num_tokens_padded[0]         sum over experts of ceil(c_e/block_m)*block_m
 */
int oracle_moe_align(const int32_t* topk_ids, int64_t T, int64_t k, int64_t E_global,
                     const int32_t* expert_map, int64_t E_local, int64_t block_m,
                     int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_tokens_padded,
                     int64_t capacity)
{
    const int64_t P = T * k;
    const int32_t sentinel = (int32_t)P;
    if (block_m <= 0 || capacity % block_m != 0)
        return -1;
    for (int64_t i = 0; i < capacity; ++i)
        sorted_ids[i] = sentinel;
    for (int64_t b = 0; b < capacity / block_m; ++b)
        expert_ids[b] = -1;
    int64_t pos = 0;
    for (int64_t e = 0; e < E_local; ++e) {
        int64_t count = 0;
        for (int64_t p = 0; p < P; ++p)
            if (local_of(topk_ids[p], E_global, expert_map, E_local) == e)
                ++count;
        if (count == 0)
            continue;
        int64_t padded = (g_mutation == MUT_ALIGN_NO_PAD)
                             ? count
                             : (count + block_m - 1) / block_m * block_m;
        if (pos + padded > capacity)
            return -1;
        int64_t r = pos;
        if (g_mutation == MUT_ALIGN_DESCENDING) {
            for (int64_t p = P - 1; p >= 0; --p)
                if (local_of(topk_ids[p], E_global, expert_map, E_local) == e)
                    sorted_ids[r++] = (int32_t)p;
        } else {
            for (int64_t p = 0; p < P; ++p)
                if (local_of(topk_ids[p], E_global, expert_map, E_local) == e)
                    sorted_ids[r++] = (int32_t)p;
        }
        for (int64_t b = pos / block_m; b < (pos + padded + block_m - 1) / block_m; ++b)
            expert_ids[b] = (int32_t)e;
        pos += padded;
    }
    num_tokens_padded[0] = (int32_t)pos;
    return 0;
}

/* ------------------------------------------------------------------------- */
/* the expert MLP of a set of rows that share one expert                     */
/* ------------------------------------------------------------------------- */
typedef struct {
    const float* W13;   /* [2I, H] dequantised */
    const float* W2;    /* [H, I]  dequantised */
    int64_t H, I;
    int64_t nrows;
    const uint16_t* const* xrows; /* nrows pointers to bf16 rows of length H */
    float* g;            /* [nrows, I] */
    float* u;            /* [nrows, I] */
    uint16_t* h;         /* [nrows, I] bf16 */
    float* y;            /* [nrows, H] */
} mlp_ctx;

/* g[r, n] = sum_c x[r, c] * W13[n, c];  u[r, n] = sum_c x[r, c] * W13[I + n, c] */
static void mlp_gate_up(void* p, int64_t b, int64_t e)
{
    mlp_ctx* m = (mlp_ctx*)p;
    const int64_t H = m->H, I = m->I;
    int64_t gate_row0 = 0, up_row0 = I;
    if (g_mutation == MUT_GATE_UP_SWAPPED) {
        gate_row0 = I;
        up_row0 = 0;
    }
    for (int64_t n = b; n < e; ++n) {
        const float* wg = m->W13 + (gate_row0 + n) * H;
        const float* wu = m->W13 + (up_row0 + n) * H;
        for (int64_t r = 0; r < m->nrows; ++r) {
            const uint16_t* x = m->xrows[r];
            float ag = 0.0f, au = 0.0f;
            for (int64_t c = 0; c < H; ++c) {
                float xv = oracle_bf16_to_f32(x[c]);
                ag += xv * wg[c];
                au += xv * wu[c];
            }
            m->g[r * I + n] = ag;
            m->u[r * I + n] = au;
            m->h[r * I + n] = oracle_f32_to_bf16(oracle_silu(ag) * au);
        }
    }
}

/* y[r, n] = sum_i h[r, i] * W2[n, i] */
static void mlp_down(void* p, int64_t b, int64_t e)
{
    mlp_ctx* m = (mlp_ctx*)p;
    const int64_t H = m->H, I = m->I;
    for (int64_t n = b; n < e; ++n) {
        for (int64_t r = 0; r < m->nrows; ++r) {
            const uint16_t* h = m->h + r * I;
            float acc = 0.0f;
            for (int64_t i = 0; i < I; ++i) {
                float w = (g_mutation == MUT_DOWN_TRANSPOSED) ? m->W2[i * H + n] : m->W2[n * I + i];
                acc += oracle_bf16_to_f32(h[i]) * w;
            }
            m->y[r * H + n] = acc;
        }
    }
}

/* Dequantise expert e and run its MLP on nrows activation rows. */
static int expert_mlp(const int32_t* w13_q, const uint16_t* w13_s, const int32_t* w2_q,
                      const uint16_t* w2_s, int64_t e, int64_t H, int64_t I, int64_t nrows,
                      const uint16_t* const* xrows, float* g, float* u, uint16_t* h, float* y)
{
    float* W13 = (float*)malloc(sizeof(float) * (size_t)(2 * I * H));
    float* W2 = (float*)malloc(sizeof(float) * (size_t)(H * I));
    if (!W13 || !W2) {
        free(W13);
        free(W2);
        return -1;
    }
    oracle_dequant(w13_q + e * (2 * I) * (H / 8), scales_at(w13_s, e * (2 * I) * (H / 32)), 2 * I, H,
                   W13);
    oracle_dequant(w2_q + e * H * (I / 8), scales_at(w2_s, e * H * (I / 32)), H, I, W2);
    mlp_ctx m = {W13, W2, H, I, nrows, xrows, g, u, h, y};
    parallel_for(I, mlp_gate_up, &m);
    parallel_for(H, mlp_down, &m);
    free(W13);
    free(W2);
    return 0;
}

/* One expert's MLP on explicit rows; exposed for tests. x: [nrows, H] bf16. */
int oracle_expert_mlp(const int32_t* w13_q, const uint16_t* w13_s, const int32_t* w2_q,
                      const uint16_t* w2_s, int64_t e, int64_t H, int64_t I, int64_t nrows,
                      const uint16_t* x, float* g, float* u, uint16_t* h, float* y)
{
    const uint16_t** rows = (const uint16_t**)malloc(sizeof(void*) * (size_t)(nrows > 0 ? nrows : 1));
    if (!rows)
        return -1;
    for (int64_t r = 0; r < nrows; ++r)
        rows[r] = x + r * H;
    int rc = expert_mlp(w13_q, w13_s, w2_q, w2_s, e, H, I, nrows, rows, g, u, h, y);
    free(rows);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* combine (R9)                                                              */
/* ------------------------------------------------------------------------- */
/* out[t, n] = RNE_bf16( sum over local slots j ascending of w[t, j] * y[t*k + j, n] ) */
static void combine(const float* y_pairs, const uint8_t* is_local, const float* topk_weights,
                    int64_t T, int64_t k, int64_t H, uint16_t* out)
{
    int64_t kk = (g_mutation == MUT_DROP_LAST_SLOT) ? k - 1 : k;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t n = 0; n < H; ++n) {
            float acc = 0.0f;
            for (int64_t j = 0; j < kk; ++j) {
                int64_t p = t * k + j;
                if (!is_local[p])
                    continue;
                float w = (g_mutation == MUT_DROP_WEIGHT) ? 1.0f : topk_weights[p];
                acc += w * y_pairs[p * H + n];
            }
            out[t * H + n] = oracle_f32_to_bf16(acc);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* indexed layer                                                             */
/* ------------------------------------------------------------------------- */
/*
 * The whole layer on the indexed (moe_align_block_size) layout.  For each
 * padded row r < num_tokens_padded whose pair p = sorted_ids[r] is not the
 * sentinel, the token t = p / k goes through the MLP of expert
 * expert_ids[r / block_m]; then the combine.  Optional outputs:
 *   h_rows [capacity, I] bf16 (rows of sentinel entries set to 0),
 *   y_pairs [T*k, H] fp32 (pairs that are not local set to 0).
 * Returns 0, or -1 on an inconsistent index / allocation failure.
 */
int oracle_moe_indexed(const uint16_t* x, int64_t T, int64_t H, int64_t I, int64_t E_local,
                       int64_t k, const int32_t* w13_q, const uint16_t* w13_s,
                       const int32_t* w2_q, const uint16_t* w2_s, const float* topk_weights,
                       const int32_t* sorted_ids, const int32_t* expert_ids,
                       const int32_t* num_tokens_padded, int64_t capacity, int64_t block_m,
                       uint16_t* out, uint16_t* h_rows, float* y_pairs_out, float* g_rows,
                       float* u_rows)
{
    const int64_t P = T * k;
    const int64_t ntp = num_tokens_padded[0];
    if (ntp < 0 || ntp > capacity || block_m <= 0)
        return -1;
    float* y_pairs = (float*)calloc((size_t)(P > 0 ? P : 1) * (size_t)H, sizeof(float));
    uint8_t* is_local = (uint8_t*)calloc((size_t)(P > 0 ? P : 1), 1);
    int64_t* rows_of = (int64_t*)malloc(sizeof(int64_t) * (size_t)(ntp > 0 ? ntp : 1));
    const uint16_t** xrows = (const uint16_t**)malloc(sizeof(void*) * (size_t)(ntp > 0 ? ntp : 1));
    int rc = 0;
    if (!y_pairs || !is_local || !rows_of || !xrows) {
        rc = -1;
        goto done;
    }
    if (h_rows)
        memset(h_rows, 0, sizeof(uint16_t) * (size_t)(capacity * I));
    if (g_rows)
        memset(g_rows, 0, sizeof(float) * (size_t)(capacity * I));
    if (u_rows)
        memset(u_rows, 0, sizeof(float) * (size_t)(capacity * I));
    for (int64_t e = 0; e < E_local && rc == 0; ++e) {
        int64_t n = 0;
        for (int64_t r = 0; r < ntp; ++r) {
            int32_t p = sorted_ids[r];
            if (p < 0 || p >= P)
                continue;
            if (expert_ids[r / block_m] != e)
                continue;
            rows_of[n] = r;
            xrows[n] = x + (p / k) * H;
            ++n;
        }
        if (n == 0)
            continue;
        float* g = (float*)malloc(sizeof(float) * (size_t)(n * I));
        float* u = (float*)malloc(sizeof(float) * (size_t)(n * I));
        uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(n * I));
        float* y = (float*)malloc(sizeof(float) * (size_t)(n * H));
        if (!g || !u || !h || !y ||
            expert_mlp(w13_q, w13_s, w2_q, w2_s, e, H, I, n, xrows, g, u, h, y) != 0) {
            rc = -1;
        } else {
            for (int64_t i = 0; i < n; ++i) {
                int64_t r = rows_of[i];
                int64_t p = sorted_ids[r];
                is_local[p] = 1;
                memcpy(y_pairs + p * H, y + i * H, sizeof(float) * (size_t)H);
                if (h_rows)
                    memcpy(h_rows + r * I, h + i * I, sizeof(uint16_t) * (size_t)I);
                if (g_rows)
                    memcpy(g_rows + r * I, g + i * I, sizeof(float) * (size_t)I);
                if (u_rows)
                    memcpy(u_rows + r * I, u + i * I, sizeof(float) * (size_t)I);
            }
        }
        free(g);
        free(u);
        free(h);
        free(y);
    }
    if (rc == 0) {
        combine(y_pairs, is_local, topk_weights, T, k, H, out);
        if (y_pairs_out)
            memcpy(y_pairs_out, y_pairs, sizeof(float) * (size_t)(P * H));
    }
done:
    free(y_pairs);
    free(is_local);
    free(rows_of);
    free(xrows);
    return rc;
}

/*
 * The second half of the indexed layer on given intermediate rows: for each
 * padded row r < num_tokens_padded with pair p = sorted_ids[r] (not the
 * sentinel), y_p = W2_e h_rows[r] (e = expert_ids[r / block_m]), then the
 * combine.  Checks a down GEMM + combine against the same intermediate that a
 * gate/up implementation produced (the bf16 rounding of h is a decision two
 * fp32 implementations may take differently).
 */
int oracle_moe_indexed_down(const uint16_t* h_rows, int64_t T, int64_t H, int64_t I,
                            int64_t E_local, int64_t k, const int32_t* w2_q, const uint16_t* w2_s,
                            const float* topk_weights, const int32_t* sorted_ids,
                            const int32_t* expert_ids, const int32_t* num_tokens_padded,
                            int64_t capacity, int64_t block_m, uint16_t* out)
{
    const int64_t P = T * k;
    const int64_t ntp = num_tokens_padded[0];
    if (ntp < 0 || ntp > capacity || block_m <= 0)
        return -1;
    float* y_pairs = (float*)calloc((size_t)(P > 0 ? P : 1) * (size_t)H, sizeof(float));
    uint8_t* is_local = (uint8_t*)calloc((size_t)(P > 0 ? P : 1), 1);
    int64_t* rows_of = (int64_t*)malloc(sizeof(int64_t) * (size_t)(ntp > 0 ? ntp : 1));
    uint16_t* hbuf = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)((ntp > 0 ? ntp : 1) * I));
    float* W2 = (float*)malloc(sizeof(float) * (size_t)(H * I));
    float* y = (float*)malloc(sizeof(float) * (size_t)((ntp > 0 ? ntp : 1) * H));
    int rc = 0;
    if (!y_pairs || !is_local || !rows_of || !hbuf || !W2 || !y) {
        rc = -1;
        goto done;
    }
    for (int64_t e = 0; e < E_local; ++e) {
        int64_t n = 0;
        for (int64_t r = 0; r < ntp; ++r) {
            int32_t p = sorted_ids[r];
            if (p < 0 || p >= P || expert_ids[r / block_m] != e)
                continue;
            rows_of[n] = r;
            memcpy(hbuf + n * I, h_rows + r * I, sizeof(uint16_t) * (size_t)I);
            ++n;
        }
        if (n == 0)
            continue;
        oracle_dequant(w2_q + e * H * (I / 8), scales_at(w2_s, e * H * (I / 32)), H, I, W2);
        mlp_ctx m = {NULL, W2, H, I, n, NULL, NULL, NULL, hbuf, y};
        parallel_for(H, mlp_down, &m);
        for (int64_t i = 0; i < n; ++i) {
            int64_t p = sorted_ids[rows_of[i]];
            is_local[p] = 1;
            memcpy(y_pairs + p * H, y + i * H, sizeof(float) * (size_t)H);
        }
    }
    combine(y_pairs, is_local, topk_weights, T, k, H, out);
done:
    free(y_pairs);
    free(is_local);
    free(rows_of);
    free(hbuf);
    free(W2);
    free(y);
    return rc;
}

/* Down GEMM + outputs of the grouped layer on given intermediate rows h_rows [M, I]. */
int oracle_moe_grouped_down(int mode, const uint16_t* h_rows, int64_t M, int64_t H, int64_t I,
                            int64_t E_local, const int32_t* m_indices, const int32_t* masked_m,
                            int64_t max_m, const int32_t* w2_q, const uint16_t* w2_s,
                            const int32_t* row_to_pair, const float* topk_weights, int64_t T,
                            int64_t k, uint16_t* out_rows, uint16_t* out_tokens)
{
    if ((mode != 0 && mode != 1) || (mode == 1 && M != E_local * max_m))
        return -1;
    float* yall = (float*)calloc((size_t)(M > 0 ? M : 1) * (size_t)H, sizeof(float));
    int64_t* rows_of = (int64_t*)malloc(sizeof(int64_t) * (size_t)(M > 0 ? M : 1));
    uint16_t* hbuf = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)((M > 0 ? M : 1) * I));
    float* W2 = (float*)malloc(sizeof(float) * (size_t)(H * I));
    float* y = (float*)malloc(sizeof(float) * (size_t)((M > 0 ? M : 1) * H));
    int rc = 0;
    if (!yall || !rows_of || !hbuf || !W2 || !y) {
        rc = -1;
        goto done;
    }
    for (int64_t r = 0; r < M * H; ++r)
        out_rows[r] = 0;
    for (int64_t e = 0; e < E_local; ++e) {
        int64_t n = 0;
        for (int64_t r = 0; r < M; ++r) {
            int valid = (mode == 0) ? (m_indices[r] == e)
                                    : ((r / max_m == e) && (r % max_m) < masked_m[e]);
            if (!valid)
                continue;
            rows_of[n] = r;
            memcpy(hbuf + n * I, h_rows + r * I, sizeof(uint16_t) * (size_t)I);
            ++n;
        }
        if (n == 0)
            continue;
        oracle_dequant(w2_q + e * H * (I / 8), scales_at(w2_s, e * H * (I / 32)), H, I, W2);
        mlp_ctx m = {NULL, W2, H, I, n, NULL, NULL, NULL, hbuf, y};
        parallel_for(H, mlp_down, &m);
        for (int64_t i = 0; i < n; ++i) {
            int64_t r = rows_of[i];
            for (int64_t c = 0; c < H; ++c)
                out_rows[r * H + c] = oracle_f32_to_bf16(y[i * H + c]);
            memcpy(yall + r * H, y + i * H, sizeof(float) * (size_t)H);
        }
    }
    if (out_tokens && row_to_pair && topk_weights) {
        const int64_t P = T * k;
        float* y_pairs = (float*)calloc((size_t)(P > 0 ? P : 1) * (size_t)H, sizeof(float));
        uint8_t* is_local = (uint8_t*)calloc((size_t)(P > 0 ? P : 1), 1);
        if (!y_pairs || !is_local) {
            rc = -1;
        } else {
            for (int64_t r = 0; r < M; ++r) {
                int valid = (mode == 0) ? (m_indices[r] >= 0)
                                        : ((r % max_m) < masked_m[r / max_m]);
                int64_t p = row_to_pair[r];
                if (!valid || p < 0 || p >= P)
                    continue;
                is_local[p] = 1;
                memcpy(y_pairs + p * H, yall + r * H, sizeof(float) * (size_t)H);
            }
            combine(y_pairs, is_local, topk_weights, T, k, H, out_tokens);
        }
        free(y_pairs);
        free(is_local);
    }
done:
    free(yall);
    free(rows_of);
    free(hbuf);
    free(W2);
    free(y);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* grouped layer: contiguous (mode 0) and masked (mode 1)                    */
/* ------------------------------------------------------------------------- */
/*
 * mode 0 (contiguous): a is [M, H]; row r belongs to expert m_indices[r], or
 *   is padding when m_indices[r] < 0.
 * mode 1 (masked): a is [E, max_m, H] (M = E*max_m); row e*max_m + i belongs
 *   to expert e when i < masked_m[e], else it is ignored.
 * out_rows [M, H] bf16: RNE_bf16(y) of each valid row, 0 on other rows.
 * Optional token combine: with row_to_pair [M] (pair id t*k+j or -1) and
 *   topk_weights [T, k], out_tokens [T, H] gets the same combine as the
 *   indexed layer over the pairs that have a valid row.
 * Optional h_rows [M, I] bf16 and y_rows [M, H] fp32 (0 on invalid rows).
 */
int oracle_moe_grouped(int mode, const uint16_t* a, int64_t M, int64_t H, int64_t I,
                       int64_t E_local, const int32_t* m_indices, const int32_t* masked_m,
                       int64_t max_m, const int32_t* w13_q, const uint16_t* w13_s,
                       const int32_t* w2_q, const uint16_t* w2_s, const int32_t* row_to_pair,
                       const float* topk_weights, int64_t T, int64_t k, uint16_t* out_rows,
                       uint16_t* out_tokens, uint16_t* h_rows, float* y_rows)
{
    if (mode != 0 && mode != 1)
        return -1;
    if (mode == 1 && M != E_local * max_m)
        return -1;
    int64_t* rows_of = (int64_t*)malloc(sizeof(int64_t) * (size_t)(M > 0 ? M : 1));
    const uint16_t** xrows = (const uint16_t**)malloc(sizeof(void*) * (size_t)(M > 0 ? M : 1));
    float* yall = (float*)calloc((size_t)(M > 0 ? M : 1) * (size_t)H, sizeof(float));
    int rc = 0;
    if (!rows_of || !xrows || !yall) {
        rc = -1;
        goto done;
    }
    for (int64_t r = 0; r < M; ++r)
        for (int64_t c = 0; c < H; ++c)
            out_rows[r * H + c] = 0;
    if (h_rows)
        memset(h_rows, 0, sizeof(uint16_t) * (size_t)(M * I));
    for (int64_t e = 0; e < E_local && rc == 0; ++e) {
        int64_t n = 0;
        for (int64_t r = 0; r < M; ++r) {
            int valid;
            if (mode == 0)
                valid = m_indices[r] == e;
            else
                valid = (r / max_m == e) && (r % max_m) < masked_m[e];
            if (!valid)
                continue;
            rows_of[n] = r;
            xrows[n] = a + r * H;
            ++n;
        }
        if (n == 0)
            continue;
        float* g = (float*)malloc(sizeof(float) * (size_t)(n * I));
        float* u = (float*)malloc(sizeof(float) * (size_t)(n * I));
        uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(n * I));
        float* y = (float*)malloc(sizeof(float) * (size_t)(n * H));
        if (!g || !u || !h || !y ||
            expert_mlp(w13_q, w13_s, w2_q, w2_s, e, H, I, n, xrows, g, u, h, y) != 0) {
            rc = -1;
        } else {
            for (int64_t i = 0; i < n; ++i) {
                int64_t r = rows_of[i];
                for (int64_t c = 0; c < H; ++c)
                    out_rows[r * H + c] = oracle_f32_to_bf16(y[i * H + c]);
                memcpy(yall + r * H, y + i * H, sizeof(float) * (size_t)H);
                if (h_rows)
                    memcpy(h_rows + r * I, h + i * I, sizeof(uint16_t) * (size_t)I);
            }
        }
        free(g);
        free(u);
        free(h);
        free(y);
    }
    if (rc == 0 && y_rows)
        memcpy(y_rows, yall, sizeof(float) * (size_t)(M * H));
    if (rc == 0 && out_tokens && row_to_pair && topk_weights) {
        const int64_t P = T * k;
        float* y_pairs = (float*)calloc((size_t)(P > 0 ? P : 1) * (size_t)H, sizeof(float));
        uint8_t* is_local = (uint8_t*)calloc((size_t)(P > 0 ? P : 1), 1);
        if (!y_pairs || !is_local) {
            rc = -1;
        } else {
            for (int64_t r = 0; r < M; ++r) {
                int valid = (mode == 0) ? (m_indices[r] >= 0)
                                        : ((r % max_m) < masked_m[r / max_m]);
                int64_t p = row_to_pair[r];
                if (!valid || p < 0 || p >= P)
                    continue;
                is_local[p] = 1;
                memcpy(y_pairs + p * H, yall + r * H, sizeof(float) * (size_t)H);
            }
            combine(y_pairs, is_local, topk_weights, T, k, H, out_tokens);
        }
        free(y_pairs);
        free(is_local);
    }
done:
    free(rows_of);
    free(xrows);
    free(yall);
    return rc;
}
