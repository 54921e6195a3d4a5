// device.cuh -- inline-PTX building blocks for sm_103a: mbarriers with bounded
// waits, TMA tile loads, cp.async, tcgen05 (TMEM alloc, MMA, commit, ld/st).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "chord_internal.h"

namespace chord {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: every kernel of the library is launched so
// that it may start while the kernel before it in the stream finishes; it
// lets its own successor be scheduled as soon as all its CTAs run, and waits
// for its predecessors (completed, their writes visible) before it touches
// any memory they may read or write
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// error word (in the caller's workspace)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void raise_error(int* err, int bits)
{
    if (err)
        atomicOr(err, bits);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait on the phase with the given parity.  Gives up after limit_ns (or
// when another role of the CTA has aborted), records CHORD_DEVERR_TIMEOUT in
// the error word, sets the CTA abort flag and returns false.  Never traps and
// never spins forever.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ bool mbar_spin(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* err, uint64_t limit_ns)
{
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 63u) == 63u) {
            if (*abort_flag)
                return false;
            if (global_timer_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                raise_error(err, CHORD_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* err, uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity))
        return true;
    return mbar_spin(bar, parity, abort_flag, err, limit_ns);
}

// The same wait with the spin loop out of line, for the waits off the
// critical path (producers, epilogue): one try_wait inline keeps those loops
// small for the instruction cache; a wait that spins pays a call.
static __device__ __noinline__ bool mbar_spin_ool(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, int* err)
{
    return mbar_spin(bar, parity, abort_flag, err, kWaitLimitNs);
}
__device__ __forceinline__ bool mbar_wait_cold(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               int* err)
{
    if (mbar_try_wait(bar, parity))
        return true;
    return mbar_spin_ool(bar, parity, abort_flag, err);
}

// Bounded wait for a phase that copies this thread issued will complete, used on
// the way out of an aborted CTA (so ignores the abort flag): the CTA must not
// end while the TMA engine still writes its shared memory.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity) && global_timer_ns() - t0 < kWaitLimitNs) {
    }
}

// ---------------------------------------------------------------------------
// TMA (tiled tensor copies, global -> shared) and cp.async
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
        "cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
        "cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            int w, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
        "cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar),
        "l"(policy)
        : "memory");
}

// Plain bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory, completing on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 16-byte cp.async with zero fill: copies src_bytes (0 or 16) and zero-fills the rest.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_8(uint32_t dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}

// arrive on bar once all earlier cp.async of this thread have landed
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows 128 B
// apart inside an 8-row group, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;          // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;  // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;          // descriptor version
    d |= static_cast<uint64_t>(2) << 61;          // 128-byte swizzle
    return d;
}

// Instruction descriptor: dense, D fp32, A and B bf16, both K-major, shape M x N.
__host__ __device__ __forceinline__ uint32_t idesc_bf16_f32(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, M = 128 rows of A, N from idesc, K = 16.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Same MMA issued by one lane that elect.sync picks; the whole warp executes the
// call with identical operands.  Issuing from a converged warp keeps the
// operands in uniform registers: measured on sm_103a, 16 back-to-back M=128
// N<=32 MMAs issue at about 22 clocks each this way against 53 clocks from a
// lane-0-only branch.
__device__ __forceinline__ void mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit_elect(uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// One K stage of MMAs (BK / 16 of them, K = 16 each) issued from one asm
// block: one elect.sync for the stage, operands as 32-bit adds on the
// descriptor's address word (address >> 4 stays below 2^14, so the adds never
// carry into the other fields).  The j-th MMA reads A columns a + 8 j and the
// B descriptor of 16-element K step j: atom column j / 4 (REG16 = that
// column's size in 16-byte units), 32-byte step j % 4 inside the swizzled row.
// accumulate = 0 makes the first MMA overwrite D.
template <int REG16>
__device__ __forceinline__ void mma_stage16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred e, p0, pt;\n\t.reg .b32 bq, bl, al;\n\t.reg .b64 bd;\n\t"
        "setp.ne.b32 p0, %5, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "mov.b32 bq, %2;\n\tmov.b64 bd, {bq, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p0;\n\t"
        "add.u32 bl, bq, 2;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 8;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 4;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 16;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 6;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 24;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bq, %2, %6;\n\tmov.b64 bd, {bq, %3};\n\tadd.u32 al, %1, 32;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 2;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 40;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 4;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 48;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 6;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 56;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bq, %2, %7;\n\tmov.b64 bd, {bq, %3};\n\tadd.u32 al, %1, 64;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 2;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 72;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 4;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 80;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 6;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 88;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bq, %2, %8;\n\tmov.b64 bd, {bq, %3};\n\tadd.u32 al, %1, 96;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 2;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 104;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 4;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 112;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 6;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 120;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "}"
        ::"r"(d_tmem), "r"(a_tmem), "r"(static_cast<uint32_t>(b_desc)),
        "r"(static_cast<uint32_t>(b_desc >> 32)), "r"(idesc), "r"(accumulate), "n"(REG16),
        "n"(2 * REG16), "n"(3 * REG16)
        : "memory");
}

template <int REG16>
__device__ __forceinline__ void mma_stage8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred e, p0, pt;\n\t.reg .b32 bq, bl, al;\n\t.reg .b64 bd;\n\t"
        "setp.ne.b32 p0, %5, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "mov.b32 bq, %2;\n\tmov.b64 bd, {bq, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p0;\n\t"
        "add.u32 bl, bq, 2;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 8;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 4;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 16;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 6;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 24;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bq, %2, %6;\n\tmov.b64 bd, {bq, %3};\n\tadd.u32 al, %1, 32;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 2;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 40;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 4;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 48;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "add.u32 bl, bq, 6;\n\tmov.b64 bd, {bl, %3};\n\tadd.u32 al, %1, 56;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [al], bd, %4, pt;\n\t"
        "}"
        ::"r"(d_tmem), "r"(a_tmem), "r"(static_cast<uint32_t>(b_desc)),
        "r"(static_cast<uint32_t>(b_desc >> 32)), "r"(idesc), "r"(accumulate), "n"(REG16)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
        "%29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]),
        "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]),
        "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

// Four consecutive fp32 reductions in one instruction (16-byte aligned address).
__device__ __forceinline__ void red_add_v4_f32(float* addr, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c),
                 "f"(d));
}

__device__ __forceinline__ uint32_t bf16x2_pack_rn(float lo, float hi)
{
    const __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&t);
}

// Fire-and-forget fp32 reduction.  No "memory" clobber: nothing in the kernel
// reads the target after it, and a clobber would serialise the caller's
// independent loads behind every reduction.
__device__ __forceinline__ void red_add_f32(float* addr, float v)
{
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v));
}

}  // namespace chord
