// ptx.cuh -- thin inline-PTX wrappers for the sm_103a features the MQA logits
// kernels use: mbarriers with transaction counts, TMA tensor copies, the
// tcgen05 tensor core (TMEM allocation, MMA, commit, TMEM loads) and a few
// register/fence helpers.  Every wait in this library is bounded: see
// wait_bounded() below.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mqa {

// Device-wide status word: bit flags set by kernels (timeouts, failed checks).
// Read and cleared by the host through mqa_device_status().
enum : unsigned {
    kDevErrTimeout = 1u,
    kDevErrBadRange = 2u,
    kDevErrBadContext = 4u,
    kDevErrBadBlock = 8u,
    kDevErrBadSchedule = 16u,
};

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel in its stream still runs;
// grid_dependency_wait() returns once that kernel has completed and its memory
// is visible, and must precede every global access that depends on it.  A
// kernel calls launch_dependents() to let its successor start early.  Both are
// no-ops without such a launch.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One arrival per warp, made by an elected lane without a divergent branch.
__device__ __forceinline__ void mbar_arrive_one_per_warp(uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// try_wait may suspend the thread for a while before reporting an incomplete
// phase.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Per-CTA wait context: a shared abort flag and a cycle budget.  A wait that
// runs out sets the flag (so every other role of the CTA stops waiting too),
// records kDevErrTimeout in the device status word and returns false.  No wait
// in this library can spin forever.
struct WaitCtx {
    volatile int* abort_flag;      // shared memory
    unsigned* status;              // device status word (global)
    long long limit;               // clock64 cycles
};

// `sleep_ns` > 0 backs off between polls: for waiters that are not on the
// critical path, so they leave issue slots to the math warps.  The abort flag
// and the clock are checked every 16 polls.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                             unsigned sleep_ns = 0)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    for (unsigned n = 1;; ++n) {
        if (sleep_ns)
            __nanosleep(sleep_ns);
        if (mbar_try_wait(bar, parity))
            return true;
        if ((n & 15) == 0) {
            if (*w.abort_flag)
                return false;
            if (clock64() - t0 > w.limit) {
                *w.abort_flag = 1;
                atomicOr(w.status, kDevErrTimeout);
                return false;
            }
        }
    }
}

// Cycle budget of a drain wait: at least 2^30 cycles (about half a second),
// whatever budget the pipeline waits were given.
__device__ __forceinline__ long long drain_limit(const WaitCtx& w)
{
    return w.limit > (1ll << 30) ? w.limit : (1ll << 30);
}

// Wait for an asynchronous operation this thread issued itself (a TMA copy, a
// tcgen05 MMA) to complete, before the CTA frees the shared memory or TMEM it
// targets.  Its completion depends on no other role of the CTA, so the abort
// flag is ignored: after another role has given up, the operations already in
// flight must still land.  Bounded by drain_limit(); running out records
// kDevErrTimeout.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, const WaitCtx& w)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    const long long limit = drain_limit(w);
    for (unsigned n = 1;; ++n) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((n & 15) == 0 && clock64() - t0 > limit) {
            *w.abort_flag = 1;
            atomicOr(w.status, kDevErrTimeout);
            return false;
        }
    }
}

// The same wait taken by a whole warp, shaped for the hot path: the whole
// loop is one PTX block whose branches are uniform (each try_wait answer is
// voted across the warp), so the compiler adds no convergence bookkeeping
// around it, and the polling loop is only the test, the vote and a clock
// compare (no shared load, no extra register: measured, an abort-flag check in
// this loop slowed the 2048 x 32768 dense call by 8 %).  Polling stops when
// the phase completes or the cycle budget is spent; a timeout records
// kDevErrTimeout, raises the CTA's abort flag (which stops the waits of the
// other roles) and returns false.  Every lane gets the same answer.
__device__ __forceinline__ bool warp_wait_fast(uint32_t bar, uint32_t parity, const WaitCtx& w)
{
    uint32_t ok;
    asm volatile(
        "{\n\t"
        ".reg .pred p;\n\t"
        ".reg .u64 t0, t1;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "vote.sync.all.pred p, p, 0xffffffff;\n\t"
        "@p bra.uni W_DONE;\n\t"
        "mov.u64 t0, %%clock64;\n\t"
        "W_LOOP:\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "vote.sync.all.pred p, p, 0xffffffff;\n\t"
        "@p bra.uni W_DONE;\n\t"
        "mov.u64 t1, %%clock64;\n\t"
        "sub.s64 t1, t1, t0;\n\t"
        "setp.lt.s64 p, t1, %3;\n\t"
        "@p bra.uni W_LOOP;\n\t"
        "mov.u32 %0, 0;\n\t"
        "bra.uni W_END;\n\t"
        "W_DONE:\n\t"
        "mov.u32 %0, 1;\n\t"
        "W_END:\n\t"
        "}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "l"(w.limit)
        : "memory");
    if (ok)
        return true;
    *w.abort_flag = 1;
    atomicOr(w.status, kDevErrTimeout);
    return false;
}

// ---------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_1d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x)
{
    asm volatile(
        "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// ------------------------------------------------------------------ tcgen05
// TMEM allocation: executed by one whole warp.  The allocated base address is
// written to shared memory at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
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

// D[tmem] (+)= A[smem] * B[smem]^T, FP8 E4M3 inputs, FP32 accumulation.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= (A * SFA)[smem] * (B * SFB)[smem]^T: MXFP8 (E4M3 elements,
// one UE8M0 scale per 32 elements of K, "scale_vec::1X"), FP32 accumulation.
// The scale factors are read from TMEM: for row m of A (M = 128), lane m,
// column sfa + m / 32; for row n of B, lane n % 32 of every lane quadrant,
// column sfb + n / 32; in either cell the byte given by the instruction
// descriptor's scale-factor ids (idesc_mx_f32).  This placement was read
// off the hardware with all-ones operands and coded scale bytes.
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                             uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// 32 rows x 128 bits of shared memory (described by sf_desc) -> TMEM lanes
// r, r + 32, r + 64, r + 96 (every lane quadrant), four 32-bit columns from
// `taddr`: row r word j lands in column taddr + j.  Asynchronous, ordered
// with the issuing thread's later tcgen05.mma.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t s_desc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(s_desc)
                 : "memory");
}

// Descriptor of a tcgen05.cp source: 32 rows of 16 bytes, one after another
// (no swizzle; eight-row core matrices 128 bytes apart).
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(128 >> 4) << 16;            // leading byte offset
    d |= static_cast<uint64_t>(128 >> 4) << 32;            // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                   // descriptor version
    return d;
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with a 128-byte (layout 2) or 64-byte (layout 4) swizzle: rows of
// `row_bytes`, groups of 8 rows `8 * row_bytes` apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t row_bytes)
{
    const uint64_t layout = (row_bytes == 128) ? 2ull : 4ull;
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);          // start address
    d |= static_cast<uint64_t>(1) << 16;                          // leading byte offset (unused)
    d |= static_cast<uint64_t>((8u * row_bytes) >> 4) << 32;       // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                          // descriptor version
    d |= layout << 61;                                            // swizzle mode
    return d;
}

// Instruction descriptor: E4M3 x E4M3 -> F32, both operands K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t M, uint32_t N)
{
    return (1u << 4)                 // D format: F32
           | (0u << 7) | (0u << 10)  // A, B format: E4M3
           | ((N >> 3) << 17)        // N / 8
           | ((M >> 4) << 24);       // M / 16
}

// Element formats of kind::f8f6f4 / kind::mxf8f6f4 operands (the A and B
// format fields of the instruction descriptor).
enum : uint32_t { kFmtE4M3 = 0u, kFmtE2M1 = 5u };

// Instruction descriptor of the block-scaled MMA (kind::mxf8f6f4): `fmt` x
// `fmt` -> F32 (E4M3, or E2M1 held one element per byte of shared memory),
// K-major, M x N, UE8M0 scales; scale-factor id `sf` (the byte of each scale
// cell) for both operands: the K-block of this MMA.
__host__ __device__ constexpr uint32_t idesc_mx_f32(uint32_t M, uint32_t N, uint32_t sf,
                                                    uint32_t fmt)
{
    return (sf << 4)                 // B scale-factor id
           | (fmt << 7) | (fmt << 10)  // A, B format
           | ((N >> 3) << 17)        // N / 8
           | (1u << 23)              // scale type: UE8M0
           | ((M >> 4) << 24)        // M / 16
           | (sf << 29);             // A scale-factor id
}

// 32 consecutive TMEM columns of this warp's 32 lanes -> 32 registers per
// thread (thread t holds lane base + t).  Waits for the load before returning.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int k = 0; k < 32; ++k)
        v[k] = __uint_as_float(r[k]);
}

// Asynchronous form: issue the load only; the registers are valid after
// tmem_wait32() on the same array (which also orders every later use of them
// after the wait).
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, float (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
          "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]),
          "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]),
          "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]),
          "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]),
          "=f"(v[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait32(float (&v)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                   "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                   "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]),
                   "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]),
                   "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]),
                   "+f"(v[30]), "+f"(v[31])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, float (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
          "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]),
          "=f"(v[13]), "=f"(v[14]), "=f"(v[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait16(float (&v)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                   "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                   "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15])
                 :
                 : "memory");
}

// 16 columns of this warp's 32 TMEM lanes, loaded and waited for in one step.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, float (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
          "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]),
          "=f"(v[13]), "=f"(v[14]), "=f"(v[15])
        : "r"(taddr)
        : "memory");
}

// 32 or 64 columns of this warp's 32 TMEM lanes, loaded and waited for in one step.
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, float (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
          "=f"(v[6]), "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]),
          "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]),
          "=f"(v[18]), "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]),
          "=f"(v[24]), "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]),
          "=f"(v[30]), "=f"(v[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld64_wait(uint32_t taddr, float (&v)[64])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
        "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
          "=f"(v[6]), "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]),
          "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]),
          "=f"(v[18]), "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]),
          "=f"(v[24]), "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]),
          "=f"(v[30]), "=f"(v[31]), "=f"(v[32]), "=f"(v[33]), "=f"(v[34]), "=f"(v[35]),
          "=f"(v[36]), "=f"(v[37]), "=f"(v[38]), "=f"(v[39]), "=f"(v[40]), "=f"(v[41]),
          "=f"(v[42]), "=f"(v[43]), "=f"(v[44]), "=f"(v[45]), "=f"(v[46]), "=f"(v[47]),
          "=f"(v[48]), "=f"(v[49]), "=f"(v[50]), "=f"(v[51]), "=f"(v[52]), "=f"(v[53]),
          "=f"(v[54]), "=f"(v[55]), "=f"(v[56]), "=f"(v[57]), "=f"(v[58]), "=f"(v[59]),
          "=f"(v[60]), "=f"(v[61]), "=f"(v[62]), "=f"(v[63])
        : "r"(taddr)
        : "memory");
}

template <int W>
__device__ __forceinline__ void tmem_ld_async(uint32_t taddr, float (&v)[W])
{
    if constexpr (W == 32)
        tmem_ld32_async(taddr, v);
    else
        tmem_ld16_async(taddr, v);
}

template <int W>
__device__ __forceinline__ void tmem_wait(float (&v)[W])
{
    if constexpr (W == 32)
        tmem_wait32(v);
    else
        tmem_wait16(v);
}

// Warp-group register budget change (all 128 threads of the warp group).
template <int N>
__device__ __forceinline__ void regs_inc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void named_bar_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace mqa
