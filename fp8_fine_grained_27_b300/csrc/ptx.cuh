// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers, TMA bulk
// tensor copies, tcgen05 (TMEM allocation, MMA, commit, loads) and the E4M3
// conversion.  Written from the public PTX ISA description of each
// instruction.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace fp8bs {

// ---------------------------------------------------------------- basics
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
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

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

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

// Device error word shared by every kernel of the library (the library is a
// single translation unit, so this is its one definition).  Kernels only
// write it (first error wins); fp8bs_get_device_error reads and clears it.
__device__ int g_fp8bs_error = 0;

enum : int { ERR_NONE = 0, ERR_TIMEOUT_PRODUCER = 1, ERR_TIMEOUT_MMA = 2,
             ERR_TIMEOUT_CONSUMER = 3, ERR_TIMEOUT_SELFTEST = 4, ERR_TIMEOUT_SPLIT = 5 };

// Bounds checks of the debug build (compiled with -DFP8BS_DEBUG).  Each
// global, shared-memory and TMEM access site checks its index against the
// extent that the kernel's arguments (or its own layout) give it; a failed
// check records the site's number in g_fp8bs_debug_site (first one wins) and
// the caller skips the access, so a bad index is reported instead of
// touching memory.  In the release build dbg_ok is the constant true and the
// checks compile away.
__device__ int g_fp8bs_debug_site = 0;

enum : int {
    DBG_QROWS_LOAD = 1, DBG_QROWS_STORE = 2, DBG_QROWS_SCALE = 3,
    DBG_QT_LOAD = 4, DBG_QT_SMEM = 5, DBG_QT_STORE = 6, DBG_QT_SCALE = 7,
    DBG_GEMM_SCALE_A = 8, DBG_GEMM_SCALE_B = 9, DBG_GEMM_TMEM = 10, DBG_GEMM_EPI_SMEM = 11,
    DBG_GEMM_STORE = 12, DBG_GEMM_GROUP = 13, DBG_GEMM_SWIGLU_STORE = 14,
    DBG_MX_STORE = 15, DBG_MX_EPI_SMEM = 16, DBG_MOE_GROUP = 17, DBG_MOE_COMBINE = 18, DBG_GEMM_SPLIT = 19,
};

__device__ __forceinline__ bool dbg_ok(bool in_bounds, int site)
{
#ifdef FP8BS_DEBUG
    if (!in_bounds) {
        atomicCAS(&g_fp8bs_debug_site, 0, site);
        return false;
    }
    return true;
#else
    (void)in_bounds;
    (void)site;
    return true;
#endif
}

// Bounded wait on an mbarrier phase.  Spins briefly, then checks the global
// timer.  `abort` is a flag in the CTA's shared memory (zeroed at the CTA's
// start): after `limit_ns` the wait records `code` in the device error word
// (first error wins), raises the flag and returns false; any wait of the same
// CTA that sees the flag raised returns false at once, so the other roles of
// a CTA give up together.  The flag belongs to one CTA of one launch, so an
// error that an earlier launch left in the device error word does not make
// later launches give up.  A null `abort` (a drain that must run to its own
// limit) never gives up early and raises nothing.
// Non-blocking test of a phase (no suspension).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The phase is tested once without suspending before the (suspending)
// try_wait loop: a try_wait on a phase that has already completed measured
// about 200 cycles, and the GEMM loops wait on many such phases (operands
// loaded chunks ahead, scale slots).  Wgrad GEMM 0.3686 -> 0.3400 ms, FFN
// GEMM +1% at equal clock, bit-identical.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int code, volatile int *abort,
                                          uint64_t limit_ns = 2000000000ull)
{
    if (mbar_test_wait(bar, parity))
        return true;
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
        if (mbar_try_wait(bar, parity))
            return true;
    const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (abort && *abort != 0)
            return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicCAS(&g_fp8bs_error, 0, code);
            if (abort)
                *abort = 1;
            return false;
        }
    }
}

// A flag in global memory that one CTA sets (release at GPU scope, after its
// data) and another CTA of the same launch waits for (acquire at GPU scope).
__device__ __forceinline__ void flag_release(uint32_t *f, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t flag_acquire(const uint32_t *f)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}

// Bounded wait until *f == v, with the give-up rules of mbar_wait.
__device__ __forceinline__ bool flag_wait(const uint32_t *f, uint32_t v, int code, volatile int *abort,
                                          uint64_t limit_ns = 2000000000ull)
{
    const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
    while (true) {
        if (flag_acquire(f) == v)
            return true;
        if (abort && *abort != 0)
            return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicCAS(&g_fp8bs_error, 0, code);
            if (abort)
                *abort = 1;
            return false;
        }
        __nanosleep(256);
    }
}

// Clock record of the GEMM kernels.  CTA 0 of each launch adds the SM cycles
// and the nanoseconds from the end of its set-up to its end, and counts the
// launch, so the host can compute the SM clock the GEMMs actually ran at (the
// board's sampled clock cannot resolve kernels of a millisecond, and the
// clock drops under the power cap).  g_fp8bs_clock = {cycles, ns, launches}.
__device__ unsigned long long g_fp8bs_clock[3];

struct KernelClock {
    unsigned long long cycles, ns;
};

__device__ __forceinline__ KernelClock kernel_clock_begin()
{
    KernelClock k;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(k.cycles));
    k.ns = globaltimer_ns();
    return k;
}

__device__ __forceinline__ void kernel_clock_end(const KernelClock &k)
{
    unsigned long long c;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
    const unsigned long long t = globaltimer_ns();
    atomicAdd(&g_fp8bs_clock[0], c - k.cycles);
    atomicAdd(&g_fp8bs_clock[1], t - k.ns);
    atomicAdd(&g_fp8bs_clock[2], 1ull);
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may be scheduled while the kernel before it in the stream is
// still running: it must not read that kernel's results (or write what that
// kernel reads) before grid_dependency_wait(), which returns once the earlier
// grid has completed and its memory is visible.  The earlier kernel calls
// grid_launch_dependents() to let the next one be scheduled before it ends.
// Without a programmatic launch both are no-ops.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Re-balance registers between warpgroups (the four warps of a warpgroup
// execute these together).
template <int N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2D tiled bulk tensor load global -> shared, completion on `bar` (tx bytes).
// x = innermost coordinate (elements), y = row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *m, int32_t x,
                                            int32_t y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Untiled bulk copy global -> shared of `bytes` (a multiple of 16; both
// addresses 16-byte aligned), completion on `bar` (tx bytes).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// ---------------------------------------------------------------- cp.async
// Asynchronous global -> shared copies of 4 or 16 bytes (any 4-/16-byte
// aligned addresses), and an mbarrier arrival that fires once every copy the
// thread issued before it has landed (counted in the barrier's expected
// arrivals: "noinc").
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// 16-byte copy that reads src_bytes (0 or 16) and zero-fills the rest
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
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

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 x E4M3 -> FP32, one instruction
// (M x N x 32).  `accumulate` selects D += versus D =.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives
// lane (base lane + i), columns col .. col+31 of TMEM.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// 16 lanes x 256 bits, 4 times along the columns: thread i of the warp
// receives, for j = 0..3, r[4j], r[4j+1] = lane (base lane + i/4), columns
// col + 8j + 2(i%4) and + 1, and r[4j+2], r[4j+3] = lane (base lane + 8 +
// i/4), the same two columns (a layout checked on the device).
__device__ __forceinline__ void tmem_ld16x4(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand stored as rows of
// 128 bytes with the 128-byte swizzle (8-row, 1024-byte atoms), as a TMA load
// with CU_TENSOR_MAP_SWIZZLE_128B writes it.  Fields: start address >> 4
// (bits 0-13), leading byte offset >> 4 (16-29, unused for this layout),
// stride byte offset >> 4 = 1024 B between 8-row groups (32-45), descriptor
// version 1 (46-47), base offset 0 (49-51, atoms are 1024-byte aligned),
// layout type 2 = 128-byte swizzle (61-63).
__device__ __forceinline__ uint64_t sdesc_k128_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor for kind::f8f6f4: D FP32 (bits 4-5 = 1), A and B
// E4M3 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at
// bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N)
{
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------- E4M3
// Two FP32 values -> two E4M3 codes, round to nearest even, saturating to
// +-448 (NaN stays NaN).  Result: low byte = lo, high byte = hi.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
    return h;
}

}  // namespace fp8bs
