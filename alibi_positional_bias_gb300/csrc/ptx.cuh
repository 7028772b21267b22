// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// tensor loads, and the tcgen05 tensor-core / tensor-memory instructions.
// Written from the PTX ISA descriptions of these instructions.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "checks.h"
#include "internal.h"

namespace alibi {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Record a device-side failure (first site wins for the detail field).
__device__ __forceinline__ void report_error(uint32_t *err, uint32_t code, uint32_t site)
{
    if (err) {
        atomicOr(err, code);
        atomicCAS(err + 1, 0u, site);
    }
}

// ------------------------------------------------------- integer division

// Division by a runtime divisor d >= 1 of numerators below 2^31 as a multiply-high,
// an add and a shift (Granlund and Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994): with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d)
// + 1, n / d = (umulhi(n, m) + n) >> l. The tensor-core kernels decode their work items
// with it at every item boundary, where a plain integer division is a long
// dependent sequence.
struct FastDiv {
    uint32_t d, m, l;
};

inline FastDiv make_fastdiv(uint32_t d)
{
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
    return FastDiv{d, static_cast<uint32_t>(m), l};
}

__device__ __forceinline__ int fdiv(int n, const FastDiv &f)
{
    const uint32_t u = static_cast<uint32_t>(n);
    return static_cast<int>((__umulhi(u, f.m) + u) >> f.l);
}

__device__ __forceinline__ int fmod_(int n, const FastDiv &f) { return n - fdiv(n, f) * static_cast<int>(f.d); }

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Programmatic dependent launch (a grid launched with programmatic stream
// serialization may start before the previous grid in its stream has finished):
// wait until the grids this one depends on have completed and their writes are
// visible; let the dependent grid launch once every CTA of this grid has issued
// this (or exited).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// This CTA's failure state, in static shared memory: the abort code one of the
// CTA's own roles raised, and the limit of every bounded wait. Their addresses are
// constants, so a wait carries no extra register. Waits give up early only on the
// CTA's own abort code, never on the device status word, so an error left
// uncollected in that word by an earlier launch does not cut a later launch short,
// while one role's timeout still stops the other roles of its CTA within a few
// hundred polls. A kernel that waits calls cta_err_init() from one thread before
// its first barrier.
static __shared__ uint32_t cta_abort;
static __shared__ uint64_t cta_wait_ns;

__device__ __forceinline__ void cta_err_init(uint64_t limit_ns)
{
    cta_abort = 0u;
    cta_wait_ns = limit_ns;
}

// Debug-checks build (-DALIBI_CHECKS): the device status word and the CTA's dynamic
// shared-memory window, against which the wrappers below test their addresses
// (predicates in checks.h). Every CTA allocates all TMEM columns of its SM.
#ifdef ALIBI_CHECKS
static __shared__ uint32_t *cta_check_word;
static __shared__ uint32_t cta_smem_lo, cta_smem_hi;
constexpr uint32_t kCheckTmemCols = 512;

__device__ __forceinline__ void check_fail(uint32_t id, uint32_t value)
{
    report_error(cta_check_word, ALIBI_DEV_CHECK, check::site(id, value));
}

__device__ __forceinline__ bool check_smem(uint32_t saddr, uint32_t bytes, uint32_t align)
{
    return check::smem_range(saddr, bytes, align, cta_smem_lo, cta_smem_hi);
}
#endif

// One thread of every kernel that uses the wrappers below calls this before the
// CTA's first barrier (a no-op outside the debug-checks build).
__device__ __forceinline__ void cta_check_init(uint32_t *dev, const void *smem, uint32_t bytes)
{
#ifdef ALIBI_CHECKS
    cta_check_word = dev;
    cta_smem_lo = smem_u32(smem);
    cta_smem_hi = cta_smem_lo + bytes;
#else
    (void)dev;
    (void)smem;
    (void)bytes;
#endif
}

// Wait until the phase with the given parity has completed, for at most the CTA's
// wait limit. Returns false on expiry, after recording ALIBI_DEV_TIMEOUT in the
// device status word `err` and in the CTA's abort code; or early if another role
// of this CTA raised an error (unless `drain`: a drain wait is for work this thread
// issued itself, which completes on its own, so it ignores the abort code and ends
// only on completion or its own time limit). The abort code and the global timer
// are read only every 256 polls, so a completed phase is noticed without extra
// latency on the critical path.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *err, uint32_t site,
                                          bool drain = false)
{
    if (mbar_test(bar, parity)) return true;  // already complete: no suspend
    uint64_t t0 = 0;
#pragma unroll 1
    for (uint32_t n = 0;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 255u) == 255u) {
            if (!drain && *(volatile uint32_t *)&cta_abort != 0u) return false;
            const uint64_t t = global_timer_ns();
            if (t0 == 0) {
                t0 = t;
            } else if (t - t0 > *(volatile uint64_t *)&cta_wait_ns) {
                report_error(err, ALIBI_DEV_TIMEOUT, site);
                *(volatile uint32_t *)&cta_abort = ALIBI_DEV_TIMEOUT;
                return false;
            }
        }
    }
}

// The same bounded wait polling with the non-suspending test: for a single issuing
// warp whose reaction time to a handoff is on the critical path (the suspending
// try_wait wakes a little later after the phase completes).
__device__ __forceinline__ bool mbar_wait_spin(uint64_t *bar, uint32_t parity, uint32_t *err, uint32_t site)
{
    uint64_t t0 = 0;
#pragma unroll 1
    for (uint32_t n = 0;; ++n) {
        if (mbar_test(bar, parity)) return true;
        if ((n & 1023u) == 1023u) {
            if (*(volatile uint32_t *)&cta_abort != 0u) return false;
            const uint64_t t = global_timer_ns();
            if (t0 == 0) {
                t0 = t;
            } else if (t - t0 > *(volatile uint64_t *)&cta_wait_ns) {
                report_error(err, ALIBI_DEV_TIMEOUT, site);
                *(volatile uint32_t *)&cta_abort = ALIBI_DEV_TIMEOUT;
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 3-D tiled load of one box into shared memory, completing on `bar`. Every load of
// the kernels is a 16 KB box (64 bf16 x 128 rows) into a 1024-byte aligned swizzle atom.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, int x, int y, int z, uint64_t *bar)
{
#ifdef ALIBI_CHECKS
    if (!check::tma_x_aligned(x)) return check_fail(check::TMA_LOAD, static_cast<uint32_t>(x));
    if (!check_smem(smem_u32(dst), 16384, 1024)) return check_fail(check::TMA_LOAD, smem_u32(dst));
#endif
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// 3-D tiled store of one box from shared memory (bulk-group completion). The
// source must stay unchanged until bulk_wait_read() has returned; rows and columns
// outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const void *tmap, const void *src, int x, int y, int z)
{
#ifdef ALIBI_CHECKS
    if (!check::tma_store_coords(x, y, z))
        return check_fail(check::TMA_STORE, static_cast<uint32_t>(x < 0 || (x & 7) ? x : (y < 0 ? y : z)));
    if (!check_smem(smem_u32(src), 1024, 16)) return check_fail(check::TMA_STORE, smem_u32(src));
#endif
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// All but the most recent committed bulk store of this thread have finished reading
// shared memory (a double-buffered source may be refilled).
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// Every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ------------------------------------------------------------------ tcgen05

// Allocate `ncols` TMEM columns (whole warp); the base address lands in *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

#ifdef ALIBI_CHECKS
// D columns (N of the instruction descriptor) inside the allocation and every shared-
// memory operand's start inside the window; a TMEM A operand's K = 16 step (8 columns).
__device__ __forceinline__ bool check_mma(uint32_t d_tmem, uint32_t idesc, const uint64_t *descs, int ndesc,
                                          int a_tmem)
{
    if (!check::tmem_cols(d_tmem, check::idesc_n(idesc), kCheckTmemCols)) {
        check_fail(check::TMEM_COLS, d_tmem);
        return false;
    }
    if (a_tmem >= 0 && !check::tmem_cols(static_cast<uint32_t>(a_tmem), 8, kCheckTmemCols)) {
        check_fail(check::TMEM_COLS, static_cast<uint32_t>(a_tmem));
        return false;
    }
    for (int i = 0; i < ndesc; ++i)
        if (!check_smem(check::desc_addr(descs[i]), 16, 16)) {
            check_fail(check::SMEM_DESC, check::desc_addr(descs[i]));
            return false;
        }
    return true;
}
#endif

// Warp-converged forms: the whole warp executes the call with identical operands
// and one elected lane (the lowest active one, i.e. the same lane every time
// the warp is converged) issues the instruction. Keeping the issuing code
// warp-uniform lets the descriptor arithmetic stay in uniform registers.
__device__ __forceinline__ void mma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
#ifdef ALIBI_CHECKS
    const uint64_t descs[2] = {a_desc, b_desc};
    if (!check_mma(d_tmem, idesc, descs, 2, -1)) return;
#endif
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Copy a 128-row x 32-byte slice of a shared-memory matrix (described like an MMA
// operand: swizzle, strides, K-step offset) into TMEM: row r to lane r, the 16 bf16
// of the slice as 8 columns of bf16 pairs, the layout an A operand read from TMEM
// takes. Ordered with the issuing thread's MMAs; tracked by its commits.
__device__ __forceinline__ void tmem_cp_w(uint32_t taddr, uint64_t s_desc)
{
#ifdef ALIBI_CHECKS
    if (!check::tmem_cols(taddr, 8, kCheckTmemCols)) return check_fail(check::TMEM_COLS, taddr);
    if (!check_smem(check::desc_addr(s_desc), 16, 16)) return check_fail(check::SMEM_DESC, check::desc_addr(s_desc));
#endif
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.cp.cta_group::1.128x256b [%0], %1;\n\t}" ::"r"(taddr),
        "l"(s_desc)
        : "memory");
}

__device__ __forceinline__ void mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
#ifdef ALIBI_CHECKS
    if (!check_mma(d_tmem, idesc, &b_desc, 1, static_cast<int>(a_tmem & 0xFFFFu))) return;
#endif
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit_w(uint64_t *bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp gets row (lane base + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
#ifdef ALIBI_CHECKS
    // warp-uniform tests (the address is), so a skipped load is skipped by the whole warp
    if (!check::tmem_cols(taddr, 32, kCheckTmemCols) || !check::tmem_lanes(taddr, threadIdx.x >> 5)) {
        check_fail(check::tmem_cols(taddr, 32, kCheckTmemCols) ? check::TMEM_LANES : check::TMEM_COLS, taddr);
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0u;
        return;
    }
#endif
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
#ifdef ALIBI_CHECKS
    if (!check::tmem_cols(taddr, 32, kCheckTmemCols) || !check::tmem_lanes(taddr, threadIdx.x >> 5))
        return check_fail(check::tmem_cols(taddr, 32, kCheckTmemCols) ? check::TMEM_LANES : check::TMEM_COLS, taddr);
#endif
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for tcgen05.mma with the 128-byte swizzle
// (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B): start address,
// leading- and stride-dimension byte offsets (16-byte units), the fixed
// descriptor version bit 46, and layout type 2 (SWIZZLE_128B) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B,
// K-major A, B K-major (b_mn_major = 0) or MN-major (1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, uint32_t b_mn_major)
{
    return (1u << 4)             // D format: f32
           | (1u << 7)           // A format: bf16
           | (1u << 10)          // B format: bf16
           | (0u << 15)          // A K-major
           | (b_mn_major << 16)  // B major-ness
           | ((N >> 3) << 17)    // N / 8
           | ((M >> 4) << 24);   // M / 16
}

// ------------------------------------------------- bias operands in smem
//
// A column bias that is the same for every tile of a head can be added by the
// tensor core: one more K=16 step whose A rows are (1, 1, 1, 0, ...) and whose B
// row for column c holds the bias value split into three bf16 terms (hi, mid,
// lo: 24 bits). Both operands live in one 128 x 64 bf16 atom with the 128-byte
// swizzle (the TMA layout: 16-byte chunk j of row r at chunk j ^ (r & 7)):
// logical chunks 0-1 hold the ones, chunks 2 + 2b and 3 + 2b bias buffer b.

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Row r of the ones operand (logical chunks 0 and 1; write both halves: j = 0, 1).
__device__ __forceinline__ void write_ones_chunk(uint8_t *aux, int r, int j)
{
    const uint4 v = j == 0 ? make_uint4(0x3F803F80u, 0x00003F80u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4 *>(aux + r * 128 + ((j ^ (r & 7)) << 4)) = v;
}

// Row r of K-step 3 (logical chunks 6-7) of the atom that holds the ones: (-1, -1, -1,
// 0, ...), the A rows that multiply a bias operand into its negation.
__device__ __forceinline__ void write_neg_ones_step3(uint8_t *aux, int r)
{
    uint8_t *row = aux + r * 128;
    *reinterpret_cast<uint4 *>(row + ((6 ^ (r & 7)) << 4)) = make_uint4(0xBF80BF80u, 0x0000BF80u, 0u, 0u);
    *reinterpret_cast<uint4 *>(row + ((7 ^ (r & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
}

// Row r of the K-step `pair` (logical chunks 2 pair, 2 pair + 1) of an atom: the
// value b as hi + mid + lo bf16 terms.
__device__ __forceinline__ void write_bias_pair(uint8_t *atom, int r, int pair, float b)
{
    const __nv_bfloat16 hi = __float2bfloat16_rn(b);
    const float r1 = b - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    const uint32_t w0 = static_cast<uint32_t>(__bfloat16_as_ushort(hi)) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(mid)) << 16);
    const uint32_t w1 = static_cast<uint32_t>(__bfloat16_as_ushort(lo));
    const int j0 = 2 * pair;
    uint8_t *row = atom + r * 128;
    *reinterpret_cast<uint4 *>(row + ((j0 ^ (r & 7)) << 4)) = make_uint4(w0, w1, 0u, 0u);
    *reinterpret_cast<uint4 *>(row + (((j0 + 1) ^ (r & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
}

// Row r of bias buffer `buf` (K-step 1 + buf of the atom that holds the ones).
__device__ __forceinline__ void write_bias_row(uint8_t *aux, int r, int buf, float b)
{
    write_bias_pair(aux, r, 1 + buf, b);
}

// ---------------------------------------------------------------- numerics

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

}  // namespace alibi
