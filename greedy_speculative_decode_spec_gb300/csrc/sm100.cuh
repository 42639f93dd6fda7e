// sm100.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100 family, here sm_103a)
// features the kernels use: mbarriers, TMA tensor loads, tcgen05 MMA / TMEM.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace spec {
namespace sm100 {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same probe with a bound on how long the thread may be suspended waiting for the
// phase (the suspend-time hint, in ns), so that a short wait limit and an abort are seen.
__device__ __forceinline__ bool mbar_try_wait_for(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
// the suspend bound of the bounded waits: the wait limit, at most 20 us
__device__ __forceinline__ uint32_t wait_hint(uint64_t timeout_ns) {
    return timeout_ns < 20000u ? (uint32_t)timeout_ns : 20000u;
}

// Non-blocking probe of a phase (mbarrier.test_wait): true if it has completed.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The polling loop of mbar_wait, kept out of line so that every wait site costs a few
// instructions of the kernel's instruction footprint. sleep_ns > 0: sleep about that long
// between probes (for threads that are not latency-critical).
static __device__ __noinline__ bool mbar_wait_loop(uint32_t bar, uint32_t parity, volatile int *abort,
                                            uint64_t timeout_ns, uint32_t sleep_ns) {
    // every probe (a try_wait may itself suspend the thread for a while) is followed by the
    // abort and time checks, so that a short limit is honoured
    const uint64_t t0 = globaltimer();
    const uint32_t hint = wait_hint(timeout_ns);
    for (;;) {
        if (mbar_try_wait_for(bar, parity, hint)) return true;
        if (sleep_ns) __nanosleep(sleep_ns);
        if (abort != nullptr && *abort) return false;
        if (globaltimer() - t0 > timeout_ns) return false;
    }
}

// The same wait by non-blocking probes (mbarrier.test_wait), for threads that share a warp
// with another thread on its own loop: a probe never holds the warp, so the other thread's
// path keeps being issued while this one waits.
static __device__ __noinline__ bool mbar_wait_poll(uint32_t bar, uint32_t parity, volatile int *abort,
                                            uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test(bar, parity)) return true;
        if ((i & 7u) == 0) {
            if (abort != nullptr && *abort) return false;
            if (globaltimer() - t0 > timeout_ns) return false;
        }
    }
}

// Waits for the phase of the given parity to complete. Gives up (returns false) when
// *abort becomes non-zero (abort may be null: then only the time limit applies) or after
// timeout_ns of wall time, so no wait can hang.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          uint64_t timeout_ns) {
    // a limit below 1 us (a test setting) is watched with non-blocking probes: a suspended
    // probe could outlast it
    if (timeout_ns < 1000u) return mbar_test(bar, parity) || mbar_wait_poll(bar, parity, abort, timeout_ns);
    return mbar_try_wait_for(bar, parity, wait_hint(timeout_ns)) || mbar_wait_loop(bar, parity, abort, timeout_ns, 0);
}

// The same wait for a thread that is not latency-critical: between probes it sleeps about
// sleep_ns, leaving the SM sub-partition's issue slots to the warps that do the math.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, volatile int *abort,
                                                uint64_t timeout_ns, uint32_t sleep_ns) {
    if (timeout_ns < 1000u) return mbar_test(bar, parity) || mbar_wait_poll(bar, parity, abort, timeout_ns);
    return mbar_try_wait_for(bar, parity, wait_hint(timeout_ns)) ||
           mbar_wait_loop(bar, parity, abort, timeout_ns, sleep_ns);
}

// ---- programmatic dependent launch ----------------------------------------------------------

// Waits until the grids this one depends on (launched before it in the stream) have completed
// and their memory is visible; returns at once for a grid launched without that dependency.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the grid launched after this one in the stream be scheduled before this grid ends (it
// still waits, in grid_dep_wait, for this grid to complete before it reads its results).
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- TMA ---------------------------------------------------------------------------------

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// ---- cp.async (16-byte global -> shared copies, L2 only) ----------------------------------

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` (without raising its expected count) once every cp.async this thread
// issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// The same copy with a zero fill: when `valid` is false no byte is read (src must still be
// a valid address) and the 16 destination bytes are written as zeros.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void cp_async_wait_dyn(uint32_t n) {
    switch (n) {
        case 0: cp_async_wait<0>(); break;
        case 1: cp_async_wait<1>(); break;
        case 2: cp_async_wait<2>(); break;
        case 3: cp_async_wait<3>(); break;
        case 4: cp_async_wait<4>(); break;
        case 5: cp_async_wait<5>(); break;
        case 6: cp_async_wait<6>(); break;
        default: cp_async_wait<7>(); break;
    }
}


__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- tcgen05 -------------------------------------------------------------------------------

// One warp allocates `ncols` TMEM columns (power of two >= 32); the base address is
// written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T, bf16 inputs, fp32 accumulator (kind::f16).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] . B[smem]^T with 16-bit float inputs: A's M rows are TMEM lanes and
// its K = 16 elements are packed two per 32-bit column (8 columns from a_tmem).
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T with 8-bit float inputs (kind::f8f6f4; the types are in
// the instruction descriptor), fp32 accumulator. One instruction covers K = 32.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp receives TMEM lane
// (quadrant base + i), columns col..col+15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// (TMA / tensor core) accesses.
// 2^x with the SFU's approximate base-2 exponential (PTX ex2.approx.ftz: about 2 ulp,
// subnormal results flushed to zero; 2^-inf = 0).
// maximum of v over the 32 lanes of the warp, in every lane (NaN inputs are ignored, as by
// fmaxf)
__device__ __forceinline__ float warp_max_f32(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes
// (64 bf16), 8-row groups 1024 bytes apart. The tile base must be 1024-byte aligned;
// stepping 16 elements along K adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);          // start address
    d |= (uint64_t)1u << 16;                          // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;    // stride byte offset: next 8-row group
    d |= (uint64_t)1u << 46;                          // descriptor version (sm_100 family)
    d |= (uint64_t)2u << 61;                          // layout: 128-byte swizzle
    return d;
}

// Shared-memory matrix descriptor: MN-major operand, 128-byte swizzle. Each row of 128
// bytes holds 64 consecutive MN elements of one K index; 8 K rows form a 1024-byte atom
// (stride byte offset 1024); the next 64 MN elements sit `lbo` bytes further.
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Shared-memory matrix descriptor, K-major operand whose rows are `row_bytes` (64 or 128)
// long with the swizzle of that width; 8-row groups `sbo` bytes apart (8 * row_bytes for a
// dense tile; 0 makes every group read the first one). The tile base must be aligned to
// 8 * row_bytes; stepping 32 bytes along K adds 32 to the start address.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr, uint32_t row_bytes, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)(row_bytes == 64 ? 4u : 2u) << 61;  // 64-byte or 128-byte swizzle
    return d;
}

// Advances a shared-memory matrix descriptor's start address by `bytes` (a multiple of 16).
// The address field holds bits 4..17 of the byte address, so for any shared-memory address
// the sum never carries out of it: two integer adds instead of a new descriptor per MMA.
__device__ __forceinline__ uint64_t desc_advance(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

// Shared-memory matrix descriptor: MN-major operand, 32-byte swizzle. Each 32-byte row holds
// 16 consecutive MN elements of one K index; 8 K rows form a 256-byte atom (stride byte
// offset 256); the next 16 MN elements sit `lbo` bytes further. The base must be 256-byte
// aligned; stepping 16 K rows adds 512 bytes to the start address.
__device__ __forceinline__ uint64_t desc_mnmajor_sw32(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((256u >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)6u << 61;  // 32-byte swizzle
    return d;
}

// Instruction descriptor, kind::f8f6f4 with E4M3 A and B (K-major), fp32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f8_e4m3(int M, int N) {
    return (1u << 4)                                  // D format: f32
           | (0u << 7)                                // A format: E4M3
           | (0u << 10)                               // B format: E4M3
           | ((uint32_t)(N >> 3) << 17)               // N / 8
           | ((uint32_t)(M >> 4) << 24);              // M / 16
}

// Instruction descriptor, kind::f16: 16-bit A and B (bf16 or f16), fp32 D, shape M x N;
// a_mn / b_mn select an MN-major operand.
__host__ __device__ constexpr uint32_t idesc_f16kind(int M, int N, bool f16_inputs, bool a_mn, bool b_mn) {
    return (1u << 4)                                  // D format: f32
           | ((f16_inputs ? 0u : 1u) << 7)            // A format: f16 (0) or bf16 (1)
           | ((f16_inputs ? 0u : 1u) << 10)           // B format
           | ((a_mn ? 1u : 0u) << 15)                 // A major
           | ((b_mn ? 1u : 0u) << 16)                 // B major
           | ((uint32_t)(N >> 3) << 17)               // N / 8
           | ((uint32_t)(M >> 4) << 24);              // M / 16
}

__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return idesc_f16kind(M, N, false, false, false);
}

}  // namespace sm100
}  // namespace spec
