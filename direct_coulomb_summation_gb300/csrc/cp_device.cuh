// cp_device.cuh -- small sm_103a device helpers written as inline PTX:
// SFU reciprocal square root, shared-memory mbarriers, 1-D bulk (TMA) copies
// from global to shared memory, and a bounded barrier wait.
#pragma once

#include <cstdint>

namespace cpmap {

// Longest a thread waits on an mbarrier before it records
// CP_DEVICE_WAIT_TIMEOUT and carries on (nanoseconds of %globaltimer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Index checks of the checked build (compiled with -DCP_BOUNDS_CHECKS):
// CP_IN(i, n, status) is true when 0 <= i < n; when it is not, the checked
// build records CP_DEVICE_RANGE (0x2) in *status and the caller skips the
// access.  In the release build every check is the constant `true`.
#ifdef CP_BOUNDS_CHECKS
__device__ __forceinline__ bool cp_in_range(long long i, long long n, unsigned int *status) {
    if (i >= 0 && i < n) return true;
    atomicOr(status, 0x2u);
    return false;
}
#define CP_IN(i, n, status) (::cpmap::cp_in_range((long long)(i), (long long)(n), (status)))
#else
// the release build only references the operands (no code is generated)
#define CP_IN(i, n, status) ((void)(i), (void)(n), true)
#endif

// rsqrt on the SFU (MUFU): one instruction, flush-to-zero variant.
__device__ __forceinline__ float sfu_rsqrt(float x) {
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two reciprocal square roots on the FMA pipe instead of the SFU, for
// positive normal inputs, returned divided by sqrt(2): v = rsqrt(x)/sqrt(2).
// The initial estimate is that of the "fast inverse square root" (integer
// 0x5f3759df - bits/2; C. Lomont, "Fast Inverse Square Root", 2003) with
// 2^22 taken off the constant, which halves it in the log domain, i.e.
// divides it by about sqrt(2).  Newton's step y <- y (3/2 - (x/2) y^2) for
// y = sqrt(2) v reads v <- v (3/2 - x v^2): it needs x itself rather than
// x/2, and written as v <- v (x v^2 - 3/2) it needs no negated operand
// either (the sign of v flips at each step, and two steps restore it).  So
// two steps cost 6 f32x2 operations instead of 7.  Relative error after the
// second step below 5e-6 (the Newton error roughly squares, times 3/2, plus
// fp32 rounding; 4.75e-6 over every fp32 in [1, 4), and the error repeats
// every factor of 4).  The caller multiplies by sqrt(2) once per sum.
__device__ __forceinline__ float2 fma_rsqrt2_scaled(float2 x) {
    float2 v = make_float2(__int_as_float(0x5ef759df - (__float_as_int(x.x) >> 1)),
                           __int_as_float(0x5ef759df - (__float_as_int(x.y) >> 1)));
    const float2 m15 = make_float2(-1.5f, -1.5f);
    v = __fmul2_rn(v, __ffma2_rn(x, __fmul2_rn(v, v), m15));
    v = __fmul2_rn(v, __ffma2_rn(x, __fmul2_rn(v, v), m15));
    return v;
}

// sqrt(2) rounded to fp32: undoes the scaling of fma_rsqrt2_scaled.
constexpr float kSqrt2 = 1.41421356f;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t arrivals) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(arrivals) : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy and the cluster.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Raises the transaction bytes that the current phase of `bar` waits for
// (without arriving): several copies can then complete on one phase.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for phase `parity` of `bar` to complete, at most kWaitLimitNs.  On
// time-out it sets CP_DEVICE_WAIT_TIMEOUT in *status and returns false; the
// caller then carries on (its data are wrong, the status says so) so that no
// thread is left behind at a later block barrier.  After a time-out the
// CTA's shared memory is undefined: a bulk copy issued before it may still
// land in a stage that is being reused, or after the CTA has exited.  The
// launch's results are then invalid, which the status word reports; the
// issuing threads stop issuing copies once one of their waits gave up.
__device__ __forceinline__ bool mbar_wait_limit(uint64_t *bar, uint32_t parity, unsigned int *status,
                                                unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, 1u /* CP_DEVICE_WAIT_TIMEOUT */);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned int *status) {
    return mbar_wait_limit(bar, parity, status, kWaitLimitNs);
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream-serialization attribute may be scheduled while the kernel before
// it on the stream is still running; pdl_wait() blocks until that kernel
// has completed and its memory operations are visible, so it comes before
// any global memory access.  pdl_launch_dependents() lets the next such
// kernel start being scheduled.  Both are no-ops without a programmatic
// dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completion counted on
// `bar` in bytes.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

}  // namespace cpmap
