// fd_device.cuh -- device-side building blocks shared by the libfd kernels:
// mbarrier pipeline primitives, bulk (TMA) global->shared copies, bounded
// waits, bf16 unpacking and the packed fp32x2 arithmetic of sm_100-family GPUs.
// Everything here is inline PTX or CUDA intrinsics for sm_103a.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace fd {

// Device status bits (see fd_device_status in fd.h).
constexpr unsigned kStatusBadPage = 1u;
constexpr unsigned kStatusTimeout = 2u;
constexpr unsigned kStatusBadSeqLen = 4u;

// Sequence length as the kernels use it: seq_lens[b] clamped to [0, L_max]
// (an out-of-range entry is recorded in `status`).
__device__ __forceinline__ int clamped_len(const int32_t* seq_lens, int b, int L_max, unsigned* status) {
    if (!seq_lens) return L_max;
    const int L = seq_lens[b];
    if (L < 0 || L > L_max) {
        if (status && threadIdx.x == 0) atomicOr(status, kStatusBadSeqLen);
        return L < 0 ? 0 : L_max;
    }
    return L;
}

// A pipeline wait gives up after this long (nanoseconds of %globaltimer) or
// this many polls, whichever comes first; the kernel then records
// kStatusTimeout and finishes without touching the stage.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr unsigned kWaitLimitPolls = 1u << 26;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes initialised barriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// Waits for the phase with the given parity to complete.  Returns false if
// the wait hit its limit (the caller records kStatusTimeout and stops).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (unsigned it = 1; it < kWaitLimitPolls; ++it) {
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 1023u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
    return false;
}

// L2 policy for data that is streamed exactly once.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk asynchronous copy global -> shared (TMA, non-tensor form); completion
// is signalled on `bar` as transaction bytes.  dst, src 16-byte aligned;
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and (in that kernel) wait for this grid's results.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Named barrier over a subset of warps (id 1..15; the count is in threads).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 16-byte shared-memory load.
__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

// bf16x2 word -> two fp32 (exact: bf16 is the top half of binary32).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float2 f2mul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 f2fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ unsigned short f32_to_bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

}  // namespace fd
