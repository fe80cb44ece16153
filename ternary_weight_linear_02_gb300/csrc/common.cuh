// common.cuh -- device helpers shared by the kernels of libternary_gb300.
//
// Code table ("三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战" §3.1):
// 00 -> 0, 01 -> +1, 10 -> -1, 11 -> 0; weight k of a packed row sits in byte
// k/4 at bits [2(k%4)+1 : 2(k%4)].
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace tl {

// ---------------------------------------------------------------------------
// Branch-free decode of a 32-bit word of 16 codes into 16-bit MMA operands.
//
// With code bits (b1 b0) the value is b0 - b1 for all four codes (00->0,
// 01->+1, 10->-1, 11->0).  Write it in sign-magnitude form: magnitude
// nz = b0 XOR b1, sign = b1.  sign_nz() rewrites every 2-bit field of w in
// place as (b1, nz): bit 2j keeps b0^b1, bit 2j+1 keeps b1.
//
// A 16-bit value whose only possible set bits are 15 (sign) and 14 is
// +-0 or +-2.0 in BOTH fp16 (exponent field 16 -> 2^1) and bf16 (exponent
// field 128 -> 2^1).  So moving field j to bits [15:14] gives exactly
// 2*t: 00 -> +0, 01 -> +2, 10 -> -2, 11 -> -0.  The factor 2 is undone
// in the fp32 epilogue (an exact power-of-two scaling).
//
// pair2(z, j) moves fields j and j+8 (0 <= j < 8) to bits [15:14] and [31:30]:
// one packed f16x2 / bf16x2 register holding {2*t_j, 2*t_{j+8}}.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t sign_nz(uint32_t w) {
    return w ^ ((w >> 1) & 0x55555555u);
}

__device__ __forceinline__ uint32_t pair2(uint32_t z, int j) {
    return (z << (14 - 2 * j)) & 0xC000C000u;
}

// ---------------------------------------------------------------------------
// 16-bit input types
// ---------------------------------------------------------------------------
struct F16 {
    using T = __half;
    static constexpr bool is_bf16 = false;
};
struct BF16 {
    using T = __nv_bfloat16;
    static constexpr bool is_bf16 = true;
};

// fp32 -> output element (round to nearest even for 16-bit outputs)
template <int OUT>
struct OutStore;
template <>
struct OutStore<0> {  // TL_F16
    static __device__ __forceinline__ void st(void *base, int64_t idx, float v) {
        reinterpret_cast<__half *>(base)[idx] = __float2half_rn(v);
    }
};
template <>
struct OutStore<1> {  // TL_BF16
    static __device__ __forceinline__ void st(void *base, int64_t idx, float v) {
        reinterpret_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(v);
    }
};
template <>
struct OutStore<2> {  // TL_F32
    static __device__ __forceinline__ void st(void *base, int64_t idx, float v) {
        reinterpret_cast<float *>(base)[idx] = v;
    }
};

__device__ __forceinline__ float h2f(uint16_t bits) {
    return __half2float(__ushort_as_half(bits));
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch and L2 prefetch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Bulk prefetch of [p, p+bytes) into L2.  p and bytes must be multiples of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Split-phase cluster barrier (all threads of the CTA execute both halves).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Cluster shared memory: the address of `saddr` (a shared::cta address) in the
// CTA of rank `rank`, and stores to such an address.
__device__ __forceinline__ uint32_t cl_map(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cl_st_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void cl_st_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cl_st_v4_f32(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Split-phase cluster barrier with release / acquire ordering of memory
// (shared::cluster included): writes before arrive are visible after wait.
__device__ __forceinline__ void cl_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cl_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// mbarrier + 1-D bulk async copy (global -> this CTA's shared memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
// make an initialised mbarrier visible to the async (bulk copy / TMA) proxy
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
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
// Bounded wait for phase `parity` of an mbarrier: gives up after ~0.5 s of
// spinning (a correct program never gets there) and reports false.
// try_wait that may suspend the thread for up to `ns` nanoseconds while the
// phase is incomplete (a waiting warp then stops competing for issue slots)
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
// Default give-up time of a bounded wait, in SM clock cycles (~0.5 s).
constexpr long long kWaitLimitDefault = 1ll << 30;

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  long long limit = kWaitLimitDefault) {
    if (mbar_try_wait(bar, parity)) return true;  // fast path: no clock read
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 200u)) return true;
        if (clock64() - t0 > limit) return false;
    }
}
// Copy `bytes` (multiple of 16; both addresses 16-byte aligned) from global
// memory into this CTA's shared memory, completing `bytes` transactions on bar.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Device status word codes (written with atomicExch; 0 = OK)
constexpr int kStatusTimeout = 7;

__device__ __forceinline__ uint2 ldg_nc_v2(const void *p) {
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

}  // namespace tl
