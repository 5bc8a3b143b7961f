// pkv_device.cuh -- device-side helpers: mbarrier + 1-D bulk-copy (TMA) PTX
// wrappers with bounded waits, element conversions, error reporting.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pkv_internal.h"

namespace pkv {

// Upper bound on mbarrier polls before a wait gives up and reports
// PKV_DEVERR_TIMEOUT.  Each poll suspends the thread until the phase
// completes or kWaitHintNs elapses, so the bound is at most about
// kWaitLimit * kWaitHintNs = 1.6 s of wall time -- far beyond any legitimate
// copy latency -- while a waiting warp issues few instructions.
constexpr uint32_t kWaitLimit = 1u << 14;
constexpr uint32_t kWaitHintNs = 100000;

__device__ __forceinline__ void report(unsigned int* err, unsigned int bit) {
    atomicOr(err, bit);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kWaitHintNs)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier.  dst,
// src and bytes must be multiples of 16.  The evict-first hint keeps
// once-read KV tiles from displacing other lines in L2.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// ---------------------------------------------------------------- elements
// Element type tags.
struct F16 {
    using storage = __half;
    static constexpr int bytes = 2;
};
struct BF16 {
    using storage = __nv_bfloat16;
    static constexpr int bytes = 2;
};
struct E4M3 {
    using storage = __nv_fp8_e4m3;
    static constexpr int bytes = 1;
};

// Convert N packed elements (N*bytes of raw storage, read as 32-bit words) to
// fp32.  bf16 -> f32 is exact (the bf16 bits are the upper half of the f32);
// f16 -> f32 and e4m3 -> f16 -> f32 use the hardware conversions (exact).
template <typename T, int N>
struct Unpack;

template <int N>
struct Unpack<BF16, N> {
    static_assert(N % 2 == 0, "");
    __device__ __forceinline__ static void run(const uint32_t* w, float* f) {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

template <int N>
struct Unpack<F16, N> {
    static_assert(N % 2 == 0, "");
    __device__ __forceinline__ static void run(const uint32_t* w, float* f) {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
            float2 x = __half22float2(h);
            f[2 * i] = x.x;
            f[2 * i + 1] = x.y;
        }
    }
};

template <int N>
struct Unpack<E4M3, N> {
    static_assert(N % 4 == 0, "");
    __device__ __forceinline__ static void run(const uint32_t* w, float* f) {
#pragma unroll
        for (int i = 0; i < N / 4; ++i) {
            __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] & 0xffffu), __NV_E4M3);
            __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] >> 16), __NV_E4M3);
            float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
            float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
            f[4 * i] = a.x;
            f[4 * i + 1] = a.y;
            f[4 * i + 2] = b.x;
            f[4 * i + 3] = b.y;
        }
    }
};

// Load N elements (N*bytes, 8- or 16-byte aligned) as 32-bit words.
template <int BYTES>
__device__ __forceinline__ void load_words(const void* p, uint32_t* w) {
    static_assert(BYTES == 4 || BYTES == 8 || BYTES == 16, "");
    if constexpr (BYTES == 16) {
        uint4 x = *reinterpret_cast<const uint4*>(p);
        w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
    } else if constexpr (BYTES == 8) {
        uint2 x = *reinterpret_cast<const uint2*>(p);
        w[0] = x.x; w[1] = x.y;
    } else {
        w[0] = *reinterpret_cast<const uint32_t*>(p);
    }
}

__device__ __forceinline__ float to_float(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ typename T::storage from_float(float x);
template <>
__device__ __forceinline__ __half from_float<F16>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<BF16>(float x) { return __float2bfloat16_rn(x); }

// ------------------------------------------- programmatic dependent launch
// Waits until the grid this launch programmatically depends on (the decode
// kernel that wrote the partials) has completed and its writes are
// visible; returns at once for a launch without that dependency.
__device__ __forceinline__ void wait_primary_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the launch that programmatically depends on this grid start its
// CTAs once every CTA of this grid has made this call (or exited).
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace pkv
