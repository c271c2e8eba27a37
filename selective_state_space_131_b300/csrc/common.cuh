// common.cuh -- shared device helpers of libm3scan (one translation unit:
// m3scan.cu includes every kernel file).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace m3 {

// Device status word.  A kernel that gives up on a bounded wait (or detects an
// inconsistent state) ORs a code in here and returns; m3_device_status() reads
// and clears it.  Never trap: the context must stay usable.
__device__ unsigned int g_status;

enum : unsigned int {
    kStatusWaitTimeout = 1u,   // an mbarrier wait ran out of its budget
    kStatusBadLaunch = 2u,     // a kernel saw launch geometry it was not built for
};

__device__ __forceinline__ void set_status(unsigned int code) { atomicOr(&g_status, code); }

// Element I/O for the two input dtypes; all arithmetic is fp32.
template <typename T>
struct IO;
template <>
struct IO<float> {
    static __device__ __forceinline__ float ld(const float* p, int64_t i) { return __ldg(p + i); }
    static __device__ __forceinline__ void st(float* p, int64_t i, float v) { p[i] = v; }
};
template <>
struct IO<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16* p, int64_t i) {
        return __bfloat162float(p[i]);
    }
    static __device__ __forceinline__ void st(__nv_bfloat16* p, int64_t i, float v) {
        p[i] = __float2bfloat16_rn(v);
    }
};

// log2(e), to evaluate exp(x) as 2^(x log2 e) with the hardware exp2.
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace m3
