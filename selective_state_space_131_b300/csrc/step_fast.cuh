// step_fast.cuh -- decode step of the Mamba-3 scan for the common shapes
// (P in {32, 64, 128}, N % 8 == 0, at most 256 threads per (b, h), R in
// {1, 2, 4}; 16-byte aligned tensors): one 128-bit-load-per-row, barrier-light kernel that keeps many
// state bytes in flight.  The generic m3_step_kernel (step_simt.cuh) serves
// every other shape.
//
// Per (b, h), the update of the Mamba-3 summary page (§3.1 eq. (5)-(6) with
// the 2x2 rotation blocks of §3.2, Proposition 3.2.1, and the rank-R input of
// §3.3), in the complex frame:
//   h' <- Rot(theta_t)(alpha h' + beta prev_B^T prev_x) + gamma B_t^T x_t,
//   y_t[r] = C_t[r]^T h'.
// Thread (g, q) of a CTA owns rows 8 g .. 8 g + 7 (four rotation pairs) and
// columns 4 q .. 4 q + 3 of the N x P fp32 state: it issues its eight 16-byte
// state loads first, reads the token's small inputs through L1, updates the
// state in registers, streams it back, and adds its rows' share of y_t;
// partial sums meet in shared memory once.
#pragma once

#include "common.cuh"
#include "ptx_sm100.cuh"

namespace m3fast {

constexpr int kRPT = 8;   // state rows per thread

template <typename T>
struct Vec;
template <>
struct Vec<float> {
    // 8 consecutive elements (32 bytes) as floats
    static __device__ __forceinline__ void ld8(const float* p, float (&o)[8]) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p));
        const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    }
    // 4 consecutive elements (16 bytes)
    static __device__ __forceinline__ void ld4(const float* p, float (&o)[4]) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p));
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    }
    // 2 consecutive elements (8 bytes)
    static __device__ __forceinline__ float2 ld2(const float* p) { return __ldg(reinterpret_cast<const float2*>(p)); }
    static __device__ __forceinline__ void st(float* p, float v) { p[0] = v; }
};
template <>
struct Vec<__nv_bfloat16> {
    static __device__ __forceinline__ float lo(uint32_t u) { return __uint_as_float(u << 16); }
    static __device__ __forceinline__ float hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
    static __device__ __forceinline__ void ld8(const __nv_bfloat16* p, float (&o)[8]) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
        o[0] = lo(a.x); o[1] = hi(a.x); o[2] = lo(a.y); o[3] = hi(a.y);
        o[4] = lo(a.z); o[5] = hi(a.z); o[6] = lo(a.w); o[7] = hi(a.w);
    }
    static __device__ __forceinline__ void ld4(const __nv_bfloat16* p, float (&o)[4]) {
        const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
        o[0] = lo(a.x); o[1] = hi(a.x); o[2] = lo(a.y); o[3] = hi(a.y);
    }
    static __device__ __forceinline__ float2 ld2(const __nv_bfloat16* p) {
        const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p));
        return make_float2(lo(u), hi(u));
    }
    static __device__ __forceinline__ void st(__nv_bfloat16* p, float v) { p[0] = __float2bfloat16_rn(v); }
};

// x - n 2 pi with n = rint(x / 2 pi): two-constant (Cody-Waite) reduction,
// 2 pi = 6.28125 + 1.9353071795864769e-3 with the first constant exact in 8 bits.
__device__ __forceinline__ float reduce_2pi(float x) {
    const float n = rintf(x * 0.15915494309189535f);
    return fmaf(-n, 1.9353071795864769e-3f, fmaf(-n, 6.28125f, x));
}

struct StepArgs {
    int H, N, P, P4;      // P4 = P / 4 threads along the columns
};

// Resident 128-thread CTAs per SM the register budget is sized for: the
// state loads of many CTAs must be in flight to cover DRAM latency, and a
// larger rank needs more registers for its inputs.
__host__ __device__ constexpr int min_ctas(int R, int maxt) { return (R == 1 ? 6 : R == 2 ? 5 : 4) * 128 / maxt; }

// blockDim = P4 * (N / 8) <= MAXT; grid = b * h.
template <typename T, int R, int MAXT>
__global__ void __launch_bounds__(MAXT, min_ctas(R, MAXT)) m3_step_fast_kernel(StepArgs a, float* __restrict__ state,
                                                           const T* __restrict__ x_t, const float* __restrict__ dt_t,
                                                           const float* __restrict__ A, const T* __restrict__ B_t,
                                                           const T* __restrict__ C_t, const float* __restrict__ lam_t,
                                                           const T* __restrict__ theta_t, const T* __restrict__ prev_B,
                                                           const T* __restrict__ prev_x, T* __restrict__ y_t) {
    extern __shared__ __align__(16) float red[];   // [warps][R][P]
    const int N = a.N, P = a.P, P4 = a.P4;
    if ((int)blockDim.x != P4 * (N / kRPT)) {
        if (threadIdx.x == 0) m3::set_status(m3::kStatusBadLaunch);
        return;
    }
    const int64_t unit = blockIdx.x;
    const int h = (int)(unit % a.H);
    const int q = threadIdx.x % P4, g = threadIdx.x / P4;
    const int n0 = g * kRPT, p0 = 4 * q;
    float* st = state + unit * (int64_t)N * P + (int64_t)n0 * P + p0;

    // 1. state loads first (the bulk of the bytes)
    float4 hs[kRPT];
#pragma unroll
    for (int i = 0; i < kRPT; ++i) hs[i] = __ldcs(reinterpret_cast<const float4*>(st + (int64_t)i * P));

    // 2. the token's scalars and this thread's slices of the inputs
    const float d = __ldg(dt_t + unit);
    const float l = lam_t ? __ldg(lam_t + unit) : 1.0f;
    const float alpha = expf(d * __ldg(A + h));
    const float beta = (1.0f - l) * d * alpha;
    const float gamma = l * d;
    float xr[R][4], pxr[R][4];
    const bool has_prev = prev_B != nullptr;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        Vec<T>::ld4(x_t + (unit * R + r) * P + p0, xr[r]);
        if (has_prev) {
            Vec<T>::ld4(prev_x + (unit * R + r) * P + p0, pxr[r]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) pxr[r][j] = 0.0f;
        }
    }
    const T* Bp = B_t + unit * R * N + n0;
    const T* Cp = C_t + unit * R * N + n0;
    const T* pBp = has_prev ? prev_B + unit * R * N + n0 : nullptr;
    float cs[kRPT / 2], sn[kRPT / 2];
    {
        float th[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (theta_t) Vec<T>::ld4(theta_t + unit * (N / 2) + n0 / 2, th);
#pragma unroll
        for (int m = 0; m < kRPT / 2; ++m) __sincosf(reduce_2pi(th[m]), &sn[m], &cs[m]);
    }

    // 3. update: rows (n0 + 2m, n0 + 2m + 1) form rotation pair k = n0 / 2 + m
    float yp[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j) yp[r][j] = 0.0f;
#pragma unroll
    for (int m = 0; m < kRPT / 2; ++m) {
        const float* h0 = reinterpret_cast<const float*>(&hs[2 * m]);
        const float* h1 = reinterpret_cast<const float*>(&hs[2 * m + 1]);
        // B, prev_B, C of this pair's two rows (L1 broadcasts: every column
        // thread of the row group reads the same values)
        float2 br[R], pbr[R], cr[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            br[r] = Vec<T>::ld2(Bp + r * N + 2 * m);
            cr[r] = Vec<T>::ld2(Cp + r * N + 2 * m);
            pbr[r] = has_prev ? Vec<T>::ld2(pBp + r * N + 2 * m) : make_float2(0.0f, 0.0f);
        }
        float o0[4], o1[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float v0 = 0.0f, v1 = 0.0f, u0 = 0.0f, u1 = 0.0f;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                v0 = fmaf(pbr[r].x, pxr[r][j], v0);
                v1 = fmaf(pbr[r].y, pxr[r][j], v1);
                u0 = fmaf(br[r].x, xr[r][j], u0);
                u1 = fmaf(br[r].y, xr[r][j], u1);
            }
            const float z0 = fmaf(alpha, h0[j], beta * v0);
            const float z1 = fmaf(alpha, h1[j], beta * v1);
            // (a, b) -> (a cos - b sin, a sin + b cos), then + gamma u
            o0[j] = fmaf(gamma, u0, fmaf(cs[m], z0, -sn[m] * z1));
            o1[j] = fmaf(gamma, u1, fmaf(sn[m], z0, cs[m] * z1));
#pragma unroll
            for (int r = 0; r < R; ++r) yp[r][j] = fmaf(cr[r].x, o0[j], fmaf(cr[r].y, o1[j], yp[r][j]));
        }
        __stcs(reinterpret_cast<float4*>(st + (int64_t)(2 * m) * P), make_float4(o0[0], o0[1], o0[2], o0[3]));
        __stcs(reinterpret_cast<float4*>(st + (int64_t)(2 * m + 1) * P), make_float4(o1[0], o1[1], o1[2], o1[3]));
    }

    // 4. y_t: sum the row groups -- lanes P4 apart in a warp, then warps in shared memory
#pragma unroll
    for (int o = P4; o < 32; o <<= 1)
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int j = 0; j < 4; ++j) yp[r][j] += __shfl_xor_sync(0xffffffffu, yp[r][j], o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    // a warp holds all P columns when P4 <= 32 (the shapes this kernel takes)
    if (lane < P4) {
#pragma unroll
        for (int r = 0; r < R; ++r)
            *reinterpret_cast<float4*>(red + (warp * R + r) * P + p0) = make_float4(yp[r][0], yp[r][1], yp[r][2], yp[r][3]);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < R * P; e += blockDim.x) {
        float acc = 0.0f;
        for (int w = 0; w < nwarps; ++w) acc += red[w * R * P + e];
        Vec<T>::st(y_t + unit * R * P + e, acc);
    }
}

// The shapes m3_step_fast_kernel takes (with every tensor 16-byte aligned):
// P / 4 a power of two between 8 and 32 (the y reduction pairs lanes P / 4
// apart), N a multiple of 8, one (b, h) in 32..256 threads.
inline bool supports(int64_t N, int64_t P, int64_t R) {
    if (R != 1 && R != 2 && R != 4) return false;
    if (N % kRPT != 0 || (P != 32 && P != 64 && P != 128)) return false;
    const int64_t threads = (P / 4) * (N / kRPT);
    return threads >= 32 && threads <= 256 && threads % 32 == 0;
}

inline int threads(int64_t N, int64_t P) { return (int)((P / 4) * (N / kRPT)); }
inline size_t smem_bytes(int64_t N, int64_t P, int64_t R) { return (size_t)(threads(N, P) / 32) * R * P * 4; }

}  // namespace m3fast
