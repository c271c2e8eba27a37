// step_ring.cuh -- decode step of the Mamba-3 scan (m3_step) with the state
// and the token's inputs staged through a shared-memory ring by untiled bulk
// copies: persistent CTAs walk the (b, h) units, and while one unit is being
// updated the copies of the next units are already in flight, so the bytes
// in flight do not depend on the registers of the update.
//
// Per (b, h) the update is that of step_fast.cuh (Mamba-3 summary page §3.1
// eq. (5)-(6) with the 2x2 rotation blocks of §3.2, Proposition 3.2.1, and the
// rank-R input of §3.3), in the complex frame:
//   h' <- Rot(theta_t)(alpha h' + beta prev_B^T prev_x) + gamma B_t^T x_t,
//   y_t[r] = C_t[r]^T h',
// with the same thread tiling: thread (g, q) owns rows 8 g .. 8 g + 7 (four
// rotation pairs) and columns 4 q .. 4 q + 3 of the N x P fp32 state.
//
// Ring: kStages stages, each holding one unit's state and inputs laid out as
// in global memory (every block a multiple of 16 bytes), filled by one thread
// with cp.async.bulk and completed on the stage's mbarrier (bounded waits: a
// wait that runs out sets the device status word and the CTA stops after the
// unit at hand, once its copies in flight have landed or their wait ran out).
// The updated state goes straight from registers to global memory; y meets in
// a double-buffered reduction area, one barrier per unit.
#pragma once

#include "common.cuh"
#include "ptx_sm100.cuh"

namespace m3ring {

constexpr int kStages = 2;   // 512 threads per SM (measured on R = 4: 3 stages 3 % and 4 stages 16 % slower)
constexpr int kRPT = 8;                        // state rows per thread
constexpr long long kWaitBudget = 4000000000LL;   // clock cycles (~2 s)

// Shared-memory layout (bytes).  Per stage: state | x | prev_x | B | C | prev_B | theta.
struct Geo {
    int H, N, P, P4, R, nthreads;
    int64_t units;
    uint32_t b_state, b_x, b_B, b_th;          // bytes per unit
    uint32_t o_x, o_px, o_B, o_C, o_pB, o_th;  // offsets inside a stage (state at 0)
    uint32_t stage_bytes, o_red, red_bytes, o_bar, smem_bytes;
};

inline uint32_t up16(uint64_t v) { return (uint32_t)((v + 15) & ~uint64_t(15)); }

inline Geo make_geo(int64_t units, int H, int N, int P, int R, int esize) {
    Geo g;
    g.H = H; g.N = N; g.P = P; g.P4 = P / 4; g.R = R;
    g.nthreads = (P / 4) * (N / kRPT);
    g.units = units;
    g.b_state = (uint32_t)N * P * 4;
    g.b_x = (uint32_t)(R * P * esize);
    g.b_B = (uint32_t)(R * N * esize);
    g.b_th = (uint32_t)(N / 2 * esize);
    uint32_t o = up16(g.b_state);
    g.o_x = o;  o += up16(g.b_x);
    g.o_px = o; o += up16(g.b_x);
    g.o_B = o;  o += up16(g.b_B);
    g.o_C = o;  o += up16(g.b_B);
    g.o_pB = o; o += up16(g.b_B);
    g.o_th = o; o += up16(g.b_th);
    g.stage_bytes = (o + 127) & ~127u;
    g.o_red = kStages * g.stage_bytes;
    g.red_bytes = (uint32_t)(g.nthreads / 32) * R * P * 4;
    g.o_bar = g.o_red + 2 * g.red_bytes;
    g.smem_bytes = g.o_bar + kStages * 8;
    return g;
}

// The shapes this kernel takes: ranks 2 and 4 (more arithmetic per state
// element; rank 1 is bound by the state round trip alone, which the plain
// kernel's eight 16-byte loads per thread already cover) in the single-step
// fast kernel's shapes whose per-unit blocks are all multiples of 16 bytes
// (the bulk copies' unit).
inline bool supports(int64_t N, int64_t P, int64_t R, int esize) {
    if (R != 2 && R != 4) return false;
    if (N % kRPT != 0 || (P != 32 && P != 64 && P != 128)) return false;
    const int64_t threads = (P / 4) * (N / kRPT);
    if (threads < 32 || threads > 256 || threads % 32 != 0) return false;
    return (R * P * esize) % 16 == 0 && (R * N * esize) % 16 == 0 && (N / 2 * esize) % 16 == 0;
}

// Loads from the shared-memory stage.
template <typename T>
struct SV;
template <>
struct SV<float> {
    static __device__ __forceinline__ void ld4(const float* p, float (&o)[4]) {
        const float4 a = *reinterpret_cast<const float4*>(p);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    }
    static __device__ __forceinline__ float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }
    static __device__ __forceinline__ void st(float* p, float v) { p[0] = v; }
};
template <>
struct SV<__nv_bfloat16> {
    static __device__ __forceinline__ float lo(uint32_t u) { return __uint_as_float(u << 16); }
    static __device__ __forceinline__ float hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
    static __device__ __forceinline__ void ld4(const __nv_bfloat16* p, float (&o)[4]) {
        const uint2 a = *reinterpret_cast<const uint2*>(p);
        o[0] = lo(a.x); o[1] = hi(a.x); o[2] = lo(a.y); o[3] = hi(a.y);
    }
    static __device__ __forceinline__ float2 ld2(const __nv_bfloat16* p) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
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

// blockDim = P4 * (N / 8) <= MAXT; grid = persistent CTAs (at most one per
// unit), each taking units blockIdx.x, blockIdx.x + gridDim.x, ...
template <typename T, int R, int MAXT>
__global__ void __launch_bounds__(MAXT, 512 / MAXT)
    m3_step_ring_kernel(const Geo g, float* __restrict__ state, const T* __restrict__ x_t,
                        const float* __restrict__ dt_t, const float* __restrict__ A, const T* __restrict__ B_t,
                        const T* __restrict__ C_t, const float* __restrict__ lam_t, const T* __restrict__ theta_t,
                        const T* __restrict__ prev_B, const T* __restrict__ prev_x, T* __restrict__ y_t) {
    extern __shared__ __align__(128) uint8_t smem[];
    if ((int)blockDim.x != g.nthreads || g.R != R) {
        if (threadIdx.x == 0) m3::set_status(m3::kStatusBadLaunch);
        return;
    }
    const int N = g.N, P = g.P, P4 = g.P4;
    const int tid = threadIdx.x, q = tid % P4, grp = tid / P4;
    const int n0 = grp * kRPT, p0 = 4 * q;
    const int warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + g.o_bar);
    const bool has_prev = prev_B != nullptr;
    const int64_t stride = gridDim.x;
    const uint32_t tx = g.b_state + g.b_x + 2 * g.b_B + (has_prev ? g.b_x + g.b_B : 0u) + (theta_t ? g.b_th : 0u);

    // one thread fills stage s with unit u
    auto issue = [&](int64_t u, int s) {
        uint8_t* st = smem + (uint32_t)s * g.stage_bytes;
        uint64_t* bar = &bars[s];
        ptx::mbar_arrive_expect_tx(bar, tx);
        ptx::bulk_g2s(st, state + u * (int64_t)N * P, g.b_state, bar);
        ptx::bulk_g2s(st + g.o_x, x_t + u * R * P, g.b_x, bar);
        ptx::bulk_g2s(st + g.o_B, B_t + u * R * N, g.b_B, bar);
        ptx::bulk_g2s(st + g.o_C, C_t + u * R * N, g.b_B, bar);
        if (has_prev) {
            ptx::bulk_g2s(st + g.o_px, prev_x + u * R * P, g.b_x, bar);
            ptx::bulk_g2s(st + g.o_pB, prev_B + u * R * N, g.b_B, bar);
        }
        if (theta_t) ptx::bulk_g2s(st + g.o_th, theta_t + u * (N / 2), g.b_th, bar);
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) ptx::mbar_init(&bars[s], 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const int64_t u0 = blockIdx.x;
    if (tid == 0)
        for (int s = 0; s < kStages; ++s) {
            const int64_t u = u0 + s * stride;
            if (u < g.units) issue(u, s);
        }
    // this unit's scalars; the next unit's are loaded one unit ahead
    float d = 0.0f, l = 1.0f, a_h = 0.0f;
    if (u0 < g.units) {
        d = __ldg(dt_t + u0);
        l = lam_t ? __ldg(lam_t + u0) : 1.0f;
        a_h = __ldg(A + (int)(u0 % g.H));
    }
    int it = 0;
    bool fail = false;
    for (int64_t u = u0; u < g.units; u += stride, ++it) {
        const int s = it % kStages;
        const uint32_t par = (uint32_t)(it / kStages) & 1u;
        const int64_t un = u + stride;
        float dn = 0.0f, ln = 1.0f, an = 0.0f;
        if (un < g.units) {
            dn = __ldg(dt_t + un);
            ln = lam_t ? __ldg(lam_t + un) : 1.0f;
            an = __ldg(A + (int)(un % g.H));
        }
        const bool ok = ptx::mbar_wait(&bars[s], par, kWaitBudget);
        if (!ok) m3::set_status(m3::kStatusWaitTimeout);
        const uint8_t* st = smem + (uint32_t)s * g.stage_bytes;

        // 1. this thread's state rows and its slices of the inputs, from the stage
        float4 hs[kRPT];
        {
            const float* hsm = reinterpret_cast<const float*>(st) + n0 * P + p0;
#pragma unroll
            for (int i = 0; i < kRPT; ++i) hs[i] = *reinterpret_cast<const float4*>(hsm + i * P);
        }
        const float alpha = expf(d * a_h);
        const float beta = (1.0f - l) * d * alpha;
        const float gamma = l * d;
        const T* xs = reinterpret_cast<const T*>(st + g.o_x);
        const T* pxs = reinterpret_cast<const T*>(st + g.o_px);
        float xr[R][4], pxr[R][4];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            SV<T>::ld4(xs + r * P + p0, xr[r]);
            if (has_prev) {
                SV<T>::ld4(pxs + r * P + p0, pxr[r]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) pxr[r][j] = 0.0f;
            }
        }
        const T* Bs = reinterpret_cast<const T*>(st + g.o_B) + n0;
        const T* Cs = reinterpret_cast<const T*>(st + g.o_C) + n0;
        const T* pBs = reinterpret_cast<const T*>(st + g.o_pB) + n0;
        float cs[kRPT / 2], sn[kRPT / 2];
        {
            float th[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (theta_t) SV<T>::ld4(reinterpret_cast<const T*>(st + g.o_th) + n0 / 2, th);
#pragma unroll
            for (int m = 0; m < kRPT / 2; ++m) __sincosf(reduce_2pi(th[m]), &sn[m], &cs[m]);
        }

        // 2. update: rows (n0 + 2m, n0 + 2m + 1) form rotation pair n0 / 2 + m; the new
        //    state goes straight to global memory
        float* gst = state + u * (int64_t)N * P + (int64_t)n0 * P + p0;
        float yp[R][4];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int j = 0; j < 4; ++j) yp[r][j] = 0.0f;
#pragma unroll
        for (int m = 0; m < kRPT / 2; ++m) {
            const float* h0 = reinterpret_cast<const float*>(&hs[2 * m]);
            const float* h1 = reinterpret_cast<const float*>(&hs[2 * m + 1]);
            float2 br[R], pbr[R], cr[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                br[r] = SV<T>::ld2(Bs + r * N + 2 * m);
                cr[r] = SV<T>::ld2(Cs + r * N + 2 * m);
                pbr[r] = has_prev ? SV<T>::ld2(pBs + r * N + 2 * m) : make_float2(0.0f, 0.0f);
            }
            float o0[4], o1[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float v0 = 0.0f, v1 = 0.0f, w0 = 0.0f, w1 = 0.0f;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    v0 = fmaf(pbr[r].x, pxr[r][j], v0);
                    v1 = fmaf(pbr[r].y, pxr[r][j], v1);
                    w0 = fmaf(br[r].x, xr[r][j], w0);
                    w1 = fmaf(br[r].y, xr[r][j], w1);
                }
                const float z0 = fmaf(alpha, h0[j], beta * v0);
                const float z1 = fmaf(alpha, h1[j], beta * v1);
                // (a, b) -> (a cos - b sin, a sin + b cos), then + gamma B x^T
                o0[j] = fmaf(gamma, w0, fmaf(cs[m], z0, -sn[m] * z1));
                o1[j] = fmaf(gamma, w1, fmaf(sn[m], z0, cs[m] * z1));
#pragma unroll
                for (int r = 0; r < R; ++r) yp[r][j] = fmaf(cr[r].x, o0[j], fmaf(cr[r].y, o1[j], yp[r][j]));
            }
            __stcs(reinterpret_cast<float4*>(gst + (int64_t)(2 * m) * P), make_float4(o0[0], o0[1], o0[2], o0[3]));
            __stcs(reinterpret_cast<float4*>(gst + (int64_t)(2 * m + 1) * P), make_float4(o1[0], o1[1], o1[2], o1[3]));
        }

        // 3. y: lanes P4 apart in a warp, then the warps in shared memory (two buffers
        //    used in turn, so one barrier per unit suffices)
#pragma unroll
        for (int o = P4; o < 32; o <<= 1)
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int j = 0; j < 4; ++j) yp[r][j] += __shfl_xor_sync(0xffffffffu, yp[r][j], o);
        float* red = reinterpret_cast<float*>(smem + g.o_red + (uint32_t)(it & 1) * g.red_bytes);
        if (lane < P4) {
#pragma unroll
            for (int r = 0; r < R; ++r)
                *reinterpret_cast<float4*>(red + (warp * R + r) * P + p0) =
                    make_float4(yp[r][0], yp[r][1], yp[r][2], yp[r][3]);
        }
        // every thread is done with stage s; a wait that ran out anywhere stops the CTA
        const bool bad = __syncthreads_or(!ok) != 0;
        if (tid == 0 && !bad) {
            const int64_t ua = u + (int64_t)kStages * stride;
            if (ua < g.units) {
                ptx::fence_proxy_async_smem();
                issue(ua, s);
            }
        }
        for (int e = tid; e < R * P; e += blockDim.x) {
            float acc = 0.0f;
            for (int w = 0; w < nwarps; ++w) acc += red[w * R * P + e];
            SV<T>::st(y_t + u * R * P + e, acc);
        }
        if (bad) {
            fail = true;
            break;
        }
        d = dn; l = ln; a_h = an;
    }
    if (fail && tid == 0) {
        // copies still in flight (the failed stage and those issued ahead) land
        // before the CTA leaves, or their bounded wait runs out
        for (int k = 0; k < kStages; ++k) {
            const int it2 = it + k;
            const int64_t u2 = (int64_t)blockIdx.x + (int64_t)it2 * stride;
            if (u2 >= g.units) break;
            (void)ptx::mbar_wait(&bars[it2 % kStages], (uint32_t)(it2 / kStages) & 1u, kWaitBudget);
        }
    }
}

}  // namespace m3ring
