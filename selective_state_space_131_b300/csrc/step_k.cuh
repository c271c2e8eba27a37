// step_k.cuh -- multi-token decode of the Mamba-3 scan (m3_step_k): k consecutive
// tokens of every (b, h) per launch, the state read and written once.  The thread
// tiling and the small helpers are those of the single-step kernel in step_fast.cuh.
#pragma once

#include "step_fast.cuh"

namespace m3fast {

// Multi-token decode (m3_step_k): k consecutive tokens of every (b, h) in one
// launch, the state read once and written once.  The thread tiling of
// m3_step_fast_kernel; the state stays in registers across the k tokens.
//
// The recurrence is carried in the augmented form
//   g_{j-1} = h'_{j-1} + c_j u_{j-1},   c_j = (1 - lambda_j) dt_j  (so beta_j = c_j alpha_j)
//   h'_j    = alpha_j Rot(theta_j) g_{j-1} + gamma_j u_j,   y_j = C_j^T h'_j
//   g_j     = h'_j + c_{j+1} u_j
// which needs no previous-token product per token (the caller's previous token
// enters once, in g_{-1}); the state written back is h' of the last token.
// The tokens' inputs are staged in shared memory in groups of kGroup with
// 16-byte cp.async copies (the latency is paid once per group, the next group
// loads while this one runs); at the start of a group the threads turn its
// angles and decays into alpha cos / alpha sin per (token, pair) and gamma, c
// per token, once for the whole CTA.  Each token's y meets in a
// double-buffered shared-memory reduction (one barrier per token).  Token
// tensors have the prefill's token-major layout: x [b, k, h, R, P],
// B / C [b, k, h, R, N], theta [b, k, h, N/2], dt / lambda [b, k, h].
constexpr int kGroup = 8;

struct StepKArgs {
    int H, N, P, P4;
    int64_t k;
    // staging layout (bytes): per token x | B | C | theta | dt, lambda; per group
    // buffer also dt, lambda of the token after the group; the previous-token
    // slot x | B; nbuf group buffers; the coefficients of one group
    int xb, nb, kb, tokb, grpb, nbuf;
};

inline StepKArgs stepk_layout(int H, int N, int P, int R, int64_t k, int es) {
    auto up16 = [](int v) { return (v + 15) & ~15; };
    StepKArgs a;
    a.H = H; a.N = N; a.P = P; a.P4 = P / 4; a.k = k;
    a.xb = R * P * es;
    a.nb = up16(R * N * es);
    a.kb = up16((N / 2) * es);
    a.tokb = a.xb + 2 * a.nb + a.kb + 16;
    a.grpb = kGroup * a.tokb + 16;
    a.nbuf = k > kGroup ? 2 : 1;
    return a;
}
// Dynamic shared memory of m3_step_k_kernel: the y reduction (2 x warps x R x P
// floats), the previous-token slot, the group buffers and one group's
// coefficients (alpha cos, alpha sin per token and pair; gamma, c per token).
inline size_t stepk_smem(const StepKArgs& a, int R) {
    const int warps = (a.P4 * (a.N / kRPT)) / 32;
    return (size_t)2 * warps * R * a.P * 4 + (size_t)(a.xb + a.nb) + (size_t)a.nbuf * a.grpb +
           (size_t)kGroup * (a.N / 2) * 8 + (size_t)kGroup * 8;
}

template <typename T>
struct SVec;
template <>
struct SVec<float> {
    static __device__ __forceinline__ void ld4(const uint8_t* p, float (&o)[4]) {
        const float4 a = *reinterpret_cast<const float4*>(p);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    }
    static __device__ __forceinline__ float2 ld2(const uint8_t* p) { return *reinterpret_cast<const float2*>(p); }
    static __device__ __forceinline__ float ld1(const uint8_t* p) { return *reinterpret_cast<const float*>(p); }
};
template <>
struct SVec<__nv_bfloat16> {
    static __device__ __forceinline__ void ld4(const uint8_t* p, float (&o)[4]) {
        const uint2 a = *reinterpret_cast<const uint2*>(p);
        o[0] = Vec<__nv_bfloat16>::lo(a.x); o[1] = Vec<__nv_bfloat16>::hi(a.x);
        o[2] = Vec<__nv_bfloat16>::lo(a.y); o[3] = Vec<__nv_bfloat16>::hi(a.y);
    }
    static __device__ __forceinline__ float2 ld2(const uint8_t* p) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
        return make_float2(Vec<__nv_bfloat16>::lo(u), Vec<__nv_bfloat16>::hi(u));
    }
    static __device__ __forceinline__ float ld1(const uint8_t* p) {
        return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
    }
};

template <typename T, int R, int MAXT>
__global__ void __launch_bounds__(MAXT, min_ctas(R, MAXT)) m3_step_k_kernel(StepKArgs a, float* __restrict__ state,
                                                        const T* __restrict__ x, const float* __restrict__ dt,
                                                        const float* __restrict__ A, const T* __restrict__ Bm,
                                                        const T* __restrict__ Cm, const float* __restrict__ lam,
                                                        const T* __restrict__ theta, const T* __restrict__ prev_B,
                                                        const T* __restrict__ prev_x, T* __restrict__ y) {
    extern __shared__ __align__(16) float red[];   // [2][warps][R][P], then the staging area
    const int N = a.N, P = a.P, P4 = a.P4, H = a.H, K = N / 2;
    constexpr int es = sizeof(T);
    if ((int)blockDim.x != P4 * (N / kRPT)) {
        if (threadIdx.x == 0) m3::set_status(m3::kStatusBadLaunch);
        return;
    }
    const int64_t unit = blockIdx.x;
    const int64_t b = unit / H;
    const int h = (int)(unit % H);
    const int q = threadIdx.x % P4, g = threadIdx.x / P4;
    const int n0 = g * kRPT, p0 = 4 * q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int nthr = blockDim.x;
    float* st = state + unit * (int64_t)N * P + (int64_t)n0 * P + p0;
    uint8_t* prev_slot = reinterpret_cast<uint8_t*>(red + 2 * nwarps * R * P);
    uint8_t* bufs = prev_slot + a.xb + a.nb;
    float* coef = reinterpret_cast<float*>(bufs + (size_t)a.nbuf * a.grpb);   // [kGroup][K][2]
    float* tokc = coef + kGroup * K * 2;                                       // [kGroup][gamma, c_next]
    const int64_t ngroups = (a.k + kGroup - 1) / kGroup;
    const bool has_theta = theta != nullptr;
    const bool theta16 = ((N / 2) * es) % 16 == 0;

    auto gbuf = [&](int64_t gi) { return bufs + (size_t)(gi % a.nbuf) * a.grpb; };
    auto slot = [&](int64_t j) { return gbuf(j / kGroup) + (j % kGroup) * a.tokb; };
    // issue the copies of group gi's tokens, and dt / lambda of the token after it
    // (every thread takes a share; lambda = NULL is written as 1 directly)
    auto issue_group = [&](int64_t gi) {
        const int64_t j0 = gi * kGroup;
        const int nt = (int)((a.k - j0) < kGroup ? (a.k - j0) : kGroup);
        const int cx = a.xb / 16, cn = (R * N * es) / 16;
        const int ck = has_theta ? (theta16 ? ((N / 2) * es) / 16 : ((N / 2) * es) / 4) : 0;
        const int per = cx + 2 * cn + ck + 2;
        for (int e = threadIdx.x; e < nt * per; e += nthr) {
            const int jj = e / per;
            int c = e - jj * per;
            const int64_t j = j0 + jj;
            const int64_t tj = (b * a.k + j) * H + h;
            uint8_t* d = slot(j);
            if (c < cx) { ptx::cp_async16(d + c * 16, reinterpret_cast<const uint8_t*>(x + tj * R * P) + c * 16); continue; }
            c -= cx;
            if (c < cn) { ptx::cp_async16(d + a.xb + c * 16, reinterpret_cast<const uint8_t*>(Bm + tj * R * N) + c * 16); continue; }
            c -= cn;
            if (c < cn) { ptx::cp_async16(d + a.xb + a.nb + c * 16, reinterpret_cast<const uint8_t*>(Cm + tj * R * N) + c * 16); continue; }
            c -= cn;
            uint8_t* dk = d + a.xb + 2 * a.nb;
            const uint8_t* sk = reinterpret_cast<const uint8_t*>(theta + tj * (N / 2));
            if (c < ck) {
                if (theta16) ptx::cp_async16(dk + c * 16, sk + c * 16);
                else ptx::cp_async4(dk + c * 4, sk + c * 4, true);
                continue;
            }
            c -= ck;
            float* ds = reinterpret_cast<float*>(dk + a.kb);
            if (c == 0) ptx::cp_async4(ds, dt + tj, true);
            else if (lam) ptx::cp_async4(ds + 1, lam + tj, true);
            else ds[1] = 1.0f;
        }
        if (threadIdx.x == 0) {
            float* nx = reinterpret_cast<float*>(gbuf(gi) + kGroup * a.tokb);
            const int64_t jn = j0 + kGroup;
            if (jn < a.k) {
                const int64_t tn = (b * a.k + jn) * H + h;
                ptx::cp_async4(nx, dt + tn, true);
                if (lam) ptx::cp_async4(nx + 1, lam + tn, true);
                else nx[1] = 1.0f;
            } else {
                nx[0] = 0.0f;
                nx[1] = 1.0f;
            }
        }
    };

    // the caller's previous token and group 0, then the state (the bulk of the bytes)
    const bool has_prev = prev_B != nullptr;
    if (has_prev) {
        for (int c = threadIdx.x; c < a.xb / 16 + (R * N * es) / 16; c += nthr) {
            if (c < a.xb / 16) ptx::cp_async16(prev_slot + c * 16, reinterpret_cast<const uint8_t*>(prev_x + unit * R * P) + c * 16);
            else ptx::cp_async16(prev_slot + a.xb + (c - a.xb / 16) * 16,
                                 reinterpret_cast<const uint8_t*>(prev_B + unit * R * N) + (c - a.xb / 16) * 16);
        }
    }
    issue_group(0);
    ptx::cp_async_commit();
    float4 hs[kRPT];
#pragma unroll
    for (int i = 0; i < kRPT; ++i) hs[i] = __ldcs(reinterpret_cast<const float4*>(st + (int64_t)i * P));
    const float A_h = __ldg(A + h);

    for (int64_t gi = 0; gi < ngroups; ++gi) {
        const int64_t j0 = gi * kGroup;
        const int nt = (int)((a.k - j0) < kGroup ? (a.k - j0) : kGroup);
        ptx::cp_async_wait_all();   // group gi (the only copies in flight)
        __syncthreads();
        // the group's coefficients: alpha cos, alpha sin per (token, pair); gamma and
        // c of the next token per token
        for (int e = threadIdx.x; e < nt * K; e += nthr) {
            const int jj = e / K, k = e - jj * K;
            const uint8_t* d = slot(j0 + jj);
            const float* sc = reinterpret_cast<const float*>(d + a.xb + 2 * a.nb + a.kb);
            const float al = expf(sc[0] * A_h);
            float sn = 0.0f, cs = 1.0f;
            if (has_theta) __sincosf(reduce_2pi(SVec<T>::ld1(d + a.xb + 2 * a.nb + k * es)), &sn, &cs);
            *reinterpret_cast<float2*>(coef + (jj * K + k) * 2) = make_float2(al * cs, al * sn);
        }
        for (int jj = threadIdx.x; jj < nt; jj += nthr) {
            const float* sc = reinterpret_cast<const float*>(slot(j0 + jj) + a.xb + 2 * a.nb + a.kb);
            const float* sn = (jj + 1 < kGroup) ? reinterpret_cast<const float*>(slot(j0 + jj + 1) + a.xb + 2 * a.nb + a.kb)
                                                : reinterpret_cast<const float*>(gbuf(gi) + kGroup * a.tokb);
            // the token after the last of the call does not exist: c = 0
            const bool last = j0 + jj + 1 >= a.k;
            tokc[2 * jj] = sc[1] * sc[0];
            tokc[2 * jj + 1] = last ? 0.0f : (1.0f - sn[1]) * sn[0];
        }
        if (gi == 0 && has_prev) {
            // g_{-1} = h'_{-1} + c_0 u_{-1}: the caller's previous token enters here once
            const float* s0 = reinterpret_cast<const float*>(slot(0) + a.xb + 2 * a.nb + a.kb);
            const float c0 = (1.0f - s0[1]) * s0[0];
            float px[R][4];
#pragma unroll
            for (int r = 0; r < R; ++r) SVec<T>::ld4(prev_slot + (r * P + p0) * es, px[r]);
#pragma unroll
            for (int i = 0; i < kRPT; ++i) {
                float* hv = reinterpret_cast<float*>(&hs[i]);
                float bb[R];
#pragma unroll
                for (int r = 0; r < R; ++r) bb[r] = SVec<T>::ld1(prev_slot + a.xb + (r * N + n0 + i) * es);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    float u = 0.0f;
#pragma unroll
                    for (int r = 0; r < R; ++r) u = fmaf(bb[r], px[r][jj], u);
                    hv[jj] = fmaf(c0, u, hv[jj]);
                }
            }
        }
        // the next group loads while this one runs (its buffer held group gi - 1)
        if (gi + 1 < ngroups) {
            issue_group(gi + 1);
            ptx::cp_async_commit();
        }
        __syncthreads();

        for (int jj = 0; jj < nt; ++jj) {
            const int64_t j = j0 + jj;
            const uint8_t* cur = slot(j);
            const float2 gc = *reinterpret_cast<const float2*>(tokc + 2 * jj);   // gamma, c_next
            float cf[8];
            {
                const float4 c0 = *reinterpret_cast<const float4*>(coef + (jj * K + n0 / 2) * 2);
                const float4 c1 = *reinterpret_cast<const float4*>(coef + (jj * K + n0 / 2) * 2 + 4);
                cf[0] = c0.x; cf[1] = c0.y; cf[2] = c0.z; cf[3] = c0.w;
                cf[4] = c1.x; cf[5] = c1.y; cf[6] = c1.z; cf[7] = c1.w;
            }
            float xr[R][4];
#pragma unroll
            for (int r = 0; r < R; ++r) SVec<T>::ld4(cur + (r * P + p0) * es, xr[r]);
            // the four columns in two packed fp32 pairs (each lane's arithmetic that of the
            // scalar form, so the same bits)
            float2 yp[R][2];
#pragma unroll
            for (int r = 0; r < R; ++r) yp[r][0] = yp[r][1] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int m = 0; m < kRPT / 2; ++m) {
                float2* h0 = reinterpret_cast<float2*>(&hs[2 * m]);
                float2* h1 = reinterpret_cast<float2*>(&hs[2 * m + 1]);
                float2 br[R], cr[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    br[r] = SVec<T>::ld2(cur + a.xb + (r * N + n0 + 2 * m) * es);
                    cr[r] = SVec<T>::ld2(cur + a.xb + a.nb + (r * N + n0 + 2 * m) * es);
                }
                const float ac = cf[2 * m], as = cf[2 * m + 1];
                const float2 ac2 = make_float2(ac, ac), as2 = make_float2(as, as), nas2 = make_float2(-as, -as);
                const float2 g2 = make_float2(gc.x, gc.x), c2 = make_float2(gc.y, gc.y);
#pragma unroll
                for (int hv = 0; hv < 2; ++hv) {
                    float2 u0 = make_float2(0.0f, 0.0f), u1 = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const float2 xv = make_float2(xr[r][2 * hv], xr[r][2 * hv + 1]);
                        u0 = __ffma2_rn(make_float2(br[r].x, br[r].x), xv, u0);
                        u1 = __ffma2_rn(make_float2(br[r].y, br[r].y), xv, u1);
                    }
                    // alpha Rot(theta) g + gamma u: (a, b) -> (ac a - as b, as a + ac b)
                    const float2 o0 = __ffma2_rn(g2, u0, __ffma2_rn(ac2, h0[hv], __fmul2_rn(nas2, h1[hv])));
                    const float2 o1 = __ffma2_rn(g2, u1, __ffma2_rn(as2, h0[hv], __fmul2_rn(ac2, h1[hv])));
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        yp[r][hv] = __ffma2_rn(make_float2(cr[r].x, cr[r].x), o0,
                                               __ffma2_rn(make_float2(cr[r].y, cr[r].y), o1, yp[r][hv]));
                    // g = h' + c_next u; c_next is 0 after the launch's last token, which
                    // so leaves h' (up to the sign of an exact zero)
                    h0[hv] = __ffma2_rn(c2, u0, o0);
                    h1[hv] = __ffma2_rn(c2, u1, o1);
                }
            }
            // y of token j: lanes P4 apart, then the warps through shared memory
#pragma unroll
            for (int o = P4; o < 32; o <<= 1)
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int hv = 0; hv < 2; ++hv) {
                        yp[r][hv].x += __shfl_xor_sync(0xffffffffu, yp[r][hv].x, o);
                        yp[r][hv].y += __shfl_xor_sync(0xffffffffu, yp[r][hv].y, o);
                    }
            float* rb = red + (j & 1) * nwarps * R * P;
            if (lane < P4) {
#pragma unroll
                for (int r = 0; r < R; ++r)
                    *reinterpret_cast<float4*>(rb + (warp * R + r) * P + p0) =
                        make_float4(yp[r][0].x, yp[r][0].y, yp[r][1].x, yp[r][1].y);
            }
            __syncthreads();
            const int64_t tj = (b * a.k + j) * H + h;
            for (int e = threadIdx.x; e < R * P; e += nthr) {
                float acc = 0.0f;
                for (int w = 0; w < nwarps; ++w) acc += rb[w * R * P + e];
                Vec<T>::st(y + tj * R * P + e, acc);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kRPT; ++i) __stcs(reinterpret_cast<float4*>(st + (int64_t)i * P), hs[i]);
}

}  // namespace m3fast
