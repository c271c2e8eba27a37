// scan_chunk.cuh -- chunked prefill of the Mamba-3 scan on CUDA cores, fp32
// arithmetic, for every shape and dtype (m3_scan_chunk_kernel).  It executes
// exactly the chunk length Q the caller asks for, so it also serves as the
// check that the chunked algebra does not depend on Q.
//
// Per (batch b, head h), chunk c of Q tokens (Q R rows (t, r)), in the rotated
// ("data-dependent RoPE") frame of the Mamba-3 summary page, Propositions
// 3.2.2 / 3.2.3, with the SSD intra-chunk / inter-chunk split of "Foundation
// Model Engineering" ch. 20.2:
//   cs_t   = sum_{i = c0}^{t} dt_i A            (chunk-local log decay)
//   Phi_t  = sum_{i <= t} theta_i               (cumulative angle, per pair)
//   B~, C~ = Rot(-Phi_t) B_t, Rot(-Phi_t) C_t
//   w_t    = gamma_t + (1 - lambda_{t+1}) dt_{t+1}    (eq. (7)'s two bands, folded)
//   S'_ij  = (C~_i . B~_j) * { exp(cs_ti - cs_tj) w_tj  if tj < ti;  gamma_ti if tj = ti;  0 }
//   y_i    = sum_j S'_ij x_j + exp(cs_ti) C~_i^T G_{c-1}
//   G_c    = exp(cs_end) G_{c-1} + sum_j exp(cs_end - cs_tj) w_tj B~_j x_j^T
// G is the augmented chunk state h_end + (1 - lambda_next) dt_next v~_end, which
// carries the trapezoid's cross-chunk beta term; final_state = Rot(Phi_{T-1}) G.
//
// One CTA of 256 threads per (b, h) sequence; every chunk goes through shared
// memory in five phases separated by barriers: load, scalars + angles, rotate,
// y (row blocks of S'), state update.  Inputs are staged in their own dtype
// (bf16 stays bf16, so a 256-row MIMO chunk fits); the rotated B~, C~ are
// rounded to that dtype once.  Every sum is fp32.  The running angle is kept
// per pair in fp64 and reduced mod 2 pi there (a few fp64 operations per token
// and pair, off the fp32 paths), so its error does not grow with the sequence.
#pragma once

#include "common.cuh"

namespace m3cs {

constexpr int kThreads = 256;
constexpr double kTwoPiD = 6.283185307179586476925286766559;

// Sizes of one launch and the shared-memory layout (byte offsets).
struct Geo {
    int Q, R, P, N, K, QR, RB, NS;   // NS: row stride of B~ / C~ (N + 1, odd)
    int64_t T;
    int H;
    int nch;
    int off_carry, off_bt, off_ct, off_x, off_sp, off_g, off_cos, off_sin, off_sc, off_dl, bytes;
};

// elem: bytes per staged element (4 for fp32 inputs, 2 for bf16).
inline Geo make_geo(int64_t T, int H, int P, int N, int R, int Q, int elem) {
    Geo g;
    g.Q = Q; g.R = R; g.P = P; g.N = N; g.K = N / 2; g.QR = Q * R;
    g.RB = g.QR < 64 ? g.QR : 64;
    g.NS = N + 1;
    g.T = T; g.H = H;
    g.nch = (int)((T + Q - 1) / Q);
    auto up = [](int x, int a) { return (x + a - 1) / a * a; };
    int o = 0;
    g.off_carry = o; o += 8 * g.K;
    g.off_bt = o;    o = up(o + elem * g.QR * g.NS, 16);
    g.off_ct = o;    o = up(o + elem * g.QR * g.NS, 16);
    g.off_x = o;     o = up(o + elem * g.QR * P, 16);
    g.off_sp = o;    o += 4 * g.RB * g.QR;
    g.off_g = o;     o += 4 * N * P;
    g.off_cos = o;   o += 4 * Q * g.K;
    g.off_sin = o;   o += 4 * Q * g.K;
    g.off_sc = o;    o += 4 * 5 * Q;            // cs | gamma | w | dec | exp(cs)
    g.off_dl = o;    o += 4 * 2 * (Q + 1);      // dt | lambda of the Q tokens and the one after
    g.bytes = up(o, 16);
    return g;
}

template <typename T>
struct Stage;
template <>
struct Stage<float> {
    static __device__ __forceinline__ float get(const float* p, int i) { return p[i]; }
    static __device__ __forceinline__ void put(float* p, int i, float v) { p[i] = v; }
};
template <>
struct Stage<__nv_bfloat16> {
    static __device__ __forceinline__ float get(const __nv_bfloat16* p, int i) { return __bfloat162float(p[i]); }
    static __device__ __forceinline__ void put(__nv_bfloat16* p, int i, float v) { p[i] = __float2bfloat16_rn(v); }
};

// x - n 2 pi, n = rint(x / 2 pi), in fp64.
__device__ __forceinline__ double reduce_2pi_d(double x) { return fma(-rint(x * (1.0 / kTwoPiD)), kTwoPiD, x); }

template <typename T>
__global__ void __launch_bounds__(kThreads) m3_scan_chunk_kernel(
    const Geo geo, const T* __restrict__ x, const float* __restrict__ dt, const float* __restrict__ A,
    const T* __restrict__ Bm, const T* __restrict__ Cm, const float* __restrict__ lam, const T* __restrict__ theta,
    T* __restrict__ y, float* __restrict__ final_state, const float* __restrict__ h0, const T* __restrict__ prev_B,
    const T* __restrict__ prev_x) {
    extern __shared__ __align__(16) uint8_t smem[];
    if (blockDim.x != kThreads) {
        if (threadIdx.x == 0) m3::set_status(m3::kStatusBadLaunch);
        return;
    }
    const int tid = threadIdx.x;
    const int Q = geo.Q, R = geo.R, P = geo.P, N = geo.N, K = geo.K, QR = geo.QR, NS = geo.NS;
    const int64_t Tn = geo.T;
    const int H = geo.H;
    const int64_t unit = blockIdx.x;
    const int64_t b = unit / H;
    const int h = (int)(unit % H);
    const float A_h = __ldg(A + h);

    double* carry = reinterpret_cast<double*>(smem + geo.off_carry);   // [K] running angle
    T* Bt = reinterpret_cast<T*>(smem + geo.off_bt);                    // [QR][NS]
    T* Ct = reinterpret_cast<T*>(smem + geo.off_ct);                    // [QR][NS]
    T* Xs = reinterpret_cast<T*>(smem + geo.off_x);                     // [QR][P]
    float* Sp = reinterpret_cast<float*>(smem + geo.off_sp);            // [RB][QR]
    float* G = reinterpret_cast<float*>(smem + geo.off_g);              // [N][P]
    float* cosv = reinterpret_cast<float*>(smem + geo.off_cos);         // [Q][K] (theta on load)
    float* sinv = reinterpret_cast<float*>(smem + geo.off_sin);         // [Q][K]
    float* sc_cs = reinterpret_cast<float*>(smem + geo.off_sc);
    float* sc_gam = sc_cs + Q;
    float* sc_w = sc_gam + Q;
    float* sc_dec = sc_w + Q;
    float* sc_ecs = sc_dec + Q;
    float* s_dt = reinterpret_cast<float*>(smem + geo.off_dl);          // [Q + 1]
    float* s_lam = s_dt + (Q + 1);                                      // [Q + 1]

    // token base offsets of this (b, h) in the [b, T, h] and [b, T, h, *] layouts
    auto tok_idx = [&](int64_t t) { return (b * Tn + t) * H + h; };

    // G_{-1}: zero, or the continuation's h0 + (1 - lambda_0) dt_0 sum_r prev_B[r] prev_x[r]^T
    {
        float bcoef = 0.0f;
        if (prev_B && Tn > 0) {
            const float d0 = __ldg(dt + tok_idx(0));
            const float l0 = lam ? __ldg(lam + tok_idx(0)) : 1.0f;
            bcoef = (1.0f - l0) * d0;
        }
        for (int e = tid; e < N * P; e += kThreads) {
            const int n = e / P, p = e % P;
            float v = h0 ? __ldg(h0 + unit * N * P + e) : 0.0f;
            if (prev_B) {
                float u = 0.0f;
                for (int r = 0; r < R; ++r)
                    u = fmaf(m3::IO<T>::ld(prev_B, (unit * R + r) * N + n), m3::IO<T>::ld(prev_x, (unit * R + r) * P + p), u);
                v = fmaf(bcoef, u, v);
            }
            G[e] = v;
        }
        for (int k = tid; k < K; k += kThreads) carry[k] = 0.0;
    }

    for (int c = 0; c < geo.nch; ++c) {
        const int64_t t0 = (int64_t)c * Q;
        const int nt = (int)((Tn - t0) < Q ? (Tn - t0) : Q);   // valid tokens of this chunk
        // ---- (1) load the chunk (zero past the end of the sequence)
        for (int e = tid; e < QR * P; e += kThreads) {
            const int row = e / P, t = row / R, rp = e - t * R * P;
            const float v = t < nt ? m3::IO<T>::ld(x, tok_idx(t0 + t) * R * P + rp) : 0.0f;
            Stage<T>::put(Xs, e, v);
        }
        for (int e = tid; e < QR * N; e += kThreads) {
            const int row = e / N, n = e % N, t = row / R, rn = e - t * R * N;
            const bool ok = t < nt;
            Stage<T>::put(Bt, row * NS + n, ok ? m3::IO<T>::ld(Bm, tok_idx(t0 + t) * R * N + rn) : 0.0f);
            Stage<T>::put(Ct, row * NS + n, ok ? m3::IO<T>::ld(Cm, tok_idx(t0 + t) * R * N + rn) : 0.0f);
        }
        for (int e = tid; e < Q * K; e += kThreads) {
            const int t = e / K, k = e % K;
            cosv[e] = (theta && t < nt) ? m3::IO<T>::ld(theta, tok_idx(t0 + t) * K + k) : 0.0f;
        }
        for (int t = tid; t <= Q; t += kThreads) {
            const bool ok = t0 + t < Tn;
            s_dt[t] = ok ? __ldg(dt + tok_idx(t0 + t)) : 0.0f;
            s_lam[t] = (ok && lam) ? __ldg(lam + tok_idx(t0 + t)) : 1.0f;
        }
        __syncthreads();

        // ---- (2a) warp 0: chunk scalars.  Lane l takes tokens [l m, l m + m).
        if (tid < 32) {
            const int lane = tid, m = (Q + 31) / 32;
            float run = 0.0f;
            for (int i = 0; i < m; ++i) {
                const int t = lane * m + i;
                if (t < Q) run = fmaf(s_dt[t], A_h, run);
            }
            float incl = run;   // inclusive scan of the lane totals
            for (int o = 1; o < 32; o <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            float acc = incl - run;   // exclusive prefix
            for (int i = 0; i < m; ++i) {
                const int t = lane * m + i;
                if (t < Q) {
                    acc = fmaf(s_dt[t], A_h, acc);
                    sc_cs[t] = acc;
                }
            }
            __syncwarp();
            // past the end (dt = 0) cs stays at the last token's value -- bit for bit, so
            // that exp(cs_end - cs) is exactly 1 there, as the scan's rounding would not
            // guarantee
            for (int t = nt + lane; t < Q; t += 32) sc_cs[t] = sc_cs[nt - 1];
            __syncwarp();
            const float cs_end = sc_cs[Q - 1];
            for (int t = lane; t < Q; t += 32) {
                const float gam = s_lam[t] * s_dt[t];
                const float w = gam + (1.0f - s_lam[t + 1]) * s_dt[t + 1];
                sc_gam[t] = gam;
                sc_w[t] = w;
                sc_dec[t] = expf(cs_end - sc_cs[t]) * w;
                sc_ecs[t] = expf(sc_cs[t]);
            }
        } else if (theta && tid < 32 + K) {
            // ---- (2b) one thread per rotation pair: the running angle in fp64,
            //      its sine and cosine per token (theta = 0 past the end)
            const int k = tid - 32;
            double s = carry[k];
            for (int t = 0; t < Q; ++t) {
                s += (double)cosv[t * K + k];
                const float a = (float)reduce_2pi_d(s);
                float sn, cn;
                sincosf(a, &sn, &cn);
                cosv[t * K + k] = cn;
                sinv[t * K + k] = sn;
            }
            carry[k] = reduce_2pi_d(s);
        }
        __syncthreads();

        // ---- (3) rotate B and C by -Phi_t: (a, b) -> (a cos + b sin, -a sin + b cos)
        if (theta) {
            for (int e = tid; e < QR * K; e += kThreads) {
                const int row = e / K, k = e % K, t = row / R;
                const float cn = cosv[t * K + k], sn = sinv[t * K + k];
                const int i0 = row * NS + 2 * k;
                const float b0 = Stage<T>::get(Bt, i0), b1 = Stage<T>::get(Bt, i0 + 1);
                const float c0 = Stage<T>::get(Ct, i0), c1 = Stage<T>::get(Ct, i0 + 1);
                Stage<T>::put(Bt, i0, fmaf(b0, cn, b1 * sn));
                Stage<T>::put(Bt, i0 + 1, fmaf(-b0, sn, b1 * cn));
                Stage<T>::put(Ct, i0, fmaf(c0, cn, c1 * sn));
                Stage<T>::put(Ct, i0 + 1, fmaf(-c0, sn, c1 * cn));
            }
            __syncthreads();
        }

        // ---- (4) y, one block of RB rows at a time.  Every thread computes 4 x 4 tiles
        //      (four rows by four columns), so that each value read from shared memory
        //      feeds four multiply-adds.
        for (int rb0 = 0; rb0 < QR; rb0 += geo.RB) {
            const int rows = (QR - rb0) < geo.RB ? (QR - rb0) : geo.RB;   // a multiple of 16
            const int jmax = ((rb0 + rows - 1) / R + 1) * R;   // columns up to the block's last token
            const int jt = (jmax + 3) / 4;                      // 4-column tiles (<= QR / 4)
            // (4a) S' = (C~ B~^T) o M for rows [rb0, rb0 + rows), columns [0, 4 jt)
            for (int tt = tid; tt < (rows / 4) * jt; tt += kThreads) {
                const int il0 = (tt / jt) * 4, j0 = (tt % jt) * 4;
                const int i0 = rb0 + il0;
                float acc[4][4];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[a][q] = 0.0f;
                if (j0 / R <= (i0 + 3) / R) {   // some entry on or below the diagonal
                    for (int n = 0; n < N; ++n) {
                        float cv[4], bv[4];
#pragma unroll
                        for (int a = 0; a < 4; ++a) cv[a] = Stage<T>::get(Ct, (i0 + a) * NS + n);
#pragma unroll
                        for (int q = 0; q < 4; ++q) bv[q] = Stage<T>::get(Bt, (j0 + q) * NS + n);
#pragma unroll
                        for (int a = 0; a < 4; ++a)
#pragma unroll
                            for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(cv[a], bv[q], acc[a][q]);
                    }
                }
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const int ti = (i0 + a) / R;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int j = j0 + q, tj = j / R;
                        float v = 0.0f;
                        if (tj <= ti) {
                            const float mk = (tj == ti) ? sc_gam[ti] : expf(sc_cs[ti] - sc_cs[tj]) * sc_w[tj];
                            v = acc[a][q] * mk;
                        }
                        Sp[(il0 + a) * QR + j] = v;
                    }
                }
            }
            __syncthreads();
            // (4b) y = S' X + diag(exp cs) C~ G_{c-1} for the block's rows, 4 x 4 tiles of (row, p)
            const int pt = P / 4;
            for (int tt = tid; tt < (rows / 4) * pt; tt += kThreads) {
                const int il0 = (tt / pt) * 4, p0 = (tt % pt) * 4;
                const int i0 = rb0 + il0;
                const int jn = ((i0 + 3) / R + 1) * R;   // columns up to the last row's token
                float acc[4][4], inter[4][4];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int q = 0; q < 4; ++q) { acc[a][q] = 0.0f; inter[a][q] = 0.0f; }
                for (int j = 0; j < jn; ++j) {
                    float sv[4], xv[4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) sv[a] = Sp[(il0 + a) * QR + j];   // zero past each row's token
#pragma unroll
                    for (int q = 0; q < 4; ++q) xv[q] = Stage<T>::get(Xs, j * P + p0 + q);
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(sv[a], xv[q], acc[a][q]);
                }
                for (int n = 0; n < N; ++n) {
                    float cv[4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) cv[a] = Stage<T>::get(Ct, (i0 + a) * NS + n);
                    const float4 g4 = *reinterpret_cast<const float4*>(G + n * P + p0);
                    const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int q = 0; q < 4; ++q) inter[a][q] = fmaf(cv[a], gv[q], inter[a][q]);
                }
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const int i = i0 + a, ti = i / R;
                    if (ti >= nt) continue;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        m3::IO<T>::st(y, tok_idx(t0 + ti) * R * P + (i - ti * R) * P + p0 + q,
                                      fmaf(sc_ecs[ti], inter[a][q], acc[a][q]));
                }
            }
            __syncthreads();
        }

        // ---- (5) G_c = exp(cs_end) G_{c-1} + sum_j dec_tj B~_j x_j^T, 4 x 4 tiles of (n, p)
        {
            const float dec_end = expf(sc_cs[Q - 1]);
            const int nt4 = (N + 3) / 4, pt = P / 4;
            for (int tt = tid; tt < nt4 * pt; tt += kThreads) {
                const int n0 = (tt / pt) * 4, p0 = (tt % pt) * 4;
                float acc[4][4];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[a][q] = 0.0f;
                for (int j = 0; j < QR; ++j) {
                    const float dj = sc_dec[j / R];
                    float bv[4], xv[4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) bv[a] = (n0 + a < N) ? dj * Stage<T>::get(Bt, j * NS + n0 + a) : 0.0f;
#pragma unroll
                    for (int q = 0; q < 4; ++q) xv[q] = Stage<T>::get(Xs, j * P + p0 + q);
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(bv[a], xv[q], acc[a][q]);
                }
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    if (n0 + a >= N) break;
                    float4* gp = reinterpret_cast<float4*>(G + (n0 + a) * P + p0);
                    const float4 g = *gp;
                    *gp = make_float4(fmaf(dec_end, g.x, acc[a][0]), fmaf(dec_end, g.y, acc[a][1]),
                                      fmaf(dec_end, g.z, acc[a][2]), fmaf(dec_end, g.w, acc[a][3]));
                }
            }
        }
        __syncthreads();
    }

    // ---- final state in the complex frame: Rot(+Phi_{T-1}) G
    if (final_state) {
        float* fs = final_state + unit * N * P;
        for (int e = tid; e < K * P; e += kThreads) {
            const int k = e / P, p = e % P;
            float sn = 0.0f, cn = 1.0f;
            if (theta) sincosf((float)carry[k], &sn, &cn);
            const float a = G[(2 * k) * P + p], bb = G[(2 * k + 1) * P + p];
            fs[(2 * k) * P + p] = fmaf(a, cn, -bb * sn);
            fs[(2 * k + 1) * P + p] = fmaf(a, sn, bb * cn);
        }
    }
}

}  // namespace m3cs
