// scan_bwd.cuh -- backward pass of the chunked Mamba-3 prefill (m3_scan_bwd)
// on CUDA cores, fp32 arithmetic, with recompute: only the chunk states are
// kept between the passes (the "recompute instead of store" of the Mamba-1
// review page, "hardware-aware algorithm" step 4; the chunked training path of
// "Foundation Model Engineering" ch. 20.2).
//
// Forward, per (b, h) and chunk c (rotated frame, as in scan_chunk.cuh):
//   S'_ij  = S_ij M_ij,  S = C~ B~^T,  M_ij = exp(cs_ti - cs_tj) w_tj (tj < ti), gamma_ti (tj = ti), 0
//   Y      = S' X + diag(exp(cs)) C~ G_{c-1}
//   G_c    = exp(cs_end) G_{c-1} + B~^T diag(s) X,   s_j = exp(cs_end - cs_tj) w_tj
//   final  = Rot(Phi_{T-1}) G_last
// Backward of one chunk, given dY and dG_c (the adjoint of G_c, carried from the
// chunk after it):
//   dS'    = dY X^T;  dS = dS' o M;  dM = dS' o S
//   dX     = S'^T dY + diag(s) B~ dG_c
//   dC~    = dS B~ + diag(exp(cs)) dY G_{c-1}^T
//   dB~    = dS^T C~ + diag(s) X dG_c^T
//   dG_{c-1} = exp(cs_end) dG_c + C~^T diag(exp(cs)) dY
//   the scalar paths: cs through M, exp(cs) and s; w through M and s; gamma
//   through M's diagonal and w; then cs_t = A sum_{k<=t} dt_k, gamma = lambda dt,
//   w_t = gamma_t + (1 - lambda_{t+1}) dt_{t+1} (its next-token part reaches the
//   first token of the chunk after, whose dt / lambda gradients are held back
//   one chunk);
//   the rotation: B~ = Rot(-Phi) B gives dB = Rot(Phi) dB~ and
//   dPhi_t = sum_r (dB~_0 B~_1 - dB~_1 B~_0 + dC~_0 C~_1 - dC~_1 C~_0) per pair,
//   dtheta_t = sum_{t' >= t} dPhi_t' (a suffix sum carried across chunks, started
//   by the final state's rotation).  Pairs whose relative angle is zero -- a token
//   with itself, the last token with the final state -- enter neither dPhi nor the
//   start of the sum: their two contributions cancel exactly, and summed they would
//   leave rounding noise of their own size in gradients that fast decay makes tiny.
//
// Pass 1 (m3_bwd_ckpt_kernel) recomputes the chunk states forward and stores
// G_{c-1} for every chunk and G_last, with the angle at each chunk start, in the
// workspace; pass 2 (m3_bwd_chunk_kernel) walks the chunks in reverse; pass 3
// (m3_bwd_dA_kernel) sums dA over the batch in a fixed order.  One CTA of 256
// threads per (b, h) in passes 1 and 2; every reduction has a fixed order, so
// the gradients are deterministic.
#pragma once

#include "common.cuh"
#include "scan_chunk.cuh"

namespace m3bwd {

using m3cs::Stage;
using m3cs::reduce_2pi_d;
constexpr int kThreads = 256;

// Sizes and shared-memory layouts of passes 1 and 2 (byte offsets).  Row
// strides are odd (N + 1, P + 1, QR + 1 floats) so that threads walking
// consecutive rows hit distinct banks.
struct Geo {
    int Q, R, P, N, K, QR, NS, PS, QS;
    int64_t T;
    int H, nch;
    // pass 2
    int o_x, o_dy, o_bt, o_ct, o_s, o_ds, o_z, o_g, o_dg, o_t2, o_xg, o_cos, o_sin, o_tok, o_row, o_dl, o_red,
        o_pend, o_dp, o_sp, bytes;
    // pass 1
    int c_bt, c_x, c_g, c_cos, c_sin, c_tok, c_dl, c_bytes;
};

// Per-token scalar slots (floats) of pass 2, each [Q]
enum { kCs = 0, kGam, kW, kS, kEcs, kDcs, kDw, kDg, kCsdt, kXs, kTokSlots };
// Per-row slots (floats), each [QR]
enum { kEbar = 0, kDsr, kRowSlots };

inline Geo make_geo(int64_t T, int H, int P, int N, int R, int Q) {
    Geo g;
    g.Q = Q; g.R = R; g.P = P; g.N = N; g.K = N / 2; g.QR = Q * R;
    g.NS = N + 1; g.PS = P + 1; g.QS = g.QR + 1;
    g.T = T; g.H = H;
    g.nch = (int)((T + Q - 1) / Q);
    int o = 0;
    auto take = [&](int floats) { const int at = o; o += 4 * floats; return at; };
    g.o_x = take(g.QR * g.PS);
    g.o_dy = take(g.QR * g.PS);
    g.o_bt = take(g.QR * g.NS);
    g.o_ct = take(g.QR * g.NS);
    g.o_s = take(g.QR * g.QS);
    g.o_ds = take(g.QR * g.QS);
    g.o_z = take(g.QR * g.QS);
    g.o_g = take(N * g.PS);
    g.o_dg = take(N * g.PS);
    g.o_t2 = take(g.QR * g.NS);
    g.o_xg = take(g.QR * g.NS);
    g.o_cos = take(Q * g.K);
    g.o_sin = take(Q * g.K);
    g.o_tok = take(kTokSlots * Q);
    g.o_row = take(kRowSlots * g.QR);
    g.o_dl = take(2 * (Q + 1));
    g.o_red = take(kThreads + 4);
    g.o_pend = take(4 + g.K);   // pending ddt / dlambda of the next chunk's first token, dA; dPhi suffix carry
    g.o_dp = take(g.QR * g.K);  // dPhi share of every row and pair
    g.o_sp = take(g.QR * g.K);  // last chunk: the final state's pair with every row
    g.bytes = (o + 15) & ~15;
    o = 0;
    g.c_bt = take(g.QR * g.NS);
    g.c_x = take(g.QR * g.PS);
    g.c_g = take(N * P);
    g.c_cos = take(Q * g.K);
    g.c_sin = take(Q * g.K);
    g.c_tok = take(2 * Q);
    g.c_dl = take(2 * (Q + 1));
    g.c_bytes = (o + 15) & ~15;
    return g;
}

// Workspace layout: chunk states [units][nch + 1][N][P] fp32, chunk-start
// angles [units][nch + 1][K] fp32 (reduced mod 2 pi), dA partials [units].
struct Work {
    float* G;
    float* phi;
    float* dA;
};
inline size_t work_bytes(int64_t units, const Geo& g) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    return up((size_t)units * (g.nch + 1) * g.N * g.P * 4) + up((size_t)units * (g.nch + 1) * g.K * 4) +
           up((size_t)units * 4);
}
inline Work work_split(void* ws, int64_t units, const Geo& g) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    uint8_t* p = static_cast<uint8_t*>(ws);
    Work w;
    w.G = reinterpret_cast<float*>(p);
    p += up((size_t)units * (g.nch + 1) * g.N * g.P * 4);
    w.phi = reinterpret_cast<float*>(p);
    p += up((size_t)units * (g.nch + 1) * g.K * 4);
    w.dA = reinterpret_cast<float*>(p);
    return w;
}

// Warp 0: chunk-local cs (natural-log units) of the Q tokens from s_dt into cs[];
// past the nt valid tokens cs repeats the last one's value bit for bit (the scan's
// rounding would not), so that exp(cs_end - cs_t) is exactly 1 for the last token.
__device__ __forceinline__ void chunk_cs(const float* s_dt, float A_h, int Q, int nt, float* cs, int lane) {
    const int m = (Q + 31) / 32;
    float run = 0.0f;
    for (int i = 0; i < m; ++i) {
        const int t = lane * m + i;
        if (t < Q) run = fmaf(s_dt[t], A_h, run);
    }
    float incl = run;
    for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    float acc = incl - run;
    for (int i = 0; i < m; ++i) {
        const int t = lane * m + i;
        if (t < Q) {
            acc = fmaf(s_dt[t], A_h, acc);
            cs[t] = acc;
        }
    }
    __syncwarp();
    for (int t = nt + lane; t < Q; t += 32) cs[t] = cs[nt - 1];
    __syncwarp();
}

// ------------------------------------------------------------------ pass 1
template <typename T>
__global__ void __launch_bounds__(kThreads) m3_bwd_ckpt_kernel(const Geo geo, Work wk, const T* __restrict__ x,
                                                               const float* __restrict__ dt,
                                                               const float* __restrict__ A, const T* __restrict__ Bm,
                                                               const float* __restrict__ lam,
                                                               const T* __restrict__ theta) {
    extern __shared__ __align__(16) uint8_t smem[];
    if (blockDim.x != kThreads) {
        if (threadIdx.x == 0) m3::set_status(m3::kStatusBadLaunch);
        return;
    }
    const int tid = threadIdx.x;
    const int Q = geo.Q, R = geo.R, P = geo.P, N = geo.N, K = geo.K, QR = geo.QR, NS = geo.NS, PS = geo.PS;
    const int64_t Tn = geo.T;
    const int H = geo.H;
    const int64_t unit = blockIdx.x, b = unit / H;
    const int h = (int)(unit % H);
    const float A_h = __ldg(A + h);
    float* Bt = reinterpret_cast<float*>(smem + geo.c_bt);
    float* Xs = reinterpret_cast<float*>(smem + geo.c_x);
    float* G = reinterpret_cast<float*>(smem + geo.c_g);
    float* cosv = reinterpret_cast<float*>(smem + geo.c_cos);
    float* sinv = reinterpret_cast<float*>(smem + geo.c_sin);
    float* cs = reinterpret_cast<float*>(smem + geo.c_tok);
    float* sdec = cs + Q;
    float* s_dt = reinterpret_cast<float*>(smem + geo.c_dl);
    float* s_lam = s_dt + (Q + 1);
    auto tok_idx = [&](int64_t t) { return (b * Tn + t) * H + h; };
    float* Gout = wk.G + unit * (int64_t)(geo.nch + 1) * N * P;
    float* Pout = wk.phi + unit * (int64_t)(geo.nch + 1) * K;

    for (int e = tid; e < N * P; e += kThreads) G[e] = 0.0f;
    double carry = 0.0;   // thread 32 + k: the running angle of pair k
    __syncthreads();
    for (int c = 0; c <= geo.nch; ++c) {
        // G_{c-1} and the angle before the chunk's first token
        for (int e = tid; e < N * P; e += kThreads) Gout[(int64_t)c * N * P + e] = G[e];
        if (tid >= 32 && tid < 32 + K) Pout[(int64_t)c * K + tid - 32] = (float)carry;
        if (c == geo.nch) break;
        const int64_t t0 = (int64_t)c * Q;
        const int nt = (int)((Tn - t0) < Q ? (Tn - t0) : Q);
        for (int e = tid; e < QR * P; e += kThreads) {
            const int row = e / P, p = e % P, t = row / R;
            Xs[row * PS + p] = t < nt ? m3::IO<T>::ld(x, tok_idx(t0 + t) * R * P + (e - t * R * P)) : 0.0f;
        }
        for (int e = tid; e < QR * N; e += kThreads) {
            const int row = e / N, n = e % N, t = row / R;
            Bt[row * NS + n] = t < nt ? m3::IO<T>::ld(Bm, tok_idx(t0 + t) * R * N + (e - t * R * N)) : 0.0f;
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
        if (tid < 32) {
            chunk_cs(s_dt, A_h, Q, nt, cs, tid);
            const float cs_end = cs[Q - 1];
            for (int t = tid; t < Q; t += 32) {
                const float w = s_lam[t] * s_dt[t] + (1.0f - s_lam[t + 1]) * s_dt[t + 1];
                sdec[t] = expf(cs_end - cs[t]) * w;
            }
        } else if (theta && tid < 32 + K) {
            const int k = tid - 32;
            for (int t = 0; t < Q; ++t) {
                carry += (double)cosv[t * K + k];
                float sn, cn;
                sincosf((float)reduce_2pi_d(carry), &sn, &cn);
                cosv[t * K + k] = cn;
                sinv[t * K + k] = sn;
            }
            carry = reduce_2pi_d(carry);
        }
        __syncthreads();
        if (theta) {
            for (int e = tid; e < QR * K; e += kThreads) {
                const int row = e / K, k = e % K, t = row / R;
                const float cn = cosv[t * K + k], sn = sinv[t * K + k];
                const float b0 = Bt[row * NS + 2 * k], b1 = Bt[row * NS + 2 * k + 1];
                Bt[row * NS + 2 * k] = fmaf(b0, cn, b1 * sn);
                Bt[row * NS + 2 * k + 1] = fmaf(-b0, sn, b1 * cn);
            }
            __syncthreads();
        }
        const float dec_end = expf(cs[Q - 1]);
        // 4 x 4 tiles of (n, p): each value read from shared memory feeds four products
        for (int tt = tid; tt < ((N + 3) / 4) * (P / 4); tt += kThreads) {
            const int n0 = (tt / (P / 4)) * 4, p0 = (tt % (P / 4)) * 4;
            float acc[4][4] = {};
            for (int j = 0; j < QR; ++j) {
                const float dj = sdec[j / R];
                float bv[4], xv[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) bv[a] = (n0 + a < N) ? dj * Bt[j * NS + n0 + a] : 0.0f;
#pragma unroll
                for (int q = 0; q < 4; ++q) xv[q] = Xs[j * PS + p0 + q];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(bv[a], xv[q], acc[a][q]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                if (n0 + a >= N) break;
#pragma unroll
                for (int q = 0; q < 4; ++q) G[(n0 + a) * P + p0 + q] = fmaf(dec_end, G[(n0 + a) * P + p0 + q], acc[a][q]);
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ pass 2
template <typename T>
__global__ void __launch_bounds__(kThreads) m3_bwd_chunk_kernel(
    const Geo geo, Work wk, const T* __restrict__ x, const float* __restrict__ dt, const float* __restrict__ A,
    const T* __restrict__ Bm, const T* __restrict__ Cm, const float* __restrict__ lam, const T* __restrict__ theta,
    const T* __restrict__ dy, const float* __restrict__ dfinal, T* __restrict__ dx, float* __restrict__ ddt,
    T* __restrict__ dB, T* __restrict__ dC, float* __restrict__ dlam, T* __restrict__ dtheta) {
    extern __shared__ __align__(16) uint8_t smem[];
    if (blockDim.x != kThreads) {
        if (threadIdx.x == 0) m3::set_status(m3::kStatusBadLaunch);
        return;
    }
    const int tid = threadIdx.x;
    const int Q = geo.Q, R = geo.R, P = geo.P, N = geo.N, K = geo.K, QR = geo.QR;
    const int NS = geo.NS, PS = geo.PS, QS = geo.QS;
    const int64_t Tn = geo.T;
    const int H = geo.H, nch = geo.nch;
    const int64_t unit = blockIdx.x, b = unit / H;
    const int h = (int)(unit % H);
    const float A_h = __ldg(A + h);
    float* Xs = reinterpret_cast<float*>(smem + geo.o_x);
    float* dYs = reinterpret_cast<float*>(smem + geo.o_dy);
    float* Bt = reinterpret_cast<float*>(smem + geo.o_bt);
    float* Ct = reinterpret_cast<float*>(smem + geo.o_ct);
    float* Sp = reinterpret_cast<float*>(smem + geo.o_s);     // S' = S o M
    float* dS = reinterpret_cast<float*>(smem + geo.o_ds);    // dS' o M
    float* Zm = reinterpret_cast<float*>(smem + geo.o_z);     // dM = dS' o S
    float* G = reinterpret_cast<float*>(smem + geo.o_g);      // G_{c-1}  [N][PS]
    float* dG = reinterpret_cast<float*>(smem + geo.o_dg);    // adjoint of G_c [N][PS]
    float* T2 = reinterpret_cast<float*>(smem + geo.o_t2);    // dY G^T, then dC~   [QR][NS]
    float* XG = reinterpret_cast<float*>(smem + geo.o_xg);    // X dG^T, then dB~   [QR][NS]
    float* cosv = reinterpret_cast<float*>(smem + geo.o_cos);
    float* sinv = reinterpret_cast<float*>(smem + geo.o_sin);
    float* tok = reinterpret_cast<float*>(smem + geo.o_tok);
    float* rowv = reinterpret_cast<float*>(smem + geo.o_row);
    float* s_dt = reinterpret_cast<float*>(smem + geo.o_dl);
    float* s_lam = s_dt + (Q + 1);
    float* red = reinterpret_cast<float*>(smem + geo.o_red);
    float* pend = reinterpret_cast<float*>(smem + geo.o_pend);   // [0] ddt, [1] dlam of token c0 + Q; [2] dA
    float* dphi_c = pend + 4;                                     // [K] suffix sum of dPhi
    float* dpr = reinterpret_cast<float*>(smem + geo.o_dp);       // [QR][K]
    float* spr = reinterpret_cast<float*>(smem + geo.o_sp);       // [QR][K]
    float* cs = tok + kCs * Q;
    float* gam = tok + kGam * Q;
    float* wv = tok + kW * Q;
    float* sv = tok + kS * Q;
    float* ecs = tok + kEcs * Q;
    float* dcs = tok + kDcs * Q;
    float* dw = tok + kDw * Q;
    float* dgm = tok + kDg * Q;
    float* csdt = tok + kCsdt * Q;
    float* xs = tok + kXs * Q;
    float* ebar = rowv + kEbar * QR;
    float* dsr = rowv + kDsr * QR;
    auto tok_idx = [&](int64_t t) { return (b * Tn + t) * H + h; };
    const float* Gin = wk.G + unit * (int64_t)(nch + 1) * N * P;
    const float* Pin = wk.phi + unit * (int64_t)(nch + 1) * K;

    // dG_last = Rot(-Phi_{T-1}) dfinal.  The final rotation's angle gradient
    // sum_p (-df_0 f_1 + df_1 f_0), f = Rot(Phi_{T-1}) G_last, starts the dtheta suffix
    // sum; it is formed in parts: here the part through G_{nch-1} (f = Rot(Phi_{T-1})
    // G_{nch-1}, decayed by the last chunk's exp(cs_end) once that is known), and in the
    // last chunk the part through each of its rows (minus that row's s-term share of
    // dPhi), without the last token's rows, whose pair with the final state has zero
    // angle and cancels exactly
    for (int e = tid; e < K * P; e += kThreads) {
        const int k = e / P, p = e % P;
        float df0 = 0.0f, df1 = 0.0f;
        if (dfinal) {
            df0 = __ldg(dfinal + unit * N * P + (2 * k) * P + p);
            df1 = __ldg(dfinal + unit * N * P + (2 * k + 1) * P + p);
        }
        float sn = 0.0f, cn = 1.0f;
        if (theta) sincosf(Pin[(int64_t)nch * K + k], &sn, &cn);
        dG[(2 * k) * PS + p] = fmaf(df0, cn, df1 * sn);
        dG[(2 * k + 1) * PS + p] = fmaf(-df0, sn, df1 * cn);
        // f = Rot(Phi) G_{nch-1}, staged in G for the angle term below
        const float* gl = Gin + (int64_t)(nch - 1) * N * P;
        const float g0 = gl[(2 * k) * P + p], g1 = gl[(2 * k + 1) * P + p];
        G[(2 * k) * PS + p] = -df0 * fmaf(g0, sn, g1 * cn) + df1 * fmaf(g0, cn, -g1 * sn);
    }
    if (tid == 0) { pend[0] = 0.0f; pend[1] = 0.0f; pend[2] = 0.0f; }
    __syncthreads();
    for (int k = tid; k < K; k += kThreads) {
        float acc = 0.0f;
        if (theta && dfinal)
            for (int p = 0; p < P; ++p) acc += G[(2 * k) * PS + p];
        dphi_c[k] = acc;
    }
    __syncthreads();

    for (int c = nch - 1; c >= 0; --c) {
        const int64_t t0 = (int64_t)c * Q;
        const int nt = (int)((Tn - t0) < Q ? (Tn - t0) : Q);
        // ---- (1) load the chunk and its checkpoint
        for (int e = tid; e < QR * P; e += kThreads) {
            const int row = e / P, p = e % P, t = row / R;
            const bool ok = t < nt;
            const int64_t gi = tok_idx(t0 + t) * R * P + (e - t * R * P);
            Xs[row * PS + p] = ok ? m3::IO<T>::ld(x, gi) : 0.0f;
            dYs[row * PS + p] = ok ? m3::IO<T>::ld(dy, gi) : 0.0f;
        }
        for (int e = tid; e < QR * N; e += kThreads) {
            const int row = e / N, n = e % N, t = row / R;
            const bool ok = t < nt;
            const int64_t gi = tok_idx(t0 + t) * R * N + (e - t * R * N);
            Bt[row * NS + n] = ok ? m3::IO<T>::ld(Bm, gi) : 0.0f;
            Ct[row * NS + n] = ok ? m3::IO<T>::ld(Cm, gi) : 0.0f;
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
        for (int e = tid; e < N * P; e += kThreads) G[(e / P) * PS + e % P] = Gin[(int64_t)c * N * P + e];
        __syncthreads();
        // ---- (2) scalars (warp 0) and angles (one thread per pair)
        if (tid < 32) {
            chunk_cs(s_dt, A_h, Q, nt, cs, tid);
            const float cs_end = cs[Q - 1];
            for (int t = tid; t < Q; t += 32) {
                gam[t] = s_lam[t] * s_dt[t];
                wv[t] = gam[t] + (1.0f - s_lam[t + 1]) * s_dt[t + 1];
                sv[t] = expf(cs_end - cs[t]) * wv[t];
                ecs[t] = expf(cs[t]);
                dcs[t] = 0.0f;
                dw[t] = 0.0f;
                dgm[t] = 0.0f;
            }
        } else if (theta && tid < 32 + K) {
            const int k = tid - 32;
            double s = (double)Pin[(int64_t)c * K + k];
            for (int t = 0; t < Q; ++t) {
                s += (double)cosv[t * K + k];
                float sn, cn;
                sincosf((float)reduce_2pi_d(s), &sn, &cn);
                cosv[t * K + k] = cn;
                sinv[t * K + k] = sn;
            }
        }
        __syncthreads();
        if (theta) {
            for (int e = tid; e < QR * K; e += kThreads) {
                const int row = e / K, k = e % K, t = row / R;
                const float cn = cosv[t * K + k], sn = sinv[t * K + k];
                const int i0 = row * NS + 2 * k;
                const float b0 = Bt[i0], b1 = Bt[i0 + 1], c0 = Ct[i0], c1 = Ct[i0 + 1];
                Bt[i0] = fmaf(b0, cn, b1 * sn);
                Bt[i0 + 1] = fmaf(-b0, sn, b1 * cn);
                Ct[i0] = fmaf(c0, cn, c1 * sn);
                Ct[i0 + 1] = fmaf(-c0, sn, c1 * cn);
            }
            __syncthreads();
        }
        // ---- (3) S' = S o M, dS = dS' o M, dM = dS' o S;  T2 = dY G^T;  XG = X dG^T
        //      (4 x 4 tiles: each value read from shared memory feeds four products; the
        //      sums keep their order)
        for (int tt = tid; tt < (QR / 4) * (QR / 4); tt += kThreads) {
            const int i0 = (tt / (QR / 4)) * 4, j0 = (tt % (QR / 4)) * 4;
            float sa[4][4] = {}, da[4][4] = {};
            if (j0 / R <= (i0 + 3) / R) {   // some entry on or below the diagonal
                for (int n = 0; n < N; ++n) {
                    float cv[4], bv[4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) { cv[a] = Ct[(i0 + a) * NS + n]; bv[a] = Bt[(j0 + a) * NS + n]; }
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int q = 0; q < 4; ++q) sa[a][q] = fmaf(cv[a], bv[q], sa[a][q]);
                }
                for (int p = 0; p < P; ++p) {
                    float yv[4], xv[4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) { yv[a] = dYs[(i0 + a) * PS + p]; xv[a] = Xs[(j0 + a) * PS + p]; }
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int q = 0; q < 4; ++q) da[a][q] = fmaf(yv[a], xv[q], da[a][q]);
                }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int i = i0 + a, ti = i / R;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j = j0 + q, tj = j / R;
                    float sp = 0.0f, dsv = 0.0f, z = 0.0f;
                    if (tj <= ti) {
                        const float m = (tj == ti) ? gam[ti] : expf(cs[ti] - cs[tj]) * wv[tj];
                        sp = sa[a][q] * m;
                        dsv = da[a][q] * m;
                        z = da[a][q] * sa[a][q];
                    }
                    Sp[i * QS + j] = sp;
                    dS[i * QS + j] = dsv;
                    Zm[i * QS + j] = z;
                }
            }
        }
        for (int tt = tid; tt < (QR / 4) * ((N + 3) / 4); tt += kThreads) {
            const int i0 = (tt / ((N + 3) / 4)) * 4, n0 = (tt % ((N + 3) / 4)) * 4;
            float a2[4][4] = {}, ax[4][4] = {};
            for (int p = 0; p < P; ++p) {
                float yv[4], xv[4], gv[4], dv[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    yv[a] = dYs[(i0 + a) * PS + p];
                    xv[a] = Xs[(i0 + a) * PS + p];
                    gv[a] = (n0 + a < N) ? G[(n0 + a) * PS + p] : 0.0f;
                    dv[a] = (n0 + a < N) ? dG[(n0 + a) * PS + p] : 0.0f;
                }
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        a2[a][q] = fmaf(yv[a], gv[q], a2[a][q]);
                        ax[a][q] = fmaf(xv[a], dv[q], ax[a][q]);
                    }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (n0 + q < N) {
                        T2[(i0 + a) * NS + n0 + q] = a2[a][q];
                        XG[(i0 + a) * NS + n0 + q] = ax[a][q];
                    }
        }
        // <dG_c, G_{c-1}>: the gradient of exp(cs_end) through the state
        {
            float acc = 0.0f;
            for (int e = tid; e < N * P; e += kThreads) acc = fmaf(dG[(e / P) * PS + e % P], G[(e / P) * PS + e % P], acc);
            red[tid] = acc;
        }
        __syncthreads();
        // ---- (4) per-row sums: ebar_i = C~_i . T2_i (exp(cs_i)'s gradient), ds_j = B~_j . XG_j (s_j's);
        //      the dM sums into the token scalars; the <dG, G> total
        for (int i = tid; i < QR; i += kThreads) {
            float a = 0.0f, d = 0.0f;
            for (int n = 0; n < N; ++n) {
                a = fmaf(Ct[i * NS + n], T2[i * NS + n], a);
                d = fmaf(Bt[i * NS + n], XG[i * NS + n], d);
            }
            ebar[i] = a;
            dsr[i] = d;
        }
        if (tid == kThreads - 1) {
            float acc = 0.0f;
            for (int i = 0; i < kThreads; ++i) acc += red[i];
            red[kThreads] = acc;
        }
        __syncthreads();
        // ---- (5) dX, dC~ (into T2), dB~ (into XG) -- each thread reads only the
        //      T2 / XG element it overwrites
        for (int tt = tid; tt < (QR / 4) * (P / 4); tt += kThreads) {
            const int j0 = (tt / (P / 4)) * 4, p0 = (tt % (P / 4)) * 4;
            float acc[4][4] = {}, st[4][4] = {};
            // rows from the first column's token on (S' is zero above each column's token)
            for (int i = (j0 / R) * R; i < QR; ++i) {
                float sv4[4], yv[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) { sv4[a] = Sp[i * QS + j0 + a]; yv[a] = dYs[i * PS + p0 + a]; }
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(sv4[a], yv[q], acc[a][q]);
            }
            for (int n = 0; n < N; ++n) {
                float bv[4], gv[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) { bv[a] = Bt[(j0 + a) * NS + n]; gv[a] = dG[n * PS + p0 + a]; }
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int q = 0; q < 4; ++q) st[a][q] = fmaf(bv[a], gv[q], st[a][q]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int j = j0 + a, tj = j / R;
                if (tj >= nt) continue;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    m3::IO<T>::st(dx, tok_idx(t0 + tj) * R * P + (j - tj * R) * P + p0 + q, fmaf(sv[tj], st[a][q], acc[a][q]));
            }
        }
        // dC~_i = sum_j dS_ij B~_j + exp(cs_i) T2_i and dB~_j = sum_i dS_ij C~_i + s_j XG_j,
        // one thread per row and rotation pair.  The same-token block's share (j, i in
        // the row's own token) is summed apart: its contributions to dPhi through B~ and
        // C~ cancel exactly (C~_i . B~_j is unchanged by a common rotation), so dPhi is
        // formed from the other terms alone, free of that cancellation.  So is the s-term
        // of the last token's rows in the last chunk (its pair with the final state).
        const bool last = (c == nch - 1);
        for (int e = tid; e < QR * K; e += kThreads) {
            const int i = e / K, k = e % K, ti = i / R;
            const int n0 = 2 * k;
            float c_off[2] = {0.0f, 0.0f}, c_dg[2] = {0.0f, 0.0f}, b_off[2] = {0.0f, 0.0f}, b_dg[2] = {0.0f, 0.0f};
            float b_s[2];
            for (int j = 0; j < ti * R; ++j) {
                const float d = dS[i * QS + j];
                c_off[0] = fmaf(d, Bt[j * NS + n0], c_off[0]);
                c_off[1] = fmaf(d, Bt[j * NS + n0 + 1], c_off[1]);
            }
            for (int j = ti * R; j < (ti + 1) * R; ++j) {
                const float d = dS[i * QS + j];
                c_dg[0] = fmaf(d, Bt[j * NS + n0], c_dg[0]);
                c_dg[1] = fmaf(d, Bt[j * NS + n0 + 1], c_dg[1]);
                const float d2 = dS[j * QS + i];
                b_dg[0] = fmaf(d2, Ct[j * NS + n0], b_dg[0]);
                b_dg[1] = fmaf(d2, Ct[j * NS + n0 + 1], b_dg[1]);
            }
            for (int i2 = (ti + 1) * R; i2 < QR; ++i2) {
                const float d = dS[i2 * QS + i];
                b_off[0] = fmaf(d, Ct[i2 * NS + n0], b_off[0]);
                b_off[1] = fmaf(d, Ct[i2 * NS + n0 + 1], b_off[1]);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                c_off[u] = fmaf(ecs[ti], T2[i * NS + n0 + u], c_off[u]);
                b_s[u] = sv[ti] * XG[i * NS + n0 + u];
            }
            if (theta) {
                // this row's share of dPhi_t[k]: d/dPhi Rot(-Phi) v = (v~_1, -v~_0)
                const float sterm = b_s[0] * Bt[i * NS + n0 + 1] - b_s[1] * Bt[i * NS + n0];
                const bool fin = last && ti == nt - 1;
                dpr[i * K + k] = b_off[0] * Bt[i * NS + n0 + 1] - b_off[1] * Bt[i * NS + n0] +
                                 c_off[0] * Ct[i * NS + n0 + 1] - c_off[1] * Ct[i * NS + n0] + (fin ? 0.0f : sterm);
                if (last) spr[i * K + k] = (fin || ti >= nt) ? 0.0f : sterm;
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                T2[i * NS + n0 + u] = c_off[u] + c_dg[u];
                XG[i * NS + n0 + u] = b_off[u] + b_s[u] + b_dg[u];
            }
        }
        // ---- (6) token scalars (warp 0): dcs, dw, dgamma from dM, exp(cs), s and <dG, G>
        if (tid < 32) {
            const float cs_end = cs[Q - 1];
            for (int t = tid; t < Q; t += 32) {
                float a_cs = 0.0f, a_w = 0.0f, a_g = 0.0f;
                for (int r = 0; r < R; ++r) {
                    const int i = t * R + r;
                    // row i (token t) against earlier tokens j: M_ij = exp(cs_t - cs_tj) w_tj
                    for (int j = 0; j < t * R; ++j) {
                        const int tj = j / R;
                        a_cs = fmaf(Zm[i * QS + j], expf(cs[t] - cs[tj]) * wv[tj], a_cs);
                    }
                    // the diagonal block: M = gamma_t
                    for (int j = t * R; j < (t + 1) * R; ++j) a_g += Zm[i * QS + j];
                    // column i (token t) under later rows i2 (token t2): M = exp(cs_t2 - cs_t) w_t
                    for (int i2 = (t + 1) * R; i2 < QR; ++i2) {
                        const float e2 = expf(cs[i2 / R] - cs[t]);
                        a_cs = fmaf(-Zm[i2 * QS + i], e2 * wv[t], a_cs);
                        a_w = fmaf(Zm[i2 * QS + i], e2, a_w);
                    }
                    // exp(cs_t) of the inter-chunk output; s_t = exp(cs_end - cs_t) w_t of the state update
                    a_cs = fmaf(ebar[i], ecs[t], a_cs);
                    a_w = fmaf(dsr[i], expf(cs_end - cs[t]), a_w);
                }
                // s_t = exp(cs_end - cs_t) w_t depends on dt_k for t < k <= end only: its
                // term x_t is added over that range below rather than as + at cs_end and
                // - at cs_t (which would cancel, inexactly, for every k <= t)
                float x = 0.0f;
                for (int r = 0; r < R; ++r) x = fmaf(dsr[t * R + r], sv[t], x);
                xs[t] = x;
                dcs[t] = a_cs;
                dw[t] = a_w;
                dgm[t] = a_g;
            }
            __syncwarp();
            if (tid == 0) {
                dcs[Q - 1] += red[kThreads] * expf(cs_end);   // cs_end through exp(cs_end) G_{c-1}
                // cs_t = A sum_{k <= t} dt_k:  with R_k = sum_{t >= k} dcs_t + sum_{t < k} x_t,
                // ddt_k += A R_k and dA += sum_k dt_k R_k
                float pre = 0.0f;
                for (int t = 0; t < Q; ++t) {
                    csdt[t] = pre;                       // sum_{t' < t} x_t'
                    pre += xs[t];
                }
                float suf = 0.0f, dA_c = 0.0f;
                for (int t = Q - 1; t >= 0; --t) {
                    suf += dcs[t];
                    const float Rk = suf + csdt[t];
                    dA_c = fmaf(s_dt[t], Rk, dA_c);
                    csdt[t] = A_h * Rk;                  // ddt_t through cs
                }
                pend[2] += dA_c;
                // w_t = gamma_t + (1 - lambda_{t+1}) dt_{t+1};  gamma_t = lambda_t dt_t
                float nd = 0.0f, nl = 0.0f;               // w_{Q-1}'s part for token c0 + Q
                for (int t = Q - 1; t >= 0; --t) {
                    const float g_t = dgm[t] + dw[t];
                    float d_dt = csdt[t] + g_t * s_lam[t];
                    float d_l = g_t * s_dt[t];
                    if (t > 0) {
                        // w_{t-1}'s next-token part (1 - lambda_t) dt_t
                        d_dt = fmaf(dw[t - 1], 1.0f - s_lam[t], d_dt);
                        d_l = fmaf(-dw[t - 1], s_dt[t], d_l);
                    }
                    if (t == Q - 1) {
                        nd = dw[t] * (1.0f - s_lam[Q]);
                        nl = -dw[t] * s_dt[Q];
                    }
                    gam[t] = d_dt;      // reused: ddt of token t (without w_{t-1} of the chunk before, for t = 0)
                    wv[t] = d_l;        // reused: dlambda of token t
                }
                // token c0 + Q (the first of the chunk processed before this one) is complete
                if (t0 + Q < Tn) {
                    ddt[tok_idx(t0 + Q)] = pend[0] + nd;
                    if (dlam) dlam[tok_idx(t0 + Q)] = pend[1] + nl;
                }
                // tokens 1 .. nt - 1 are complete; token 0 waits for the chunk before
                for (int t = 1; t < nt; ++t) {
                    ddt[tok_idx(t0 + t)] = gam[t];
                    if (dlam) dlam[tok_idx(t0 + t)] = wv[t];
                }
                pend[0] = gam[0];
                pend[1] = wv[0];
                if (c == 0) {
                    ddt[tok_idx(0)] = gam[0];
                    if (dlam) dlam[tok_idx(0)] = wv[0];
                }
            }
        }
        __syncthreads();
        // ---- (7) rotation: dB, dC rotated back (dPhi was formed in (5));
        //      dtheta = suffix sums (thread per pair)
        if (theta) {
            for (int e = tid; e < QR * K; e += kThreads) {
                const int row = e / K, k = e % K, t = row / R;
                const float cn = cosv[t * K + k], sn = sinv[t * K + k];
                const int i0 = row * NS + 2 * k;
                const float db0 = XG[i0], db1 = XG[i0 + 1], dc0 = T2[i0], dc1 = T2[i0 + 1];
                // dB = Rot(+Phi) dB~, dC likewise
                const float ob0 = fmaf(db0, cn, -db1 * sn), ob1 = fmaf(db0, sn, db1 * cn);
                const float oc0 = fmaf(dc0, cn, -dc1 * sn), oc1 = fmaf(dc0, sn, dc1 * cn);
                XG[i0] = ob0; XG[i0 + 1] = ob1; T2[i0] = oc0; T2[i0 + 1] = oc1;
            }
            __syncthreads();
            for (int k = tid; k < K; k += kThreads) {
                float acc = dphi_c[k];
                if (c == nch - 1) {
                    // the final state's angle term: through G_{nch-1}, decayed over the chunk,
                    // and through the chunk's rows but the last token's
                    acc *= expf(cs[Q - 1]);
                    for (int i = 0; i < QR; ++i) acc -= spr[i * K + k];
                }
                for (int t = Q - 1; t >= 0; --t) {
                    float v = 0.0f;
                    for (int r = 0; r < R; ++r) v += dpr[(t * R + r) * K + k];
                    acc += v;
                    if (t < nt) m3::IO<T>::st(dtheta, tok_idx(t0 + t) * K + k, acc);
                }
                dphi_c[k] = acc;
            }
        }
        // dB, dC of the chunk's valid rows
        for (int e = tid; e < QR * N; e += kThreads) {
            const int row = e / N, n = e % N, t = row / R;
            if (t < nt) {
                const int64_t gi = tok_idx(t0 + t) * R * N + (e - t * R * N);
                m3::IO<T>::st(dB, gi, XG[row * NS + n]);
                m3::IO<T>::st(dC, gi, T2[row * NS + n]);
            }
        }
        // ---- (8) dG_{c-1} = exp(cs_end) dG_c + C~^T diag(exp(cs)) dY  (C~ still rotated)
        {
            const float dec_end = expf(cs[Q - 1]);
            for (int tt = tid; tt < ((N + 3) / 4) * (P / 4); tt += kThreads) {
                const int n0 = (tt / (P / 4)) * 4, p0 = (tt % (P / 4)) * 4;
                float acc[4][4] = {};
                for (int i = 0; i < QR; ++i) {
                    const float ei = ecs[i / R];
                    float cv[4], yv[4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        cv[a] = (n0 + a < N) ? Ct[i * NS + n0 + a] * ei : 0.0f;
                        yv[a] = dYs[i * PS + p0 + a];
                    }
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(cv[a], yv[q], acc[a][q]);
                }
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    if (n0 + a >= N) break;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dG[(n0 + a) * PS + p0 + q] = fmaf(dec_end, dG[(n0 + a) * PS + p0 + q], acc[a][q]);
                }
            }
        }
        __syncthreads();
    }
    if (tid == 0) wk.dA[unit] = pend[2];
}

// ------------------------------------------------------------------ pass 3
// dA[h] = sum_b dA_part[b, h], in batch order.
__global__ void m3_bwd_dA_kernel(const float* __restrict__ part, int64_t batch, int H, float* __restrict__ dA) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H) return;
    float acc = 0.0f;
    for (int64_t b = 0; b < batch; ++b) acc += part[b * H + h];
    dA[h] = acc;
}

}  // namespace m3bwd
