// step_simt.cuh -- fp32 SIMT kernels of libm3scan:
//   * m3_step_kernel: one decode step for every (b, h), state streamed from HBM
//     with 128-bit loads/stores (memory bound: ~2 x 16 KB of state per head).
//   * m3_scan_seq_kernel: the prefill evaluated one token at a time with the
//     state held in registers (the exact recurrence, no chunking).  It serves
//     fp32 inputs (whose 1e-4 tolerance rules out bf16 tensor cores) and every
//     shape the tensor-core kernel does not cover.
//
// Both evaluate the complex-frame update of the Mamba-3 summary page (§3.1
// eq. (5)-(6) with the rotation blocks of §3.2, Proposition 3.2.1, and the
// rank-R input of §3.3):
//   h' <- Rot(theta_t)(alpha h' + beta u_{t-1}) + gamma u_t,  y_t[r] = C_t[r]^T h'
// Thread geometry: thread (tk, q) owns the 4 columns p = 4q..4q+3 of the
// row pairs (2k, 2k+1), k = tk + i*TK for i < NPT, of one head's N x P state.
#pragma once

#include "common.cuh"

namespace m3 {

// Per-token inputs staged in shared memory as fp32, in this order.
struct TokLayout {
    int x, B, C, cs, sn, dt, lam, size;
    __host__ __device__ TokLayout(int R, int P, int N) {
        const int K = N / 2;
        x = 0;
        B = x + R * P;
        C = B + R * N;
        cs = C + R * N;
        sn = cs + K;
        dt = sn + K;
        lam = dt + 1;
        size = ((lam + 1 + 3) / 4) * 4;
    }
};

struct SimtArgs {
    int R, P, N, K, P4, TK;
};

// Source of flat element e of one token's input block.
template <typename T>
struct TokSource {
    const T* x;       // R*P elements of this token
    const T* B;       // R*N
    const T* C;       // R*N
    const T* theta;   // K, or nullptr
    const float* dt;  // 1
    const float* lam; // 1, or nullptr

    __device__ __forceinline__ float load(int e, const SimtArgs& a) const {
        const int RP = a.R * a.P, RN = a.R * a.N;
        if (e < RP) return IO<T>::ld(x, e);
        e -= RP;
        if (e < RN) return IO<T>::ld(B, e);
        e -= RN;
        if (e < RN) return IO<T>::ld(C, e);
        e -= RN;
        if (e < a.K) return theta ? IO<T>::ld(theta, e) : 0.0f;
        e -= a.K;
        if (e == 0) return __ldg(dt);
        return lam ? __ldg(lam) : 1.0f;
    }
    // Where flat element e goes in the shared token block (theta -> cs/sn
    // handled by the caller).
    static __device__ __forceinline__ int slot(int e, const SimtArgs& a, const TokLayout& L) {
        const int RP = a.R * a.P, RN = a.R * a.N;
        if (e < RP + 2 * RN) return e;  // x, B, C are contiguous in both
        e -= RP + 2 * RN;
        if (e < a.K) return -1 - e;     // theta element k -> (cs[k], sn[k])
        return e == a.K ? L.dt : L.lam;
    }
};

__device__ __forceinline__ void store_tok(float* tok, const TokLayout& L, const SimtArgs& a, int e,
                                          float v, int slot) {
    if (slot >= 0) {
        tok[slot] = v;
    } else {
        const int k = -1 - slot;
        float s, c;
        sincosf(v, &s, &c);
        tok[L.cs + k] = c;
        tok[L.sn + k] = s;
    }
}

// The recurrence step for this thread's pairs.  `cur` holds token t,
// `prv` holds token t-1 (its B and x only are read).  Adds this thread's
// rows' share of y_t into yp[r][j] (p = 4q + j).
template <int NPT>
__device__ __forceinline__ void step_pairs(float (&h)[NPT][2][4], float (&yp)[8][4], const float* cur,
                                           const float* prv, const TokLayout& L, const SimtArgs& a,
                                           float A_h, int q, int tk) {
    const float d = cur[L.dt];
    const float l = cur[L.lam];
    const float alpha = expf(d * A_h);
    const float beta = (1.0f - l) * d * alpha;
    const float gamma = l * d;
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j) yp[r][j] = 0.0f;
#pragma unroll
    for (int i = 0; i < NPT; ++i) {
        const int k = tk + i * a.TK;
        const float c = cur[L.cs + k], s = cur[L.sn + k];
        float u0[4] = {0, 0, 0, 0}, u1[4] = {0, 0, 0, 0}, v0[4] = {0, 0, 0, 0}, v1[4] = {0, 0, 0, 0};
        for (int r = 0; r < a.R; ++r) {
            const float b0 = cur[L.B + r * a.N + 2 * k], b1 = cur[L.B + r * a.N + 2 * k + 1];
            const float4 xv = *reinterpret_cast<const float4*>(cur + L.x + r * a.P + 4 * q);
            const float pb0 = prv[L.B + r * a.N + 2 * k], pb1 = prv[L.B + r * a.N + 2 * k + 1];
            const float4 pxv = *reinterpret_cast<const float4*>(prv + L.x + r * a.P + 4 * q);
            const float xs[4] = {xv.x, xv.y, xv.z, xv.w};
            const float pxs[4] = {pxv.x, pxv.y, pxv.z, pxv.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                u0[j] += b0 * xs[j];
                u1[j] += b1 * xs[j];
                v0[j] += pb0 * pxs[j];
                v1[j] += pb1 * pxs[j];
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float z0 = alpha * h[i][0][j] + beta * v0[j];
            const float z1 = alpha * h[i][1][j] + beta * v1[j];
            h[i][0][j] = c * z0 - s * z1 + gamma * u0[j];
            h[i][1][j] = s * z0 + c * z1 + gamma * u1[j];
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            if (r < a.R) {
                const float c0 = cur[L.C + r * a.N + 2 * k], c1 = cur[L.C + r * a.N + 2 * k + 1];
#pragma unroll
                for (int j = 0; j < 4; ++j) yp[r][j] += c0 * h[i][0][j] + c1 * h[i][1][j];
            }
        }
    }
}

// Write this thread's y partials to red[tk][r][p].
__device__ __forceinline__ void put_partials(float* red, const float (&yp)[8][4], const SimtArgs& a,
                                             int q, int tk) {
    for (int r = 0; r < a.R; ++r)
        *reinterpret_cast<float4*>(red + (tk * a.R + r) * a.P + 4 * q) =
            make_float4(yp[r][0], yp[r][1], yp[r][2], yp[r][3]);
}

// y[e] = sum_tk red[tk][e], e < R*P, fixed order (deterministic).
template <typename T>
__device__ __forceinline__ void reduce_y(const float* red, const SimtArgs& a, T* y_out) {
    const int RP = a.R * a.P;
    for (int e = threadIdx.x; e < RP; e += blockDim.x) {
        float acc = 0.0f;
        for (int t = 0; t < a.TK; ++t) acc += red[t * RP + e];
        IO<T>::st(y_out, e, acc);
    }
}

// ---------------------------------------------------------------------------
// Decode step: grid = b*h blocks, blockDim = TK * P4.
// Shared memory: cur token block, prev block, red[TK][R][P].
template <typename T, int NPT>
__global__ void __launch_bounds__(512) m3_step_kernel(SimtArgs a, int64_t H, float* __restrict__ state,
                                                      const T* __restrict__ x_t, const float* __restrict__ dt_t,
                                                      const float* __restrict__ A,
                                                      const T* __restrict__ B_t, const T* __restrict__ C_t,
                                                      const float* __restrict__ lam_t,
                                                      const T* __restrict__ theta_t,
                                                      const T* __restrict__ prev_B,
                                                      const T* __restrict__ prev_x, T* __restrict__ y_t) {
    extern __shared__ __align__(16) float smem[];
    const TokLayout L(a.R, a.P, a.N);
    float* cur = smem;
    float* prv = smem + L.size;
    float* red = prv + L.size;
    if (blockDim.x != a.TK * a.P4) {
        if (threadIdx.x == 0) set_status(kStatusBadLaunch);
        return;
    }
    const int64_t unit = blockIdx.x;  // b * H + h
    const int h_idx = (int)(unit % H);
    const int q = threadIdx.x % a.P4, tk = threadIdx.x / a.P4;
    const int64_t NP = (int64_t)a.N * a.P;
    float* st = state + unit * NP;

    // 1. state loads first (the bulk of the bytes): rows 2k, 2k+1, columns 4q..4q+3
    float h[NPT][2][4];
#pragma unroll
    for (int i = 0; i < NPT; ++i) {
        const int k = tk + i * a.TK;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const float4 v = __ldcs(reinterpret_cast<const float4*>(st + (2 * k + rr) * (int64_t)a.P + 4 * q));
            h[i][rr][0] = v.x; h[i][rr][1] = v.y; h[i][rr][2] = v.z; h[i][rr][3] = v.w;
        }
    }
    // 2. this token's inputs and the previous token's B, x into shared memory
    TokSource<T> src;
    src.x = x_t + unit * a.R * a.P;
    src.B = B_t + unit * a.R * a.N;
    src.C = C_t + unit * a.R * a.N;
    src.theta = theta_t ? theta_t + unit * a.K : nullptr;
    src.dt = dt_t + unit;
    src.lam = lam_t ? lam_t + unit : nullptr;
    const int E = a.R * a.P + 2 * a.R * a.N + a.K + 2;
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        store_tok(cur, L, a, e, src.load(e, a), TokSource<T>::slot(e, a, L));
    for (int e = threadIdx.x; e < a.R * a.P; e += blockDim.x)
        prv[L.x + e] = prev_x ? IO<T>::ld(prev_x + unit * a.R * a.P, e) : 0.0f;
    for (int e = threadIdx.x; e < a.R * a.N; e += blockDim.x)
        prv[L.B + e] = prev_B ? IO<T>::ld(prev_B + unit * a.R * a.N, e) : 0.0f;
    __syncthreads();

    // 3. update and write back the state (streaming stores), y partials
    float yp[8][4];
    step_pairs<NPT>(h, yp, cur, prv, L, a, __ldg(A + h_idx), q, tk);
#pragma unroll
    for (int i = 0; i < NPT; ++i) {
        const int k = tk + i * a.TK;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
            __stcs(reinterpret_cast<float4*>(st + (2 * k + rr) * (int64_t)a.P + 4 * q),
                   make_float4(h[i][rr][0], h[i][rr][1], h[i][rr][2], h[i][rr][3]));
    }
    put_partials(red, yp, a, q, tk);
    __syncthreads();
    reduce_y<T>(red, a, y_t + unit * a.R * a.P);
}

// ---------------------------------------------------------------------------
// Sequential prefill: grid = b*h blocks; the state stays in registers for the
// whole sequence.  Shared memory: 3 rotating token blocks (t-1, t, t+1) and
// 2 rotating partial buffers.  One __syncthreads per token.
constexpr int kSeqPrefetch = 8;  // input elements each thread prefetches into registers

template <typename T, int NPT>
__global__ void __launch_bounds__(512) m3_scan_seq_kernel(SimtArgs a, int64_t T_len, int64_t H,
                                                          const T* __restrict__ x, const float* __restrict__ dt,
                                                          const float* __restrict__ A,
                                                          const T* __restrict__ Bm, const T* __restrict__ Cm,
                                                          const float* __restrict__ lam,
                                                          const T* __restrict__ theta, T* __restrict__ y,
                                                          float* __restrict__ final_state,
                                                          const float* __restrict__ h0,
                                                          const T* __restrict__ prev_B,
                                                          const T* __restrict__ prev_x) {
    extern __shared__ __align__(16) float smem[];
    const TokLayout L(a.R, a.P, a.N);
    float* tok[3] = {smem, smem + L.size, smem + 2 * L.size};
    float* red[2] = {smem + 3 * L.size, smem + 3 * L.size + a.TK * a.R * a.P};
    if (blockDim.x != a.TK * a.P4) {
        if (threadIdx.x == 0) set_status(kStatusBadLaunch);
        return;
    }
    const int64_t unit = blockIdx.x;
    const int64_t b = unit / H, hh = unit % H;
    const int q = threadIdx.x % a.P4, tk = threadIdx.x / a.P4;
    const float A_h = __ldg(A + hh);
    const int E = a.R * a.P + 2 * a.R * a.N + a.K + 2;

    auto source = [&](int64_t t) {
        const int64_t bth = (b * T_len + t) * H + hh;
        TokSource<T> s;
        s.x = x + bth * a.R * a.P;
        s.B = Bm + bth * a.R * a.N;
        s.C = Cm + bth * a.R * a.N;
        s.theta = theta ? theta + bth * a.K : nullptr;
        s.dt = dt + bth;
        s.lam = lam ? lam + bth : nullptr;
        return s;
    };

    // token -1: the previous token's x and B of a continuation (zero for a fresh
    // sequence); token 0 loaded synchronously
    for (int e = threadIdx.x; e < L.size; e += blockDim.x) tok[2][e] = 0.0f;
    __syncthreads();
    if (prev_B) {
        for (int e = threadIdx.x; e < a.R * a.P; e += blockDim.x)
            tok[2][L.x + e] = IO<T>::ld(prev_x + unit * a.R * a.P, e);
        for (int e = threadIdx.x; e < a.R * a.N; e += blockDim.x)
            tok[2][L.B + e] = IO<T>::ld(prev_B + unit * a.R * a.N, e);
    }
    if (T_len > 0) {
        const TokSource<T> s0 = source(0);
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            store_tok(tok[0], L, a, e, s0.load(e, a), TokSource<T>::slot(e, a, L));
    }
    __syncthreads();

    float h[NPT][2][4];
#pragma unroll
    for (int i = 0; i < NPT; ++i)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int k = tk + i * a.TK;
            float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (h0) v = __ldg(reinterpret_cast<const float4*>(h0 + (unit * a.N + 2 * k + rr) * (int64_t)a.P + 4 * q));
            h[i][rr][0] = v.x; h[i][rr][1] = v.y; h[i][rr][2] = v.z; h[i][rr][3] = v.w;
        }

    for (int64_t t = 0; t < T_len; ++t) {
        float* cur = tok[t % 3];
        float* prv = tok[(t + 2) % 3];
        float* nxt = tok[(t + 1) % 3];
        const bool has_next = (t + 1 < T_len);
        // (a) prefetch token t+1 into registers
        float pre[kSeqPrefetch];
        TokSource<T> sn;
        if (has_next) {
            sn = source(t + 1);
#pragma unroll
            for (int i = 0; i < kSeqPrefetch; ++i) {
                const int e = threadIdx.x + i * blockDim.x;
                pre[i] = (e < E) ? sn.load(e, a) : 0.0f;
            }
        }
        // (b) the step for token t
        float yp[8][4];
        step_pairs<NPT>(h, yp, cur, prv, L, a, A_h, q, tk);
        float* rb = red[t & 1];
        put_partials(rb, yp, a, q, tk);
        // (c) stage token t+1
        if (has_next) {
#pragma unroll
            for (int i = 0; i < kSeqPrefetch; ++i) {
                const int e = threadIdx.x + i * blockDim.x;
                if (e < E) store_tok(nxt, L, a, e, pre[i], TokSource<T>::slot(e, a, L));
            }
            for (int e = threadIdx.x + kSeqPrefetch * blockDim.x; e < E; e += blockDim.x)
                store_tok(nxt, L, a, e, sn.load(e, a), TokSource<T>::slot(e, a, L));
        }
        __syncthreads();
        // (d) y_t
        reduce_y<T>(rb, a, y + ((b * T_len + t) * H + hh) * a.R * a.P);
    }

    if (final_state) {
        float* fs = final_state + unit * (int64_t)a.N * a.P;
#pragma unroll
        for (int i = 0; i < NPT; ++i) {
            const int k = tk + i * a.TK;
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
                *reinterpret_cast<float4*>(fs + (2 * k + rr) * (int64_t)a.P + 4 * q) =
                    make_float4(h[i][rr][0], h[i][rr][1], h[i][rr][2], h[i][rr][3]);
        }
    }
}

}  // namespace m3
