// scan_ws.cuh -- chunked tensor-core prefill of the Mamba-3 scan (bf16 inputs,
// fp32 state), warp-specialised so that consecutive chunks overlap.
//
// The math is the chunked evaluation in the rotated ("data-dependent RoPE")
// frame (Mamba-3 summary page, "Mamba-3: Expressive SSM with MIMO", §3.1-§3.3,
// Propositions 3.2.2 / 3.2.3; SSD intra/inter-chunk split of "Foundation Model
// Engineering" ch. 20.2).  Per (batch b, head h), chunk c of Q tokens (Q*R = 64
// tile rows), chunk-local log decay cs_t = sum_{i=c0}^{t} dt_i A, cumulative
// angle Phi_t = sum_{i<=t} theta_i, B~ = Rot(-Phi) B, C~ = Rot(-Phi) C:
//
//   S       = C~ B~^T                                       (tcgen05 -> TMEM)
//   S'      = S o M,  M_ij = exp(cs_i - cs_j) w_j (j < i), gamma_i (j = i), 0 (j > i)
//             w_j = gamma_j + (1 - lambda_{j+1}) dt_{j+1}   (eq. (7)'s decay x two-band, folded)
//   Y_intra = S' X                                          (tcgen05 -> TMEM)
//   Y_inter = C~ G_{c-1}                                    (tcgen05 -> TMEM)
//   y       = Y_intra + diag(exp(cs)) Y_inter               (epilogue)
//   dG      = (diag(exp(cs_end - cs) w) B~)^T X             (tcgen05 -> TMEM)
//   G_c     = exp(cs_end) G_{c-1} + dG                      (fp32 registers)
//
// G_c = h_end + (1 - lambda_next) dt_next v~_end is the augmented chunk state: it
// carries the trapezoid's cross-chunk beta term.  final_state = Rot(Phi_{T-1}) G.
//
// The factorised mask: inside a 16-row block J with reference token r (its last
// token), for rows i whose token lies after the block,
//   exp(cs_i - cs_j) w_j = exp(cs_i - cs_r) * [exp(cs_r - cs_j) w_j],
// both factors <= 1 (cs decreases along the chunk), so the products cannot
// overflow; only the diagonal block needs one exp per element.
//
// Roles (256 threads, one CTA per (b, h), two CTAs per SM when N = 64):
//   warpgroup 0 (threads 0-127), chunk c+1: scalars (warp 0, from dt / lambda it
//     copied into shared memory one chunk ahead), cumulative angles, rotation of
//     B and C in shared memory (with the fused B / C normalisation first, in the
//     NORM variants), the scaled copy B~'.  Lane 0 of warp 1 issues Phi and
//     Y_inter, lane 0 of warp 2 issues S and dG.
//   warpgroup 1 (threads 128-255), chunk c: mask S -> S', G update, y epilogue;
//     thread 128 issues the TMA store of y, lane 0 of warp 5 issues Y_intra and
//     lane 0 of warp 6 every TMA load: two stages, each filled in two parts when
//     the rotation is on (theta + B as soon as S has read them, C + x after
//     Y_intra), in one part otherwise.
// Every mbarrier wait is bounded; a wait that runs out sets the device status
// word, the decision to stop is voted at the next named barrier (uniform in the
// warpgroup), and the CTA waits (bounded) for its copies and MMAs in flight and
// frees its TMEM before it returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "m3scan.h"
#include "ptx_sm100.cuh"

namespace m3ws {

constexpr int kWG = 128;
constexpr int kThreads = 2 * kWG;
constexpr int kRows = 64;                       // tile rows per chunk = Q * R
constexpr int kP = 64;                          // headdim
constexpr long long kWaitBudget = 4000000000LL; // clock cycles (~2 s) before a wait gives up
constexpr float kTwoPi = 6.283185307179586f;
constexpr uint32_t kBarWG0 = 1, kBarWG1 = 2;
// Warpgroup 0's MMA issuers, one lane in each of two warps other than warp 0
// (which computes the chunk scalars), so that no warp carries two serial jobs.
constexpr int kEarlyIssuer = 32;   // Phi(c), Y_inter(c-1)
constexpr int kLateIssuer = 64;    // S(c), dG(c)
// Warpgroup 1's serial jobs, likewise one lane in each of three warps.
constexpr int kYIssuer = 2 * 64 + 32;   // (warp 5) Y_intra(c)
constexpr int kLoader = 2 * 64 + 64;    // (warp 6) the TMA loads of every chunk
// Largest decay span (log2 units) across one 16-row mask block for which the
// diagonal block is evaluated in factorised form; beyond it, exactly.
constexpr float kSpanMax = 96.0f;
// High word of every 128-byte-swizzled operand descriptor here (SBO = 1024).
constexpr uint32_t kDescHi = ptx::sdesc_hi(1024, ptx::kSwz128);

__host__ __device__ constexpr int align1k(int x) { return (x + 1023) & ~1023; }
__host__ __device__ constexpr int align16(int x) { return (x + 15) & ~15; }

template <int NSLAB, int R, bool ROT, bool NORM = false>
struct Cfg {
    static constexpr int Q = kRows / R;          // tokens per chunk
    static constexpr int N = 64 * NSLAB;         // state size
    static constexpr int K = N / 2;              // rotation pairs
    static constexpr int KG = N / 8;             // 16-byte groups per row (4 pairs each)
    static constexpr int TB = 16 / R;            // tokens per 16-row mask block
    static constexpr int TILE = kRows * 128;     // one 64-column slab of a 64-row bf16 tile
    // stage (TMA destination): x | B slabs | C slabs | theta
    static constexpr int ST_X = 0;
    static constexpr int ST_B = ST_X + TILE;
    static constexpr int ST_C = ST_B + NSLAB * TILE;
    static constexpr int ST_TH = ST_C + NSLAB * TILE;
    static constexpr int TH_BYTES = ROT ? Q * K * 2 : 0;
    static constexpr int ST_BYTES = align1k(ST_TH + TH_BYTES);
    // With the rotation, a stage fills in two parts: theta and B, which the
    // prologue needs first and which are free again once S has been computed,
    // then C and x, free once Y_inter and Y_intra have been computed.  Without
    // it, the prologue needs all tiles at once and part a carries them all.
    static constexpr uint32_t TX_A = ROT ? TILE * NSLAB + TH_BYTES : TILE * (1 + 2 * NSLAB);
    static constexpr uint32_t TX_B = TILE * (1 + NSLAB);
    static constexpr int OFF_BD = 2 * ST_BYTES;               // B~' (2 stages)
    static constexpr int OFF_SP = OFF_BD + 2 * NSLAB * TILE;  // S' (K-major)
    static constexpr int OFF_G = OFF_SP + TILE;               // G bf16 [N][P] (MN-major)
    static constexpr int OFF_Y = OFF_G + N * 128;             // y staging (TMA store source)
    static constexpr int OFF_L = OFF_Y + TILE;                // L: [64 rows][64 tokens] 0/1, K-major
    // per-chunk scalars in three buffers (chunk c in buffer c % 3): warp 0 writes chunk
    // c's while warpgroup 1 may still read chunk c - 1's and c - 2's (a warpgroup-0
    // warp that starts chunk c knows only that chunk c - 3's output has been stored)
    static constexpr int OFF_SC = OFF_L + TILE;
    static constexpr int SC_CS = 0, SC_W = Q, SC_GAM = 2 * Q, SC_SCB = 3 * Q, SC_SCF = 4 * Q, SC_SDF = 5 * Q,
                         SC_DEC = 6 * Q;
    static constexpr int SC_STRIDE = 6 * Q + 4;               // floats per buffer
    static constexpr int OFF_CARRY = align16(OFF_SC + 3 * SC_STRIDE * 4);  // float [2][K]: angle carry
    // dt and lambda of a chunk's Q tokens and the token after it, per stage: float [2][2][DL]
    static constexpr int DL = (Q + 1 + 3) & ~3;
    static constexpr int OFF_DL = OFF_CARRY + 2 * K * 4;
    // with the B / C normalisation: its scales and this head's biases, float [4][N]
    static constexpr int OFF_NRM = OFF_DL + 2 * 2 * DL * 4;
    static constexpr int SMEM_BYTES = OFF_NRM + (NORM ? 4 * N * 4 : 0) + 1024;  // + alignment slack
    // theta tile [Q][K] as the MN-major B operand of Phi = L theta: 64-byte
    // swizzle for K = 32 pairs, 128-byte swizzle for K = 64
    static constexpr uint32_t TH_SBO = (K == 32) ? 512 : 1024;
    static constexpr uint32_t TH_K16 = 2 * TH_SBO;            // bytes per 16 tokens
    // TMEM columns: S / Y_intra double-buffered, dG, Y_inter
    static constexpr uint32_t TM_SY0 = 0, TM_DG = 128, TM_YI = 192, TM_COLS = 256;
    static_assert(Q <= 64, "scalar lanes hold two tokens each");
    static_assert(K == 32 || K == 64, "theta tile width");
    static_assert(TB * R == 16, "mask blocks");
};

struct Params {
    int64_t T;
    int H;
    int nchunks;
    const float* dt;
    const float* A;
    const float* lam;    // may be null (lambda = 1)
    float* final_state;  // may be null
    // continuation (all may be null): the state before the first token (complex
    // frame, fp32 [b, h, N, P]) and the token before it (bf16 [b, h, R, N] / [b, h, R, P])
    const float* h0;
    const __nv_bfloat16* prev_B;
    const __nv_bfloat16* prev_x;
    // B / C normalisation (all null without it): scales [N], biases [h, N], epsilon
    const float* norm_wB;
    const float* norm_wC;
    const float* norm_bB;
    const float* norm_bC;
    float norm_eps;
    // chunk checkpoints for the backward pass (CKPT variants only): the fp32 state
    // G_{c-1} at the start of every chunk c and G_last, [b h][nch + 1][N][P], and
    // the angle carry (reduced mod 2 pi) at the same points, [b h][nch + 1][K]
    float* ck_G;
    float* ck_phi;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}
// n consecutive floats from shared memory (n = 8, 4: 16-byte aligned; n = 2: 8-byte aligned).
template <int n>
__device__ __forceinline__ void load_tok(const float* p, float (&out)[n]) {
    if constexpr (n == 2) {
        const float2 a = *reinterpret_cast<const float2*>(p);
        out[0] = a.x; out[1] = a.y;
    } else {
#pragma unroll
        for (int q = 0; q < n; q += 4) {
            const float4 a = *reinterpret_cast<const float4*>(p + q);
            out[q] = a.x; out[q + 1] = a.y; out[q + 2] = a.z; out[q + 3] = a.w;
        }
    }
}

// The two bf16 of a packed word as floats (bf16 is the top half of an fp32).
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// x - n 2 pi with n = rint(x / 2 pi), in [-pi, pi]: Cody and Waite's
// two-constant reduction (2 pi = kC1 + kC2 with kC1 = 201/32 exact in 8 bits,
// so n kC1 is exact for |n| < 2^16 and the error is about |n| ulp(kC2)).
constexpr float kC1 = 6.28125f;
constexpr float kC2 = 1.9353071795864769e-3f;
__device__ __forceinline__ float reduce_2pi(float x) {
    const float n = rintf(x * (1.0f / kTwoPi));
    return fmaf(-n, kC2, fmaf(-n, kC1, x));
}
// sin / cos of x: the reduction above, then the hardware sin / cos (absolute
// error ~1e-6 on [-pi, pi]).
__device__ __forceinline__ void sincos_reduced(float x, float* s, float* c) {
    __sincosf(reduce_2pi(x), s, c);
}
// 1 / sqrt(ss / n + eps) of a row's sum of squares ss over n channels, kept
// finite for an all-zero row (the zero-filled rows past the end of a sequence)
// when eps is 0: such a row then normalises to 0 instead of 0 * inf = NaN.
__device__ __forceinline__ float rms_inv(float ss, float inv_n, float eps) {
    return rsqrtf(fmaxf(fmaf(ss, inv_n, eps), 1.17549435e-38f));
}

// 1 / RMS of a 64- or 128-element bf16 row held as two half rows in lanes l and
// l ^ 16 (GPT 16-byte groups each): the squares summed in packed fp32 pairs on two
// accumulators, so the dependent chain is GPT * 2 deep instead of GPT * 8.
template <int GPT>
__device__ __forceinline__ float row_rms_inv(const uint4 (&v)[GPT], float inv_n, float eps) {
    float2 s0 = make_float2(0.0f, 0.0f), s1 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int g = 0; g < GPT; ++g) {
        const uint32_t pv[4] = {v[g].x, v[g].y, v[g].z, v[g].w};
        float2 e0 = make_float2(bf_lo(pv[0]), bf_hi(pv[0])), e1 = make_float2(bf_lo(pv[1]), bf_hi(pv[1]));
        float2 e2 = make_float2(bf_lo(pv[2]), bf_hi(pv[2])), e3 = make_float2(bf_lo(pv[3]), bf_hi(pv[3]));
        s0 = __ffma2_rn(e0, e0, s0);
        s1 = __ffma2_rn(e1, e1, s1);
        s0 = __ffma2_rn(e2, e2, s0);
        s1 = __ffma2_rn(e3, e3, s1);
    }
    float ss = (s0.x + s1.x) + (s0.y + s1.y);
    ss += __shfl_xor_sync(0xffffffffu, ss, 16);
    return rms_inv(ss, inv_n, eps);
}
// Byte offset of the 16-byte group g of row `row` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int row, int g) {
    return (uint32_t)(row * 128 + (((g & 7) ^ (row & 7)) << 4) + (g >> 3) * (kRows * 128));
}

template <int NSLAB, int R, bool ROT, bool NORM, bool CKPT = false>
__global__ void __launch_bounds__(kThreads, (NSLAB == 1 ? 2 : 1))
    m3_scan_ws_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_B,
                      const __grid_constant__ CUtensorMap map_C, const __grid_constant__ CUtensorMap map_th,
                      const __grid_constant__ CUtensorMap map_y, const Params prm) {
    using CF = Cfg<NSLAB, R, ROT, NORM>;
    // CKPT: the backward pass's checkpoint run, which needs the chunk states and
    // angles only: C is not loaded, and S, the mask, Y_intra, Y_inter and the
    // output are skipped; map_y then describes the fp32 checkpoints
    // [b h (nch + 1)][N][P] (box 32 x 64 x 1, 128-byte swizzle), which leave
    // through a shared-memory tile by TMA stores
    static_assert(!(CKPT && NORM), "no checkpoint run with the fused normalisation");
    constexpr int Q = CF::Q, N = CF::N, K = CF::K, TILE = CF::TILE;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t bar_lda[2], bar_ldb[2], bar_sd[2], bar_syfree[2], bar_dgfree, bar_yi, bar_y, bar_phi, bar_fin[3];
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;

    if (blockDim.x != kThreads) {
        if (threadIdx.x == 0) m3::set_status(m3::kStatusBadLaunch);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x;
    const int h = unit % prm.H;
    const int b = unit / prm.H;
    const int64_t T = prm.T;
    const int nch = prm.nchunks;
    const float A_l2 = __ldg(prm.A + h) * m3::kLog2e;

    float* scal0 = reinterpret_cast<float*>(smem + CF::OFF_SC);
    float* s_carry = reinterpret_cast<float*>(smem + CF::OFF_CARRY);
    uint8_t* t_sp = smem + CF::OFF_SP;
    uint8_t* t_g = smem + CF::OFF_G;
    uint8_t* t_y = smem + CF::OFF_Y;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&bar_lda[s], 1);
            ptx::mbar_init(&bar_ldb[s], 1);
            ptx::mbar_init(&bar_sd[s], 1);
            ptx::mbar_init(&bar_syfree[s], 1);
        }
        for (int k = 0; k < 3; ++k) ptx::mbar_init(&bar_fin[k], 1);
        ptx::mbar_init(&bar_dgfree, 1);
        ptx::mbar_init(&bar_yi, 1);
        ptx::mbar_init(&bar_y, 1);
        ptx::mbar_init(&bar_phi, 1);
        ptx::fence_mbar_init();
        abort_s = 0;
    }
    if (warp == 0) {
        ptx::tmem_alloc(&tmem_base_s, CF::TM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid < 2 * K) s_carry[tid] = 0.0f;
    if constexpr (NORM) {
        // the scales and this head's biases: with the rotation per pair of channels
        // (n, n + 1), (w[n], w[n + 1], b[n], b[n + 1]) at 2 n for B and at 2 N + 2 n
        // for C; without it B and C interleaved per channel, (wB[n], wC[n]) at 2 n
        // and (bB[n], bC[n]) at 2 N + 2 n
        float* nrm = reinterpret_cast<float*>(smem + CF::OFF_NRM);
        for (int i = tid; i < N; i += kThreads) {
            const float v[4] = {__ldg(prm.norm_wB + i), __ldg(prm.norm_wC + i), __ldg(prm.norm_bB + (int64_t)h * N + i),
                                __ldg(prm.norm_bC + (int64_t)h * N + i)};
            if (ROT) {
                const int o = 2 * (i & ~1) + (i & 1);
                nrm[o] = v[0];
                nrm[o + 2] = v[2];
                nrm[2 * N + o] = v[1];
                nrm[2 * N + o + 2] = v[3];
            } else {
                nrm[2 * i] = v[0];
                nrm[2 * i + 1] = v[1];
                nrm[2 * N + 2 * i] = v[2];
                nrm[2 * N + 2 * i + 1] = v[3];
            }
        }
    }
    // fp32 chunk state G, rows owned by the consumer threads (M = 64 accumulator
    // layout for N = 64: row 16 w + lane % 16, columns 32 (lane / 16) + [0, 32);
    // M = 128 layout for N = 128: row 32 w + lane, all 64 columns)
    constexpr int GC = (N == 64) ? 32 : 64;
    float G[GC];
#pragma unroll
    for (int p = 0; p < GC; ++p) G[p] = 0.0f;
    // A continuation starts from the augmented state G_{-1} = h_{-1} + (1 - lambda_0)
    // dt_0 prev_B^T prev_x (the RoPE frame of this call starts at angle 0, so the
    // complex-frame state is also the rotated-frame state); warpgroup 1 holds it in
    // its fp32 registers and puts the bf16 copy Y_inter(0) reads in shared memory.
    const bool has_init = (prm.h0 != nullptr) || (prm.prev_B != nullptr);
    if (has_init && tid >= kWG && tid < 2 * kWG) {
        const int w1 = warp - 4;
        const int g_row = (N == 64) ? (w1 * 16 + (lane & 15)) : (w1 * 32 + lane);
        const int col0 = (N == 64) ? (lane >> 4) * 32 : 0;
        const int64_t i0 = ((int64_t)b * T) * prm.H + h;             // token 0 of this (b, h)
        const float d0 = T > 0 ? __ldg(prm.dt + i0) : 0.0f;
        const float l0 = (T > 0 && prm.lam) ? __ldg(prm.lam + i0) : 1.0f;
        const float bcoef = (1.0f - l0) * d0;
        const int64_t uh = (int64_t)b * prm.H + h;
#pragma unroll
        for (int p = 0; p < GC; ++p) {
            float v = prm.h0 ? __ldg(prm.h0 + (uh * N + g_row) * kP + col0 + p) : 0.0f;
            if (prm.prev_B) {
                float u = 0.0f;
                for (int r = 0; r < R; ++r)
                    u = fmaf(__bfloat162float(prm.prev_B[(uh * R + r) * N + g_row]),
                             __bfloat162float(prm.prev_x[(uh * R + r) * kP + col0 + p]), u);
                v = fmaf(bcoef, u, v);
            }
            G[p] = v;
        }
#pragma unroll
        for (int g = 0; g < GC / 8; ++g)
            *reinterpret_cast<uint4*>(t_g + swz(g_row, col0 / 8 + g)) =
                make_uint4(pack_bf16(G[g * 8 + 0], G[g * 8 + 1]), pack_bf16(G[g * 8 + 2], G[g * 8 + 3]),
                           pack_bf16(G[g * 8 + 4], G[g * 8 + 5]), pack_bf16(G[g * 8 + 6], G[g * 8 + 7]));
    }
    // L[i][t] = 1 for t <= token(i) = i / R (and t < Q), else 0: 64 x 64 bf16, 128-byte swizzle
    for (int e = tid; e < kRows * 8; e += kThreads) {
        const int i = e >> 3, g = e & 7;
        uint32_t wv[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int t0 = g * 8 + 2 * m;
            const uint32_t lo = (t0 <= i / R && t0 < Q) ? 0x3F80u : 0u;        // bf16 1.0
            const uint32_t hi = (t0 + 1 <= i / R && t0 + 1 < Q) ? 0x3F80u : 0u;
            wv[m] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(smem + CF::OFF_L + swz(i, g)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    // TMA loads of chunk c into stage c % 2 (issued by thread kLoader only):
    // part a (theta and B; every tile without the rotation) and part b (C and x)
    auto issue_loads_a = [&](int c) {
        const int s = c & 1;
        uint8_t* st = smem + s * CF::ST_BYTES;
        const int t0 = c * Q;
        // (the checkpoint run reads no C)
        ptx::mbar_arrive_expect_tx(&bar_lda[s], CF::TX_A - ((CKPT && !ROT) ? NSLAB * TILE : 0u));
        if (ROT) ptx::tma_load_4d(st + CF::ST_TH, &map_th, &bar_lda[s], 0, h, t0, b);
#pragma unroll
        for (int sl = 0; sl < NSLAB; ++sl) {
            ptx::tma_load_5d(st + CF::ST_B + sl * TILE, &map_B, &bar_lda[s], sl * 64, 0, h, t0, b);
            if (!ROT && !CKPT) ptx::tma_load_5d(st + CF::ST_C + sl * TILE, &map_C, &bar_lda[s], sl * 64, 0, h, t0, b);
        }
        if (!ROT) ptx::tma_load_5d(st + CF::ST_X, &map_x, &bar_lda[s], 0, 0, h, t0, b);
    };
    auto issue_loads_b = [&](int c) {
        if (!ROT) return;
        const int s = c & 1;
        uint8_t* st = smem + s * CF::ST_BYTES;
        const int t0 = c * Q;
        ptx::mbar_arrive_expect_tx(&bar_ldb[s], CF::TX_B - (CKPT ? NSLAB * TILE : 0u));
        if (!CKPT) {
#pragma unroll
            for (int sl = 0; sl < NSLAB; ++sl)
                ptx::tma_load_5d(st + CF::ST_C + sl * TILE, &map_C, &bar_ldb[s], sl * 64, 0, h, t0, b);
        }
        ptx::tma_load_5d(st + CF::ST_X, &map_x, &bar_ldb[s], 0, 0, h, t0, b);
    };
    int last_a = -1, last_b = -1;   // thread kLoader only: the last chunk of each part loaded
    bool aborted = false;

    if (tid < kWG) {
        // ======================= warpgroup 0: prologue + S / dG issue =======================
        // Lane 0 of warp 1 turns the chunk's theta tile into the cumulative angles
        // of every tile row with one MMA, Phi_rows = L theta (L[i][t] = 1 for
        // t <= token(i)), into the S/Y TMEM buffer of the stage.  Thread
        // (warp w, lane l) then owns tile row 16 w + l % 16 and the rotation
        // pairs [PH (l / 16), PH (l / 16) + PH): it reads those angles with the
        // 16x32bx2 TMEM shape, rotates its half of the B and C rows in shared
        // memory (bank-conflict free under the 128-byte swizzle) and writes its
        // half of the scaled copy B~'.  Warp 0 computes the chunk scalars (lane l
        // holds tokens l and l + 32) into the chunk's scalar buffer.
        constexpr int PH = K / 2;               // pairs per thread
        constexpr int GPT = PH / 4;             // 16-byte groups per thread
        const int row = warp * 16 + (lane & 15);
        const int hf = lane >> 4;
        const int tok = row / R;
        float* carry_buf = reinterpret_cast<float*>(smem + CF::OFF_CARRY);   // [2][K]
        // warp 0 only: dt / lambda of chunk c's tokens and of the token after it
        // (zero past the end), copied into shared memory one chunk ahead
        float* s_dl = reinterpret_cast<float*>(smem + CF::OFF_DL);   // [stage][dt | lambda][DL]
        auto prefetch_scalars = [&](int c) {
            float* dst = s_dl + (c & 1) * 2 * CF::DL;
            for (int tt = lane; tt <= Q; tt += 32) {
                const int64_t t = (int64_t)c * Q + tt;
                const bool ok = t < T;
                const int64_t idx = ok ? ((int64_t)b * T + t) * prm.H + h : 0;
                ptx::cp_async4(dst + tt, prm.dt + idx, ok);
                if (prm.lam) ptx::cp_async4(dst + CF::DL + tt, prm.lam + idx, ok);
            }
            ptx::cp_async_commit();
        };
        if (warp == 0) prefetch_scalars(0);
        // thread kEarlyIssuer only: the MMAs of step (0) for chunk c (c = nch: the last Y_inter)
        auto issue_early = [&](int c) {
            const int s = c & 1;
            bool ok = true;
            if (c >= 2) ok = ptx::mbar_wait(&bar_syfree[s], ((c >> 1) - 1) & 1, kWaitBudget);
            if (ok && ROT && c < nch) ok = ptx::mbar_wait(&bar_lda[s], (c >> 1) & 1, kWaitBudget);
            if (!ok) {
                m3::set_status(m3::kStatusWaitTimeout);
                abort_s = 1;
                return;
            }
            ptx::tc_fence_after();
            if (ROT && c < nch) {
                const uint32_t l_lo = ptx::sdesc_lo(ptx::smem_u32(smem + CF::OFF_L), 16);
                const uint32_t th_lo = ptx::sdesc_lo(ptx::smem_u32(smem + s * CF::ST_BYTES + CF::ST_TH), K * 2);
                constexpr uint32_t id_phi = ptx::idesc_bf16(kRows, K, false, true);
                constexpr uint32_t th_hi = ptx::sdesc_hi(CF::TH_SBO, K == 32 ? ptx::kSwz64 : ptx::kSwz128);
#pragma unroll
                for (int k16 = 0; k16 < Q / 16; ++k16)
                    ptx::umma_bf16_lo<kDescHi, th_hi>(tmem + CF::TM_SY0 + 64u * s, l_lo + k16 * 2,
                                                       th_lo + k16 * (CF::TH_K16 >> 4), id_phi, k16 > 0);
                ptx::umma_commit(&bar_phi);
            }
            if (!CKPT && (c >= 2 || (c == 1 && (prm.h0 != nullptr || prm.prev_B != nullptr)))) {
                // Y_inter(c-1) = C~_{c-1} G_{c-2} (G: bf16 [N][P] rows, MN-major; G_{-1}
                // is the continuation's initial state)
                const uint32_t c_lo =
                    ptx::sdesc_lo(ptx::smem_u32(smem + ((c - 1) & 1) * CF::ST_BYTES + CF::ST_C), 16);
                const uint32_t g_lo = ptx::sdesc_lo(ptx::smem_u32(t_g), N * 128);
                constexpr uint32_t id_y = ptx::idesc_bf16(kRows, kP, false, true);
#pragma unroll
                for (int k16 = 0; k16 < N / 16; ++k16) {
                    const uint32_t ko = ((k16 >> 2) * TILE + (k16 & 3) * 32) >> 4;
                    ptx::umma_bf16_lo<kDescHi, kDescHi>(tmem + CF::TM_YI, c_lo + ko, g_lo + k16 * 128, id_y, k16 > 0);
                }
                ptx::umma_commit(&bar_yi);
            }
        };

        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            uint8_t* st = smem + s * CF::ST_BYTES;
            float* sc = scal0 + (c % 3) * CF::SC_STRIDE;
            const uint32_t tm_sy = tmem + CF::TM_SY0 + 64u * s;
            // (0) thread kEarlyIssuer, once chunk c-2's output has been read (its S/Y buffer and
            //     Y_inter free): Phi_rows = L theta -> TMEM S/Y[s] when chunk c's tiles
            //     are in, and Y_inter(c-1) = C~_{c-1} G_{c-2} -> TMEM Y_inter, which
            //     warpgroup 1 needs halfway through chunk c-1
            if (tid == kEarlyIssuer) issue_early(c);
            // the issuing lane's warp reconverges before its other lanes wait: a lane
            // parked in mbarrier.try_wait can hold back a diverged lane of its warp
            __syncwarp();

            // (1) warp 0: chunk scalars for tokens lane (u = 0) and 32 + lane (u = 1):
            //     cs (log2 units), gamma, w, B~' row scale, mask column weights
            if (warp == 0) {
                ptx::cp_async_wait_all();   // this chunk's dt / lambda (copied during chunk c-1)
                __syncwarp();
                if (c + 1 < nch) prefetch_scalars(c + 1);
                const float* sdt = s_dl + s * 2 * CF::DL;
                const float* slm = sdt + CF::DL;
                float d_cur[2], l_cur[2], dnext[2], lnext[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    // token t = 32 u + lane and the one after it (t + 1 <= Q wherever used)
                    const int t = u * 32 + lane;
                    const bool in = t < Q;
                    d_cur[u] = in ? sdt[t] : 0.0f;
                    dnext[u] = in ? sdt[t + 1] : 0.0f;
                    l_cur[u] = (in && prm.lam) ? slm[t] : 1.0f;
                    lnext[u] = (in && prm.lam) ? slm[t + 1] : 1.0f;
                }
                float cs[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    float a = d_cur[u] * A_l2;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float v = __shfl_up_sync(0xffffffffu, a, o);
                        if (lane >= o) a += v;
                    }
                    cs[u] = a;
                }
                cs[1] += __shfl_sync(0xffffffffu, cs[0], 31);
                const float cs_end = (Q == 64) ? __shfl_sync(0xffffffffu, cs[1], 31) : __shfl_sync(0xffffffffu, cs[0], Q - 1);
                const int ref = (lane / CF::TB) * CF::TB + CF::TB - 1;   // last token of the mask block
                const int first = (lane / CF::TB) * CF::TB;                // its first token
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float cs_ref = __shfl_sync(0xffffffffu, cs[u], ref);
                    const float cs_first = __shfl_sync(0xffffffffu, cs[u], first);
                    const float gam = l_cur[u] * d_cur[u];
                    const float w = gam + (1.0f - lnext[u]) * dnext[u];
                    const int t = u * 32 + lane;
                    if (t < Q) {
                        sc[CF::SC_CS + t] = cs[u];
                        sc[CF::SC_GAM + t] = gam;
                        sc[CF::SC_W + t] = w;
                        sc[CF::SC_SCB + t] = m3::ex2_approx(cs_end - cs[u]) * w;
                        sc[CF::SC_SCF + t] = m3::ex2_approx(cs_ref - cs[u]) * w;
                        // >= w; bounded by 2^kSpanMax w wherever the consumer uses it
                        sc[CF::SC_SDF + t] = m3::ex2_approx(fminf(cs_first - cs[u], kSpanMax)) * w;
                    }
                }
                if (lane == 0) sc[CF::SC_DEC] = m3::ex2_approx(cs_end);
            }

            // (2) this chunk's tiles; the angles of this thread's row and pairs
            bool fail = !ptx::mbar_wait(&bar_lda[s], (c >> 1) & 1, kWaitBudget);
            if constexpr (NORM && ROT) {
                // B / C normalisation of the Mamba-3 block (§3.4), B's part: each row
                // (one token and rank) divided by its RMS over N, scaled and given this
                // head's bias in fp32 and rounded to bf16 in place, before the angles
                // (no sine or cosine is live yet).  The two halves of a row sit in lanes
                // l and l ^ 16.
                const float* nrm = reinterpret_cast<const float*>(smem + CF::OFF_NRM);   // B's (w, w, b, b) per pair
                uint8_t* sbn = st + CF::ST_B;
                uint4 v[GPT];
#pragma unroll
                for (int g = 0; g < GPT; ++g) v[g] = *reinterpret_cast<const uint4*>(sbn + swz(row, hf * GPT + g));
                const float inv = row_rms_inv(v, 1.0f / N, prm.norm_eps);
                const float2 inv2 = make_float2(inv, inv);
#pragma unroll
                for (int g = 0; g < GPT; ++g) {
                    uint32_t* pv = reinterpret_cast<uint32_t*>(&v[g]);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int n = (hf * GPT + g) * 8 + 2 * m;   // column of the pair's first element
                        const float4 wb = *reinterpret_cast<const float4*>(nrm + 2 * n);
                        const float2 u = __ffma2_rn(__fmul2_rn(make_float2(bf_lo(pv[m]), bf_hi(pv[m])), inv2),
                                                    make_float2(wb.x, wb.y), make_float2(wb.z, wb.w));
                        pv[m] = pack_bf16(u.x, u.y);
                    }
                    *reinterpret_cast<uint4*>(sbn + swz(row, hf * GPT + g)) = v[g];
                }
            }
            float cn[PH], sn[PH];
            if (ROT) {
                if (!fail) fail = !ptx::mbar_wait(&bar_phi, c & 1, kWaitBudget);
                __syncwarp();   // tcgen05.ld below is warp-aligned
                ptx::tc_fence_after();
                const float* cin = carry_buf + s * K + hf * PH;
                if constexpr (CKPT) {
                    // the angle before chunk c's first token, for the backward pass
                    if (row == 0) {
                        float* dst = prm.ck_phi + ((int64_t)unit * (nch + 1) + c) * K + hf * PH;
#pragma unroll
                        for (int q = 0; q < PH; ++q) dst[q] = cin[q];
                    }
                }
                float* cout = carry_buf + (s ^ 1) * K + hf * PH;
                const uint32_t taddr = tm_sy + ((uint32_t)(warp * 32) << 16);
#pragma unroll
                for (int q = 0; q < PH; q += 16) {
                    uint32_t v[16];
                    if constexpr (PH == 16) ptx::tmem_ld16x2_16h(taddr, v);       // pairs [16 hf, 16 hf + 16)
                    else ptx::tmem_ld16x2_16(taddr + q, v);                          // pairs 32 hf + q + [0, 16)
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        const float4 cv = *reinterpret_cast<const float4*>(cin + q + e);
                        const float car[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const float phi = car[m] + __uint_as_float(v[e + m]);
                            sincos_reduced(phi, &sn[q + e + m], &cn[q + e + m]);
                            // the chunk's last row carries its angles to the next chunk
                            if (row == kRows - 1) cout[q + e + m] = reduce_2pi(phi);
                        }
                    }
                }
                ptx::tc_fence_before();
            }

            // (3) rotate this thread's half rows of B, C in place (B~, C~); after
            //     warp 0's scalars are in, write B~' = scale * B~
            {
                uint8_t* sb = st + CF::ST_B;
                uint8_t* scc = st + CF::ST_C;
                uint8_t* bd = smem + CF::OFF_BD + s * NSLAB * TILE;
                uint4 vb[GPT];
#pragma unroll
                for (int g = 0; g < GPT; ++g) vb[g] = *reinterpret_cast<const uint4*>(sb + swz(row, hf * GPT + g));
                if constexpr (NORM && ROT) {
                    // C's normalisation (B's ran in step (2)), then the joint rotation of
                    // the plain path: C's row sum of squares over one 16-byte group at a
                    // time, then per group normalise C, rotate B and C, store both
                    if (!fail) fail = !ptx::mbar_wait(&bar_ldb[s], (c >> 1) & 1, kWaitBudget);   // C and x
                    const float* nrm = reinterpret_cast<const float*>(smem + CF::OFF_NRM) + 2 * N;   // C's
                    float ic;
                    {
                        uint4 q[GPT];
#pragma unroll
                        for (int g = 0; g < GPT; ++g) q[g] = *reinterpret_cast<const uint4*>(scc + swz(row, hf * GPT + g));
                        ic = row_rms_inv(q, 1.0f / N, prm.norm_eps);
                    }
                    const float2 ic2 = make_float2(ic, ic);
#pragma unroll
                    for (int g = 0; g < GPT; ++g) {
                        const uint32_t off = swz(row, hf * GPT + g);
                        uint4 q = *reinterpret_cast<const uint4*>(scc + off);
                        uint32_t* pb = reinterpret_cast<uint32_t*>(&vb[g]);
                        uint32_t* pc = reinterpret_cast<uint32_t*>(&q);
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const int n = (hf * GPT + g) * 8 + 2 * m;
                            const float4 wb = *reinterpret_cast<const float4*>(nrm + 2 * n);
                            const float2 cq = __ffma2_rn(__fmul2_rn(make_float2(bf_lo(pc[m]), bf_hi(pc[m])), ic2),
                                                         make_float2(wb.x, wb.y), make_float2(wb.z, wb.w));
                            // Rot(-phi): (a, b) -> (a cos + b sin, -a sin + b cos), for the B pair
                            // and the normalised C pair at once: u = (a_B, a_C), v = (b_B, b_C)
                            const float2 u = make_float2(bf_lo(pb[m]), cq.x);
                            const float2 v = make_float2(bf_hi(pb[m]), cq.y);
                            const float co = cn[g * 4 + m], si = sn[g * 4 + m];
                            const float2 c2 = make_float2(co, co), s2 = make_float2(si, si), ns2 = make_float2(-si, -si);
                            const float2 u2 = __ffma2_rn(u, c2, __fmul2_rn(v, s2));
                            const float2 v2 = __ffma2_rn(v, c2, __fmul2_rn(u, ns2));
                            pb[m] = pack_bf16(u2.x, v2.x);
                            pc[m] = pack_bf16(u2.y, v2.y);
                        }
                        *reinterpret_cast<uint4*>(sb + off) = vb[g];
                        *reinterpret_cast<uint4*>(scc + off) = q;
                    }
                } else if constexpr (NORM) {
                    // the same normalisation without a rotation: B and C together in packed
                    // fp32x2 math, u = (a_B, a_C), v = (b_B, b_C) for a pair's elements (a, b)
                    // (without theta every tile of the chunk is already in)
                    uint4 vc[GPT];
#pragma unroll
                    for (int g = 0; g < GPT; ++g) vc[g] = *reinterpret_cast<const uint4*>(scc + swz(row, hf * GPT + g));
                    // (B row, C row) sums of squares on two accumulators (half the dependent chain)
                    float2 ss = make_float2(0.0f, 0.0f), s1 = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int g = 0; g < GPT; ++g) {
                        const uint32_t* pb = reinterpret_cast<const uint32_t*>(&vb[g]);
                        const uint32_t* pc = reinterpret_cast<const uint32_t*>(&vc[g]);
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const float2 u = make_float2(bf_lo(pb[m]), bf_lo(pc[m]));
                            const float2 v = make_float2(bf_hi(pb[m]), bf_hi(pc[m]));
                            ss = __ffma2_rn(u, u, ss);
                            s1 = __ffma2_rn(v, v, s1);
                        }
                    }
                    ss.x += s1.x;
                    ss.y += s1.y;
                    // the tiles are unpacked again below rather than kept as 64 fp32 values
#pragma unroll
                    for (int g = 0; g < GPT; ++g) {
                        asm volatile("" : "+r"(vb[g].x), "+r"(vb[g].y), "+r"(vb[g].z), "+r"(vb[g].w));
                        asm volatile("" : "+r"(vc[g].x), "+r"(vc[g].y), "+r"(vc[g].z), "+r"(vc[g].w));
                    }
                    ss.x += __shfl_xor_sync(0xffffffffu, ss.x, 16);
                    ss.y += __shfl_xor_sync(0xffffffffu, ss.y, 16);
                    const float2 inv = make_float2(rms_inv(ss.x, 1.0f / N, prm.norm_eps),
                                                   rms_inv(ss.y, 1.0f / N, prm.norm_eps));
                    const float* nrm = reinterpret_cast<const float*>(smem + CF::OFF_NRM);
#pragma unroll
                    for (int g = 0; g < GPT; ++g) {
                        uint32_t* pb = reinterpret_cast<uint32_t*>(&vb[g]);
                        uint32_t* pc = reinterpret_cast<uint32_t*>(&vc[g]);
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const int n = (hf * GPT + g) * 8 + 2 * m;   // column of the pair's first element
                            const float4 w = *reinterpret_cast<const float4*>(nrm + 2 * n);           // wB, wC at n, n + 1
                            const float4 bi = *reinterpret_cast<const float4*>(nrm + 2 * N + 2 * n);  // biases likewise
                            const float2 u = __ffma2_rn(__fmul2_rn(make_float2(bf_lo(pb[m]), bf_lo(pc[m])), inv),
                                                        make_float2(w.x, w.y), make_float2(bi.x, bi.y));
                            const float2 v = __ffma2_rn(__fmul2_rn(make_float2(bf_hi(pb[m]), bf_hi(pc[m])), inv),
                                                        make_float2(w.z, w.w), make_float2(bi.z, bi.w));
                            pb[m] = pack_bf16(u.x, v.x);
                            pc[m] = pack_bf16(u.y, v.y);
                        }
                        const uint32_t off = swz(row, hf * GPT + g);
                        *reinterpret_cast<uint4*>(sb + off) = vb[g];
                        *reinterpret_cast<uint4*>(scc + off) = vc[g];
                        asm volatile("" ::: "memory");   // the next group's scale / bias loads stay behind
                    }
                } else if (ROT && CKPT) {
                    // B~ alone, kept in registers for B~' (S is not formed); x must be in
                    // before dG
                    if (!fail) fail = !ptx::mbar_wait(&bar_ldb[s], (c >> 1) & 1, kWaitBudget);   // x
#pragma unroll
                    for (int g = 0; g < GPT; ++g) {
                        uint32_t* pb = reinterpret_cast<uint32_t*>(&vb[g]);
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            // Rot(-phi): (a, b) -> (a cos + b sin, -a sin + b cos)
                            const float a = bf_lo(pb[m]), bb = bf_hi(pb[m]);
                            const float co = cn[g * 4 + m], si = sn[g * 4 + m];
                            pb[m] = pack_bf16(fmaf(a, co, bb * si), fmaf(bb, co, a * -si));
                        }
                    }
                } else if (ROT) {
                    if (!fail) fail = !ptx::mbar_wait(&bar_ldb[s], (c >> 1) & 1, kWaitBudget);   // C and x
                    uint4 vc[GPT];
#pragma unroll
                    for (int g = 0; g < GPT; ++g) vc[g] = *reinterpret_cast<const uint4*>(scc + swz(row, hf * GPT + g));
#pragma unroll
                    for (int g = 0; g < GPT; ++g) {
                        uint32_t* pb = reinterpret_cast<uint32_t*>(&vb[g]);
                        uint32_t* pc = reinterpret_cast<uint32_t*>(&vc[g]);
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            // Rot(-phi): (a, b) -> (a cos + b sin, -a sin + b cos), for the
                            // B pair and the C pair at once: u = (a_B, a_C), v = (b_B, b_C)
                            const float2 u = make_float2(bf_lo(pb[m]), bf_lo(pc[m]));
                            const float2 v = make_float2(bf_hi(pb[m]), bf_hi(pc[m]));
                            const float co = cn[g * 4 + m], si = sn[g * 4 + m];
                            const float2 c2 = make_float2(co, co), s2 = make_float2(si, si), ns2 = make_float2(-si, -si);
                            const float2 u2 = __ffma2_rn(u, c2, __fmul2_rn(v, s2));
                            const float2 v2 = __ffma2_rn(v, c2, __fmul2_rn(u, ns2));
                            pb[m] = pack_bf16(u2.x, v2.x);
                            pc[m] = pack_bf16(u2.y, v2.y);
                        }
                        const uint32_t off = swz(row, hf * GPT + g);
                        *reinterpret_cast<uint4*>(sb + off) = vb[g];
                        *reinterpret_cast<uint4*>(scc + off) = vc[g];
                    }
                }
                ptx::bar_sync(kBarWG0, kWG);   // warp 0's scalars are in shared memory
                const float rs = sc[CF::SC_SCB + tok];
#pragma unroll
                for (int g = 0; g < GPT; ++g) {
                    // B~' = scale * B~ (from the rounded B~, as the MMA sees it)
                    const uint32_t* pb = reinterpret_cast<const uint32_t*>(&vb[g]);
                    *reinterpret_cast<uint4*>(bd + swz(row, hf * GPT + g)) =
                        make_uint4(pack_bf16(bf_lo(pb[0]) * rs, bf_hi(pb[0]) * rs),
                                   pack_bf16(bf_lo(pb[1]) * rs, bf_hi(pb[1]) * rs),
                                   pack_bf16(bf_lo(pb[2]) * rs, bf_hi(pb[2]) * rs),
                                   pack_bf16(bf_lo(pb[3]) * rs, bf_hi(pb[3]) * rs));
                }
            }
            ptx::fence_proxy_async_smem();
            if (fail) { m3::set_status(m3::kStatusWaitTimeout); abort_s = 1; }
            if (ptx::bar_sync_or(kBarWG0, kWG, fail || abort_s)) { aborted = true; break; }

            // (5) thread kLateIssuer: S = C~ B~^T -> TMEM S/Y[s];  dG = B~'^T X -> TMEM dG
            if (tid == kLateIssuer) {
                bool ok = true;
                if (c >= 1) ok = ptx::mbar_wait(&bar_dgfree, (c - 1) & 1, kWaitBudget);
                if (!ok) {
                    m3::set_status(m3::kStatusWaitTimeout);
                    abort_s = 1;
                } else {
                    ptx::tc_fence_after();
                    const uint32_t c_lo = ptx::sdesc_lo(ptx::smem_u32(st + CF::ST_C), 16);
                    const uint32_t b_lo = ptx::sdesc_lo(ptx::smem_u32(st + CF::ST_B), 16);
                    const uint32_t x_lo = ptx::sdesc_lo(ptx::smem_u32(st + CF::ST_X), TILE);
                    const uint32_t bd_lo = ptx::sdesc_lo(ptx::smem_u32(smem + CF::OFF_BD + s * NSLAB * TILE), TILE);
                    constexpr uint32_t id_s = ptx::idesc_bf16(kRows, kRows, false, false);
                    constexpr uint32_t id_g = ptx::idesc_bf16(N, kP, true, true);
                    const uint32_t tm_s = tmem + CF::TM_SY0 + 64u * s;
                    if constexpr (!CKPT) {
#pragma unroll
                        for (int k16 = 0; k16 < N / 16; ++k16) {   // K = state (K-major slabs)
                            const uint32_t ko = ((k16 >> 2) * TILE + (k16 & 3) * 32) >> 4;
                            ptx::umma_bf16_lo<kDescHi, kDescHi>(tm_s, c_lo + ko, b_lo + ko, id_s, k16 > 0);
                        }
                    }
#pragma unroll
                    for (int k16 = 0; k16 < kRows / 16; ++k16)   // K = rows (MN-major operands)
                        ptx::umma_bf16_lo<kDescHi, kDescHi>(tmem + CF::TM_DG, bd_lo + k16 * 128, x_lo + k16 * 128, id_g,
                                                             k16 > 0);
                    ptx::umma_commit(&bar_sd[s]);
                }
            }
            __syncwarp();   // as above, for the S / dG issuer's warp
        }
        if (!CKPT && tid == kEarlyIssuer && !aborted && (nch >= 2 || prm.h0 != nullptr || prm.prev_B != nullptr))
            issue_early(nch);   // Y_inter(nch - 1)
        if (warp == 0) ptx::cp_async_wait_all();   // a stop may leave a scalar copy in flight
    } else {
        // ======================= warpgroup 1: mask, state, output =======================
        const int w1 = warp - 4;
        const bool leader = (tid == kWG);
        const int i_row = w1 * 16 + (lane & 15);      // tile row of S / Y held by this thread
        const int hc = lane >> 4;                     // column half: [32 hc, 32 hc + 32)
        const int ti = i_row / R;                     // its token
        const uint32_t lane_base = (uint32_t)(w1 * 32) << 16;
        const int g_row = (N == 64) ? i_row : (w1 * 32 + lane);

        if (tid == kLoader) {
            for (int c = 0; c < 2 && c < nch; ++c) {
                issue_loads_a(c);
                issue_loads_b(c);
                last_a = last_b = c;
            }
        }
        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            uint8_t* st = smem + s * CF::ST_BYTES;
            const float* sc = scal0 + (c % 3) * CF::SC_STRIDE;
            const uint32_t tm_sy = tmem + lane_base + CF::TM_SY0 + 64u * s;
            // (1) S_c and dG_c are in TMEM
            bool fail = !ptx::mbar_wait(&bar_sd[s], (c >> 1) & 1, kWaitBudget);
            __syncwarp();   // tcgen05.ld / wait::ld below are warp-aligned
            ptx::tc_fence_after();
            // theta and B of stage s have been read (Phi_c before S_c; S_c is done):
            // part a of chunk c + 2
            if (ROT && tid == kLoader && !fail && c + 2 < nch) {
                issue_loads_a(c + 2);
                last_a = c + 2;
            }
            if constexpr (CKPT) {
                // x is free once dG_c is done: the rest of chunk c + 2
                if (tid == kLoader && !fail && c + 2 < nch) {
                    if (ROT) {
                        issue_loads_b(c + 2);
                        last_b = c + 2;
                    } else {
                        issue_loads_a(c + 2);
                        last_a = c + 2;
                    }
                }
            }
            const float cs_i = sc[CF::SC_CS + ti];
            if constexpr (!CKPT) {
            // S_c, block J (columns 16 J + [0, 16)) in v[8 J, 8 J + 8): this thread
            // holds columns 16 J + 8 hc + [0, 8) (waited for in the mask below)
            uint32_t v[32];
#pragma unroll
            for (int J = 0; J < 4; ++J) ptx::tmem_ld16x2_8(tm_sy + 16 * J, *reinterpret_cast<uint32_t(*)[8]>(&v[8 * J]));
            // (2) mask: S' = S o M for this thread's row, 8 columns in each of the
            //     four 16-row blocks; the block kind (below / diagonal / above)
            //     is the same for the whole warp
            {
                constexpr int TB = CF::TB;
                constexpr int TPC = 8 / R;                         // tokens under 8 columns
                const float gam_i = sc[CF::SC_GAM + ti];
#pragma unroll
                for (int J = 0; J < 4; ++J) {
                    const int t0 = (16 * J + 8 * hc) / R;         // first token of these columns
                    float mk[TPC];
                    if (J < w1) {
                        // strictly below the diagonal block: exp(cs_i - cs_r) * [exp(cs_r - cs_j) w_j]
                        const float u = m3::ex2_approx(cs_i - sc[CF::SC_CS + J * TB + TB - 1]);
                        load_tok<TPC>(sc + CF::SC_SCF + t0, mk);
#pragma unroll
                        for (int e = 0; e < TPC; ++e) mk[e] *= u;
                    } else if (J == w1) {
                        // diagonal block: exp(cs_i - cs_f) * [exp(cs_f - cs_j) w_j] around the
                        // block's first token f while its decay span stays below 2^kSpanMax
                        // (both factors finite), else one exp per token
                        const float cs_f = sc[CF::SC_CS + J * TB];
                        if (cs_f - sc[CF::SC_CS + J * TB + TB - 1] <= kSpanMax) {
                            const float e_i = m3::ex2_approx(cs_i - cs_f);
                            load_tok<TPC>(sc + CF::SC_SDF + t0, mk);
#pragma unroll
                            for (int e = 0; e < TPC; ++e) mk[e] *= e_i;
                        } else {
#pragma unroll
                            for (int e = 0; e < TPC; ++e)
                                mk[e] = m3::ex2_approx(cs_i - sc[CF::SC_CS + t0 + e]) * sc[CF::SC_W + t0 + e];
                        }
#pragma unroll
                        for (int e = 0; e < TPC; ++e)
                            mk[e] = (t0 + e < ti) ? mk[e] : (t0 + e == ti ? gam_i : 0.0f);
                    } else {
#pragma unroll
                        for (int e = 0; e < TPC; ++e) mk[e] = 0.0f;
                    }
                    if (J == 0) {
                        __syncwarp();
                        ptx::tmem_ld_wait();
                    }
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const float2 sv = __fmul2_rn(
                            make_float2(__uint_as_float(v[8 * J + e]), __uint_as_float(v[8 * J + e + 1])),
                            make_float2(mk[e / R], mk[(e + 1) / R]));
                        o[e / 2] = pack_bf16(sv.x, sv.y);
                    }
                    *reinterpret_cast<uint4*>(t_sp + swz(i_row, 2 * J + hc)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            }   // !CKPT
            // (3) G_c = exp(cs_end) G_{c-1} + dG_c (fp32)
            if constexpr (CKPT) {
                // G_{-1} for the backward pass (rows and columns as held here); the later
                // checkpoints leave through the staging tile below
                if (c == 0) {
                    float* dst = prm.ck_G + (((int64_t)unit * (nch + 1)) * N + g_row) * kP + ((N == 64) ? hc * 32 : 0);
#pragma unroll
                    for (int p4 = 0; p4 < GC / 4; ++p4)
                        *reinterpret_cast<float4*>(dst + 4 * p4) =
                            make_float4(G[4 * p4], G[4 * p4 + 1], G[4 * p4 + 2], G[4 * p4 + 3]);
                }
            }
            __syncwarp();
            {
                const float dec = sc[CF::SC_DEC];
                if constexpr (N == 64) {
                    uint32_t v[32];
                    ptx::tmem_ld16x2_32(tmem + lane_base + CF::TM_DG, v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int p = 0; p < 32; p += 2) {
                        const float2 g2 = __ffma2_rn(make_float2(dec, dec), make_float2(G[p], G[p + 1]),
                                                     make_float2(__uint_as_float(v[p]), __uint_as_float(v[p + 1])));
                        G[p] = g2.x; G[p + 1] = g2.y;
                    }
                } else {
#pragma unroll
                    for (int c32 = 0; c32 < 2; ++c32) {
                        uint32_t v[32];
                        ptx::tmem_ld32(tmem + lane_base + CF::TM_DG + c32 * 32, v);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int p = 0; p < 32; p += 2) {
                            const float2 g2 = __ffma2_rn(make_float2(dec, dec),
                                                         make_float2(G[c32 * 32 + p], G[c32 * 32 + p + 1]),
                                                         make_float2(__uint_as_float(v[p]), __uint_as_float(v[p + 1])));
                            G[c32 * 32 + p] = g2.x; G[c32 * 32 + p + 1] = g2.y;
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::fence_proxy_async_smem();
            if (leader) ptx::bulk_wait_read0();   // the previous y store has left the staging tile
            if (fail) { m3::set_status(m3::kStatusWaitTimeout); abort_s = 1; }
            if (ptx::bar_sync_or(kBarWG1, kWG, fail || abort_s)) { aborted = true; break; }
            if (leader) ptx::mbar_arrive(&bar_dgfree);
            if constexpr (CKPT) {
                static_assert(!CKPT || N == 64, "checkpoint run: N = 64");
                // no output: the S/Y buffer of stage s (it held Phi_c only) is free
                if (leader) ptx::mbar_arrive(&bar_syfree[s]);
                if (c + 1 < nch) {
                    // G_c (checkpoint slot c + 1) into the staging tile (the S', G and y
                    // buffers, unused here): two [64 rows][32 floats] boxes, 128-byte
                    // swizzled (conflict-free: the eight rows of a quarter-warp land in
                    // eight 16-byte columns); the previous stores have read it (the
                    // leader waited before the barrier above)
                    uint8_t* box = smem + CF::OFF_SP + hc * (64 * 128);
#pragma unroll
                    for (int p4 = 0; p4 < 8; ++p4)
                        *reinterpret_cast<float4*>(box + g_row * 128 + ((p4 ^ (g_row & 7)) << 4)) =
                            make_float4(G[4 * p4], G[4 * p4 + 1], G[4 * p4 + 2], G[4 * p4 + 3]);
                    ptx::fence_proxy_async_smem();
                    ptx::bar_sync(kBarWG1, kWG);
                    if (leader) {
                        const int slot = (int)((int64_t)unit * (nch + 1) + c + 1);
                        ptx::tma_store_3d(&map_y, smem + CF::OFF_SP, 0, 0, slot);
                        ptx::tma_store_3d(&map_y, smem + CF::OFF_SP + 64 * 128, 32, 0, slot);
                        ptx::bulk_commit();
                    }
                }
                continue;
            }
            if (tid == kYIssuer) {
                ptx::tc_fence_after();
                // Y_intra = S' X -> TMEM S/Y[s] (S has been read by every thread)
                const uint32_t sp_lo = ptx::sdesc_lo(ptx::smem_u32(t_sp), 16);
                const uint32_t x_lo = ptx::sdesc_lo(ptx::smem_u32(st + CF::ST_X), TILE);
                constexpr uint32_t id_y = ptx::idesc_bf16(kRows, kP, false, true);
#pragma unroll
                for (int k16 = 0; k16 < kRows / 16; ++k16)
                    ptx::umma_bf16_lo<kDescHi, kDescHi>(tmem + CF::TM_SY0 + 64u * s, sp_lo + k16 * 2, x_lo + k16 * 128,
                                                         id_y, k16 > 0);
                ptx::umma_commit(&bar_y);
            }
            __syncwarp();   // as above, for the Y_intra issuer's warp
            // (4) G_{c-1} is no longer read: store the bf16 copy of G_c
            fail = false;
            // chunk c has an inter-chunk term (always for a continuation); the flag is
            // re-read from the kernel parameters rather than kept in a register
            const bool cont = (prm.h0 != nullptr) || (prm.prev_B != nullptr);
            const bool has_yi = (c > 0) || cont;
            if (has_yi) fail = !ptx::mbar_wait(&bar_yi, (cont ? c : c - 1) & 1, kWaitBudget);
            if constexpr (N == 64) {
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    *reinterpret_cast<uint4*>(t_g + swz(g_row, hc * 4 + g)) =
                        make_uint4(pack_bf16(G[g * 8 + 0], G[g * 8 + 1]), pack_bf16(G[g * 8 + 2], G[g * 8 + 3]),
                                   pack_bf16(G[g * 8 + 4], G[g * 8 + 5]), pack_bf16(G[g * 8 + 6], G[g * 8 + 7]));
            } else {
#pragma unroll
                for (int g = 0; g < 8; ++g)
                    *reinterpret_cast<uint4*>(t_g + swz(g_row, g)) =
                        make_uint4(pack_bf16(G[g * 8 + 0], G[g * 8 + 1]), pack_bf16(G[g * 8 + 2], G[g * 8 + 3]),
                                   pack_bf16(G[g * 8 + 4], G[g * 8 + 5]), pack_bf16(G[g * 8 + 6], G[g * 8 + 7]));
            }
            // (5) Y_intra done: C and x of stage s are free -> part b of chunk c + 2
            //     (without the rotation, every tile of chunk c + 2)
            if (!fail) fail = !ptx::mbar_wait(&bar_y, c & 1, kWaitBudget);
            __syncwarp();
            ptx::tc_fence_after();
            if (tid == kLoader && !fail && c + 2 < nch) {
                if (ROT) {
                    issue_loads_b(c + 2);
                    last_b = c + 2;
                } else {
                    issue_loads_a(c + 2);
                    last_a = c + 2;
                }
            }
            // (6) y = Y_intra + exp(cs) Y_inter -> bf16 staging -> TMA store
            {
                const float e = m3::ex2_approx(cs_i);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t ya[16], yb[16];
                    ptx::tmem_ld16x2_16(tm_sy + q * 16, ya);
                    if (has_yi) ptx::tmem_ld16x2_16(tmem + lane_base + CF::TM_YI + q * 16, yb);
                    ptx::tmem_ld_wait();
                    float y[16];
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float2 a2 = make_float2(__uint_as_float(ya[j]), __uint_as_float(ya[j + 1]));
                        float2 r2 = a2;
                        if (has_yi)
                            r2 = __ffma2_rn(make_float2(e, e), make_float2(__uint_as_float(yb[j]), __uint_as_float(yb[j + 1])),
                                            a2);
                        y[j] = r2.x; y[j + 1] = r2.y;
                    }
                    // columns 32 hc + 16 q + [0, 16) -> groups 4 hc + 2 q, +1
#pragma unroll
                    for (int g = 0; g < 2; ++g)
                        *reinterpret_cast<uint4*>(t_y + swz(i_row, hc * 4 + q * 2 + g)) =
                            make_uint4(pack_bf16(y[g * 8 + 0], y[g * 8 + 1]), pack_bf16(y[g * 8 + 2], y[g * 8 + 3]),
                                       pack_bf16(y[g * 8 + 4], y[g * 8 + 5]), pack_bf16(y[g * 8 + 6], y[g * 8 + 7]));
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            if (fail) { m3::set_status(m3::kStatusWaitTimeout); abort_s = 1; }
            if (ptx::bar_sync_or(kBarWG1, kWG, fail || abort_s)) { aborted = true; break; }
            if (leader) {
                ptx::tma_store_5d(&map_y, t_y, 0, 0, h, c * Q, b);
                ptx::bulk_commit();
                ptx::mbar_arrive(&bar_syfree[s]);
            }
        }

        if (leader) ptx::bulk_wait0();   // every y store is complete
    }

    // ---- final state = Rot(Phi_{T-1}) G in the complex frame.  The angle carry
    // was written by warpgroup 0 before its last barrier; the CTA barrier below
    // makes it visible.  A stop anywhere (abort_s) skips the write.
    __syncthreads();
    aborted = (abort_s != 0);
    if constexpr (CKPT) {
        // G_last and the final angle, after the last chunk (slot nch)
        if (!aborted && tid >= kWG) {
            const int w1 = warp - 4;
            const int g_row = (N == 64) ? (w1 * 16 + (lane & 15)) : (w1 * 32 + lane);
            float* dst = prm.ck_G + (((int64_t)unit * (nch + 1) + nch) * N + g_row) * kP + ((N == 64) ? (lane >> 4) * 32 : 0);
#pragma unroll
            for (int p4 = 0; p4 < GC / 4; ++p4)
                *reinterpret_cast<float4*>(dst + 4 * p4) = make_float4(G[4 * p4], G[4 * p4 + 1], G[4 * p4 + 2], G[4 * p4 + 3]);
        }
        if (!aborted && tid < K)
            prm.ck_phi[((int64_t)unit * (nch + 1) + nch) * K + tid] = ROT ? s_carry[(nch & 1) * K + tid] : 0.0f;
    }
    if (!aborted && prm.final_state && tid >= kWG) {
        const int w1 = warp - 4;
        const int g_row = (N == 64) ? (w1 * 16 + (lane & 15)) : (w1 * 32 + lane);
        const int col0 = (N == 64) ? (lane >> 4) * 32 : 0;
        float cn = 1.0f, sn = 0.0f;
        if (ROT) sincosf(s_carry[(nch & 1) * K + (g_row >> 1)], &sn, &cn);
        const bool even = (g_row & 1) == 0;
        float* fs = prm.final_state + (((int64_t)b * prm.H + h) * N + g_row) * kP + col0;
#pragma unroll
        for (int p4 = 0; p4 < GC / 4; ++p4) {
            float o[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float mine = G[p4 * 4 + u];
                const float other = __shfl_xor_sync(0xffffffffu, mine, 1);   // row partner 2k <-> 2k+1
                // (a, b) -> (a cos - b sin, a sin + b cos)
                o[u] = ROT ? (even ? cn * mine - sn * other : sn * other + cn * mine) : mine;
            }
            *reinterpret_cast<float4*>(fs + p4 * 4) = make_float4(o[0], o[1], o[2], o[3]);
        }
    }
    if (aborted && tid == kWG) ptx::bulk_wait0();   // y stores still in flight
    if (aborted && tid == kLoader) {
        // stopped early: wait (bounded) for the loads still in flight
        // (the two stages last received chunks last - 1 and last of each part)
        for (int k = 0; k < 2; ++k) {
            const int ca = last_a - k, cb = last_b - k;
            if (ca >= 0) (void)ptx::mbar_wait(&bar_lda[ca & 1], (ca >> 1) & 1, kWaitBudget);
            if (ROT && cb >= 0) (void)ptx::mbar_wait(&bar_ldb[cb & 1], (cb >> 1) & 1, kWaitBudget);
        }
    }
    if (aborted && (tid == kEarlyIssuer || tid == kLateIssuer || tid == kYIssuer)) {
        // every MMA this thread issued has completed once this commit arrives
        const int k = (tid == kEarlyIssuer) ? 0 : (tid == kLateIssuer ? 1 : 2);
        ptx::umma_commit(&bar_fin[k]);
        (void)ptx::mbar_wait(&bar_fin[k], 0, kWaitBudget);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc(tmem, CF::TM_COLS);
}

}  // namespace m3ws

// ----------------------------------------------------------------------------- host side
namespace m3ws {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// The shapes this kernel takes: bf16, P = 64, N in {64, 128}, R in {1, 2, 4}.
// The chunk is Q = 64 / R tokens (64 tile rows) whatever d.chunk asks for.
inline bool supports(const m3_dims& d) {
    if (d.dtype != M3_BF16 || d.headdim != kP) return false;
    if (d.dstate != 64 && d.dstate != 128) return false;
    if (d.rank != 1 && d.rank != 2 && d.rank != 4) return false;
    if (d.heads > 65535 || d.seqlen > INT32_MAX / 2 || d.batch > 65535) return false;
    return true;
}

// 5-D map over a [b, T, h, R, inner] bf16 tensor: box (64, R, 1, Q, 1), 128-byte swizzle.
inline bool make_map5(CUtensorMap* m, const void* base, const m3_dims& d, int inner, int Q) {
    const cuuint64_t R = (cuuint64_t)d.rank;
    cuuint64_t dims[5] = {(cuuint64_t)inner, R, (cuuint64_t)d.heads, (cuuint64_t)d.seqlen, (cuuint64_t)d.batch};
    cuuint64_t strides[4] = {(cuuint64_t)inner * 2, R * inner * 2, (cuuint64_t)d.heads * R * inner * 2,
                             (cuuint64_t)d.seqlen * d.heads * R * inner * 2};
    cuuint32_t box[5] = {64, (cuuint32_t)R, 1, (cuuint32_t)Q, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over theta [b, T, h, K] bf16: box (K, 1, Q, 1); the tile is the
// MN-major operand of the angle MMA, so it lands 64-byte swizzled (K = 32
// pairs, 64-byte rows) or 128-byte swizzled (K = 64).
inline bool make_map_theta(CUtensorMap* m, const void* base, const m3_dims& d, int Q) {
    const cuuint64_t K = (cuuint64_t)d.dstate / 2;
    cuuint64_t dims[4] = {K, (cuuint64_t)d.heads, (cuuint64_t)d.seqlen, (cuuint64_t)d.batch};
    cuuint64_t strides[3] = {K * 2, (cuuint64_t)d.heads * K * 2, (cuuint64_t)d.seqlen * d.heads * K * 2};
    cuuint32_t box[4] = {(cuuint32_t)K, 1, (cuuint32_t)Q, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle sw = (K == 32) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NSLAB, int R, bool ROT, bool NORM, bool CKPT = false>
int launch_cfg(const m3_dims& d, const CUtensorMap* maps, const Params& prm, cudaStream_t s) {
    using CF = Cfg<NSLAB, R, ROT, NORM>;
    auto k = m3_scan_ws_kernel<NSLAB, R, ROT, NORM, CKPT>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_BYTES) != cudaSuccess)
        return M3_ERR_CUDA;
    k<<<(unsigned)(d.batch * d.heads), kThreads, CF::SMEM_BYTES, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4],
                                                                      prm);
    return cudaGetLastError() == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

template <int NSLAB, bool ROT, bool NORM, bool CKPT = false>
int launch_r(const m3_dims& d, const CUtensorMap* maps, const Params& prm, cudaStream_t s) {
    switch (d.rank) {
        case 1: return launch_cfg<NSLAB, 1, ROT, NORM, CKPT>(d, maps, prm, s);
        case 2: return launch_cfg<NSLAB, 2, ROT, NORM, CKPT>(d, maps, prm, s);
        case 4: return launch_cfg<NSLAB, 4, ROT, NORM, CKPT>(d, maps, prm, s);
    }
    return M3_ERR_UNSUPPORTED;
}

template <int NSLAB, bool NORM>
int launch_n(const m3_dims& d, const CUtensorMap* maps, const Params& prm, bool rot, cudaStream_t s) {
    return rot ? launch_r<NSLAB, true, NORM>(d, maps, prm, s) : launch_r<NSLAB, false, NORM>(d, maps, prm, s);
}

inline int launch(const m3_dims& d, const void* x, const float* dt, const float* A, const void* B, const void* C,
                  const float* lam, const void* theta, const float* h0, const void* prev_B, const void* prev_x,
                  void* y, float* final_state, cudaStream_t s, const float* norm_wB = nullptr,
                  const float* norm_wC = nullptr, const float* norm_bB = nullptr, const float* norm_bC = nullptr,
                  float norm_eps = 0.0f, float* ck_G = nullptr, float* ck_phi = nullptr) {
    if (!supports(d)) return M3_ERR_UNSUPPORTED;
    const void* tma_ptrs[] = {x, B, C, theta, y};
    for (const void* p : tma_ptrs)
        if (p && (reinterpret_cast<uintptr_t>(p) & 15u)) return M3_ERR_ALIGN;
    if (!encode_fn()) return M3_ERR_CUDA;
    const int Q = kRows / (int)d.rank;
    CUtensorMap maps[5];
    memset(maps, 0, sizeof(maps));
    if (!make_map5(&maps[0], x, d, kP, Q) || !make_map5(&maps[1], B, d, (int)d.dstate, Q) ||
        !make_map5(&maps[2], C, d, (int)d.dstate, Q) || !make_map5(&maps[4], y, d, kP, Q))
        return M3_ERR_CUDA;
    const bool rot = theta != nullptr;
    if (rot && !make_map_theta(&maps[3], theta, d, Q)) return M3_ERR_CUDA;
    if (!rot) maps[3] = maps[0];   // never read
    Params prm;
    prm.T = d.seqlen;
    prm.H = (int)d.heads;
    prm.nchunks = (int)((d.seqlen + Q - 1) / Q);
    prm.dt = dt;
    prm.A = A;
    prm.lam = lam;
    prm.final_state = final_state;
    prm.h0 = h0;
    prm.prev_B = static_cast<const __nv_bfloat16*>(prev_B);
    prm.prev_x = static_cast<const __nv_bfloat16*>(prev_x);
    prm.norm_wB = norm_wB;
    prm.norm_wC = norm_wC;
    prm.norm_bB = norm_bB;
    prm.norm_bC = norm_bC;
    prm.norm_eps = norm_eps;
    prm.ck_G = ck_G;
    prm.ck_phi = ck_phi;
    const bool norm = norm_wB != nullptr;
    if (ck_G) {
        // the checkpointing forward of the backward pass: N = 64, no normalisation;
        // no y, the map of the fp32 checkpoints [b h (nch + 1)][N][P] instead
        if (d.dstate != 64 || norm) return M3_ERR_UNSUPPORTED;
        if (reinterpret_cast<uintptr_t>(ck_G) & 15u) return M3_ERR_ALIGN;
        const int64_t slots = d.batch * d.heads * (int64_t)(prm.nchunks + 1);
        if (slots >= INT32_MAX) return M3_ERR_UNSUPPORTED;
        cuuint64_t dims[3] = {(cuuint64_t)kP, 64, (cuuint64_t)slots};
        cuuint64_t strides[2] = {(cuuint64_t)kP * 4, (cuuint64_t)64 * kP * 4};
        cuuint32_t box[3] = {32, 64, 1};
        cuuint32_t es[3] = {1, 1, 1};
        if (encode_fn()(&maps[4], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ck_G, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return M3_ERR_CUDA;
        return rot ? launch_r<1, true, false, true>(d, maps, prm, s) : launch_r<1, false, false, true>(d, maps, prm, s);
    }
    if (d.dstate == 64)
        return norm ? launch_n<1, true>(d, maps, prm, rot, s) : launch_n<1, false>(d, maps, prm, rot, s);
    return norm ? launch_n<2, true>(d, maps, prm, rot, s) : launch_n<2, false>(d, maps, prm, rot, s);
}

}  // namespace m3ws
