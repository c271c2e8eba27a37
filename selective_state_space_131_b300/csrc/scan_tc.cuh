// scan_tc.cuh -- chunked tensor-core (tcgen05 / TMEM / TMA) prefill of the
// Mamba-3 scan for bf16 inputs, fp32 state.
//
// The math (per batch row b and head h; Mamba-3 summary page §3.1-§3.3):
// work in the rotated ("data-dependent RoPE") frame of Propositions 3.2.2 /
// 3.2.3, B~_t = Rot(Phi_t)^T B_t, C~_t = Rot(Phi_t)^T C_t with the cumulative
// angle Phi_t = sum_{i<=t} theta_i, where the recurrence has a scalar decay:
//     h_t = alpha_t h_{t-1} + beta_t v~_{t-1} + gamma_t v~_t,  y_t = C~_t^T h_t.
// Split the sequence in chunks (the SSD intra/inter-chunk split of the
// Mamba-2 chapter page, "Foundation Model Engineering" ch. 20.2 §2).  With
// the chunk-local log decay cs_t = sum_{i=c0}^{t} dt_i A, eq. (7)'s mask
// L = decay x two-band folds into one lower-triangular matrix
//     M_ij = exp(cs_i - cs_j) w_j (j < i),  M_ii = gamma_i,  0 (j > i),
//     w_j  = gamma_j + (1 - lambda_{j+1}) dt_{j+1}   (= gamma_j + beta_{j+1}/alpha_{j+1}),
// and the state carried between chunks is the augmented
//     G_c = h_end + (1 - lambda_next) dt_next v~_end
//         = exp(cs_end) G_{c-1} + sum_j exp(cs_end - cs_j) w_j v~_j,
// which carries the trapezoid's cross-chunk beta term with no extra buffer.
// Per chunk:
//     S  = C~ B~^T                      (tcgen05, bf16 -> fp32 in TMEM)
//     S' = S o M                        (registers, -> bf16 in shared memory)
//     Y  = S' X + diag(exp(cs)) C~ G_{c-1}   (tcgen05, both into one TMEM accumulator)
//     dG = (diag(exp(cs_end - cs) w) B~)^T X  (tcgen05)
//     G_c = exp(cs_end) G_{c-1} + dG    (fp32, registers)
// and the final state is Rot(Phi_{T-1}) G_last (back to the complex frame).
// MIMO rank R: rows are (token, r) pairs; the mask is shared by the R x R
// blocks of a token pair.
//
// One CTA (128 threads) per (b, h); the chunks of a sequence are processed in
// order (the state chain); TMA double-buffers the next chunk's x, B, C, theta
// while the current one computes.  Every mbarrier wait is bounded.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "m3scan.h"
#include "ptx_sm100.cuh"

namespace m3tc {

constexpr int kThreads = 128;
constexpr int kStages = 2;
constexpr long long kWaitBudget = 4000000000LL;   // clock cycles (~2 s) before a wait gives up
constexpr float kTwoPi = 6.283185307179586f;

__host__ __device__ constexpr int align1k(int x) { return (x + 1023) & ~1023; }
__host__ __device__ constexpr int imax(int a, int b) { return a > b ? a : b; }

// Tile geometry and shared-memory map.  ROWS = Q * R rows per chunk (64 or
// 128), NSLAB = N / 64, R = rank; P = 64.
template <int ROWS, int NSLAB, int R, bool ROT>
struct Cfg {
    static constexpr int Q = ROWS / R;            // tokens per chunk
    static constexpr int N = 64 * NSLAB;
    static constexpr int K = N / 2;               // rotation pairs
    static constexpr int TILE = ROWS * 128;       // one 64-column slab of a ROWS-row bf16 tile
    static constexpr int M_S = ROWS;              // MMA M of S and Y
    static constexpr int M_G = N;                 // MMA M of dG
    // stage (TMA destination)
    static constexpr int ST_X = 0;
    static constexpr int ST_B = ST_X + TILE;
    static constexpr int ST_C = ST_B + NSLAB * TILE;
    static constexpr int ST_TH = ST_C + NSLAB * TILE;
    static constexpr int TH_BYTES = ROT ? Q * K * 2 : 0;
    static constexpr int ST_BYTES = align1k(ST_TH + TH_BYTES);
    static constexpr int TX_BYTES = TILE * (1 + 2 * NSLAB) + TH_BYTES;
    // operand tiles
    static constexpr int OFF_CD = kStages * ST_BYTES;                   // C~' = exp(cs) C~ ; later S'
    static constexpr int CD_BYTES = imax(NSLAB, ROWS / 64) * TILE;
    static constexpr int OFF_BD = OFF_CD + CD_BYTES;                    // B~' ; later y staging
    static constexpr int OFF_G = OFF_BD + NSLAB * TILE;                 // G (bf16, [N][64] MN-major)
    static constexpr int OFF_PHI = OFF_G + N * 128;                     // Phi [Q][K] fp32
    static constexpr int OFF_SCAL = OFF_PHI + (ROT ? Q * K * 4 : 0);
    // scalars (floats): cs[Q], w[Q], gam[Q], d[Q+1], l[Q+1], warp sums[4], theta partials [4][K]
    static constexpr int SC_CS = 0, SC_W = Q, SC_GAM = 2 * Q, SC_D = 3 * Q, SC_L = 4 * Q + 1,
                         SC_WS = 5 * Q + 2, SC_PART = 5 * Q + 6;
    static constexpr int SCAL_FLOATS = SC_PART + 4 * K;
    static constexpr int OFF_CARRY = align1k(OFF_SCAL + SCAL_FLOATS * 4);  // double carry[K]
    static constexpr int SMEM_BYTES = OFF_CARRY + K * 8 + 1024;          // + alignment slack
    // TMEM columns
    static constexpr int TM_S = 0, TM_Y = ROWS, TM_G = ROWS + 64, TM_COLS = 256;
    static_assert(ROWS == 64 || ROWS == 128, "rows per chunk");
    static_assert(TM_G + 64 <= TM_COLS, "tmem budget");
};

struct Params {
    int64_t T;      // sequence length
    int H;          // heads
    int nchunks;
    const float* dt;
    const float* A;
    const float* lam;   // may be null
    float* final_state; // may be null
};

// TMEM row of an accumulator with M rows held by (warp, lane), or -1.
template <int M>
__device__ __forceinline__ int tmem_row(int warp, int lane) {
    if (M == 128) return warp * 32 + lane;
    return lane < 16 ? warp * 16 + lane : -1;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(v);
}

// sin/cos of x: reduce to [-pi, pi] with one constant, then the hardware
// sin/cos (accurate to ~1e-6 absolute on that range).
__device__ __forceinline__ void sincos_reduced(float x, float* s, float* c) {
    const float n = rintf(x * (1.0f / kTwoPi));
    const float r = fmaf(-n, kTwoPi, x);
    __sincosf(r, s, c);
}

template <int ROWS, int NSLAB, int R, bool ROT>
__global__ void __launch_bounds__(kThreads, 1)
    m3_scan_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_B,
                      const __grid_constant__ CUtensorMap map_C, const __grid_constant__ CUtensorMap map_th,
                      const __grid_constant__ CUtensorMap map_y, const Params prm) {
    using CF = Cfg<ROWS, NSLAB, R, ROT>;
    constexpr int Q = CF::Q, N = CF::N, K = CF::K, TILE = CF::TILE;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t bar_full[kStages];
    __shared__ uint64_t bar_mma1, bar_mma2;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x;
    const int h = unit % prm.H;
    const int b = unit / prm.H;
    const int64_t T = prm.T;
    const float A_l2 = __ldg(prm.A + h) * m3::kLog2e;

    float* scal = reinterpret_cast<float*>(smem + CF::OFF_SCAL);
    float* s_cs = scal + CF::SC_CS;
    float* s_w = scal + CF::SC_W;
    float* s_gam = scal + CF::SC_GAM;
    float* s_d = scal + CF::SC_D;
    float* s_l = scal + CF::SC_L;
    float* s_ws = scal + CF::SC_WS;
    float* s_part = scal + CF::SC_PART;
    double* s_carry = reinterpret_cast<double*>(smem + CF::OFF_CARRY);
    float* s_phi = reinterpret_cast<float*>(smem + CF::OFF_PHI);
    uint8_t* t_cd = smem + CF::OFF_CD;   // C~' then S'
    uint8_t* t_bd = smem + CF::OFF_BD;   // B~' then y staging
    uint8_t* t_g = smem + CF::OFF_G;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) ptx::mbar_init(&bar_full[s], 1);
        ptx::mbar_init(&bar_mma1, 1);
        ptx::mbar_init(&bar_mma2, 1);
        ptx::fence_mbar_init();
        abort_s = 0;
        ptx::tma_prefetch_map(&map_x);
        ptx::tma_prefetch_map(&map_B);
        ptx::tma_prefetch_map(&map_C);
        ptx::tma_prefetch_map(&map_y);
        if (ROT) ptx::tma_prefetch_map(&map_th);
    }
    if (warp == 0) {
        ptx::tmem_alloc(&tmem_base_s, CF::TM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid < K) s_carry[tid] = 0.0;
    // G tile starts at zero (G_{-1} = 0)
    for (int i = tid; i < N * 128 / 16; i += kThreads) reinterpret_cast<uint4*>(t_g)[i] = make_uint4(0, 0, 0, 0);
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    auto issue_loads = [&](int c) {
        const int s = c % kStages;
        uint8_t* st = smem + s * CF::ST_BYTES;
        const int t0 = c * Q;
        ptx::mbar_arrive_expect_tx(&bar_full[s], CF::TX_BYTES);
        ptx::tma_load_5d(st + CF::ST_X, &map_x, &bar_full[s], 0, 0, h, t0, b);
#pragma unroll
        for (int sl = 0; sl < NSLAB; ++sl) {
            ptx::tma_load_5d(st + CF::ST_B + sl * TILE, &map_B, &bar_full[s], sl * 64, 0, h, t0, b);
            ptx::tma_load_5d(st + CF::ST_C + sl * TILE, &map_C, &bar_full[s], sl * 64, 0, h, t0, b);
        }
        if (ROT) ptx::tma_load_4d(st + CF::ST_TH, &map_th, &bar_full[s], 0, h, t0, b);
    };
    const int nch = prm.nchunks;
    if (tid == 0) {
        for (int c = 0; c < kStages && c < nch; ++c) issue_loads(c);
    }

    // dt / lambda of tokens c0 .. c0 + Q (Q + 1 values) for the next chunk, in registers
    auto load_scalars = [&](int c, float& dv, float& lv, float& dn, float& ln) {
        const int64_t t = (int64_t)c * Q + tid;
        dv = 0.0f; lv = 1.0f; dn = 0.0f; ln = 1.0f;
        if (tid < Q && t < T) {
            const int64_t idx = ((int64_t)b * T + t) * prm.H + h;
            dv = __ldg(prm.dt + idx);
            if (prm.lam) lv = __ldg(prm.lam + idx);
        }
        const int64_t tn = (int64_t)(c + 1) * Q;
        if (tid == 0 && tn < T) {
            const int64_t idx = ((int64_t)b * T + tn) * prm.H + h;
            dn = __ldg(prm.dt + idx);
            if (prm.lam) ln = __ldg(prm.lam + idx);
        }
    };
    float d_cur, l_cur, dn_cur, ln_cur;
    load_scalars(0, d_cur, l_cur, dn_cur, ln_cur);

    float G[64];   // fp32 state rows owned by this thread (dG layout)
#pragma unroll
    for (int p = 0; p < 64; ++p) G[p] = 0.0f;
    const int g_row = tmem_row<CF::M_G>(warp, lane);
    const int s_row = tmem_row<CF::M_S>(warp, lane);
    // A failed bounded wait sets abort_s; every thread reads it only after a
    // __syncthreads, so the decision to stop is uniform across the CTA.
    auto wait_or_abort = [&](uint64_t* bar, uint32_t parity) {
        if (!ptx::mbar_wait(bar, parity, kWaitBudget)) {
            m3::set_status(m3::kStatusWaitTimeout);
            abort_s = 1;
        }
    };
    int loads_issued = (nch < kStages) ? nch : kStages;   // meaningful in thread 0 only
    int chunks_landed = 0;
    int mma_wait_failed = 0;                                // bit 0: bar_mma1, bit 1: bar_mma2
    int fail_parity = 0;
    bool ok = true;

    for (int c = 0; c < nch; ++c) {
        const int s = c % kStages;
        uint8_t* st = smem + s * CF::ST_BYTES;
        // prefetch next chunk's scalars
        float d_nx = 0.0f, l_nx = 1.0f, dn_nx = 0.0f, ln_nx = 1.0f;
        if (c + 1 < nch) load_scalars(c + 1, d_nx, l_nx, dn_nx, ln_nx);

        // ---- phase 1: scalars -> cs (log2 units), gamma, w
        if (tid < Q) {
            s_d[tid] = d_cur;
            s_l[tid] = l_cur;
        }
        if (tid == 0) {
            s_d[Q] = dn_cur;
            s_l[Q] = ln_cur;
        }
        float a = (tid < Q) ? d_cur * A_l2 : 0.0f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float v = __shfl_up_sync(0xffffffffu, a, o);
            if (lane >= o) a += v;
        }
        if (lane == 31) s_ws[warp] = a;
        // ---- phase 2a: per-segment angle sums
        constexpr int SEG = ROT ? kThreads / K : 1;
        constexpr int SEGLEN = ROT ? Q / SEG : 1;
        const int th_k = tid % K, th_sg = tid / K;
        const __nv_bfloat16* s_th = reinterpret_cast<const __nv_bfloat16*>(st + CF::ST_TH);
        // wait for this chunk's tiles
        wait_or_abort(&bar_full[s], (c / kStages) & 1);
        float th_acc = 0.0f;
        if (ROT) {
#pragma unroll 4
            for (int i = 0; i < SEGLEN; ++i) th_acc += __bfloat162float(s_th[(th_sg * SEGLEN + i) * K + th_k]);
            s_part[th_sg * K + th_k] = th_acc;
        }
        if (tid == 0) ptx::bulk_wait_read0();   // previous y store has left the staging tile
        __syncthreads();
        if (abort_s) { ok = false; break; }
        chunks_landed = c + 1;
        {
            float off = 0.0f;
            for (int w = 0; w < warp; ++w) off += s_ws[w];
            if (tid < Q) s_cs[tid] = a + off;
        }
        if (ROT) {
            // ---- phase 2b: cumulative angles Phi[t][k] (carry + prefix)
            float run = (float)s_carry[th_k];
            for (int sg = 0; sg < th_sg; ++sg) run += s_part[sg * K + th_k];
#pragma unroll 4
            for (int i = 0; i < SEGLEN; ++i) {
                const int t = th_sg * SEGLEN + i;
                run += __bfloat162float(s_th[t * K + th_k]);
                s_phi[t * K + th_k] = run;
            }
        }
        __syncthreads();
        if (tid < Q) {
            const float d = s_d[tid], l = s_l[tid];
            const float dn = s_d[tid + 1], ln = s_l[tid + 1];
            s_gam[tid] = l * d;
            s_w[tid] = l * d + (1.0f - ln) * dn;
        }
        __syncthreads();
        const float cs_end = s_cs[Q - 1];

        // ---- phase 3: rotate B, C; write C~ (in place), C~', B~ (in place), B~'
        {
            constexpr int CH = N / 8;                     // 16-byte chunks per row
            constexpr int ITEMS = ROWS * CH;
            uint8_t* sb = st + CF::ST_B;
            uint8_t* sc = st + CF::ST_C;
#pragma unroll 2
            for (int e = tid; e < ITEMS; e += kThreads) {
                const int row = e / CH, q8 = e % CH;
                const int t = row / R;
                const int slab = q8 >> 3, cc = q8 & 7;
                const uint32_t off = slab * TILE + row * 128 + ((cc ^ (row & 7)) << 4);
                uint4 vb = *reinterpret_cast<const uint4*>(sb + off);
                uint4 vc = *reinterpret_cast<const uint4*>(sc + off);
                const float cs_t = s_cs[t];
                const float sc_c = exp2f(cs_t);
                const float sc_b = exp2f(cs_end - cs_t) * s_w[t];
                uint32_t* pb = reinterpret_cast<uint32_t*>(&vb);
                uint32_t* pc = reinterpret_cast<uint32_t*>(&vc);
                uint4 ob, oc;
                uint32_t* qb = reinterpret_cast<uint32_t*>(&ob);
                uint32_t* qc = reinterpret_cast<uint32_t*>(&oc);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    float2 bb = unpack_bf16(pb[m]);
                    float2 cv = unpack_bf16(pc[m]);
                    if (ROT) {
                        const int k = q8 * 4 + m;
                        float sn, cn;
                        sincos_reduced(s_phi[t * K + k], &sn, &cn);
                        // Rot(-phi): (a, b) -> (a cos + b sin, -a sin + b cos)
                        const float b0 = bb.x * cn + bb.y * sn, b1 = bb.y * cn - bb.x * sn;
                        const float c0 = cv.x * cn + cv.y * sn, c1 = cv.y * cn - cv.x * sn;
                        bb = make_float2(b0, b1);
                        cv = make_float2(c0, c1);
                        pb[m] = pack_bf16(b0, b1);
                        pc[m] = pack_bf16(c0, c1);
                    }
                    qb[m] = pack_bf16(bb.x * sc_b, bb.y * sc_b);
                    qc[m] = pack_bf16(cv.x * sc_c, cv.y * sc_c);
                }
                if (ROT) {
                    *reinterpret_cast<uint4*>(sb + off) = vb;
                    *reinterpret_cast<uint4*>(sc + off) = vc;
                }
                *reinterpret_cast<uint4*>(t_bd + off) = ob;
                *reinterpret_cast<uint4*>(t_cd + off) = oc;
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();

        // ---- phase 4: S = C~ B~^T ; dG = B~'^T X ; Y = C~' G_{c-1}
        if (tid == 0) {
            ptx::tc_fence_after();
            const uint32_t a_c = ptx::smem_u32(st + CF::ST_C), a_b = ptx::smem_u32(st + CF::ST_B);
            const uint32_t a_x = ptx::smem_u32(st + CF::ST_X);
            const uint32_t a_bd = ptx::smem_u32(t_bd), a_cd = ptx::smem_u32(t_cd), a_g = ptx::smem_u32(t_g);
            constexpr uint32_t id_s = ptx::idesc_bf16(CF::M_S, ROWS, false, false);
            constexpr uint32_t id_g = ptx::idesc_bf16(CF::M_G, 64, true, true);
            constexpr uint32_t id_y = ptx::idesc_bf16(CF::M_S, 64, false, true);
#pragma unroll
            for (int k16 = 0; k16 < N / 16; ++k16) {   // K = N (state dim), K-major slabs
                const uint32_t ko = (k16 >> 2) * TILE + (k16 & 3) * 32;
                ptx::umma_bf16(tmem + CF::TM_S, ptx::sdesc_sw128(a_c + ko, 16, 1024),
                               ptx::sdesc_sw128(a_b + ko, 16, 1024), id_s, k16 > 0);
            }
#pragma unroll
            for (int k16 = 0; k16 < ROWS / 16; ++k16) {   // K = rows (j), MN-major operands
                ptx::umma_bf16(tmem + CF::TM_G, ptx::sdesc_sw128(a_bd + k16 * 2048, TILE, 1024),
                               ptx::sdesc_sw128(a_x + k16 * 2048, TILE, 1024), id_g, k16 > 0);
            }
            if (c > 0) {
#pragma unroll
                for (int k16 = 0; k16 < N / 16; ++k16) {   // K = N, A K-major, G MN-major [n][p]
                    const uint32_t ko = (k16 >> 2) * TILE + (k16 & 3) * 32;
                    ptx::umma_bf16(tmem + CF::TM_Y, ptx::sdesc_sw128(a_cd + ko, 16, 1024),
                                   ptx::sdesc_sw128(a_g + k16 * 2048, N * 128, 1024), id_y, k16 > 0);
                }
            }
            ptx::umma_commit(&bar_mma1);
        }
        __syncwarp();
        if (!ptx::mbar_wait(&bar_mma1, c & 1, kWaitBudget)) {
            m3::set_status(m3::kStatusWaitTimeout);
            abort_s = 1;
            mma_wait_failed |= 1;
            fail_parity = c & 1;
        }
        __syncwarp();
        ptx::tc_fence_after();

        // ---- phase 5a: S' = S o M -> bf16, K-major slabs of 64 columns (t_cd)
        {
            const int i = s_row;
            const int ti = (i >= 0) ? i / R : 0;
            const float cs_i = s_cs[ti], gam_i = s_gam[ti];
#pragma unroll
            for (int c32 = 0; c32 < ROWS / 32; ++c32) {
                uint32_t v[32];
                ptx::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + CF::TM_S + c32 * 32, v);
                ptx::tmem_ld_wait();
                if (i >= 0) {
#pragma unroll
                    for (int g8 = 0; g8 < 4; ++g8) {
                        uint32_t o[4];
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            float sv[2];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int j = c32 * 32 + g8 * 8 + m * 2 + u;
                                const int tj = j / R;
                                float mk;
                                if (tj > ti) mk = 0.0f;
                                else if (tj == ti) mk = gam_i;
                                else mk = exp2f(cs_i - s_cs[tj]) * s_w[tj];
                                sv[u] = __uint_as_float(v[g8 * 8 + m * 2 + u]) * mk;
                            }
                            o[m] = pack_bf16(sv[0], sv[1]);
                        }
                        const int j0 = c32 * 32 + g8 * 8;
                        const uint32_t off = (j0 >> 6) * TILE + i * 128 + ((((j0 & 63) >> 3) ^ (i & 7)) << 4);
                        *reinterpret_cast<uint4*>(t_cd + off) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
        }
        // ---- phase 5b: G = exp(cs_end) G + dG ; bf16 copy (MN-major [n][p]) for the next chunk
        {
            const float dec = exp2f(cs_end);
#pragma unroll
            for (int c32 = 0; c32 < 2; ++c32) {
                uint32_t v[32];
                ptx::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + CF::TM_G + c32 * 32, v);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int p = 0; p < 32; ++p) G[c32 * 32 + p] = fmaf(dec, G[c32 * 32 + p], __uint_as_float(v[p]));
            }
            if (g_row >= 0) {
#pragma unroll
                for (int g8 = 0; g8 < 8; ++g8) {
                    const uint32_t off = g_row * 128 + ((g8 ^ (g_row & 7)) << 4);
                    *reinterpret_cast<uint4*>(t_g + off) =
                        make_uint4(pack_bf16(G[g8 * 8 + 0], G[g8 * 8 + 1]), pack_bf16(G[g8 * 8 + 2], G[g8 * 8 + 3]),
                                   pack_bf16(G[g8 * 8 + 4], G[g8 * 8 + 5]), pack_bf16(G[g8 * 8 + 6], G[g8 * 8 + 7]));
                }
            }
        }
        // angle carry: Phi at the chunk's last token, reduced mod 2 pi (fp64)
        if (ROT && tid < K) {
            double acc = s_carry[tid];
            for (int sg = 0; sg < SEG; ++sg) acc += (double)s_part[sg * K + tid];
            acc -= 6.283185307179586 * rint(acc * (1.0 / 6.283185307179586));
            s_carry[tid] = acc;
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        if (abort_s) { ok = false; break; }

        // ---- phase 6: Y += S' X
        if (tid == 0) {
            ptx::tc_fence_after();
            const uint32_t a_sp = ptx::smem_u32(t_cd), a_x = ptx::smem_u32(st + CF::ST_X);
            constexpr uint32_t id_y = ptx::idesc_bf16(CF::M_S, 64, false, true);
#pragma unroll
            for (int k16 = 0; k16 < ROWS / 16; ++k16) {
                const uint32_t ko = (k16 >> 2) * TILE + (k16 & 3) * 32;
                ptx::umma_bf16(tmem + CF::TM_Y, ptx::sdesc_sw128(a_sp + ko, 16, 1024),
                               ptx::sdesc_sw128(a_x + k16 * 2048, TILE, 1024), id_y, (c > 0 || k16 > 0) ? 1u : 0u);
            }
            ptx::umma_commit(&bar_mma2);
        }
        __syncwarp();
        if (!ptx::mbar_wait(&bar_mma2, c & 1, kWaitBudget)) {
            m3::set_status(m3::kStatusWaitTimeout);
            abort_s = 1;
            mma_wait_failed |= 2;
            fail_parity = c & 1;
        }
        __syncwarp();
        ptx::tc_fence_after();

        // ---- phase 7: y tile -> bf16 staging (t_bd, 128B-swizzled rows) -> TMA store
        {
            const int i = s_row;
#pragma unroll
            for (int c32 = 0; c32 < 2; ++c32) {
                uint32_t v[32];
                ptx::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + CF::TM_Y + c32 * 32, v);
                ptx::tmem_ld_wait();
                if (i >= 0) {
#pragma unroll
                    for (int g8 = 0; g8 < 4; ++g8) {
                        const int q = c32 * 4 + g8;
                        const uint32_t off = i * 128 + ((q ^ (i & 7)) << 4);
                        *reinterpret_cast<uint4*>(t_bd + off) = make_uint4(
                            pack_bf16(__uint_as_float(v[g8 * 8 + 0]), __uint_as_float(v[g8 * 8 + 1])),
                            pack_bf16(__uint_as_float(v[g8 * 8 + 2]), __uint_as_float(v[g8 * 8 + 3])),
                            pack_bf16(__uint_as_float(v[g8 * 8 + 4]), __uint_as_float(v[g8 * 8 + 5])),
                            pack_bf16(__uint_as_float(v[g8 * 8 + 6]), __uint_as_float(v[g8 * 8 + 7])));
                    }
                }
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        if (abort_s) { ok = false; break; }
        if (tid == 0) {
            ptx::tma_store_5d(&map_y, t_bd, 0, 0, h, c * Q, b);
            ptx::bulk_commit();
            if (c + kStages < nch) {
                issue_loads(c + kStages);
                loads_issued = c + kStages + 1;
            }
        }
        d_cur = d_nx; l_cur = l_nx; dn_cur = dn_nx; ln_cur = ln_nx;
    }

    // ---- epilogue: final state = Rot(Phi_{T-1}) G (complex frame)
    if (ok && prm.final_state) {
        float cn = 1.0f, sn = 0.0f;
        if (ROT && g_row >= 0) {
            const float ang = (float)s_carry[g_row >> 1];
            sincosf(ang, &sn, &cn);
        }
        const bool even = g_row >= 0 && (g_row & 1) == 0;
        float* fs = prm.final_state + (((int64_t)b * prm.H + h) * N + (g_row >= 0 ? g_row : 0)) * 64;
#pragma unroll
        for (int p4 = 0; p4 < 16; ++p4) {
            float o[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float mine = G[p4 * 4 + u];
                const float other = ROT ? __shfl_xor_sync(0xffffffffu, mine, 1) : 0.0f;
                // rows (2k, 2k+1): (a, b) -> (a cos - b sin, a sin + b cos)
                o[u] = ROT ? (even ? cn * mine - sn * other : sn * other + cn * mine) : mine;
            }
            if (g_row >= 0) *reinterpret_cast<float4*>(fs + p4 * 4) = make_float4(o[0], o[1], o[2], o[3]);
        }
    }
    if (tid == 0) {
        ptx::bulk_wait0();
        if (!ok) {
            // stopped early: wait (bounded) for the copies and MMAs still in
            // flight before the shared memory and TMEM are released
            for (int cc = chunks_landed; cc < loads_issued; ++cc)
                (void)ptx::mbar_wait(&bar_full[cc % kStages], (cc / kStages) & 1, kWaitBudget);
        }
    }
    if (!ok && lane == 0 && warp == 0) {
        if (mma_wait_failed & 1) (void)ptx::mbar_wait(&bar_mma1, fail_parity, kWaitBudget);
        if (mma_wait_failed & 2) (void)ptx::mbar_wait(&bar_mma2, fail_parity, kWaitBudget);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, CF::TM_COLS);
}

// ----------------------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

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

// Tile rows per chunk the kernel uses for dims d (0 = unsupported).
inline int tile_rows(const m3_dims& d) {
    const int R = (int)d.rank;
    if (d.dtype != M3_BF16 || d.headdim != 64) return 0;
    if (d.dstate != 64 && d.dstate != 128) return 0;
    if (R != 1 && R != 2 && R != 4) return 0;
    if (d.heads > 65535 || d.seqlen > INT32_MAX / 2) return 0;
    const int rows = (int)d.chunk * R;
    if (d.dstate == 128) return 64;                 // shared-memory budget: 64-row tiles
    return rows <= 64 ? 64 : 128;
}

inline bool supports(const m3_dims& d) { return tile_rows(d) != 0; }

template <int ROWS, int NSLAB, int R, bool ROT>
int launch_cfg(const m3_dims& d, const CUtensorMap* maps, const Params& prm, cudaStream_t s) {
    using CF = Cfg<ROWS, NSLAB, R, ROT>;
    auto k = m3_scan_tc_kernel<ROWS, NSLAB, R, ROT>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_BYTES) != cudaSuccess)
        return M3_ERR_CUDA;
    k<<<(unsigned)(d.batch * d.heads), kThreads, CF::SMEM_BYTES, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4],
                                                                      prm);
    return cudaGetLastError() == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

template <int ROWS, int NSLAB, bool ROT>
int launch_r(const m3_dims& d, const CUtensorMap* maps, const Params& prm, cudaStream_t s) {
    switch (d.rank) {
        case 1: return launch_cfg<ROWS, NSLAB, 1, ROT>(d, maps, prm, s);
        case 2: return launch_cfg<ROWS, NSLAB, 2, ROT>(d, maps, prm, s);
        case 4: return launch_cfg<ROWS, NSLAB, 4, ROT>(d, maps, prm, s);
    }
    return M3_ERR_UNSUPPORTED;
}

// 5-D map over a [b, T, h, R, inner] bf16 tensor: box (64, R, 1, Q, 1), 128B swizzle.
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

// 4-D map over theta [b, T, h, K] bf16: box (K, 1, Q, 1), no swizzle.
inline bool make_map_theta(CUtensorMap* m, const void* base, const m3_dims& d, int Q) {
    const cuuint64_t K = (cuuint64_t)d.dstate / 2;
    cuuint64_t dims[4] = {K, (cuuint64_t)d.heads, (cuuint64_t)d.seqlen, (cuuint64_t)d.batch};
    cuuint64_t strides[3] = {K * 2, (cuuint64_t)d.heads * K * 2, (cuuint64_t)d.seqlen * d.heads * K * 2};
    cuuint32_t box[4] = {(cuuint32_t)K, 1, (cuuint32_t)Q, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int launch(const m3_dims& d, const void* x, const float* dt, const float* A, const void* B, const void* C,
                  const float* lam, const void* theta, void* y, float* final_state, cudaStream_t s) {
    const int rows = tile_rows(d);
    if (!rows) return M3_ERR_UNSUPPORTED;
    const void* tma_ptrs[] = {x, B, C, theta, y};
    for (const void* p : tma_ptrs)
        if (p && (reinterpret_cast<uintptr_t>(p) & 15u)) return M3_ERR_ALIGN;
    if (!encode_fn()) return M3_ERR_CUDA;
    const int Q = rows / (int)d.rank;
    CUtensorMap maps[5];
    memset(maps, 0, sizeof(maps));
    if (!make_map5(&maps[0], x, d, 64, Q) || !make_map5(&maps[1], B, d, (int)d.dstate, Q) ||
        !make_map5(&maps[2], C, d, (int)d.dstate, Q) || !make_map5(&maps[4], y, d, 64, Q))
        return M3_ERR_CUDA;
    const bool rot = theta != nullptr;
    if (rot && !make_map_theta(&maps[3], theta, d, Q)) return M3_ERR_CUDA;
    if (!rot) maps[3] = maps[0];
    Params prm;
    prm.T = d.seqlen;
    prm.H = (int)d.heads;
    prm.nchunks = (int)((d.seqlen + Q - 1) / Q);
    prm.dt = dt;
    prm.A = A;
    prm.lam = lam;
    prm.final_state = final_state;
    if (d.dstate == 64) {
        if (rows == 64) return rot ? launch_r<64, 1, true>(d, maps, prm, s) : launch_r<64, 1, false>(d, maps, prm, s);
        return rot ? launch_r<128, 1, true>(d, maps, prm, s) : launch_r<128, 1, false>(d, maps, prm, s);
    }
    return rot ? launch_r<64, 2, true>(d, maps, prm, s) : launch_r<64, 2, false>(d, maps, prm, s);
}

}  // namespace m3tc
