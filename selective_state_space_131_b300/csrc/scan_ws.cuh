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
//   warpgroup 0 (threads 0-127), chunk c+1: scalars (cs, gamma, w, scales),
//     cumulative angles, rotation of B and C in shared memory, the scaled copy
//     B~'; then thread 0 issues S and dG.
//   warpgroup 1 (threads 128-255), chunk c: mask S -> S', issue Y_inter and
//     Y_intra, G update, y epilogue + TMA store; thread 128 also issues every
//     TMA load (two stages ahead of warpgroup 0).
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

__host__ __device__ constexpr int align1k(int x) { return (x + 1023) & ~1023; }
__host__ __device__ constexpr int align16(int x) { return (x + 15) & ~15; }

template <int NSLAB, int R, bool ROT>
struct Cfg {
    static constexpr int Q = kRows / R;          // tokens per chunk
    static constexpr int N = 64 * NSLAB;         // state size
    static constexpr int K = N / 2;              // rotation pairs
    static constexpr int KG = N / 8;             // 16-byte groups per row (4 pairs each)
    static constexpr int NSEG = kWG / KG;        // token segments of the angle scan
    static constexpr int TPS = Q / NSEG;         // tokens per segment
    static constexpr int TB = 16 / R;            // tokens per 16-row mask block
    static constexpr int TILE = kRows * 128;     // one 64-column slab of a 64-row bf16 tile
    // stage (TMA destination): x | B slabs | C slabs | theta
    static constexpr int ST_X = 0;
    static constexpr int ST_B = ST_X + TILE;
    static constexpr int ST_C = ST_B + NSLAB * TILE;
    static constexpr int ST_TH = ST_C + NSLAB * TILE;
    static constexpr int TH_BYTES = ROT ? Q * K * 2 : 0;
    static constexpr int ST_BYTES = align1k(ST_TH + TH_BYTES);
    static constexpr uint32_t TX_BYTES = TILE * (1 + 2 * NSLAB) + TH_BYTES;
    static constexpr int OFF_BD = 2 * ST_BYTES;               // B~' (2 stages)
    static constexpr int OFF_SP = OFF_BD + 2 * NSLAB * TILE;  // S' (K-major)
    static constexpr int OFF_G = OFF_SP + TILE;               // G bf16 [N][P] (MN-major)
    static constexpr int OFF_Y = OFF_G + N * 128;             // y staging (TMA store source)
    static constexpr int OFF_SC = OFF_Y + TILE;               // per-stage scalars
    static constexpr int SC_CS = 0, SC_W = Q, SC_GAM = 2 * Q, SC_SCB = 3 * Q, SC_SCF = 4 * Q, SC_DEC = 5 * Q;
    static constexpr int SC_STRIDE = 5 * Q + 4;               // floats per stage
    static constexpr int OFF_DL = OFF_SC + 2 * SC_STRIDE * 4; // dt[Q+1], lambda[Q+1]
    static constexpr int OFF_WS = align16(OFF_DL + 2 * (Q + 1) * 4);  // warp sums [4]
    static constexpr int OFF_PART = OFF_WS + 16;              // angle partials [4 warps][KG][4]
    static constexpr int OFF_CARRY = align16(OFF_PART + 4 * KG * 16);  // double [K]
    static constexpr int SMEM_BYTES = OFF_CARRY + K * 8 + 1024;        // + alignment slack
    // TMEM columns: S / Y_intra double-buffered, dG, Y_inter
    static constexpr uint32_t TM_SY0 = 0, TM_DG = 128, TM_YI = 192, TM_COLS = 256;
    static_assert(NSEG * TPS == Q, "angle segments must tile the chunk");
    static_assert(Q % 32 == 0 || Q <= 32, "scalar scan");
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
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(v);
}
// sin / cos of x: one reduction to [-pi, pi] by a multiple of 2 pi, then the
// hardware sin / cos (absolute error ~1e-6 on that range).
__device__ __forceinline__ void sincos_reduced(float x, float* s, float* c) {
    const float n = rintf(x * (1.0f / kTwoPi));
    __sincosf(fmaf(-n, kTwoPi, x), s, c);
}
// Byte offset of the 16-byte group g of row `row` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int row, int g) {
    return (uint32_t)(row * 128 + (((g & 7) ^ (row & 7)) << 4) + (g >> 3) * (kRows * 128));
}

template <int NSLAB, int R, bool ROT>
__global__ void __launch_bounds__(kThreads, (NSLAB == 1 ? 2 : 1))
    m3_scan_ws_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_B,
                      const __grid_constant__ CUtensorMap map_C, const __grid_constant__ CUtensorMap map_th,
                      const __grid_constant__ CUtensorMap map_y, const Params prm) {
    using CF = Cfg<NSLAB, R, ROT>;
    constexpr int Q = CF::Q, N = CF::N, K = CF::K, KG = CF::KG, TPS = CF::TPS, TILE = CF::TILE;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t bar_full[2], bar_sd[2], bar_syfree[2], bar_dgfree, bar_yi, bar_y, bar_fin[2];
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
    float* s_d = reinterpret_cast<float*>(smem + CF::OFF_DL);
    float* s_l = s_d + (Q + 1);
    float* s_ws = reinterpret_cast<float*>(smem + CF::OFF_WS);
    float* s_part = reinterpret_cast<float*>(smem + CF::OFF_PART);
    double* s_carry = reinterpret_cast<double*>(smem + CF::OFF_CARRY);
    uint8_t* t_sp = smem + CF::OFF_SP;
    uint8_t* t_g = smem + CF::OFF_G;
    uint8_t* t_y = smem + CF::OFF_Y;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&bar_full[s], 1);
            ptx::mbar_init(&bar_sd[s], 1);
            ptx::mbar_init(&bar_syfree[s], 1);
            ptx::mbar_init(&bar_fin[s], 1);
        }
        ptx::mbar_init(&bar_dgfree, 1);
        ptx::mbar_init(&bar_yi, 1);
        ptx::mbar_init(&bar_y, 1);
        ptx::fence_mbar_init();
        abort_s = 0;
    }
    if (warp == 0) {
        ptx::tmem_alloc(&tmem_base_s, CF::TM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid < K) s_carry[tid] = 0.0;
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    // TMA loads of chunk c into stage c % 2 (issued by thread kWG only).
    auto issue_loads = [&](int c) {
        const int s = c & 1;
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
    int last_load[2] = {-1, -1};     // thread kWG only: last chunk loaded into each stage
    bool aborted = false;
    // fp32 chunk state G, rows owned by the consumer threads (M = 64 accumulator
    // layout for N = 64: row 16 w + lane % 16, columns 32 (lane / 16) + [0, 32);
    // M = 128 layout for N = 128: row 32 w + lane, all 64 columns)
    constexpr int GC = (N == 64) ? 32 : 64;
    float G[GC];
#pragma unroll
    for (int p = 0; p < GC; ++p) G[p] = 0.0f;

    if (tid < kWG) {
        // ======================= warpgroup 0: prologue + S / dG issue =======================
        const int kg = tid % KG, seg = tid / KG;
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

        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            uint8_t* st = smem + s * CF::ST_BYTES;
            float* sc = scal0 + s * CF::SC_STRIDE;
            float d_nx = 0.0f, l_nx = 1.0f, dn_nx = 0.0f, ln_nx = 1.0f;
            if (c + 1 < nch) load_scalars(c + 1, d_nx, l_nx, dn_nx, ln_nx);

            // (1) dt / lambda staging, warp scan of dt A (log2 units)
            if (tid < Q) { s_d[tid] = d_cur; s_l[tid] = l_cur; }
            if (tid == 0) { s_d[Q] = dn_cur; s_l[Q] = ln_cur; }
            float a = (tid < Q) ? d_cur * A_l2 : 0.0f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, a, o);
                if (lane >= o) a += v;
            }
            if (lane == 31) s_ws[warp] = a;
            // this chunk's tiles
            bool fail = !ptx::mbar_wait(&bar_full[s], (c >> 1) & 1, kWaitBudget);
            // angle partial sums of this thread's tokens for its 4 pairs
            float ph[4] = {0.0f, 0.0f, 0.0f, 0.0f}, own[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const __nv_bfloat16* s_th = reinterpret_cast<const __nv_bfloat16*>(st + CF::ST_TH);
            if (ROT) {   // unconditional: the shuffles below need the whole warp
#pragma unroll
                for (int i = 0; i < TPS; ++i) {
                    const uint2 raw = *reinterpret_cast<const uint2*>(s_th + (seg * TPS + i) * K + kg * 4);
                    const float2 t01 = unpack_bf16(raw.x), t23 = unpack_bf16(raw.y);
                    own[0] += t01.x; own[1] += t01.y; own[2] += t23.x; own[3] += t23.y;
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) ph[m] = own[m];
                // inclusive scan over the segments of this warp with the same kg
#pragma unroll
                for (int o = KG; o < 32; o <<= 1) {
                    float v[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) v[m] = __shfl_up_sync(0xffffffffu, ph[m], o);
                    if (lane >= o) {
#pragma unroll
                        for (int m = 0; m < 4; ++m) ph[m] += v[m];
                    }
                }
                if (lane >= 32 - KG) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) s_part[(warp * KG + kg) * 4 + m] = ph[m];
                }
            }
            if (fail) { m3::set_status(m3::kStatusWaitTimeout); abort_s = 1; }
            if (ptx::bar_sync_or(kBarWG0, kWG, fail || abort_s)) { aborted = true; break; }

            // (2) cs, gamma, w; angle at the start of this thread's segment
            float cs_t = 0.0f;
            if (tid < Q) {
                float off = 0.0f;
                for (int w = 0; w < warp; ++w) off += s_ws[w];
                cs_t = a + off;
                const float d = s_d[tid], l = s_l[tid], dn = s_d[tid + 1], ln = s_l[tid + 1];
                sc[CF::SC_CS + tid] = cs_t;
                sc[CF::SC_GAM + tid] = l * d;
                sc[CF::SC_W + tid] = l * d + (1.0f - ln) * dn;
            }
            float phi[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (ROT) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    // exclusive prefix: carry + earlier warps + earlier segments of this warp
                    float run = (float)s_carry[kg * 4 + m];
                    for (int w = 0; w < warp; ++w) run += s_part[(w * KG + kg) * 4 + m];
                    phi[m] = run + (ph[m] - own[m]);
                }
            }
            ptx::bar_sync(kBarWG0, kWG);

            // (3) per-token scales: B~' rows, factorised mask columns, chunk decay
            if (tid < Q) {
                const float cs_end = sc[CF::SC_CS + Q - 1];
                const int ref = (tid / CF::TB) * CF::TB + CF::TB - 1;
                const float w = sc[CF::SC_W + tid];
                sc[CF::SC_SCB + tid] = exp2f(cs_end - cs_t) * w;
                sc[CF::SC_SCF + tid] = exp2f(sc[CF::SC_CS + ref] - cs_t) * w;
                if (tid == 0) sc[CF::SC_DEC] = exp2f(cs_end);
            }
            ptx::bar_sync(kBarWG0, kWG);

            // (4) rotate B, C in place (B~, C~) and write B~' = scb * B~
            {
                uint8_t* sb = st + CF::ST_B;
                uint8_t* scc = st + CF::ST_C;
                uint8_t* bd = smem + CF::OFF_BD + s * NSLAB * TILE;
#pragma unroll
                for (int i = 0; i < TPS; ++i) {
                    const int t = seg * TPS + i;
                    float cn[4], sn[4];
                    if (ROT) {
                        const uint2 raw = *reinterpret_cast<const uint2*>(s_th + t * K + kg * 4);
                        const float2 t01 = unpack_bf16(raw.x), t23 = unpack_bf16(raw.y);
                        phi[0] += t01.x; phi[1] += t01.y; phi[2] += t23.x; phi[3] += t23.y;
#pragma unroll
                        for (int m = 0; m < 4; ++m) sincos_reduced(phi[m], &sn[m], &cn[m]);
                    }
                    const float scb = sc[CF::SC_SCB + t];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const int row = t * R + r;
                        const uint32_t off = swz(row, kg);
                        uint4 vb = *reinterpret_cast<const uint4*>(sb + off);
                        uint4 ob;
                        uint32_t* pb = reinterpret_cast<uint32_t*>(&vb);
                        uint32_t* qb = reinterpret_cast<uint32_t*>(&ob);
                        if (ROT) {
                            uint4 vc = *reinterpret_cast<const uint4*>(scc + off);
                            uint32_t* pc = reinterpret_cast<uint32_t*>(&vc);
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                // Rot(-phi): (a, b) -> (a cos + b sin, -a sin + b cos)
                                const float2 bb = unpack_bf16(pb[m]), cv = unpack_bf16(pc[m]);
                                const float b0 = bb.x * cn[m] + bb.y * sn[m], b1 = bb.y * cn[m] - bb.x * sn[m];
                                const float c0 = cv.x * cn[m] + cv.y * sn[m], c1 = cv.y * cn[m] - cv.x * sn[m];
                                pb[m] = pack_bf16(b0, b1);
                                pc[m] = pack_bf16(c0, c1);
                            }
                            *reinterpret_cast<uint4*>(sb + off) = vb;
                            *reinterpret_cast<uint4*>(scc + off) = vc;
                        }
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const float2 bb = unpack_bf16(pb[m]);
                            qb[m] = pack_bf16(bb.x * scb, bb.y * scb);
                        }
                        *reinterpret_cast<uint4*>(bd + off) = ob;
                    }
                }
                // angle carry at the chunk's last token, reduced mod 2 pi in fp64
                if (ROT && seg == CF::NSEG - 1) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        double v = (double)phi[m];
                        v -= 6.283185307179586 * rint(v * (1.0 / 6.283185307179586));
                        s_carry[kg * 4 + m] = v;
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            if (ptx::bar_sync_or(kBarWG0, kWG, abort_s)) { aborted = true; break; }

            // (5) thread 0: S = C~ B~^T -> TMEM S/Y[s];  dG = B~'^T X -> TMEM dG
            if (tid == 0) {
                bool ok = true;
                if (c >= 1) ok = ptx::mbar_wait(&bar_dgfree, (c - 1) & 1, kWaitBudget);
                if (ok && c >= 2) ok = ptx::mbar_wait(&bar_syfree[s], ((c >> 1) - 1) & 1, kWaitBudget);
                if (!ok) {
                    m3::set_status(m3::kStatusWaitTimeout);
                    abort_s = 1;
                } else {
                    ptx::tc_fence_after();
                    const uint32_t a_c = ptx::smem_u32(st + CF::ST_C), a_b = ptx::smem_u32(st + CF::ST_B);
                    const uint32_t a_x = ptx::smem_u32(st + CF::ST_X);
                    const uint32_t a_bd = ptx::smem_u32(smem + CF::OFF_BD + s * NSLAB * TILE);
                    constexpr uint32_t id_s = ptx::idesc_bf16(kRows, kRows, false, false);
                    constexpr uint32_t id_g = ptx::idesc_bf16(N, kP, true, true);
                    const uint32_t tm_s = tmem + CF::TM_SY0 + 64u * s;
#pragma unroll
                    for (int k16 = 0; k16 < N / 16; ++k16) {   // K = state (K-major slabs)
                        const uint32_t ko = (k16 >> 2) * TILE + (k16 & 3) * 32;
                        ptx::umma_bf16(tm_s, ptx::sdesc_sw128(a_c + ko, 16, 1024), ptx::sdesc_sw128(a_b + ko, 16, 1024),
                                       id_s, k16 > 0);
                    }
#pragma unroll
                    for (int k16 = 0; k16 < kRows / 16; ++k16) {   // K = rows (MN-major operands)
                        ptx::umma_bf16(tmem + CF::TM_DG, ptx::sdesc_sw128(a_bd + k16 * 2048, TILE, 1024),
                                       ptx::sdesc_sw128(a_x + k16 * 2048, TILE, 1024), id_g, k16 > 0);
                    }
                    ptx::umma_commit(&bar_sd[s]);
                }
            }
            d_cur = d_nx; l_cur = l_nx; dn_cur = dn_nx; ln_cur = ln_nx;
        }
    } else {
        // ======================= warpgroup 1: mask, state, output =======================
        const int w1 = warp - 4;
        const bool leader = (tid == kWG);
        const int i_row = w1 * 16 + (lane & 15);      // tile row of S / Y held by this thread
        const int hc = lane >> 4;                     // column half: [32 hc, 32 hc + 32)
        const int ti = i_row / R;                     // its token
        const uint32_t lane_base = (uint32_t)(w1 * 32) << 16;
        const int g_row = (N == 64) ? i_row : (w1 * 32 + lane);

        if (leader) {
            for (int c = 0; c < 2 && c < nch; ++c) {
                issue_loads(c);
                last_load[c] = c;
            }
        }
        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            uint8_t* st = smem + s * CF::ST_BYTES;
            const float* sc = scal0 + s * CF::SC_STRIDE;
            const uint32_t tm_sy = tmem + lane_base + CF::TM_SY0 + 64u * s;
            // (1) S_c and dG_c are in TMEM
            bool fail = !ptx::mbar_wait(&bar_sd[s], (c >> 1) & 1, kWaitBudget);
            ptx::tc_fence_after();
            if (leader && !fail && c > 0) {
                // Y_inter = C~ G_{c-1} (G: bf16 [N][P] rows, MN-major)
                const uint32_t a_c = ptx::smem_u32(st + CF::ST_C), a_g = ptx::smem_u32(t_g);
                constexpr uint32_t id_y = ptx::idesc_bf16(kRows, kP, false, true);
#pragma unroll
                for (int k16 = 0; k16 < N / 16; ++k16) {
                    const uint32_t ko = (k16 >> 2) * TILE + (k16 & 3) * 32;
                    ptx::umma_bf16(tmem + CF::TM_YI, ptx::sdesc_sw128(a_c + ko, 16, 1024),
                                   ptx::sdesc_sw128(a_g + k16 * 2048, N * 128, 1024), id_y, k16 > 0);
                }
                ptx::umma_commit(&bar_yi);
            }
            // (2) mask: S' = S o M for this thread's row and 32 columns
            const float cs_i = sc[CF::SC_CS + ti];
            {
                uint32_t v[32];
                ptx::tmem_ld16x2_32(tm_sy, v);
                ptx::tmem_ld_wait();
                const float gam_i = sc[CF::SC_GAM + ti];
                uint32_t o[16];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int J = hc * 2 + half;                   // 16-row block of these 16 columns
                    if (J < w1) {
                        const float u = exp2f(cs_i - sc[CF::SC_CS + J * CF::TB + CF::TB - 1]);
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 2) {
                            const int j = J * 16 + jj;
                            const float m0 = u * sc[CF::SC_SCF + j / R], m1 = u * sc[CF::SC_SCF + (j + 1) / R];
                            o[half * 8 + jj / 2] = pack_bf16(__uint_as_float(v[half * 16 + jj]) * m0,
                                                             __uint_as_float(v[half * 16 + jj + 1]) * m1);
                        }
                    } else if (J == w1) {
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 2) {
                            float mm[2];
#pragma unroll
                            for (int u2 = 0; u2 < 2; ++u2) {
                                const int tj = (J * 16 + jj + u2) / R;
                                mm[u2] = (tj < ti) ? exp2f(cs_i - sc[CF::SC_CS + tj]) * sc[CF::SC_W + tj]
                                                   : (tj == ti ? gam_i : 0.0f);
                            }
                            o[half * 8 + jj / 2] = pack_bf16(__uint_as_float(v[half * 16 + jj]) * mm[0],
                                                             __uint_as_float(v[half * 16 + jj + 1]) * mm[1]);
                        }
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) o[half * 8 + jj] = 0u;
                    }
                }
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    *reinterpret_cast<uint4*>(t_sp + swz(i_row, hc * 4 + g)) =
                        make_uint4(o[g * 4 + 0], o[g * 4 + 1], o[g * 4 + 2], o[g * 4 + 3]);
            }
            // (3) G_c = exp(cs_end) G_{c-1} + dG_c (fp32)
            {
                const float dec = sc[CF::SC_DEC];
                if constexpr (N == 64) {
                    uint32_t v[32];
                    ptx::tmem_ld16x2_32(tmem + lane_base + CF::TM_DG, v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int p = 0; p < 32; ++p) G[p] = fmaf(dec, G[p], __uint_as_float(v[p]));
                } else {
#pragma unroll
                    for (int c32 = 0; c32 < 2; ++c32) {
                        uint32_t v[32];
                        ptx::tmem_ld32(tmem + lane_base + CF::TM_DG + c32 * 32, v);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int p = 0; p < 32; ++p)
                            G[c32 * 32 + p] = fmaf(dec, G[c32 * 32 + p], __uint_as_float(v[p]));
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::fence_proxy_async_smem();
            if (leader) ptx::bulk_wait_read0();   // the previous y store has left the staging tile
            if (fail) { m3::set_status(m3::kStatusWaitTimeout); abort_s = 1; }
            if (ptx::bar_sync_or(kBarWG1, kWG, fail || abort_s)) { aborted = true; break; }
            if (leader) {
                ptx::tc_fence_after();
                ptx::mbar_arrive(&bar_dgfree);
                // Y_intra = S' X -> TMEM S/Y[s] (S has been read by every thread)
                const uint32_t a_sp = ptx::smem_u32(t_sp), a_x = ptx::smem_u32(st + CF::ST_X);
                constexpr uint32_t id_y = ptx::idesc_bf16(kRows, kP, false, true);
#pragma unroll
                for (int k16 = 0; k16 < kRows / 16; ++k16)
                    ptx::umma_bf16(tmem + CF::TM_SY0 + 64u * s, ptx::sdesc_sw128(a_sp + k16 * 32, 16, 1024),
                                   ptx::sdesc_sw128(a_x + k16 * 2048, TILE, 1024), id_y, k16 > 0);
                ptx::umma_commit(&bar_y);
            }
            // (4) G_{c-1} is no longer read: store the bf16 copy of G_c
            fail = false;
            if (c > 0) fail = !ptx::mbar_wait(&bar_yi, (c - 1) & 1, kWaitBudget);
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
            // (5) Y_intra done: stage s is free -> TMA of chunk c + 2
            if (!fail) fail = !ptx::mbar_wait(&bar_y, c & 1, kWaitBudget);
            ptx::tc_fence_after();
            if (leader && !fail && c + 2 < nch) {
                issue_loads(c + 2);
                last_load[s] = c + 2;
            }
            // (6) y = Y_intra + exp(cs) Y_inter -> bf16 staging -> TMA store
            {
                const float e = exp2f(cs_i);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t ya[16], yb[16];
                    ptx::tmem_ld16x2_16(tm_sy + q * 16, ya);
                    if (c > 0) ptx::tmem_ld16x2_16(tmem + lane_base + CF::TM_YI + q * 16, yb);
                    ptx::tmem_ld_wait();
                    float y[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        y[j] = (c > 0) ? fmaf(e, __uint_as_float(yb[j]), __uint_as_float(ya[j])) : __uint_as_float(ya[j]);
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
    if (!aborted && prm.final_state && tid >= kWG) {
        const int w1 = warp - 4;
        const int g_row = (N == 64) ? (w1 * 16 + (lane & 15)) : (w1 * 32 + lane);
        const int col0 = (N == 64) ? (lane >> 4) * 32 : 0;
        float cn = 1.0f, sn = 0.0f;
        if (ROT) sincosf((float)s_carry[g_row >> 1], &sn, &cn);
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
    if (aborted && tid == kWG) {
        // stopped early: wait (bounded) for the stores and loads still in flight
        ptx::bulk_wait0();
        for (int s = 0; s < 2; ++s)
            if (last_load[s] >= 0) (void)ptx::mbar_wait(&bar_full[s], (last_load[s] >> 1) & 1, kWaitBudget);
    }
    if (aborted && (tid == 0 || tid == kWG)) {
        // every MMA this thread issued has completed once this commit arrives
        const int wg = tid / kWG;
        ptx::umma_commit(&bar_fin[wg]);
        (void)ptx::mbar_wait(&bar_fin[wg], 0, kWaitBudget);
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

template <int NSLAB, int R, bool ROT>
int launch_cfg(const m3_dims& d, const CUtensorMap* maps, const Params& prm, cudaStream_t s) {
    using CF = Cfg<NSLAB, R, ROT>;
    auto k = m3_scan_ws_kernel<NSLAB, R, ROT>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_BYTES) != cudaSuccess)
        return M3_ERR_CUDA;
    k<<<(unsigned)(d.batch * d.heads), kThreads, CF::SMEM_BYTES, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4],
                                                                      prm);
    return cudaGetLastError() == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

template <int NSLAB, bool ROT>
int launch_r(const m3_dims& d, const CUtensorMap* maps, const Params& prm, cudaStream_t s) {
    switch (d.rank) {
        case 1: return launch_cfg<NSLAB, 1, ROT>(d, maps, prm, s);
        case 2: return launch_cfg<NSLAB, 2, ROT>(d, maps, prm, s);
        case 4: return launch_cfg<NSLAB, 4, ROT>(d, maps, prm, s);
    }
    return M3_ERR_UNSUPPORTED;
}

inline int launch(const m3_dims& d, const void* x, const float* dt, const float* A, const void* B, const void* C,
                  const float* lam, const void* theta, void* y, float* final_state, cudaStream_t s) {
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
    if (d.dstate == 64) return rot ? launch_r<1, true>(d, maps, prm, s) : launch_r<1, false>(d, maps, prm, s);
    return rot ? launch_r<2, true>(d, maps, prm, s) : launch_r<2, false>(d, maps, prm, s);
}

}  // namespace m3ws
