// scan_bwd_tc.cuh -- reverse pass of the backward (m3_scan_bwd) on the tensor
// cores for the tensor-core prefill's shapes with N = P = 64 (bf16, R in
// {1, 2, 4}, chunk R = 64 rows).  Pass 1 is the forward tensor-core kernel with
// its chunk checkpoints (scan_ws.cuh, CKPT); pass 3 is m3bwd::m3_bwd_dA_kernel.
//
// Per (b, h), chunks in reverse, the chunk backward of scan_bwd.cuh (rotated
// frame, 64-row tiles, i / j rows, n state, p head columns):
//   batch 1 (tcgen05, TMEM):  S = C~ B~^T,  dS' = dY X^T,  T2 = dY G^T,  XG = X dG^T
//   epilogue 1:  M, S' = S o M, dS = dS' o M (bf16 tiles), dM = dS' o S sums into
//                the token scalars; exp(cs) and s gradients from T2, XG
//   batch 2:     dX = S'^T dY + B~' dG,  dC~ = dS B~,  dB~ = dS^T C~,  dGu = C~'^T dY
//                (B~' = diag(s) B~, C~' = diag(exp(cs)) C~)
//   epilogue 2:  dx; dG_{c-1} = exp(cs_end) dG_c + dGu (fp32 registers, bf16 tile);
//                dC~ += diag(exp(cs)) T2, dB~ += diag(s) XG, rotated back by Phi;
//                dPhi per row and pair; dtheta as suffix sums; dt, lambda, A.
// Every operand is one 64 x 64 bf16 tile, 128-byte swizzled, stored [row][col]
// and read K-major or MN-major as the product needs (as in scan_ws.cuh).
// 256 threads: the two warpgroups read different accumulators in the
// epilogues; thread 32 issues the MMAs and the TMA loads, thread 0 the bulk
// copies of the checkpoints and the TMA stores of each chunk's dx, dB and dC
// tiles (staged in the S', dS and C~' buffers once the products that read them
// are done).  Waits are bounded: a wait that runs out sets the device status
// word, the stop is voted at the next barrier, and the CTA waits (bounded) for
// its work in flight.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx_sm100.cuh"
#include "scan_bwd.cuh"

namespace m3bwdtc {

constexpr int kThreads = 256;
constexpr int kT = 64;                      // tile rows / columns
constexpr int TILE = kT * 128;              // bytes of one 64 x 64 bf16 tile
constexpr long long kWaitBudget = 4000000000LL;
constexpr uint32_t kDescHi = ptx::sdesc_hi(1024, ptx::kSwz128);
constexpr uint32_t kIdKK = ptx::idesc_bf16(64, 64, false, false);
constexpr uint32_t kIdKM = ptx::idesc_bf16(64, 64, false, true);
constexpr uint32_t kIdMM = ptx::idesc_bf16(64, 64, true, true);

// shared memory (bytes, 1024-aligned tiles): per stage x | B | C | dY | theta
// ([Q][32] bf16, unswizzled), then the tiles of one chunk
constexpr int ST_X = 0, ST_B = TILE, ST_C = 2 * TILE, ST_DY = 3 * TILE, ST_TH = 4 * TILE;
constexpr int ST_BYTES = 4 * TILE + 4096;
constexpr int OFF_G = 2 * ST_BYTES;        // G_{c-1} bf16 [n][p]
constexpr int OFF_DG = OFF_G + TILE;       // dG_c bf16 [n][p]
constexpr int OFF_SP = OFF_DG + TILE;      // S' [i][j]
constexpr int OFF_DS = OFF_SP + TILE;      // dS [i][j]
constexpr int OFF_BD = OFF_DS + TILE;      // B~' [j][n]
constexpr int OFF_CD = OFF_BD + TILE;      // C~' [i][n]
constexpr int OFF_ZM = OFF_CD + TILE;      // fp32 [64][65]: dM o M below the diagonal blocks
constexpr int OFF_ZE = OFF_ZM + 64 * 65 * 4;   // fp32 [64][65]: dM o E (E = exp(cs_i - cs_j))
constexpr int OFF_F = OFF_ZE + 64 * 65 * 4;    // fp32 scratch, see below
// float offsets inside OFF_F
constexpr int F_CS = 0, F_GAM = 64, F_W = 128, F_S = 192, F_ECS = 256, F_EEND = 320;     // per token
// [row or token][pair] arrays use a row stride of KS = 33 floats: threads that walk
// rows at a fixed pair then hit distinct banks
constexpr int KS = 33;
constexpr int F_COS = 384, F_SIN = F_COS + 64 * KS;                                      // [Q][KS]
constexpr int F_RZM = F_SIN + 64 * KS, F_RG = F_RZM + 64, F_EBAR = F_RG + 64, F_DSR = F_EBAR + 64;   // per row
constexpr int F_DPR = F_DSR + 64;                                                        // [64 rows][KS]
constexpr int F_DL = F_DPR + 64 * KS;                                                    // [2][dt | lam][68]
constexpr int F_RED = F_DL + 2 * 2 * 68;                                                 // [8]: <dG, G> partials
constexpr int F_PEND = F_RED + 8;                                                        // ddt, dlam, dA
constexpr int F_DPHI = F_PEND + 4;                                                       // [32] dtheta suffix carry
constexpr int F_PHI0 = F_DPHI + 32;                                                      // [32] angle at chunk start
constexpr int F_DTOK = F_PHI0 + 32;                                                      // [2][64] ddt, dlam of the chunk
constexpr int F_CZM = F_DTOK + 128, F_CZE = F_CZM + 64;                                  // per column
constexpr int F_SEG = F_CZE + 64;                                                        // [4][32] segment totals
constexpr int F_DSD = F_SEG + 128;                                                       // [64][4] dS, same-token block
constexpr int F_END = F_DSD + 256;
constexpr int OFF_GB = (OFF_F + F_END * 4 + 1023) & ~1023;   // fp32 G checkpoint, 2 stages x [64][64]
constexpr int OFF_DTH = OFF_GB + 2 * 64 * 64 * 4;   // bf16 [64 tokens][32 pairs]: dtheta staging
constexpr int SMEM_BYTES = OFF_DTH + 64 * 32 * 2 + 1024;
// TMEM columns
constexpr uint32_t TM_S = 0, TM_DSP = 64, TM_T2 = 128, TM_XG = 192, TM_DX = 256, TM_DC = 320, TM_DB = 384,
                   TM_DGU = 448, TM_COLS = 512;

struct Params {
    int64_t T;
    int H, nch;
    const float* dt;
    const float* A;
    const float* lam;
    const __nv_bfloat16* theta;
    const float* dfinal;
    const float* ck_G;
    const float* ck_phi;
    float* dA_part;
    __nv_bfloat16* dx;
    float* ddt;
    __nv_bfloat16* dB;
    __nv_bfloat16* dC;
    float* dlam;
    __nv_bfloat16* dtheta;
};

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float lo16(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float hi16(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t swz(int row, int g) {   // 16-byte group g of a row, 128-byte swizzle
    return (uint32_t)(row * 128 + (((g & 7) ^ (row & 7)) << 4));
}
// 32 consecutive columns [32 hc, 32 hc + 32) of row `row` of a tile as floats
__device__ __forceinline__ void tile_row32(const uint8_t* t, int row, int hc, float (&o)[32]) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint4 v = *reinterpret_cast<const uint4*>(t + swz(row, 4 * hc + g));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            o[8 * g + 2 * m] = lo16(u[m]);
            o[8 * g + 2 * m + 1] = hi16(u[m]);
        }
    }
}
// the 8 columns of 16-byte group gg of row `row` of a tile as floats
__device__ __forceinline__ void tile_row8(const uint8_t* t, int row, int gg, float (&o)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(t + swz(row, gg));
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        o[2 * m] = lo16(u[m]);
        o[2 * m + 1] = hi16(u[m]);
    }
}
// 16 columns: 16-byte groups gg, gg + 1 of row `row`
__device__ __forceinline__ void tile_put16(uint8_t* t, int row, int gg, const float (&v)[16]) {
#pragma unroll
    for (int g = 0; g < 2; ++g)
        *reinterpret_cast<uint4*>(t + swz(row, gg + g)) =
            make_uint4(pack2(v[8 * g], v[8 * g + 1]), pack2(v[8 * g + 2], v[8 * g + 3]),
                       pack2(v[8 * g + 4], v[8 * g + 5]), pack2(v[8 * g + 6], v[8 * g + 7]));
}
__device__ __forceinline__ void tile_put32(uint8_t* t, int row, int hc, const float (&v)[32]) {
#pragma unroll
    for (int g = 0; g < 4; ++g)
        *reinterpret_cast<uint4*>(t + swz(row, 4 * hc + g)) =
            make_uint4(pack2(v[8 * g], v[8 * g + 1]), pack2(v[8 * g + 2], v[8 * g + 3]),
                       pack2(v[8 * g + 4], v[8 * g + 5]), pack2(v[8 * g + 6], v[8 * g + 7]));
}
// x - n 2 pi (two-constant reduction), as in scan_ws.cuh
__device__ __forceinline__ float red2pi(float x) {
    const float n = rintf(x * 0.15915494309189535f);
    return fmaf(-n, 1.9353071795864769e-3f, fmaf(-n, 6.28125f, x));
}

template <int R>
__global__ void __launch_bounds__(kThreads, 1)
    m3_bwd_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_B,
                     const __grid_constant__ CUtensorMap map_C, const __grid_constant__ CUtensorMap map_dy,
                     const __grid_constant__ CUtensorMap map_th, const __grid_constant__ CUtensorMap map_dx,
                     const __grid_constant__ CUtensorMap map_dB, const __grid_constant__ CUtensorMap map_dC,
                     const __grid_constant__ CUtensorMap map_dth, const Params prm) {
    constexpr int Q = kT / R;      // tokens per chunk
    constexpr int K = 32;          // rotation pairs (N = 64)
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t bar_ld[2], bar_ck[2], bar_m1, bar_m2, bar_fin;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;
    if (blockDim.x != kThreads) {
        if (threadIdx.x == 0) m3::set_status(m3::kStatusBadLaunch);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wg = warp >> 2, wq = warp & 3;
    const int unit = blockIdx.x;
    const int h = unit % prm.H, b = unit / prm.H;
    const int64_t T = prm.T;
    const int nch = prm.nch;
    const float A_h = __ldg(prm.A + h);
    const float A_l2 = A_h * m3::kLog2e;
    // accumulator row / column half owned by this thread in the epilogues
    const int row = wq * 16 + (lane & 15);
    const int hc = lane >> 4;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    float* F = reinterpret_cast<float*>(smem + OFF_F);
    float* zm = reinterpret_cast<float*>(smem + OFF_ZM);
    float* ze = reinterpret_cast<float*>(smem + OFF_ZE);
    auto tok_idx = [&](int64_t t) { return ((int64_t)b * T + t) * prm.H + h; };

    if (tid == 0) {
        ptx::mbar_init(&bar_ld[0], 1);
        ptx::mbar_init(&bar_ld[1], 1);
        ptx::mbar_init(&bar_ck[0], 1);
        ptx::mbar_init(&bar_ck[1], 1);
        ptx::mbar_init(&bar_m1, 1);
        ptx::mbar_init(&bar_m2, 1);
        ptx::mbar_init(&bar_fin, 1);
        ptx::fence_mbar_init();
        abort_s = 0;
    }
    if (warp == 0) {
        ptx::tmem_alloc(&tmem_base_s, TM_COLS);
        ptx::tmem_relinquish();
    }
    // TMA loads of chunk c into stage st (thread 32 only); dt / lambda of chunk c's
    // tokens and the one after (zero / one past the end) by warp 2 with cp.async
    int ld_count[2] = {0, 0};   // thread 32: loads issued per stage
    auto issue_loads = [&](int c, int st) {
        ++ld_count[st];
        uint8_t* base = smem + st * ST_BYTES;
        const int t0 = c * Q;
        const bool rot = prm.theta != nullptr;
        ptx::mbar_arrive_expect_tx(&bar_ld[st], 4 * TILE + (rot ? Q * K * 2 : 0));
        ptx::tma_load_5d(base + ST_X, &map_x, &bar_ld[st], 0, 0, h, t0, b);
        ptx::tma_load_5d(base + ST_B, &map_B, &bar_ld[st], 0, 0, h, t0, b);
        ptx::tma_load_5d(base + ST_C, &map_C, &bar_ld[st], 0, 0, h, t0, b);
        ptx::tma_load_5d(base + ST_DY, &map_dy, &bar_ld[st], 0, 0, h, t0, b);
        if (rot) ptx::tma_load_4d(base + ST_TH, &map_th, &bar_ld[st], 0, h, t0, b);
    };
    // thread 0: checkpoint slot c (the fp32 64 x 64 state, 16 KB, contiguous) into
    // stage st of the fp32 buffer with one bulk copy (one instruction instead of a
    // 16-byte copy per thread and vector)
    int ck_count[2] = {0, 0};   // thread 0: copies issued per stage
    auto issue_ckpt = [&](int c, int st) {
        ++ck_count[st];
        ptx::mbar_arrive_expect_tx(&bar_ck[st], 64 * 64 * 4);
        ptx::bulk_g2s(smem + OFF_GB + st * 16384, prm.ck_G + ((int64_t)unit * (prm.nch + 1) + c) * 64 * 64,
                      64 * 64 * 4, &bar_ck[st]);
    };
    // warpgroup 0 (idle while warpgroup 1 runs the mask's column sums and the token
    // scalars): dtheta of chunk cc from its rows' dPhi (F_DPR), suffix sums over the
    // 64 rows in four segments of 16 (warp = segment, lane = pair), carried from the
    // chunks after it; the sum at a token's first row is that token's dtheta
    auto dtheta_chunk = [&](int cc) {
        const int seg = warp;
        constexpr int RS = 16;
        const int64_t tc0 = (int64_t)cc * Q;
        __nv_bfloat16* dth = reinterpret_cast<__nv_bfloat16*>(smem + OFF_DTH);   // [token][pair]
        // the previous chunk's dtheta store has read the staging tile before the
        // barrier below lets any thread write it
        if (tid == 0) ptx::bulk_wait_read0();
        float v[RS];
        float tot = 0.0f;
#pragma unroll
        for (int q = 0; q < RS; ++q) {
            v[q] = F[F_DPR + (seg * RS + q) * KS + lane];
            tot += v[q];
        }
        F[F_SEG + seg * 32 + lane] = tot;
        ptx::bar_sync(3, 128);
        float acc = F[F_DPHI + lane];
        for (int s2 = seg + 1; s2 < 4; ++s2) acc += F[F_SEG + s2 * 32 + lane];
#pragma unroll
        for (int q = RS - 1; q >= 0; --q) {
            const int rw = seg * RS + q;
            acc += v[q];
            if (rw % R == 0) dth[(rw / R) * K + lane] = __float2bfloat16_rn(acc);   // past T: clipped
        }
        ptx::fence_proxy_async_smem();
        ptx::bar_sync(3, 128);   // every thread has read F_DPHI and written its dtheta
        if (seg == 0) F[F_DPHI + lane] = acc;
        if (tid == 0) {
            // the chunk's dtheta [Q tokens][32 pairs] in one TMA store
            ptx::tma_store_4d(&map_dth, dth, 0, h, (int)tc0, b);
            ptx::bulk_commit();
        }
    };
    auto issue_scalars = [&](int c, int st) {
        float* dst = F + F_DL + st * 2 * 68;
        for (int tt = lane; tt <= Q; tt += 32) {
            const int64_t t = (int64_t)c * Q + tt;
            const bool ok = t < T;
            const int64_t idx = ok ? tok_idx(t) : 0;
            ptx::cp_async4(dst + tt, prm.dt + idx, ok);
            if (prm.lam) ptx::cp_async4(dst + 68 + tt, prm.lam + idx, ok);
        }
        ptx::cp_async_commit();
    };

    // dG_last = Rot(-Phi_{T-1}) dfinal, held in fp32 by warpgroup 0 (rows n =
    // `row`, columns 32 hc ..); the final rotation's angle gradient
    // sum_p (-df_0 f_1 + df_1 f_0), f = Rot(Phi) G_last, starts the dtheta carry.  Here
    // its part through G_{nch-1} (f = Rot(Phi) G_{nch-1}); the last chunk decays it and
    // adds the part through its own rows
    float dG[32];
    const int64_t ckb = (int64_t)unit * (nch + 1);
    if (tid < 32) F[F_DPHI + tid] = 0.0f;
    if (tid == 0) { F[F_PEND] = 0.0f; F[F_PEND + 1] = 0.0f; F[F_PEND + 2] = 0.0f; }
    __syncthreads();
    if (wg == 0) {
        const int k = row >> 1;
        const bool even = (row & 1) == 0;
        float sn = 0.0f, cn = 1.0f;
        if (prm.theta) __sincosf(red2pi(__ldg(prm.ck_phi + ckb * K + (int64_t)nch * K + k)), &sn, &cn);
        float dphi = 0.0f;
#pragma unroll
        for (int p = 0; p < 32; ++p) {
            const float df = prm.dfinal ? __ldg(prm.dfinal + ((int64_t)unit * 64 + row) * 64 + 32 * hc + p) : 0.0f;
            const float dfo = __shfl_xor_sync(0xffffffffu, df, 1);   // the pair partner's row
            const float g = __ldg(prm.ck_G + ((ckb + nch - 1) * 64 + row) * 64 + 32 * hc + p);
            const float go = __shfl_xor_sync(0xffffffffu, g, 1);
            // Rot(-phi) (df0, df1) = (df0 c + df1 s, -df0 s + df1 c)
            dG[p] = even ? fmaf(df, cn, dfo * sn) : fmaf(-dfo, sn, df * cn);
            if (even) {
                const float f0 = fmaf(g, cn, -go * sn), f1 = fmaf(g, sn, go * cn);
                dphi = fmaf(-df, f1, fmaf(dfo, f0, dphi));
            }
        }
        // sum the 64 columns of pair k: the two column halves (lanes l, l ^ 16)
        dphi += __shfl_xor_sync(0xffffffffu, dphi, 16);
        if (even && hc == 0 && prm.theta && prm.dfinal) F[F_DPHI + k] = dphi;
        tile_put32(smem + OFF_DG, row, hc, dG);
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    if (tid == 32) issue_loads(nch - 1, (nch - 1) & 1);
    if (warp == 7) issue_scalars(nch - 1, (nch - 1) & 1);
    if (tid == 0) issue_ckpt(nch - 1, (nch - 1) & 1);
    bool fail = false;
    float dA_acc = 0.0f;

    for (int c = nch - 1; c >= 0 && !fail; --c) {
        const int st = c & 1;
        uint8_t* sbase = smem + st * ST_BYTES;
        const int64_t t0 = (int64_t)c * Q;
        const int nt = (int)((T - t0) < Q ? (T - t0) : Q);
        // the next chunk (in reverse) into the other stage, free since the
        // previous iteration's batch 2 completed
        if (c > 0 && tid == 32) issue_loads(c - 1, st ^ 1);
        if (c > 0 && tid == 0) issue_ckpt(c - 1, st ^ 1);   // its stage was read last iteration
        // ---- (1) checkpoint G_{c-1} (warpgroup 0: fp32 slice for <dG, G>, bf16 tile;
        //      the next chunk's slice prefetched); dt / lambda (warp 7)
        if (wg == 0) {
            // slot c (copied during the chunk before)
            if (!ptx::mbar_wait(&bar_ck[st], ((nch - 1 - c) >> 1) & 1, kWaitBudget)) {
                m3::set_status(m3::kStatusWaitTimeout);
                abort_s = 1;
            }
            float gsl[32];
            const float* src = reinterpret_cast<const float*>(smem + OFF_GB) + st * 4096 + row * 64 + 32 * hc;
#pragma unroll
            for (int p4 = 0; p4 < 8; ++p4) {
                const float4 v = *reinterpret_cast<const float4*>(src + 4 * p4);
                gsl[4 * p4] = v.x; gsl[4 * p4 + 1] = v.y; gsl[4 * p4 + 2] = v.z; gsl[4 * p4 + 3] = v.w;
            }
            tile_put32(smem + OFF_G, row, hc, gsl);
            float part = 0.0f;
#pragma unroll
            for (int p = 0; p < 32; ++p) part = fmaf(dG[p], gsl[p], part);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (lane == 0) F[F_RED + wq] = part;
        }
        if (warp == 7) {
            ptx::cp_async_wait_all();   // this chunk's dt / lambda
            __syncwarp();
            if (c > 0) issue_scalars(c - 1, st ^ 1);
        }
        float phi0 = 0.0f;   // warpgroup 1: the angle of pair `lane` before the chunk
        if (wg == 1 && prm.theta) phi0 = __ldg(prm.ck_phi + (ckb + c) * K + lane);
        ptx::fence_proxy_async_smem();   // the G tile, for the MMAs below
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
        if (tid == 32) {
            // the products that need neither the rotation nor the mask, as soon as the
            // tiles are in: dS' = dY X^T, T2 = dY G^T, XG = X dG^T
            if (!ptx::mbar_wait(&bar_ld[st], ((nch - 1 - c) >> 1) & 1, kWaitBudget)) {
                m3::set_status(m3::kStatusWaitTimeout);
                abort_s = 1;
            } else {
                ptx::tc_fence_after();
                const uint32_t x_lo = ptx::sdesc_lo(ptx::smem_u32(sbase + ST_X), 16);
                const uint32_t y_lo = ptx::sdesc_lo(ptx::smem_u32(sbase + ST_DY), 16);
                const uint32_t g_lo = ptx::sdesc_lo(ptx::smem_u32(smem + OFF_G), 16);
                const uint32_t d_lo = ptx::sdesc_lo(ptx::smem_u32(smem + OFF_DG), 16);
#pragma unroll
                for (int k = 0; k < 4; ++k) {   // K-major operands: 16 columns = +32 bytes
                    ptx::umma_bf16_lo<kDescHi, kDescHi>(tmem + TM_DSP, y_lo + 2 * k, x_lo + 2 * k, kIdKK, k > 0);
                    ptx::umma_bf16_lo<kDescHi, kDescHi>(tmem + TM_T2, y_lo + 2 * k, g_lo + 2 * k, kIdKK, k > 0);
                    ptx::umma_bf16_lo<kDescHi, kDescHi>(tmem + TM_XG, x_lo + 2 * k, d_lo + 2 * k, kIdKK, k > 0);
                }
            }
        }
        __syncwarp();   // warp 1 reconverges before its other lanes wait: a lane parked in
                        // mbarrier.try_wait can hold back the issuing lane of its warp
        if (warp == 0) {
            // chunk-local cs (log2 units), gamma, w, s = 2^(cs_end - cs) w, exp(cs)
            const float* sdt = F + F_DL + st * 2 * 68;
            const float* slm = sdt + 68;
            float dcur[2], lcur[2], dn[2], ln[2], cs[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = u * 32 + lane;
                const bool in = t < Q;
                dcur[u] = in ? sdt[t] : 0.0f;
                dn[u] = in ? sdt[t + 1] : 0.0f;
                lcur[u] = (in && prm.lam) ? slm[t] : 1.0f;
                ln[u] = (in && prm.lam) ? slm[t + 1] : 1.0f;
                float a = dcur[u] * A_l2;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float v = __shfl_up_sync(0xffffffffu, a, o);
                    if (lane >= o) a += v;
                }
                cs[u] = a;
            }
            cs[1] += __shfl_sync(0xffffffffu, cs[0], 31);
            // cs_end is the last valid token's cs, and past it (dt = 0) cs repeats that
            // value bit for bit, so that 2^(cs_end - cs) is exactly 1 for the last token
            const int lt = nt - 1;   // uniform over the warp
            const float cs_end = __shfl_sync(0xffffffffu, (lt < 32) ? cs[0] : cs[1], lt & 31);
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (u * 32 + lane > lt) cs[u] = cs_end;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = u * 32 + lane;
                if (t < Q) {
                    const float gam = lcur[u] * dcur[u];
                    const float w = gam + (1.0f - ln[u]) * dn[u];
                    F[F_CS + t] = cs[u];
                    F[F_GAM + t] = gam;
                    F[F_W + t] = w;
                    F[F_EEND + t] = m3::ex2_approx(cs_end - cs[u]);
                    F[F_S + t] = m3::ex2_approx(cs_end - cs[u]) * w;
                    F[F_ECS + t] = m3::ex2_approx(cs[u]);
                }
            }
        }
        if (wg == 1 && prm.theta) {
            // the cumulative angle of every token and pair: 4 segments of Q / 4 tokens
            // per pair (warp 4 + seg), fp32 from the checkpointed angle at the chunk start
            const int seg = warp - 4;
            constexpr int QS = Q / 4;
            bool ok = ptx::mbar_wait(&bar_ld[st], ((nch - 1 - c) >> 1) & 1, kWaitBudget);
            if (!ok) { m3::set_status(m3::kStatusWaitTimeout); abort_s = 1; }
            const __nv_bfloat16* th = reinterpret_cast<const __nv_bfloat16*>(sbase + ST_TH);
            float loc[QS];
            float run = 0.0f;
#pragma unroll
            for (int q = 0; q < QS; ++q) {
                run += __bfloat162float(th[(seg * QS + q) * K + lane]);
                loc[q] = run;
            }
            F[F_SEG + seg * 32 + lane] = run;
            ptx::bar_sync(1, 128);
            float off = phi0;
            for (int s2 = 0; s2 < seg; ++s2) off += F[F_SEG + s2 * 32 + lane];
            off = red2pi(off);
#pragma unroll
            for (int q = 0; q < QS; ++q) {
                float sn, co;
                __sincosf(red2pi(off + loc[q]), &sn, &co);
                F[F_COS + (seg * QS + q) * KS + lane] = co;
                F[F_SIN + (seg * QS + q) * KS + lane] = sn;
            }
        }
        // ---- (2) the tiles are in; rotate B, C in place (B~, C~) and write B~' and C~'
        //      (the previous chunk's gradient stores have read the C~', S' and dS tiles)
        if (!ptx::mbar_wait(&bar_ld[st], ((nch - 1 - c) >> 1) & 1, kWaitBudget)) {
            m3::set_status(m3::kStatusWaitTimeout);
            abort_s = 1;
        }
        if (tid == 0) ptx::bulk_wait_read0();
        __syncthreads();
        if (abort_s) { fail = true; break; }
        {
            const int r2 = tid >> 2, qq = tid & 3;     // row, quarter: 16 columns = 8 pairs
            const int t = r2 / R;
            uint8_t* tb = sbase + ST_B;
            uint8_t* tc = sbase + ST_C;
            const float sj = F[F_S + t], ei = F[F_ECS + t];
#pragma unroll
            for (int g2 = 0; g2 < 2; ++g2) {
                const int g = 2 * qq + g2;
                const uint32_t off = swz(r2, g);
                uint4 vb = *reinterpret_cast<const uint4*>(tb + off);
                uint4 vc = *reinterpret_cast<const uint4*>(tc + off);
                uint32_t* pb = reinterpret_cast<uint32_t*>(&vb);
                uint32_t* pc = reinterpret_cast<uint32_t*>(&vc);
                uint32_t ob[4], oc[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    // the B and C pairs side by side in packed fp32: u = (a_B, a_C), v = (b_B, b_C)
                    float2 u = make_float2(lo16(pb[m]), lo16(pc[m])), v = make_float2(hi16(pb[m]), hi16(pc[m]));
                    if (prm.theta) {
                        const int k = g * 4 + m;
                        const float co = F[F_COS + t * KS + k], si = F[F_SIN + t * KS + k];
                        // Rot(-phi): (a, b) -> (a cos + b sin, -a sin + b cos)
                        const float2 co2 = make_float2(co, co), si2 = make_float2(si, si), nsi2 = make_float2(-si, -si);
                        const float2 nu = __ffma2_rn(u, co2, __fmul2_rn(v, si2));
                        const float2 nv = __ffma2_rn(u, nsi2, __fmul2_rn(v, co2));
                        u = nu;
                        v = nv;
                    }
                    pb[m] = pack2(u.x, v.x);
                    pc[m] = pack2(u.y, v.y);
                    // scaled copies from the rounded values the MMAs see
                    const float2 sb = __fmul2_rn(make_float2(lo16(pb[m]), hi16(pb[m])), make_float2(sj, sj));
                    const float2 scl = __fmul2_rn(make_float2(lo16(pc[m]), hi16(pc[m])), make_float2(ei, ei));
                    ob[m] = pack2(sb.x, sb.y);
                    oc[m] = pack2(scl.x, scl.y);
                }
                *reinterpret_cast<uint4*>(tb + off) = vb;
                *reinterpret_cast<uint4*>(tc + off) = vc;
                *reinterpret_cast<uint4*>(smem + OFF_BD + off) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
                *reinterpret_cast<uint4*>(smem + OFF_CD + off) = make_uint4(oc[0], oc[1], oc[2], oc[3]);
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
        // ---- (3) S = C~ B~^T (commit: epilogue 1 waits for it and the products before
        //      it); then dGu = C~'^T dY and dX := B~' dG, which need no mask
        if (tid == 32) {
            const uint32_t b_lo = ptx::sdesc_lo(ptx::smem_u32(sbase + ST_B), 16);
            const uint32_t c_lo = ptx::sdesc_lo(ptx::smem_u32(sbase + ST_C), 16);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                ptx::umma_bf16_lo<kDescHi, kDescHi>(tmem + TM_S, c_lo + 2 * k, b_lo + 2 * k, kIdKK, k > 0);
            ptx::umma_commit(&bar_m1);
            const uint32_t y_mn = ptx::sdesc_lo(ptx::smem_u32(sbase + ST_DY), TILE);
            const uint32_t bd_k = ptx::sdesc_lo(ptx::smem_u32(smem + OFF_BD), 16);
            const uint32_t dg_mn = ptx::sdesc_lo(ptx::smem_u32(smem + OFF_DG), TILE);
            const uint32_t cd_mn = ptx::sdesc_lo(ptx::smem_u32(smem + OFF_CD), TILE);
#pragma unroll
            for (int k = 0; k < 4; ++k) {   // MN-major operands: 16 K rows = +2048 bytes
                ptx::umma_bf16_lo<kDescHi, kDescHi>(tmem + TM_DGU, cd_mn + 128 * k, y_mn + 128 * k, kIdMM, k > 0);
                ptx::umma_bf16_lo<kDescHi, kDescHi>(tmem + TM_DX, bd_k + 2 * k, dg_mn + 128 * k, kIdKM, k > 0);
            }
        }
        __syncwarp();
        if (!ptx::mbar_wait(&bar_m1, (nch - 1 - c) & 1, kWaitBudget)) {
            m3::set_status(m3::kStatusWaitTimeout);
            abort_s = 1;
        }
        __syncwarp();
        ptx::tc_fence_after();
        // ---- (4) epilogue 1
        float eT[32];     // warpgroup 1: exp(cs_i) T2 (row i) or s_j XG (row j), kept for (6)
        float sX[32];
        if (wg == 0) {
            // S, dS' of row i, columns 32 hc ..: mask, S', dS, dM -- in two halves of 16
            // columns, to keep the registers in bounds
            const int ti = row / R;
            const float cs_i = F[F_CS + ti], gam_i = F[F_GAM + ti];
            float rzm = 0.0f, rg = 0.0f;
            float dsd[R];   // dS of the same-token block (selected, no dynamic register index)
#pragma unroll
            for (int r = 0; r < R; ++r) dsd[r] = 0.0f;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t vs[16], vd[16];
                ptx::tmem_ld16x2_16(tmem + lane_base + TM_S + 16 * half, vs);
                ptx::tmem_ld16x2_16(tmem + lane_base + TM_DSP + 16 * half, vd);
                ptx::tmem_ld_wait();
                float sp[16], ds[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int j = 32 * hc + 16 * half + e, tj = j / R;
                    const float S = __uint_as_float(vs[e]), dSp = __uint_as_float(vd[e]);
                    float m = 0.0f, ez = 0.0f;
                    if (tj < ti) {
                        ez = m3::ex2_approx(cs_i - F[F_CS + tj]);
                        m = ez * F[F_W + tj];
                    } else if (tj == ti) {
                        m = gam_i;
                    }
                    sp[e] = S * m;
                    // the tile takes dS without the same-token block, which epilogue 2 adds
                    // in fp32 (so that dPhi can be formed without it)
                    ds[e] = (tj == ti) ? 0.0f : dSp * m;
#pragma unroll
                    for (int r = 0; r < R; ++r) dsd[r] += (j == ti * R + r) ? dSp * gam_i : 0.0f;
                    const float z = dSp * S;
                    const float zmv = (tj < ti) ? z * m : 0.0f;
                    rzm += zmv;
                    if (tj == ti) rg += z;
                    zm[row * 65 + j] = zmv;
                    ze[row * 65 + j] = (tj < ti) ? z * ez : 0.0f;
                }
                tile_put16(smem + OFF_SP, row, 4 * hc + 2 * half, sp);
                tile_put16(smem + OFF_DS, row, 4 * hc + 2 * half, ds);
            }
            rzm += __shfl_xor_sync(0xffffffffu, rzm, 16);
            rg += __shfl_xor_sync(0xffffffffu, rg, 16);
            if (hc == 0) {
                F[F_RZM + row] = rzm;
                F[F_RG + row] = rg;
            }
            if ((ti * R) / 32 == hc) {   // the block lies in this thread's column half
#pragma unroll
                for (int r = 0; r < R; ++r) F[F_DSD + row * 4 + r] = dsd[r];
            }
        } else {
            // T2 (row i: ebar_i = C~_i . T2_i) and XG (row j: ds_j = B~_j . XG_j)
            uint32_t vt[32], vx[32];
            ptx::tmem_ld16x2_32(tmem + lane_base + TM_T2, vt);
            ptx::tmem_ld16x2_32(tmem + lane_base + TM_XG, vx);
            ptx::tmem_ld_wait();
            float cr[32], br[32];
            tile_row32(sbase + ST_C, row, hc, cr);
            tile_row32(sbase + ST_B, row, hc, br);
            const int t = row / R;
            const float ei = F[F_ECS + t], sj = F[F_S + t];
            float eb = 0.0f, dsr = 0.0f;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float t2 = __uint_as_float(vt[e]), xg = __uint_as_float(vx[e]);
                eb = fmaf(cr[e], t2, eb);
                dsr = fmaf(br[e], xg, dsr);
                eT[e] = ei * t2;
                sX[e] = sj * xg;
            }
            eb += __shfl_xor_sync(0xffffffffu, eb, 16);
            dsr += __shfl_xor_sync(0xffffffffu, dsr, 16);
            if (hc == 0) {
                F[F_EBAR + row] = eb;
                F[F_DSR + row] = dsr;
            }
            if (c == nch - 1 && prm.theta) {
                // last chunk: this row's s-term share of dPhi, i.e. minus its pair with the
                // final state, for the start of the dtheta sum (the last token's rows
                // excluded: that pair has zero angle); nothing reads F_DPR yet
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    F[F_DPR + row * KS + 16 * hc + m] =
                        (t >= nt - 1) ? 0.0f : sX[2 * m] * br[2 * m + 1] - sX[2 * m + 1] * br[2 * m];
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
        if (abort_s) { fail = true; break; }
        // ---- (5) the masked products (thread 32): dX += S'^T dY, dC~ = dS B~,
        //      dB~ = dS^T C~; meanwhile the token scalars (warp 4) and the previous
        //      chunk's dtheta (warps 6, 7)
        if (tid == 32) {
            const uint32_t y_mn = ptx::sdesc_lo(ptx::smem_u32(sbase + ST_DY), TILE);
            const uint32_t b_mn = ptx::sdesc_lo(ptx::smem_u32(sbase + ST_B), TILE);
            const uint32_t c_mn = ptx::sdesc_lo(ptx::smem_u32(sbase + ST_C), TILE);
            const uint32_t sp_mn = ptx::sdesc_lo(ptx::smem_u32(smem + OFF_SP), TILE);
            const uint32_t ds_k = ptx::sdesc_lo(ptx::smem_u32(smem + OFF_DS), 16);
            const uint32_t ds_mn = ptx::sdesc_lo(ptx::smem_u32(smem + OFF_DS), TILE);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                ptx::umma_bf16_lo<kDescHi, kDescHi>(tmem + TM_DX, sp_mn + 128 * k, y_mn + 128 * k, kIdMM, 1);
                ptx::umma_bf16_lo<kDescHi, kDescHi>(tmem + TM_DC, ds_k + 2 * k, b_mn + 128 * k, kIdKM, k > 0);
                ptx::umma_bf16_lo<kDescHi, kDescHi>(tmem + TM_DB, ds_mn + 128 * k, c_mn + 128 * k, kIdMM, k > 0);
            }
            ptx::umma_commit(&bar_m2);
        }
        __syncwarp();
        if (wg == 0 && prm.theta && c + 1 < nch) dtheta_chunk(c + 1);
        if (wg == 1) {
            // column sums of dM o M (threads 128-191) and dM o E (192-255)
            const int j = (tid - 128) & 63;
            const float* src = (tid < 192) ? zm : ze;
            float a0 = 0.0f, a1 = 0.0f;
#pragma unroll 8
            for (int i = 0; i < 64; i += 2) {
                a0 += src[i * 65 + j];
                a1 += src[(i + 1) * 65 + j];
            }
            F[(tid < 192 ? F_CZM : F_CZE) + j] = a0 + a1;
            ptx::bar_sync(2, 128);
            if (warp == 6 && prm.theta && c == nch - 1) {
                // the final state's angle term: the part through G_{nch-1}, decayed over
                // the chunk, and the part through the chunk's rows but the last token's
                float acc = F[F_DPHI + lane] * m3::ex2_approx(F[F_CS + Q - 1]);
                for (int r2 = 0; r2 < 64; ++r2) acc -= F[F_DPR + r2 * KS + lane];
                F[F_DPHI + lane] = acc;
            }
        }
        if (warp == 4) {
            const float cs_end = F[F_CS + Q - 1];
            const float gdot = F[F_RED] + F[F_RED + 1] + F[F_RED + 2] + F[F_RED + 3];
            // per token (lane: tokens lane, lane + 32): dcs, dw, dgamma; x_t, the gradient
            // of s_t = exp(cs_end - cs_t) w_t through its decay, which depends on dt_k for
            // t < k <= end only: it is added over that range (R_k below) rather than as +
            // at cs_end and - at cs_t, which would cancel, inexactly, for every k <= t
            float dcs[2], dw[2], dg[2], xs[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = u * 32 + lane;
                dcs[u] = 0.0f; dw[u] = 0.0f; dg[u] = 0.0f; xs[u] = 0.0f;
                if (t < Q) {
                    const float s_t = F[F_S + t], ecs_t = F[F_ECS + t], ee = F[F_EEND + t];
                    for (int r = 0; r < R; ++r) {
                        const int i = t * R + r;
                        dcs[u] += F[F_RZM + i] - F[F_CZM + i] + F[F_EBAR + i] * ecs_t;
                        dw[u] += F[F_CZE + i] + F[F_DSR + i] * ee;
                        dg[u] += F[F_RG + i];
                        xs[u] = fmaf(F[F_DSR + i], s_t, xs[u]);
                    }
                }
            }
            // cs_end: through exp(cs_end) G_{c-1} (cs here in log2 units; the gradients are
            // with respect to the natural-log cs: d/dcs 2^(x log2 e) = value)
            const float dcs_end = gdot * m3::ex2_approx(cs_end);
            if (Q == 64) { if (lane == 31) dcs[1] += dcs_end; }
            else if (lane == Q - 1) dcs[0] += dcs_end;
            // R_k = sum_{t >= k} dcs_t + sum_{t < k} x_t;  ddt_k += A R_k;  dA += sum_k dt_k R_k
            const float* sdt = F + F_DL + st * 2 * 68;
            const float* slm = sdt + 68;
            float sfx[2];
            {
                // suffix sums of dcs over the 64 tokens (lane u * 32 + lane)
                float a1 = dcs[1];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float v = __shfl_down_sync(0xffffffffu, a1, o);
                    if (lane + o < 32) a1 += v;
                }
                float a0 = dcs[0];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float v = __shfl_down_sync(0xffffffffu, a0, o);
                    if (lane + o < 32) a0 += v;
                }
                sfx[1] = a1;
                sfx[0] = a0 + __shfl_sync(0xffffffffu, a1, 0);
                // exclusive prefix sums of x
                float p0 = xs[0], p1 = xs[1];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float v0 = __shfl_up_sync(0xffffffffu, p0, o);
                    const float v1 = __shfl_up_sync(0xffffffffu, p1, o);
                    if (lane >= o) { p0 += v0; p1 += v1; }
                }
                // exclusive: the previous lane's inclusive sum (never "inclusive - own",
                // which cancels against an x of much larger size)
                const float tot0 = __shfl_sync(0xffffffffu, p0, 31);
                const float e0 = __shfl_up_sync(0xffffffffu, p0, 1), e1 = __shfl_up_sync(0xffffffffu, p1, 1);
                sfx[0] += (lane == 0) ? 0.0f : e0;
                sfx[1] += (lane == 0) ? tot0 : tot0 + e1;
            }
            float dA_c = 0.0f;
            {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int t = u * 32 + lane;
                    if (t < Q) dA_c = fmaf(sdt[t], sfx[u], dA_c);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dA_c += __shfl_xor_sync(0xffffffffu, dA_c, o);
            }
            // dt / lambda per token: gamma = lambda dt; w_t = gamma_t + (1 - lambda_{t+1}) dt_{t+1}
            float nd = 0.0f, nl = 0.0f;
            // dw of the token before: shuffled by every lane, then chosen
            const float up0 = __shfl_up_sync(0xffffffffu, dw[0], 1);
            const float up1 = __shfl_up_sync(0xffffffffu, dw[1], 1);
            const float last0 = __shfl_sync(0xffffffffu, dw[0], 31);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = u * 32 + lane;
                const float dw_prev = (u == 0) ? up0 : (lane == 0 ? last0 : up1);
                if (t < Q) {
                    const float g_t = dg[u] + dw[u];
                    const float lam_t = prm.lam ? slm[t] : 1.0f;
                    float d_dt = A_h * sfx[u] + g_t * lam_t;
                    float d_l = g_t * sdt[t];
                    if (t > 0) {
                        d_dt = fmaf(dw_prev, 1.0f - lam_t, d_dt);
                        d_l = fmaf(-dw_prev, sdt[t], d_l);
                    }
                    F[F_DTOK + t] = d_dt;
                    F[F_DTOK + 64 + t] = d_l;
                    if (t == Q - 1) {
                        const float lam_n = prm.lam ? slm[Q] : 1.0f;
                        nd = dw[u] * (1.0f - lam_n);
                        nl = -dw[u] * sdt[Q];
                    }
                }
            }
            __syncwarp();
            if (lane == (Q - 1) % 32) {
                // token c0 + Q (the first of the chunk processed before) is complete
                if (t0 + Q < T) {
                    prm.ddt[tok_idx(t0 + Q)] = F[F_PEND] + nd;
                    if (prm.dlam) prm.dlam[tok_idx(t0 + Q)] = F[F_PEND + 1] + nl;
                }
            }
            __syncwarp();
            for (int t = 1 + lane; t < nt; t += 32) {
                prm.ddt[tok_idx(t0 + t)] = F[F_DTOK + t];
                if (prm.dlam) prm.dlam[tok_idx(t0 + t)] = F[F_DTOK + 64 + t];
            }
            if (lane == 0) {
                F[F_PEND] = F[F_DTOK];
                F[F_PEND + 1] = F[F_DTOK + 64];
                if (c == 0) {
                    prm.ddt[tok_idx(0)] = F[F_DTOK];
                    if (prm.dlam) prm.dlam[tok_idx(0)] = F[F_DTOK + 64];
                }
                dA_acc += dA_c;
            }
        }
        ptx::bar_sync(4, kThreads);   // warpgroup 0's dtheta has read F_DPR before epilogue 2 rewrites it
        if (!ptx::mbar_wait(&bar_m2, (nch - 1 - c) & 1, kWaitBudget)) {
            m3::set_status(m3::kStatusWaitTimeout);
            abort_s = 1;
        }
        __syncwarp();
        ptx::tc_fence_after();
        // ---- (6) epilogue 2
        if (wg == 0) {
            // dx of row j; dG_{c-1} = exp(cs_end) dG_c + dGu (rows n)
            uint32_t vx[32], vg[32];
            ptx::tmem_ld16x2_32(tmem + lane_base + TM_DX, vx);
            ptx::tmem_ld16x2_32(tmem + lane_base + TM_DGU, vg);
            ptx::tmem_ld_wait();
            // dx of row j into the staging tile (the S' buffer, free once the masked
            // products are done; rows past the sequence end are clipped by the store)
#pragma unroll
            for (int g = 0; g < 4; ++g)
                *reinterpret_cast<uint4*>(smem + OFF_SP + swz(row, 4 * hc + g)) =
                    make_uint4(pack2(__uint_as_float(vx[8 * g]), __uint_as_float(vx[8 * g + 1])),
                               pack2(__uint_as_float(vx[8 * g + 2]), __uint_as_float(vx[8 * g + 3])),
                               pack2(__uint_as_float(vx[8 * g + 4]), __uint_as_float(vx[8 * g + 5])),
                               pack2(__uint_as_float(vx[8 * g + 6]), __uint_as_float(vx[8 * g + 7])));
            const float dec = m3::ex2_approx(F[F_CS + Q - 1]);
#pragma unroll
            for (int p = 0; p < 32; ++p) dG[p] = fmaf(dec, dG[p], __uint_as_float(vg[p]));
            tile_put32(smem + OFF_DG, row, hc, dG);
        } else {
            // dC~ (row i) and dB~ (row j): the MMA terms plus the held ones, rotated
            // back by Phi; this row's share of dPhi per pair
            uint32_t vc[32], vb[32];
            ptx::tmem_ld16x2_32(tmem + lane_base + TM_DC, vc);
            ptx::tmem_ld16x2_32(tmem + lane_base + TM_DB, vb);
            ptx::tmem_ld_wait();
            const int t = row / R;
            // the same-token block's share of dC~ (row i: sum over j in i's token of
            // dS_ij B~_j) and of dB~ (row j: sum over i in j's token of dS_ij C~_i), in
            // fp32 (the products above left it out): its contributions to dPhi through
            // B~ and C~ cancel exactly (C~_i . B~_j is unchanged by a common rotation), so
            // dPhi is formed without it, free of that cancellation.  Likewise the s-term
            // of the last token's rows in the last chunk (its pair with the final state).
            // Eight columns (four pairs) at a time, to keep the registers in bounds.
            float d_io[R], d_oi[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                d_io[r] = F[F_DSD + row * 4 + r];
                d_oi[r] = F[F_DSD + (t * R + r) * 4 + (row - t * R)];
            }
            const bool fin = (c == nch - 1) && t == nt - 1;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                float cr[8], br[8], cdg[8], bdg[8];
                tile_row8(sbase + ST_C, row, 4 * hc + g, cr);
                tile_row8(sbase + ST_B, row, 4 * hc + g, br);
#pragma unroll
                for (int e = 0; e < 8; ++e) { cdg[e] = 0.0f; bdg[e] = 0.0f; }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float vb2[8], vc2[8];
                    tile_row8(sbase + ST_B, t * R + r, 4 * hc + g, vb2);
                    tile_row8(sbase + ST_C, t * R + r, 4 * hc + g, vc2);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        cdg[e] = fmaf(d_io[r], vb2[e], cdg[e]);
                        bdg[e] = fmaf(d_oi[r], vc2[e], bdg[e]);
                    }
                }
                uint32_t pc[4], pb[4];
#pragma unroll
                for (int mm = 0; mm < 4; ++mm) {
                    const int m = 4 * g + mm, k = 16 * hc + m, e = 2 * mm;
                    // f: the terms that enter dPhi; d: the whole dC~ / dB~
                    const float fc0 = __uint_as_float(vc[2 * m]) + eT[2 * m];
                    const float fc1 = __uint_as_float(vc[2 * m + 1]) + eT[2 * m + 1];
                    const float vb0 = __uint_as_float(vb[2 * m]), vb1 = __uint_as_float(vb[2 * m + 1]);
                    const float fb0 = fin ? vb0 : vb0 + sX[2 * m], fb1 = fin ? vb1 : vb1 + sX[2 * m + 1];
                    const float dc0 = fc0 + cdg[e], dc1 = fc1 + cdg[e + 1];
                    const float db0 = vb0 + sX[2 * m] + bdg[e], db1 = vb1 + sX[2 * m + 1] + bdg[e + 1];
                    float co = 1.0f, si = 0.0f;
                    if (prm.theta) { co = F[F_COS + t * KS + k]; si = F[F_SIN + t * KS + k]; }
                    // dC = Rot(+phi) dC~, dB likewise: (a cos - b sin, a sin + b cos)
                    pc[mm] = pack2(fmaf(dc0, co, -dc1 * si), fmaf(dc0, si, dc1 * co));
                    pb[mm] = pack2(fmaf(db0, co, -db1 * si), fmaf(db0, si, db1 * co));
                    // d/dphi Rot(-phi) v = (v~_1, -v~_0)
                    F[F_DPR + row * KS + k] = fb0 * br[e + 1] - fb1 * br[e] + fc0 * cr[e + 1] - fc1 * cr[e];
                }
                // into the staging tiles (the dS and C~' buffers, free here)
                *reinterpret_cast<uint4*>(smem + OFF_DS + swz(row, 4 * hc + g)) = make_uint4(pc[0], pc[1], pc[2], pc[3]);
                *reinterpret_cast<uint4*>(smem + OFF_CD + swz(row, 4 * hc + g)) = make_uint4(pb[0], pb[1], pb[2], pb[3]);
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
        if (tid == 0) {
            // dx, dC, dB of the chunk: one TMA store each from the staging tiles
            // (their reads are waited for before the tiles are written again)
            ptx::tma_store_5d(&map_dx, smem + OFF_SP, 0, 0, h, (int)t0, b);
            ptx::tma_store_5d(&map_dC, smem + OFF_DS, 0, 0, h, (int)t0, b);
            ptx::tma_store_5d(&map_dB, smem + OFF_CD, 0, 0, h, (int)t0, b);
            ptx::bulk_commit();
        }
        __syncthreads();
    }
    // dtheta of chunk 0 (the last chunk processed)
    if (!fail && wg == 0 && prm.theta) dtheta_chunk(0);
    if (tid == 0) ptx::bulk_wait0();   // every gradient tile stored
    if (tid == 128) prm.dA_part[unit] = dA_acc;   // warp 4 lane 0 accumulated it
    if (fail && tid == 0) {
        // stopped early: the checkpoint copies in flight land (bounded wait)
        for (int s2 = 0; s2 < 2; ++s2)
            if (ck_count[s2] > 0) (void)ptx::mbar_wait(&bar_ck[s2], (ck_count[s2] - 1) & 1, kWaitBudget);
    }
    if (fail && tid == 32) {
        // stopped early: wait (bounded) for the last load of each stage
        for (int s2 = 0; s2 < 2; ++s2)
            if (ld_count[s2] > 0) (void)ptx::mbar_wait(&bar_ld[s2], (ld_count[s2] - 1) & 1, kWaitBudget);
    }
    if (fail && tid == 32) {
        // every MMA issued has completed once this commit arrives
        ptx::umma_commit(&bar_fin);
        (void)ptx::mbar_wait(&bar_fin, 0, kWaitBudget);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc(tmem, TM_COLS);
}

}  // namespace m3bwdtc
