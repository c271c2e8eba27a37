// m3scan.cu -- the C ABI of libm3scan.so (declared in include/m3scan.h):
// host-side validation, kernel selection and launch.  Every kernel of the
// library is compiled in this one translation unit.
#include <cuda_runtime.h>

#include <cstdint>
#include <cmath>
#include <cstring>
#include <mutex>

#include "m3scan.h"
#include "common.cuh"
#include "step_simt.cuh"
#include "step_fast.cuh"
#include "step_k.cuh"
#include "step_ring.cuh"
#include "scan_ws.cuh"
#include "scan_chunk.cuh"
#include "scan_bwd.cuh"
#include "scan_bwd_tc.cuh"
#include "selftest.cuh"

namespace {

using m3::SimtArgs;
using m3::TokLayout;

constexpr size_t kMaxSmem = 227 * 1024;

bool aligned(const void* p, uintptr_t bytes) { return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) == 0; }
bool aligned16(const void* p) { return aligned(p, 16); }

// Validates the sizes shared by both entry points.
int check_dims(const m3_dims* d, bool need_chunk) {
    if (!d) return M3_ERR_NULL;
    if (d->dtype != M3_F32 && d->dtype != M3_BF16) return M3_ERR_DTYPE;
    if (d->reserved != 0) return M3_ERR_SHAPE;
    if (d->batch < 0 || d->seqlen < 0 || d->heads < 1) return M3_ERR_SHAPE;
    if (d->headdim < 4 || d->headdim > 256 || d->headdim % 4 != 0) return M3_ERR_SHAPE;
    if (d->dstate < 2 || d->dstate > 256 || d->dstate % 2 != 0) return M3_ERR_SHAPE;
    if (d->rank < 1 || d->rank > 8) return M3_ERR_SHAPE;
    if (need_chunk && d->chunk != 16 && d->chunk != 32 && d->chunk != 64 && d->chunk != 128)
        return M3_ERR_SHAPE;
    if (d->batch * d->heads > INT32_MAX) return M3_ERR_SHAPE;
    return M3_OK;
}

// SIMT geometry: NPT row pairs per thread, TK threads along pairs, P/4 along P.
bool simt_geometry(const m3_dims* d, SimtArgs* a, int* npt, int* block) {
    const int N = (int)d->dstate, P = (int)d->headdim, R = (int)d->rank;
    const int K = N / 2, P4 = P / 4, units = K * P4;
    int n = 1;
    while (units / n > 256 && K % (2 * n) == 0 && n < 8) n *= 2;
    if (units / n > 512) return false;
    a->R = R; a->P = P; a->N = N; a->K = K; a->P4 = P4; a->TK = K / n;
    *npt = n;
    *block = a->TK * P4;
    return true;
}

size_t step_smem_bytes(const SimtArgs& a) {
    const TokLayout L(a.R, a.P, a.N);
    return sizeof(float) * (2 * (size_t)L.size + (size_t)a.TK * a.R * a.P);
}
size_t seq_smem_bytes(const SimtArgs& a) {
    const TokLayout L(a.R, a.P, a.N);
    return sizeof(float) * (3 * (size_t)L.size + 2 * (size_t)a.TK * a.R * a.P);
}

template <typename K>
int prepare(K kernel, size_t smem) {
    if (smem > kMaxSmem) return M3_ERR_UNSUPPORTED;
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return M3_ERR_CUDA;
    }
    return M3_OK;
}

int launch_status() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

template <typename T, int NPT>
int launch_step(const m3_dims* d, const SimtArgs& a, int block, float* state, const void* x_t, const float* dt_t,
                const float* A, const void* B_t, const void* C_t, const float* lam_t, const void* theta_t,
                const void* prev_B, const void* prev_x, void* y_t, cudaStream_t s) {
    auto k = m3::m3_step_kernel<T, NPT>;
    const size_t smem = step_smem_bytes(a);
    int rc = prepare(k, smem);
    if (rc != M3_OK) return rc;
    k<<<(unsigned)(d->batch * d->heads), block, smem, s>>>(
        a, d->heads, state, (const T*)x_t, dt_t, A, (const T*)B_t, (const T*)C_t, lam_t, (const T*)theta_t,
        (const T*)prev_B, (const T*)prev_x, (T*)y_t);
    return launch_status();
}

template <typename T, int NPT>
int launch_seq(const m3_dims* d, const SimtArgs& a, int block, const void* x, const float* dt, const float* A,
               const void* B, const void* C, const float* lam, const void* theta, void* y, float* final_state,
               const float* h0, const void* prev_B, const void* prev_x, cudaStream_t s) {
    auto k = m3::m3_scan_seq_kernel<T, NPT>;
    const size_t smem = seq_smem_bytes(a);
    int rc = prepare(k, smem);
    if (rc != M3_OK) return rc;
    k<<<(unsigned)(d->batch * d->heads), block, smem, s>>>(a, d->seqlen, d->heads, (const T*)x, dt, A, (const T*)B,
                                                          (const T*)C, lam, (const T*)theta, (T*)y, final_state, h0,
                                                          (const T*)prev_B, (const T*)prev_x);
    return launch_status();
}

template <typename T>
int dispatch_seq(const m3_dims* d, const void* x, const float* dt, const float* A, const void* B, const void* C,
                 const float* lam, const void* theta, void* y, float* fs, const float* h0, const void* pB,
                 const void* px, cudaStream_t s) {
    SimtArgs a;
    int npt, block;
    if (!simt_geometry(d, &a, &npt, &block)) return M3_ERR_UNSUPPORTED;
    switch (npt) {
        case 1: return launch_seq<T, 1>(d, a, block, x, dt, A, B, C, lam, theta, y, fs, h0, pB, px, s);
        case 2: return launch_seq<T, 2>(d, a, block, x, dt, A, B, C, lam, theta, y, fs, h0, pB, px, s);
        case 4: return launch_seq<T, 4>(d, a, block, x, dt, A, B, C, lam, theta, y, fs, h0, pB, px, s);
        case 8: return launch_seq<T, 8>(d, a, block, x, dt, A, B, C, lam, theta, y, fs, h0, pB, px, s);
    }
    return M3_ERR_UNSUPPORTED;
}

template <typename T>
int dispatch_step(const m3_dims* d, float* state, const void* x_t, const float* dt_t, const float* A,
                  const void* B_t, const void* C_t, const float* lam_t, const void* theta_t, const void* prev_B,
                  const void* prev_x, void* y_t, cudaStream_t s) {
    SimtArgs a;
    int npt, block;
    if (!simt_geometry(d, &a, &npt, &block)) return M3_ERR_UNSUPPORTED;
    switch (npt) {
        case 1: return launch_step<T, 1>(d, a, block, state, x_t, dt_t, A, B_t, C_t, lam_t, theta_t, prev_B, prev_x, y_t, s);
        case 2: return launch_step<T, 2>(d, a, block, state, x_t, dt_t, A, B_t, C_t, lam_t, theta_t, prev_B, prev_x, y_t, s);
        case 4: return launch_step<T, 4>(d, a, block, state, x_t, dt_t, A, B_t, C_t, lam_t, theta_t, prev_B, prev_x, y_t, s);
        case 8: return launch_step<T, 8>(d, a, block, state, x_t, dt_t, A, B_t, C_t, lam_t, theta_t, prev_B, prev_x, y_t, s);
    }
    return M3_ERR_UNSUPPORTED;
}

// Geometry of the chunked CUDA-core kernel for `d` (inputs staged in their dtype).
m3cs::Geo chunk_geo(const m3_dims* d) {
    return m3cs::make_geo(d->seqlen, (int)d->heads, (int)d->headdim, (int)d->dstate, (int)d->rank, (int)d->chunk,
                          d->dtype == M3_F32 ? 4 : 2);
}

template <typename T>
int launch_chunk(const m3_dims* d, const void* x, const float* dt, const float* A, const void* B, const void* C,
                 const float* lam, const void* theta, void* y, float* fs, const float* h0, const void* pB,
                 const void* px, cudaStream_t s) {
    const m3cs::Geo g = chunk_geo(d);
    auto k = m3cs::m3_scan_chunk_kernel<T>;
    int rc = prepare(k, (size_t)g.bytes);
    if (rc != M3_OK) return rc;
    k<<<(unsigned)(d->batch * d->heads), m3cs::kThreads, g.bytes, s>>>(
        g, (const T*)x, dt, A, (const T*)B, (const T*)C, lam, (const T*)theta, (T*)y, fs, h0, (const T*)pB,
        (const T*)px);
    return launch_status();
}

// The decode step for the common shapes (step_fast.cuh); every tensor is
// 16-byte aligned (checked by the caller).
template <typename T>
int launch_step_fast(const m3_dims* d, float* state, const void* x_t, const float* dt_t, const float* A,
                     const void* B_t, const void* C_t, const float* lam_t, const void* theta_t, const void* prev_B,
                     const void* prev_x, void* y_t, cudaStream_t s) {
    m3fast::StepArgs a;
    a.H = (int)d->heads;
    a.N = (int)d->dstate;
    a.P = (int)d->headdim;
    a.P4 = a.P / 4;
    const int block = m3fast::threads(d->dstate, d->headdim);
    const size_t smem = m3fast::smem_bytes(d->dstate, d->headdim, d->rank);
    const unsigned grid = (unsigned)(d->batch * d->heads);
#define M3_STEP_FAST(RR, MT)                                                                                  \
    m3fast::m3_step_fast_kernel<T, RR, MT><<<grid, block, smem, s>>>(a, state, (const T*)x_t, dt_t, A,          \
                                                                     (const T*)B_t, (const T*)C_t, lam_t,       \
                                                                     (const T*)theta_t, (const T*)prev_B,       \
                                                                     (const T*)prev_x, (T*)y_t)
    const bool small = block <= 128;
    switch (d->rank) {
        case 1: if (small) M3_STEP_FAST(1, 128); else M3_STEP_FAST(1, 256); break;
        case 2: if (small) M3_STEP_FAST(2, 128); else M3_STEP_FAST(2, 256); break;
        case 4: if (small) M3_STEP_FAST(4, 128); else M3_STEP_FAST(4, 256); break;
        default: return M3_ERR_UNSUPPORTED;
    }
#undef M3_STEP_FAST
    return launch_status();
}

// The decode step through the shared-memory ring (step_ring.cuh): persistent
// CTAs, as many as fit on the device at once; every tensor is 16-byte aligned
// and every per-unit block a multiple of 16 bytes (checked by the caller).
template <typename T>
int launch_step_ring(const m3_dims* d, float* state, const void* x_t, const float* dt_t, const float* A,
                     const void* B_t, const void* C_t, const float* lam_t, const void* theta_t, const void* prev_B,
                     const void* prev_x, void* y_t, cudaStream_t s) {
    const m3ring::Geo g = m3ring::make_geo(d->batch * d->heads, (int)d->heads, (int)d->dstate, (int)d->headdim,
                                           (int)d->rank, (int)sizeof(T));
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return M3_ERR_CUDA;
    int rc = M3_OK;
#define M3_STEP_RING(RR, MT)                                                                                    \
    do {                                                                                                        \
        auto k = m3ring::m3_step_ring_kernel<T, RR, MT>;                                                        \
        rc = prepare(k, g.smem_bytes);                                                                          \
        if (rc != M3_OK) return rc;                                                                             \
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, g.nthreads, g.smem_bytes) != cudaSuccess || \
            per_sm < 1)                                                                                         \
            return M3_ERR_UNSUPPORTED;                                                                          \
        const int64_t want = (int64_t)sms * per_sm;                                                             \
        const unsigned grid = (unsigned)(g.units < want ? g.units : want);                                      \
        k<<<grid, g.nthreads, g.smem_bytes, s>>>(g, state, (const T*)x_t, dt_t, A, (const T*)B_t, (const T*)C_t,   \
                                                lam_t, (const T*)theta_t, (const T*)prev_B, (const T*)prev_x,      \
                                                (T*)y_t);                                                       \
    } while (0)
    const bool small = g.nthreads <= 128;
    switch (d->rank) {
        case 2: if (small) M3_STEP_RING(2, 128); else M3_STEP_RING(2, 256); break;
        case 4: if (small) M3_STEP_RING(4, 128); else M3_STEP_RING(4, 256); break;
        default: return M3_ERR_UNSUPPORTED;
    }
#undef M3_STEP_RING
    return launch_status();
}

// The multi-token decode kernel for the common shapes (step_k.cuh); every
// tensor it reads with vector loads is 16-byte aligned (checked by the caller).
template <typename T>
int launch_step_k(const m3_dims* d, float* state, const void* x, const float* dt, const float* A, const void* B,
                  const void* C, const float* lam, const void* theta, const void* prev_B, const void* prev_x, void* y,
                  cudaStream_t s) {
    const m3fast::StepKArgs a = m3fast::stepk_layout((int)d->heads, (int)d->dstate, (int)d->headdim, (int)d->rank,
                                                     d->seqlen, (int)sizeof(T));
    const int block = m3fast::threads(d->dstate, d->headdim);
    const size_t smem = m3fast::stepk_smem(a, (int)d->rank);
    int rc = M3_OK;
    switch (d->rank) {
        case 1: rc = prepare(m3fast::m3_step_k_kernel<T, 1, 128>, smem); if (rc == M3_OK) rc = prepare(m3fast::m3_step_k_kernel<T, 1, 256>, smem); break;
        case 2: rc = prepare(m3fast::m3_step_k_kernel<T, 2, 128>, smem); if (rc == M3_OK) rc = prepare(m3fast::m3_step_k_kernel<T, 2, 256>, smem); break;
        case 4: rc = prepare(m3fast::m3_step_k_kernel<T, 4, 128>, smem); if (rc == M3_OK) rc = prepare(m3fast::m3_step_k_kernel<T, 4, 256>, smem); break;
        default: return M3_ERR_UNSUPPORTED;
    }
    if (rc != M3_OK) return rc;
    const unsigned grid = (unsigned)(d->batch * d->heads);
#define M3_STEP_K(RR, MT)                                                                                   \
    m3fast::m3_step_k_kernel<T, RR, MT><<<grid, block, smem, s>>>(a, state, (const T*)x, dt, A, (const T*)B,    \
                                                                  (const T*)C, lam, (const T*)theta,            \
                                                                  (const T*)prev_B, (const T*)prev_x, (T*)y)
    const bool small = block <= 128;
    switch (d->rank) {
        case 1: if (small) M3_STEP_K(1, 128); else M3_STEP_K(1, 256); break;
        case 2: if (small) M3_STEP_K(2, 128); else M3_STEP_K(2, 256); break;
        case 4: if (small) M3_STEP_K(4, 128); else M3_STEP_K(4, 256); break;
        default: return M3_ERR_UNSUPPORTED;
    }
#undef M3_STEP_K
    return launch_status();
}

// The tensor-core kernel takes its shapes when the chunk is one 64-row tile
// (Q R = 64); every other chunk runs on the chunked CUDA-core kernel when its
// shared memory fits, else on the token-serial kernel.
int scan_algorithm(const m3_dims* d) {
    if (check_dims(d, true) != M3_OK) return M3_ALGO_NONE;
    if (m3ws::supports(*d) && d->chunk * d->rank == m3ws::kRows) return M3_ALGO_CHUNKED_TC;
    if ((size_t)chunk_geo(d).bytes <= kMaxSmem && d->heads <= INT32_MAX) return M3_ALGO_CHUNKED_SIMT;
    SimtArgs a;
    int npt, block;
    if (!simt_geometry(d, &a, &npt, &block) || seq_smem_bytes(a) > kMaxSmem) return M3_ALGO_NONE;
    return M3_ALGO_SEQUENTIAL;
}

// The backward pass: chunk * R <= 64 rows, and both passes' shared memory fits.
m3bwd::Geo bwd_geo(const m3_dims* d) {
    return m3bwd::make_geo(d->seqlen, (int)d->heads, (int)d->headdim, (int)d->dstate, (int)d->rank, (int)d->chunk);
}
bool bwd_supported(const m3_dims* d) {
    if (d->chunk * d->rank > 64) return false;
    const m3bwd::Geo g = bwd_geo(d);
    return (size_t)g.bytes <= kMaxSmem && (size_t)g.c_bytes <= kMaxSmem;
}

// The tensor-core backward: bf16, N = P = 64, R in {1, 2, 4}, one 64-row tile per
// chunk, every tensor the TMA reads or writes 16-byte aligned.
bool bwd_tc_shape(const m3_dims* d, const void* const* ptrs, int n) {
    if (!m3ws::supports(*d) || d->dstate != 64 || d->chunk * d->rank != m3ws::kRows) return false;
    for (int i = 0; i < n; ++i)
        if (ptrs[i] && !aligned16(ptrs[i])) return false;
    return true;
}

// 4-D map over theta [b, T, h, K] bf16, box (K, 1, Q, 1), no swizzle: the tile
// lands as [Q][K] rows of 2 K bytes.
bool make_map_theta_plain(CUtensorMap* m, const void* base, const m3_dims& d, int Q) {
    const cuuint64_t K = (cuuint64_t)d.dstate / 2;
    cuuint64_t dims[4] = {K, (cuuint64_t)d.heads, (cuuint64_t)d.seqlen, (cuuint64_t)d.batch};
    cuuint64_t strides[3] = {K * 2, (cuuint64_t)d.heads * K * 2, (cuuint64_t)d.seqlen * d.heads * K * 2};
    cuuint32_t box[4] = {(cuuint32_t)K, 1, (cuuint32_t)Q, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return m3ws::encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_bwd_tc(const m3_dims* d, const void* x, const float* dt, const float* A, const void* B, const void* C,
                  const float* lam, const void* theta, const void* dy, const float* dfinal, void* dx, float* ddt,
                  float* dA, void* dB, void* dC, float* dlam, void* dtheta, const m3bwd::Work& w, cudaStream_t s) {
    // pass 1: the forward tensor-core kernel's checkpoint run (the chunk states and
    // angles only; dx is passed as its y but not written)
    int rc = m3ws::launch(*d, x, dt, A, B, C, lam, theta, nullptr, nullptr, nullptr, dx, nullptr, s, nullptr,
                          nullptr, nullptr, nullptr, 0.0f, w.G, w.phi);
    if (rc != M3_OK) return rc;
    // pass 2
    const int Q = m3ws::kRows / (int)d->rank;
    CUtensorMap maps[9];
    memset(maps, 0, sizeof(maps));
    // inputs: x, B, C, dy, theta; the gradient tiles the kernel stores: dx, dB, dC, dtheta
    if (!m3ws::make_map5(&maps[0], x, *d, 64, Q) || !m3ws::make_map5(&maps[1], B, *d, 64, Q) ||
        !m3ws::make_map5(&maps[2], C, *d, 64, Q) || !m3ws::make_map5(&maps[3], dy, *d, 64, Q) ||
        !m3ws::make_map5(&maps[5], dx, *d, 64, Q) || !m3ws::make_map5(&maps[6], dB, *d, 64, Q) ||
        !m3ws::make_map5(&maps[7], dC, *d, 64, Q))
        return M3_ERR_CUDA;
    if (theta) {
        if (!make_map_theta_plain(&maps[4], theta, *d, Q) || !make_map_theta_plain(&maps[8], dtheta, *d, Q))
            return M3_ERR_CUDA;
    } else {
        maps[4] = maps[0];   // never read
        maps[8] = maps[0];   // never written
    }
    m3bwdtc::Params prm;
    prm.T = d->seqlen;
    prm.H = (int)d->heads;
    prm.nch = (int)((d->seqlen + Q - 1) / Q);
    prm.dt = dt;
    prm.A = A;
    prm.lam = lam;
    prm.theta = static_cast<const __nv_bfloat16*>(theta);
    prm.dfinal = dfinal;
    prm.ck_G = w.G;
    prm.ck_phi = w.phi;
    prm.dA_part = w.dA;
    prm.dx = static_cast<__nv_bfloat16*>(dx);
    prm.ddt = ddt;
    prm.dB = static_cast<__nv_bfloat16*>(dB);
    prm.dC = static_cast<__nv_bfloat16*>(dC);
    prm.dlam = dlam;
    prm.dtheta = static_cast<__nv_bfloat16*>(dtheta);
    const unsigned grid = (unsigned)(d->batch * d->heads);
#define M3_BWD_TC(RR)                                                                                           \
    {                                                                                                          \
        auto k = m3bwdtc::m3_bwd_tc_kernel<RR>;                                                                \
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, m3bwdtc::SMEM_BYTES) !=       \
            cudaSuccess)                                                                                       \
            return M3_ERR_CUDA;                                                                                \
        k<<<grid, m3bwdtc::kThreads, m3bwdtc::SMEM_BYTES, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4],     \
                                                               maps[5], maps[6], maps[7], maps[8], prm);       \
    }
    switch (d->rank) {
        case 1: M3_BWD_TC(1); break;
        case 2: M3_BWD_TC(2); break;
        case 4: M3_BWD_TC(4); break;
        default: return M3_ERR_UNSUPPORTED;
    }
#undef M3_BWD_TC
    m3bwd::m3_bwd_dA_kernel<<<(unsigned)((d->heads + 127) / 128), 128, 0, s>>>(w.dA, d->batch, (int)d->heads, dA);
    return launch_status();
}

template <typename T>
int launch_bwd(const m3_dims* d, const void* x, const float* dt, const float* A, const void* B, const void* C,
               const float* lam, const void* theta, const void* dy, const float* dfinal, void* dx, float* ddt,
               float* dA, void* dB, void* dC, float* dlam, void* dtheta, void* ws, cudaStream_t s) {
    const m3bwd::Geo g = bwd_geo(d);
    const int64_t units = d->batch * d->heads;
    const m3bwd::Work w = m3bwd::work_split(ws, units, g);
    if constexpr (sizeof(T) == 2) {
        const void* tma_ptrs[] = {x, B, C, theta, dy, dx, dB, dC, dtheta};
        if (bwd_tc_shape(d, tma_ptrs, 9))
            return launch_bwd_tc(d, x, dt, A, B, C, lam, theta, dy, dfinal, dx, ddt, dA, dB, dC, dlam, dtheta, w, s);
    }
    auto k1 = m3bwd::m3_bwd_ckpt_kernel<T>;
    auto k2 = m3bwd::m3_bwd_chunk_kernel<T>;
    int rc = prepare(k1, (size_t)g.c_bytes);
    if (rc == M3_OK) rc = prepare(k2, (size_t)g.bytes);
    if (rc != M3_OK) return rc;
    k1<<<(unsigned)units, m3bwd::kThreads, g.c_bytes, s>>>(g, w, (const T*)x, dt, A, (const T*)B, lam,
                                                           (const T*)theta);
    k2<<<(unsigned)units, m3bwd::kThreads, g.bytes, s>>>(g, w, (const T*)x, dt, A, (const T*)B, (const T*)C, lam,
                                                         (const T*)theta, (const T*)dy, dfinal, (T*)dx, ddt, (T*)dB,
                                                         (T*)dC, dlam, (T*)dtheta);
    m3bwd::m3_bwd_dA_kernel<<<(unsigned)((d->heads + 127) / 128), 128, 0, s>>>(w.dA, d->batch, (int)d->heads, dA);
    return launch_status();
}

}  // namespace

extern "C" {

size_t m3_scan_bwd_workspace_size(const m3_dims* d) {
    if (check_dims(d, true) != M3_OK || !bwd_supported(d)) return 0;
    return m3bwd::work_bytes(d->batch * d->heads, bwd_geo(d));
}

int m3_scan_bwd(const m3_dims* d, const void* x, const float* dt, const float* A, const void* B, const void* C,
                const float* lambda, const void* theta, const void* dy, const float* dfinal, void* dx, float* ddt,
                float* dA, void* dB, void* dC, float* dlambda, void* dtheta, void* workspace,
                size_t workspace_bytes, void* stream) {
    int rc = check_dims(d, true);
    if (rc != M3_OK) return rc;
    const bool has_tokens = d->batch > 0 && d->seqlen > 0;
    if (!dA) return M3_ERR_NULL;
    if (has_tokens && (!x || !dt || !A || !B || !C || !dy || !dx || !ddt || !dB || !dC)) return M3_ERR_NULL;
    if (has_tokens && ((lambda != nullptr && !dlambda) || (theta != nullptr && !dtheta))) return M3_ERR_NULL;
    const uintptr_t es = d->dtype == M3_F32 ? 4 : 2;
    const void* elem_ptrs[] = {x, B, C, theta, dy, dx, dB, dC, dtheta};
    for (const void* p : elem_ptrs)
        if (p && !aligned(p, es)) return M3_ERR_ALIGN;
    const void* f32_ptrs[] = {dt, A, lambda, dfinal, ddt, dA, dlambda};
    for (const void* p : f32_ptrs)
        if (p && !aligned(p, 4)) return M3_ERR_ALIGN;
    if (!bwd_supported(d)) return M3_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!has_tokens) {
        // no token: y does not exist and the final state is zero whatever the
        // inputs, so every gradient is zero; only dA has elements
        return cudaMemsetAsync(dA, 0, sizeof(float) * d->heads, s) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
    }
    const size_t need = m3bwd::work_bytes(d->batch * d->heads, bwd_geo(d));
    if (!workspace || workspace_bytes < need) return M3_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return M3_ERR_ALIGN;
    return d->dtype == M3_F32 ? launch_bwd<float>(d, x, dt, A, B, C, lambda, theta, dy, dfinal, dx, ddt, dA, dB, dC,
                                                  dlambda, dtheta, workspace, s)
                              : launch_bwd<__nv_bfloat16>(d, x, dt, A, B, C, lambda, theta, dy, dfinal, dx, ddt, dA,
                                                          dB, dC, dlambda, dtheta, workspace, s);
}

size_t m3_scan_workspace_size(const m3_dims* d) {
    (void)d;
    return 0;
}

int m3_scan_algorithm(const m3_dims* d) { return scan_algorithm(d); }

int m3_scan_fwd_from(const m3_dims* d, const void* x, const float* dt, const float* A, const void* B, const void* C,
                     const float* lambda, const void* theta, const float* initial_state, const void* prev_B,
                     const void* prev_x, void* y, float* final_state, void* workspace, size_t workspace_bytes,
                     void* stream) {
    int rc = check_dims(d, true);
    if (rc != M3_OK) return rc;
    (void)workspace;
    (void)workspace_bytes;
    const bool has_tokens = d->batch > 0 && d->seqlen > 0;
    if (has_tokens && (!x || !dt || !A || !B || !C || !y)) return M3_ERR_NULL;
    if (d->batch > 0 && !A) return M3_ERR_NULL;
    if ((prev_B == nullptr) != (prev_x == nullptr)) return M3_ERR_NULL;
    const uintptr_t es = d->dtype == M3_F32 ? 4 : 2;
    const void* elem_ptrs[] = {x, B, C, theta, y, prev_B, prev_x};
    for (const void* p : elem_ptrs)
        if (p && !aligned(p, es)) return M3_ERR_ALIGN;
    const void* f32_ptrs[] = {dt, A, lambda};
    for (const void* p : f32_ptrs)
        if (p && !aligned(p, 4)) return M3_ERR_ALIGN;
    if (final_state && !aligned16(final_state)) return M3_ERR_ALIGN;
    if (initial_state && !aligned16(initial_state)) return M3_ERR_ALIGN;
    const int algo = scan_algorithm(d);
    if (algo == M3_ALGO_NONE) return M3_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d->batch == 0) return M3_OK;
    const size_t state_bytes = sizeof(float) * d->batch * d->heads * d->dstate * d->headdim;
    if (d->seqlen == 0) {
        // no token: the state passes through unchanged (the previous token's
        // input is carried by the caller, not folded into the state)
        if (!final_state) return M3_OK;
        const cudaError_t e = initial_state
                                  ? cudaMemcpyAsync(final_state, initial_state, state_bytes, cudaMemcpyDeviceToDevice, s)
                                  : cudaMemsetAsync(final_state, 0, state_bytes, s);
        return e == cudaSuccess ? M3_OK : M3_ERR_CUDA;
    }
    if (algo == M3_ALGO_CHUNKED_TC)
        return m3ws::launch(*d, x, dt, A, B, C, lambda, theta, initial_state, prev_B, prev_x, y, final_state, s);
    if (algo == M3_ALGO_CHUNKED_SIMT)
        return d->dtype == M3_F32
                   ? launch_chunk<float>(d, x, dt, A, B, C, lambda, theta, y, final_state, initial_state, prev_B,
                                         prev_x, s)
                   : launch_chunk<__nv_bfloat16>(d, x, dt, A, B, C, lambda, theta, y, final_state, initial_state,
                                                 prev_B, prev_x, s);
    if (d->dtype == M3_F32)
        return dispatch_seq<float>(d, x, dt, A, B, C, lambda, theta, y, final_state, initial_state, prev_B, prev_x, s);
    return dispatch_seq<__nv_bfloat16>(d, x, dt, A, B, C, lambda, theta, y, final_state, initial_state, prev_B, prev_x,
                                       s);
}

int m3_scan_fwd(const m3_dims* d, const void* x, const float* dt, const float* A, const void* B, const void* C,
                const float* lambda, const void* theta, void* y, float* final_state, void* workspace,
                size_t workspace_bytes, void* stream) {
    return m3_scan_fwd_from(d, x, dt, A, B, C, lambda, theta, nullptr, nullptr, nullptr, y, final_state, workspace,
                            workspace_bytes, stream);
}

int m3_scan_fwd_bcnorm(const m3_dims* d, const void* x, const float* dt, const float* A, const void* B,
                       const void* C, const float* lambda, const void* theta, const float* norm_B, const float* norm_C,
                       const float* bias_B, const float* bias_C, float eps, void* y, float* final_state,
                       void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_dims(d, true);
    if (rc != M3_OK) return rc;
    (void)workspace;
    (void)workspace_bytes;
    const bool has_tokens = d->batch > 0 && d->seqlen > 0;
    if (has_tokens && (!x || !dt || !A || !B || !C || !y)) return M3_ERR_NULL;
    if (!norm_B || !norm_C || !bias_B || !bias_C) return M3_ERR_NULL;
    if (!(eps >= 0.0f) || eps == INFINITY) return M3_ERR_VALUE;
    const uintptr_t es = d->dtype == M3_F32 ? 4 : 2;
    const void* elem_ptrs[] = {x, B, C, theta, y};
    for (const void* p : elem_ptrs)
        if (p && !aligned(p, es)) return M3_ERR_ALIGN;
    const void* f32_ptrs[] = {dt, A, lambda, norm_B, norm_C, bias_B, bias_C};
    for (const void* p : f32_ptrs)
        if (p && !aligned(p, 4)) return M3_ERR_ALIGN;
    if (final_state && !aligned16(final_state)) return M3_ERR_ALIGN;
    if (scan_algorithm(d) != M3_ALGO_CHUNKED_TC) return M3_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d->batch == 0) return M3_OK;
    if (d->seqlen == 0) {
        if (!final_state) return M3_OK;
        const size_t state_bytes = sizeof(float) * d->batch * d->heads * d->dstate * d->headdim;
        return cudaMemsetAsync(final_state, 0, state_bytes, s) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
    }
    return m3ws::launch(*d, x, dt, A, B, C, lambda, theta, nullptr, nullptr, nullptr, y, final_state, s, norm_B, norm_C,
                        bias_B, bias_C, eps);
}

int m3_step(const m3_dims* d, float* state, const void* x_t, const float* dt_t, const float* A, const void* B_t,
            const void* C_t, const float* lambda_t, const void* theta_t, const void* prev_B, const void* prev_x,
            void* y_t, void* stream) {
    int rc = check_dims(d, false);
    if (rc != M3_OK) return rc;
    if (d->batch > 0 && (!state || !x_t || !dt_t || !A || !B_t || !C_t || !y_t)) return M3_ERR_NULL;
    if ((prev_B == nullptr) != (prev_x == nullptr)) return M3_ERR_NULL;
    const uintptr_t es = d->dtype == M3_F32 ? 4 : 2;
    const void* elem_ptrs[] = {x_t, B_t, C_t, theta_t, prev_B, prev_x, y_t};
    for (const void* p : elem_ptrs)
        if (p && !aligned(p, es)) return M3_ERR_ALIGN;
    const void* f32_ptrs[] = {dt_t, A, lambda_t};
    for (const void* p : f32_ptrs)
        if (p && !aligned(p, 4)) return M3_ERR_ALIGN;
    if (state && !aligned16(state)) return M3_ERR_ALIGN;
    if (m3fast::supports(d->dstate, d->headdim, d->rank)) {
        const void* vec_ptrs[] = {state, x_t, B_t, C_t, theta_t, prev_B, prev_x};
        bool ok16 = true;
        for (const void* p : vec_ptrs) ok16 = ok16 && (!p || aligned16(p));
        if (ok16) {
            if (d->batch == 0) return M3_OK;
            cudaStream_t s = static_cast<cudaStream_t>(stream);
            if (m3ring::supports(d->dstate, d->headdim, d->rank, (int)es))
                return d->dtype == M3_F32
                           ? launch_step_ring<float>(d, state, x_t, dt_t, A, B_t, C_t, lambda_t, theta_t, prev_B,
                                                     prev_x, y_t, s)
                           : launch_step_ring<__nv_bfloat16>(d, state, x_t, dt_t, A, B_t, C_t, lambda_t, theta_t,
                                                             prev_B, prev_x, y_t, s);
            return d->dtype == M3_F32
                       ? launch_step_fast<float>(d, state, x_t, dt_t, A, B_t, C_t, lambda_t, theta_t, prev_B, prev_x,
                                                 y_t, s)
                       : launch_step_fast<__nv_bfloat16>(d, state, x_t, dt_t, A, B_t, C_t, lambda_t, theta_t, prev_B,
                                                         prev_x, y_t, s);
        }
    }
    SimtArgs a;
    int npt, block;
    if (!simt_geometry(d, &a, &npt, &block) || step_smem_bytes(a) > kMaxSmem) return M3_ERR_UNSUPPORTED;
    if (d->batch == 0) return M3_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d->dtype == M3_F32)
        return dispatch_step<float>(d, state, x_t, dt_t, A, B_t, C_t, lambda_t, theta_t, prev_B, prev_x, y_t, s);
    return dispatch_step<__nv_bfloat16>(d, state, x_t, dt_t, A, B_t, C_t, lambda_t, theta_t, prev_B, prev_x, y_t,
                                        s);
}

int m3_step_k(const m3_dims* d, float* state, const void* x, const float* dt, const float* A, const void* B,
              const void* C, const float* lambda, const void* theta, const void* prev_B, const void* prev_x, void* y,
              void* stream) {
    int rc = check_dims(d, false);
    if (rc != M3_OK) return rc;
    const bool work = d->batch > 0 && d->seqlen > 0;
    if (work && (!state || !x || !dt || !A || !B || !C || !y)) return M3_ERR_NULL;
    if ((prev_B == nullptr) != (prev_x == nullptr)) return M3_ERR_NULL;
    const uintptr_t es = d->dtype == M3_F32 ? 4 : 2;
    const void* elem_ptrs[] = {x, B, C, theta, prev_B, prev_x, y};
    for (const void* p : elem_ptrs)
        if (p && !aligned(p, es)) return M3_ERR_ALIGN;
    const void* f32_ptrs[] = {dt, A, lambda};
    for (const void* p : f32_ptrs)
        if (p && !aligned(p, 4)) return M3_ERR_ALIGN;
    if (state && !aligned16(state)) return M3_ERR_ALIGN;
    if (!work) return M3_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (m3fast::supports(d->dstate, d->headdim, d->rank)) {
        const void* vec_ptrs[] = {state, x, B, C, theta, prev_B, prev_x};
        bool ok16 = true;
        for (const void* p : vec_ptrs) ok16 = ok16 && (!p || aligned16(p));
        if (ok16)
            return d->dtype == M3_F32
                       ? launch_step_k<float>(d, state, x, dt, A, B, C, lambda, theta, prev_B, prev_x, y, s)
                       : launch_step_k<__nv_bfloat16>(d, state, x, dt, A, B, C, lambda, theta, prev_B, prev_x, y, s);
    }
    // other shapes: the continued prefill with the state as both its initial and
    // its final state (every prefill kernel reads a (b, h) state before it
    // writes it, in the same CTA), in chunks of the CUDA-core kernels
    m3_dims dc = *d;
    dc.chunk = (16 * d->rank == m3ws::kRows) ? 32 : 16;
    return m3_scan_fwd_from(&dc, x, dt, A, B, C, lambda, theta, state, prev_B, prev_x, y, state, nullptr, 0,
                            stream);
}

// ---------------------------------------------------------------------------
// Backward pass without caller-provided workspace, for callers that cannot
// allocate device memory (a host whose allocator belongs to another runtime or
// framework, a process running under a fixed memory budget, code that must not
// touch the allocator inside a serving loop).  Its scratch is one fixed array in
// this library's device image: every GPU that loads the library holds it until
// the process exits.
}  // extern "C"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB
static __device__ __align__(256) uint8_t g_bwd_scratch[kNoAllocScratchBytes];

// The context current on the calling thread (driver API, looked up once through
// the runtime): the per-device caches below are keyed by it, so that a device
// reset (a new primary context, where the old addresses and handles are void)
// makes them look up again instead of using stale ones.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
int current_context(CUcontext* out) {
    static CtxGetCurrentFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p)
            return M3_ERR_CUDA;
        fn = reinterpret_cast<CtxGetCurrentFn>(p);
    }
    if (fn(out) == CUDA_SUCCESS && *out) return M3_OK;
    // no context current on this thread yet: the runtime makes the device's primary one
    if (cudaFree(nullptr) != cudaSuccess) return M3_ERR_CUDA;
    return fn(out) == CUDA_SUCCESS && *out ? M3_OK : M3_ERR_CUDA;
}

// The device address of g_bwd_scratch, looked up once per device and context
// with that device current (in host code the array's name is a host-side
// stand-in, not a device address).
constexpr int kMaxScratchDevices = 256;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxScratchDevices];
CUcontext g_scratch_ctx[kMaxScratchDevices];

int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return M3_ERR_CUDA;
    if (dev < 0 || dev >= kMaxScratchDevices) return M3_ERR_UNSUPPORTED;
    CUcontext ctx = nullptr;
    if (current_context(&ctx) != M3_OK) return M3_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) return M3_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_addr[dev];
    return M3_OK;
}

}  // namespace

extern "C" {

int m3_scan_bwd_noalloc(const m3_dims* d, const void* x, const float* dt, const float* A, const void* B,
                        const void* C, const float* lambda, const void* theta, const void* dy, const float* dfinal,
                        void* dx, float* ddt, float* dA, void* dB, void* dC, float* dlambda, void* dtheta,
                        void* stream) {
    const int rc = check_dims(d, true);
    if (rc != M3_OK) return rc;
    const bool has_tokens = d->batch > 0 && d->seqlen > 0;
    if (has_tokens && bwd_supported(d) &&
        m3bwd::work_bytes(d->batch * d->heads, bwd_geo(d)) > kNoAllocScratchBytes)
        return M3_ERR_WORKSPACE;   // these sizes need more than the fixed scratch holds
    void* scratch = nullptr;
    if (has_tokens) {
        const int src = scratch_address(&scratch);
        if (src != M3_OK) return src;
    }
    return m3_scan_bwd(d, x, dt, A, B, C, lambda, theta, dy, dfinal, dx, ddt, dA, dB, dC, dlambda, dtheta, scratch,
                       has_tokens ? kNoAllocScratchBytes : 0, stream);
}

}  // extern "C"

namespace {

// ---- prefill from and to host memory (m3_scan_fwd_host)
// Per slice of the batch a staging set in the caller's workspace: the inputs
// x, dt, B, C, lambda, theta and the outputs y, final_state of `slice` batch
// rows; two sets used in turn, after the heads' A.
inline size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

struct HostSet {
    size_t x, dt, B, C, lam, th, y, fs, bytes;   // byte offsets inside a set; its size
};

HostSet host_set(const m3_dims* d, int64_t slice) {
    const size_t es = d->dtype == M3_F32 ? 4 : 2;
    const size_t units = (size_t)slice * d->seqlen * d->heads;   // (b, t, h) of one slice
    HostSet hs;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += up256(bytes);
        return at;
    };
    hs.x = take(units * d->rank * d->headdim * es);
    hs.dt = take(units * 4);
    hs.B = take(units * d->rank * d->dstate * es);
    hs.C = take(units * d->rank * d->dstate * es);
    hs.lam = take(units * 4);
    hs.th = take(units * (d->dstate / 2) * es);
    hs.y = take(units * d->rank * d->headdim * es);
    hs.fs = take((size_t)slice * d->heads * d->dstate * d->headdim * 4);
    hs.bytes = o;
    return hs;
}

// batch rows per slice: as asked (at most the batch), or an eighth of the batch
int64_t host_slice(const m3_dims* d, int64_t slice) {
    const int64_t b = d->batch > 0 ? d->batch : 1;
    if (slice > 0) return slice < b ? slice : b;
    return (b + 7) / 8;
}

size_t host_ws_bytes(const m3_dims* d, int64_t slice) {
    return up256((size_t)d->heads * 4) + 2 * host_set(d, slice).bytes;
}

// The library's two copy streams (host to device, device to host) and its
// events, per device: made on the device's first call and kept (handles only,
// no device memory).  A call holds g_pipe_mu while it enqueues, so that calls
// from several host threads do not interleave their event records.  (Splitting
// a slice's uploads over two streams measured the same: the host-to-device
// copies are bound by the link, not by one copy engine.)
struct HostPipe {
    CUcontext ctx = nullptr;   // the context the handles belong to
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t fork = nullptr, in[2] = {nullptr, nullptr}, done[2] = {nullptr, nullptr},
                out[2] = {nullptr, nullptr};
};
constexpr int kMaxPipeDevices = 256;
std::mutex g_pipe_mu;
HostPipe g_pipe[kMaxPipeDevices];

int pipe_for(int dev, HostPipe** out) {
    HostPipe& p = g_pipe[dev];
    CUcontext ctx = nullptr;
    if (current_context(&ctx) != M3_OK) return M3_ERR_CUDA;
    // handles made in an earlier context (before a device reset) are void: made again
    // (the old ones went with their context)
    if (!p.up || p.ctx != ctx) {
        HostPipe q;
        q.ctx = ctx;
        bool ok = cudaStreamCreateWithFlags(&q.up, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&q.down, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&q.fork, cudaEventDisableTiming) == cudaSuccess;
        for (int k = 0; k < 2 && ok; ++k)
            ok = cudaEventCreateWithFlags(&q.in[k], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&q.done[k], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&q.out[k], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            cudaEvent_t evs[] = {q.fork, q.in[0], q.in[1], q.done[0], q.done[1], q.out[0], q.out[1]};
            for (cudaEvent_t e : evs)
                if (e) cudaEventDestroy(e);
            if (q.up) cudaStreamDestroy(q.up);
            if (q.down) cudaStreamDestroy(q.down);
            return M3_ERR_CUDA;
        }
        p = q;
    }
    *out = &p;
    return M3_OK;
}

}  // namespace

extern "C" {

size_t m3_scan_fwd_host_workspace_size(const m3_dims* d, int64_t slice) {
    if (check_dims(d, true) != M3_OK || slice < 0 || d->batch == 0) return 0;
    return host_ws_bytes(d, host_slice(d, slice));
}

int m3_scan_fwd_host(const m3_dims* d, const void* x, const float* dt, const float* A, const void* B, const void* C,
                     const float* lambda, const void* theta, void* y, float* final_state, int64_t slice,
                     void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_dims(d, true);
    if (rc != M3_OK) return rc;
    if (slice < 0) return M3_ERR_VALUE;
    const bool has_tokens = d->batch > 0 && d->seqlen > 0;
    if (has_tokens && (!x || !dt || !B || !C || !y)) return M3_ERR_NULL;
    if (d->batch > 0 && !A) return M3_ERR_NULL;
    const uintptr_t es = d->dtype == M3_F32 ? 4 : 2;
    const void* elem_ptrs[] = {x, B, C, theta, y};
    for (const void* p : elem_ptrs)
        if (p && !aligned(p, es)) return M3_ERR_ALIGN;
    const void* f32_ptrs[] = {dt, A, lambda, final_state};
    for (const void* p : f32_ptrs)
        if (p && !aligned(p, 4)) return M3_ERR_ALIGN;
    if (scan_algorithm(d) == M3_ALGO_NONE) return M3_ERR_UNSUPPORTED;
    if (d->batch == 0) return M3_OK;
    const int64_t sl = host_slice(d, slice);
    if (!workspace || workspace_bytes < host_ws_bytes(d, sl)) return M3_ERR_WORKSPACE;
    if (((uintptr_t)workspace & 255) != 0) return M3_ERR_ALIGN;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return M3_ERR_CUDA;
    if (dev < 0 || dev >= kMaxPipeDevices) return M3_ERR_UNSUPPORTED;

    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe* p = nullptr;
    rc = pipe_for(dev, &p);
    if (rc != M3_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const HostSet hs = host_set(d, sl);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* A_d = reinterpret_cast<float*>(ws);
    uint8_t* sets = ws + up256((size_t)d->heads * 4);
    // bytes per batch row of each array
    const size_t th_units = (size_t)d->seqlen * d->heads;
    const size_t r_x = th_units * d->rank * d->headdim * es, r_f = th_units * 4;
    const size_t r_B = th_units * d->rank * d->dstate * es, r_th = th_units * (d->dstate / 2) * es;
    const size_t r_fs = (size_t)d->heads * d->dstate * d->headdim * 4;
    const auto up = cudaMemcpyHostToDevice, down = cudaMemcpyDeviceToHost;
    bool ok = true;
    auto chk = [&](cudaError_t e) { ok = ok && e == cudaSuccess; };
    auto at = [](const void* base, size_t off) { return static_cast<const uint8_t*>(base) + off; };

    // the workspace is free once the caller's earlier work on `stream` is done
    chk(cudaEventRecord(p->fork, s));
    chk(cudaStreamWaitEvent(p->up, p->fork, 0));
    chk(cudaMemcpyAsync(A_d, A, (size_t)d->heads * 4, up, p->up));
    const int64_t nsl = (d->batch + sl - 1) / sl;
    int scan_rc = M3_OK;
    int64_t last = -1;
    for (int64_t i = 0; i < nsl && ok && scan_rc == M3_OK; ++i) {
        const int k = (int)(i & 1);
        const int64_t b0 = i * sl, nb = (d->batch - b0) < sl ? (d->batch - b0) : sl;
        uint8_t* st = sets + k * hs.bytes;
        // host -> device, once the set's previous slice has been read back
        if (i >= 2) chk(cudaStreamWaitEvent(p->up, p->out[k], 0));
        if (has_tokens) {
            chk(cudaMemcpyAsync(st + hs.x, at(x, b0 * r_x), nb * r_x, up, p->up));
            chk(cudaMemcpyAsync(st + hs.dt, at(dt, b0 * r_f), nb * r_f, up, p->up));
            chk(cudaMemcpyAsync(st + hs.B, at(B, b0 * r_B), nb * r_B, up, p->up));
            chk(cudaMemcpyAsync(st + hs.C, at(C, b0 * r_B), nb * r_B, up, p->up));
            if (lambda) chk(cudaMemcpyAsync(st + hs.lam, at(lambda, b0 * r_f), nb * r_f, up, p->up));
            if (theta) chk(cudaMemcpyAsync(st + hs.th, at(theta, b0 * r_th), nb * r_th, up, p->up));
        }
        chk(cudaEventRecord(p->in[k], p->up));
        // the slice's scan on the caller's stream
        chk(cudaStreamWaitEvent(s, p->in[k], 0));
        if (!ok) break;
        m3_dims ds = *d;
        ds.batch = nb;
        scan_rc = m3_scan_fwd(&ds, st + hs.x, reinterpret_cast<const float*>(st + hs.dt), A_d, st + hs.B,
                              st + hs.C, lambda ? reinterpret_cast<const float*>(st + hs.lam) : nullptr,
                              theta ? st + hs.th : nullptr, st + hs.y,
                              final_state ? reinterpret_cast<float*>(st + hs.fs) : nullptr, nullptr, 0, stream);
        chk(cudaEventRecord(p->done[k], s));
        // device -> host
        chk(cudaStreamWaitEvent(p->down, p->done[k], 0));
        if (has_tokens) chk(cudaMemcpyAsync(static_cast<uint8_t*>(y) + b0 * r_x, st + hs.y, nb * r_x, down, p->down));
        if (final_state)
            chk(cudaMemcpyAsync(reinterpret_cast<uint8_t*>(final_state) + b0 * r_fs, st + hs.fs, nb * r_fs, down,
                                p->down));
        chk(cudaEventRecord(p->out[k], p->down));
        last = i;
    }
    // `stream` completes after both copy streams (each in order): the last read-back
    // and every copy into the workspace
    if (last >= 0) chk(cudaStreamWaitEvent(s, p->out[last & 1], 0));
    chk(cudaEventRecord(p->fork, p->up));
    chk(cudaStreamWaitEvent(s, p->fork, 0));
    if (scan_rc != M3_OK) return scan_rc;
    return ok ? M3_OK : M3_ERR_CUDA;
}

int m3_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return M3_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, m3::g_status, sizeof(v)) != cudaSuccess) return M3_ERR_CUDA;
    if (v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(m3::g_status, &zero, sizeof(zero)) != cudaSuccess) return M3_ERR_CUDA;
        return M3_ERR_DEVICE;
    }
    return M3_OK;
}

int m3_selftest_wait_timeout(long long budget_cycles, void* stream) {
    if (budget_cycles < 1 || budget_cycles > 4000000000LL) return M3_ERR_VALUE;
    m3::m3_wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(budget_cycles);
    return launch_status();
}

const char* m3_status_string(int status) {
    switch (status) {
        case M3_OK: return "ok";
        case M3_ERR_NULL: return "a required pointer is NULL";
        case M3_ERR_SHAPE: return "a size is out of range";
        case M3_ERR_DTYPE: return "unknown dtype";
        case M3_ERR_ALIGN: return "a pointer is not aligned as required";
        case M3_ERR_CUDA: return "a CUDA call or kernel launch failed";
        case M3_ERR_UNSUPPORTED: return "no kernel for these sizes";
        case M3_ERR_DEVICE: return "a kernel reported a device-side error";
        case M3_ERR_WORKSPACE: return "workspace too small";
        case M3_ERR_VALUE: return "a scalar argument is out of range";
    }
    return "unknown status";
}

}  // extern "C"
