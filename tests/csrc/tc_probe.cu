// tc_probe.cu -- unit tests of the library's tcgen05 / TMA wrappers
// (selective_state_space_131_b300/csrc/ptx_sm100.cuh): one CTA runs a single
// UMMA with operands staged in 128-byte-swizzled shared memory in either
// K-major or MN-major layout, and dumps all 128 TMEM lanes; a second kernel
// loads a tile with TMA (128-byte swizzle) and dumps the shared-memory image.
// Built by tests/test_tc_wrappers.py; every index is bounded by the sizes
// checked in the host functions below.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx_sm100.cuh"

namespace {

constexpr int kThreads = 128;

// A tile of `rows` (M or N index) x K, bf16, K-major: slab s of 64 K holds
// rows x 128 bytes.  MN-major: block m of 64 rows holds K x 128 bytes.
__device__ uint32_t tile_offset(int mode, int rows, int K, int r, int k) {
    if (mode == 0) return (uint32_t)(k / 64) * rows * 128u + ptx::sw128_offset(r, k % 64);
    if (mode == 2) return ptx::sw64_offset(k, r);   // MN-major, 64-byte swizzle, rows = 32
    return (uint32_t)(r / 64) * K * 128u + ptx::sw128_offset(k, r % 64);
}

// First 1024-byte-aligned address (in the shared window) of the dynamic buffer.
__device__ uint8_t* align1024(uint8_t* p) {
    const uint32_t s = ptx::smem_u32(p);
    return p + ((1024u - (s & 1023u)) & 1023u);
}

__global__ void umma_probe_kernel(int M, int N, int K, int a_mn, int b_mn, int half_split,
                                  const __nv_bfloat16* A, const __nv_bfloat16* B, float* D, unsigned* status) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    uint8_t* sa = smem;                                  // M x K
    uint8_t* sb = smem + (size_t)M * K * 2;              // N x K (1024-aligned: M*K*2 is)
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

    for (int i = tid; i < M * K; i += kThreads) {
        const int r = i / K, k = i % K;
        *reinterpret_cast<__nv_bfloat16*>(sa + tile_offset(a_mn, M, K, r, k)) = A[i];
    }
    for (int i = tid; i < N * K; i += kThreads) {
        const int r = i / K, k = i % K;
        *reinterpret_cast<__nv_bfloat16*>(sb + tile_offset(b_mn, N, K, r, k)) = B[i];
    }
    ptx::fence_proxy_async_smem();
    if (tid == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(&tmem_base, 256);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (tid == 0) {
        const uint32_t a0 = ptx::smem_u32(sa), b0 = ptx::smem_u32(sb);
        const uint32_t idesc = ptx::idesc_bf16(M, N, a_mn != 0, b_mn != 0);   // b_mn 2: MN-major too
        for (int k16 = 0; k16 < K / 16; ++k16) {
            uint64_t ad, bd;
            if (a_mn) ad = ptx::sdesc_sw128(a0 + k16 * 2048u, (uint32_t)K * 128u, 1024u);
            else ad = ptx::sdesc_sw128(a0 + (k16 / 4) * M * 128u + (k16 % 4) * 32u, 16u, 1024u);
            if (b_mn == 2) bd = ptx::sdesc_sw64(b0 + k16 * 1024u, 64u, 512u);
            else if (b_mn) bd = ptx::sdesc_sw128(b0 + k16 * 2048u, (uint32_t)K * 128u, 1024u);
            else bd = ptx::sdesc_sw128(b0 + (k16 / 4) * N * 128u + (k16 % 4) * 32u, 16u, 1024u);
            ptx::umma_bf16(tmem, ad, bd, idesc, k16 > 0 ? 1u : 0u);
        }
        ptx::umma_commit(&bar);
    }
    __syncwarp();
    const bool ok = ptx::mbar_wait(&bar, 0, 2000000000LL);
    if (!ok && lane == 0) atomicOr(status, 1u);
    ptx::tc_fence_after();
    if (ok && !half_split) {
        for (int c = 0; c < N; c += 16) {
            uint32_t v[16];
            ptx::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);   // N is a multiple of 16
            ptx::tmem_ld_wait();
            for (int j = 0; j < 16; ++j) D[(size_t)(warp * 32 + lane) * N + c + j] = __uint_as_float(v[j]);
        }
    } else if (ok) {
        // 16x32bx2: thread t < 16 -> lane t, columns [c, c+32); t >= 16 -> lane t-16, [c+32, c+64).
        // Written to D row (16 * warp + t % 16) of an M-row image.
        for (int c = 0; c < N; c += 64) {
            uint32_t v[32];
            ptx::tmem_ld16x2_32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);
            ptx::tmem_ld_wait();
            const int row = warp * 16 + (lane & 15), c0 = c + (lane >> 4) * 32;
            for (int j = 0; j < 32; ++j) D[(size_t)row * N + c0 + j] = __uint_as_float(v[j]);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, 256);
}

__global__ void tma_probe_kernel(const __grid_constant__ CUtensorMap map, int rows, int c1, int c2,
                                 uint8_t* out, unsigned* status) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const uint32_t bytes = (uint32_t)rows * 128u;
    if (threadIdx.x == 0) {
        ptx::mbar_arrive_expect_tx(&bar, bytes);
        ptx::tma_load_3d(smem, &map, &bar, 0, c1, c2);
    }
    const bool ok = ptx::mbar_wait(&bar, 0, 2000000000LL);
    if (!ok) {
        if (threadIdx.x == 0) atomicOr(status, 1u);
        return;
    }
    for (uint32_t i = threadIdx.x; i < bytes; i += blockDim.x) out[i] = smem[i];
}

}  // namespace

extern "C" {

// D[128][N] <- TMEM lanes x columns after D = A[M][K] * B[N][K]^T; with
// half_split (M = 64 only) D[64][N] <- the rows read with the 16x32bx2 shape.
// M in {64, 128}, N in {64, 128, 256}, K in {64, 128}; MN-major needs
// M (or N) a multiple of 64.  Returns a cudaError_t, or -1 for bad sizes.
__attribute__((visibility("default"))) int probe_umma(int M, int N, int K, int a_mn, int b_mn, int half_split,
                                                      const void* A, const void* B, float* D,
                                                      unsigned* status) {
    if (!(M == 64 || M == 128) || !(N == 32 || N == 64 || N == 128 || N == 256) || !(K == 64 || K == 128)) return -1;
    if (half_split && M != 64) return -1;
    if ((b_mn == 2) != (N == 32)) return -1;   // the 64-byte-swizzled operand is 32 wide
    const size_t smem = (size_t)(M + N) * K * 2 + 1024;
    cudaFuncSetAttribute(umma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    umma_probe_kernel<<<1, kThreads, smem>>>(M, N, K, a_mn, b_mn, half_split, (const __nv_bfloat16*)A,
                                             (const __nv_bfloat16*)B, D, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    return (int)cudaDeviceSynchronize();
}

// TMA load of a [rows][64] bf16 box at coordinates (0, c1, c2) of a 3D tensor
// [d2][d1][64] (row stride 128 bytes) with 128-byte swizzle; the raw
// shared-memory image (rows * 128 bytes) goes to out.
__attribute__((visibility("default"))) int probe_tma(const void* src, int d1, int d2, int rows, int c1, int c2,
                                                     uint8_t* out, unsigned* status) {
    if (rows < 1 || rows > 256 || d1 < 1 || d2 < 1) return -1;
    typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || !fn)
        return -2;
    CUtensorMap map;
    cuuint64_t dims[3] = {64, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t strides[2] = {128, (cuuint64_t)d1 * 128};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = ((EncodeFn)fn)(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(src), dims, strides,
                                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return -3;
    const size_t smem = (size_t)rows * 128 + 1024;
    cudaFuncSetAttribute(tma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    tma_probe_kernel<<<1, 128, smem>>>(map, rows, c1, c2, out, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    return (int)cudaDeviceSynchronize();
}

}  // extern "C"
