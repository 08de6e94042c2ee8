// Test-only probe of the tcgen05 building blocks used by libkda: one CTA loads
// A and B from global memory into 128B-swizzled shared-memory tiles in the
// K-major or MN-major layouts the KDA kernel uses, runs D = A*B with
// tcgen05.mma (M = 128, bf16 in, fp32 out), and copies D out of tensor memory.
// The pytest suite compares D with torch.matmul.  A second probe runs the bounded
// mbarrier wait on a barrier nothing completes, to check that it gives up.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../gated_delta_rule_52_gb300/csrc/sm103.cuh"

using namespace kda::sm103;

namespace {

constexpr int M = 128;

// A: row-major [M][K] in global.  B: row-major [K][N] in global.  The MMA runs with
// mma_m rows (64 or 128; with 64 it reads the first 64 rows of the A tile); D returns
// all 128 TMEM lanes, which start out NaN.
__global__ void __launch_bounds__(128, 1)
probe_kernel(const __nv_bfloat16 *A, const __nv_bfloat16 *B, float *D, int N, int K, int a_mn,
             int b_mn, int fp16, int *status, int mma_m) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *sA = smem;                      // M*K*2 bytes
    unsigned char *sB = smem + M * K * 2;          // N*K*2 bytes
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // A tile
    for (int idx = tid; idx < M * K; idx += blockDim.x) {
        const int m = idx / K, k = idx % K;
        uint32_t off;
        if (!a_mn) off = (k / 64) * (M * 128) + sw128_off(m, k % 64);       // K-major [m][k]
        else off = (m / 64) * (K * 128) + sw128_off(k, m % 64);             // MN-major [k][m]
        if (fp16) *reinterpret_cast<__half *>(sA + off) = __float2half_rn(__bfloat162float(A[idx]));
        else *reinterpret_cast<__nv_bfloat16 *>(sA + off) = A[idx];
    }
    for (int idx = tid; idx < K * N; idx += blockDim.x) {
        const int k = idx / N, n = idx % N;
        uint32_t off;
        if (!b_mn) off = (k / 64) * (N * 128) + sw128_off(n, k % 64);       // K-major [n][k]
        else off = (n / 64) * (K * 128) + sw128_off(k, n % 64);             // MN-major [k][n]
        if (fp16) *reinterpret_cast<__half *>(sB + off) = __float2half_rn(__bfloat162float(B[idx]));
        else *reinterpret_cast<__nv_bfloat16 *>(sB + off) = B[idx];
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    {
        float nanv[16];
        for (int j = 0; j < 16; ++j) nanv[j] = __int_as_float(0x7fc00000);
        for (int c0 = 0; c0 < N; c0 += 16) tmem_st16(tmem_addr(tbase, warp * 32, c0), nanv);
        tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid == 0) {
        const uint32_t idesc = idesc_f16kind(mma_m, N, a_mn != 0, b_mn != 0, fp16 != 0);
        const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
        for (int ks = 0; ks < K / 16; ++ks) {
            uint64_t ad, bd;
            if (!a_mn) ad = sdesc_sw128(a0 + (ks / 4) * (M * 128) + (ks % 4) * 32, 16, 1024);
            else ad = sdesc_sw128(a0 + ks * 2048, K * 128, 1024);
            if (!b_mn) bd = sdesc_sw128(b0 + (ks / 4) * (N * 128) + (ks % 4) * 32, 16, 1024);
            else bd = sdesc_sw128(b0 + ks * 2048, K * 128, 1024);
            mma_bf16(tbase, ad, bd, idesc, ks > 0);
        }
        mma_commit(&bar);
    }
    if (!mbar_wait(&bar, 0, 2000000000ull)) {
        if (lane == 0) atomicExch(status, 1);
    }
    tc_fence_after();
    const int row = warp * 32 + lane;
    for (int c0 = 0; c0 < N; c0 += 16) {
        float r[16];
        tmem_ld16(tmem_addr(tbase, warp * 32, c0), r);
        tmem_ld_wait();
        for (int j = 0; j < 16; ++j) D[row * N + c0 + j] = r[j];
    }
    // TMEM store/load round trip on the last 16 columns (lane/column encoding).
    {
        float w[16], r[16];
        for (int j = 0; j < 16; ++j) w[j] = (float)(row * 1000 + j);
        tmem_st16(tmem_addr(tbase, warp * 32, 240), w);
        tmem_st_wait();
        tmem_ld16(tmem_addr(tbase, warp * 32, 240), r);
        tmem_ld_wait();
        for (int j = 0; j < 16; ++j)
            if (r[j] != w[j]) atomicExch(status, 2);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}

}  // namespace

extern "C" int kda_probe_mma_m(const void *A, const void *B, float *D, int mma_m, int N, int K,
                               int a_mn, int b_mn, int fp16, int *status, void *stream) {
    if (N < 16 || N > 256 || N % 16 || (b_mn && N % 64) || K < 16 || K > 128 || K % 64 ||
        (mma_m != 64 && mma_m != 128) || (mma_m == 64 && a_mn))
        return 1;
    const size_t smem = 1024 + (size_t)(M + N) * K * 2;
    cudaError_t e = cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return 2;
    probe_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16 *>(A), static_cast<const __nv_bfloat16 *>(B), D, N, K,
        a_mn, b_mn, fp16, status, mma_m);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int kda_probe_mma(const void *A, const void *B, float *D, int N, int K, int a_mn,
                             int b_mn, int fp16, int *status, void *stream) {
    return kda_probe_mma_m(A, B, D, 128, N, K, a_mn, b_mn, fp16, status, stream);
}

// ---------------------------------------------------------------------------
// TMA probe: one 3-D tiled load (box 64 channels x 1 head x 64 tokens, 128B
// swizzle) from a bf16 [T][H][128] tensor, read back through sw128_off.
#include <cuda.h>

namespace {

__global__ void tma_probe_kernel(const __grid_constant__ CUtensorMap tmap, int h, int t0, int c0,
                                 __nv_bfloat16 *out, int *status) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *tile = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&bar, 64 * 64 * 2);
        tma_load_3d(tile, &tmap, &bar, c0, h, t0);
    }
    if (!mbar_wait(&bar, 0, 2000000000ull)) {
        if (threadIdx.x == 0) atomicExch(status, 1);
        return;
    }
    for (int idx = threadIdx.x; idx < 64 * 64; idx += blockDim.x) {
        const int t = idx / 64, c = idx % 64;
        out[idx] = *reinterpret_cast<const __nv_bfloat16 *>(tile + sw128_off(t, c));
    }
}

// The bounded mbarrier wait every libkda kernel uses, on a barrier that nothing
// arrives on (arrive == 0) or that one thread has completed (arrive == 1): out[0] = 1
// if the wait succeeded, 2 if it gave up; out[1] = nanoseconds spent in it.
__global__ void wait_probe_kernel(unsigned long long limit_ns, int arrive, unsigned long long *out) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (arrive) mbar_arrive(&bar);
        const uint64_t t0 = globaltimer_ns();
        const bool ok = mbar_wait(&bar, 0, limit_ns);
        out[1] = globaltimer_ns() - t0;
        out[0] = ok ? 1ull : 2ull;
    }
}

}  // namespace

extern "C" int kda_probe_tma(const void *src, int T, int H, int h, int t0, int c0, void *out,
                             int *status, void *stream) {
    CUtensorMap tm;
    cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {256, (cuuint64_t)H * 256};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = cuTensorMapEncodeTiled(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                                        const_cast<void *>(src), dims, strides, box, estr,
                                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return 10 + (int)r;
    tma_probe_kernel<<<1, 128, 2048 + 8192, static_cast<cudaStream_t>(stream)>>>(
        tm, h, t0, c0, static_cast<__nv_bfloat16 *>(out), status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int kda_probe_wait(unsigned long long limit_ns, int arrive, unsigned long long *out,
                              void *stream) {
    if (limit_ns > 1000000000ull) return 1;   // at most 1 s
    wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, arrive, out);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
