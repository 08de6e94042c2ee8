// Device helpers shared by the chunked (UT/WY) prefill kernels: chunk constants,
// the decay-factor table indexing, mma.sync TF32 fragments of fp32 tiles, packed
// operand-row stores into 128B-swizzled tiles, the TMA tensor maps of the token
// tensors and the device error word.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace chunk {

using namespace sm103;

constexpr int C = kChunk;
constexpr int DK = kHeadDim;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWait = 2000000000ull;   // 2 s per wait
constexpr int LDA = 68;             // fp32 row stride of A and T (16-byte aligned rows)
constexpr int kFacRows = 14;       // rows of the per-chunk decay-factor table (fac_base)

// First row of the key variant of row block bt (rows of blocks 0..bt rescaled to the
// start of block bt) in the stacked variant operand.
__device__ __forceinline__ int variant_off(int bt) { return 8 * bt * (bt + 1); }

// mma.sync operand fragments (g = lane / 4, q = lane % 4) of a row-major fp32
// tile in shared memory: A (16 x 8) at a, B (8 x 8) at b.  The fp32 bit patterns
// go to the tf32 MMA as they are (it uses the leading 19 bits, i.e. truncates);
// an explicit round-to-nearest conversion cost 3.5% of the prefill time and moved
// the parity figures by at most a few percent of their size.
__device__ __forceinline__ void frag_a(const float *a, int lda, int lane, uint32_t (&f)[4]) {
    const int g = lane >> 2, q = lane & 3;
    f[0] = __float_as_uint(a[g * lda + q]);
    f[1] = __float_as_uint(a[(g + 8) * lda + q]);
    f[2] = __float_as_uint(a[g * lda + q + 4]);
    f[3] = __float_as_uint(a[(g + 8) * lda + q + 4]);
}
__device__ __forceinline__ void frag_b(const float *b, int ldb, int lane, uint32_t (&f)[2]) {
    const int g = lane >> 2, q = lane & 3;
    f[0] = __float_as_uint(b[q * ldb + g]);
    f[1] = __float_as_uint(b[(q + 4) * ldb + g]);
}

// Stores a 16 x 8 accumulator tile (times `sign`) at d (row stride ldd).
__device__ __forceinline__ void store_16x8(float *d, int ldd, int lane, const float (&acc)[4],
                                           float sign) {
    const int g = lane >> 2, q = lane & 3;
    d[g * ldd + 2 * q] = sign * acc[0];
    d[g * ldd + 2 * q + 1] = sign * acc[1];
    d[(g + 8) * ldd + 2 * q] = sign * acc[2];
    d[(g + 8) * ldd + 2 * q + 1] = sign * acc[3];
}

// Rows of the decay-factor table of one chunk (per 16-token block b and channel):
// fac_base(b) + 0: 2^Gs[b], + 1: 2^(G_C - Gs[b]), + 1 + (bt - b): 2^(Gs[bt] - Gs[b])
// for bt > b, with Gs[b] the cumulative log2 decay before block b and G_C the
// chunk total.
__device__ __forceinline__ int fac_base(int b) { return b * (11 - b) / 2; }

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool fp16) {
    return fp16 ? pack_f16(lo, hi) : pack_bf16(lo, hi);
}
template <bool FP16>
__device__ __forceinline__ void st_pack16(uint32_t base, int row, int col0, const float (&v)[16]) {
    sts128(base + sw128_off(row, col0), pack2(v[0], v[1], FP16), pack2(v[2], v[3], FP16),
           pack2(v[4], v[5], FP16), pack2(v[6], v[7], FP16));
    sts128(base + sw128_off(row, col0 + 8), pack2(v[8], v[9], FP16), pack2(v[10], v[11], FP16),
           pack2(v[12], v[13], FP16), pack2(v[14], v[15], FP16));
}

// fp16 operand range: true when x lies beyond +-65504 (or is NaN), where its fp16 copy
// would not hold it.
__device__ __forceinline__ bool f16_out(float x) { return !(fabsf(x) <= 65504.f); }
// st_pack16 that also records whether any value leaves the fp16 range (fp16 tiles only).
template <bool FP16>
__device__ __forceinline__ void st_pack16(uint32_t base, int row, int col0, const float (&v)[16], bool &bad) {
    if (FP16) {
#pragma unroll
        for (int e = 0; e < 16; ++e) bad |= f16_out(v[e]);
    }
    st_pack16<FP16>(base, row, col0, v);
}
// bf16 -> fp16 of a 16-byte vector in place, recording values beyond the fp16 range.
__device__ __forceinline__ uint4 bf16_to_f16x8(uint4 x, bool &bad) {
    const float a0 = bf16lo(x.x), a1 = bf16hi(x.x), b0 = bf16lo(x.y), b1 = bf16hi(x.y);
    const float c0 = bf16lo(x.z), c1 = bf16hi(x.z), d0 = bf16lo(x.w), d1 = bf16hi(x.w);
    bad |= f16_out(a0) | f16_out(a1) | f16_out(b0) | f16_out(b1) | f16_out(c0) | f16_out(c1) |
           f16_out(d0) | f16_out(d1);
    return make_uint4(pack_f16(a0, a1), pack_f16(b0, b1), pack_f16(c0, c1), pack_f16(d0, d1));
}

struct TmaMaps {
    CUtensorMap q, k, g, v;
};

// Records (first error wins) that this thread met a value beyond the fp16 operand range.
__device__ __forceinline__ void flag_range(const Params &p, bool bad) {
    if (bad && p.err) atomicCAS(p.err, 0, kErrRange);
}

__device__ __forceinline__ void set_err(const Params &p) {
    if (p.err) atomicExch(p.err, kErrTimeout);
}

// Host: the driver's tensor-map encoder and the 3-D tiled map of a [rows, H, 128] bf16
// token tensor (64 tokens x 64 channels per box, 128-byte swizzle).
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

inline bool encode_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t H) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)DK, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)DK * 2, (cuuint64_t)H * DK * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace chunk
}  // namespace kda
