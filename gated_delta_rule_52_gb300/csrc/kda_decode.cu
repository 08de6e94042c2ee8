// KDA forward for calls with few tokens per sequence (decode and short
// multi-token steps): the token recurrence applied directly, one token at a
// time, with the state held in registers.
//
// Per (sequence, head), with S the K x V state (FlashKDA README "Kernel API"
// semantics; the same activations as the chunked kernel):
//   S <- Diag(alpha_t) S;  u = beta_t (v_t - S^T k_hat_t);  S <- S + k_hat_t u^T;
//   out_t = scale * S^T q_hat_t
// which is S_t = (I - beta k k^T) Diag(alpha) S_{t-1} + beta k v^T written so that
// each state column needs only its own dot products.
//
// Work split: one CTA per (sequence, head, 32-column slice of V); 128 threads,
// thread = (state column v of the slice, 32-row group of K), so each thread keeps
// 32 fp32 state values in registers.  Per token the CTA computes the normalised
// q, k and the decay factors once (one channel per thread) into shared memory,
// then every thread updates its 32 values; the two column sums over K (S^T k and
// S^T q) combine the four row groups through shared memory.  The state crosses
// HBM once in and once out per call, which bounds the kernel for short steps.
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int DK = kHeadDim;
constexpr int VS = 32;                // state columns per CTA
constexpr int NTD = 128;              // threads per CTA
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf(const __nv_bfloat16 *p, int64_t i) { return __bfloat162float(p[i]); }

__global__ void __launch_bounds__(NTD) kda_decode_kernel(Params p) {
    __shared__ float alpha[DK], kn[DK], qn[DK];
    __shared__ float red[2][4][VS];
    __shared__ float nrm[2][4];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t unit = blockIdx.x / (DK / VS);
    const int vs = blockIdx.x % (DK / VS);
    const int64_t h = unit % p.H, n = unit / p.H;
    int64_t b, t0, len;
    seq_range(p, n, b, t0, len);
    const int64_t row_base = b * p.T + t0;

    const int v = vs * VS + lane;       // this thread's state column
    const int c0 = warp * 32;           // its 32 rows of K
    const size_t state_base = (size_t)(n * p.H + h) * DK * DK;
    float s[32];
    if (p.init) {
        if (p.state_type == kStateBF16) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                reinterpret_cast<const __nv_bfloat16 *>(p.init) + state_base + (size_t)v * DK + c0);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 w = src[i];
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[8 * i + 2 * j] = __uint_as_float(ws[j] << 16);
                    s[8 * i + 2 * j + 1] = __uint_as_float(ws[j] & 0xFFFF0000u);
                }
            }
        } else {
            const float4 *src = reinterpret_cast<const float4 *>(
                reinterpret_cast<const float *>(p.init) + state_base + (size_t)v * DK + c0);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 w = src[i];
                s[4 * i] = w.x; s[4 * i + 1] = w.y; s[4 * i + 2] = w.z; s[4 * i + 3] = w.w;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = 0.f;
    }

    // gate constants of this head for channel c = tid (log2 units)
    const float a2 = -__expf(p.A_log[h]) * kLog2e;
    const float b2 = a2 * p.dt_bias[h * DK + tid];
    const float lb2 = p.lower_bound * kLog2e;

    for (int64_t t = 0; t < len; ++t) {
        const int64_t row = row_base + t;
        const int64_t tok = (row * p.H + h) * DK;
        // activations of this token, one channel per thread
        const float qc = bf(p.q, tok + tid), kc = bf(p.k, tok + tid), gc = bf(p.g, tok + tid);
        const float beta = 1.f / (1.f + exp2f(-bf(p.beta, row * p.H + h) * kLog2e));
        const float vv = bf(p.v, tok + v);
        float sq = qc * qc, sk = kc * kc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
        }
        if (lane == 0) {
            nrm[0][warp] = sq;
            nrm[1][warp] = sk;
        }
        const float gk2 = lb2 * __fdividef(1.f, 1.f + exp2f(fmaf(gc, a2, b2)));
        alpha[tid] = exp2f(gk2);
        __syncthreads();
        const float rq = rsqrtf(nrm[0][0] + nrm[0][1] + nrm[0][2] + nrm[0][3] + 1e-6f);
        const float rk = rsqrtf(nrm[1][0] + nrm[1][1] + nrm[1][2] + nrm[1][3] + 1e-6f);
        kn[tid] = kc * rk;
        qn[tid] = qc * rq;
        __syncthreads();

        // decay, then the column sum S^T k_hat over this thread's 32 rows
        float ks = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            s[i] *= alpha[c0 + i];
            ks = fmaf(kn[c0 + i], s[i], ks);
        }
        red[0][warp][lane] = ks;
        __syncthreads();
        const float u = beta * (vv - (red[0][0][lane] + red[0][1][lane] + red[0][2][lane] + red[0][3][lane]));
        float os = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            s[i] = fmaf(kn[c0 + i], u, s[i]);
            os = fmaf(qn[c0 + i], s[i], os);
        }
        red[1][warp][lane] = os;
        __syncthreads();
        if (warp == 0)
            p.out[tok + v] = __float2bfloat16(
                p.scale * (red[1][0][lane] + red[1][1][lane] + red[1][2][lane] + red[1][3][lane]));
    }

    if (p.fin) {
        if (p.state_type == kStateBF16) {
            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.fin) + state_base +
                                                   (size_t)v * DK + c0);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __nv_bfloat162 pr = __floats2bfloat162_rn(s[8 * i + 2 * j], s[8 * i + 2 * j + 1]);
                    w[j] = *reinterpret_cast<const uint32_t *>(&pr);
                }
                dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        } else {
            float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.fin) + state_base +
                                                     (size_t)v * DK + c0);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_float4(s[4 * i], s[4 * i + 1], s[4 * i + 2], s[4 * i + 3]);
        }
    }
}

}  // namespace

cudaError_t launch_decode(const Params &p, cudaStream_t stream) {
    const int64_t units = p.n_seqs * p.H;
    if (units == 0) return cudaSuccess;
    kda_decode_kernel<<<(unsigned)(units * (DK / VS)), NTD, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
