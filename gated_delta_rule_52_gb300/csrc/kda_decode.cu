// KDA forward for decode: calls of one token row (kda_fwd sends those here).  The
// token recurrence applied once, in fp32, with the state held in registers.
//
// Per (sequence, head), with S the K x V state (FlashKDA README "Kernel API"
// semantics; the same activations as the chunked kernel):
//   S <- Diag(alpha) S;  u = beta (v - S^T k_hat);  S <- S + k_hat u^T;
//   out = scale * S^T q_hat
// which is S_t = (I - beta k k^T) Diag(alpha) S_{t-1} + beta k v^T written so that
// each state column needs only its own dot products.
//
// Work split: one warp per (sequence, head, 8 state columns), independent of every
// other warp.  The state crosses HBM once in and once out, so the kernel is bound by
// it.  Earlier designs were slower:
// - one CTA per 32-column slice: the state went through a shared tile, the per-token
//   vectors were computed once into shared memory, and the column sums combined four
//   warps through shared memory; 0.103 ms for 64 x 64 heads against 0.085 ms here;
// - before that, one column and 32 rows per thread: every lane read the same rows of
//   the per-token vectors, and the shared-memory load path was the bound.
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

using namespace sm103;

constexpr int DK = kHeadDim;
constexpr float kLog2e = 1.4426950408889634f;

// One-token calls (T = 1): warp = (sequence, head, 8 state columns).  Lane = (column
// quad cl, channel chunk r): it holds columns 8 cg + 4 cl + i (i = 0..3) at channels
// 4 r .. 4 r + 3 and 64 + 4 r .. 64 + 4 r + 3, 32 fp32 values, moved straight between
// global memory and registers (a warp instruction reads or writes 256 contiguous bytes
// of each of two state rows).  Every warp forms the token's activations for its own
// channels and sums over K with shuffles among the 16 lanes of its column quad: no
// shared memory, no block barrier.
constexpr int kWarps1 = 8;   // warps per CTA
__global__ void __launch_bounds__(32 * kWarps1) kda_decode1_kernel(Params p) {
    const int lane = threadIdx.x & 31;
    const int64_t task = (int64_t)blockIdx.x * kWarps1 + (threadIdx.x >> 5);
    const int64_t tasks = p.n_seqs * p.H * (DK / 8);
    if (task >= tasks) return;
    const int cg = (int)(task % (DK / 8));
    const int64_t unit = task / (DK / 8), h = unit % p.H, n = unit / p.H;
    int64_t b, t0, len;
    seq_range(p, n, b, t0, len);
    const int cl = lane >> 4, r = lane & 15;
    const int vb = 8 * cg + 4 * cl;                 // first of this lane's 4 columns
    const int ca = 4 * r, cb = 64 + 4 * r;          // its two channel chunks
    const size_t sbase = (size_t)(n * p.H + h) * DK * DK;
    const bool sbf = p.state_type == kStateBF16;

    float2 s[4][4];   // [column i][channel pair: ca, ca+2, cb, cb+2]
    if (p.init) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const size_t row = sbase + (size_t)(vb + i) * DK;
            if (sbf) {
                const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(p.init) + row;
                const uint2 a = *reinterpret_cast<const uint2 *>(src + ca);
                const uint2 c = *reinterpret_cast<const uint2 *>(src + cb);
                s[i][0] = bf16x2_to_f2(a.x); s[i][1] = bf16x2_to_f2(a.y);
                s[i][2] = bf16x2_to_f2(c.x); s[i][3] = bf16x2_to_f2(c.y);
            } else {
                const float *src = reinterpret_cast<const float *>(p.init) + row;
                const float4 a = *reinterpret_cast<const float4 *>(src + ca);
                const float4 c = *reinterpret_cast<const float4 *>(src + cb);
                s[i][0] = make_float2(a.x, a.y); s[i][1] = make_float2(a.z, a.w);
                s[i][2] = make_float2(c.x, c.y); s[i][3] = make_float2(c.z, c.w);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = make_float2(0.f, 0.f);
    }

    if (len > 0) {
        const int64_t tok = ((b * p.T + t0) * p.H + h) * DK;
        const uint2 qa = *reinterpret_cast<const uint2 *>(p.q + tok + ca), qc = *reinterpret_cast<const uint2 *>(p.q + tok + cb);
        const uint2 ka = *reinterpret_cast<const uint2 *>(p.k + tok + ca), kc = *reinterpret_cast<const uint2 *>(p.k + tok + cb);
        const uint2 ga = *reinterpret_cast<const uint2 *>(p.g + tok + ca), gc = *reinterpret_cast<const uint2 *>(p.g + tok + cb);
        const uint2 vv = *reinterpret_cast<const uint2 *>(p.v + tok + vb);
        const float bl = __bfloat162float(p.beta[(b * p.T + t0) * p.H + h]);
        const float4 da = *reinterpret_cast<const float4 *>(p.dt_bias + h * DK + ca);
        const float4 dc = *reinterpret_cast<const float4 *>(p.dt_bias + h * DK + cb);
        const float a2 = -__expf(p.A_log[h]) * kLog2e, lb2 = p.lower_bound * kLog2e;
        const float2 q2[4] = {bf16x2_to_f2(qa.x), bf16x2_to_f2(qa.y), bf16x2_to_f2(qc.x), bf16x2_to_f2(qc.y)};
        const float2 k2[4] = {bf16x2_to_f2(ka.x), bf16x2_to_f2(ka.y), bf16x2_to_f2(kc.x), bf16x2_to_f2(kc.y)};
        const float2 g2[4] = {bf16x2_to_f2(ga.x), bf16x2_to_f2(ga.y), bf16x2_to_f2(gc.x), bf16x2_to_f2(gc.y)};
        const float2 db[4] = {make_float2(da.x, da.y), make_float2(da.z, da.w), make_float2(dc.x, dc.y),
                              make_float2(dc.z, dc.w)};
        // norms over K: this lane's 8 channels, then the 16 lanes of the column quad
        float2 sq2 = make_float2(0.f, 0.f), sk2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            sq2 = fma2(q2[e], q2[e], sq2);
            sk2 = fma2(k2[e], k2[e], sk2);
        }
        float sq = sq2.x + sq2.y, sk = sk2.x + sk2.y;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
        }
        const float rq = rsqrtf(sq + 1e-6f), rk = rsqrtf(sk + 1e-6f);
        const float beta = 1.f / (1.f + exp2f(-bl * kLog2e));
        float2 al[4], kn[4], qn[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 z = fma2(make_float2(a2, a2), add2(g2[e], db[e]), make_float2(0.f, 0.f));
            al[e] = make_float2(exp2f(lb2 * __fdividef(1.f, 1.f + exp2f(z.x))),
                                exp2f(lb2 * __fdividef(1.f, 1.f + exp2f(z.y))));
            kn[e] = mul2(k2[e], make_float2(rk, rk));
            qn[e] = mul2(q2[e], make_float2(rq, rq));
        }
        const float2 vf[2] = {bf16x2_to_f2(vv.x), bf16x2_to_f2(vv.y)};
        float o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s[i][e] = mul2(s[i][e], al[e]);
                acc = fma2(kn[e], s[i][e], acc);
            }
            float ks = acc.x + acc.y;
#pragma unroll
            for (int o2 = 1; o2 < 16; o2 <<= 1) ks += __shfl_xor_sync(0xffffffffu, ks, o2);
            const float vi = (i & 1) ? vf[i >> 1].y : vf[i >> 1].x;
            const float u = beta * (vi - ks);
            float2 oc = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s[i][e] = fma2(kn[e], make_float2(u, u), s[i][e]);
                oc = fma2(qn[e], s[i][e], oc);
            }
            float os = oc.x + oc.y;
#pragma unroll
            for (int o2 = 1; o2 < 16; o2 <<= 1) os += __shfl_xor_sync(0xffffffffu, os, o2);
            o[i] = p.scale * os;
        }
        if (r == 0)
            *reinterpret_cast<uint2 *>(p.out + tok + vb) = make_uint2(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]));
    }

    if (p.fin) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const size_t row = sbase + (size_t)(vb + i) * DK;
            if (sbf) {
                __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.fin) + row;
                *reinterpret_cast<uint2 *>(dst + ca) = make_uint2(pack_bf16(s[i][0].x, s[i][0].y), pack_bf16(s[i][1].x, s[i][1].y));
                *reinterpret_cast<uint2 *>(dst + cb) = make_uint2(pack_bf16(s[i][2].x, s[i][2].y), pack_bf16(s[i][3].x, s[i][3].y));
            } else {
                float *dst = reinterpret_cast<float *>(p.fin) + row;
                *reinterpret_cast<float4 *>(dst + ca) = make_float4(s[i][0].x, s[i][0].y, s[i][1].x, s[i][1].y);
                *reinterpret_cast<float4 *>(dst + cb) = make_float4(s[i][2].x, s[i][2].y, s[i][3].x, s[i][3].y);
            }
        }
    }
}
}  // namespace

cudaError_t launch_decode(const Params &p, cudaStream_t stream) {
    if (p.T != 1) return cudaErrorInvalidValue;   // calls of more rows run the short-step kernel
    const int64_t tasks = p.n_seqs * p.H * (DK / 8);
    if (tasks == 0) return cudaSuccess;
    kda_decode1_kernel<<<(unsigned)((tasks + kWarps1 - 1) / kWarps1), 32 * kWarps1, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
