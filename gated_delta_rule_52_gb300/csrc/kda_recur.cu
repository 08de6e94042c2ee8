// KDA forward with the gate that has no lower bound (safe_gate off in the FlashKDA
// usage notes): the token recurrence over whole sequences, state in registers.
//
// Gate: gk = -exp(A_log[h]) * softplus(g + dt_bias[h]), a per-token log decay with no
// floor (the FlashKDA README "Kernel API" names A_log the log-gate parameter and
// dt_bias the gate bias; with the lower bound gone the activation is the softplus rate
// scaled by exp(A_log)).  The chunked kernels factor exp(G_t - G_i) into per-token
// factors 2^(+-G) inside 16-token blocks; that needs the decay over a block to stay
// inside the fp32 exponent range, which the lower bound guarantees.  Here one token
// may decay by e^-60 or more, so the recurrence runs token by token,
//   S <- Diag(alpha) S;  u = beta (v - S^T k_hat);  S <- S + k_hat u^T;
//   out = scale * S^T q_hat,
// where any decay down to zero is exact in fp32.
//
// Work split as in the one-token kernel: warp = (sequence, head, 8 state columns),
// lane = (column quad, channel chunk) holding 4 columns x 8 channels; per token each
// warp forms the activations of its channels and sums over K with shuffles among the
// 16 lanes of its column quad.  The next token's inputs are loaded while the current
// one is computed.
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

using namespace sm103;

constexpr int DK = kHeadDim;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kWarpsR = 8;   // warps per CTA

// One token's raw inputs for one lane: q, k, g at channels ca..ca+3 and cb..cb+3,
// v at the lane's 4 columns, the beta logit.
struct TokIn {
    uint2 qa, qc, ka, kc, ga, gc, vv;
    float bl;
};

__device__ __forceinline__ void load_tok(const Params &p, int64_t row, int64_t h, int ca, int cb,
                                         int vb, TokIn &x) {
    const int64_t tok = (row * p.H + h) * DK;
    x.qa = *reinterpret_cast<const uint2 *>(p.q + tok + ca);
    x.qc = *reinterpret_cast<const uint2 *>(p.q + tok + cb);
    x.ka = *reinterpret_cast<const uint2 *>(p.k + tok + ca);
    x.kc = *reinterpret_cast<const uint2 *>(p.k + tok + cb);
    x.ga = *reinterpret_cast<const uint2 *>(p.g + tok + ca);
    x.gc = *reinterpret_cast<const uint2 *>(p.g + tok + cb);
    x.vv = *reinterpret_cast<const uint2 *>(p.v + tok + vb);
    x.bl = __bfloat162float(p.beta[row * p.H + h]);
}

// log2(1 + 2^-y) for y >= 0: the lg2 unit where 2^-y is not tiny, else the first two
// terms of the series (relative error below 1e-7 there).
__device__ __forceinline__ float log2_1p_exp2_neg(float y) {
    const float e = exp2f(-y);
    return e > 1e-3f ? __log2f(1.f + e) : e * (1.f - 0.5f * e) * kLog2e;
}

__global__ void __launch_bounds__(32 * kWarpsR) kda_recur_kernel(Params p) {
    const int lane = threadIdx.x & 31;
    const int64_t task = (int64_t)blockIdx.x * kWarpsR + (threadIdx.x >> 5);
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

    // per-head constants: the gate bias of this lane's channels (in log2 units) and
    // -exp(A_log) (the softplus below is in log2 units, so alpha = 2^(ea * sp2))
    float2 db[4];
    {
        const float4 da = *reinterpret_cast<const float4 *>(p.dt_bias + h * DK + ca);
        const float4 dc = *reinterpret_cast<const float4 *>(p.dt_bias + h * DK + cb);
        db[0] = make_float2(da.x * kLog2e, da.y * kLog2e); db[1] = make_float2(da.z * kLog2e, da.w * kLog2e);
        db[2] = make_float2(dc.x * kLog2e, dc.y * kLog2e); db[3] = make_float2(dc.z * kLog2e, dc.w * kLog2e);
    }
    const float ea = -__expf(p.A_log[h]);
    const float2 l2e = make_float2(kLog2e, kLog2e);

    TokIn nxt;
    if (len > 0) load_tok(p, b * p.T + t0, h, ca, cb, vb, nxt);
    for (int64_t t = 0; t < len; ++t) {
        const TokIn cur = nxt;
        const int64_t row = b * p.T + t0 + t;
        if (t + 1 < len) load_tok(p, row + 1, h, ca, cb, vb, nxt);

        const float2 q2[4] = {bf16x2_to_f2(cur.qa.x), bf16x2_to_f2(cur.qa.y), bf16x2_to_f2(cur.qc.x),
                              bf16x2_to_f2(cur.qc.y)};
        const float2 k2[4] = {bf16x2_to_f2(cur.ka.x), bf16x2_to_f2(cur.ka.y), bf16x2_to_f2(cur.kc.x),
                              bf16x2_to_f2(cur.kc.y)};
        const float2 g2[4] = {bf16x2_to_f2(cur.ga.x), bf16x2_to_f2(cur.ga.y), bf16x2_to_f2(cur.gc.x),
                              bf16x2_to_f2(cur.gc.y)};
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
        const float beta = 1.f / (1.f + exp2f(-cur.bl * kLog2e));
        // alpha = exp(-exp(A_log) softplus(x)) with x = g + dt_bias; in log2 units
        // softplus(x) log2(e) = max(y, 0) + log2(1 + 2^-|y|), y = x log2(e)
        float2 al[4], kn[4], qn[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 y = fma2(g2[e], l2e, db[e]);
            const float spx = fmaxf(y.x, 0.f) + log2_1p_exp2_neg(fabsf(y.x));
            const float spy = fmaxf(y.y, 0.f) + log2_1p_exp2_neg(fabsf(y.y));
            al[e] = make_float2(exp2f(ea * spx), exp2f(ea * spy));
            kn[e] = mul2(k2[e], make_float2(rk, rk));
            qn[e] = mul2(q2[e], make_float2(rq, rq));
        }
        const float2 vf[2] = {bf16x2_to_f2(cur.vv.x), bf16x2_to_f2(cur.vv.y)};
        // decay, then k_hat^T S per column (the four columns' sums interleaved)
        float ks[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s[i][e] = mul2(s[i][e], al[e]);
                acc = fma2(kn[e], s[i][e], acc);
            }
            ks[i] = acc.x + acc.y;
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1)
#pragma unroll
            for (int i = 0; i < 4; ++i) ks[i] += __shfl_xor_sync(0xffffffffu, ks[i], o);
        float os[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float vi = (i & 1) ? vf[i >> 1].y : vf[i >> 1].x;
            const float u = beta * (vi - ks[i]);
            float2 oc = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s[i][e] = fma2(kn[e], make_float2(u, u), s[i][e]);
                oc = fma2(qn[e], s[i][e], oc);
            }
            os[i] = oc.x + oc.y;
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1)
#pragma unroll
            for (int i = 0; i < 4; ++i) os[i] += __shfl_xor_sync(0xffffffffu, os[i], o);
        if (r == 0)
            *reinterpret_cast<uint2 *>(p.out + (row * p.H + h) * DK + vb) =
                make_uint2(pack_bf16(p.scale * os[0], p.scale * os[1]), pack_bf16(p.scale * os[2], p.scale * os[3]));
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

cudaError_t launch_recur(const Params &p, cudaStream_t stream) {
    const int64_t tasks = p.n_seqs * p.H * (DK / 8);
    if (tasks == 0) return cudaSuccess;
    kda_recur_kernel<<<(unsigned)((tasks + kWarpsR - 1) / kWarpsR), 32 * kWarpsR, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
