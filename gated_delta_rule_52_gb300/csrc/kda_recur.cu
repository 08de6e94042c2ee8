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
// Work split: two CTAs of 8 warps per (sequence, head), 64 state columns each; warp =
// 8 columns, lane = (column quad, channel chunk) holding 4 columns x 8 channels of the
// state for the whole sequence.  The tokens go in blocks of 16: (A) all 256 threads
// form the block's activations once (thread = token x 8 channels: norms by shuffles
// over 16 threads, beta, the gate) into shared memory with the block's v rows, then
// (B) every warp runs the block's 16 steps from there, summing over K with shuffles
// among the 16 lanes of a column quad.  The next block's raw inputs are loaded during
// (B).  Against one warp per 8 columns forming every token's activations itself, this
// halves the time (the activations were computed 16 times per token).  Calls with at most
// one CTA per SM sum k_hat^T and q_hat^T of the decayed state in one reduction per token
// (kOneSum); larger calls keep the second sum after the update.
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

using namespace sm103;

constexpr int DK = kHeadDim;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kWarpsR = 8;   // warps per CTA

// log2(1 + 2^-y) for y >= 0: the lg2 unit where 2^-y is not tiny, else the first two
// terms of the series (relative error below 1e-7 there).
__device__ __forceinline__ float log2_1p_exp2_neg(float y) {
    const float e = exp2f(-y);
    return e > 1e-3f ? __log2f(1.f + e) : e * (1.f - 0.5f * e) * kLog2e;
}

// Tokens per staged block: the CTA forms the block's activations once in shared
// memory, then every warp runs the block's recurrence steps from there.
constexpr int TB = 16;

// kOneSum: k_hat^T S' and q_hat^T S' of the decayed state S' = Diag(alpha) S summed in
// one reduction, out = q_hat^T S' + (q_hat . k_hat) u (a shorter chain per token, faster
// with one CTA per SM); otherwise q_hat^T S is summed after the update, which overlaps the
// next token's decay (faster when two CTAs share an SM).
template <bool kOneSum>
__global__ void __launch_bounds__(32 * kWarpsR) kda_recur_kernel(Params p) {
    __shared__ __align__(16) float qs[TB][DK], kks[TB][DK], als[TB][DK];
    __shared__ float bs[TB], qks[TB];
    __shared__ __align__(16) __nv_bfloat16 vs[TB][DK];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t unit = blockIdx.x >> 1;   // two CTAs (64 columns each) per (sequence, head)
    const int qc = (int)(blockIdx.x & 1);
    if (unit >= p.n_seqs * p.H) return;     // the grid is exactly 2 CTAs per unit; never taken
    const int64_t h = unit % p.H, n = unit / p.H;
    int64_t b, t0, len;
    seq_range(p, n, b, t0, len);
    const int64_t row0 = b * p.T + t0;
    // recurrence role: lane = (column quad, channel chunk)
    const int cl = lane >> 4, r = lane & 15;
    const int vb = 64 * qc + 8 * warp + 4 * cl;     // first of this lane's 4 columns
    const int ca = 4 * r, cb = 64 + 4 * r;          // its two channel chunks
    // activation role: thread = (token of the block, 8 consecutive channels)
    const int aj = tid >> 4, ac = 8 * (tid & 15);
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

    // the activation role's gate bias (log2 units) and -exp(A_log)
    float2 db[4];
    {
        const float4 d0 = *reinterpret_cast<const float4 *>(p.dt_bias + h * DK + ac);
        const float4 d1 = *reinterpret_cast<const float4 *>(p.dt_bias + h * DK + ac + 4);
        db[0] = make_float2(d0.x * kLog2e, d0.y * kLog2e); db[1] = make_float2(d0.z * kLog2e, d0.w * kLog2e);
        db[2] = make_float2(d1.x * kLog2e, d1.y * kLog2e); db[3] = make_float2(d1.z * kLog2e, d1.w * kLog2e);
    }
    const float ea = -__expf(p.A_log[h]);
    const float2 l2e = make_float2(kLog2e, kLog2e);

    // raw inputs of the next block, loaded one block ahead
    uint4 xq = make_uint4(0u, 0u, 0u, 0u), xk = xq, xg = xq;
    float xb = 0.f;
    uint4 xv = make_uint4(0u, 0u, 0u, 0u);
    auto load_block = [&](int64_t blk) {
        const int64_t j = blk + aj;
        if (j < len) {
            const int64_t tok = ((row0 + j) * p.H + h) * DK + ac;
            xq = *reinterpret_cast<const uint4 *>(p.q + tok);
            xk = *reinterpret_cast<const uint4 *>(p.k + tok);
            xg = *reinterpret_cast<const uint4 *>(p.g + tok);
            xv = *reinterpret_cast<const uint4 *>(p.v + tok);
            if ((tid & 15) == 0) xb = __bfloat162float(p.beta[(row0 + j) * p.H + h]);
        }
    };
    if (len > 0) load_block(0);

    for (int64_t blk = 0; blk < len; blk += TB) {
        const int L = (int)((len - blk) < TB ? (len - blk) : TB);
        // (A) activations of the block's tokens into shared memory
        {
            const bool ok = aj < L;
            const uint32_t qw[4] = {xq.x, xq.y, xq.z, xq.w}, kw[4] = {xk.x, xk.y, xk.z, xk.w},
                           gw[4] = {xg.x, xg.y, xg.z, xg.w};
            float2 q2[4], k2[4];
            float2 sq2 = make_float2(0.f, 0.f), sk2 = make_float2(0.f, 0.f), sqk2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                q2[e] = bf16x2_to_f2(qw[e]);
                k2[e] = bf16x2_to_f2(kw[e]);
                sq2 = fma2(q2[e], q2[e], sq2);
                sk2 = fma2(k2[e], k2[e], sk2);
                if (kOneSum) sqk2 = fma2(q2[e], k2[e], sqk2);
            }
            float sq = sq2.x + sq2.y, sk = sk2.x + sk2.y, sqk = sqk2.x + sqk2.y;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
                if (kOneSum) sqk += __shfl_xor_sync(0xffffffffu, sqk, o);
            }
            const float rq = rsqrtf(sq + 1e-6f), rk = rsqrtf(sk + 1e-6f);
            float2 al[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 y = fma2(bf16x2_to_f2(gw[e]), l2e, db[e]);
                const float spx = fmaxf(y.x, 0.f) + log2_1p_exp2_neg(fabsf(y.x));
                const float spy = fmaxf(y.y, 0.f) + log2_1p_exp2_neg(fabsf(y.y));
                al[e] = make_float2(exp2f(ea * spx), exp2f(ea * spy));
                q2[e] = mul2(q2[e], make_float2(rq, rq));
                k2[e] = mul2(k2[e], make_float2(rk, rk));
            }
            const float beta = 1.f / (1.f + exp2f(-xb * kLog2e));
            __syncthreads();   // the previous block's steps are done with the tiles
            if (ok) {
                float4 *dq = reinterpret_cast<float4 *>(&qs[aj][ac]);
                float4 *dk = reinterpret_cast<float4 *>(&kks[aj][ac]);
                float4 *da = reinterpret_cast<float4 *>(&als[aj][ac]);
                dq[0] = make_float4(q2[0].x, q2[0].y, q2[1].x, q2[1].y);
                dq[1] = make_float4(q2[2].x, q2[2].y, q2[3].x, q2[3].y);
                dk[0] = make_float4(k2[0].x, k2[0].y, k2[1].x, k2[1].y);
                dk[1] = make_float4(k2[2].x, k2[2].y, k2[3].x, k2[3].y);
                da[0] = make_float4(al[0].x, al[0].y, al[1].x, al[1].y);
                da[1] = make_float4(al[2].x, al[2].y, al[3].x, al[3].y);
                if ((tid & 15) == 0) {
                    bs[aj] = beta;
                    qks[aj] = sqk * rq * rk;   // q_hat . k_hat (used with kOneSum)
                }
                *reinterpret_cast<uint4 *>(&vs[aj][ac]) = xv;
            }
        }
        if (blk + TB < len) load_block(blk + TB);
        __syncthreads();   // the block's activations are in shared memory

        // (B) the block's recurrence steps
#pragma unroll 1
        for (int j = 0; j < L; ++j) {
            const float4 qa = *reinterpret_cast<const float4 *>(&qs[j][ca]);
            const float4 qb = *reinterpret_cast<const float4 *>(&qs[j][cb]);
            const float4 ka = *reinterpret_cast<const float4 *>(&kks[j][ca]);
            const float4 kb = *reinterpret_cast<const float4 *>(&kks[j][cb]);
            const float4 aa = *reinterpret_cast<const float4 *>(&als[j][ca]);
            const float4 ab = *reinterpret_cast<const float4 *>(&als[j][cb]);
            const float beta = bs[j], qk = qks[j];
            const float2 qn[4] = {make_float2(qa.x, qa.y), make_float2(qa.z, qa.w), make_float2(qb.x, qb.y),
                                  make_float2(qb.z, qb.w)};
            const float2 kn[4] = {make_float2(ka.x, ka.y), make_float2(ka.z, ka.w), make_float2(kb.x, kb.y),
                                  make_float2(kb.z, kb.w)};
            const float2 al[4] = {make_float2(aa.x, aa.y), make_float2(aa.z, aa.w), make_float2(ab.x, ab.y),
                                  make_float2(ab.z, ab.w)};
            const uint2 vw = *reinterpret_cast<const uint2 *>(&vs[j][vb]);
            const float2 vf[2] = {bf16x2_to_f2(vw.x), bf16x2_to_f2(vw.y)};
            float ks[4], os[4];
            if (kOneSum) {
                float qsum[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float2 ak = make_float2(0.f, 0.f), aq = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        s[i][e] = mul2(s[i][e], al[e]);
                        ak = fma2(kn[e], s[i][e], ak);
                        aq = fma2(qn[e], s[i][e], aq);
                    }
                    ks[i] = ak.x + ak.y;
                    qsum[i] = aq.x + aq.y;
                }
#pragma unroll
                for (int o = 1; o < 16; o <<= 1)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        ks[i] += __shfl_xor_sync(0xffffffffu, ks[i], o);
                        qsum[i] += __shfl_xor_sync(0xffffffffu, qsum[i], o);
                    }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float u = beta * (((i & 1) ? vf[i >> 1].y : vf[i >> 1].x) - ks[i]);
                    os[i] = fmaf(qk, u, qsum[i]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[i][e] = fma2(kn[e], make_float2(u, u), s[i][e]);
                }
            } else {
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
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float u = beta * (((i & 1) ? vf[i >> 1].y : vf[i >> 1].x) - ks[i]);
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
            }
            if (r == 0)
                *reinterpret_cast<uint2 *>(p.out + ((row0 + blk + j) * p.H + h) * DK + vb) =
                    make_uint2(pack_bf16(p.scale * os[0], p.scale * os[1]),
                               pack_bf16(p.scale * os[2], p.scale * os[3]));
        }
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
    const int64_t units = p.n_seqs * p.H;
    if (units == 0) return cudaSuccess;
    int sms = 0;
    const cudaError_t e = sm_count(sms);
    if (e != cudaSuccess) return e;
    // one CTA per SM or fewer: the latency of the per-token chain decides, so one sum
    if (units * 2 <= sms)
        kda_recur_kernel<true><<<(unsigned)(units * 2), 32 * kWarpsR, 0, stream>>>(p);
    else
        kda_recur_kernel<false><<<(unsigned)(units * 2), 32 * kWarpsR, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
