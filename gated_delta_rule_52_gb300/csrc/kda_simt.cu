// Correctness-first KDA forward kernel: the chunked UT/WY form in fp32 on the
// CUDA cores, one CTA per (sequence, head, 64-wide slice of V).
//
// Per chunk of C = 64 tokens with entering state S0 (K x V), cumulative log
// decay G_r = sum_{s<=r} gk_s per channel:
//   A[t,i] = beta_t sum_c k[t,c] k[i,c] exp(G[t,c]-G[i,c])   (i < t)
//   M[t,i] =        sum_c q[t,c] k[i,c] exp(G[t,c]-G[i,c])   (i <= t)
//   Ti     = (I + A)^-1                         (forward substitution)
//   U      = Ti beta (V - (K*exp(G)) S0)
//   O      = scale ((Q*exp(G)) S0 + M U)
//   S_C    = Diag(exp(G_C)) S0 + (K*exp(G_C - G))^T U
// which is the token recurrence of the KDA forward (FlashKDA README "Kernel
// API") unrolled over the chunk.  Every exponent evaluated is <= 0.
//
// This kernel is the plain reference shape of the algorithm on the GPU; the
// tensor-core kernel keeps the same chunk algebra.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int C = kChunk;
constexpr int DK = kHeadDim;
constexpr int VS = 64;          // V columns per CTA
constexpr int NSLICE = kHeadDim / VS;
constexpr int NT = 256;
constexpr int DKP = DK + 1;     // padded row strides (floats) against bank conflicts
constexpr int VSP = VS + 1;
constexpr int CP = C + 1;

struct SimtSmem {
    float q[C * DKP];    // q_hat, then q_hat * exp(G)
    float k[C * DKP];    // k_hat, then k_hat * exp(G)
    float G[C * DKP];    // gk, then G (cumulative), then kbar = k_hat * exp(G_C - G)
    float S[DK * VSP];   // state slice S[c][v]
    float v[C * VSP];    // v slice, then U
    float R[C * VSP];    // beta * (v - (K*exp(G)) S)
    float A[C * CP];
    float M[C * CP];
    float Ti[C * CP];
    float beta[C];
    float gC[DK];        // G_C (log) per channel
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__global__ void __launch_bounds__(NT, 1) kda_simt_kernel(Params p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SimtSmem &s = *reinterpret_cast<SimtSmem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    int64_t unit = blockIdx.x;
    const int slice = (int)(unit % NSLICE);
    unit /= NSLICE;
    const int64_t h = unit % p.H;
    const int64_t n = unit / p.H;
    int64_t b, t0, len;
    seq_range(p, n, b, t0, len);
    const int v0 = slice * VS;
    const float a_h = __expf(p.A_log[h]);
    const float lb = p.lower_bound;
    const float *dtb = p.dt_bias + h * DK;
    const size_t state_base = (size_t)(n * p.H + h) * DK * DK;

    for (int idx = tid; idx < DK * VS; idx += NT) {
        const int c = idx % DK, vv = idx / DK;
        float x = 0.f;
        if (p.init) {
            const size_t off = state_base + (size_t)(v0 + vv) * DK + c;
            x = p.state_type == kStateBF16
                    ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.init)[off])
                    : reinterpret_cast<const float *>(p.init)[off];
        }
        s.S[c * VSP + vv] = x;
    }
    __syncthreads();

    for (int64_t cs = 0; cs < len; cs += C) {
        const int L = (int)((len - cs) < C ? (len - cs) : C);
        const size_t tok0 = (size_t)(b * p.T + t0 + cs);

        for (int idx = tid; idx < C * DK; idx += NT) {
            const int t = idx / DK, c = idx % DK;
            float qv = 0.f, kv = 0.f, gv = 0.f;
            if (t < L) {
                const size_t off = ((tok0 + t) * p.H + h) * DK + c;
                qv = __bfloat162float(p.q[off]);
                kv = __bfloat162float(p.k[off]);
                gv = __bfloat162float(p.g[off]);
            }
            s.q[t * DKP + c] = qv;
            s.k[t * DKP + c] = kv;
            s.G[t * DKP + c] = gv;
        }
        for (int idx = tid; idx < C * VS; idx += NT) {
            const int t = idx / VS, vv = idx % VS;
            float x = 0.f;
            if (t < L) x = __bfloat162float(p.v[((tok0 + t) * p.H + h) * DK + v0 + vv]);
            s.v[t * VSP + vv] = x;
        }
        if (tid < C) {
            float bt = 0.f;
            if (tid < L) {
                const float bl = __bfloat162float(p.beta[(tok0 + tid) * p.H + h]);
                bt = 1.f / (1.f + __expf(-bl));
            }
            s.beta[tid] = bt;
        }
        __syncthreads();

        // L2 norms and the gate; rows t >= L keep q = k = 0 and gk = 0.
        for (int t = warp; t < C; t += NT / 32) {
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int j = 0; j < DK / 32; ++j) {
                const int c = lane + 32 * j;
                const float a = s.q[t * DKP + c], bb = s.k[t * DKP + c];
                sq += a * a;
                sk += bb * bb;
            }
            sq = warp_sum(sq);
            sk = warp_sum(sk);
            const float rq = rsqrtf(sq + 1e-6f), rk = rsqrtf(sk + 1e-6f);
#pragma unroll
            for (int j = 0; j < DK / 32; ++j) {
                const int c = lane + 32 * j;
                s.q[t * DKP + c] *= rq;
                s.k[t * DKP + c] *= rk;
                float gk = 0.f;
                if (t < L) {
                    const float x = a_h * (s.G[t * DKP + c] + dtb[c]);
                    gk = lb / (1.f + __expf(-x));
                }
                s.G[t * DKP + c] = gk;
            }
        }
        __syncthreads();

        if (tid < DK) {
            float acc = 0.f;
            for (int t = 0; t < C; ++t) {
                acc += s.G[t * DKP + tid];
                s.G[t * DKP + tid] = acc;
            }
        }
        __syncthreads();

        for (int pi = tid; pi < C * C; pi += NT) {
            const int t = pi / C, i = pi % C;
            float sa = 0.f, sm = 0.f;
            if (i <= t) {
                for (int c = 0; c < DK; ++c) {
                    const float e = __expf(s.G[t * DKP + c] - s.G[i * DKP + c]);
                    const float ki = s.k[i * DKP + c] * e;
                    sa += s.k[t * DKP + c] * ki;
                    sm += s.q[t * DKP + c] * ki;
                }
            }
            s.A[t * CP + i] = (i < t) ? s.beta[t] * sa : 0.f;
            s.M[t * CP + i] = sm;
        }
        if (tid < DK) s.gC[tid] = s.G[(C - 1) * DKP + tid];
        __syncthreads();

        // Ti = (I + A)^-1, unit lower triangular, one row per step.
        for (int t = 0; t < C; ++t) {
            if (tid < C) {
                const int j = tid;
                float x = (j == t) ? 1.f : 0.f;
                if (j < t)
                    for (int i = j; i < t; ++i) x -= s.A[t * CP + i] * s.Ti[i * CP + j];
                s.Ti[t * CP + j] = x;
            }
            __syncthreads();
        }

        for (int idx = tid; idx < C * DK; idx += NT) {
            const int t = idx / DK, c = idx % DK;
            const float Gv = s.G[t * DKP + c];
            const float e = __expf(Gv);
            const float kk = s.k[t * DKP + c];
            s.q[t * DKP + c] *= e;
            s.k[t * DKP + c] = kk * e;
            s.G[t * DKP + c] = kk * __expf(s.gC[c] - Gv);
        }
        __syncthreads();

        for (int idx = tid; idx < C * VS; idx += NT) {
            const int t = idx / VS, vv = idx % VS;
            float acc = 0.f;
            for (int c = 0; c < DK; ++c) acc += s.k[t * DKP + c] * s.S[c * VSP + vv];
            s.R[t * VSP + vv] = s.beta[t] * (s.v[t * VSP + vv] - acc);
        }
        __syncthreads();

        for (int idx = tid; idx < C * VS; idx += NT) {
            const int t = idx / VS, vv = idx % VS;
            float acc = 0.f;
            for (int j = 0; j <= t; ++j) acc += s.Ti[t * CP + j] * s.R[j * VSP + vv];
            s.v[t * VSP + vv] = acc;   // U
        }
        __syncthreads();

        for (int idx = tid; idx < C * VS; idx += NT) {
            const int t = idx / VS, vv = idx % VS;
            float acc = 0.f;
            for (int c = 0; c < DK; ++c) acc += s.q[t * DKP + c] * s.S[c * VSP + vv];
            for (int i = 0; i <= t; ++i) acc += s.M[t * CP + i] * s.v[i * VSP + vv];
            if (t < L) p.out[((tok0 + t) * p.H + h) * DK + v0 + vv] = __float2bfloat16(p.scale * acc);
        }
        __syncthreads();

        for (int idx = tid; idx < DK * VS; idx += NT) {
            const int c = idx / VS, vv = idx % VS;
            float acc = __expf(s.gC[c]) * s.S[c * VSP + vv];
            for (int i = 0; i < C; ++i) acc += s.G[i * DKP + c] * s.v[i * VSP + vv];
            s.S[c * VSP + vv] = acc;
        }
        __syncthreads();
    }

    if (p.fin) {
        for (int idx = tid; idx < DK * VS; idx += NT) {
            const int c = idx % DK, vv = idx / DK;
            const size_t off = state_base + (size_t)(v0 + vv) * DK + c;
            const float x = s.S[c * VSP + vv];
            if (p.state_type == kStateBF16)
                reinterpret_cast<__nv_bfloat16 *>(p.fin)[off] = __float2bfloat16(x);
            else
                reinterpret_cast<float *>(p.fin)[off] = x;
        }
    }
}

}  // namespace

cudaError_t launch_simt(const Params &p, cudaStream_t stream) {
    const size_t smem = sizeof(SimtSmem);
    cudaError_t e = cudaFuncSetAttribute(kda_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t units = p.n_seqs * p.H * NSLICE;
    if (units == 0) return cudaSuccess;
    kda_simt_kernel<<<(unsigned)units, NT, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
