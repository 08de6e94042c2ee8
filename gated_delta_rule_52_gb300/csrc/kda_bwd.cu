// KDA backward: gradients of L = sum(dout * out) + sum(dfinal * final_state) with
// respect to every input of the forward (q, k, v, g, beta logits, A_log, dt_bias and
// the initial state), fp32.
//
// The pages ship the forward only (the FlashKDA Q&A, its notes on training); this is
// the derivative of that forward (the token recurrence of the gated delta rule with
// one decay rate per key channel, FlashKDA README "Kernel API" for the inputs), taken
// in reverse token order.  With S'_t = Diag(alpha_t) S_{t-1}, w_t = v_t - S'_t^T k_t,
// u_t = beta_t w_t, S_t = S'_t + k_t u_t^T and o_t = scale S_t^T q_t (q, k normalised),
// the reverse step carries dS = dL/dS_t:
//   dq_t = scale S_t do_t;  dS += scale q_t do_t^T;  du = dS^T k_t;  dv_t = beta_t du;
//   dbeta_t = du . w_t;  dx = -beta_t du;  dS' = dS + k_t dx^T;
//   dk_t = dS u_t + S'_t dx;  dalpha_t = rowsum(dS' * S_{t-1});  dS = Diag(alpha_t) dS'.
//
// Two kernels:
//   kda_bwd_state_kernel: one CTA of 512 threads per (sequence, head) unit, persistent
//     over the units.  A forward sweep stores the state at the start of every 64-token
//     chunk (checkpoints); then, chunk by chunk in reverse, the chunk's states are
//     recomputed from its checkpoint into a per-CTA scratch of 64 states, and the
//     reverse step runs over the chunk's tokens.  The K x V state (fp32) lives in
//     registers: thread = 4 key channels x 8 value columns.  It writes dv and, per
//     token, dq_hat, dk_hat, dalpha and dbeta (of beta itself) into dq, dk, dg, dbeta.
//   kda_bwd_act_kernel: the activations' derivatives per token row: the L2 norms, the
//     beta sigmoid, alpha = exp(gk) and the gate (bounded or not), in place on dq, dk,
//     dg, dbeta, and the sums over tokens of dA_log and ddt_bias.
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int DKB = kHeadDim;   // K = V = 128
constexpr int NTB = 512;        // threads of the state kernel
constexpr int CB = 64;          // tokens per chunk
constexpr int64_t kStateElems = (int64_t)DKB * DKB;

// shared memory of the state kernel (floats)
constexpr int SB_Q = 0;                  // [64][128] q_hat
constexpr int SB_K = SB_Q + CB * DKB;    // [64][128] k_hat
constexpr int SB_A = SB_K + CB * DKB;    // [64][128] alpha = exp(gk)
constexpr int SB_V = SB_A + CB * DKB;    // [64][128] v
constexpr int SB_D = SB_V + CB * DKB;    // [64][128] dout
constexpr int SB_W = SB_D + CB * DKB;    // [64][128] w = v - S'^T k_hat (reverse pass)
constexpr int SB_RED = SB_W + CB * DKB;  // [16][128] column-sum partials, one row per warp
constexpr int SB_VEC = SB_RED + 16 * DKB;   // [128] a column vector for every thread
constexpr int SB_BETA = SB_VEC + DKB;       // [64] beta
constexpr int SB_MISC = SB_BETA + CB;       // [4] dbeta partials of warps 0-3
constexpr int SB_FLOATS = SB_MISC + 4;
constexpr size_t kBwdSmem = (size_t)SB_FLOATS * 4;
static_assert(kBwdSmem <= 232448, "shared memory budget");

struct BwdArgs {
    const __nv_bfloat16 *dout;   // [B,T,H,V]
    const float *dfinal;         // [N,H,V,K] or null (zero)
    float *dq, *dk, *dv, *dg, *dbeta;   // token gradients
    float *dA_log, *ddt_bias;    // [H], [H,K]: summed over tokens (zeroed before)
    float *dinit;                // [N,H,V,K] or null
    float *ckpt;                 // chunk-start states, kStateElems floats per slot
    float *tok;                  // per CTA: CB states (the chunk's S_{t-1})
    int unbounded;
};

// First packed token row of sequence n and its length.
__device__ __forceinline__ void bwd_span(const Params &p, int64_t n, int64_t &row0, int64_t &len) {
    if (p.cu_seqlens) {
        row0 = p.cu_seqlens[n];
        len = p.cu_seqlens[n + 1] - row0;
    } else {
        row0 = n * p.T;
        len = p.T;
    }
}

// Checkpoint slot of chunk ci of unit (n, h): sequence n owns chunk slots
// [floor(row0 / 64) + n, floor(row0 / 64) + n + nchunks), which never overlap.
__device__ __forceinline__ int64_t ckpt_slot(int64_t row0, int64_t n, int64_t ci, int64_t h, int64_t H) {
    return ((row0 / CB + n + ci) * H + h);
}

// The gate's log decay of one element (bounded: lb sigmoid(a x); else -a softplus(x)).
__device__ __forceinline__ float gate_gk(float x, float a, float lb, int unbounded) {
    if (unbounded) {
        const float sp = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
        return -a * sp;
    }
    return lb / (1.f + expf(-a * x));
}

__device__ __forceinline__ float4 bf16x4_to_f4(uint2 w) {
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
// Sum over the 16 lanes of a half-warp (the threads that share four key channels).
__device__ __forceinline__ float half_sum(float x) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Loads the chunk of packed token rows [row, row + L) of head h into shared memory:
// q_hat, k_hat, alpha, v, beta (and dout).  Rows t >= L hold q_hat = k_hat = v = dout = 0,
// alpha = 1, beta = 0, a step that leaves the state as it is.  Warp w takes tokens
// w, w + 16, ...; lane = four channels.
__device__ void bwd_prepare(const Params &p, const BwdArgs &b, float *sm, int64_t row, int L, int64_t h,
                            bool with_dout) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float a = expf(p.A_log[h]);
    const float4 dtb = reinterpret_cast<const float4 *>(p.dt_bias + h * DKB)[lane];
    for (int t = warp; t < CB; t += NTB / 32) {
        float4 qn = make_float4(0.f, 0.f, 0.f, 0.f), kn = qn, vv = qn, dd = qn;
        float4 al = make_float4(1.f, 1.f, 1.f, 1.f);
        float be = 0.f;
        if (t < L) {   // warp-uniform
            const int64_t tok = (row + t) * p.H + h;
            const float4 q = bf16x4_to_f4(reinterpret_cast<const uint2 *>(p.q + tok * DKB)[lane]);
            const float4 k = bf16x4_to_f4(reinterpret_cast<const uint2 *>(p.k + tok * DKB)[lane]);
            const float4 g = bf16x4_to_f4(reinterpret_cast<const uint2 *>(p.g + tok * DKB)[lane]);
            vv = bf16x4_to_f4(reinterpret_cast<const uint2 *>(p.v + tok * DKB)[lane]);
            if (with_dout) dd = bf16x4_to_f4(reinterpret_cast<const uint2 *>(b.dout + tok * DKB)[lane]);
            const float sq = warp_sum(q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w);
            const float sk = warp_sum(k.x * k.x + k.y * k.y + k.z * k.z + k.w * k.w);
            const float rq = 1.f / sqrtf(sq + 1e-6f), rk = 1.f / sqrtf(sk + 1e-6f);
            qn = make_float4(q.x * rq, q.y * rq, q.z * rq, q.w * rq);
            kn = make_float4(k.x * rk, k.y * rk, k.z * rk, k.w * rk);
            al = make_float4(expf(gate_gk(g.x + dtb.x, a, p.lower_bound, b.unbounded)),
                             expf(gate_gk(g.y + dtb.y, a, p.lower_bound, b.unbounded)),
                             expf(gate_gk(g.z + dtb.z, a, p.lower_bound, b.unbounded)),
                             expf(gate_gk(g.w + dtb.w, a, p.lower_bound, b.unbounded)));
            be = 1.f / (1.f + expf(-__bfloat162float(p.beta[tok])));
        }
        reinterpret_cast<float4 *>(sm + SB_Q + t * DKB)[lane] = qn;
        reinterpret_cast<float4 *>(sm + SB_K + t * DKB)[lane] = kn;
        reinterpret_cast<float4 *>(sm + SB_A + t * DKB)[lane] = al;
        reinterpret_cast<float4 *>(sm + SB_V + t * DKB)[lane] = vv;
        reinterpret_cast<float4 *>(sm + SB_D + t * DKB)[lane] = dd;
        if (lane == 0) sm[SB_BETA + t] = be;
    }
}

// Column sums over all 128 key channels: part[j] is this thread's sum over its four
// channels for column 8 cg + j.  Leaves one partial per warp in SB_RED and syncs; the
// caller's threads 0-127 then add the 16 partials of their column.
__device__ __forceinline__ void col_partials(float *sm, const float (&part)[8]) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, cg = tid & 15;
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = part[j] + __shfl_xor_sync(0xffffffffu, part[j], 16);
    if (lane < 16) {
        float4 *r = reinterpret_cast<float4 *>(sm + SB_RED + warp * DKB + 8 * cg);
        r[0] = make_float4(x[0], x[1], x[2], x[3]);
        r[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
    __syncthreads();
}
__device__ __forceinline__ float col_total(const float *sm, int col) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 16; ++w) s += sm[SB_RED + w * DKB + col];
    return s;
}

// One forward step on the register tile s (rows r0.., columns c0..) of token t of the
// chunk: S' = Diag(alpha) S; w = v - S'^T k_hat (into SB_W when store_w); S = S' + beta k_hat w^T.
__device__ __forceinline__ void fwd_step(float *sm, float (&s)[4][8], int t, int r0, int c0, bool store_w) {
    const int tid = threadIdx.x;
    const float4 a4 = *reinterpret_cast<const float4 *>(sm + SB_A + t * DKB + r0);
    const float4 k4 = *reinterpret_cast<const float4 *>(sm + SB_K + t * DKB + r0);
    const float a[4] = {a4.x, a4.y, a4.z, a4.w}, kk[4] = {k4.x, k4.y, k4.z, k4.w};
    float part[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        part[j] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s[i][j] *= a[i];
            part[j] = fmaf(kk[i], s[i][j], part[j]);
        }
    }
    col_partials(sm, part);
    if (tid < DKB) {
        const float wv = sm[SB_V + t * DKB + tid] - col_total(sm, tid);
        sm[SB_VEC + tid] = wv;
        if (store_w) sm[SB_W + t * DKB + tid] = wv;
    }
    __syncthreads();
    const float be = sm[SB_BETA + t];
    const float4 w0 = *reinterpret_cast<const float4 *>(sm + SB_VEC + c0);
    const float4 w1 = *reinterpret_cast<const float4 *>(sm + SB_VEC + c0 + 4);
    const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float bk = be * kk[i];
#pragma unroll
        for (int j = 0; j < 8; ++j) s[i][j] = fmaf(bk, w[j], s[i][j]);
    }
}

// Register tile <-> a state stored thread-major (8 float4 per thread, coalesced).
__device__ __forceinline__ void tile_store(float *dst, const float (&s)[4][8]) {
    float4 *d = reinterpret_cast<float4 *>(dst) + threadIdx.x * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        d[2 * i] = make_float4(s[i][0], s[i][1], s[i][2], s[i][3]);
        d[2 * i + 1] = make_float4(s[i][4], s[i][5], s[i][6], s[i][7]);
    }
}
__device__ __forceinline__ void tile_load(const float *src, float (&s)[4][8]) {
    const float4 *d = reinterpret_cast<const float4 *>(src) + threadIdx.x * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 x = d[2 * i], y = d[2 * i + 1];
        s[i][0] = x.x; s[i][1] = x.y; s[i][2] = x.z; s[i][3] = x.w;
        s[i][4] = y.x; s[i][5] = y.y; s[i][6] = y.z; s[i][7] = y.w;
    }
}

// One reverse step of token t of the chunk (packed token row `row`): ds is dL/dS_t on
// entry and dL/dS_{t-1} on exit; sp the state S_{t-1}.
__device__ __forceinline__ void bwd_step(const Params &p, const BwdArgs &b, float *sm, float (&ds)[4][8],
                                         const float (&sp)[4][8], int t, int64_t tok, int r0, int c0) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, cg = tid & 15;
    const float4 a4 = *reinterpret_cast<const float4 *>(sm + SB_A + t * DKB + r0);
    const float4 k4 = *reinterpret_cast<const float4 *>(sm + SB_K + t * DKB + r0);
    const float4 q4 = *reinterpret_cast<const float4 *>(sm + SB_Q + t * DKB + r0);
    const float a[4] = {a4.x, a4.y, a4.z, a4.w}, kk[4] = {k4.x, k4.y, k4.z, k4.w};
    const float qq[4] = {q4.x, q4.y, q4.z, q4.w};
    float w[8], dd[8];
    {
        const float4 w0 = *reinterpret_cast<const float4 *>(sm + SB_W + t * DKB + c0);
        const float4 w1 = *reinterpret_cast<const float4 *>(sm + SB_W + t * DKB + c0 + 4);
        const float4 d0 = *reinterpret_cast<const float4 *>(sm + SB_D + t * DKB + c0);
        const float4 d1 = *reinterpret_cast<const float4 *>(sm + SB_D + t * DKB + c0 + 4);
        w[0] = w0.x; w[1] = w0.y; w[2] = w0.z; w[3] = w0.w; w[4] = w1.x; w[5] = w1.y; w[6] = w1.z; w[7] = w1.w;
        dd[0] = d0.x; dd[1] = d0.y; dd[2] = d0.z; dd[3] = d0.w; dd[4] = d1.x; dd[5] = d1.y; dd[6] = d1.z; dd[7] = d1.w;
    }
    const float be = sm[SB_BETA + t], sc = p.scale;
    // dq_hat = scale S_t do with S_t = Diag(alpha) S_{t-1} + beta k_hat w^T;  dS += scale q_hat do^T
    float xq[4], part[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float x = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            x = fmaf(fmaf(a[i], sp[i][j], be * kk[i] * w[j]), dd[j], x);
            ds[i][j] = fmaf(sc * qq[i], dd[j], ds[i][j]);
        }
        xq[i] = x;
    }
    // du = dS^T k_hat (column sums)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        part[j] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) part[j] = fmaf(ds[i][j], kk[i], part[j]);
    }
    col_partials(sm, part);
    if (tid < DKB) {
        const float du = col_total(sm, tid);
        sm[SB_VEC + tid] = du;
        b.dv[tok * DKB + tid] = be * du;
        const float pb = warp_sum(du * sm[SB_W + t * DKB + tid]);   // warps 0-3, whole warps
        if (lane == 0) sm[SB_MISC + warp] = pb;
    }
    __syncthreads();
    float dx[8];
    {
        const float4 u0 = *reinterpret_cast<const float4 *>(sm + SB_VEC + c0);
        const float4 u1 = *reinterpret_cast<const float4 *>(sm + SB_VEC + c0 + 4);
        dx[0] = -be * u0.x; dx[1] = -be * u0.y; dx[2] = -be * u0.z; dx[3] = -be * u0.w;
        dx[4] = -be * u1.x; dx[5] = -be * u1.y; dx[6] = -be * u1.z; dx[7] = -be * u1.w;
    }
    // dk_hat = dS (beta w) + S' dx;  dS' = dS + k_hat dx^T;  dalpha = rowsum(dS' * S_{t-1});
    // dS_{t-1} = Diag(alpha) dS'
    float yk[4], za[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float y = 0.f, z = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            y = fmaf(ds[i][j], be * w[j], y);
            y = fmaf(a[i] * sp[i][j], dx[j], y);
            const float dsp = fmaf(kk[i], dx[j], ds[i][j]);
            z = fmaf(dsp, sp[i][j], z);
            ds[i][j] = a[i] * dsp;
        }
        yk[i] = y;
        za[i] = z;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        xq[i] = half_sum(xq[i]);
        yk[i] = half_sum(yk[i]);
        za[i] = half_sum(za[i]);
    }
    if (cg == 0) {
        *reinterpret_cast<float4 *>(b.dq + tok * DKB + r0) = make_float4(sc * xq[0], sc * xq[1], sc * xq[2], sc * xq[3]);
        *reinterpret_cast<float4 *>(b.dk + tok * DKB + r0) = make_float4(yk[0], yk[1], yk[2], yk[3]);
        *reinterpret_cast<float4 *>(b.dg + tok * DKB + r0) = make_float4(za[0], za[1], za[2], za[3]);
    }
    if (tid == 0) b.dbeta[tok] = sm[SB_MISC] + sm[SB_MISC + 1] + sm[SB_MISC + 2] + sm[SB_MISC + 3];
}

__global__ void __launch_bounds__(NTB, 1) kda_bwd_state_kernel(Params p, BwdArgs b) {
    extern __shared__ __align__(16) float sm[];
    const int tid = threadIdx.x, rg = tid >> 4, cg = tid & 15;
    const int r0 = 4 * rg, c0 = 8 * cg;
    const int64_t units = p.n_seqs * p.H;
    float *tokst = b.tok + (size_t)blockIdx.x * CB * kStateElems;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int64_t n = u / p.H, h = u % p.H;
        int64_t row0, len;
        bwd_span(p, n, row0, len);
        const int nch = (int)((len + CB - 1) / CB);
        const size_t soff = (size_t)(n * p.H + h) * kStateElems;   // [V][K] state of the unit
        float s[4][8];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) s[i][j] = 0.f;
        if (p.init) {   // S[c][v] = init[v][c]
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const size_t off = soff + (size_t)(c0 + j) * DKB + r0;
                const float4 x = p.state_type == kStateBF16
                                     ? bf16x4_to_f4(*reinterpret_cast<const uint2 *>(
                                           reinterpret_cast<const __nv_bfloat16 *>(p.init) + off))
                                     : *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p.init) + off);
                s[0][j] = x.x; s[1][j] = x.y; s[2][j] = x.z; s[3][j] = x.w;
            }
        }
        // forward sweep: the state at the start of every chunk
        for (int ci = 0; ci < nch; ++ci) {
            const int L = (int)(len - (int64_t)ci * CB < CB ? len - (int64_t)ci * CB : CB);
            tile_store(b.ckpt + ckpt_slot(row0, n, ci, h, p.H) * kStateElems, s);
            __syncthreads();   // every reader of the previous chunk's tiles is done
            bwd_prepare(p, b, sm, row0 + (int64_t)ci * CB, L, h, false);
            __syncthreads();
            for (int t = 0; t < L; ++t) fwd_step(sm, s, t, r0, c0, false);
        }
        // reverse: dS from the final-state gradient, then chunk by chunk
        float ds[4][8];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) ds[i][j] = 0.f;
        if (b.dfinal) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 x = *reinterpret_cast<const float4 *>(b.dfinal + soff + (size_t)(c0 + j) * DKB + r0);
                ds[0][j] = x.x; ds[1][j] = x.y; ds[2][j] = x.z; ds[3][j] = x.w;
            }
        }
        for (int ci = nch - 1; ci >= 0; --ci) {
            const int L = (int)(len - (int64_t)ci * CB < CB ? len - (int64_t)ci * CB : CB);
            const int64_t crow = row0 + (int64_t)ci * CB;
            tile_load(b.ckpt + ckpt_slot(row0, n, ci, h, p.H) * kStateElems, s);
            __syncthreads();
            bwd_prepare(p, b, sm, crow, L, h, true);
            __syncthreads();
            for (int t = 0; t < L; ++t) {   // S_{t-1} of every token, and w
                tile_store(tokst + (size_t)t * kStateElems, s);
                fwd_step(sm, s, t, r0, c0, true);
            }
            for (int t = L - 1; t >= 0; --t) {   // this thread's own stores: no fence needed
                float sp[4][8];
                tile_load(tokst + (size_t)t * kStateElems, sp);
                bwd_step(p, b, sm, ds, sp, t, (crow + t) * p.H + h, r0, c0);
            }
        }
        if (b.dinit) {   // dinit[v][c] = dS_0[c][v]
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float4 *>(b.dinit + soff + (size_t)(c0 + j) * DKB + r0) =
                    make_float4(ds[0][j], ds[1][j], ds[2][j], ds[3][j]);
        }
    }
}

// Derivatives of the activations, one warp per token row of one head (lane = four
// channels), 64 rows per block; in place on dq (dq_hat in), dk (dk_hat in), dg (dalpha
// in) and dbeta (of beta in, of the logit out).  dA_log and ddt_bias receive one atomic
// add per block and channel.
constexpr int kActRows = 64;
__global__ void __launch_bounds__(256) kda_bwd_act_kernel(Params p, BwdArgs b, int64_t rows) {
    __shared__ float red[8][DKB];
    __shared__ float reda[8];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t h = blockIdx.y;
    const float a = expf(p.A_log[h]), lb = p.lower_bound;
    const float4 dtb4 = reinterpret_cast<const float4 *>(p.dt_bias + h * DKB)[lane];
    const float dtb[4] = {dtb4.x, dtb4.y, dtb4.z, dtb4.w};
    float acct[4] = {0.f, 0.f, 0.f, 0.f}, acca = 0.f;
    for (int r = warp; r < kActRows; r += 8) {
        const int64_t row = (int64_t)blockIdx.x * kActRows + r;
        if (row >= rows) break;   // warp-uniform
        const int64_t tok = row * p.H + h;
        // the L2 norms: x_hat = x / n, n = sqrt(|x|^2 + eps): dx = dx_hat / n - x (x . dx_hat) / n^3
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const __nv_bfloat16 *xp = which == 0 ? p.q : p.k;
            float *gp = which == 0 ? b.dq : b.dk;
            const float4 x = bf16x4_to_f4(reinterpret_cast<const uint2 *>(xp + tok * DKB)[lane]);
            float4 *dp = reinterpret_cast<float4 *>(gp + tok * DKB) + lane;
            const float4 dh = *dp;
            const float sq = warp_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w);
            const float xd = warp_sum(x.x * dh.x + x.y * dh.y + x.z * dh.z + x.w * dh.w);
            const float nrm = sqrtf(sq + 1e-6f), inv = 1.f / nrm, c3 = xd * inv * inv * inv;
            *dp = make_float4(dh.x * inv - x.x * c3, dh.y * inv - x.y * c3, dh.z * inv - x.z * c3,
                              dh.w * inv - x.w * c3);
        }
        if (lane == 0) {
            const float be = 1.f / (1.f + expf(-__bfloat162float(p.beta[tok])));
            b.dbeta[tok] = b.dbeta[tok] * be * (1.f - be);
        }
        // the gate: alpha = exp(gk)
        const float4 g4 = bf16x4_to_f4(reinterpret_cast<const uint2 *>(p.g + tok * DKB)[lane]);
        float4 *gp = reinterpret_cast<float4 *>(b.dg + tok * DKB) + lane;
        const float4 da4 = *gp;
        const float gg[4] = {g4.x, g4.y, g4.z, g4.w}, dal[4] = {da4.x, da4.y, da4.z, da4.w};
        float dgo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float x = gg[e] + dtb[e];
            if (b.unbounded) {   // gk = -a softplus(x): dgk/dx = -a sigmoid(x), dgk/dA_log = gk
                const float gk = -a * (fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))));
                const float dgk = dal[e] * expf(gk);
                dgo[e] = dgk * (-a / (1.f + expf(-x)));
                acca = fmaf(dgk, gk, acca);
            } else {   // gk = lb sigmoid(z), z = a x: dgk/dz = lb s (1 - s), dz/dx = a, dz/dA_log = z
                const float sgm = 1.f / (1.f + expf(-a * x));
                const float dz = dal[e] * expf(lb * sgm) * lb * sgm * (1.f - sgm);
                dgo[e] = dz * a;
                acca = fmaf(dz, a * x, acca);
            }
            acct[e] += dgo[e];
        }
        *gp = make_float4(dgo[0], dgo[1], dgo[2], dgo[3]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) red[warp][4 * lane + e] = acct[e];
    acca = warp_sum(acca);
    if (lane == 0) reda[warp] = acca;
    __syncthreads();
    if (tid < DKB) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += red[w][tid];
        atomicAdd(b.ddt_bias + h * DKB + tid, s);
    }
    if (tid == 0) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += reda[w];
        atomicAdd(b.dA_log + h, s);
    }
}

size_t ckpt_bytes(const Params &p) {
    const int64_t slots = ((p.B * p.T) / CB + p.n_seqs + 1) * p.H;
    return (size_t)slots * kStateElems * 4;
}

}  // namespace

size_t bwd_scratch_bytes(const Params &p, int sms) {
    const int64_t units = p.n_seqs * p.H;
    const int64_t grid = units < sms ? units : sms;
    return ckpt_bytes(p) + (size_t)grid * CB * kStateElems * 4;
}

cudaError_t launch_bwd(const Params &p, const BwdGrads &g, int unbounded, unsigned char *ws, int sms,
                       cudaStream_t stream) {
    const int64_t units = p.n_seqs * p.H;
    BwdArgs b;
    b.dout = g.dout;
    b.dfinal = g.dfinal;
    b.dq = g.dq;
    b.dk = g.dk;
    b.dv = g.dv;
    b.dg = g.dg;
    b.dbeta = g.dbeta;
    b.dA_log = g.dA_log;
    b.ddt_bias = g.ddt_bias;
    b.dinit = g.dinit;
    b.unbounded = unbounded;
    b.ckpt = reinterpret_cast<float *>(ws);
    b.tok = reinterpret_cast<float *>(ws + ckpt_bytes(p));
    cudaError_t e = cudaSuccess;
    if (p.H > 0) {
        if ((e = cudaMemsetAsync(b.dA_log, 0, sizeof(float) * (size_t)p.H, stream)) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(b.ddt_bias, 0, sizeof(float) * (size_t)(p.H * DKB), stream)) != cudaSuccess)
            return e;
    }
    if (units == 0) return cudaSuccess;
    static std::atomic<bool> attr_done[kMaxDevices];
    e = once_per_device(attr_done, [](int) {
        return cudaFuncSetAttribute(kda_bwd_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kBwdSmem);
    });
    if (e != cudaSuccess) return e;
    const int64_t grid = units < sms ? units : sms;
    kda_bwd_state_kernel<<<(unsigned)grid, NTB, kBwdSmem, stream>>>(p, b);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t rows = p.B * p.T;
    if (rows > 0) {
        kda_bwd_act_kernel<<<dim3((unsigned)((rows + kActRows - 1) / kActRows), (unsigned)p.H), 256, 0, stream>>>(
            p, b, rows);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace kda
