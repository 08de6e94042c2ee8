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
// Every value column v of the state evolves on its own (the per-token vectors alpha,
// k, beta are shared, the columns never mix), and so does its gradient; only dq, dk,
// dalpha and dbeta sum over the columns.  So:
//   kda_bwd_state_kernel: a CTA of 8 warps takes 32 value columns of one (sequence,
//     head) unit (four CTAs per unit, persistent over units x column slices), a warp
//     four columns, lane = 4 key channels x 4 columns of the fp32 state in registers.
//     The recurrence and its reverse run warp by warp with no CTA barrier per token:
//     column sums are warp shuffles.  A forward sweep stores the slice's state at the
//     start of every 16-token chunk; then chunk by chunk in reverse the chunk's states
//     are recomputed into a per-CTA scratch and the reverse step runs over its tokens.
//     The slice's shares of dq_hat, dk_hat, dalpha and dbeta go into shared per-token
//     slots (shared-memory atomic adds over the warps) and, once per chunk, to a
//     partial buffer per slice; dv and the initial state's gradient are the slice's own.
//   kda_bwd_act_kernel: per token row, the four slices' shares summed, then the
//     activations' derivatives: the L2 norms, the beta sigmoid, alpha = exp(gk) and the
//     gate (bounded or not); dq, dk, dg, dbeta written, dA_log and ddt_bias summed.
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int DKB = kHeadDim;   // K = V = 128
constexpr int NTB = 256;        // threads of the state kernel: 8 warps
constexpr int NSL = 4;          // value-column slices per unit (CTAs per unit)
constexpr int CWB = DKB / NSL;  // 32 columns per CTA, 4 per warp
constexpr int CPW = 4;          // columns per warp
constexpr int CB = 16;          // tokens per chunk (the scratch of all CTAs stays in L2)
constexpr int kSlice = DKB * CWB;   // floats of one slice of a state

// shared memory of the state kernel (floats)
constexpr int SB_Q = 0;                    // [CB][128] q_hat
constexpr int SB_K = SB_Q + CB * DKB;      // [CB][128] k_hat
constexpr int SB_A = SB_K + CB * DKB;      // [CB][128] alpha = exp(gk)
constexpr int SB_V = SB_A + CB * DKB;      // [CB][32] v of the slice
constexpr int SB_D = SB_V + CB * CWB;      // [CB][32] dout of the slice
constexpr int SB_W = SB_D + CB * CWB;      // [CB][32] w = v - S'^T k_hat of the slice
constexpr int SB_GQ = SB_W + CB * CWB;     // [CB][128] the slice's share of dq_hat
constexpr int SB_GK = SB_GQ + CB * DKB;    // [CB][128] ... of dk_hat
constexpr int SB_GA = SB_GK + CB * DKB;    // [CB][128] ... of dalpha
constexpr int SB_GB = SB_GA + CB * DKB;    // [CB] ... of dbeta
constexpr int SB_BETA = SB_GB + CB;        // [CB] beta
constexpr int SB_FLOATS = SB_BETA + CB;
constexpr size_t kBwdSmem = (size_t)SB_FLOATS * 4;
static_assert(2 * (kBwdSmem + 1024) <= 233472, "two CTAs per SM");

struct BwdArgs {
    const __nv_bfloat16 *dout;   // [B,T,H,V]
    const float *dfinal;         // [N,H,V,K] or null (zero)
    float *dq, *dk, *dv, *dg, *dbeta;   // token gradients
    float *dA_log, *ddt_bias;    // [H], [H,K]: summed over tokens (zeroed before)
    float *dinit;                // [N,H,V,K] or null
    float *ckpt;                 // chunk-start slices, kSlice floats per slot
    float *tok;                  // per CTA: CB slices (the chunk's S_{t-1})
    float *pq, *pk, *pa, *pb;    // per slice: shares of dq_hat, dk_hat, dalpha [rows H 128], dbeta [rows H]
    int64_t prow;                // rows H: the stride of one slice in pq, pk, pa (x 128) and pb
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

// Checkpoint slot of chunk ci of unit (n, h), slice sl: sequence n owns chunk slots
// [floor(row0 / CB) + n, floor(row0 / CB) + n + nchunks), which never overlap.
__device__ __forceinline__ int64_t ckpt_slot(int64_t row0, int64_t n, int64_t ci, int64_t h, int64_t H, int sl) {
    return ((row0 / CB + n + ci) * H + h) * NSL + sl;
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

// Loads the chunk of packed token rows [row, row + L) of head h: q_hat, k_hat, alpha
// (all channels), beta, and v (and dout) of the slice's columns vb .. vb + 31; rows
// t >= L hold q_hat = k_hat = v = dout = 0, alpha = 1, beta = 0.  Clears the gradient
// slots.  Warp w takes tokens w, w + 16; lane = four channels.
__device__ void bwd_prepare(const Params &p, const BwdArgs &b, float *sm, int64_t row, int L, int64_t h,
                            int vb, bool with_dout) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float a = expf(p.A_log[h]);
    const float4 dtb = reinterpret_cast<const float4 *>(p.dt_bias + h * DKB)[lane];
    for (int t = warp; t < CB; t += NTB / 32) {
        float4 qn = make_float4(0.f, 0.f, 0.f, 0.f), kn = qn;
        float4 al = make_float4(1.f, 1.f, 1.f, 1.f);
        float vv = 0.f, dd = 0.f, be = 0.f;
        if (t < L) {   // warp-uniform
            const int64_t tok = (row + t) * p.H + h;
            const float4 q = bf16x4_to_f4(reinterpret_cast<const uint2 *>(p.q + tok * DKB)[lane]);
            const float4 k = bf16x4_to_f4(reinterpret_cast<const uint2 *>(p.k + tok * DKB)[lane]);
            const float4 g = bf16x4_to_f4(reinterpret_cast<const uint2 *>(p.g + tok * DKB)[lane]);
            vv = __bfloat162float(p.v[tok * DKB + vb + lane]);
            if (with_dout) dd = __bfloat162float(b.dout[tok * DKB + vb + lane]);
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
        sm[SB_V + t * CWB + lane] = vv;
        sm[SB_D + t * CWB + lane] = dd;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        reinterpret_cast<float4 *>(sm + SB_GQ + t * DKB)[lane] = z;
        reinterpret_cast<float4 *>(sm + SB_GK + t * DKB)[lane] = z;
        reinterpret_cast<float4 *>(sm + SB_GA + t * DKB)[lane] = z;
        if (lane == 0) {
            sm[SB_BETA + t] = be;
            sm[SB_GB + t] = 0.f;
        }
    }
}

// A lane's tile: key channels lane + 32 i (i < 4) of the warp's four value columns j (a
// stride of 32 channels, so that the lanes of a warp hit 32 different shared-memory banks).
// Stored thread-major (four float4 per thread, coalesced) in checkpoints and scratch.
__device__ __forceinline__ void tile_store(float *dst, const float (&s)[4][CPW]) {
    float4 *d = reinterpret_cast<float4 *>(dst) + threadIdx.x * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_float4(s[i][0], s[i][1], s[i][2], s[i][3]);
}
__device__ __forceinline__ void tile_load(const float *src, float (&s)[4][CPW]) {
    const float4 *d = reinterpret_cast<const float4 *>(src) + threadIdx.x * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 x = d[i];
        s[i][0] = x.x; s[i][1] = x.y; s[i][2] = x.z; s[i][3] = x.w;
    }
}

// Sums of four columns over the warp's 32 lanes, every lane receiving all four: two
// exchanges halve the columns a lane carries (lane bit 4, then bit 3), three more finish
// the one left (lane 8 j then holds column j's sum), four broadcasts hand them round.
__device__ __forceinline__ void col_sums4(const float (&x)[CPW], float (&out)[CPW]) {
    const int lane = threadIdx.x & 31;
    const bool b4 = lane & 16, b3 = lane & 8;
    const float y0 = (b4 ? x[2] : x[0]) + __shfl_xor_sync(0xffffffffu, b4 ? x[0] : x[2], 16);
    const float y1 = (b4 ? x[3] : x[1]) + __shfl_xor_sync(0xffffffffu, b4 ? x[1] : x[3], 16);
    float z = (b3 ? y1 : y0) + __shfl_xor_sync(0xffffffffu, b3 ? y0 : y1, 8);
    z += __shfl_xor_sync(0xffffffffu, z, 4);
    z += __shfl_xor_sync(0xffffffffu, z, 2);
    z += __shfl_xor_sync(0xffffffffu, z, 1);
#pragma unroll
    for (int j = 0; j < CPW; ++j) out[j] = __shfl_sync(0xffffffffu, z, 8 * j);
}

// One forward step of token t on the warp's four columns: S' = Diag(alpha) S;
// w = v - S'^T k_hat (into SB_W when store_w); S = S' + beta k_hat w^T.
__device__ __forceinline__ void fwd_step(float *sm, float (&s)[4][CPW], int t, bool store_w) {
    const int lane = threadIdx.x & 31, lc = CPW * (threadIdx.x >> 5);
    const float4 v4 = *reinterpret_cast<const float4 *>(sm + SB_V + t * CWB + lc);
    float a[4], kk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        a[i] = sm[SB_A + t * DKB + lane + 32 * i];
        kk[i] = sm[SB_K + t * DKB + lane + 32 * i];
    }
    float part[CPW] = {0.f, 0.f, 0.f, 0.f}, ks[CPW];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < CPW; ++j) {
            s[i][j] *= a[i];
            part[j] = fmaf(kk[i], s[i][j], part[j]);
        }
    col_sums4(part, ks);
    const float w[CPW] = {v4.x - ks[0], v4.y - ks[1], v4.z - ks[2], v4.w - ks[3]};
    if (store_w && lane == 0)
        *reinterpret_cast<float4 *>(sm + SB_W + t * CWB + lc) = make_float4(w[0], w[1], w[2], w[3]);
    const float be = sm[SB_BETA + t];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float bk = be * kk[i];
#pragma unroll
        for (int j = 0; j < CPW; ++j) s[i][j] = fmaf(bk, w[j], s[i][j]);
    }
}

// One reverse step of token t on the warp's four columns: ds is dL/dS_t on entry and
// dL/dS_{t-1} on exit; sp the state S_{t-1}.  The warp's shares of dq_hat, dk_hat,
// dalpha and dbeta go to the token's slots by shared-memory atomic adds.
__device__ __forceinline__ void bwd_step(const Params &p, const BwdArgs &b, float *sm, float (&ds)[4][CPW],
                                         const float (&sp)[4][CPW], int t, int64_t tok, int vb) {
    const int lane = threadIdx.x & 31, lc = CPW * (threadIdx.x >> 5);
    const float4 w4 = *reinterpret_cast<const float4 *>(sm + SB_W + t * CWB + lc);
    const float4 d4 = *reinterpret_cast<const float4 *>(sm + SB_D + t * CWB + lc);
    float a[4], kk[4], qq[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        a[i] = sm[SB_A + t * DKB + lane + 32 * i];
        kk[i] = sm[SB_K + t * DKB + lane + 32 * i];
        qq[i] = sm[SB_Q + t * DKB + lane + 32 * i];
    }
    const float w[CPW] = {w4.x, w4.y, w4.z, w4.w}, dd[CPW] = {d4.x, d4.y, d4.z, d4.w};
    const float be = sm[SB_BETA + t], sc = p.scale;
    // dq_hat = scale S_t do, S_t = Diag(alpha) S_{t-1} + beta k_hat w^T;  dS += scale q_hat do^T
    float xq[4], part[CPW] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float x = 0.f;
        const float bk = be * kk[i], sq = sc * qq[i];
#pragma unroll
        for (int j = 0; j < CPW; ++j) {
            x = fmaf(fmaf(a[i], sp[i][j], bk * w[j]), dd[j], x);
            ds[i][j] = fmaf(sq, dd[j], ds[i][j]);
            part[j] = fmaf(ds[i][j], kk[i], part[j]);
        }
        xq[i] = sc * x;
    }
    // du = dS^T k_hat (sums over the key channels)
    float du[CPW];
    col_sums4(part, du);
    if (lane < CPW) {
        const float dl = lane == 0 ? du[0] : (lane == 1 ? du[1] : (lane == 2 ? du[2] : du[3]));
        b.dv[tok * DKB + vb + lc + lane] = be * dl;
    }
    if (lane == 0)
        atomicAdd(sm + SB_GB + t, du[0] * w[0] + du[1] * w[1] + du[2] * w[2] + du[3] * w[3]);
    float dx[CPW];
#pragma unroll
    for (int j = 0; j < CPW; ++j) dx[j] = -be * du[j];
    // dk_hat = dS (beta w) + S' dx;  dS' = dS + k_hat dx^T;  dalpha = rowsum(dS' * S_{t-1});
    // dS_{t-1} = Diag(alpha) dS'
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float y = 0.f, z = 0.f;
#pragma unroll
        for (int j = 0; j < CPW; ++j) {
            y = fmaf(ds[i][j], be * w[j], y);
            y = fmaf(a[i] * sp[i][j], dx[j], y);
            const float dsp = fmaf(kk[i], dx[j], ds[i][j]);
            z = fmaf(dsp, sp[i][j], z);
            ds[i][j] = a[i] * dsp;
        }
        atomicAdd(sm + SB_GQ + t * DKB + lane + 32 * i, xq[i]);
        atomicAdd(sm + SB_GK + t * DKB + lane + 32 * i, y);
        atomicAdd(sm + SB_GA + t * DKB + lane + 32 * i, z);
    }
}

__global__ void __launch_bounds__(NTB, 2) kda_bwd_state_kernel(Params p, BwdArgs b) {
    extern __shared__ __align__(16) float sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t work = p.n_seqs * p.H * NSL;
    float *tokst = b.tok + (size_t)blockIdx.x * CB * kSlice;
    for (int64_t wi = blockIdx.x; wi < work; wi += gridDim.x) {
        const int64_t u = wi / NSL, n = u / p.H, h = u % p.H;
        const int sl = (int)(wi % NSL), vb = sl * CWB, col = vb + CPW * warp;
        int64_t row0, len;
        bwd_span(p, n, row0, len);
        const int nch = (int)((len + CB - 1) / CB);
        const size_t soff = (size_t)(n * p.H + h) * DKB * DKB;   // [V][K] state of the unit
        // the slice's share of the token gradients: slice 0 into the outputs, the others
        // into the partial buffers
        float *gq = sl == 0 ? b.dq : b.pq + (size_t)(sl - 1) * b.prow * DKB;
        float *gk = sl == 0 ? b.dk : b.pk + (size_t)(sl - 1) * b.prow * DKB;
        float *ga = sl == 0 ? b.dg : b.pa + (size_t)(sl - 1) * b.prow * DKB;
        float *gb = sl == 0 ? b.dbeta : b.pb + (size_t)(sl - 1) * b.prow;
        float s[4][CPW];
#pragma unroll
        for (int j = 0; j < CPW; ++j)   // S[c][v] = init[v][c]
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const size_t off = soff + (size_t)(col + j) * DKB + lane + 32 * i;
                s[i][j] = !p.init ? 0.f
                          : p.state_type == kStateBF16
                              ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.init)[off])
                              : reinterpret_cast<const float *>(p.init)[off];
            }
        // forward sweep: the slice's state at the start of every chunk
        for (int ci = 0; ci < nch; ++ci) {
            const int L = (int)(len - (int64_t)ci * CB < CB ? len - (int64_t)ci * CB : CB);
            tile_store(b.ckpt + ckpt_slot(row0, n, ci, h, p.H, sl) * kSlice, s);
            __syncthreads();   // every reader of the previous chunk's shared data is done
            bwd_prepare(p, b, sm, row0 + (int64_t)ci * CB, L, h, vb, false);
            __syncthreads();
            for (int t = 0; t < L; ++t) fwd_step(sm, s, t, false);
        }
        // reverse: dS from the final-state gradient, then chunk by chunk
        float ds[4][CPW];
#pragma unroll
        for (int j = 0; j < CPW; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                ds[i][j] = b.dfinal ? b.dfinal[soff + (size_t)(col + j) * DKB + lane + 32 * i] : 0.f;
        for (int ci = nch - 1; ci >= 0; --ci) {
            const int L = (int)(len - (int64_t)ci * CB < CB ? len - (int64_t)ci * CB : CB);
            const int64_t crow = row0 + (int64_t)ci * CB;
            tile_load(b.ckpt + ckpt_slot(row0, n, ci, h, p.H, sl) * kSlice, s);
            __syncthreads();
            bwd_prepare(p, b, sm, crow, L, h, vb, true);
            __syncthreads();
            for (int t = 0; t < L; ++t) {   // S_{t-1} of every token, and w
                tile_store(tokst + (size_t)t * kSlice, s);
                fwd_step(sm, s, t, true);
            }
            __syncwarp();   // lane 0's w stores are visible to the warp
            float sp[4][CPW], spn[4][CPW];
            tile_load(tokst + (size_t)(L - 1) * kSlice, sp);
            for (int t = L - 1; t >= 0; --t) {   // this thread's own stores: no fence needed
                if (t > 0) tile_load(tokst + (size_t)(t - 1) * kSlice, spn);
                bwd_step(p, b, sm, ds, sp, t, (crow + t) * p.H + h, vb);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < CPW; ++j) sp[i][j] = spn[i][j];
            }
            __syncthreads();   // every warp's slot additions are in
            for (int e = tid; e < L * DKB; e += NTB) {
                const int t = e >> 7, r = e & (DKB - 1);
                const int64_t o = ((crow + t) * p.H + h) * DKB + r;
                gq[o] = sm[SB_GQ + t * DKB + r];
                gk[o] = sm[SB_GK + t * DKB + r];
                ga[o] = sm[SB_GA + t * DKB + r];
            }
            for (int t = tid; t < L; t += NTB) gb[(crow + t) * p.H + h] = sm[SB_GB + t];
        }
        if (b.dinit) {   // dinit[v][c] = dS_0[c][v] on the slice's columns
#pragma unroll
            for (int j = 0; j < CPW; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) b.dinit[soff + (size_t)(col + j) * DKB + lane + 32 * i] = ds[i][j];
        }
    }
}

// Per token row of one head (a warp per row, lane = four channels, 64 rows per block):
// the four slices' shares of dq_hat, dk_hat, dalpha, dbeta summed (slice 0's sit in the
// outputs already), then the derivatives of the L2 norms, the beta sigmoid, alpha =
// exp(gk) and the gate; dq, dk, dg, dbeta written.  dA_log and ddt_bias take one atomic
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
    const size_t sstride = (size_t)b.prow * DKB;
    float acct[4] = {0.f, 0.f, 0.f, 0.f}, acca = 0.f;
    auto share4 = [&](float *out, const float *part, int64_t tok) {   // slice 0 + the others
        float4 x = reinterpret_cast<const float4 *>(out + tok * DKB)[lane];
#pragma unroll
        for (int sl = 0; sl < NSL - 1; ++sl) {
            const float4 y = reinterpret_cast<const float4 *>(part + sl * sstride + tok * DKB)[lane];
            x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
        }
        return x;
    };
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
            const float4 dh = share4(gp, which == 0 ? b.pq : b.pk, tok);
            const float sq = warp_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w);
            const float xd = warp_sum(x.x * dh.x + x.y * dh.y + x.z * dh.z + x.w * dh.w);
            const float inv = 1.f / sqrtf(sq + 1e-6f), c3 = xd * inv * inv * inv;
            reinterpret_cast<float4 *>(gp + tok * DKB)[lane] =
                make_float4(dh.x * inv - x.x * c3, dh.y * inv - x.y * c3, dh.z * inv - x.z * c3,
                            dh.w * inv - x.w * c3);
        }
        if (lane == 0) {
            float dbe = b.dbeta[tok];
#pragma unroll
            for (int sl = 0; sl < NSL - 1; ++sl) dbe += b.pb[sl * b.prow + tok];
            const float be = 1.f / (1.f + expf(-__bfloat162float(p.beta[tok])));
            b.dbeta[tok] = dbe * be * (1.f - be);
        }
        // the gate: alpha = exp(gk)
        const float4 g4 = bf16x4_to_f4(reinterpret_cast<const uint2 *>(p.g + tok * DKB)[lane]);
        const float4 da4 = share4(b.dg, b.pa, tok);
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
        reinterpret_cast<float4 *>(b.dg + tok * DKB)[lane] = make_float4(dgo[0], dgo[1], dgo[2], dgo[3]);
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

struct BwdLayout {
    size_t ckpt, tok, part, total;
    int64_t grid;
};
BwdLayout bwd_layout(const Params &p, int sms) {
    BwdLayout l;
    const int64_t work = p.n_seqs * p.H * NSL;
    l.grid = work < 2 * (int64_t)sms ? work : 2 * (int64_t)sms;   // two CTAs per SM
    const int64_t slots = ((p.B * p.T) / CB + p.n_seqs + 1) * p.H * NSL;
    const int64_t prow = p.B * p.T * p.H;
    l.ckpt = 0;
    l.tok = (size_t)slots * kSlice * 4;
    l.part = l.tok + (size_t)l.grid * CB * kSlice * 4;
    l.total = l.part + (size_t)(NSL - 1) * (size_t)prow * (3 * DKB + 1) * 4;
    return l;
}

}  // namespace

size_t bwd_scratch_bytes(const Params &p, int sms) { return bwd_layout(p, sms).total; }

cudaError_t launch_bwd(const Params &p, const BwdGrads &g, int unbounded, unsigned char *ws, int sms,
                       cudaStream_t stream) {
    const BwdLayout l = bwd_layout(p, sms);
    const int64_t prow = p.B * p.T * p.H;
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
    b.ckpt = reinterpret_cast<float *>(ws + l.ckpt);
    b.tok = reinterpret_cast<float *>(ws + l.tok);
    float *part = reinterpret_cast<float *>(ws + l.part);
    b.pq = part;
    b.pk = part + (size_t)(NSL - 1) * prow * DKB;
    b.pa = part + (size_t)2 * (NSL - 1) * prow * DKB;
    b.pb = part + (size_t)3 * (NSL - 1) * prow * DKB;
    b.prow = prow;
    cudaError_t e = cudaSuccess;
    if (p.H > 0) {
        if ((e = cudaMemsetAsync(b.dA_log, 0, sizeof(float) * (size_t)p.H, stream)) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(b.ddt_bias, 0, sizeof(float) * (size_t)(p.H * DKB), stream)) != cudaSuccess)
            return e;
    }
    if (p.n_seqs * p.H == 0) return cudaSuccess;
    static std::atomic<bool> attr_done[kMaxDevices];
    e = once_per_device(attr_done, [](int) {
        return cudaFuncSetAttribute(kda_bwd_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kBwdSmem);
    });
    if (e != cudaSuccess) return e;
    kda_bwd_state_kernel<<<(unsigned)l.grid, NTB, kBwdSmem, stream>>>(p, b);
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
