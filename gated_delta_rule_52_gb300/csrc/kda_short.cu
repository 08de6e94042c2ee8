// KDA forward for short multi-token steps (2..64 token rows per call, or the
// sequences of at most 64 tokens of a mixed-length varlen call): the sequence's
// tokens form chunks of 16 of the UT/WY form, evaluated with warp-level tensor-core
// MMAs (mma.sync m16n8k16, fp32 accumulation), the state kept in registers from one
// 16-token block to the next.
//
// Per (sequence, head) and 16-token block of L <= 16 tokens, with G the cumulative
// log decay from the start of the block (every exponent below is <= 0 except 2^-G,
// which stays below 2^116 since each token's log decay is >= the lower bound of -5):
//   A[t,i] = beta_t sum_c k_hat[t,c] k_hat[i,c] 2^(G[t,c]-G[i,c])   (i < t)
//   M[t,i] =        sum_c q_hat[t,c] k_hat[i,c] 2^(G[t,c]-G[i,c])   (i <= t)
//   T' = (I + A)^-1 Diag(beta);   U = T' (V - K_hat Gamma S)
//   O  = scale (Q_hat Gamma S + M U);   S <- Diag(Gamma_L) S + Kbar^T U
// with Gamma = 2^G, Gamma_L its last row and Kbar = k_hat 2^(G_L - G) (the
// chunk equations of the tensor-core path; FlashKDA README "Kernel API" semantics).
//
// Work split: one CTA of 8 warps per (sequence, head).  Warp w owns state rows
// v = 16w .. 16w+15 (storage [V][K]) as fp32 MMA accumulators in registers; the
// same registers, packed to fp16, are the B operand of (K_hat Gamma; Q_hat Gamma) S^T,
// so no warp needs another warp's state.  The CTA shares the per-block operands:
// - the gate and the decayed q/k tiles (threads = channel pairs and token halves);
// - the norms and beta;
// - A and M from one bf16 MMA each (raw q/k times 2^G against k times 2^-G, the
//   norms applied in fp32 afterwards, as in the chunked kernel);
// - the 16 x 16 inverse by forward substitution (on warp 2, after its own products).
// CTAs are persistent (two per SM): a unit's token rows are copied in while the
// previous unit finishes, and its state is prefetched into L2 at the same time.  The
// row norms of k are folded into U (U' = Diag(1/|k|) U) and out of M and Kbar, so
// every fp16 tile is the raw input times decay factors in [0, 1].
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

using namespace sm103;

constexpr int DK = kHeadDim;
constexpr int NTS = 256;            // 8 warps
constexpr int LT = 16;              // token rows of the step (padded with zeros)
constexpr int RS = 136;             // row stride (halves) of the [16|32][128] tiles: 272 B
constexpr int RS16 = 24;            // row stride (halves) of the 16 x 16 tiles: 48 B
constexpr float kLog2e = 1.4426950408889634f;

struct ShortSmem {
    __nv_bfloat16 q[LT][RS], k[LT][RS], g[LT][RS], v[LT][RS];   // raw inputs, zero rows >= L
    __nv_bfloat16 kp[LT][RS], qp[LT][RS], kn[LT][RS];            // k 2^G, q 2^G, k 2^-G (bf16)
    __half y[2 * LT][RS];        // [k 2^G; q 2^G] (fp16)
    __half kc[LT][RS];           // k 2^(G_L - G) (fp16)
    float a[LT][LT + 1];         // A (fp32)
    __half tp[LT][RS16];         // T' = (I + A)^-1 Diag(beta)
    __half mp[LT][RS16];         // M' = Diag(1/|q|) raw M (without the 1/|k_i| factor)
    __half wr[8][LT][RS16];      // per warp: R = V - K_hat Gamma S^T, its 16 columns
    __half wu[8][LT][RS16];      // per warp: U' = Diag(1/|k|) U, its 16 columns
    float gam[DK];               // Gamma_L
    float rq[LT], rk[LT], beta[LT];
};

// m16n8k16 MMAs, fp32 accumulate in place.  Fragments (g = lane / 4, q = lane % 4):
// A a0 (g, 2q..2q+1), a1 (g+8, ..), a2 (g, 2q+8..), a3 (g+8, 2q+8..); B b0 (k 2q..2q+1,
// n g), b1 (k 2q+8.., n g); D d0,d1 (g, 2q..2q+1), d2,d3 (g+8, 2q..2q+1).
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16x(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Four 8x8 b16 matrices; lane l gives the address of row (l & 7) of matrix l >> 3.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(row))
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(row))
                 : "memory");
}
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// fp16 pair of operand values, recording in `bad` any value beyond +-65504 (or NaN)
__device__ __forceinline__ uint32_t h2c(bool &bad, float lo, float hi) {
    bad |= !(fabsf(lo) <= 65504.f) | !(fabsf(hi) <= 65504.f);
    return pack_f16(lo, hi);
}
// Bulk prefetch of a contiguous global range into L2 (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Column of channel c in every channel-indexed tile (a permutation inside each
// block of 16 channels).  For each of its two state rows a thread holds channels
// 16 i + 4 qq + 0..3 (i = 0..7): eight 16-byte pieces of the [V][K] row, so a warp's
// load instruction covers 64 contiguous bytes of each of 8 rows.  In the MMA
// fragments these channels are z[2i] (+0, +1) and z[2i+1] (+2, +3); tau puts every
// channel where those fragments expect it: k = 2 qq + e (+0, +1) or 8 + 2 qq + e
// (+2, +3) in k step i of the X products, and n = 2 qq + e in n tile 2i (+0, +1) or
// 2i + 1 (+2, +3) of the state update.
__device__ __forceinline__ int tau(int c) {
    return (c & ~15) | (((c >> 1) & 1) << 3) | (((c >> 2) & 3) << 1) | (c & 1);
}

// kMulti: calls of more than 16 token rows (several blocks per unit); a separate
// instantiation keeps the single-block case free of the block loop's registers.
template <bool kMulti>
__global__ void __launch_bounds__(NTS, 2) kda_short_kernel(Params p) {
    bool rbad = false;   // some fp16 operand value (k, q, state, R, T', U') beyond +-65504
    extern __shared__ __align__(16) unsigned char dsm[];
    ShortSmem &sm = *reinterpret_cast<ShortSmem *>(dsm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, qq = lane & 3;
    const int v0 = 16 * warp + gq;   // this thread's state rows: v0 and v0 + 8
    const int64_t units = p.n_seqs * p.H;
    const size_t selt = p.state_type == kStateBF16 ? 2 : 4;

    // Token rows of 16-token block sc of unit u into the q, k, g, v tiles (16-byte
    // asynchronous copies for the rows that exist, zeros for the rest), committed as
    // one cp.async group.
    auto load_inputs = [&](int64_t u, int sc) {
        const int64_t uh = u % p.H, un = u / p.H;
        int64_t ub, ut0, ulen;
        seq_range(p, un, ub, ut0, ulen);
        const int64_t first = ut0 + LT * sc, rows = ulen - LT * sc;
        for (int i = tid; i < 4 * LT * 16; i += NTS) {
            const int x = i >> 8, t = (i >> 4) & 15, ch = i & 15;
            __nv_bfloat16 *dst = (x == 0 ? &sm.q[t][8 * ch] : x == 1 ? &sm.k[t][8 * ch]
                                  : x == 2 ? &sm.g[t][8 * ch] : &sm.v[t][8 * ch]);
            if (t < rows) {
                const __nv_bfloat16 *src = (x == 0 ? p.q : x == 1 ? p.k : x == 2 ? p.g : p.v) +
                                           ((ub * p.T + first + t) * p.H + uh) * DK + 8 * ch;
                cp_async16(dst, src);
            } else {
                *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    // Persistent CTAs, unit after unit; a unit's tokens in blocks of 16, the state in
    // the z registers from the first block to the last.  The next block's (or the next
    // unit's first block's) token rows are copied in as soon as the current ones are
    // dead (after the second barrier), and the next unit's state is prefetched into L2
    // at the same point.
    // In a mixed-length call the units longer than kShortMaxT tokens are the cluster
    // kernel's: this kernel steps over them (the next unit it takes, from u on).
    auto next_unit = [&](int64_t u) -> int64_t {
        if (!p.mixed) return u;
        for (; u < units; u += gridDim.x) {
            int64_t ub, ut0, ulen;
            seq_range(p, u / p.H, ub, ut0, ulen);
            if (ulen <= kShortMaxT) break;
        }
        return u;
    };
    const int64_t first_unit = next_unit(blockIdx.x);
    if (first_unit < units) load_inputs(first_unit, 0);
    for (int64_t unit = first_unit; unit < units; unit = next_unit(unit + gridDim.x)) {
        const int64_t h = unit % p.H, n = unit / p.H;
        int64_t b, t0, len64;
        seq_range(p, n, b, t0, len64);
        const int Lseq = (int)len64;   // <= 64 (the packed batch has at most 64 token rows)
        const int nsub = kMulti && Lseq > LT ? (Lseq + LT - 1) / LT : 1;   // a zero-length unit: one empty block
        const size_t state_base = (size_t)(n * p.H + h) * DK * DK;
        const int64_t row_first = b * p.T + t0;

        // ---- this warp's state rows as MMA accumulators: z[2i + r][e] (rows v0) and
        // z[2i + r][2 + e] (rows v0 + 8) hold channel 16 i + 4 qq + 2 r + e
        float z[16][4];
        if (p.init) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = 16 * i + 4 * qq;
                if (p.state_type == kStateBF16) {
                    const __nv_bfloat16 *s0 = reinterpret_cast<const __nv_bfloat16 *>(p.init) + state_base;
                    const uint2 w0 = *reinterpret_cast<const uint2 *>(s0 + (size_t)v0 * DK + c);
                    const uint2 w1 = *reinterpret_cast<const uint2 *>(s0 + (size_t)(v0 + 8) * DK + c);
                    z[2 * i][0] = __uint_as_float(w0.x << 16); z[2 * i][1] = __uint_as_float(w0.x & 0xFFFF0000u);
                    z[2 * i + 1][0] = __uint_as_float(w0.y << 16); z[2 * i + 1][1] = __uint_as_float(w0.y & 0xFFFF0000u);
                    z[2 * i][2] = __uint_as_float(w1.x << 16); z[2 * i][3] = __uint_as_float(w1.x & 0xFFFF0000u);
                    z[2 * i + 1][2] = __uint_as_float(w1.y << 16); z[2 * i + 1][3] = __uint_as_float(w1.y & 0xFFFF0000u);
                } else {
                    const float *s0 = reinterpret_cast<const float *>(p.init) + state_base;
                    const float4 x0 = *reinterpret_cast<const float4 *>(s0 + (size_t)v0 * DK + c);
                    const float4 x1 = *reinterpret_cast<const float4 *>(s0 + (size_t)(v0 + 8) * DK + c);
                    z[2 * i][0] = x0.x; z[2 * i][1] = x0.y; z[2 * i + 1][0] = x0.z; z[2 * i + 1][1] = x0.w;
                    z[2 * i][2] = x1.x; z[2 * i][3] = x1.y; z[2 * i + 1][2] = x1.z; z[2 * i + 1][3] = x1.w;
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) z[j][0] = z[j][1] = z[j][2] = z[j][3] = 0.f;
        }

        // the z registers -> final_state (bf16 or fp32), 16-byte pieces as they were loaded
        auto store_state = [&]() {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = 16 * i + 4 * qq;
                if (p.state_type == kStateBF16) {
                    __nv_bfloat16 *s0 = reinterpret_cast<__nv_bfloat16 *>(p.fin) + state_base;
                    *reinterpret_cast<uint2 *>(s0 + (size_t)v0 * DK + c) =
                        make_uint2(pack_bf16(z[2 * i][0], z[2 * i][1]), pack_bf16(z[2 * i + 1][0], z[2 * i + 1][1]));
                    *reinterpret_cast<uint2 *>(s0 + (size_t)(v0 + 8) * DK + c) =
                        make_uint2(pack_bf16(z[2 * i][2], z[2 * i][3]), pack_bf16(z[2 * i + 1][2], z[2 * i + 1][3]));
                } else {
                    float *s0 = reinterpret_cast<float *>(p.fin) + state_base;
                    *reinterpret_cast<float4 *>(s0 + (size_t)v0 * DK + c) =
                        make_float4(z[2 * i][0], z[2 * i][1], z[2 * i + 1][0], z[2 * i + 1][1]);
                    *reinterpret_cast<float4 *>(s0 + (size_t)(v0 + 8) * DK + c) =
                        make_float4(z[2 * i][2], z[2 * i][3], z[2 * i + 1][2], z[2 * i + 1][3]);
                }
            }
        };
        for (int sc = 0; sc < nsub; ++sc) {
            const int L = !kMulti ? Lseq : (Lseq - LT * sc < LT ? Lseq - LT * sc : LT);   // rows of this block
            const int64_t row_base = row_first + LT * sc;
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            __syncthreads();

            if (tid < DK) {
                // ---- gate (log2 units) and its running sum G over the step, two channels
                // per thread, tokens 8 hf .. 8 hf + 7 (the partner lane holds the other half);
                // then the decayed tiles at the permuted columns
                const int c0 = 2 * (tid >> 1), hf = tid & 1, col = tau(c0);
                const float a2 = -__expf(p.A_log[h]) * kLog2e;
                const float2 a2v = make_float2(a2, a2);
                const float2 b2 = make_float2(a2 * p.dt_bias[h * DK + c0], a2 * p.dt_bias[h * DK + c0 + 1]);
                const float lb2 = p.lower_bound * kLog2e;
                float2 run = make_float2(0.f, 0.f), Gs[8];
#pragma unroll
                for (int tt = 0; tt < 8; ++tt) {
                    const int t = 8 * hf + tt;
                    if (t < L) {
                        const float2 zz = fma2(bf16x2_to_f2(*reinterpret_cast<const uint32_t *>(&sm.g[t][c0])), a2v, b2);
                        run.x += lb2 * __fdividef(1.f, 1.f + exp2f(zz.x));
                        run.y += lb2 * __fdividef(1.f, 1.f + exp2f(zz.y));
                    }
                    Gs[tt] = run;
                }
                const float2 other = make_float2(__shfl_xor_sync(0xffffffffu, run.x, 1),
                                                 __shfl_xor_sync(0xffffffffu, run.y, 1));
                const float2 GL = add2(run, other);
                const float2 off = hf ? other : make_float2(0.f, 0.f);
                const float2 eL = make_float2(exp2f(GL.x), exp2f(GL.y));
#pragma unroll
                for (int tt = 0; tt < 8; ++tt) {
                    const int t = 8 * hf + tt;
                    const float2 G = add2(Gs[tt], off);
                    const float2 e = make_float2(exp2f(G.x), exp2f(G.y));
                    const float2 ei = make_float2(exp2f(-G.x), exp2f(-G.y));
                    const float2 ec = mul2(eL, ei);   // 2^(G_L - G) <= 1
                    const float2 kx = bf16x2_to_f2(*reinterpret_cast<const uint32_t *>(&sm.k[t][c0]));
                    const float2 qx = bf16x2_to_f2(*reinterpret_cast<const uint32_t *>(&sm.q[t][c0]));
                    const float2 ke = mul2(kx, e), qe = mul2(qx, e), ki = mul2(kx, ei), kc = mul2(kx, ec);
                    *reinterpret_cast<uint32_t *>(&sm.kp[t][col]) = pack_bf16(ke.x, ke.y);
                    *reinterpret_cast<uint32_t *>(&sm.qp[t][col]) = pack_bf16(qe.x, qe.y);
                    *reinterpret_cast<uint32_t *>(&sm.kn[t][col]) = pack_bf16(ki.x, ki.y);
                    *reinterpret_cast<uint32_t *>(&sm.y[t][col]) = h2c(rbad, ke.x, ke.y);
                    *reinterpret_cast<uint32_t *>(&sm.y[LT + t][col]) = h2c(rbad, qe.x, qe.y);
                    *reinterpret_cast<uint32_t *>(&sm.kc[t][col]) = h2c(rbad, kc.x, kc.y);
                }
                if (hf == 0) *reinterpret_cast<float2 *>(&sm.gam[col]) = eL;
            } else {
                // ---- row norms of q and k (warps 4-7, four tokens each) and beta
                const int w4 = warp - 4;
#pragma unroll
                for (int tt = 0; tt < 4; ++tt) {
                    const int t = 4 * w4 + tt;
                    const uint2 qw = *reinterpret_cast<const uint2 *>(&sm.q[t][4 * lane]);
                    const uint2 kw = *reinterpret_cast<const uint2 *>(&sm.k[t][4 * lane]);
                    float sq = 0.f, sk = 0.f;
                    const uint32_t qa[2] = {qw.x, qw.y}, ka[2] = {kw.x, kw.y};
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const float q0 = __uint_as_float(qa[i] << 16), q1 = __uint_as_float(qa[i] & 0xFFFF0000u);
                        const float k0 = __uint_as_float(ka[i] << 16), k1 = __uint_as_float(ka[i] & 0xFFFF0000u);
                        sq = fmaf(q0, q0, fmaf(q1, q1, sq));
                        sk = fmaf(k0, k0, fmaf(k1, k1, sk));
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        sq += __shfl_xor_sync(0xffffffffu, sq, o);
                        sk += __shfl_xor_sync(0xffffffffu, sk, o);
                    }
                    if (lane == 0) {
                        sm.rq[t] = t < L ? rsqrtf(sq + 1e-6f) : 0.f;
                        sm.rk[t] = t < L ? rsqrtf(sk + 1e-6f) : 0.f;
                    }
                }
                if (tid >= NTS - LT) {
                    const int t = tid - (NTS - LT);
                    const float bl = t < L ? __bfloat162float(p.beta[(row_base + t) * p.H + h]) : 0.f;
                    sm.beta[t] = t < L ? 1.f / (1.f + exp2f(-bl * kLog2e)) : 0.f;
                }
            }
            __syncthreads();

            // ---- A (warp 0) and M' (warp 1): raw [k 2^G | q 2^G] x (k 2^-G)^T in bf16
            if (warp < 2) {
                const __nv_bfloat16 (*lhs)[RS] = warp == 0 ? sm.kp : sm.qp;
                float d[2][4] = {};
#pragma unroll
                for (int s = 0; s < DK / 16; ++s) {
                    uint32_t af[4], bf[4];
                    ldsm_x4(af, &lhs[(lane & 7) + 8 * ((lane >> 3) & 1)][16 * s + 8 * (lane >> 4)]);
                    ldsm_x4(bf, &sm.kn[(lane & 7) + 8 * (lane >> 4)][16 * s + 8 * ((lane >> 3) & 1)]);
                    mma_bf16x(d[0], af, bf[0], bf[1]);
                    mma_bf16x(d[1], af, bf[2], bf[3]);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int t = gq + 8 * hr, i0 = 8 * nt + 2 * qq;
                        if (warp == 0) {
                            const float f = sm.beta[t] * sm.rk[t];
                            sm.a[t][i0] = i0 < t ? f * sm.rk[i0] * d[nt][2 * hr] : 0.f;
                            sm.a[t][i0 + 1] = i0 + 1 < t ? f * sm.rk[i0 + 1] * d[nt][2 * hr + 1] : 0.f;
                        } else {
                            const float f = sm.rq[t];
                            *reinterpret_cast<uint32_t *>(&sm.mp[t][i0]) =
                                h2c(rbad, i0 <= t ? f * d[nt][2 * hr] : 0.f, i0 + 1 <= t ? f * d[nt][2 * hr + 1] : 0.f);
                        }
                    }
                }
                if (warp == 0) {   // A is in shared memory: release warp 2 (no wait here)
                    __syncwarp();
                    asm volatile("bar.arrive 1, 64;" ::: "memory");
                }
            }
            // ---- X = [k 2^G; q 2^G] S^T for this warp's 16 state rows (B from the z registers)
            float x[2][2][4] = {};   // [k rows | q rows][column half][fragment]
#pragma unroll
            for (int s = 0; s < DK / 16; ++s) {
                uint32_t a0[4], a1[4];
                ldsm_x4(a0, &sm.y[(lane & 7) + 8 * ((lane >> 3) & 1)][16 * s + 8 * (lane >> 4)]);
                ldsm_x4(a1, &sm.y[LT + (lane & 7) + 8 * ((lane >> 3) & 1)][16 * s + 8 * (lane >> 4)]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const uint32_t b0 = h2c(rbad, z[2 * s][2 * nt], z[2 * s][2 * nt + 1]);
                    const uint32_t b1 = h2c(rbad, z[2 * s + 1][2 * nt], z[2 * s + 1][2 * nt + 1]);
                    mma_f16(x[0][nt], a0, b0, b1);
                    mma_f16(x[1][nt], a1, b0, b1);
                }
            }
            // R = V - K_hat Gamma S^T (rows scaled by 1/|k_t|), fp16, into this warp's tile
            const float rk0 = sm.rk[gq], rk1 = sm.rk[gq + 8], rq0 = sm.rq[gq], rq1 = sm.rq[gq + 8];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int vl = 8 * nt + 2 * qq, vg = 16 * warp + vl;
                const float2 va = bf16x2_to_f2(*reinterpret_cast<const uint32_t *>(&sm.v[gq][vg]));
                const float2 vb = bf16x2_to_f2(*reinterpret_cast<const uint32_t *>(&sm.v[gq + 8][vg]));
                *reinterpret_cast<uint32_t *>(&sm.wr[warp][gq][vl]) =
                    h2c(rbad, va.x - rk0 * x[0][nt][0], va.y - rk0 * x[0][nt][1]);
                *reinterpret_cast<uint32_t *>(&sm.wr[warp][gq + 8][vl]) =
                    h2c(rbad, vb.x - rk1 * x[0][nt][2], vb.y - rk1 * x[0][nt][3]);
                x[1][nt][0] *= rq0; x[1][nt][1] *= rq0; x[1][nt][2] *= rq1; x[1][nt][3] *= rq1;
            }
            if (warp == 2) {
                // T = (I + A)^-1 by forward substitution, lane = column j (right-looking:
                // once x[r] is final it is added into every later row), then T' = T Diag(beta).
                // On warp 2 after its own products, once warp 0 has A in shared memory.
                asm volatile("bar.sync 1, 64;" ::: "memory");
                const int j = lane & (LT - 1);   // lanes 16-31 repeat the columns, without stores
                float acc[LT], xs[LT];
#pragma unroll
                for (int r = 0; r < LT; ++r) acc[r] = 0.f;
#pragma unroll
                for (int r = 0; r < LT; ++r) {
                    xs[r] = r == j ? 1.f : (r < j ? 0.f : -acc[r]);
#pragma unroll
                    for (int r2 = r + 1; r2 < LT; ++r2) acc[r2] = fmaf(sm.a[r2][r], xs[r], acc[r2]);
                }
                const float bj = sm.beta[j];
                if (lane < LT) {
#pragma unroll
                    for (int r = 0; r < LT; ++r) {
                        rbad |= !(fabsf(xs[r] * bj) <= 65504.f);
                        sm.tp[r][j] = __float2half_rn(xs[r] * bj);
                    }
                }
            }
            __syncthreads();   // T' (warp 2), M' (warp 1) and every warp's R are in shared memory
            if (sc + 1 < nsub) {   // q, k, g, v are dead: the next block's rows go in
                load_inputs(unit, sc + 1);
            } else if (next_unit(unit + gridDim.x) < units) {   // or the next unit's first block
                const int64_t nu = next_unit(unit + gridDim.x);
                load_inputs(nu, 0);
                if (tid == 0 && p.init)
                    prefetch_l2(static_cast<const unsigned char *>(p.init) + (size_t)nu * DK * DK * selt,
                                (uint32_t)(DK * DK * selt));
            }

            // ---- U = T' R, U' = Diag(1/|k|) U (fp16)
            {
                uint32_t af[4], bf[4];
                ldsm_x4(af, &sm.tp[(lane & 7) + 8 * ((lane >> 3) & 1)][8 * (lane >> 4)]);
                ldsm_x4_t(bf, &sm.wr[warp][(lane & 7) + 8 * ((lane >> 3) & 1)][8 * (lane >> 4)]);
                float u[2][4] = {};
                mma_f16(u[0], af, bf[0], bf[1]);
                mma_f16(u[1], af, bf[2], bf[3]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int vl = 8 * nt + 2 * qq;
                    *reinterpret_cast<uint32_t *>(&sm.wu[warp][gq][vl]) = h2c(rbad, rk0 * u[nt][0], rk0 * u[nt][1]);
                    *reinterpret_cast<uint32_t *>(&sm.wu[warp][gq + 8][vl]) = h2c(rbad, rk1 * u[nt][2], rk1 * u[nt][3]);
                }
            }
            __syncwarp();

            // ---- O = scale (Q_hat Gamma S^T + M' U') -> out
            {
                uint32_t af[4], bf[4];
                ldsm_x4(af, &sm.mp[(lane & 7) + 8 * ((lane >> 3) & 1)][8 * (lane >> 4)]);
                ldsm_x4_t(bf, &sm.wu[warp][(lane & 7) + 8 * ((lane >> 3) & 1)][8 * (lane >> 4)]);
                mma_f16(x[1][0], af, bf[0], bf[1]);
                mma_f16(x[1][1], af, bf[2], bf[3]);
                const float sc = p.scale;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int vg = 16 * warp + 8 * nt + 2 * qq;
                    if (gq < L)
                        *reinterpret_cast<uint32_t *>(p.out + ((row_base + gq) * p.H + h) * DK + vg) =
                            pack_bf16(sc * x[1][nt][0], sc * x[1][nt][1]);
                    if (gq + 8 < L)
                        *reinterpret_cast<uint32_t *>(p.out + ((row_base + gq + 8) * p.H + h) * DK + vg) =
                            pack_bf16(sc * x[1][nt][2], sc * x[1][nt][3]);
                }
            }

            // ---- S^T <- S^T Diag(Gamma_L) + U'^T (k 2^(G_L - G)), fp32 in the z registers
            if (p.fin || sc + 1 < nsub) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float2 gm = *reinterpret_cast<const float2 *>(&sm.gam[8 * j + 2 * qq]);
                    z[j][0] *= gm.x; z[j][1] *= gm.y; z[j][2] *= gm.x; z[j][3] *= gm.y;
                }
                uint32_t af[4];
                // A = U'^T (rows v, columns t): transposed 8x8 blocks of the [t][v] tile
                ldsm_x4_t(af, &sm.wu[warp][(lane & 7) + 8 * (lane >> 4)][8 * ((lane >> 3) & 1)]);
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    uint32_t bf[4];
                    ldsm_x4_t(bf, &sm.kc[(lane & 7) + 8 * ((lane >> 3) & 1)][8 * j + 8 * (lane >> 4)]);
                    mma_f16(z[j], af, bf[0], bf[1]);
                    mma_f16(z[j + 1], af, bf[2], bf[3]);
                }
                if (!kMulti && p.fin) store_state();
            }
        }   // blocks of the unit
        if (kMulti && p.fin) store_state();
    }
    if (rbad && p.err) atomicCAS(p.err, 0, kErrRange);   // an fp16 operand left its range
}

}  // namespace

cudaError_t launch_short(const Params &p, cudaStream_t stream) {
    const int64_t units = p.n_seqs * p.H;
    if (units == 0) return cudaSuccess;
    const int bytes = (int)sizeof(ShortSmem);
    const bool multi = p.T > LT;
    static std::atomic<bool> attr_done[2][kMaxDevices];
    cudaError_t e = once_per_device(attr_done[multi], [&](int) {
        return multi ? cudaFuncSetAttribute(kda_short_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)
                     : cudaFuncSetAttribute(kda_short_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    });
    if (e != cudaSuccess) return e;
    int sms = 0;
    if ((e = sm_count(sms)) != cudaSuccess) return e;
    const int64_t grid = units < 2 * (int64_t)sms ? units : 2 * (int64_t)sms;   // two CTAs per SM
    if (multi)
        kda_short_kernel<true><<<(unsigned)grid, NTS, bytes, stream>>>(p);
    else
        kda_short_kernel<false><<<(unsigned)grid, NTS, bytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
