// KDA forward on sm_103a with a two-CTA cluster per (sequence, head).
//
// The chunk algebra is the one of the tensor-core path (the KDA token recurrence
// of the FlashKDA README "Kernel API" unrolled over 64-token chunks; S is K x V,
// G the in-chunk cumulative log decay, Gamma = exp(G)):
//   A[t,i] = beta_t sum_c k[t,c] k[i,c] exp(G[t,c]-G[i,c])  (i < t)
//   M[t,i] =        sum_c q[t,c] k[i,c] exp(G[t,c]-G[i,c])  (i <= t)
//   T' = (I + A)^-1 Diag(beta);  W = T' (K_hat*Gamma);  U = T' V - W S
//   O  = scale ((Q_hat*Gamma) S + M U);   S <- Diag(Gamma_C) S + Kbar^T U
//
// Work split.  Only the last two lines are sequential across chunks; everything
// before them depends on the chunk's own inputs.  So:
//   CTA rank 0 ("front") runs the chunk-parallel part one chunk ahead:
//     warps 0-7  prologue of chunk m: gate, norms, block-local decay, the
//                operands of G1 and the chain's K_hat*Gamma, Q_hat*Gamma, Kbar;
//                issues G1 = [Kp; Qp] x Kn^T into a double-buffered TMEM slot;
//     warps 8-11 solver of chunk m-1: A and M out of TMEM, the blocked
//                inverse, T' (fp16);
//     warp 12    control: issues G1, ships the prologue's tiles, prefetches
//                the next raw tiles, so the prologue never waits on the chain;
//     both groups ship their tiles into the chain CTA's shared memory with bulk
//     shared->shared copies that complete as transaction bytes on the chain's
//     per-slot mbarrier.
//   CTA rank 1 ("chain") owns the whole state (V = 128) in tensor memory:
//     G2u = [T'; 0] x V and G3 = [-W; Q_hat*Gamma] x S  -> U | Q Gamma S
//     U readout, S decay
//     G4 = Kbar^T U -> S,  G5 = [0; M] x U -> O
//     O and S readout; W for the next chunk (G2w = [T'; 0] x K_hat*Gamma) is
//     computed and read out beside this, off the sequential path.
// Flow control: the chain arrives remotely on the front's "slot free" barriers
// (per-slot tiles K_bar, M, Gamma_C) and "single free" barrier (single-buffered
// tiles T', K_hat*Gamma, Q_hat*Gamma); the front waits on them before shipping.
//
// Precision and exponent handling are those of the single-CTA path: G1 on bf16
// operands of the raw q/k scaled by 16-token-block-local decay factors, the
// other GEMMs on fp16 operands, fp32 accumulators, fp32 state.  Every wait is
// bounded (2 s); a timeout sets the device error word and both CTAs unwind.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

using namespace sm103;

constexpr int C = kChunk;
constexpr int DK = kHeadDim;
constexpr int NT = 416;            // 13 warps in both CTAs
constexpr int NP = 256;            // front prologue group: warps 0-7
constexpr int NS = 128;            // front solver group: warps 8-11
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWait = 2000000000ull;   // 2 s per wait
constexpr int LDA = 68;             // fp32 row stride of A and T (16-byte aligned rows)
constexpr uint32_t kChunkBytes = 16384 * 3 + 512 + 8192 * 2;   // front -> chain per chunk
constexpr int kOrderMax = 256;     // varlen batches up to this many sequences run longest first

// ---- front shared memory
constexpr uint32_t F_RAW = 0;          // 2 slots x {q, k, g}: 16 KB each, 2 x [64 t][64 c]
constexpr uint32_t F_SLOT = 49152;
constexpr uint32_t F_AMA = 98304;      // [Kp; Qp]: 2 x [128][64] bf16
constexpr uint32_t F_AMB = 131072;     // Kn variants: 2 x [160][64] bf16
constexpr uint32_t F_MST = 172032;     // M staging fp16 [64 t][64 i]
constexpr uint32_t F_AMAT = 180224;    // A fp32 [64][68]; T' staging (fp16) after the inverse
constexpr uint32_t F_TF = 197632;      // T fp32 [64][68]
constexpr uint32_t F_ZS = 215040;      // inverse scratch fp32 [3][16][16]
// ---- chain shared memory
constexpr uint32_t C_B2 = 0;           // K_hat*Gamma 2 x [64 i][64 c] | V 2 x [64 t][64 v] (MN-major)
constexpr uint32_t C_G3A = 32768;      // [-W; Q_hat*Gamma]: 2 x [128][64] (K-major)
constexpr uint32_t C_KB = 65536;       // 2 slots x Kbar 2 x [64 i][64 c] (MN-major)
constexpr uint32_t C_TZM = 98304;      // T' | Z | M0 | Z | M1, each [64][64] (K-major)
constexpr uint32_t C_SB = 139264;      // S fp16 2 x [128 c][64 v] (MN-major)
constexpr uint32_t C_UT = 172032;      // U fp16 2 x [64 i][64 v] (MN-major)
constexpr uint32_t SMALL = 218112;     // common offset in both CTAs (remote addresses)

struct Small {
    float rq[2][C], rk[2][C], beta[2][C];   // front, per slot
    float btot[4][DK];                       // front
    float gamC_f[2][DK];                     // front: exp(G_C) per slot (copy source)
    float gamC_c[2][DK];                     // chain: copy destination
    uint64_t raw_full[2], g1_done[2], am_free[2], s_done[2], slot_free[2], single_free, pdone[2];
    uint64_t full[2], v_full, mma_bar, w_bar;
    uint32_t tmem_base;
    int abort_p, abort_s, abort_c;
};
constexpr uint32_t SMEM_BYTES = SMALL + sizeof(Small) + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

__device__ __forceinline__ int variant_off(int bt) { return 8 * bt * (bt + 1); }

// G1's A-operand rows hold the 16-token blocks in the order 0, 3, 1, 2, so that
// each 32-lane TMEM quarter of the result needs 80 of the 160 variant columns
// (blocks 0 and 3: variants 0 and 3; blocks 1 and 2: variants 1 and 2).
__device__ __forceinline__ int row_block_of(int blk) { return (0x1320 >> (4 * blk)) & 0xF; }
__device__ __forceinline__ int block_of_row_block(int rb) { return (0x2130 >> (4 * rb)) & 0xF; }

// 16x16 = 16xK * Kx16 block product on the tensor cores (mma.sync, tf32 operands
// rounded to nearest, fp32 accumulation).
// A(r, k) = a[r * lda + k], B(k, c) = b[k * ldb + c]; acc holds two 16x8 tiles.
template <int K>
__device__ __forceinline__ void block_mma_16x16(const float *a, int lda, const float *b, int ldb,
                                                int lane, float (&acc)[2][4]) {
    const int g = lane >> 2, q = lane & 3;
    float av[K / 8][4], bv[K / 8][2][2];
#pragma unroll
    for (int kk = 0; kk < K / 8; ++kk) {   // all operand loads first
        av[kk][0] = a[g * lda + 8 * kk + q];
        av[kk][1] = a[(g + 8) * lda + 8 * kk + q];
        av[kk][2] = a[g * lda + 8 * kk + q + 4];
        av[kk][3] = a[(g + 8) * lda + 8 * kk + q + 4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            bv[kk][nt][0] = b[(8 * kk + q) * ldb + 8 * nt + g];
            bv[kk][nt][1] = b[(8 * kk + q + 4) * ldb + 8 * nt + g];
        }
    }
#pragma unroll
    for (int kk = 0; kk < K / 8; ++kk) {
        uint32_t ah[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ah[i] = to_tf32(av[kk][i]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            uint32_t bh[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) bh[i] = to_tf32(bv[kk][nt][i]);
            mma_tf32_16x8x8(acc[nt], ah, bh);
        }
    }
}

// Off-diagonal levels of the blocked inverse on one warp per block pair (bt, ba),
// bt - ba = D: Z = sum_{ba <= m < bt} A[bt][m] T[m][ba], T[bt][ba] = -T[bt][bt] Z.
template <int D>
__device__ __forceinline__ void inverse_level_mma(const float *Amat, float *Tf, float *Zs, int wq,
                                                  int lane) {
    if (wq < 4 - D) {
        const int ba = wq, bt = ba + D, g = lane >> 2, q = lane & 3;
        float z[2][4] = {};
        block_mma_16x16<16 * D>(Amat + (16 * bt) * LDA + 16 * ba, LDA, Tf + (16 * ba) * LDA + 16 * ba,
                                LDA, lane, z);
        float *zt = Zs + wq * 256;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            zt[g * 16 + 8 * nt + 2 * q] = z[nt][0];
            zt[g * 16 + 8 * nt + 2 * q + 1] = z[nt][1];
            zt[(g + 8) * 16 + 8 * nt + 2 * q] = z[nt][2];
            zt[(g + 8) * 16 + 8 * nt + 2 * q + 1] = z[nt][3];
        }
        __syncwarp();
        float t2[2][4] = {};
        block_mma_16x16<16>(Tf + (16 * bt) * LDA + 16 * bt, LDA, zt, 16, lane, t2);
        float *dst = Tf + (16 * bt) * LDA + 16 * ba;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            dst[g * LDA + 8 * nt + 2 * q] = -t2[nt][0];
            dst[g * LDA + 8 * nt + 2 * q + 1] = -t2[nt][1];
            dst[(g + 8) * LDA + 8 * nt + 2 * q] = -t2[nt][2];
            dst[(g + 8) * LDA + 8 * nt + 2 * q + 1] = -t2[nt][3];
        }
    }
}

// One off-diagonal level of the blocked inverse T = (I + A)^-1 (16x16 blocks):
// for every block pair (bt, ba) with bt - ba = D,
//   Z = sum_{ba <= m < bt} A[bt][m] T[m][ba],   T[bt][ba] = -T[bt][bt] Z.
// Each task computes four adjacent columns of one row (float4 accumulators).
template <int D>
__device__ __forceinline__ void inverse_level(const float *Amat, float *Tf, float *Zs, int stid,
                                              int nthreads, uint32_t bar_id) {
    constexpr int NTASK = (4 - D) * 64;
    for (int task = stid; task < NTASK; task += nthreads) {
        const int ba = task >> 6, r = (task >> 2) & 15, jg = task & 3, bt = ba + D;
        const float *arow = Amat + (16 * bt + r) * LDA + 16 * ba;
        const float *tcol = Tf + (16 * ba) * LDA + 16 * ba + 4 * jg;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 16 * D; ++q) {
            const float a = arow[q];
            const float4 tv = *reinterpret_cast<const float4 *>(tcol + q * LDA);
            acc.x = fmaf(a, tv.x, acc.x);
            acc.y = fmaf(a, tv.y, acc.y);
            acc.z = fmaf(a, tv.z, acc.z);
            acc.w = fmaf(a, tv.w, acc.w);
        }
        *reinterpret_cast<float4 *>(Zs + ba * 256 + r * 16 + 4 * jg) = acc;
    }
    named_bar(bar_id, nthreads);
    for (int task = stid; task < NTASK; task += nthreads) {
        const int ba = task >> 6, r = (task >> 2) & 15, jg = task & 3, bt = ba + D;
        const float *trow = Tf + (16 * bt + r) * LDA + 16 * bt;   // T[bt][bt] row (zero above r)
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float a = trow[q];
            const float4 z = *reinterpret_cast<const float4 *>(Zs + ba * 256 + q * 16 + 4 * jg);
            acc.x = fmaf(a, z.x, acc.x);
            acc.y = fmaf(a, z.y, acc.y);
            acc.z = fmaf(a, z.z, acc.z);
            acc.w = fmaf(a, z.w, acc.w);
        }
        *reinterpret_cast<float4 *>(Tf + (16 * bt + r) * LDA + 16 * ba + 4 * jg) =
            make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    }
    named_bar(bar_id, nthreads);
}

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

struct TmaMaps {
    CUtensorMap q, k, g, v;
};

__device__ __forceinline__ void set_err(const Params &p) {
    if (p.err) atomicExch(p.err, 8);
}

// ============================================================== front CTA
__device__ __forceinline__ void run_front(const TmaMaps &maps, const Params &p, unsigned char *smem,
                                          Small &sm, uint32_t tmem, int64_t h, int64_t row_base,
                                          int64_t len, int nchunks) {
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t chain_small = mapa_shared(smem_u32(&sm), 1);
    auto chain_addr = [&](uint32_t off) { return mapa_shared(sbase + off, 1); };
    auto chain_bar = [&](uint64_t *local_bar) {
        return chain_small + (smem_u32(local_bar) - smem_u32(&sm));
    };

    auto issue_raw = [&](int chunk) {
        const int s = chunk & 1;
        const int row = (int)(row_base + (int64_t)chunk * C);
        unsigned char *base = smem + F_RAW + s * F_SLOT;
        mbar_arrive_expect_tx(&sm.raw_full[s], 3 * 16384);
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_3d(base + kb * 8192, &maps.q, &sm.raw_full[s], kb * 64, (int)h, row);
            tma_load_3d(base + 16384 + kb * 8192, &maps.k, &sm.raw_full[s], kb * 64, (int)h, row);
            tma_load_3d(base + 32768 + kb * 8192, &maps.g, &sm.raw_full[s], kb * 64, (int)h, row);
        }
    };

    if (tid < NP) {
        // ------------------------------------------------ prologue group
        const float a2 = -__expf(p.A_log[h]) * kLog2e;
        const float lb2 = p.lower_bound * kLog2e;
        const int blk = warp >> 1;                   // 16-token block
        const int arow0 = 16 * row_block_of(blk);    // its rows in G1's A operand
        const int c = (warp & 1) * 64 + 2 * lane;    // channel pair (c, c+1)
        const int kb = c >> 6, cc = c & 63;
        const float b0 = a2 * p.dt_bias[h * DK + c], b1 = a2 * p.dt_bias[h * DK + c + 1];
        for (int m = 0; m < nchunks; ++m) {
            const int s = m & 1;
            const int64_t cs = (int64_t)m * C;
            const int L = (int)((len - cs) < C ? (len - cs) : C);
            const int64_t row0 = row_base + cs;
            const uint32_t rq_off = F_RAW + s * F_SLOT, rk_off = rq_off + 16384, rg_off = rq_off + 32768;
            if (tid == 0) {
                bool ok = mbar_wait(&sm.raw_full[s], (m >> 1) & 1, kWait);
                if (ok && m >= 2) ok = mbar_wait(&sm.s_done[s], ((m - 2) >> 1) & 1, kWait);
                if (!ok) { set_err(p); sm.abort_p = 1; }
            }
            named_bar(1, NP);
            if (sm.abort_p) break;

            // beta logits: global loads issued first, consumed after the norms
            float bl0 = 0.f, bl1 = 0.f;
            if (warp == 0) {
                if (lane < L) bl0 = __bfloat162float(p.beta[(row0 + lane) * p.H + h]);
                if (lane + 32 < L) bl1 = __bfloat162float(p.beta[(row0 + lane + 32) * p.H + h]);
            }
            // norms: half-warps take one row each (8 channels per lane, 16-byte loads)
            {
                const int hw = lane >> 4, l16 = lane & 15;
                const int kbb = l16 >> 3, col = (l16 & 7) * 8;
                float sq[4], sk[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int t = warp + (NP / 32) * (2 * u + hw);
                    const uint32_t off = kbb * 8192 + sw128_off(t, col);
                    const uint4 qv = *reinterpret_cast<const uint4 *>(smem + rq_off + off);
                    const uint4 kv = *reinterpret_cast<const uint4 *>(smem + rk_off + off);
                    const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
                    float a = 0.f, b = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        a = fmaf(bf16lo(qw[i]), bf16lo(qw[i]), a);
                        a = fmaf(bf16hi(qw[i]), bf16hi(qw[i]), a);
                        b = fmaf(bf16lo(kw[i]), bf16lo(kw[i]), b);
                        b = fmaf(bf16hi(kw[i]), bf16hi(kw[i]), b);
                    }
                    sq[u] = a;
                    sk[u] = b;
                }
#pragma unroll
                for (int o = 8; o > 0; o >>= 1)
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        sq[u] += __shfl_xor_sync(0xffffffffu, sq[u], o);
                        sk[u] += __shfl_xor_sync(0xffffffffu, sk[u], o);
                    }
                if (l16 == 0) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int t = warp + (NP / 32) * (2 * u + hw);
                        sm.rq[s][t] = t < L ? rsqrtf(sq[u] + 1e-6f) : 0.f;
                        sm.rk[s][t] = t < L ? rsqrtf(sk[u] + 1e-6f) : 0.f;
                    }
                }
            }
            if (warp == 0) {
                sm.beta[s][lane] = lane < L ? 1.f / (1.f + exp2f(-bl0 * kLog2e)) : 0.f;
                sm.beta[s][lane + 32] = lane + 32 < L ? 1.f / (1.f + exp2f(-bl1 * kLog2e)) : 0.f;
            }

            // gate and block-local cumulative decay (log2 units)
            float H0[16], H1[16];
            {
                float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const int t = blk * 16 + r;
                    const uint32_t gv =
                        *reinterpret_cast<const uint32_t *>(smem + rg_off + kb * 8192 + sw128_off(t, cc));
                    if (t < L) {
                        acc0 += lb2 * __fdividef(1.f, 1.f + exp2f(fmaf(bf16lo(gv), a2, b0)));
                        acc1 += lb2 * __fdividef(1.f, 1.f + exp2f(fmaf(bf16hi(gv), a2, b1)));
                    }
                    H0[r] = acc0;
                    H1[r] = acc1;
                }
                sm.btot[blk][c] = acc0;
                sm.btot[blk][c + 1] = acc1;
            }
            named_bar(1, NP);

            float Gs0[4], Gs1[4], s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                Gs0[bb] = s0;
                Gs1[bb] = s1;
                s0 += sm.btot[bb][c];
                s1 += sm.btot[bb][c + 1];
            }
            if (blk == 0) {
                sm.gamC_f[s][c] = exp2f(s0);
                sm.gamC_f[s][c + 1] = exp2f(s1);
            }
            const float Fs0 = exp2f(Gs0[blk]), Fs1 = exp2f(Gs1[blk]);
            const float FC0 = exp2f(s0 - Gs0[blk]), FC1 = exp2f(s1 - Gs1[blk]);
            float D0[4], D1[4];
#pragma unroll
            for (int bt = 0; bt < 4; ++bt) {
                D0[bt] = bt > blk ? exp2f(Gs0[bt] - Gs0[blk]) : 1.f;
                D1[bt] = bt > blk ? exp2f(Gs1[bt] - Gs1[blk]) : 1.f;
            }
            // [Kp; Qp] and Kn are free once G1 of the previous chunk completed
            if (tid == 0 && m >= 1) {
                if (!mbar_wait(&sm.g1_done[(m - 1) & 1], ((m - 1) >> 1) & 1, kWait)) {
                    set_err(p);
                    sm.abort_p = 1;
                }
            }
            named_bar(1, NP);
            if (sm.abort_p) break;

#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int t = blk * 16 + r;
                const uint32_t off = kb * 8192 + sw128_off(t, cc);
                const uint32_t qv = *reinterpret_cast<const uint32_t *>(smem + rq_off + off);
                const uint32_t kv = *reinterpret_cast<const uint32_t *>(smem + rk_off + off);
                const float rq = sm.rq[s][t], rk = sm.rk[s][t];
                const float q0 = t < L ? bf16lo(qv) : 0.f, q1 = t < L ? bf16hi(qv) : 0.f;
                const float k0 = t < L ? bf16lo(kv) : 0.f, k1 = t < L ? bf16hi(kv) : 0.f;
                const float e10 = exp2f(H0[r]), e11 = exp2f(H1[r]);
                const float e20 = exp2f(-H0[r]), e21 = exp2f(-H1[r]);
                const float kp0 = k0 * e10, kp1 = k1 * e11;
                const float qp0 = q0 * e10, qp1 = q1 * e11;
                const float kn0 = k0 * e20, kn1 = k1 * e21;
                *reinterpret_cast<uint32_t *>(smem + F_AMA + kb * 16384 + sw128_off(arow0 + r, cc)) =
                    pack_bf16(kp0, kp1);
                *reinterpret_cast<uint32_t *>(smem + F_AMA + kb * 16384 +
                                              sw128_off(64 + arow0 + r, cc)) = pack_bf16(qp0, qp1);
#pragma unroll
                for (int bt = 0; bt < 4; ++bt) {
                    if (bt >= blk) {
                        const int row = variant_off(bt) + t;
                        *reinterpret_cast<uint32_t *>(smem + F_AMB + kb * 20480 + sw128_off(row, cc)) =
                            pack_bf16(kn0 * D0[bt], kn1 * D1[bt]);
                    }
                }
                // chain operands, in place of the raw tiles (same layouts)
                *reinterpret_cast<uint32_t *>(smem + rq_off + off) =
                    pack_f16(qp0 * (Fs0 * rq), qp1 * (Fs1 * rq));        // Q_hat*Gamma
                *reinterpret_cast<uint32_t *>(smem + rk_off + off) =
                    pack_f16(kp0 * (Fs0 * rk), kp1 * (Fs1 * rk));        // K_hat*Gamma
                *reinterpret_cast<uint32_t *>(smem + rg_off + off) =
                    pack_f16(kn0 * (FC0 * rk), kn1 * (FC1 * rk));        // Kbar
            }
            fence_proxy_async_smem();
            named_bar(1, NP);

            if (tid == 0) mbar_arrive(&sm.pdone[s]);   // operands and rq/rk/beta of chunk m ready
        }
    } else if (warp == 12) {
        // ------------------------------------------------ control warp (lane 0)
        if (lane == 0) {
            if (nchunks > 0) issue_raw(0);
            if (nchunks > 1) issue_raw(1);
            for (int m = 0; m < nchunks; ++m) {
                const int s = m & 1;
                const uint32_t rq_off = F_RAW + s * F_SLOT, rk_off = rq_off + 16384, rg_off = rq_off + 32768;
                bool ok = mbar_wait(&sm.pdone[s], (m >> 1) & 1, kWait);
                if (ok && m >= 2) ok = mbar_wait(&sm.am_free[s], ((m - 2) >> 1) & 1, kWait);
                if (ok) {
                    tc_fence_after();
                    const uint32_t id = idesc_bf16(128, 160, false, false);
                    for (int ks = 0; ks < DK / 16; ++ks) {
                        const uint64_t ad =
                            sdesc_sw128(sbase + F_AMA + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                        const uint64_t bd =
                            sdesc_sw128(sbase + F_AMB + (ks >> 2) * 20480 + (ks & 3) * 32, 16, 1024);
                        mma_bf16(tmem + 256 * s, ad, bd, id, ks > 0);
                    }
                    mma_commit(&sm.g1_done[s]);
                }
                if (ok && m >= 2) ok = mbar_wait_cluster(&sm.slot_free[s], ((m - 2) >> 1) & 1, kWait);
                const uint32_t full = chain_bar(&sm.full[s]);
                if (ok) {
                    bulk_copy_to_peer(chain_addr(C_KB + s * 16384), sbase + rg_off, 16384, full);
                    bulk_copy_to_peer(chain_small + (smem_u32(&sm.gamC_c[s][0]) - smem_u32(&sm)),
                                      smem_u32(&sm.gamC_f[s][0]), 512, full);
                }
                if (ok && m >= 1) ok = mbar_wait_cluster(&sm.single_free, (m - 1) & 1, kWait);
                if (ok) {
                    bulk_copy_to_peer(chain_addr(C_G3A + 8192), sbase + rq_off, 8192, full);
                    bulk_copy_to_peer(chain_addr(C_G3A + 16384 + 8192), sbase + rq_off + 8192, 8192, full);
                    bulk_copy_to_peer(chain_addr(C_B2), sbase + rk_off, 16384, full);
                }
                bulk_commit();
                bulk_wait_read0();
                if (!ok) {
                    set_err(p);
                    sm.abort_p = 1;
                    sm.abort_s = 1;
                    break;
                }
                if (m + 2 < nchunks) issue_raw(m + 2);
            }
            bulk_wait0();
        }
    } else {
        // ------------------------------------------------ solver group
        const int stid = tid - NP, sw = warp - 8;          // sw = TMEM lane quarter
        float *Amat = reinterpret_cast<float *>(smem + F_AMAT);
        float *Tf = reinterpret_cast<float *>(smem + F_TF);
        float *Zs = reinterpret_cast<float *>(smem + F_ZS);
        for (int m = 0; m < nchunks; ++m) {
            const int s = m & 1;
            if (stid == 0) {
                bulk_wait_read0();   // previous T'/M staging shipped
                if (!mbar_wait(&sm.pdone[s], (m >> 1) & 1, kWait) ||
                    !mbar_wait(&sm.g1_done[s], (m >> 1) & 1, kWait)) {
                    set_err(p);
                    sm.abort_s = 1;
                }
            }
            named_bar(2, NS);
            if (sm.abort_s) break;
            tc_fence_after();

            // A (fp32, beta_t/|k_t| x 1/|k_i|, strictly lower) and M (fp16, 1/|q_t| x 1/|k_i|)
            {
                const bool is_m = sw >= 2;
                const int lr = (sw & 1) * 32 + lane;            // row within the A or M half
                const int bt = block_of_row_block(lr >> 4);
                const int t = 16 * bt + (lr & 15);
                const float rowf = is_m ? sm.rq[s][t] : sm.beta[s][t] * sm.rk[s][t];
                for (int i = 16 * (bt + 1); i < 64; i += 16) {
                    if (is_m) {
                        sts128(sbase + F_MST + sw128_off(t, i), 0, 0, 0, 0);
                        sts128(sbase + F_MST + sw128_off(t, i + 8), 0, 0, 0, 0);
                    } else {
                        float4 *dst = reinterpret_cast<float4 *>(Amat + t * LDA + i);
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) dst[e4] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                // this quarter's five 16-column chunks: {0, 6..9} or {1..5}
                auto chunk_of = [&](int k) { return (sw & 1) ? 1 + k : (k == 0 ? 0 : 5 + k); };
                auto emit = [&](int jj, float (&r)[16]) {
                    const int vo = variant_off(bt);
                    if (16 * jj >= vo && 16 * jj < vo + 16 * (bt + 1)) {
                        const int ib = 16 * jj - vo;
                        const float4 *rk4 = reinterpret_cast<const float4 *>(&sm.rk[s][ib]);
                        float cf[16];
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) {
                            const float4 x = rk4[e4];
                            cf[4 * e4] = x.x; cf[4 * e4 + 1] = x.y; cf[4 * e4 + 2] = x.z; cf[4 * e4 + 3] = x.w;
                        }
                        const int lim = is_m ? t - ib : t - ib - 1;   // last column kept
#pragma unroll
                        for (int e = 0; e < 16; ++e) r[e] = (e <= lim) ? rowf * cf[e] * r[e] : 0.f;
                        if (is_m) {
                            st_pack16<true>(sbase + F_MST, t, ib, r);
                        } else {
                            float4 *dst = reinterpret_cast<float4 *>(Amat + t * LDA + ib);
#pragma unroll
                            for (int e4 = 0; e4 < 4; ++e4)
                                dst[e4] = make_float4(r[4 * e4], r[4 * e4 + 1], r[4 * e4 + 2], r[4 * e4 + 3]);
                        }
                    }
                };
                float r0[16], r1[16], r2[16];
                tmem_ld16(tmem_addr(tmem, sw * 32, 256 * s + 16 * chunk_of(0)), r0);
                tmem_ld16(tmem_addr(tmem, sw * 32, 256 * s + 16 * chunk_of(1)), r1);
                tmem_ld16(tmem_addr(tmem, sw * 32, 256 * s + 16 * chunk_of(2)), r2);
                tmem_ld_wait();
                emit(chunk_of(0), r0);
                emit(chunk_of(1), r1);
                emit(chunk_of(2), r2);
                tmem_ld16(tmem_addr(tmem, sw * 32, 256 * s + 16 * chunk_of(3)), r0);
                tmem_ld16(tmem_addr(tmem, sw * 32, 256 * s + 16 * chunk_of(4)), r1);
                tmem_ld_wait();
                emit(chunk_of(3), r0);
                emit(chunk_of(4), r1);
            }
            tc_fence_before();
            named_bar(2, NS);
            if (stid == 0) mbar_arrive(&sm.am_free[s]);

            // T = (I + A)^-1: 16x16 diagonal blocks, then off-diagonal block levels
            if (stid < 64) {
                const int bb = stid >> 4, j = stid & 15;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) x[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
                for (int r = 1; r < 16; ++r) {
                    float acc = 0.f;
#pragma unroll
                    for (int q = 0; q < r; ++q)
                        acc = fmaf(Amat[(16 * bb + r) * LDA + 16 * bb + q], x[q], acc);
                    if (r > j) x[r] = -acc;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Tf[(16 * bb + r) * LDA + 16 * bb + j] = x[r];
            }
            named_bar(2, NS);
            inverse_level_mma<1>(Amat, Tf, Zs, sw, lane);
            named_bar(2, NS);
            inverse_level_mma<2>(Amat, Tf, Zs, sw, lane);
            named_bar(2, NS);
            inverse_level_mma<3>(Amat, Tf, Zs, sw, lane);
            named_bar(2, NS);
            // T' = T Diag(beta), fp16, into the staging tile (over the dead A)
            {
                const int t = stid >> 1, i0 = (stid & 1) * 32;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float r[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int i = i0 + 16 * hh + e;
                        r[e] = (i <= t) ? Tf[t * LDA + i] * sm.beta[s][i] : 0.f;
                    }
                    st_pack16<true>(sbase + F_AMAT, t, i0 + 16 * hh, r);
                }
            }
            fence_proxy_async_smem();
            named_bar(2, NS);
            if (stid == 0) {
                mbar_arrive(&sm.s_done[s]);
                bool ok = true;
                const uint32_t full = chain_bar(&sm.full[s]);
                if (m >= 2) ok = mbar_wait_cluster(&sm.slot_free[s], ((m - 2) >> 1) & 1, kWait);
                if (ok) bulk_copy_to_peer(chain_addr(C_TZM + 16384 + s * 16384), sbase + F_MST, 8192, full);
                if (ok && m >= 1) ok = mbar_wait_cluster(&sm.single_free, (m - 1) & 1, kWait);
                if (ok) bulk_copy_to_peer(chain_addr(C_TZM), sbase + F_AMAT, 8192, full);
                bulk_commit();
                if (!ok) { set_err(p); sm.abort_s = 1; sm.abort_p = 1; }
            }
        }
        if (stid == 0) bulk_wait0();
    }
}

// ============================================================== chain CTA
__device__ __forceinline__ void run_chain(const TmaMaps &maps, const Params &p, unsigned char *smem,
                                          Small &sm, uint32_t tmem, int64_t n, int64_t h,
                                          int64_t row_base, int64_t len, int nchunks) {
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = (warp >> 2) & 1;   // warps 0-7: (lane quarter, column half)
    const uint32_t D_S = tmem, D_W = tmem + 128, D_U = tmem + 256;
    const uint32_t front_small = mapa_shared(smem_u32(&sm), 0);
    auto front_bar = [&](uint64_t *local_bar) {
        return front_small + (smem_u32(local_bar) - smem_u32(&sm));
    };
    const size_t state_base = (size_t)(n * p.H + h) * DK * DK;

    auto issue_v = [&](int chunk) {
        const int row = (int)(row_base + (int64_t)chunk * C);
        mbar_arrive_expect_tx(&sm.v_full, 16384);
        tma_load_3d(smem + C_B2 + 16384, &maps.v, &sm.v_full, 0, (int)h, row);
        tma_load_3d(smem + C_B2 + 16384 + 8192, &maps.v, &sm.v_full, 64, (int)h, row);
    };
    // waits done by thread 0 and published to the CTA; returns true to abort
    auto lead_wait = [&](bool ok) -> bool {
        if (tid == 0 && !ok) { set_err(p); sm.abort_c = 1; }
        __syncthreads();
        return sm.abort_c != 0;
    };
    auto convert_v = [&]() {
        for (int k16 = tid; k16 < 1024; k16 += NT) {
            uint4 *ptr = reinterpret_cast<uint4 *>(smem + C_B2 + 16384 + k16 * 16);
            uint4 x = *ptr;
            x.x = pack_f16(bf16lo(x.x), bf16hi(x.x));
            x.y = pack_f16(bf16lo(x.y), bf16hi(x.y));
            x.z = pack_f16(bf16lo(x.z), bf16hi(x.z));
            x.w = pack_f16(bf16lo(x.w), bf16hi(x.w));
            *ptr = x;
        }
    };
    // -W (D_W lanes 0..63) -> rows 0..63 of the G3 A operand; warps 8, 9
    auto read_w = [&]() {
        if (warp == 8 || warp == 9) {
            const int t = (warp - 8) * 32 + lane;
            for (int jj = 0; jj < 8; ++jj) {
                float r[16];
                tmem_ld16(tmem_addr(D_W, (warp & 3) * 32, 16 * jj), r);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) r[e] = -r[e];
                st_pack16<true>(sbase + C_G3A + (jj >> 2) * 16384, t, (16 * jj) & 63, r);
            }
        }
    };
    // D_S columns of this warp (lane quarter, column half) times g, written back
    auto scale_s = [&](float g) {
        float r[4][16];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
            tmem_ld16(tmem_addr(D_S, quarter * 32, 64 * half + 16 * jj), r[jj]);
        tmem_ld_wait();
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
            for (int e = 0; e < 16; ++e) r[jj][e] *= g;
            tmem_st16(tmem_addr(D_S, quarter * 32, 64 * half + 16 * jj), r[jj]);
        }
        tmem_st_wait();
    };
    auto issue_g2w = [&]() {
        const uint32_t id = idesc_fp16(128, 128, false, true);
        for (int ks = 0; ks < C / 16; ++ks)
            mma_bf16(D_W, sdesc_sw128(sbase + C_TZM + ks * 32, 16, 1024),
                     sdesc_sw128(sbase + C_B2 + ks * 2048, 8192, 1024), id, ks > 0);
        mma_commit(&sm.w_bar);
    };

    // zero tiles (rows 64..127 of [T'; 0], rows 0..63 of [0; M0] and [0; M1])
    for (int k16 = tid; k16 < 512; k16 += NT) {
        sts128(sbase + C_TZM + 8192 + k16 * 16, 0, 0, 0, 0);
        sts128(sbase + C_TZM + 24576 + k16 * 16, 0, 0, 0, 0);
    }
    // initial state -> D_S (fp32) and S fp16 operand copy; warps 0-7
    if (warp < 8) {
        const int c = quarter * 32 + lane;
        for (int jj = 0; jj < 4; ++jj) {
            const int v0 = 64 * half + 16 * jj;
            float r[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                float x = 0.f;
                if (p.init) {
                    const size_t off = state_base + (size_t)(v0 + e) * DK + c;
                    x = p.state_type == kStateBF16
                            ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.init)[off])
                            : reinterpret_cast<const float *>(p.init)[off];
                }
                r[e] = x;
            }
            tmem_st16(tmem_addr(D_S, quarter * 32, 64 * half + 16 * jj), r);
            st_pack16<true>(sbase + C_SB + half * 16384, c, 16 * jj, r);
        }
        tmem_st_wait();
    }
    if (tid == 0) {
        if (nchunks > 0) {
            mbar_arrive_expect_tx(&sm.full[0], kChunkBytes);
            issue_v(0);
        }
        if (nchunks > 1) mbar_arrive_expect_tx(&sm.full[1], kChunkBytes);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    uint32_t ph_mma = 0;
    if (nchunks > 0) {
        bool ok = true;
        if (tid == 0) {
            ok = mbar_wait(&sm.full[0], 0, kWait) && mbar_wait(&sm.v_full, 0, kWait);
        }
        if (lead_wait(ok)) nchunks = 0;
        if (nchunks > 0) {
            tc_fence_after();
            if (warp < 8) scale_s(sm.gamC_c[0][quarter * 32 + lane]);
            convert_v();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                issue_g2w();
                ok = mbar_wait(&sm.w_bar, 0, kWait);
            }
            if (lead_wait(ok)) nchunks = 0;
            tc_fence_after();
            read_w();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
        }
    }

    for (int m = 0; m < nchunks; ++m) {
        const int s = m & 1;
        const int64_t cs = (int64_t)m * C;
        const int L = (int)((len - cs) < C ? (len - cs) : C);
        const int64_t row0 = row_base + cs;
        bool ok = true;

        // (a) U~ = T' V and U = U~ - W S, Q Gamma S
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idv = idesc_fp16(128, 128, false, true);
            for (int ks = 0; ks < C / 16; ++ks)
                mma_bf16(D_U, sdesc_sw128(sbase + C_TZM + ks * 32, 16, 1024),
                         sdesc_sw128(sbase + C_B2 + 16384 + ks * 2048, 8192, 1024), idv, ks > 0);
            for (int ks = 0; ks < DK / 16; ++ks)
                mma_bf16(D_U, sdesc_sw128(sbase + C_G3A + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                         sdesc_sw128(sbase + C_SB + ks * 2048, 16384, 1024), idv, true);
            mma_commit(&sm.mma_bar);
            ok = mbar_wait(&sm.mma_bar, ph_mma, kWait);
        }
        ph_mma ^= 1u;
        if (lead_wait(ok)) break;
        tc_fence_after();

        // (b) U -> fp16 operand; S *= Gamma_C; release T', K_hat*Gamma, Q_hat*Gamma, V
        if (tid == 0) {
            mbar_arrive_remote(front_bar(&sm.single_free));
            if (m + 1 < nchunks) issue_v(m + 1);
        }
        if (warp == 8 || warp == 9) {
            const int t = (warp - 8) * 32 + lane;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                float r[4][16];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    tmem_ld16(tmem_addr(D_U, (warp & 3) * 32, 64 * hb + 16 * jj), r[jj]);
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) st_pack16<true>(sbase + C_UT + hb * 8192, t, 16 * jj, r[jj]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // (c) S += Kbar^T U ; O += M U ; then W of the next chunk
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id4 = idesc_fp16(128, 128, true, true);
            const uint32_t id5 = idesc_fp16(128, 128, false, true);
            for (int ks = 0; ks < C / 16; ++ks)
                mma_bf16(D_S, sdesc_sw128(sbase + C_KB + s * 16384 + ks * 2048, 8192, 1024),
                         sdesc_sw128(sbase + C_UT + ks * 2048, 8192, 1024), id4, true);
            for (int ks = 0; ks < C / 16; ++ks)
                mma_bf16(D_U, sdesc_sw128(sbase + C_TZM + 8192 + s * 16384 + ks * 32, 16, 1024),
                         sdesc_sw128(sbase + C_UT + ks * 2048, 8192, 1024), id5, true);
            mma_commit(&sm.mma_bar);
            if (m + 1 < nchunks) {
                ok = mbar_wait(&sm.full[s ^ 1], ((m + 1) >> 1) & 1, kWait);
                if (ok) {
                    tc_fence_after();
                    issue_g2w();
                }
            }
            ok = ok && mbar_wait(&sm.mma_bar, ph_mma, kWait);
            if (ok && m + 1 < nchunks)
                ok = mbar_wait(&sm.w_bar, (m + 1) & 1, kWait) &&
                     mbar_wait(&sm.v_full, (m + 1) & 1, kWait);
            if (ok) {
                if (m + 2 < nchunks) mbar_arrive_expect_tx(&sm.full[s], kChunkBytes);
                mbar_arrive_remote(front_bar(&sm.slot_free[s]));
            }
        }
        ph_mma ^= 1u;
        if (lead_wait(ok)) break;
        tc_fence_after();

        // (d) S -> fp16 operand, S *= Gamma_C of the next chunk; O -> out; next -W and V
        if (warp < 8) {
            const int c = quarter * 32 + lane;
            float r[4][16];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                tmem_ld16(tmem_addr(D_S, quarter * 32, 64 * half + 16 * jj), r[jj]);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) st_pack16<true>(sbase + C_SB + half * 16384, c, 16 * jj, r[jj]);
            if (m + 1 < nchunks) {
                const float g = sm.gamC_c[s ^ 1][c];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) r[jj][e] *= g;
                    tmem_st16(tmem_addr(D_S, quarter * 32, 64 * half + 16 * jj), r[jj]);
                }
                tmem_st_wait();
            }
        } else if (warp == 10 || warp == 11) {
            const int t = (warp - 10) * 32 + lane;
            const float sc = p.scale;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                float r[4][16];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    tmem_ld16(tmem_addr(D_U, (warp & 3) * 32, 64 * hb + 16 * jj), r[jj]);
                tmem_ld_wait();
                if (t < L) {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((row0 + t) * p.H + h) * DK +
                                                               64 * hb + 16 * jj);
                        const float *x = r[jj];
                        dst[0] = make_uint4(pack_bf16(sc * x[0], sc * x[1]), pack_bf16(sc * x[2], sc * x[3]),
                                            pack_bf16(sc * x[4], sc * x[5]), pack_bf16(sc * x[6], sc * x[7]));
                        dst[1] = make_uint4(pack_bf16(sc * x[8], sc * x[9]), pack_bf16(sc * x[10], sc * x[11]),
                                            pack_bf16(sc * x[12], sc * x[13]), pack_bf16(sc * x[14], sc * x[15]));
                    }
                }
            }
        }
        if (m + 1 < nchunks) {
            read_w();
            convert_v();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    }

    // final state from the fp32 master
    if (!sm.abort_c && p.fin && warp < 8) {
        tc_fence_after();
        const int c = quarter * 32 + lane;
        for (int jj = 0; jj < 4; ++jj) {
            float r[16];
            tmem_ld16(tmem_addr(D_S, quarter * 32, 64 * half + 16 * jj), r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const size_t off = state_base + (size_t)(64 * half + 16 * jj + e) * DK + c;
                if (p.state_type == kStateBF16)
                    reinterpret_cast<__nv_bfloat16 *>(p.fin)[off] = __float2bfloat16(r[e]);
                else
                    reinterpret_cast<float *>(p.fin)[off] = r[e];
            }
        }
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NT, 1)
kda_cluster_kernel(const __grid_constant__ TmaMaps maps, Params p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small &sm = *reinterpret_cast<Small *>(smem + SMALL);
    const uint32_t rank = cluster_ctarank();
    const int64_t unit = cluster_id_x();
    const int64_t h = unit % p.H;
    int64_t n = unit / p.H;
    // Varlen: clusters take sequences longest first, so the longest recurrences
    // start in the first wave.  Every CTA ranks the lengths itself (no host sync,
    // no workspace); batches with more than kOrderMax sequences keep their order.
    if (p.cu_seqlens && p.n_seqs > 1 && p.n_seqs <= kOrderMax) {
        int64_t *lens = reinterpret_cast<int64_t *>(smem);   // scratch before any TMA
        int *sel = reinterpret_cast<int *>(smem + 8 * kOrderMax);
        for (int i = threadIdx.x; i < p.n_seqs; i += NT) lens[i] = p.cu_seqlens[i + 1] - p.cu_seqlens[i];
        if (threadIdx.x == 0) *sel = (int)n;
        __syncthreads();
        for (int i = threadIdx.x; i < p.n_seqs; i += NT) {
            const int64_t li = lens[i];
            int64_t r = 0;
            for (int j = 0; j < p.n_seqs; ++j) {
                const int64_t lj = lens[j];
                r += (lj > li) || (lj == li && j < i);
            }
            if (r == n) *sel = i;
        }
        __syncthreads();
        n = *sel;
        __syncthreads();
    }
    int64_t b, t0, len;
    seq_range(p, n, b, t0, len);
    const int64_t row_base = b * p.T + t0;
    const int nchunks = (int)((len + C - 1) / C);

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.raw_full[i], 1);
            mbar_init(&sm.g1_done[i], 1);
            mbar_init(&sm.am_free[i], 1);
            mbar_init(&sm.s_done[i], 1);
            mbar_init(&sm.slot_free[i], 1);
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.pdone[i], 1);
        }
        mbar_init(&sm.single_free, 1);
        mbar_init(&sm.v_full, 1);
        mbar_init(&sm.mma_bar, 1);
        mbar_init(&sm.w_bar, 1);
        sm.abort_p = sm.abort_s = sm.abort_c = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync();   // both CTAs' barriers exist before any remote operation
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (rank == 0)
        run_front(maps, p, smem, sm, tmem, h, row_base, len, nchunks);
    else
        run_chain(maps, p, smem, sm, tmem, n, h, row_base, len, nchunks);

    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no CTA leaves while its peer may still signal it
    if (threadIdx.x < 32) tmem_dealloc(tmem, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

bool encode_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t H) {
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

}  // namespace

cudaError_t launch_cluster(const Params &p, cudaStream_t stream) {
    const int64_t units = p.n_seqs * p.H;
    if (units == 0) return cudaSuccess;
    TmaMaps maps;
    const int64_t rows = p.B * p.T > 0 ? p.B * p.T : 1;
    const void *dummy = p.q ? (const void *)p.q : (const void *)p.A_log;
    if (!encode_map(&maps.q, p.q ? p.q : dummy, rows, p.H) ||
        !encode_map(&maps.k, p.k ? p.k : dummy, rows, p.H) ||
        !encode_map(&maps.g, p.g ? p.g : dummy, rows, p.H) ||
        !encode_map(&maps.v, p.v ? p.v : dummy, rows, p.H))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kda_cluster_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kda_cluster_kernel<<<(unsigned)(2 * units), NT, SMEM_BYTES, stream>>>(maps, p);
    return cudaGetLastError();
}

}  // namespace kda
