// KDA forward on the sm_103a tensor cores: one CTA per (sequence, head, 64-wide
// slice of V), chunks of C = 64 tokens processed in order, tcgen05 MMAs with
// fp32 accumulators in tensor memory, TMA loads of q/k/g/v.
//
// Chunk algebra (the KDA token recurrence of the FlashKDA README "Kernel API"
// unrolled over a chunk; S is K x V, S0 the state entering the chunk, G the
// in-chunk cumulative log decay per channel, Gamma = exp(G)):
//   A[t,i] = beta_t sum_c k[t,c] k[i,c] exp(G[t,c]-G[i,c])  (i < t)
//   M[t,i] =        sum_c q[t,c] k[i,c] exp(G[t,c]-G[i,c])  (i <= t)
//   T      = (I + A)^-1,   T' = T Diag(beta)
//   W      = T' (K*Gamma),  U~ = T' V,  U = U~ - W S0
//   O      = scale ((Q*Gamma) S0 + M U)
//   S_C    = Diag(Gamma_C) S0 + (K*exp(G_C - G))^T U
//
// Exponent handling.  The gate bounds the per-token log decay to (lb, 0] with
// lb >= -5, so within a 16-token block |G_t - G_start| < 80 and exp of it fits
// in fp32/bf16.  Each token is scaled relative to its own 16-token block start
// (E1 = exp(H) <= 1, E2 = exp(-H) >= 1 with H = G - G_start); the A/M GEMM's B
// operand holds, for every row block bt, the keys rescaled to bt's start
// ("variants"), so every product the GEMM forms for a needed (t, i) pair is
// exp(G_t - G_i) <= 1 computed from bounded factors.
//
// GEMMs per chunk (all M = 128, fp32 accumulators).  G1 takes bf16 operands built
// from the raw (unnormalised) bf16 q and k, so its block-scaled factors keep bf16's
// exponent range and an undecayed key enters exactly; the 1/|q|, 1/|k| factors are
// applied to the 64x64 A and M after the GEMM.  G2..G5 take fp16 operands, whose
// values are bounded (T', normalised K*Gamma, V, -W, Q*Gamma, S, Kbar, U, M) and
// gain 3 mantissa bits over bf16, which keeps the fp32 final state within 1e-3
// relative of the exact one even without decay.  Values beyond fp16's range
// (|x| > 65504: e.g. an initial state of that size) are not supported.
//   G1  [Kp; Qp] (128x128, K-major)  x  Kn^T (160 variant rows)   -> A | M raw
//   G2  [T'; 0]  (128x64, K-major)   x  [K*Gamma | V] (MN-major)  -> W | U~
//   G3  [-W; Q*Gamma] (K-major)      x  S (MN-major, fp16 copy)   -> U | Q Gamma S
//   G4  Kbar (MN-major)              x  U (MN-major)              -> S (+= onto decayed S)
//   G5  [0; M] (K-major)             x  U (MN-major)              -> O (+= Q Gamma S)
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

using namespace sm103;

constexpr int C = kChunk;
constexpr int DK = kHeadDim;
constexpr int VS = 64;                 // V columns per CTA
constexpr int NSLICE = kHeadDim / VS;
constexpr int NT = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimit = 2000000000ull;  // 2 s per wait, then KDA_ERR_TIMEOUT

// Tensor-memory columns (512 allocated; lanes = rows of each MMA's D).
constexpr uint32_t COL_S = 0;      // S[c][v]           64 cols
constexpr uint32_t COL_W = 64;     // W[t][c]          128 cols (lanes 64..127 zero)
constexpr uint32_t COL_U = 192;    // U[t][v] / O[t][v] 64 cols (O in lanes 64..127)
constexpr uint32_t COL_AM = 256;   // A|M raw          160 cols
constexpr uint32_t TMEM_COLS = 512;

// Shared-memory map (byte offsets from a 1024-aligned base).
constexpr uint32_t SM_RQ = 0;                  // raw q: 2 x [64 t][64 c]
constexpr uint32_t SM_RK = SM_RQ + 16384;      // raw k
constexpr uint32_t SM_RG = SM_RK + 16384;      // raw g
constexpr uint32_t SM_B2 = SM_RG + 16384;      // K*Gamma: 2 x [64 i][64 c] (MN-major), then
constexpr uint32_t SM_RV = SM_B2 + 16384;      //   raw v [64 t][64 v]: B of G2 spans both
constexpr uint32_t SM_AMA = SM_RV + 8192;      // [Kp; Qp]: 2 x [128][64]
constexpr uint32_t SM_AMB = SM_AMA + 32768;    // Kn variants: 2 x [160][64]
constexpr uint32_t SM_G3A = SM_AMB + 40960;    // [-W; Q*Gamma]: 2 x [128][64]
constexpr uint32_t SM_SB = SM_G3A + 32768;     // S bf16 [128 c][64 v] (MN-major)
constexpr uint32_t SM_KB = SM_SB + 16384;      // Kbar: 2 x [64 i][64 c] (MN-major)
constexpr uint32_t SM_UT = SM_KB + 16384;      // U [64 i][64 v] (MN-major)
constexpr uint32_t SM_SMALL = SM_UT + 8192;
// Reused after G1 has consumed [Kp; Qp] and Kn (region SM_AMA .. +72 KB):
constexpr uint32_t SM_TZM = SM_AMA;            // T' [64][64], 0 [64][64], M [64][64]
constexpr uint32_t SM_AMAT = SM_AMA + 24576;   // fp32 [64][65]
constexpr uint32_t SM_TF = SM_AMAT + 16640;    // fp32 [64][65]
constexpr uint32_t SM_ZS = SM_TF + 16640;      // fp32 [3][16][16] inverse scratch
constexpr int LDA = 65;

struct Small {
    float rq[C], rk[C], beta[C];
    float btot[4][DK];     // per 16-token block: sum of log2 decays
    float gamC[DK];        // exp(G_C)
    uint64_t bar_qkg, bar_v, bar_mma;
    uint32_t tmem_base;
    int fail;
};
constexpr uint32_t SMEM_BYTES = SM_SMALL + sizeof(Small) + 1024;

// Row offset of B-operand variant bt inside the Kn tile.
__device__ __forceinline__ int variant_off(int bt) { return 8 * bt * (bt + 1); }

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool fp16) {
    return fp16 ? pack_f16(lo, hi) : pack_bf16(lo, hi);
}

// 16 consecutive 16-bit values of one row of a 128B-swizzled tile (two 16-byte
// chunks), as bf16 or fp16.
template <bool FP16 = false>
__device__ __forceinline__ void st_pack16(uint32_t base, int row, int col0, const float (&v)[16]) {
    sts128(base + sw128_off(row, col0), pack2(v[0], v[1], FP16), pack2(v[2], v[3], FP16),
           pack2(v[4], v[5], FP16), pack2(v[6], v[7], FP16));
    sts128(base + sw128_off(row, col0 + 8), pack2(v[8], v[9], FP16), pack2(v[10], v[11], FP16),
           pack2(v[12], v[13], FP16), pack2(v[14], v[15], FP16));
}

struct TmaMaps {
    CUtensorMap q, k, g, v;
};

__global__ void __launch_bounds__(NT, 1)
kda_tc_kernel(const __grid_constant__ TmaMaps maps, Params p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    Small &sm = *reinterpret_cast<Small *>(smem + SM_SMALL);
    float *Amat = reinterpret_cast<float *>(smem + SM_AMAT);
    float *Tf = reinterpret_cast<float *>(smem + SM_TF);
    float *Zs = reinterpret_cast<float *>(smem + SM_ZS);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int64_t unit = blockIdx.x;
    const int slice = (int)(unit % NSLICE);
    unit /= NSLICE;
    const int64_t h = unit % p.H;
    const int64_t n = unit / p.H;
    int64_t b, t0, len;
    seq_range(p, n, b, t0, len);
    const int v0 = slice * VS;
    const int64_t row_base = b * p.T + t0;   // flattened [B*T] row of the sequence's first token
    const size_t state_base = (size_t)(n * p.H + h) * DK * DK;
    const int nchunks = (int)((len + C - 1) / C);

    if (tid == 0) {
        mbar_init(&sm.bar_qkg, 1);
        mbar_init(&sm.bar_v, 1);
        mbar_init(&sm.bar_mma, 1);
        fence_mbar_init();
        sm.fail = 0;
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    auto issue_qkg = [&](int chunk) {
        const int row = (int)(row_base + (int64_t)chunk * C);
        mbar_arrive_expect_tx(&sm.bar_qkg, 3 * 16384);
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_3d(smem + SM_RQ + kb * 8192, &maps.q, &sm.bar_qkg, kb * 64, (int)h, row);
            tma_load_3d(smem + SM_RK + kb * 8192, &maps.k, &sm.bar_qkg, kb * 64, (int)h, row);
            tma_load_3d(smem + SM_RG + kb * 8192, &maps.g, &sm.bar_qkg, kb * 64, (int)h, row);
        }
    };
    auto issue_v = [&](int chunk) {
        const int row = (int)(row_base + (int64_t)chunk * C);
        mbar_arrive_expect_tx(&sm.bar_v, 8192);
        tma_load_3d(smem + SM_RV, &maps.v, &sm.bar_v, v0, (int)h, row);
    };
    if (tid == 0 && nchunks > 0) {
        issue_qkg(0);
        issue_v(0);
    }

    // Initial state -> TMEM (fp32 master) and the bf16 operand copy.
    if (warp >= 4) {
        const int c = (warp - 4) * 32 + lane;
        for (int jj = 0; jj < VS / 16; ++jj) {
            float r[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                float x = 0.f;
                if (p.init) {
                    const size_t off = state_base + (size_t)(v0 + 16 * jj + e) * DK + c;
                    x = p.state_type == kStateBF16
                            ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.init)[off])
                            : reinterpret_cast<const float *>(p.init)[off];
                }
                r[e] = x;
            }
            tmem_st16(tmem_addr(tmem, (warp - 4) * 32, COL_S + 16 * jj), r);
            st_pack16<true>(sbase + SM_SB, c, 16 * jj, r);
        }
        tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const float a2 = -__expf(p.A_log[h]) * kLog2e;   // exp(-a x) = exp2(a2 x)
    const float lb2 = p.lower_bound * kLog2e;         // log2-domain lower bound
    uint32_t ph_qkg = 0, ph_v = 0, ph_mma = 0;
    bool failed = false;

    auto wait_all = [&](uint64_t *bar, uint32_t &ph) -> bool {
        const bool ok = mbar_wait(bar, ph, kWaitLimit);
        ph ^= 1u;
        if (!ok && p.err) atomicExch(p.err, (int)8);
        return __syncthreads_or(!ok) != 0;
    };

    for (int ch = 0; ch < nchunks && !failed; ++ch) {
        const int64_t cs = (int64_t)ch * C;
        const int L = (int)((len - cs) < C ? (len - cs) : C);
        const int64_t row0 = row_base + cs;

        // ---- P1: wait q/k/g, row norms, beta
        if (wait_all(&sm.bar_qkg, ph_qkg)) { failed = true; break; }
        for (int t = warp; t < C; t += NT / 32) {
            const int kb = lane >> 4, col = (lane * 4) & 63;
            const uint32_t off = kb * 8192 + sw128_off(t, col);
            const uint2 qv = *reinterpret_cast<const uint2 *>(smem + SM_RQ + off);
            const uint2 kv = *reinterpret_cast<const uint2 *>(smem + SM_RK + off);
            float sq = bf16lo(qv.x) * bf16lo(qv.x) + bf16hi(qv.x) * bf16hi(qv.x) +
                       bf16lo(qv.y) * bf16lo(qv.y) + bf16hi(qv.y) * bf16hi(qv.y);
            float sk = bf16lo(kv.x) * bf16lo(kv.x) + bf16hi(kv.x) * bf16hi(kv.x) +
                       bf16lo(kv.y) * bf16lo(kv.y) + bf16hi(kv.y) * bf16hi(kv.y);
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
        if (warp == 0) {
            for (int t = lane; t < C; t += 32) {
                float bt = 0.f;
                if (t < L) {
                    const float bl = __bfloat162float(p.beta[(row0 + t) * p.H + h]);
                    bt = 1.f / (1.f + exp2f(-bl * kLog2e));
                }
                sm.beta[t] = bt;
            }
        }
        __syncthreads();

        // ---- P2: gate, block-local cumulative decay, GEMM operands
        const int blk = warp >> 1;               // 16-token block of this thread
        const int c = (warp & 1) * 64 + 2 * lane; // channel pair (c, c+1)
        const int kb = c >> 6, cc = c & 63;
        float H0[16], H1[16];
        {
            const float b0 = a2 * p.dt_bias[h * DK + c], b1 = a2 * p.dt_bias[h * DK + c + 1];
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int t = blk * 16 + r;
                const uint32_t gv =
                    *reinterpret_cast<const uint32_t *>(smem + SM_RG + kb * 8192 + sw128_off(t, cc));
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
        __syncthreads();
        {
            float Gs0[4], Gs1[4];
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                Gs0[bb] = s0;
                Gs1[bb] = s1;
                s0 += sm.btot[bb][c];
                s1 += sm.btot[bb][c + 1];
            }
            // s0, s1 = G_C (log2 units)
            if (blk == 0) {
                sm.gamC[c] = exp2f(s0);
                sm.gamC[c + 1] = exp2f(s1);
            }
            const float Fs0 = exp2f(Gs0[blk]), Fs1 = exp2f(Gs1[blk]);
            const float FC0 = exp2f(s0 - Gs0[blk]), FC1 = exp2f(s1 - Gs1[blk]);
            float D0[4], D1[4];
#pragma unroll
            for (int bt = 0; bt < 4; ++bt) {
                D0[bt] = bt > blk ? exp2f(Gs0[bt] - Gs0[blk]) : 1.f;
                D1[bt] = bt > blk ? exp2f(Gs1[bt] - Gs1[blk]) : 1.f;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int t = blk * 16 + r;
                const uint32_t off = kb * 8192 + sw128_off(t, cc);
                const uint32_t qv = *reinterpret_cast<const uint32_t *>(smem + SM_RQ + off);
                const uint32_t kv = *reinterpret_cast<const uint32_t *>(smem + SM_RK + off);
                const float rq = sm.rq[t], rk = sm.rk[t];
                // raw inputs (rows t >= L are masked by rq = rk = 0 and beta = 0)
                const float q0 = t < L ? bf16lo(qv) : 0.f, q1 = t < L ? bf16hi(qv) : 0.f;
                const float k0 = t < L ? bf16lo(kv) : 0.f, k1 = t < L ? bf16hi(kv) : 0.f;
                const float e10 = exp2f(H0[r]), e11 = exp2f(H1[r]);
                const float e20 = exp2f(-H0[r]), e21 = exp2f(-H1[r]);
                const float kp0 = k0 * e10, kp1 = k1 * e11;
                const float qp0 = q0 * e10, qp1 = q1 * e11;
                const float kn0 = k0 * e20, kn1 = k1 * e21;
                // G1 A operand: rows t (keys) and 64 + t (queries)
                *reinterpret_cast<uint32_t *>(smem + SM_AMA + kb * 16384 + sw128_off(t, cc)) =
                    pack_bf16(kp0, kp1);
                *reinterpret_cast<uint32_t *>(smem + SM_AMA + kb * 16384 + sw128_off(64 + t, cc)) =
                    pack_bf16(qp0, qp1);
                // G1 B operand: token t in every variant bt >= blk
#pragma unroll
                for (int bt = 0; bt < 4; ++bt) {
                    if (bt >= blk) {
                        const int row = variant_off(bt) + t;
                        *reinterpret_cast<uint32_t *>(smem + SM_AMB + kb * 20480 +
                                                      sw128_off(row, cc)) =
                            pack_bf16(kn0 * D0[bt], kn1 * D1[bt]);
                    }
                }
                // G2 B operand: normalised K*Gamma (MN-major [i][c])
                *reinterpret_cast<uint32_t *>(smem + SM_B2 + off) =
                    pack_f16(kp0 * (Fs0 * rk), kp1 * (Fs1 * rk));
                // G3 A operand rows 64..127: normalised Q*Gamma
                *reinterpret_cast<uint32_t *>(smem + SM_G3A + kb * 16384 + sw128_off(64 + t, cc)) =
                    pack_f16(qp0 * (Fs0 * rq), qp1 * (Fs1 * rq));
                // G4 A operand: normalised Kbar = k_hat exp(G_C - G) (MN-major [i][c])
                *reinterpret_cast<uint32_t *>(smem + SM_KB + off) =
                    pack_f16(kn0 * (FC0 * rk), kn1 * (FC1 * rk));
            }
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- G1
        if (tid == 0) {
            tc_fence_after();
            if (ch + 1 < nchunks) issue_qkg(ch + 1);   // raw q/k/g consumed
            const uint32_t id = idesc_bf16(128, 160, false, false);
            for (int ks = 0; ks < DK / 16; ++ks) {
                const uint64_t ad = sdesc_sw128(sbase + SM_AMA + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(sbase + SM_AMB + (ks >> 2) * 20480 + (ks & 3) * 32, 16, 1024);
                mma_bf16(tmem + COL_AM, ad, bd, id, ks > 0);
            }
            mma_commit(&sm.bar_mma);
        }
        if (wait_all(&sm.bar_mma, ph_mma)) { failed = true; break; }
        tc_fence_after();

        // ---- P4: A (fp32, beta-scaled, strictly lower) and M (bf16, lower incl. diagonal)
        if (warp < 4) {
            const bool is_m = warp >= 2;
            const int t = (warp & 1) * 32 + lane;
            const int bt = t >> 4;
            const int jlo = (warp & 1) ? 3 : 0, jhi = (warp & 1) ? 10 : 3;
            const float rowf = is_m ? sm.rq[t] : sm.beta[t] * sm.rk[t];
            // zero the part above the diagonal block
            for (int i = 16 * (bt + 1); i < 64; i += 16) {
                if (is_m) {
                    sts128(sbase + SM_TZM + 16384 + sw128_off(t, i), 0, 0, 0, 0);
                    sts128(sbase + SM_TZM + 16384 + sw128_off(t, i + 8), 0, 0, 0, 0);
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) Amat[t * LDA + i + e] = 0.f;
                }
            }
            for (int jj = jlo; jj < jhi; ++jj) {
                float r[16];
                tmem_ld16(tmem_addr(tmem, warp * 32, COL_AM + 16 * jj), r);
                tmem_ld_wait();
                const int vo = variant_off(bt);
                if (16 * jj >= vo && 16 * jj < vo + 16 * (bt + 1)) {
                    const int ib = 16 * jj - vo;
                    // column factor 1/|k_i|; row factor 1/|q_t| (M) or beta_t/|k_t| (A)
                    if (is_m) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            r[e] = (ib + e <= t) ? rowf * sm.rk[ib + e] * r[e] : 0.f;
                        st_pack16<true>(sbase + SM_TZM + 16384, t, ib, r);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            Amat[t * LDA + ib + e] = (ib + e < t) ? rowf * sm.rk[ib + e] * r[e] : 0.f;
                    }
                }
            }
        } else {
            // zero tile between T' and M (A operand rows 64..127 of G2, rows 0..63 of G5)
            const int i = tid - 128;
            for (int k = i; k < 512; k += 128)
                sts128(sbase + SM_TZM + 8192 + k * 16, 0, 0, 0, 0);
        }
        __syncthreads();

        // ---- P5: T = (I + A)^-1, blocked: 16x16 diagonal blocks, then off-diagonal levels
        if (tid < 64) {
            const int bb = tid >> 4, j = tid & 15;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) acc = fmaf(Amat[(16 * bb + r) * LDA + 16 * bb + m], x[m], acc);
                if (r > j) x[r] = -acc;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Tf[(16 * bb + r) * LDA + 16 * bb + j] = x[r];
        }
        __syncthreads();
        for (int d = 1; d < 4; ++d) {
            const int cnt = (4 - d) * 256;
            for (int e = tid; e < cnt; e += NT) {
                const int ba = e >> 8, r = (e >> 4) & 15, j = e & 15, bt = ba + d;
                float acc = 0.f;
                for (int m = 16 * ba; m < 16 * bt; ++m)
                    acc = fmaf(Amat[(16 * bt + r) * LDA + m], Tf[m * LDA + 16 * ba + j], acc);
                Zs[e] = acc;
            }
            __syncthreads();
            for (int e = tid; e < cnt; e += NT) {
                const int ba = e >> 8, r = (e >> 4) & 15, j = e & 15, bt = ba + d;
                float acc = 0.f;
                for (int s = 0; s <= r; ++s)
                    acc = fmaf(Tf[(16 * bt + r) * LDA + 16 * bt + s], Zs[(ba << 8) + s * 16 + j], acc);
                Tf[(16 * bt + r) * LDA + 16 * ba + j] = -acc;
            }
            __syncthreads();
        }
        {
            const int t = tid >> 2, i0 = (tid & 3) * 16;
            float r[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int i = i0 + e;
                r[e] = (i <= t) ? Tf[t * LDA + i] * sm.beta[i] : 0.f;
            }
            st_pack16<true>(sbase + SM_TZM, t, i0, r);
        }
        // V (bf16 from TMA) -> fp16 in place, the B operand type of G2
        if (!mbar_wait(&sm.bar_v, ph_v, kWaitLimit)) {
            if (p.err) atomicExch(p.err, 8);
            sm.fail = 1;
        }
        ph_v ^= 1u;
        for (int k16 = tid; k16 < 512; k16 += NT) {
            uint4 *ptr = reinterpret_cast<uint4 *>(smem + SM_RV + k16 * 16);
            uint4 x = *ptr;
            x.x = pack_f16(bf16lo(x.x), bf16hi(x.x));
            x.y = pack_f16(bf16lo(x.y), bf16hi(x.y));
            x.z = pack_f16(bf16lo(x.z), bf16hi(x.z));
            x.w = pack_f16(bf16lo(x.w), bf16hi(x.w));
            *ptr = x;
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- G2: [W | U~] = [T'; 0] x [K*Gamma | V]
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_fp16(128, 192, false, true);
            for (int ks = 0; ks < C / 16; ++ks) {
                const uint64_t ad = sdesc_sw128(sbase + SM_TZM + ks * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(sbase + SM_B2 + ks * 2048, 8192, 1024);
                mma_bf16(tmem + COL_W, ad, bd, id, ks > 0);
            }
            mma_commit(&sm.bar_mma);
        }
        if (wait_all(&sm.bar_mma, ph_mma) || sm.fail) { failed = true; break; }
        tc_fence_after();
        if (tid == 0 && ch + 1 < nchunks) issue_v(ch + 1);   // raw v consumed by G2

        // ---- P7: -W -> rows 0..63 of the G3 A operand
        if (warp == 0 || warp == 1 || warp == 4 || warp == 5) {
            const int t = (warp & 1) * 32 + lane;
            const int jbase = warp >= 4 ? 4 : 0;
            for (int jj = jbase; jj < jbase + 4; ++jj) {
                float r[16];
                tmem_ld16(tmem_addr(tmem, (warp & 3) * 32, COL_W + 16 * jj), r);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) r[e] = -r[e];
                st_pack16<true>(sbase + SM_G3A + (jj >> 2) * 16384, t, (16 * jj) & 63, r);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- G3: U = U~ - W S0 (lanes 0..63), Q Gamma S0 (lanes 64..127)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_fp16(128, 64, false, true);
            for (int ks = 0; ks < DK / 16; ++ks) {
                const uint64_t ad = sdesc_sw128(sbase + SM_G3A + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(sbase + SM_SB + ks * 2048, 16384, 1024);
                mma_bf16(tmem + COL_U, ad, bd, id, true);
            }
            mma_commit(&sm.bar_mma);
        }
        if (wait_all(&sm.bar_mma, ph_mma)) { failed = true; break; }
        tc_fence_after();

        // ---- P9: U -> bf16 (MN-major [i][v]); decay the fp32 state by Gamma_C
        if (warp < 2) {
            const int t = warp * 32 + lane;
            for (int jj = 0; jj < VS / 16; ++jj) {
                float r[16];
                tmem_ld16(tmem_addr(tmem, warp * 32, COL_U + 16 * jj), r);
                tmem_ld_wait();
                st_pack16<true>(sbase + SM_UT, t, 16 * jj, r);
            }
        } else if (warp >= 4) {
            const int cch = (warp - 4) * 32 + lane;
            const float gmc = sm.gamC[cch];
            for (int jj = 0; jj < VS / 16; ++jj) {
                float r[16];
                tmem_ld16(tmem_addr(tmem, (warp - 4) * 32, COL_S + 16 * jj), r);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) r[e] *= gmc;
                tmem_st16(tmem_addr(tmem, (warp - 4) * 32, COL_S + 16 * jj), r);
            }
            tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- G4: S += Kbar^T U ;  G5: O += M U
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id4 = idesc_fp16(128, 64, true, true);
            const uint32_t id5 = idesc_fp16(128, 64, false, true);
            for (int ks = 0; ks < C / 16; ++ks) {
                const uint64_t ad = sdesc_sw128(sbase + SM_KB + ks * 2048, 8192, 1024);
                const uint64_t bd = sdesc_sw128(sbase + SM_UT + ks * 2048, 8192, 1024);
                mma_bf16(tmem + COL_S, ad, bd, id4, true);
            }
            for (int ks = 0; ks < C / 16; ++ks) {
                const uint64_t ad = sdesc_sw128(sbase + SM_TZM + 8192 + ks * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(sbase + SM_UT + ks * 2048, 8192, 1024);
                mma_bf16(tmem + COL_U, ad, bd, id5, true);
            }
            mma_commit(&sm.bar_mma);
        }
        if (wait_all(&sm.bar_mma, ph_mma)) { failed = true; break; }
        tc_fence_after();

        // ---- P11: O -> out (rows t < L); S -> bf16 operand copy
        if (warp == 2 || warp == 3) {
            const int t = (warp - 2) * 32 + lane;
            for (int jj = 0; jj < VS / 16; ++jj) {
                float r[16];
                tmem_ld16(tmem_addr(tmem, warp * 32, COL_U + 16 * jj), r);
                tmem_ld_wait();
                if (t < L) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((row0 + t) * p.H + h) * DK + v0 + 16 * jj);
                    const float s = p.scale;
                    dst[0] = make_uint4(pack_bf16(s * r[0], s * r[1]), pack_bf16(s * r[2], s * r[3]),
                                        pack_bf16(s * r[4], s * r[5]), pack_bf16(s * r[6], s * r[7]));
                    dst[1] = make_uint4(pack_bf16(s * r[8], s * r[9]), pack_bf16(s * r[10], s * r[11]),
                                        pack_bf16(s * r[12], s * r[13]), pack_bf16(s * r[14], s * r[15]));
                }
            }
        } else if (warp >= 4) {
            const int cch = (warp - 4) * 32 + lane;
            for (int jj = 0; jj < VS / 16; ++jj) {
                float r[16];
                tmem_ld16(tmem_addr(tmem, (warp - 4) * 32, COL_S + 16 * jj), r);
                tmem_ld_wait();
                st_pack16<true>(sbase + SM_SB, cch, 16 * jj, r);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    // Final state from the fp32 master.
    if (!failed && p.fin && warp >= 4) {
        const int cch = (warp - 4) * 32 + lane;
        for (int jj = 0; jj < VS / 16; ++jj) {
            float r[16];
            tmem_ld16(tmem_addr(tmem, (warp - 4) * 32, COL_S + 16 * jj), r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const size_t off = state_base + (size_t)(v0 + 16 * jj + e) * DK + cch;
                if (p.state_type == kStateBF16)
                    reinterpret_cast<__nv_bfloat16 *>(p.fin)[off] = __float2bfloat16(r[e]);
                else
                    reinterpret_cast<float *>(p.fin)[off] = r[e];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// cuTensorMapEncodeTiled, resolved through the runtime so that the library has no
// link-time dependency on the driver library (it loads on hosts without a GPU).
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

cudaError_t launch_tc(const Params &p, cudaStream_t stream) {
    const int64_t units = p.n_seqs * p.H * NSLICE;
    if (units == 0) return cudaSuccess;
    TmaMaps maps;
    const int64_t rows = p.B * p.T > 0 ? p.B * p.T : 1;
    const void *dummy = p.q ? (const void *)p.q : (const void *)p.A_log;
    if (!encode_map(&maps.q, p.q ? p.q : dummy, rows, p.H) ||
        !encode_map(&maps.k, p.k ? p.k : dummy, rows, p.H) ||
        !encode_map(&maps.g, p.g ? p.g : dummy, rows, p.H) ||
        !encode_map(&maps.v, p.v ? p.v : dummy, rows, p.H))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kda_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kda_tc_kernel<<<(unsigned)units, NT, SMEM_BYTES, stream>>>(maps, p);
    return cudaGetLastError();
}

}  // namespace kda
