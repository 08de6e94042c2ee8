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
//     warps 0-7  prologue of chunk m: gate, block-local decay, the operands
//                of G1 = [Kp; Qp] x Kn^T and the chain's K_hat*Gamma,
//                Q_hat*Gamma, Kbar;
//     warps 13-15 beside the gate: row norms of q and k, beta;
//     warps 8-11 solver of chunk m-1: A and M out of TMEM, the blocked
//                inverse, T' (fp16);
//     warp 12    control: issues G1 into a double-buffered TMEM slot, writes the
//                prologue's chain tiles (Kbar, Q_hat*Gamma, K_hat*Gamma,
//                exp(G_C)) to a workspace slot in global memory (L2) with bulk
//                stores and signals the chain, and reloads the raw tile slot two
//                chunks ahead once the stores have read it;
//     the solver ships T' and M into a double-buffered slot of the chain CTA's
//     shared memory with bulk shared->shared copies that complete as
//     transaction bytes on the chain's per-slot mbarrier.
//   CTA rank 1 ("chain") owns the whole state (V = 128) in tensor memory:
//     G2u = [T'; 0] x V and G3 = [-W; Q_hat*Gamma] x S  -> U | Q Gamma S
//     U readout, S decay; bulk loads of the next chunk's workspace tiles
//     G4 = Kbar^T U -> S,  G5 = [0; M] x U -> O
//     O and S readout; W for the next chunk (G2w = [T'; 0] x K_hat*Gamma) is
//     computed and read out beside this, off the sequential path (16 warps:
//     S by warps 0-7, -W by 8/9/12/13, O by 10/11/14/15, one column half each).
// Flow control: the chain arrives remotely on the front's "slot free" (T' and M
// of a slot) and "workspace free" barriers, the front on the chain's
// "workspace ready" barrier; each side waits before writing into the other's
// buffers.
//
// Precision and exponent handling: G1 on bf16
// operands of the raw q/k scaled by 16-token-block-local decay factors, the
// other GEMMs on fp16 operands, fp32 accumulators, fp32 state.  Every wait is
// bounded (2 s); a timeout sets the device error word and both CTAs unwind.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_chunk.cuh"

namespace kda {
namespace {

using namespace sm103;
using namespace chunk;

constexpr int NT = 512;            // 16 warps in both CTAs
constexpr int NP = 256;            // front prologue group: warps 0-7
constexpr int NS = 128;            // front solver group: warps 8-11
constexpr int NH = 96;             // front helper group (norms, beta): warps 13-15
constexpr int kHelp0 = 416;        // first helper thread
// Threads that wait on mbarriers for their group (and publish through a named
// barrier): warp 1 for the prologue, warp 10 for the solver, so that the waiting
// threads of the front sit on different schedulers (warp 12, the control warp,
// shares its scheduler with neither).
constexpr int kProLead = 32;       // thread index
constexpr int kSolLead = 64;       // index within the solver group
constexpr uint32_t kChunkBytes = 16384 * 3 + 512 + 8192 * 2;   // front -> chain per chunk
constexpr uint32_t WS_KB = 0, WS_QG = 16384, WS_KG = 32768, WS_GC = 49152;   // workspace slot layout
constexpr int kOrderMax = 256;     // varlen batches up to this many sequences run longest first

// ---- front shared memory
constexpr uint32_t F_RAW = 0;          // 2 slots x {q, k, g}: 16 KB each, 2 x [64 t][64 c]
constexpr uint32_t F_SLOT = 49152;
constexpr uint32_t F_AMA = 98304;      // [Kp; Qp]: 2 x [128][64] bf16
constexpr uint32_t F_AMB = 131072;     // Kn variants: 2 x [160][64] bf16
constexpr uint32_t F_MST = 172032;     // M staging fp16 [64 t][64 i]
constexpr uint32_t F_AMAT = 180224;    // A fp32 [64][68]; T' staging (fp16) after the inverse
constexpr uint32_t F_TF = 197632;      // T fp32 [64][68]
// ---- chain shared memory
constexpr uint32_t C_B2 = 0;           // K_hat*Gamma 2 x [64 i][64 c] | V 2 x [64 t][64 v] (MN-major)
constexpr uint32_t C_G3A = 32768;      // [-W; Q_hat*Gamma]: 2 x [128][64] (K-major)
constexpr uint32_t C_KB = 65536;       // 2 slots x Kbar 2 x [64 i][64 c] (MN-major)
constexpr uint32_t C_TZM = 98304;      // T'0 | Z | M0 | Z | M1, each [64][64] (K-major)
constexpr uint32_t C_SB = 139264;      // S fp16 2 x [128 c][64 v] (MN-major)
constexpr uint32_t C_UT = 172032;      // U fp16 2 x [64 i][64 v] (MN-major)
constexpr uint32_t C_T1 = 188416;      // T'1 | Z, each [64][64] (K-major)
constexpr uint32_t SMALL = 218112;     // common offset in both CTAs (remote addresses)

struct Small {
    float rq[2][C], rk[2][C], beta[2][C];   // front, per slot
    float btot[4][DK];                       // front
    float fac[kFacRows][DK];                 // front: decay factors, see fac_base
    float gamC_f[2][DK];                     // front: exp(G_C) per slot (copy source)
    float gamC_c[2][DK];                     // chain: copy destination
    uint64_t raw_full[2], g1_done[2], am_free[2], s_done[2], slot_free[2], pdone[2];
    uint64_t full[2], v_full, mma_bar, w_bar;
    uint64_t gready[2], gfree[2];   // workspace slot written (chain side) / loaded (front side)
    uint32_t tmem_base;
    int abort_p, abort_s, abort_c;
    int dec_p, dec_s;   // a group's abort decision, written by its lead thread only, before a barrier
};
constexpr uint32_t SMEM_BYTES = SMALL + sizeof(Small) + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// ============================================================== front CTA
__device__ __forceinline__ void run_front(const TmaMaps &maps, const Params &p, unsigned char *smem,
                                          Small &sm, uint32_t tmem, int64_t unit, int64_t h,
                                          int64_t row_base, int64_t len, int nchunks) {
    unsigned char *wsu = p.ws + unit * kWsBytesPerUnit;   // this cluster's workspace
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
        // Thread layout for the gate and the operands: warp = (16-token block, 64-channel
        // half), lane = (4-token quarter of the block, 8-channel group); every access to
        // the tiles is one 16-byte vector (8 channels of one token).
        const float a2 = -__expf(p.A_log[h]) * kLog2e;
        const float lb2 = p.lower_bound * kLog2e;
        const int blk = warp >> 1, kh = warp & 1;
        const int cg = lane & 7, qr = lane >> 3;
        const int c0 = 64 * kh + 8 * cg;             // first of this thread's 8 channels
        const uint32_t kho = kh * 8192;              // the half inside a raw tile
        float2 bias[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            bias[i] = make_float2(a2 * p.dt_bias[h * DK + c0 + 2 * i], a2 * p.dt_bias[h * DK + c0 + 2 * i + 1]);
        for (int m = 0; m < nchunks; ++m) {
            const int s = m & 1;
            const int64_t cs = (int64_t)m * C;
            const int L = (int)((len - cs) < C ? (len - cs) : C);
            const uint32_t rq_off = F_RAW + s * F_SLOT, rk_off = rq_off + 16384, rg_off = rq_off + 32768;
            if (tid == kProLead) {
                bool ok = mbar_wait(&sm.raw_full[s], (m >> 1) & 1, kWait);
                if (ok && m >= 2) ok = mbar_wait(&sm.s_done[s], ((m - 2) >> 1) & 1, kWait);
                if (!ok) { set_err(p); sm.abort_p = 1; }
                sm.dec_p = sm.abort_p;
            }
            named_bar(1, NP + NH);   // with the helpers: raw tiles of chunk m are in
            if (sm.dec_p) break;

            // gate (log2 units) and its block-local inclusive cumulative sum H (channel pairs)
            float2 H[4][4];
            {
                const float2 a2v = make_float2(a2, a2), lb2v = make_float2(lb2, lb2);
                const float2 one = make_float2(1.f, 1.f);
                float2 acc[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = 16 * blk + 4 * qr + j;
                    const uint4 gv = *reinterpret_cast<const uint4 *>(smem + rg_off + kho + sw128_off(t, 8 * cg));
                    if (t < L) {
                        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float2 z = fma2(bf16x2_to_f2(gw[i]), a2v, bias[i]);
                            const float2 d = add2(make_float2(exp2f(z.x), exp2f(z.y)), one);
                            acc[i] = fma2(lb2v, make_float2(__fdividef(1.f, d.x), __fdividef(1.f, d.y)), acc[i]);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) H[j][i] = acc[i];
                }
                // add the totals of the earlier quarters (lanes 8 and 16 apart share channels)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float2 v = acc[i];
                    float2 u = make_float2(__shfl_up_sync(0xffffffffu, v.x, 8), __shfl_up_sync(0xffffffffu, v.y, 8));
                    if (qr >= 1) v = add2(v, u);
                    u = make_float2(__shfl_up_sync(0xffffffffu, v.x, 16), __shfl_up_sync(0xffffffffu, v.y, 16));
                    if (qr >= 2) v = add2(v, u);
                    float2 ex = make_float2(__shfl_up_sync(0xffffffffu, v.x, 8), __shfl_up_sync(0xffffffffu, v.y, 8));
                    if (qr == 0) ex = make_float2(0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < 4; ++j) H[j][i] = add2(H[j][i], ex);
                    acc[i] = v;
                }
                if (qr == 3) {
                    float4 *bt4 = reinterpret_cast<float4 *>(&sm.btot[blk][c0]);
                    bt4[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
                    bt4[1] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
                }
            }
            named_bar(1, NP + NH);   // gate totals, and the helpers' norms and beta

            // decay factors per (block, channel): thread = channel, two blocks each
            {
                const int c = tid & (DK - 1), bh = tid >> 7;
                float Gs[4], tot = 0.f;
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
                    Gs[bb] = tot;
                    tot += sm.btot[bb][c];
                }
                if (bh == 0) sm.gamC_f[s][c] = exp2f(tot);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    if ((b >> 1) != bh) continue;
                    float *f = &sm.fac[fac_base(b)][c];
                    f[0] = exp2f(Gs[b]);
                    f[DK] = exp2f(tot - Gs[b]);
#pragma unroll
                    for (int bt = b + 1; bt < 4; ++bt) f[(1 + bt - b) * DK] = exp2f(Gs[bt] - Gs[b]);
                }
            }
            // [Kp; Qp] and Kn are free once G1 of the previous chunk completed
            if (tid == kProLead) {
                if (m >= 1 && !mbar_wait(&sm.g1_done[(m - 1) & 1], ((m - 1) >> 1) & 1, kWait)) {
                    set_err(p);
                    sm.abort_p = 1;
                }
                sm.dec_p = sm.abort_p;
            }
            named_bar(3, NP);
            if (sm.dec_p) {
                named_bar(1, NP + NH);   // the helpers read the decision at their next barrier
                break;
            }

            // Operands.  G1 (bf16, raw q/k times block-local decay): Kp = k 2^H and
            // Qp = q 2^H at rows 32 blk + r and 32 blk + 16 + r of [Kp; Qp]; key
            // variants Kn(bt) = k 2^(Gs[bt] - Gs[blk] - H) at row variant_off(bt) + t for
            // bt >= blk.  Chain (fp16, in place of the raw tiles): Q_hat*Gamma,
            // K_hat*Gamma and Kbar = k_hat 2^(G_C - G).
            {
                const int fb = fac_base(blk);
                const float4 *fs4 = reinterpret_cast<const float4 *>(&sm.fac[fb][c0]);
                const float4 *fc4 = reinterpret_cast<const float4 *>(&sm.fac[fb + 1][c0]);
                const float4 fsa = fs4[0], fsb = fs4[1], fca = fc4[0], fcb = fc4[1];
                const float2 Fs[4] = {make_float2(fsa.x, fsa.y), make_float2(fsa.z, fsa.w), make_float2(fsb.x, fsb.y),
                                      make_float2(fsb.z, fsb.w)};
                const float2 FC[4] = {make_float2(fca.x, fca.y), make_float2(fca.z, fca.w), make_float2(fcb.x, fcb.y),
                                      make_float2(fcb.z, fcb.w)};
                const uint32_t ama = sbase + F_AMA + kh * 16384, amb = sbase + F_AMB + kh * 20480;
#pragma unroll 2
                for (int j = 0; j < 4; ++j) {
                    const int r = 4 * qr + j, t = 16 * blk + r;
                    const uint32_t off = kho + sw128_off(t, 8 * cg);
                    uint4 qv = *reinterpret_cast<const uint4 *>(smem + rq_off + off);
                    uint4 kv = *reinterpret_cast<const uint4 *>(smem + rk_off + off);
                    if (t >= L) qv = kv = make_uint4(0u, 0u, 0u, 0u);
                    const float rq = sm.rq[s][t], rk = sm.rk[s][t];
                    const float2 rq2 = make_float2(rq, rq), rk2 = make_float2(rk, rk);
                    const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
                    uint32_t wkp[4], wqp[4], wq[4], wk[4], wb[4], wn[4];
                    float2 kn[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 k2 = bf16x2_to_f2(kw[i]), q2 = bf16x2_to_f2(qw[i]);
                        const float2 e1 = make_float2(exp2f(H[0][i].x), exp2f(H[0][i].y));
                        const float2 e2 = make_float2(exp2f(-H[0][i].x), exp2f(-H[0][i].y));
                        const float2 kp = mul2(k2, e1), qp = mul2(q2, e1);
                        kn[i] = mul2(k2, e2);
                        wkp[i] = pack_bf16(kp.x, kp.y);
                        wqp[i] = pack_bf16(qp.x, qp.y);
                        wn[i] = pack_bf16(kn[i].x, kn[i].y);
                        const float2 xq = mul2(qp, mul2(Fs[i], rq2));     // Q_hat*Gamma
                        const float2 xk = mul2(kp, mul2(Fs[i], rk2));     // K_hat*Gamma
                        const float2 xb = mul2(kn[i], mul2(FC[i], rk2));  // Kbar
                        wq[i] = pack_f16(xq.x, xq.y);
                        wk[i] = pack_f16(xk.x, xk.y);
                        wb[i] = pack_f16(xb.x, xb.y);
                    }
                    sts128(ama + sw128_off(32 * blk + r, 8 * cg), wkp[0], wkp[1], wkp[2], wkp[3]);
                    sts128(ama + sw128_off(32 * blk + 16 + r, 8 * cg), wqp[0], wqp[1], wqp[2], wqp[3]);
                    sts128(amb + sw128_off(variant_off(blk) + t, 8 * cg), wn[0], wn[1], wn[2], wn[3]);
                    sts128(sbase + rq_off + off, wq[0], wq[1], wq[2], wq[3]);
                    sts128(sbase + rk_off + off, wk[0], wk[1], wk[2], wk[3]);
                    sts128(sbase + rg_off + off, wb[0], wb[1], wb[2], wb[3]);
#pragma unroll 1
                    for (int bt = blk + 1; bt < 4; ++bt) {
                        const float4 *d4 = reinterpret_cast<const float4 *>(&sm.fac[fb + 1 + bt - blk][c0]);
                        const float4 da = d4[0], db = d4[1];
                        const float2 v0 = mul2(kn[0], make_float2(da.x, da.y)), v1 = mul2(kn[1], make_float2(da.z, da.w));
                        const float2 v2 = mul2(kn[2], make_float2(db.x, db.y)), v3 = mul2(kn[3], make_float2(db.z, db.w));
                        sts128(amb + sw128_off(variant_off(bt) + t, 8 * cg), pack_bf16(v0.x, v0.y), pack_bf16(v1.x, v1.y),
                               pack_bf16(v2.x, v2.y), pack_bf16(v3.x, v3.y));
                    }
#pragma unroll
                    for (int jj = 0; jj < 3; ++jj)
#pragma unroll
                        for (int i = 0; i < 4; ++i) H[jj][i] = H[jj + 1][i];
                }
            }
            fence_proxy_async_smem();
            named_bar(3, NP);

            if (tid == kProLead) mbar_arrive(&sm.pdone[s]);   // operands and rq/rk/beta of chunk m ready
        }
    } else if (tid >= kHelp0) {
        // ------------------------------------------------ helper group
        // Row norms (one thread per row of q or k) and beta, beside the prologue's gate;
        // published to the prologue by the barrier that ends its gate step.
        const int htid = tid - kHelp0;
        auto load_logit = [&](int mm) {
            const int64_t cs = (int64_t)mm * C;
            const int Lm = (int)((len - cs) < C ? (len - cs) : C);
            return htid < Lm ? __bfloat162float(p.beta[(row_base + cs + htid) * p.H + h]) : 0.f;
        };
        float nb = 0.f;   // logit of token htid, loaded one chunk ahead
        if (htid < C && nchunks > 0) nb = load_logit(0);
        for (int m = 0; m < nchunks; ++m) {
            const int s = m & 1;
            const int64_t cs = (int64_t)m * C;
            const int L = (int)((len - cs) < C ? (len - cs) : C);
            const uint32_t rq_off = F_RAW + s * F_SLOT, rk_off = rq_off + 16384;
            named_bar(1, NP + NH);
            if (sm.dec_p) break;
            const float bl = nb;
            if (htid < C && m + 1 < nchunks) nb = load_logit(m + 1);
            for (int i = htid; i < 2 * C; i += NH) {
                const int t = i >> 1;
                const uint32_t base = (i & 1) ? rk_off : rq_off;
                float2 acc[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) acc[u] = make_float2(0.f, 0.f);
#pragma unroll
                for (int c16 = 0; c16 < 16; ++c16) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(
                        smem + base + (c16 >> 3) * 8192 + sw128_off(t, (c16 & 7) * 8));
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 x = bf16x2_to_f2(w[u]);
                        acc[u] = fma2(x, x, acc[u]);
                    }
                }
                const float2 s01 = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
                const float r = t < L ? rsqrtf(s01.x + s01.y + 1e-6f) : 0.f;
                if (i & 1) sm.rk[s][t] = r;
                else sm.rq[s][t] = r;
            }
            if (htid < C) sm.beta[s][htid] = htid < L ? 1.f / (1.f + exp2f(-bl * kLog2e)) : 0.f;
            named_bar(1, NP + NH);
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
                // Kbar, Q_hat*Gamma, K_hat*Gamma and exp(G_C) of chunk m go to workspace
                // slot s (L2) once the chain has loaded chunk m - 2 from it; the chain
                // pulls them with bulk loads.  (Shared-to-shared copies between the two
                // SMs move ~14 bytes per cycle; the slot round trip through L2 frees the
                // raw tiles sooner.)
                if (ok && m >= 2) ok = mbar_wait_cluster(&sm.gfree[s], ((m - 2) >> 1) & 1, kWait);
                unsigned char *slot = wsu + s * kWsSlot;
                if (ok) {
                    bulk_store(slot + WS_KB, smem + rg_off, 16384);
                    bulk_store(slot + WS_QG, smem + rq_off, 16384);
                    bulk_store(slot + WS_KG, smem + rk_off, 16384);
                    bulk_store(slot + WS_GC, &sm.gamC_f[s][0], 512);
                }
                bulk_commit();
                bulk_wait_read0();   // raw tiles and exp(G_C) of slot s may be overwritten
                if (!ok) {
                    set_err(p);
                    sm.abort_p = 1;
                    sm.abort_s = 1;
                    break;
                }
                if (m + 2 < nchunks) issue_raw(m + 2);
                bulk_wait0();        // the stores are complete in global memory
                fence_proxy_async_global();
                mbar_arrive_remote(chain_bar(&sm.gready[s]));
            }
            bulk_wait0();
        }
    } else {
        // ------------------------------------------------ solver group
        // Warp sw reads TMEM lane quarter sw of G1 = rows of token block sw: lanes 0-15
        // are A rows (Kp), lanes 16-31 M rows (Qp); it needs the sw + 1 chunks of 16
        // columns of variant sw.
        const int stid = tid - NP, sw = warp - 8;
        bool rbad = false;   // a T' or M value beyond the fp16 range
        float *Amat = reinterpret_cast<float *>(smem + F_AMAT);
        float *Tf = reinterpret_cast<float *>(smem + F_TF);
        // the M staging tile above the diagonal blocks stays zero for the whole run
        for (int k16 = stid; k16 < 512; k16 += NS) sts128(sbase + F_MST + k16 * 16, 0u, 0u, 0u, 0u);
        // T above its diagonal blocks is never written: zero once, so T' needs no mask
        for (int k4 = stid; k4 < 64 * LDA / 4; k4 += NS)
            reinterpret_cast<float4 *>(Tf)[k4] = make_float4(0.f, 0.f, 0.f, 0.f);
        named_bar(2, NS);
        for (int m = 0; m < nchunks; ++m) {
            const int s = m & 1;
            if (stid == kSolLead) {
                bulk_wait_read0();   // previous T'/M staging shipped
                if (!mbar_wait(&sm.pdone[s], (m >> 1) & 1, kWait) ||
                    !mbar_wait(&sm.g1_done[s], (m >> 1) & 1, kWait)) {
                    set_err(p);
                    sm.abort_s = 1;
                }
                sm.dec_s = sm.abort_s;
            }
            named_bar(2, NS);
            if (sm.dec_s) break;
            tc_fence_after();

            // A (fp32, beta_t/|k_t| x 1/|k_i|; only i < t is used later) and
            // M (fp16, 1/|q_t| x 1/|k_i|, zero for i > t); all column loads in flight at once
            {
                const bool is_m = lane >= 16;
                const int t = 16 * sw + (lane & 15);
                const float rowf = is_m ? sm.rq[s][t] : sm.beta[s][t] * sm.rk[s][t];
                const uint32_t col0 = 256 * s + variant_off(sw);
                float r[4][16];
                tmem_ld16(tmem_addr(tmem, 32 * sw, col0), r[0]);
                if (sw >= 1) tmem_ld16(tmem_addr(tmem, 32 * sw, col0 + 16), r[1]);
                if (sw >= 2) tmem_ld16(tmem_addr(tmem, 32 * sw, col0 + 32), r[2]);
                if (sw >= 3) tmem_ld16(tmem_addr(tmem, 32 * sw, col0 + 48), r[3]);
                tmem_ld_wait();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    if (kk > sw) break;
                    const float4 *rk4 = reinterpret_cast<const float4 *>(&sm.rk[s][16 * kk]);
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) {
                        const float4 x = rk4[e4];
                        const float2 f0 = mul2(make_float2(rowf, rowf), make_float2(x.x, x.y));
                        const float2 f1 = mul2(make_float2(rowf, rowf), make_float2(x.z, x.w));
                        const float2 y0 = mul2(f0, make_float2(r[kk][4 * e4], r[kk][4 * e4 + 1]));
                        const float2 y1 = mul2(f1, make_float2(r[kk][4 * e4 + 2], r[kk][4 * e4 + 3]));
                        r[kk][4 * e4] = y0.x; r[kk][4 * e4 + 1] = y0.y;
                        r[kk][4 * e4 + 2] = y1.x; r[kk][4 * e4 + 3] = y1.y;
                    }
                    if (is_m) {
                        if (kk == sw) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) r[kk][e] = e <= (lane & 15) ? r[kk][e] : 0.f;
                        }
                        st_pack16<true>(sbase + F_MST, t, 16 * kk, r[kk], rbad);
                    } else {
                        float4 *dst = reinterpret_cast<float4 *>(Amat + t * LDA + 16 * kk);
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4)
                            dst[e4] = make_float4(r[kk][4 * e4], r[kk][4 * e4 + 1], r[kk][4 * e4 + 2],
                                                  r[kk][4 * e4 + 3]);
                    }
                }
            }
            tc_fence_before();
            named_bar(2, NS);
            if (stid == kSolLead) mbar_arrive(&sm.am_free[s]);

            // T = (I + A)^-1 in 16x16 blocks.  Diagonal blocks: forward substitution,
            // thread = (block, column j), updating all later rows after each solved row.
            if (stid < 64) {
                const int bb = stid >> 4, j = stid & 15;
                const float *Ab = Amat + (16 * bb) * LDA + 16 * bb;
                float acc[16], x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) acc[r] = 0.f;
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    x[q] = q == j ? 1.f : (q < j ? 0.f : -acc[q]);
#pragma unroll
                    for (int r = q + 1; r < 16; ++r) acc[r] = fmaf(Ab[r * LDA + q], x[q], acc[r]);
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Tf[(16 * bb + r) * LDA + 16 * bb + j] = x[r];
            }
            named_bar(2, NS);
            // B[bt][m] = T[bt][bt] A[bt][m] for m < bt, in place of A's blocks: twelve
            // 16x8 tiles (bt, nt), three per warp, all operands loaded before the MMAs
            {
                uint32_t fa[3][2][4], fb[3][2][2];
#pragma unroll
                for (int u = 0; u < 3; ++u) {
                    const int idx = sw + 4 * u;
                    const int bt = idx < 2 ? 1 : (idx < 6 ? 2 : 3);
                    const int nt = idx - (bt == 1 ? 0 : (bt == 2 ? 2 : 6));
                    const float *Tb = Tf + (16 * bt) * LDA + 16 * bt;
                    const float *Ab = Amat + (16 * bt) * LDA + 8 * nt;
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        frag_a(Tb + 8 * ks, LDA, lane, fa[u][ks]);
                        frag_b(Ab + 8 * ks * LDA, LDA, lane, fb[u][ks]);
                    }
                }
                float acc[3][4];
#pragma unroll
                for (int u = 0; u < 3; ++u) {
                    acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
                    mma_tf32_16x8x8(acc[u], fa[u][0], fb[u][0]);
                    mma_tf32_16x8x8(acc[u], fa[u][1], fb[u][1]);
                }
                __syncwarp();
#pragma unroll
                for (int u = 0; u < 3; ++u) {
                    const int idx = sw + 4 * u;
                    const int bt = idx < 2 ? 1 : (idx < 6 ? 2 : 3);
                    const int nt = idx - (bt == 1 ? 0 : (bt == 2 ? 2 : 6));
                    store_16x8(Amat + (16 * bt) * LDA + 8 * nt, LDA, lane, acc[u], 1.f);
                }
            }
            named_bar(2, NS);
            // Off-diagonal blocks of column block ba (warp ba), right-looking: once
            // T[m][ba] is final, B[bt][m] T[m][ba] is added to the sum of every bt > m,
            // and T[m+1][ba] = -(its completed sum).
            if (sw <= 2) {
                const int ba = sw;
                float P[3][2][4];   // [bt - 1][n tile]
#pragma unroll
                for (int i = 0; i < 3; ++i)
#pragma unroll
                    for (int n = 0; n < 2; ++n) P[i][n][0] = P[i][n][1] = P[i][n][2] = P[i][n][3] = 0.f;
#pragma unroll
                for (int m = 0; m < 3; ++m) {
                    if (m < ba) continue;
                    uint32_t tb[2][2][2];
                    const float *Tm = Tf + (16 * m) * LDA + 16 * ba;
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
#pragma unroll
                        for (int n = 0; n < 2; ++n) frag_b(Tm + 8 * ks * LDA + 8 * n, LDA, lane, tb[ks][n]);
#pragma unroll
                    for (int bt = m + 1; bt < 4; ++bt) {
                        uint32_t fa[2][4];
                        const float *Bp = Amat + (16 * bt) * LDA + 16 * m;
                        frag_a(Bp, LDA, lane, fa[0]);
                        frag_a(Bp + 8, LDA, lane, fa[1]);
#pragma unroll
                        for (int n = 0; n < 2; ++n) {
                            mma_tf32_16x8x8(P[bt - 1][n], fa[0], tb[0][n]);
                            mma_tf32_16x8x8(P[bt - 1][n], fa[1], tb[1][n]);
                        }
                    }
                    float *dst = Tf + (16 * (m + 1)) * LDA + 16 * ba;
                    store_16x8(dst, LDA, lane, P[m][0], -1.f);
                    store_16x8(dst + 8, LDA, lane, P[m][1], -1.f);
                    __syncwarp();
                }
            }
            named_bar(2, NS);
            // T' = T Diag(beta), fp16, into the staging tile (over the dead A)
            {
                const int t = stid >> 1, i0 = (stid & 1) * 32;
                const float4 *b4 = reinterpret_cast<const float4 *>(&sm.beta[s][i0]);
                const float4 *t4 = reinterpret_cast<const float4 *>(Tf + t * LDA + i0);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float r[16];
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) {
                        const float4 tv = t4[4 * hh + e4], bv = b4[4 * hh + e4];
                        const float2 y0 = mul2(make_float2(tv.x, tv.y), make_float2(bv.x, bv.y));
                        const float2 y1 = mul2(make_float2(tv.z, tv.w), make_float2(bv.z, bv.w));
                        r[4 * e4] = y0.x; r[4 * e4 + 1] = y0.y; r[4 * e4 + 2] = y1.x; r[4 * e4 + 3] = y1.y;
                    }
                    st_pack16<true>(sbase + F_AMAT, t, i0 + 16 * hh, r, rbad);
                }
            }
            fence_proxy_async_smem();
            named_bar(2, NS);
            if (stid == kSolLead) {
                mbar_arrive(&sm.s_done[s]);
                bool ok = true;
                const uint32_t full = chain_bar(&sm.full[s]);
                if (m >= 2) ok = mbar_wait_cluster(&sm.slot_free[s], ((m - 2) >> 1) & 1, kWait);
                if (ok) {
                    bulk_copy_to_peer(chain_addr(s ? C_T1 : C_TZM), sbase + F_AMAT, 8192, full);
                    bulk_copy_to_peer(chain_addr(C_TZM + 16384 + s * 16384), sbase + F_MST, 8192, full);
                }
                bulk_commit();
                if (!ok) { set_err(p); sm.abort_s = 1; sm.abort_p = 1; }
            }
        }
        flag_range(p, rbad);
        if (stid == kSolLead) bulk_wait0();
    }
}

// ============================================================== chain CTA
__device__ __forceinline__ void run_chain(const TmaMaps &maps, const Params &p, unsigned char *smem,
                                          Small &sm, uint32_t tmem, int64_t unit, int64_t n, int64_t h,
                                          int64_t row_base, int64_t len, int nchunks) {
    const unsigned char *wsu = p.ws + unit * kWsBytesPerUnit;   // this cluster's workspace
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = (warp >> 2) & 1;   // TMEM lane quarter; column half
    const uint32_t D_S = tmem, D_W = tmem + 128, D_U = tmem + 256;
    const uint32_t front_small = mapa_shared(smem_u32(&sm), 0);
    auto front_bar = [&](uint64_t *local_bar) {
        return front_small + (smem_u32(local_bar) - smem_u32(&sm));
    };
    const size_t state_base = (size_t)(n * p.H + h) * DK * DK;

    auto issue_v = [&](int chunk) {
        if (!p.v) {   // values taken as zero (the tile stays zero): only the phase completes
            mbar_arrive(&sm.v_full);
            return;
        }
        const int row = (int)(row_base + (int64_t)chunk * C);
        mbar_arrive_expect_tx(&sm.v_full, 16384);
        tma_load_3d(smem + C_B2 + 16384, &maps.v, &sm.v_full, 0, (int)h, row);
        tma_load_3d(smem + C_B2 + 16384 + 8192, &maps.v, &sm.v_full, 64, (int)h, row);
    };
    // Thread 0: the workspace tiles of chunk j into their operand buffers (on full[j & 1]),
    // once the front has written them; returns false if that wait gave up.
    auto load_chunk = [&](int j) -> bool {
        const int sj = j & 1;
        if (!mbar_wait_cluster(&sm.gready[sj], (j >> 1) & 1, kWait)) return false;
        fence_proxy_async_global();
        const unsigned char *slot = wsu + sj * kWsSlot;
        const uint32_t fb = smem_u32(&sm.full[sj]);
        bulk_load(sbase + C_KB + sj * 16384, slot + WS_KB, 16384, fb);
        bulk_load(sbase + C_G3A + 8192, slot + WS_QG, 8192, fb);
        bulk_load(sbase + C_G3A + 16384 + 8192, slot + WS_QG + 8192, 8192, fb);
        bulk_load(sbase + C_B2, slot + WS_KG, 16384, fb);
        bulk_load(smem_u32(&sm.gamC_c[sj][0]), slot + WS_GC, 512, fb);
        return true;
    };
    // waits done by thread 0 and published to the CTA; returns true to abort
    auto lead_wait = [&](bool ok) -> bool {
        if (tid == 0 && !ok) { set_err(p); sm.abort_c = 1; }
        __syncthreads();
        return sm.abort_c != 0;
    };
    bool rbad = false;   // a V, U, W or state value beyond the fp16 range
    auto convert_v = [&]() {
        for (int k16 = tid; k16 < 1024; k16 += NT) {
            uint4 *ptr = reinterpret_cast<uint4 *>(smem + C_B2 + 16384 + k16 * 16);
            *ptr = bf16_to_f16x8(*ptr, rbad);
        }
    };
    // -W (D_W lanes 0..63) -> rows 0..63 of the G3 A operand: warps 8, 9, 12, 13
    // (lane quarter 0/1, one column half each)
    auto read_w = [&]() {
        if (warp == 8 || warp == 9 || warp == 12 || warp == 13) {
            const int t = quarter * 32 + lane;
            {
                const int cb = half;
                float r[4][16];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) tmem_ld16(tmem_addr(D_W, quarter * 32, 64 * cb + 16 * jj), r[jj]);
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) r[jj][e] = -r[jj][e];
                    st_pack16<true>(sbase + C_G3A + cb * 16384, t, 16 * jj, r[jj], rbad);
                }
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
    auto issue_g2w = [&](int j) {   // W of chunk j (its T' slot)
        const uint32_t id = idesc_fp16(128, 128, false, true);
        for (int ks = 0; ks < C / 16; ++ks)
            mma_bf16(D_W, sdesc_sw128(sbase + ((j & 1) ? C_T1 : C_TZM) + ks * 32, 16, 1024),
                     sdesc_sw128(sbase + C_B2 + ks * 2048, 8192, 1024), id, ks > 0);
        mma_commit(&sm.w_bar);
    };

    // zero tiles (rows 64..127 of [T'; 0], rows 0..63 of [0; M0] and [0; M1])
    for (int k16 = tid; k16 < 512; k16 += NT) {
        sts128(sbase + C_TZM + 8192 + k16 * 16, 0, 0, 0, 0);
        sts128(sbase + C_TZM + 24576 + k16 * 16, 0, 0, 0, 0);
        sts128(sbase + C_T1 + 8192 + k16 * 16, 0, 0, 0, 0);
    }
    if (!p.v)
        for (int k16 = tid; k16 < 1024; k16 += NT) sts128(sbase + C_B2 + 16384 + k16 * 16, 0, 0, 0, 0);
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
            st_pack16<true>(sbase + C_SB + half * 16384, c, 16 * jj, r, rbad);
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
            ok = load_chunk(0) && mbar_wait(&sm.full[0], 0, kWait) && mbar_wait(&sm.v_full, 0, kWait);
            if (ok) mbar_arrive_remote(front_bar(&sm.gfree[0]));
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
                issue_g2w(0);
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
                mma_bf16(D_U, sdesc_sw128(sbase + (s ? C_T1 : C_TZM) + ks * 32, 16, 1024),
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
            if (m + 1 < nchunks) {
                issue_v(m + 1);
                if (!load_chunk(m + 1)) set_err(p);   // the full wait of step (c) then gives up too
            }
        }
        if (warp < 8 && quarter < 2) {   // warps 0, 1, 4, 5: lane quarter 0/1, column half
            const int t = quarter * 32 + lane;
            float r[4][16];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) tmem_ld16(tmem_addr(D_U, quarter * 32, 64 * half + 16 * jj), r[jj]);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) st_pack16<true>(sbase + C_UT + half * 8192, t, 16 * jj, r[jj], rbad);
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
                    mbar_arrive_remote(front_bar(&sm.gfree[s ^ 1]));
                    tc_fence_after();
                    issue_g2w(m + 1);
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
            for (int jj = 0; jj < 4; ++jj) st_pack16<true>(sbase + C_SB + half * 16384, c, 16 * jj, r[jj], rbad);
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
        } else if (warp == 10 || warp == 11 || warp == 14 || warp == 15) {
            // O rows (D_U lanes 64..127): lane quarter 2/3, one column half each
            const int t = (quarter - 2) * 32 + lane;
            const float sc = p.scale;
            {
                const int hb = half;
                float r[4][16];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    tmem_ld16(tmem_addr(D_U, (warp & 3) * 32, 64 * hb + 16 * jj), r[jj]);
                tmem_ld_wait();
                if (t < L && p.out) {
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

    flag_range(p, rbad);
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
    // 1024-byte alignment (128B-swizzled tiles) by pointer arithmetic on the shared
    // array itself, so that every access through `smem` stays a shared-memory access
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
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
    if (p.mixed && len <= kShortMaxT) return;   // the short-step kernel's (both CTAs agree)
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
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.gready[i], 1);
            mbar_init(&sm.gfree[i], 1);
        }
        mbar_init(&sm.v_full, 1);
        mbar_init(&sm.mma_bar, 1);
        mbar_init(&sm.w_bar, 1);
        sm.abort_p = sm.abort_s = sm.abort_c = 0;
        sm.dec_p = sm.dec_s = 0;
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
        run_front(maps, p, smem, sm, tmem, unit, h, row_base, len, nchunks);
    else
        run_chain(maps, p, smem, sm, tmem, unit, n, h, row_base, len, nchunks);

    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no CTA leaves while its peer may still signal it
    if (threadIdx.x < 32) tmem_dealloc(tmem, 512);
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
    static std::atomic<bool> attr_done[kMaxDevices];
    cudaError_t e = once_per_device(attr_done, [](int) {
        return cudaFuncSetAttribute(kda_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    });
    if (e != cudaSuccess) return e;
    kda_cluster_kernel<<<(unsigned)(2 * units), NT, SMEM_BYTES, stream>>>(maps, p);
    return cudaGetLastError();
}

}  // namespace kda
