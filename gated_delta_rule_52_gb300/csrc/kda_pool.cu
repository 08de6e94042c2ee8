// KDA forward on sm_103a with a persistent pool of CTAs: "fronts" run the
// chunk-parallel part of every chunk of every (sequence, head) unit, "chains" run
// the sequential state recurrence, one unit at a time each.  Fronts hand each chunk's
// operands to its chain through a ring of slots in global memory (resident in L2).
//
// The chunk algebra is that of the UT/WY (chunked) form of the KDA token recurrence
// (FlashKDA README "Kernel API"; the recurrence is the gated delta rule with one decay
// rate per key channel), over 64-token chunks with S the K x V state entering the chunk,
// G the in-chunk cumulative log decay and Gamma = exp(G):
//   A[t,i] = beta_t sum_c k[t,c] k[i,c] exp(G[t,c]-G[i,c])  (i < t)
//   M[t,i] =        sum_c q[t,c] k[i,c] exp(G[t,c]-G[i,c])  (i <= t)
//   T' = (I + A)^-1 Diag(beta);  W = T' (K_hat*Gamma);  U = T' V - W S
//   O  = scale ((Q_hat*Gamma) S + M U);   S <- Diag(Gamma_C) S + Kbar^T U
// Everything up to the last line's inputs depends only on the chunk's own tokens; only
// the last line's two products carry the state from chunk to chunk.
//
// Grid: one CTA per SM, launched cooperatively (all CTAs resident at once, which the
// flag waits between CTAs need).  CTAs 0 .. nc-1 are chains, the rest fronts.
//   Fixed-length calls: chain c owns units c, c + nc, ...; its packets (chunks) j = 0,
//   1, ... are chunk j % nchunks of unit c + (j / nchunks) nc.  Front f takes the
//   packets of global index i = f, f + nf, f + 2 nf, ... in the order i = j * nc + c
//   (packet j of chain c), so fronts produce packets in the order the chains consume
//   them.
//   Varlen calls: a one-CTA plan (pool_plan_kernel) sorts the sequences longest first
//   and deals their (sequence, head) units to the chains in snake order (round w gives
//   unit w nc + c to chain c in even rounds, w nc + nc - 1 - c in odd ones), so that
//   every chain gets about the same number of packets.  Global index i then runs over
//   steps j, and within a step over the chains that still have a packet j, longest
//   chain first; the plan writes that list of packets for the fronts.
//   Either way the packet of lowest index not yet produced can always be produced (the
//   slot it needs holds a packet of lower index, which its chain consumes), so the pool
//   cannot deadlock.
// Packet (c, j) goes through ring slot (c, j % D): the front waits until the chain
// has loaded packet j - D out of it ("freed" flag), stores the packet, then sets
// the slot's "ready" flag; the chain's loader warp waits for "ready", bulk-loads the
// packet and sets "freed".  Flags hold the packet index + 1; every call clears them (a
// stream-ordered memset before the launch), so neither a reused workspace nor a replayed
// CUDA graph can meet a flag that matches too early.
//
// Front CTA (per packet, pipelined as in the cluster kernel's front): warps 0-7 the
// prologue (gate, block-local decay, the operands of G1 = [Kp; Qp] x Kn^T and the
// chain tiles K_hat*Gamma, Q_hat*Gamma, Kbar), warps 13-15 row norms and beta, warp 12
// G1 and the ring stores of the chain tiles, warps 8-11 the A/M readout, the blocked
// inverse and T', stored with M.
// Chain CTA: the state steps on tcgen05 with the fp32 state in TMEM (roles at
// pool_chain); in the state-only runs of the sequence-parallel path it carries a second
// state with values of zero beside the first (DUAL).
//
// Precision: G1 on bf16 operands of the raw q/k scaled by 16-token-block-local decay
// factors, the other GEMMs on fp16 operands, fp32 accumulators, fp32 state.  Every wait
// is bounded (2 s); a timeout sets the device error word and the CTA unwinds.
#include <type_traits>

#include "kda_chunk.cuh"

namespace kda {
namespace {

using namespace sm103;
using namespace chunk;

constexpr int NT = 512;            // 16 warps
constexpr int kLoaderWarp = 12;    // chain: ring loader (the control warp in a front)
constexpr int NP = 256;            // front prologue group: warps 0-7
constexpr int NS = 128;            // front solver group: warps 8-11
constexpr int NH = 96;             // front helper group (norms, beta): warps 13-15
constexpr int kHelp0 = 416;        // first helper thread
constexpr int kProLead = 32;       // thread that waits for the prologue group (warp 1)
constexpr int kSolLead = 64;       // index within the solver group of its waiting thread (warp 10)
constexpr uint32_t kChunkBytes = 16384 * 3 + 512 + 8192 * 2;   // one packet
// ring slot layout: Kbar, Q_hat*Gamma, K_hat*Gamma (fp16 tiles), exp(G_C) (fp32), T', M (fp16)
constexpr uint32_t RS_KB = 0, RS_QG = 16384, RS_KG = 32768, RS_GC = 49152, RS_TP = 49664, RS_MM = 57856;
static_assert(RS_MM + 8192 == kChunkBytes, "ring slot layout");

// ---- front shared memory
constexpr uint32_t F_RAW = 0;          // 2 slots x {q, k, g}: 16 KB each, 2 x [64 t][64 c]
constexpr uint32_t F_SLOT = 49152;
constexpr uint32_t F_AMA = 98304;      // [Kp; Qp]: 2 x [128][64] bf16
constexpr uint32_t F_AMB = 131072;     // Kn variants: 2 x [160][64] bf16
constexpr uint32_t F_MST = 172032;     // M staging fp16 [64 t][64 i]
constexpr uint32_t F_AMAT = 180224;    // A fp32 [64][68]; T' staging (fp16) after the inverse
constexpr uint32_t F_TF = 197632;      // T fp32 [64][68]
// ---- chain shared memory
constexpr uint32_t C_SH = 0;           // S^T fp16: 2 x [128 c][64 v] (A, MN-major)
constexpr uint32_t C_UH = 32768;       // U^T fp16: [128 v][64 t] (K-major)
constexpr uint32_t C_WT = 49152;       // -W^T fp16: [128 c][64 t] (B, MN-major)
constexpr uint32_t C_V = 65536;        // 2 buffers x V [64 t][128 v] as 2 x [64][64] (bf16 -> fp16)
constexpr uint32_t C_PK = 98304;       // 2 packet slots
constexpr uint32_t C_PKSLOT = 65536;
constexpr uint32_t PK_KB = 0, PK_QG = 16384, PK_KG = 32768, PK_TP = 49152, PK_MM = 57344;
constexpr uint32_t C_END = C_PK + 2 * C_PKSLOT;
// chain with a second state (state-only runs): no O, so no Q_hat*Gamma or M in a packet;
// the second state's S^T and U^T copies take their place
constexpr uint32_t C2_SHP = 98304;      // second S^T fp16: 2 x [128 c][64 v]
constexpr uint32_t C2_UHP = 131072;     // second U^T fp16: [128 v][64 t]
constexpr uint32_t C2_PK = 147456;      // 2 packet slots: Kbar, K_hat*Gamma, T'
constexpr uint32_t C2_PKSLOT = 40960;
constexpr uint32_t P2_KB = 0, P2_KG = 16384, P2_TP = 32768;
static_assert(C2_PK + 2 * C2_PKSLOT <= C_END, "second-state chain layout");
constexpr uint32_t F_END = F_TF + 64 * LDA * 4;

// Rows of the decay-factor table of one chunk (per 16-token block b and channel c), with
// Gs[b] the cumulative log2 decay before block b, G_C the chunk total and mu[b] half of
// block b's total (the shift of the operand factors, see the prologue):
//   pool_fac_base(b) + 0: 2^(Gs[b] + mu[b])       Q_hat Gamma, K_hat Gamma (with 2^(H - mu))
//                    + 1: 2^(G_C - Gs[b] - mu[b]) Kbar (with 2^(mu - H))
//                    + 2: 2^(mu[b])               b < 3: turns 2^(mu - H) into 2^(Gs[b+1] - G)
//                    + 2 + (bt - b): 2^(Gs[bt] - Gs[b+1] + mu[bt])  key variant of row block bt > b
// Every entry is at most 1.  Each variant is the product of two factors at most 1
// (2^(Gs[b+1] - G) first, then the table entry), so where a factor underflows the term
// it belongs to is below 2^-37 of the largest one.  With the lower bound, mu = 0 and the
// variant of row block bt is 2^-H times the single entry 2^(Gs[bt] - Gs[b]) (row + 2 +
// (bt - b); the row + 2 entry is unused): every block decays by at most 2^-115, so
// neither factor leaves the fp32 range.
constexpr int kPoolFacRows = 17;
__device__ __forceinline__ int pool_fac_base(int b) { return b == 0 ? 0 : (b == 1 ? 6 : (b == 2 ? 11 : 15)); }

struct FrontSmall {
    float rq[3][C], rk[3][C], beta[3][C];   // per norm slot (task % 3)
    float btot[4][DK];
    float fac[kPoolFacRows][DK];             // decay factors, see pool_fac_base
    float gamC_f[2][DK];                     // exp(G_C) per slot (store source)
    float gb[2][DK];                         // gate bias a2 * dt_bias[h] per slot (log2 units)
    float ga[2];                             // a2 = -exp(A_log[h]) log2(e) per slot
    uint64_t raw_full[2], g1_done[2], am_free[2];
    // the prologue's "task m ready", per task % 3: the prologue runs at most three tasks
    // ahead of the solver (s_done), so no waiter falls a whole phase behind
    uint64_t pdone[3];
    uint64_t s_done[3];   // the solver is done with norm slot task % 3
    unsigned int ctl_count;   // tasks whose chain tiles the control warp has stored (complete)
    int abort_p, abort_s;
    int dec_p, dec_s;   // a group's abort decision, written by its lead thread only, before a barrier
};
struct ChainSmall {
    float gamC[2][DK];   // exp(G_C) of the packet in each slot
    // Barriers that complete once per packet are per packet parity ([2]) wherever a
    // waiter could otherwise fall two phases behind
    uint64_t full_e[2], full_l[2], vfull[2], vconv[2], u_done[2], o_done[2];
    uint64_t w_done, s_done, o_free, sh_ready, s_scaled, uh_ready, wt_ready, fin;
    uint64_t up_done;    // G3u of the second state (runs with a second state only)
    int abort;
};
constexpr uint32_t F_SMALL = F_END;
constexpr uint32_t C_SMALL = C_END;
constexpr uint32_t COMMON_A = (F_SMALL + sizeof(FrontSmall) > C_SMALL + sizeof(ChainSmall)
                                   ? F_SMALL + sizeof(FrontSmall)
                                   : C_SMALL + sizeof(ChainSmall));
constexpr uint32_t COMMON = (COMMON_A + 15u) & ~15u;   // TMEM base address
constexpr uint32_t SMEM_BYTES = COMMON + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// ---------------------------------------------------------------- ring and flags
// Ring depth D (slots per chain).  Any D >= 1 is free of deadlock: the publication of a
// packet waits only on work of its own front and on ring slots of packets of lower index
// (a front publishes its previous packet before it waits for anything of the next one).
// D is a matter of speed: with about nf / nc fronts per chain, D > nf / nc plus a few
// slots (at least kRingMin) lets the fronts run ahead of the chains without waiting on
// the ring.
constexpr int kRingMin = 8;
__host__ __device__ constexpr int64_t ring_depth(int64_t nc, int64_t nf) {
    return nf / nc + 6 > kRingMin ? nf / nc + 6 : kRingMin;
}

// Device side of the ring: D slots of kChunkBytes per chain, and per chain D "ready"
// words then D "freed" words.
struct PoolArgs {
    unsigned char *ring;
    unsigned long long *flags;
    int nc, nf;                 // chain CTAs, front CTAs
    int depth;                  // ring slots per chain
    int nchunks;                // chunks per unit (fixed-length calls)
    int waves;                  // ceil(units / nc)
    // varlen calls: the plan of pool_plan_kernel (null for fixed-length calls)
    const int4 *plist;          // packets in production order: {chain, packet, first row, h << 8 | rows}
    const int *order;           // the sequences the pool takes, longest first
    const int *chain_len;       // packets per chain
    const int *counts;          // [0] packets in all, [1] units the pool takes

    __device__ unsigned char *slot(int64_t c, int64_t j) const {
        return ring + ((size_t)c * depth + (size_t)(j % depth)) * kChunkBytes;
    }
    __device__ unsigned long long *ready(int64_t c, int64_t j) const {
        return flags + (size_t)c * 2 * depth + (size_t)(j % depth);
    }
    __device__ unsigned long long *freed(int64_t c, int64_t j) const {
        return flags + (size_t)c * 2 * depth + depth + (size_t)(j % depth);
    }
    __device__ unsigned long long tag(int64_t j) const { return (unsigned long long)j + 1ull; }
};

__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long *ptr) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ptr) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned long long *ptr, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(ptr), "l"(v) : "memory");
}
__device__ __forceinline__ void st_release_cta(unsigned int *ptr, unsigned int v) {
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(ptr)), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire_cta(const unsigned int *ptr) {
    unsigned int v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(ptr)) : "memory");
    return v;
}
// Waits until *ptr == want (another CTA's release store), giving up after limit_ns.
__device__ __forceinline__ bool wait_flag(const unsigned long long *ptr, unsigned long long want,
                                          uint64_t limit_ns) {
    if (ld_acquire_gpu(ptr) == want) return true;
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(ptr) != want)
        if (globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

// The packets of one front in order: global index i = f, f + nf, ...; i = j * nc + c.
// The decomposition is carried along incrementally (no 64-bit divisions per packet).
struct TaskIt {
    int64_t i, end;       // current global index; one past the last
    int units, H, nf, nc, nchunks, dj, dc;   // dj, dc: nf / nc and nf % nc
    int c, m, w;          // chain, chunk of the unit, wave (unit = c + w nc)
    // the current packet
    int64_t j, row;       // packet index of its chain, first token row in [B*T]
    int h, L;             // head; its token rows (<= 64)

    __device__ bool decode(const Params &p) {
        const int u = c + w * nc;
        if (u >= units) return false;
        const int n = u / H;
        h = u - n * H;
        j = (int64_t)w * nchunks + m;
        row = (int64_t)n * p.T + (int64_t)m * C;
        const int64_t rem = p.T - (int64_t)m * C;
        L = (int)(rem < C ? rem : C);
        return true;
    }
    // moves (c, m, w) on by nf global indices
    __device__ void step() {
        c += dc;
        int add = dj;
        if (c >= nc) {
            c -= nc;
            ++add;
        }
        m += add;
        while (m >= nchunks) {
            m -= nchunks;
            ++w;
        }
    }
    __device__ void advance(const Params &p) {
        for (i += nf, step(); i < end; i += nf, step())
            if (decode(p)) return;
    }
    __device__ void start(int f, const PoolArgs &a, int64_t units_, const Params &p) {
        units = (int)units_;
        H = (int)p.H;
        nf = a.nf;
        nc = a.nc;
        nchunks = a.nchunks;
        dj = nf / nc;
        dc = nf - dj * nc;
        end = (int64_t)a.waves * nchunks * nc;
        i = f;
        c = f % nc;
        const int jf = f / nc;
        m = jf % nchunks;
        w = jf / nchunks;
        if (i < end && !decode(p)) advance(p);
    }
    __device__ bool valid() const { return i < end; }
};

// The packets of one front of a varlen call, from the plan's list (the entry one step
// ahead is loaded a task early, so that its latency is hidden).
struct TaskItV {
    int64_t i, end;
    int nf;
    const int4 *pl;
    int4 nxt;
    int c, h, L;
    int64_t j, row;
    __device__ void take(const int4 e) {
        c = e.x;
        j = e.y;
        row = e.z;
        h = e.w >> 8;
        L = e.w & 0xff;
    }
    __device__ void start(int f, const PoolArgs &a, int64_t, const Params &) {
        pl = a.plist;
        nf = a.nf;
        end = a.counts[0];
        i = f;
        if (i < end) take(pl[i]);
        if (i + nf < end) nxt = pl[i + nf];
    }
    __device__ void advance(const Params &) {
        i += nf;
        if (i < end) take(nxt);
        if (i + nf < end) nxt = pl[i + nf];
    }
    __device__ bool valid() const { return i < end; }
};

// Varlen: unit of chain c in snake round w (see the plan), and the walk over a chain's
// packets that skips units without tokens.
struct UnitV {
    int64_t row0;    // first token row of the sequence
    int64_t sbase;   // element offset of the (sequence, head) state
    int h, len, nch;
    bool valid;
};
__device__ __forceinline__ UnitV unit_v(const Params &p, const PoolArgs &a, int c, int64_t w, int64_t U) {
    UnitV u;
    const int64_t k = w * a.nc + ((w & 1) ? (a.nc - 1 - c) : c);
    u.valid = k < U;
    u.row0 = u.sbase = 0;
    u.h = u.len = u.nch = 0;
    if (!u.valid) return u;
    const int64_t sq = k / p.H;
    u.h = (int)(k - sq * p.H);
    const int n = a.order[sq];
    u.row0 = p.cu_seqlens[n];
    u.len = (int)(p.cu_seqlens[n + 1] - u.row0);
    u.nch = (u.len + C - 1) / C;
    u.sbase = ((int64_t)n * p.H + u.h) * DK * DK;
    return u;
}
struct PkWalkV {
    UnitV u;
    int64_t w, U;
    int m, c;
    __device__ void skip(const Params &p, const PoolArgs &a) {
        while (u.valid && m >= u.nch) {
            ++w;
            m = 0;
            u = unit_v(p, a, c, w, U);
        }
    }
    __device__ void start(const Params &p, const PoolArgs &a, int c_) {
        c = c_;
        U = a.counts[1];
        w = 0;
        m = 0;
        u = unit_v(p, a, c, 0, U);
        skip(p, a);
    }
    __device__ void next(const Params &p, const PoolArgs &a) {
        ++m;
        skip(p, a);
    }
    __device__ int64_t row() const { return u.row0 + (int64_t)m * C; }
    __device__ int rows() const { return u.len - m * C < C ? u.len - m * C : C; }
};

// ============================================================== front CTA
// UB: the gate without a lower bound, gk = -exp(A_log) softplus(g + dt_bias), each
// token's log2 decay raised to at least kMinGate2 (see the gate step).
constexpr float kMinGate2 = -14.f;

template <bool VL, bool UB>
__device__ __forceinline__ void pool_front(const TmaMaps &maps, const Params &p, const PoolArgs &a,
                                           unsigned char *smem, FrontSmall &sm, uint32_t tmem, int f) {
    using TaskIt = typename std::conditional<VL, TaskItV, ::kda::TaskIt>::type;
    const int64_t units = p.n_seqs * p.H;
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // raw q, k, g tiles of packet `t` into raw slot m & 1
    auto issue_raw = [&](int m, const TaskIt &t) {
        const int s = m & 1;
        unsigned char *base = smem + F_RAW + s * F_SLOT;
        mbar_arrive_expect_tx(&sm.raw_full[s], 3 * 16384);
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_3d(base + kb * 8192, &maps.q, &sm.raw_full[s], kb * 64, (int)t.h, (int)t.row);
            tma_load_3d(base + 16384 + kb * 8192, &maps.k, &sm.raw_full[s], kb * 64, (int)t.h, (int)t.row);
            tma_load_3d(base + 32768 + kb * 8192, &maps.g, &sm.raw_full[s], kb * 64, (int)t.h, (int)t.row);
        }
    };

    if (tid < NP) {
        // ------------------------------------------------ prologue group
        // Thread layout for the gate and the operands: warp = (16-token block, 64-channel
        // half), lane = (4-token quarter of the block, 8-channel group); every access to
        // the tiles is one 16-byte vector (8 channels of one token).
        const float lb2 = p.lower_bound * kLog2e;
        const int blk = warp >> 1, kh = warp & 1;
        const int cg = lane & 7, qr = lane >> 3;
        const int c0 = 64 * kh + 8 * cg;             // first of this thread's 8 channels
        const uint32_t kho = kh * 8192;              // the half inside a raw tile
        TaskIt it;
        it.start(f, a, units, p);
        for (int m = 0; it.valid(); ++m, it.advance(p)) {   // m: this front's task count
            const int s = m & 1;
            const int L = it.L;
            const uint32_t rq_off = F_RAW + s * F_SLOT, rk_off = rq_off + 16384, rg_off = rq_off + 32768;
            if (tid == kProLead) {
                bool ok = mbar_wait(&sm.raw_full[s], (m >> 1) & 1, kWait);
                if (ok && m >= 3) ok = mbar_wait(&sm.s_done[m % 3], ((m - 3) / 3) & 1, kWait);
                if (!ok) { set_err(p); sm.abort_p = 1; }
                sm.dec_p = sm.abort_p;
            }
            named_bar(1, NP + NH);   // with the helpers: raw tiles and gate parameters of task m are in
            if (sm.dec_p) break;
            const float a2 = sm.ga[s];
            float2 bias[4];
            {
                const float4 *gb4 = reinterpret_cast<const float4 *>(&sm.gb[s][c0]);
                const float4 ba = gb4[0], bb = gb4[1];
                bias[0] = make_float2(ba.x, ba.y);
                bias[1] = make_float2(ba.z, ba.w);
                bias[2] = make_float2(bb.x, bb.y);
                bias[3] = make_float2(bb.z, bb.w);
            }

            // gate (log2 units) and its block-local inclusive cumulative sum H (channel pairs)
            float2 H[4][4];
            {
                const float2 a2v = make_float2(a2, a2), lb2v = make_float2(lb2, lb2);
                const float2 one = make_float2(1.f, 1.f), l2ev = make_float2(kLog2e, kLog2e);
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
                            if constexpr (UB) {
                                // y = (g + dt_bias) log2 e; softplus in log2 units is
                                // max(y, 0) + log2(1 + 2^-|y|).  Where 2^-|y| is tiny, 1 + 2^-|y|
                                // rounds and the last term carries an absolute error of about
                                // 2e-7, so the per-token log2 decay (rate times softplus) one
                                // below 4e-6 at rates up to 16: far below the rounding of the
                                // fp32 in-chunk sums of those decays
                                const float2 y = fma2(bf16x2_to_f2(gw[i]), l2ev, bias[i]);
                                const float2 u = add2(make_float2(exp2f(-fabsf(y.x)), exp2f(-fabsf(y.y))), one);
                                const float2 sp = make_float2(fmaxf(y.x, 0.f) + __log2f(u.x), fmaxf(y.y, 0.f) + __log2f(u.y));
                                const float2 gk = mul2(a2v, sp);
                                acc[i] = add2(acc[i], make_float2(fmaxf(gk.x, kMinGate2), fmaxf(gk.y, kMinGate2)));
                            } else {
                                const float2 z = fma2(bf16x2_to_f2(gw[i]), a2v, bias[i]);
                                const float2 d = add2(make_float2(exp2f(z.x), exp2f(z.y)), one);
                                acc[i] = fma2(lb2v, make_float2(__fdividef(1.f, d.x), __fdividef(1.f, d.y)), acc[i]);
                            }
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
                // UB: H relative to mu = half the block's total decay (lane 24 + cg holds
                // the total), so that the row factors 2^(H - mu) and the diagonal key factors
                // 2^(mu - H) both stay within 2^(+-total / 2).  With the lower bound a block
                // decays by at most 2^-115 and mu = 0 (no shift) keeps every factor in range.
                if constexpr (UB) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 mu = make_float2(-0.5f * __shfl_sync(0xffffffffu, acc[i].x, 24 + cg),
                                                      -0.5f * __shfl_sync(0xffffffffu, acc[i].y, 24 + cg));
#pragma unroll
                        for (int j = 0; j < 4; ++j) H[j][i] = add2(H[j][i], mu);
                    }
                }
            }
            named_bar(1, NP + NH);   // gate totals, and the helpers' norms and beta

            // decay factors per (block, channel): thread = channel, two blocks each
            {
                const int c = tid & (DK - 1), bh = tid >> 7;
                float Gs[4], mu[4], tot = 0.f;
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
                    const float bt = sm.btot[bb][c];
                    Gs[bb] = tot;
                    mu[bb] = UB ? 0.5f * bt : 0.f;   // the prologue's shift of block bb (same value)
                    tot += bt;
                }
                if (bh == 0) sm.gamC_f[s][c] = exp2f(tot);
                // with mu[b] = half of block b's total (the shift of the operand factors):
                // Q/K times 2^G = (2^(H - mu)) 2^(Gs + mu); Kbar = (2^(mu - H)) 2^(G_C - Gs - mu);
                // key variant of row block bt = (2^(mu - H)) 2^(Gs[bt] - Gs[b] + mu[bt] - mu[b]);
                // every table factor is at most 1
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    if ((b >> 1) != bh) continue;
                    float *f = &sm.fac[pool_fac_base(b)][c];
                    f[0] = exp2f(Gs[b] + mu[b]);
                    f[DK] = exp2f(tot - Gs[b] - mu[b]);
                    if constexpr (UB) {
                        if (b < 3) {
                            f[2 * DK] = exp2f(mu[b]);
                            const float gs_next = Gs[b] + 2.f * mu[b];   // Gs[b + 1]
#pragma unroll
                            for (int bt = b + 1; bt < 4; ++bt) f[(2 + bt - b) * DK] = exp2f(Gs[bt] - gs_next + mu[bt]);
                        }
                    } else {   // one step: 2^-H times 2^(Gs[bt] - Gs[b]) (at least 2^-115)
#pragma unroll
                        for (int bt = b + 1; bt < 4; ++bt) f[(2 + bt - b) * DK] = exp2f(Gs[bt] - Gs[b]);
                    }
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

            // Operands (H here is the block-local decay minus mu).  G1 (bf16, raw q/k times
            // block-local decay): Kp = k 2^H and Qp = q 2^H at rows 32 blk + r and
            // 32 blk + 16 + r of [Kp; Qp]; key variants at row variant_off(bt) + t:
            // k 2^-H for bt = blk, k 2^(Gs[bt] - G + mu[bt]) for bt > blk.  Chain (fp16, in
            // place of the raw tiles): Q_hat*Gamma, K_hat*Gamma and Kbar = k_hat 2^(G_C - G).
            {
                const int fb = pool_fac_base(blk);
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
                    const float rq = sm.rq[m % 3][t], rk = sm.rk[m % 3][t];
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
                    if (UB && blk < 3) {   // 2^(mu - H) -> 2^(Gs[blk+1] - G), at most 1 (before the variants)
                        const float4 *m4 = reinterpret_cast<const float4 *>(&sm.fac[fb + 2][c0]);
                        const float4 ma = m4[0], mb = m4[1];
                        kn[0] = mul2(kn[0], make_float2(ma.x, ma.y));
                        kn[1] = mul2(kn[1], make_float2(ma.z, ma.w));
                        kn[2] = mul2(kn[2], make_float2(mb.x, mb.y));
                        kn[3] = mul2(kn[3], make_float2(mb.z, mb.w));
                    }
#pragma unroll 1
                    for (int bt = blk + 1; bt < 4; ++bt) {
                        const float4 *d4 = reinterpret_cast<const float4 *>(&sm.fac[fb + 2 + bt - blk][c0]);
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

            if (tid == kProLead) mbar_arrive(&sm.pdone[m % 3]);   // operands and rq/rk/beta of chunk m ready
        }
    } else if (tid >= kHelp0 && tid < kHelp0 + NH) {
        // ------------------------------------------------ helper group
        // Row norms (one thread per row of q or k) and beta, beside the prologue's gate;
        // published to the prologue by the barrier that ends its gate step.
        const int htid = tid - kHelp0;
        auto load_logit = [&](const TaskIt &t) {
            return htid < t.L ? __bfloat162float(p.beta[(t.row + htid) * p.H + t.h]) : 0.f;
        };
        TaskIt it, nx;
        it.start(f, a, units, p);
        nx = it;
        nx.advance(p);
        // the gate parameters of task t into slot ps (read by the prologue after the
        // first barrier of that task)
        auto stage_gate = [&](const TaskIt &t, int ps) {
            if constexpr (UB) {   // softplus argument bias (log2 units) and the rate -exp(A_log)
                const float a = -__expf(p.A_log[t.h]);
                for (int cch = htid; cch < DK; cch += NH) sm.gb[ps][cch] = kLog2e * p.dt_bias[t.h * DK + cch];
                if (htid == 0) sm.ga[ps] = a;
            } else {
                const float a2 = -__expf(p.A_log[t.h]) * kLog2e;
                for (int cch = htid; cch < DK; cch += NH) sm.gb[ps][cch] = a2 * p.dt_bias[t.h * DK + cch];
                if (htid == 0) sm.ga[ps] = a2;
            }
        };
        float nb = 0.f;   // logit of token htid, loaded one task ahead
        if (it.valid()) {
            if (htid < C) nb = load_logit(it);
            stage_gate(it, 0);
        }
        for (int m = 0; it.valid(); ++m, it.advance(p), nx.advance(p)) {
            const int s = m & 1;
            const int L = it.L;
            const uint32_t rq_off = F_RAW + s * F_SLOT, rk_off = rq_off + 16384;
            named_bar(1, NP + NH);
            if (sm.dec_p) break;
            if (nx.valid()) stage_gate(nx, s ^ 1);
            const float bl = nb;
            if (htid < C && nx.valid()) nb = load_logit(nx);
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
                if (i & 1) sm.rk[m % 3][t] = r;
                else sm.rq[m % 3][t] = r;
            }
            if (htid < C) sm.beta[m % 3][htid] = htid < L ? 1.f / (1.f + exp2f(-bl * kLog2e)) : 0.f;
            named_bar(1, NP + NH);
        }
    } else if (warp == 12) {
        // ------------------------------------------------ control warp (lane 0)
        if (lane == 0) {
            TaskIt it, ahead, nx;
            it.start(f, a, units, p);
            ahead = it;
            nx = it;
            nx.advance(p);
            unsigned long long fv = 0;   // this task's ring-slot "freed" flag, read ahead
            if (it.valid() && it.j >= a.depth) fv = ld_acquire_gpu(a.freed(it.c, it.j));
            int issued = 0;   // raw tile loads requested
            if (ahead.valid()) { issue_raw(0, ahead); ++issued; }
            ahead.advance(p);
            if (ahead.valid()) { issue_raw(1, ahead); ++issued; }
            ahead.advance(p);
            int m = 0;
            for (; it.valid(); ++m, it.advance(p), ahead.advance(p), nx.advance(p)) {
                const int s = m & 1;
                bool ok = mbar_wait(&sm.pdone[m % 3], (m / 3) & 1, kWait);
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
                // Kbar, Q_hat*Gamma, K_hat*Gamma and exp(G_C) of the task go to its ring slot
                // once the chain has loaded the packet that slot held before (its "freed"
                // flag was read one task ahead, so that the load latency is hidden)
                if (ok && it.j >= a.depth && fv != a.tag(it.j - a.depth))
                    ok = wait_flag(a.freed(it.c, it.j), a.tag(it.j - a.depth), kWait);
                fv = 0;
                if (nx.valid() && nx.j >= a.depth) fv = ld_acquire_gpu(a.freed(nx.c, nx.j));
                if (ok) {
                    const uint32_t rq_off = F_RAW + s * F_SLOT, rk_off = rq_off + 16384, rg_off = rq_off + 32768;
                    unsigned char *slot = a.slot(it.c, it.j);
                    fence_proxy_async_global();
                    bulk_store(slot + RS_KB, smem + rg_off, 16384);
                    bulk_store(slot + RS_QG, smem + rq_off, 16384);
                    bulk_store(slot + RS_KG, smem + rk_off, 16384);
                    bulk_store(slot + RS_GC, &sm.gamC_f[s][0], 512);
                    bulk_commit();
                    bulk_wait_read0();   // raw tiles and exp(G_C) of slot s may be overwritten
                    if (ahead.valid()) { issue_raw(m + 2, ahead); ++issued; }
                    bulk_wait0();        // the stores are complete in global memory
                    fence_proxy_async_global();
                    st_release_cta(&sm.ctl_count, (unsigned)(m + 1));
                }
                if (!ok) {
                    set_err(p);
                    sm.abort_p = 1;
                    sm.abort_s = 1;
                    break;
                }
            }
            bulk_wait0();
            // after an abort, raw loads of tasks nobody processes may be in flight: no copy
            // into this CTA's shared memory may outlive it (bounded waits)
            for (int k = m; k < issued; ++k) mbar_wait(&sm.raw_full[k & 1], (k >> 1) & 1, kWait);
        }
    } else {
        // ------------------------------------------------ solver group
        // Warp sw reads TMEM lane quarter sw of G1 = rows of token block sw: lanes 0-15
        // are A rows (Kp), lanes 16-31 M rows (Qp); it needs the sw + 1 chunks of 16
        // columns of variant sw.
        const int stid = tid - NP, sw = warp - 8;
        float *Amat = reinterpret_cast<float *>(smem + F_AMAT);
        float *Tf = reinterpret_cast<float *>(smem + F_TF);
        // the M staging tile above the diagonal blocks stays zero for the whole run
        for (int k16 = stid; k16 < 512; k16 += NS) sts128(sbase + F_MST + k16 * 16, 0u, 0u, 0u, 0u);
        // T above its diagonal blocks is never written: zero once, so T' needs no mask
        for (int k4 = stid; k4 < 64 * LDA / 4; k4 += NS)
            reinterpret_cast<float4 *>(Tf)[k4] = make_float4(0.f, 0.f, 0.f, 0.f);
        named_bar(2, NS);
        unsigned long long *pub_flag = nullptr, pub_tag = 0;   // the lead's packet awaiting publication
        bool rbad = false;   // a T' or M value beyond the fp16 range
        TaskIt it;
        it.start(f, a, units, p);
        for (int m = 0; it.valid(); ++m, it.advance(p)) {
            const int s = m & 1;
            if (stid == kSolLead) {
                bulk_wait_read0();   // the previous T'/M staging is shipped
                if (!mbar_wait(&sm.pdone[m % 3], (m / 3) & 1, kWait) ||
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
                const float rowf = is_m ? sm.rq[m % 3][t] : sm.beta[m % 3][t] * sm.rk[m % 3][t];
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
                    const float4 *rk4 = reinterpret_cast<const float4 *>(&sm.rk[m % 3][16 * kk]);
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
                const float4 *b4 = reinterpret_cast<const float4 *>(&sm.beta[m % 3][i0]);
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
                mbar_arrive(&sm.s_done[m % 3]);
                // The previous packet is published first: its T'/M stores were issued a
                // task ago and the control warp's stores of it were complete before them,
                // so this costs no wait, and a publication never waits on a ring slot.
                if (pub_flag) {
                    bulk_wait0();
                    fence_proxy_async_global();
                    st_release_gpu(pub_flag, pub_tag);
                    pub_flag = nullptr;
                }
                // T' and M complete the packet, once the control warp has stored the rest
                // (which also means the slot's earlier packet is out).  The packet is
                // published one task later, so that the solver does not wait for the
                // completion of its stores here.
                bool ok = true;
                if (ld_acquire_cta(&sm.ctl_count) <= (unsigned)m) {
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_cta(&sm.ctl_count) <= (unsigned)m)
                        if (globaltimer_ns() - t0 > kWait || *(volatile int *)&sm.abort_s) { ok = false; break; }
                }
                if (ok) {
                    unsigned char *slot = a.slot(it.c, it.j);
                    bulk_store(slot + RS_TP, smem + F_AMAT, 8192);
                    bulk_store(slot + RS_MM, smem + F_MST, 8192);
                    bulk_commit();
                    pub_flag = a.ready(it.c, it.j);
                    pub_tag = a.tag(it.j);
                } else {
                    set_err(p);
                    sm.abort_s = 1;
                    sm.abort_p = 1;
                }
            }
        }
        flag_range(p, rbad);
        if (stid == kSolLead) {
            bulk_wait0();
            if (pub_flag && !sm.abort_s) {
                fence_proxy_async_global();
                st_release_gpu(pub_flag, pub_tag);
            }
        }
    }
}

// ============================================================== chain CTA
// Chain c runs units c, c + nc, ...; its packets j = 0, 1, ... are chunk j % nchunks of
// unit c + (j / nchunks) nc, in that order.
//
// The accumulators the sequential path reads out span all 128 TMEM lanes (one lane per
// value column v, or per key channel c), so four warps on four schedulers read them:
//   G2w: W^T    = (K_hat*Gamma)^T T'^T            [c x t]  (one packet ahead)
//   G2u: U^T    = V^T T'^T                        [v x t]  (one packet ahead)
//   G3u: U^T   += S^T (-W^T)                      [v x t]  (needs S of this chunk)
//   G4 : S     += Kbar^T U                        [c x v]  (S pre-scaled by Gamma_C)
//   G3o: O      = (Q_hat*Gamma) S                 [t x v]  (A rows 64-127; lanes 64-127)
//   G5 : O     += M U                             [t x v]
// The sequential path per chunk is G3u -> U readout -> G4 -> S readout; the MMA warp
// issues G2w of the next packet between G3u and G4, and G3o, G5 and the next G2u after G4.
// Roles (warp w reaches TMEM lanes 32 (w % 4) ..): warps 0-7 the state (S readout to
// its fp16 operand copy, decay by the next Gamma_C, initial and final state) and the
// conversion of the next V to fp16, 8-11 the U and -W^T readouts, 12 the loader (ring
// packets, V), 13 the MMA issuer, 14-15 the O readout (token rows, 16-byte stores).
// With a second state (DUAL; state-only runs of the sequence-parallel path) there is no
// O: G3o, G5 and the O readout drop out, and a second state S_2 with values of zero runs
// beside S on the same packets (G3u: U_2^T = S_2^T (-W^T); G4: S_2 += Kbar^T U_2), its
// accumulators in the O columns and its operand copies in the shared memory that the
// packets' Q_hat*Gamma and M parts leave free.
template <bool VL, bool DUAL>
__device__ __forceinline__ void pool_chain(const TmaMaps &maps, const Params &p, const PoolArgs &a,
                                           unsigned char *smem, ChainSmall &cs, uint32_t tmem, int c) {
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;
    // TMEM columns: S, W^T, two U^T buffers, then O, or (second state) S_2 and U_2^T
    const uint32_t D_S = tmem, D_W = tmem + 128, D_U0 = tmem + 192, D_O = tmem + 320;
    const uint32_t D_S2 = tmem + 320, D_U2 = tmem + 448;
    constexpr uint32_t O_PK = DUAL ? C2_PK : C_PK, O_SLOT = DUAL ? C2_PKSLOT : C_PKSLOT;
    constexpr uint32_t O_KB = DUAL ? P2_KB : PK_KB, O_KG = DUAL ? P2_KG : PK_KG, O_TP = DUAL ? P2_TP : PK_TP;
    const int nchunks = a.nchunks;
    const int64_t units = p.n_seqs * p.H;
    const int64_t nunits = VL ? 0 : (units - c + a.nc - 1) / a.nc;
    const int64_t npk = VL ? (int64_t)a.chain_len[c] : nunits * nchunks;   // this chain's packets
    auto pk_unit = [&](int64_t j) { return (int64_t)c + (j / nchunks) * a.nc; };
    auto pk_row = [&](int64_t j) {   // first token row of packet j in the [B*T] token rows
        return (pk_unit(j) / p.H) * p.T + (j % nchunks) * (int64_t)C;
    };
    auto pk_slot = [&](int64_t j) { return sbase + O_PK + (uint32_t)(j & 1) * O_SLOT; };
    auto par2 = [](int64_t j) { return (uint32_t)((j >> 1) & 1); };   // phase of a [j & 1] barrier
    auto par1 = [](int64_t j) { return (uint32_t)(j & 1); };          // phase of a per-packet barrier
    // bounded wait that also gives up once another role has aborted
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar, parity)) {
            if (*(volatile int *)&cs.abort) return false;
            if (globaltimer_ns() - t0 > kWait) {
                set_err(p);
                *(volatile int *)&cs.abort = 1;
                return false;
            }
        }
        return true;
    };
    auto warp_arrive = [&](uint64_t *bar) {   // one arrival per warp, after all its lanes
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
    };

    if (warp == kLoaderWarp) {
        // ------------------------------------------------ loader: V and the ring packets
        // Three tracks, advanced by one thread in whatever order their conditions allow:
        //   early(je)  K_hat*Gamma, T' of a published packet into slot je & 1 once G2u of
        //              packet je - 2 is done (u_done);
        //   late(jl)   Kbar, Q_hat*Gamma, M, exp(G_C) once G5 of packet jl - 2 is done (o_done);
        //   release(jr) the ring slot of packet jr once both of its parts have landed.
        if (lane != 0) return;
        int64_t je = 0, jl = 0, jr = 0;
        bool ready_je = false;   // packet je seen published
        [&]() {
            uint64_t t0 = globaltimer_ns();
            while (jr < npk) {
                bool progress = false;
                if (*(volatile int *)&cs.abort) return;
                if (je < npk && je < jr + 2 && (je < 2 || mbar_try_wait(&cs.u_done[je & 1], par2(je - 2)))) {
                    if (!ready_je) ready_je = ld_acquire_gpu(a.ready(c, je)) == a.tag(je);
                    if (ready_je) {
                        fence_proxy_async_global();
                        const unsigned char *slot = a.slot(c, je);
                        const uint32_t dst = pk_slot(je), fb = smem_u32(&cs.full_e[je & 1]);
                        mbar_arrive_expect_tx(&cs.full_e[je & 1], 16384 + 8192);
                        bulk_load(dst + O_KG, slot + RS_KG, 16384, fb);
                        bulk_load(dst + O_TP, slot + RS_TP, 8192, fb);
                        ++je;
                        ready_je = false;
                        progress = true;
                    }
                }
                if (jl < je && (jl < 2 || mbar_try_wait(&cs.o_done[jl & 1], par2(jl - 2)))) {
                    const unsigned char *slot = a.slot(c, jl);
                    const uint32_t dst = pk_slot(jl), fb = smem_u32(&cs.full_l[jl & 1]);
                    if constexpr (DUAL) {   // no O: Kbar and exp(G_C) only
                        mbar_arrive_expect_tx(&cs.full_l[jl & 1], 16384 + 512);
                        bulk_load(dst + O_KB, slot + RS_KB, 16384, fb);
                    } else {
                        mbar_arrive_expect_tx(&cs.full_l[jl & 1], 16384 * 2 + 8192 + 512);
                        bulk_load(dst + PK_KB, slot + RS_KB, 16384, fb);
                        bulk_load(dst + PK_QG, slot + RS_QG, 16384, fb);
                        bulk_load(dst + PK_MM, slot + RS_MM, 8192, fb);
                    }
                    bulk_load(smem_u32(&cs.gamC[jl & 1][0]), slot + RS_GC, 512, fb);
                    ++jl;
                    progress = true;
                }
                if (jr < jl && mbar_try_wait(&cs.full_e[jr & 1], par2(jr)) &&
                    mbar_try_wait(&cs.full_l[jr & 1], par2(jr))) {
                    fence_proxy_async_global();
                    st_release_gpu(a.freed(c, jr), a.tag(jr));
                    ++jr;
                    progress = true;
                }
                if (progress) {
                    t0 = globaltimer_ns();
                } else if (globaltimer_ns() - t0 > kWait) {
                    set_err(p);
                    *(volatile int *)&cs.abort = 1;
                    return;
                }
            }
        }();
        // no copy into this CTA's shared memory may outlive it: wait (bounded) for the
        // last ones requested (release waited for every part up to jr)
        for (int64_t k = jr; k < je; ++k) mbar_wait(&cs.full_e[k & 1], par2(k), kWait);
        for (int64_t k = jr; k < jl; ++k) mbar_wait(&cs.full_l[k & 1], par2(k), kWait);
        return;
    }

    if (warp == 13) {
        // ------------------------------------------------ MMA issuer
        if (lane != 0) return;
        [&]() {
            const uint32_t id_n64_mk = idesc_fp16(128, 64, true, false);    // A MN-major, B K-major
            const uint32_t id_n64_mm = idesc_fp16(128, 64, true, true);     // A MN-major, B MN-major
            const uint32_t id_n128_mk = idesc_fp16(128, 128, true, false);  // A MN-major, B K-major
            const uint32_t id_n128_km = idesc_fp16(128, 128, false, true);  // A K-major, B MN-major
            const uint32_t id_n128_kk = idesc_fp16(128, 128, false, false); // A K-major, B K-major
            const uint64_t dSH = sdesc_sw128(sbase + C_SH, 16384, 1024);    // S^T, A MN-major
            const uint64_t dWT = sdesc_sw128(sbase + C_WT, 16384, 1024);    // -W^T, B MN-major
            const uint64_t dUH = sdesc_sw128(sbase + C_UH, 16, 1024);       // U^T as A / U as B, K-major
            const uint64_t dSH2 = sdesc_sw128(sbase + C2_SHP, 16384, 1024);  // second state's S^T
            const uint64_t dUH2 = sdesc_sw128(sbase + C2_UHP, 16, 1024);     // second state's U
            auto issue_g2w = [&](int64_t jn) {   // G2w of packet jn
                const uint32_t pk = pk_slot(jn);
                const uint64_t dKG = sdesc_sw128(pk + O_KG, 8192, 1024);
                const uint64_t dTP = sdesc_sw128(pk + O_TP, 16, 1024);
                tc_fence_after();
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_bf16(D_W, dKG + (uint64_t)(ks * 128), dTP + (uint64_t)(ks * 2), id_n64_mk, ks > 0);
                mma_commit(&cs.w_done);
            };
            auto issue_g2u = [&](int64_t jn) {   // G2u of packet jn, once its V is fp16
                const uint64_t dTP = sdesc_sw128(pk_slot(jn) + O_TP, 16, 1024);
                const uint64_t dV = sdesc_sw128(sbase + C_V + (uint32_t)(jn & 1) * 16384, 8192, 1024);
                if (!wait(&cs.vconv[jn & 1], par2(jn))) return false;
                tc_fence_after();
                const uint32_t du = D_U0 + (uint32_t)(jn & 1) * 64;
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_bf16(du, dV + (uint64_t)(ks * 128), dTP + (uint64_t)(ks * 2), id_n64_mk, ks > 0);
                return true;
            };
            if (npk > 0) {
                if (!wait(&cs.full_e[0], 0)) return;
                issue_g2w(0);
                if (!issue_g2u(0)) return;
            }
            for (int64_t j = 0; j < npk; ++j) {
                const int sj = (int)(j & 1);
                const uint32_t pk = pk_slot(j);
                const uint32_t du = D_U0 + (uint32_t)sj * 64;
                // G3u: U^T += S^T (-W^T)
                if (!wait(&cs.sh_ready, par1(j)) || !wait(&cs.wt_ready, par1(j))) return;
                tc_fence_after();
                for (int ks = 0; ks < DK / 16; ++ks)
                    mma_bf16(du, dSH + (uint64_t)(ks * 128), dWT + (uint64_t)(ks * 128), id_n64_mm, true);
                mma_commit(&cs.u_done[sj]);
                if constexpr (DUAL) {
                    // the second state, values of zero: U_2^T = S_2^T (-W^T)
                    for (int ks = 0; ks < DK / 16; ++ks)
                        mma_bf16(D_U2, dSH2 + (uint64_t)(ks * 128), dWT + (uint64_t)(ks * 128), id_n64_mm, ks > 0);
                    mma_commit(&cs.up_done);
                    // G4 on both states: S += Kbar^T U
                    if (!wait(&cs.full_l[sj], par2(j)) || !wait(&cs.uh_ready, par1(j)) ||
                        !wait(&cs.s_scaled, par1(j)))
                        return;
                    tc_fence_after();
                    const uint64_t dKB = sdesc_sw128(pk + O_KB, 8192, 1024);
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_bf16(D_S, dKB + (uint64_t)(ks * 128), dUH + (uint64_t)(ks * 2), id_n128_mk, true);
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_bf16(D_S2, dKB + (uint64_t)(ks * 128), dUH2 + (uint64_t)(ks * 2), id_n128_mk, true);
                    mma_commit(&cs.s_done);
                    mma_commit(&cs.o_done[sj]);   // the packet's late part is consumed
                    if (j + 1 < npk) {
                        if (!wait(&cs.full_e[sj ^ 1], par2(j + 1))) return;
                        issue_g2w(j + 1);
                        if (!issue_g2u(j + 1)) return;
                    }
                    continue;
                }
                // G2w of the next packet right behind G3u when its operands are in (D_W
                // was read out before G3u), so that its readout overlaps this chunk's
                const bool more = j + 1 < npk;
                bool g2w_early = false;
                if (more && mbar_try_wait(&cs.full_e[sj ^ 1], par2(j + 1))) {
                    issue_g2w(j + 1);
                    g2w_early = true;
                }
                // G3o: O = (Q_hat Gamma) S into lanes 64-127 (the A operand starts 64 rows
                // before Q_hat Gamma; rows 0-63 of O are unused), right behind G3u, so that
                // the S copy is free again when G4 completes
                if (!wait(&cs.full_l[sj], par2(j))) return;
                if (j >= 1 && !wait(&cs.o_free, par1(j - 1))) return;
                tc_fence_after();
                {
                    const uint64_t dQG = sdesc_sw128(pk + PK_QG - 8192, 16, 1024);
                    for (int ks = 0; ks < DK / 16; ++ks)
                        mma_bf16(D_O, dQG + (uint64_t)((ks >> 2) * 512 + (ks & 3) * 2), dSH + (uint64_t)(ks * 128),
                                 id_n128_km, ks > 0);
                }
                // G4: S += Kbar^T U
                if (!wait(&cs.uh_ready, par1(j)) || !wait(&cs.s_scaled, par1(j))) return;
                tc_fence_after();
                {
                    const uint64_t dKB = sdesc_sw128(pk + PK_KB, 8192, 1024);
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_bf16(D_S, dKB + (uint64_t)(ks * 128), dUH + (uint64_t)(ks * 2), id_n128_mk, true);
                    mma_commit(&cs.s_done);
                }
                // otherwise G2w of the next packet here, so that its readout runs beside the
                // S readout
                if (more && !g2w_early) {
                    if (!wait(&cs.full_e[sj ^ 1], par2(j + 1))) return;
                    issue_g2w(j + 1);
                }
                // G5: O += M U
                {
                    const uint64_t dMM = sdesc_sw128(pk + PK_MM - 8192, 16, 1024);
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_bf16(D_O, dMM + (uint64_t)(ks * 2), dUH + (uint64_t)(ks * 2), id_n128_kk, true);
                    mma_commit(&cs.o_done[sj]);
                }
                // G2u of the next packet (U^T buffer (j + 1) & 1 was read out for packet j - 1)
                if (more && !issue_g2u(j + 1)) return;
            }
        }();
        // every MMA issued here completes before the CTA releases its tensor memory
        mma_commit(&cs.fin);
        mbar_wait(&cs.fin, 0, kWait);
        return;
    }

    if (warp >= 14) {
        // ------------------------------------------------ O readout: token rows (TMEM lanes 64-127)
        if constexpr (DUAL) return;   // state-only: no O
        const int t = (quarter - 2) * 32 + lane;   // token of the chunk
        PkWalkV ow;   // varlen: this packet's unit
        if (VL) ow.start(p, a, c);
        for (int64_t j = 0; j < npk; ++j, VL ? ow.next(p, a) : void()) {
            if (!wait(&cs.o_done[j & 1], par2(j))) return;
            tc_fence_after();
            uint32_t pk0[32];   // columns 0-63 as bf16 pairs
            float r[4][16];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) tmem_ld16(tmem_addr(D_O, quarter * 32, 16 * jj), r[jj]);
            tmem_ld_wait();
            const float sc = p.scale;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int e = 0; e < 8; ++e) pk0[8 * jj + e] = pack_bf16(sc * r[jj][2 * e], sc * r[jj][2 * e + 1]);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) tmem_ld16(tmem_addr(D_O, quarter * 32, 64 + 16 * jj), r[jj]);
            tmem_ld_wait();
            tc_fence_before();
            warp_arrive(&cs.o_free);
            int rows;
            if constexpr (VL) {
                rows = ow.rows();
            } else {
                const int rem = (int)(p.T - (j % nchunks) * (int64_t)C);
                rows = rem < C ? rem : C;
            }
            if (p.out && t < rows) {
                int64_t orow, oh;
                if constexpr (VL) {
                    orow = ow.row();
                    oh = ow.u.h;
                } else {
                    const int64_t u = pk_unit(j);
                    orow = pk_row(j);
                    oh = u % p.H;
                }
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((orow + t) * p.H + oh) * DK);
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8)
                    dst[q8] = make_uint4(pk0[4 * q8], pk0[4 * q8 + 1], pk0[4 * q8 + 2], pk0[4 * q8 + 3]);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    dst[8 + 2 * jj] = make_uint4(pack_bf16(sc * r[jj][0], sc * r[jj][1]), pack_bf16(sc * r[jj][2], sc * r[jj][3]),
                                                 pack_bf16(sc * r[jj][4], sc * r[jj][5]), pack_bf16(sc * r[jj][6], sc * r[jj][7]));
                    dst[9 + 2 * jj] = make_uint4(pack_bf16(sc * r[jj][8], sc * r[jj][9]), pack_bf16(sc * r[jj][10], sc * r[jj][11]),
                                                 pack_bf16(sc * r[jj][12], sc * r[jj][13]), pack_bf16(sc * r[jj][14], sc * r[jj][15]));
                }
            }
        }
        return;
    }

    if (warp >= 8) {
        // ------------------------------------------------ U and -W^T readouts (lane quarter)
        const int lv = quarter * 32 + lane;   // this thread's TMEM lane: v for U, c for W
        bool rbad = false;                    // a V, U or W value beyond the fp16 range
        auto read64 = [&](uint32_t col, float (&r)[4][16]) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) tmem_ld16(tmem_addr(col, quarter * 32, 16 * jj), r[jj]);
            tmem_ld_wait();
        };
        auto w_readout = [&](int64_t jw) -> bool {   // -W^T of packet jw
            if (!wait(&cs.w_done, par1(jw))) return false;
            tc_fence_after();
            float r[4][16];
            read64(D_W, r);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
                for (int e = 0; e < 16; ++e) r[jj][e] = -r[jj][e];
                st_pack16<true>(sbase + C_WT, lv, 16 * jj, r[jj], rbad);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(&cs.wt_ready);
            return true;
        };
        // V of packet jv into V buffer jv & 1 (warp 8, lane 0), free once G2u of packet
        // jv - 2 is done
        int64_t v_issued = 0;
        PkWalkV vw;   // varlen: the unit of the next V to load (issued in packet order)
        if (VL && warp == 8 && lane == 0) vw.start(p, a, c);
        auto issue_v = [&](int64_t jv) {
            const int sv = (int)(jv & 1);
            int row, h;
            if (VL) {
                row = (int)vw.row();
                h = vw.u.h;
                vw.next(p, a);
            } else {
                row = (int)pk_row(jv);
                h = (int)(pk_unit(jv) % p.H);
            }
            if (p.v) {
                unsigned char *vb = smem + C_V + sv * 16384;
                mbar_arrive_expect_tx(&cs.vfull[sv], 16384);
                tma_load_3d(vb, &maps.v, &cs.vfull[sv], 0, h, row);
                tma_load_3d(vb + 8192, &maps.v, &cs.vfull[sv], 64, h, row);
            } else {
                mbar_arrive(&cs.vfull[sv]);   // values of zero: the buffer stays zero
            }
            v_issued = jv + 1;
        };
        const bool vlead = warp == 8 && lane == 0;
        [&]() {
        if (vlead) {
            if (npk > 0) issue_v(0);
            if (npk > 1) issue_v(1);
        }
        if (npk > 0 && !w_readout(0)) return;
        for (int64_t j = 0; j < npk; ++j) {
            const int sj = (int)(j & 1);
            // U^T -> fp16 rows of U^T (K-major)
            if (!wait(&cs.u_done[sj], par2(j))) return;
            // G2u of packet j is done: V of packet j + 2 may land in its buffer
            if (vlead && j + 2 < npk) issue_v(j + 2);
            tc_fence_after();
            {
                float r[4][16];
                read64(D_U0 + (uint32_t)sj * 64, r);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) st_pack16<true>(sbase + C_UH, lv, 16 * jj, r[jj], rbad);
                if constexpr (DUAL) {   // and the second state's
                    if (!wait(&cs.up_done, par1(j))) return;
                    tc_fence_after();
                    read64(D_U2, r);
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) st_pack16<true>(sbase + C2_UHP, lv, 16 * jj, r[jj], rbad);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(&cs.uh_ready);
            if (j + 1 < npk && !w_readout(j + 1)) return;
        }
        }();
        flag_range(p, rbad);
        // no V copy into this CTA's shared memory may outlive it (bounded waits)
        if (vlead)
            for (int64_t k = v_issued - 2; k < v_issued; ++k)
                if (k >= 0) mbar_wait(&cs.vfull[k & 1], par2(k), kWait);
        return;
    }

    // ------------------------------------------------ state warps 0-7 (lane quarter, column half)
    const int half = warp >> 2;
    const int cc = quarter * 32 + lane;   // key channel (TMEM lane of D_S)
    auto ld_s = [&](float (&r)[4][16], uint32_t col) {   // this warp's part of S (col D_S) or S_2
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) tmem_ld16(tmem_addr(col, quarter * 32, 64 * half + 16 * jj), r[jj]);
        tmem_ld_wait();
    };
    bool rbad = false;   // a state (or V) value beyond the fp16 range of its operand copy
    // V of packet jv to fp16, in place (the 256 threads of warps 0-7, while their state
    // waits for G4)
    auto convert_v = [&](int64_t jv) -> bool {
        const int sv = (int)(jv & 1);
        if (!wait(&cs.vfull[sv], par2(jv))) return false;
        for (int k16 = tid; k16 < 1024; k16 += 256) {
            uint4 *ptr = reinterpret_cast<uint4 *>(smem + C_V + sv * 16384 + k16 * 16);
            *ptr = bf16_to_f16x8(*ptr, rbad);
        }
        fence_proxy_async_smem();
        warp_arrive(&cs.vconv[sv]);
        return true;
    };
    if (!p.v) {
        // values of zero (a state-only run): both V buffers hold zeros for the whole run;
        // each thread clears the pieces it converts later (same index pattern)
        for (int sv = 0; sv < 2; ++sv)
            for (int k16 = tid; k16 < 1024; k16 += 256)
                *reinterpret_cast<uint4 *>(smem + C_V + sv * 16384 + k16 * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (npk > 0 && !convert_v(0)) return;
    int64_t j = 0;
    const int64_t U = VL ? (int64_t)a.counts[1] : 0;
    for (int64_t w = 0;; ++w) {
        // the chain's unit of round w: its state offset and chunk count
        size_t state_base;
        int nch;
        if constexpr (VL) {
            const UnitV u = unit_v(p, a, c, w, U);
            if (!u.valid) break;
            if (u.nch == 0) {
                // a sequence without tokens: its final state is its initial state
                if (p.fin) {
                    const int64_t n16 = (int64_t)DK * DK * (p.state_type == kStateBF16 ? 2 : 4) / 16;
                    const int64_t b16 = u.sbase * (p.state_type == kStateBF16 ? 2 : 4) / 16;
                    uint4 *dst = reinterpret_cast<uint4 *>(p.fin) + b16;
                    const uint4 *src = p.init ? reinterpret_cast<const uint4 *>(p.init) + b16 : nullptr;
                    for (int64_t e = tid; e < n16; e += 256) dst[e] = src ? src[e] : make_uint4(0u, 0u, 0u, 0u);
                }
                if (DUAL && p.fin2) {   // the second state (fp32) likewise
                    const int64_t n16 = (int64_t)DK * DK * 4 / 16, b16 = u.sbase * 4 / 16;
                    uint4 *dst = reinterpret_cast<uint4 *>(p.fin2) + b16;
                    const uint4 *src = p.init2 ? reinterpret_cast<const uint4 *>(p.init2) + b16 : nullptr;
                    for (int64_t e = tid; e < n16; e += 256) dst[e] = src ? src[e] : make_uint4(0u, 0u, 0u, 0u);
                }
                continue;
            }
            state_base = (size_t)u.sbase;
            nch = u.nch;
        } else {
            if (w >= nunits) break;
            const int64_t unit = (int64_t)c + w * a.nc;
            const int64_t h = unit % p.H, n = unit / p.H;
            state_base = (size_t)(n * p.H + h) * DK * DK;
            nch = nchunks;
        }
        // the unit's initial states (the previous unit's final states are out of TMEM)
        auto ld_init = [&](float (&r)[4][16], bool second) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const size_t off = state_base + (size_t)(64 * half + 16 * jj + e) * DK + cc;
                    float x = 0.f;
                    if (second) {
                        if (p.init2) x = p.init2[off];
                    } else if (p.init) {
                        x = p.state_type == kStateBF16
                                ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.init)[off])
                                : reinterpret_cast<const float *>(p.init)[off];
                    }
                    r[jj][e] = x;
                }
        };
        for (int m = 0; m < nch; ++m, ++j) {
            const int sj = (int)(j & 1);
            float r[4][16];
            if (m == 0) {
                ld_init(r, false);
            } else {
                if (!wait(&cs.s_done, par1(j - 1))) return;
                tc_fence_after();
                ld_s(r, D_S);
            }
            // the S^T operand of this chunk (G3o of the previous one, which read the last
            // copy, completed before G4 did)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) st_pack16<true>(sbase + C_SH + half * 16384, cc, 16 * jj, r[jj], rbad);
            if constexpr (DUAL) {   // and the second state's (r then holds S_2)
                if (m == 0) ld_init(r, true);
                else ld_s(r, D_S2);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) st_pack16<true>(sbase + C2_SHP + half * 16384, cc, 16 * jj, r[jj], rbad);
            }
            fence_proxy_async_smem();
            warp_arrive(&cs.sh_ready);
            // D_S = Diag(Gamma_C) S, the decayed state G4 accumulates onto
            if (!wait(&cs.full_l[sj], par2(j))) return;
            const float g = cs.gamC[sj][cc];
            if constexpr (DUAL) {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) r[jj][e] *= g;
                    tmem_st16(tmem_addr(D_S2, quarter * 32, 64 * half + 16 * jj), r[jj]);
                }
                if (m == 0) ld_init(r, false);   // the first state again
                else ld_s(r, D_S);
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
                for (int e = 0; e < 16; ++e) r[jj][e] *= g;
                tmem_st16(tmem_addr(D_S, quarter * 32, 64 * half + 16 * jj), r[jj]);
            }
            tmem_st_wait();
            tc_fence_before();
            warp_arrive(&cs.s_scaled);
            if (j + 1 < npk && !convert_v(j + 1)) return;
        }
        // final state from the fp32 master
        if (!wait(&cs.s_done, par1(j - 1))) return;
        tc_fence_after();
        if (p.fin) {
            float r[4][16];
            ld_s(r, D_S);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const size_t off = state_base + (size_t)(64 * half + 16 * jj + e) * DK + cc;
                    if (p.state_type == kStateBF16)
                        reinterpret_cast<__nv_bfloat16 *>(p.fin)[off] = __float2bfloat16(r[jj][e]);
                    else
                        reinterpret_cast<float *>(p.fin)[off] = r[jj][e];
                }
        }
        if (DUAL && p.fin2) {
            float r[4][16];
            ld_s(r, D_S2);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    p.fin2[state_base + (size_t)(64 * half + 16 * jj + e) * DK + cc] = r[jj][e];
        }
        tc_fence_before();
    }
    flag_range(p, rbad);
}

template <bool VL, bool UB, bool DUAL>
__global__ void __launch_bounds__(NT, 1)
kda_pool_kernel(const __grid_constant__ TmaMaps maps, Params p, PoolArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment (128B-swizzled tiles) by pointer arithmetic on the shared
    // array itself, so that every access through `smem` stays a shared-memory access
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint32_t *tmem_base = reinterpret_cast<uint32_t *>(smem + COMMON);
    const int cta = (int)blockIdx.x;
    const bool chain = cta < a.nc;
    FrontSmall &fs = *reinterpret_cast<FrontSmall *>(smem + F_SMALL);
    ChainSmall &cs = *reinterpret_cast<ChainSmall *>(smem + C_SMALL);

    if (threadIdx.x == 0) {
        if (chain) {
            for (int i = 0; i < 2; ++i) {
                mbar_init(&cs.full_e[i], 1);
                mbar_init(&cs.full_l[i], 1);
                mbar_init(&cs.vfull[i], 1);
                mbar_init(&cs.vconv[i], 8);     // the eight state warps
                mbar_init(&cs.u_done[i], 1);
                mbar_init(&cs.o_done[i], 1);
            }
            mbar_init(&cs.o_free, 2);           // the two O readout warps
            mbar_init(&cs.w_done, 1);
            mbar_init(&cs.s_done, 1);
            mbar_init(&cs.sh_ready, 8);         // the eight state warps
            mbar_init(&cs.s_scaled, 8);
            mbar_init(&cs.uh_ready, 4);
            mbar_init(&cs.wt_ready, 4);
            mbar_init(&cs.fin, 1);
            mbar_init(&cs.up_done, 1);
            cs.abort = 0;
        } else {
            for (int i = 0; i < 2; ++i) {
                mbar_init(&fs.raw_full[i], 1);
                mbar_init(&fs.g1_done[i], 1);
                mbar_init(&fs.am_free[i], 1);
            }
            fs.ctl_count = 0;
            for (int i = 0; i < 3; ++i) {
                mbar_init(&fs.s_done[i], 1);
                mbar_init(&fs.pdone[i], 1);
            }
            fs.abort_p = fs.abort_s = 0;
            fs.dec_p = fs.dec_s = 0;
        }
        fence_mbar_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base;

    if (chain)
        pool_chain<VL, DUAL>(maps, p, a, smem, cs, tmem, cta);
    else
        pool_front<VL, UB>(maps, p, a, smem, fs, tmem, cta - a.nc);

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- varlen plan
// One CTA.  (1) The sequences the pool takes (all of them, or in a mixed-length call
// those of more than kShortMaxT tokens), sorted by chunk count, longest first, ties by
// index (bitonic sort of 64-bit keys in shared memory).  (2) Their (sequence, head)
// units in that order, dealt to the chains in snake order; each chain's packet count.
// (3) The chains ranked by packet count; off[j] = sum over chains of min(count, j), the
// global index of the first packet of step j.  (4) The list of packets in global order:
// packet j of the chain of rank r has index off[j] + r.
constexpr int kPlanThreads = 1024;
constexpr int kMaxChains = 512;

__global__ void __launch_bounds__(kPlanThreads)
pool_plan_kernel(Params p, PoolArgs a, int *order, int *chain_len, int *counts, int *off, int4 *plist,
                 int npad) {
    __shared__ unsigned long long key[kPoolMaxSeqs];
    __shared__ int cl[kMaxChains], rk[kMaxChains];
    __shared__ int s_n, s_lmax;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int N = (int)p.n_seqs, nc = a.nc;
    const int64_t H = p.H;
    if (tid == 0) {
        s_n = 0;
        s_lmax = 0;
    }
    for (int n = tid; n < npad; n += kPlanThreads) {
        unsigned long long k = 0;   // zero: not the pool's (sorts last)
        if (n < N) {
            const int64_t len = p.cu_seqlens[n + 1] - p.cu_seqlens[n];
            if (!(p.mixed && len <= kShortMaxT))
                k = ((unsigned long long)((len + C - 1) / C) << 32) | (unsigned long long)(0xffffffffu - (unsigned)n);
        }
        key[n] = k;
    }
    __syncthreads();
    for (int size = 2; size <= npad; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = tid; t < npad / 2; t += kPlanThreads) {
                const int lo = 2 * t - (t & (stride - 1)), hi = lo + stride;
                const unsigned long long x = key[lo], y = key[hi];
                if ((x < y) == ((lo & size) == 0)) {   // descending where (lo & size) == 0
                    key[lo] = y;
                    key[hi] = x;
                }
            }
            __syncthreads();
        }
    for (int sq = tid; sq < npad; sq += kPlanThreads)
        if (key[sq] != 0 && (sq + 1 == npad || key[sq + 1] == 0)) s_n = sq + 1;
    for (int sq = tid; sq < N; sq += kPlanThreads)
        if (key[sq] != 0) order[sq] = (int)(0xffffffffu - (unsigned)(key[sq] & 0xffffffffu));
    __syncthreads();
    const int64_t U = (int64_t)s_n * H;
    if (tid < nc) {
        int64_t tot = 0;
        for (int64_t w = 0;; ++w) {
            const int64_t k = w * nc + ((w & 1) ? (nc - 1 - tid) : tid);
            if (k >= U) break;
            tot += (int64_t)(key[k / H] >> 32);
        }
        cl[tid] = (int)tot;
        chain_len[tid] = (int)tot;
        atomicMax(&s_lmax, (int)tot);
    }
    __syncthreads();
    if (tid < nc) {
        int r = 0;
        for (int d = 0; d < nc; ++d) r += cl[d] > cl[tid] || (cl[d] == cl[tid] && d < tid);
        rk[tid] = r;
    }
    const int lmax = s_lmax;
    for (int j = tid; j <= lmax; j += kPlanThreads) {
        int64_t o = 0;
        for (int d = 0; d < nc; ++d) o += cl[d] < j ? cl[d] : j;
        off[j] = (int)o;
    }
    if (tid == 0) {
        int64_t tot = 0;
        for (int d = 0; d < nc; ++d) tot += cl[d];
        counts[0] = (int)tot;
        counts[1] = (int)U;
    }
    __syncthreads();
    for (int c = warp; c < nc; c += kPlanThreads / 32) {
        int64_t j = 0;
        for (int64_t w = 0;; ++w) {
            const int64_t k = w * nc + ((w & 1) ? (nc - 1 - c) : c);
            if (k >= U) break;
            const int64_t sq = k / H;
            const int h = (int)(k - sq * H);
            const int n = (int)(0xffffffffu - (unsigned)(key[sq] & 0xffffffffu));
            const int64_t t0 = p.cu_seqlens[n];
            const int len = (int)(p.cu_seqlens[n + 1] - t0);
            const int nch = (len + C - 1) / C;
            for (int m = lane; m < nch; m += 32) {
                const int rows = len - m * C < C ? len - m * C : C;
                plist[off[j + m] + rk[c]] = make_int4(c, (int)(j + m), (int)(t0 + (int64_t)m * C), (h << 8) | rows);
            }
            j += nch;
        }
    }
}

}  // namespace

int64_t pool_chains(int64_t units, int sms) {
    // A chain runs its units one after another, about 7K cycles per chunk; the fronts
    // take every chunk of every unit, about 9.5K cycles each, on the SMs the chains
    // leave.  In units of one unit's chunk count the run takes about
    //   max(ceil(units / nc) * 7, units * 9.5 / (sms - nc)),
    // and nc (at most half the SMs) minimises it; on a tie, the fewer chains.
    int64_t cap = sms / 2;
    if (cap > units) cap = units;
    if (cap < 1) return 1;
    int64_t best = 1;
    double best_t = 0.0;
    for (int64_t nc = 1; nc <= cap; ++nc) {
        const double tc = (double)((units + nc - 1) / nc) * 14.0, tf = (double)units * 19.0 / (double)(sms - nc);
        const double t = tc > tf ? tc : tf;
        if (nc == 1 || t < best_t) {
            best = nc;
            best_t = t;
        }
    }
    return best;
}

// Workspace layout: the ring (nc x D packet slots), its flags (2 D words per chain), and
// for varlen calls the plan: order [N], chain_len [nc], counts [4], off [P + 1] and the
// packet list [P] (16-byte entries), P = H (ceil(T / 64) + N) bounding the packet count.
namespace {
struct PoolLayout {
    size_t flags, order, chain_len, counts, off, plist, total;
};
size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }
PoolLayout pool_layout(int64_t N, int64_t H, int64_t T, bool varlen, int sms) {
    const int64_t units = N * H;
    const int64_t nc = pool_chains(units, sms);
    const int64_t D = ring_depth(nc, sms - nc);
    PoolLayout l;
    l.flags = (size_t)nc * D * kChunkBytes;
    size_t x = l.flags + (size_t)nc * 2 * D * sizeof(unsigned long long);
    l.order = l.chain_len = l.counts = l.off = l.plist = 0;
    if (varlen) {
        const int64_t P = H * ((T + C - 1) / C + N);
        l.order = up256(x);
        l.chain_len = up256(l.order + 4 * (size_t)N);
        l.counts = up256(l.chain_len + 4 * (size_t)nc);
        l.off = up256(l.counts + 16);
        l.plist = up256(l.off + 4 * (size_t)(P + 1));
        x = l.plist + 16 * (size_t)P;
    }
    l.total = x;
    return l;
}
}  // namespace

size_t pool_scratch_bytes(const Params &p, int sms) {
    return pool_layout(p.n_seqs, p.H, p.T, p.cu_seqlens != nullptr, sms).total;
}
size_t pool_scratch_bytes_varlen(int64_t N, int64_t H, int64_t T, int sms) {
    return pool_layout(N, H, T, true, sms).total;
}

bool pool_takes(const Params &p, int sms) {
    if (!p.cu_seqlens) return true;
    const int64_t P = p.H * ((p.T + C - 1) / C + p.n_seqs);
    return p.n_seqs <= kPoolMaxSeqs && pool_chains(p.n_seqs * p.H, sms) <= kMaxChains && P < (int64_t(1) << 30) &&
           p.T < (int64_t(1) << 30) && p.H < (int64_t(1) << 22);
}

cudaError_t launch_pool(const Params &p, int sms, cudaStream_t stream, bool plan_ready) {
    const int64_t units = p.n_seqs * p.H;
    if (units == 0) return cudaSuccess;
    const int64_t nc = pool_chains(units, sms);
    const int64_t nf = sms - nc;
    const bool vl = p.cu_seqlens != nullptr;
    const int64_t nchunks = vl ? 0 : (p.T + C - 1) / C;
    if (nf < 1 || (!vl && nchunks < 1)) return cudaErrorInvalidValue;
    if (vl && !pool_takes(p, sms)) return cudaErrorInvalidValue;
    // a second state: varlen, state-only
    if (p.fin2 && (!vl || p.out)) return cudaErrorInvalidValue;
    const PoolLayout l = pool_layout(p.n_seqs, p.H, p.T, vl, sms);
    PoolArgs a = {};
    a.nc = (int)nc;
    a.nf = (int)nf;
    a.nchunks = (int)nchunks;
    a.waves = vl ? 0 : (int)((units + nc - 1) / nc);
    a.ring = p.ws;
    a.depth = (int)ring_depth(nc, nf);
    a.flags = reinterpret_cast<unsigned long long *>(p.ws + l.flags);
    if (vl) {
        a.order = reinterpret_cast<const int *>(p.ws + l.order);
        a.chain_len = reinterpret_cast<const int *>(p.ws + l.chain_len);
        a.counts = reinterpret_cast<const int *>(p.ws + l.counts);
        a.plist = reinterpret_cast<const int4 *>(p.ws + l.plist);
    }
    TmaMaps maps;
    const int64_t rows = p.B * p.T;
    if (!encode_map(&maps.q, p.q, rows, p.H) || !encode_map(&maps.k, p.k, rows, p.H) ||
        !encode_map(&maps.g, p.g, rows, p.H) || !encode_map(&maps.v, p.v, rows, p.H))
        return cudaErrorInvalidValue;
    static std::atomic<bool> attr_done[kMaxDevices];
    cudaError_t e = once_per_device(attr_done, [](int) {
        const int sb = (int)SMEM_BYTES;
        cudaError_t r = cudaFuncSetAttribute(kda_pool_kernel<false, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, sb);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(kda_pool_kernel<true, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, sb);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(kda_pool_kernel<false, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, sb);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(kda_pool_kernel<true, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, sb);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(kda_pool_kernel<true, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, sb);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(kda_pool_kernel<true, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, sb);
        return r;
    });
    if (e != cudaSuccess) return e;
    if (vl && !plan_ready) {
        int npad = 1;
        while (npad < p.n_seqs) npad <<= 1;
        pool_plan_kernel<<<1, kPlanThreads, 0, stream>>>(
            p, a, reinterpret_cast<int *>(p.ws + l.order), reinterpret_cast<int *>(p.ws + l.chain_len),
            reinterpret_cast<int *>(p.ws + l.counts), reinterpret_cast<int *>(p.ws + l.off),
            reinterpret_cast<int4 *>(p.ws + l.plist), npad < 2 ? 2 : npad);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nc + nf));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the flags of this call start at zero (no packet index + 1 is zero)
    e = cudaMemsetAsync(a.flags, 0, (size_t)nc * 2 * a.depth * sizeof(unsigned long long), stream);
    if (e != cudaSuccess) return e;
    if (p.fin2)
        e = p.unbounded ? cudaLaunchKernelEx(&cfg, kda_pool_kernel<true, true, true>, maps, p, a)
                        : cudaLaunchKernelEx(&cfg, kda_pool_kernel<true, false, true>, maps, p, a);
    else if (p.unbounded)
        e = vl ? cudaLaunchKernelEx(&cfg, kda_pool_kernel<true, true, false>, maps, p, a)
               : cudaLaunchKernelEx(&cfg, kda_pool_kernel<false, true, false>, maps, p, a);
    else
        e = vl ? cudaLaunchKernelEx(&cfg, kda_pool_kernel<true, false, false>, maps, p, a)
               : cudaLaunchKernelEx(&cfg, kda_pool_kernel<false, false, false>, maps, p, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kda
