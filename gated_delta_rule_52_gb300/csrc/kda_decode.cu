// KDA forward for decode (kda_fwd runs it for calls of one token row; it handles
// up to 16): the token recurrence applied directly, one token at a time, with
// the state held in registers.
//
// Per (sequence, head), with S the K x V state (FlashKDA README "Kernel API"
// semantics; the same activations as the chunked kernel):
//   S <- Diag(alpha_t) S;  u = beta_t (v_t - S^T k_hat_t);  S <- S + k_hat_t u^T;
//   out_t = scale * S^T q_hat_t
// which is S_t = (I - beta k k^T) Diag(alpha) S_{t-1} + beta k v^T written so that
// each state column needs only its own dot products.
//
// Work split: one CTA per (sequence, head, 32-column slice of V); 128 threads,
// thread = (quad of state columns, 8-row group of K), so each thread keeps 4 x 8
// fp32 state values in registers and reads only its own 8 rows of the per-token
// vectors (the decay factors, k_hat and q_hat, computed once per token into shared
// memory, one channel per thread).  The column sums over K (S^T k and S^T q)
// combine the 16 row groups by two shuffles inside each warp and through shared
// memory across the four warps.  (The first version gave each thread one column
// and 32 rows: every lane then read the same 32 rows of all three vectors per
// token, and the shared-memory load path was the bound.)  The state crosses
// HBM once in and once out per call, which bounds the kernel for short steps.
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

using namespace sm103;

constexpr int DK = kHeadDim;
constexpr int VS = 32;                // state columns per CTA
constexpr int NTD = 128;              // threads per CTA
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf(const __nv_bfloat16 *p, int64_t i) { return __bfloat162float(p[i]); }

// 16-byte asynchronous copy global -> shared (both 16-byte aligned)
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}

// Dynamic shared memory for a call of T token rows (T <= kDecodeMaxT):
//   tile   fp32 [32][128]  state slice staging; then the normalised k and q of every
//                          token ([T][128] each) while the tokens run
//   tin    bf16 [3][T][128] q, k, g of every token
//   tv     bf16 [T][32]     v, this slice
//   alf    fp32 [T][128]    decay factors
//   tb     fp32 [16]        beta logits, then beta
__host__ __device__ constexpr int decode_smem_bytes(int T) { return VS * DK * 4 + T * (3 * DK * 2 + VS * 2 + DK * 4) + 16 * 4; }

__global__ void __launch_bounds__(NTD, 6) kda_decode_kernel(Params p) {
    extern __shared__ __align__(16) unsigned char dsm[];
    __shared__ __align__(16) float red[2][4][VS];   // per-warp column sums: [0] S^T k, [1] S^T q
    __shared__ float rnq[kDecodeMaxT], rnk[kDecodeMaxT];
    const int Tm = (int)p.T;
    float *tile = reinterpret_cast<float *>(dsm);
    __nv_bfloat16 *tin = reinterpret_cast<__nv_bfloat16 *>(dsm + VS * DK * 4);   // [3][Tm][DK]
    __nv_bfloat16 *tv = tin + 3 * Tm * DK;                                       // [Tm][VS]
    float *alf = reinterpret_cast<float *>(tv + Tm * VS);                        // [Tm][DK]
    float *tb = alf + Tm * DK;                                                   // [16]
    float *knt = tile, *qnt = tile + Tm * DK;                                    // [Tm][DK] each
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t unit = blockIdx.x / (DK / VS);
    const int vs = blockIdx.x % (DK / VS);
    const int64_t h = unit % p.H, n = unit / p.H;
    int64_t b, t0, len;
    seq_range(p, n, b, t0, len);
    const int64_t row_base = b * p.T + t0;

    const int cq = lane & 7;            // columns 4 cq .. 4 cq + 3 of the slice
    const int rg = warp * 4 + (lane >> 3);   // rows 8 rg .. 8 rg + 7 of K
    const size_t state_base = (size_t)(n * p.H + h) * DK * DK;
    // Token inputs of the whole call (at most kDecodeMaxT tokens) into shared memory
    // with 16-byte asynchronous copies, issued before the state load so the two
    // latencies overlap; the token loop then reads only shared memory.
    for (int i = tid; i < (int)len * 48; i += NTD) {
        const int t = i / 48, j = i % 48, x = j >> 4, ch = j & 15;
        const __nv_bfloat16 *src = (x == 0 ? p.q : (x == 1 ? p.k : p.g)) + ((row_base + t) * p.H + h) * DK + 8 * ch;
        cp_async16(&tin[(x * Tm + t) * DK + 8 * ch], src);
    }
    for (int i = tid; i < (int)len * 4; i += NTD) {
        const int t = i >> 2, ch = i & 3;
        cp_async16(&tv[t * VS + 8 * ch], p.v + ((row_base + t) * p.H + h) * DK + vs * VS + 8 * ch);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (tid < len) tb[tid] = bf(p.beta, (row_base + tid) * p.H + h);

    // gate constants of this head for channel c = tid (log2 units)
    const float a2 = -__expf(p.A_log[h]) * kLog2e;
    const float b2 = a2 * p.dt_bias[h * DK + tid];
    const float lb2 = p.lower_bound * kLog2e;

    // The state slice (32 rows v of 128 fp32, 16 KB contiguous) moves between HBM and
    // the registers through a shared tile: global accesses are whole 512-byte rows per
    // warp instruction, and 16-byte chunk q of row v sits at chunk q ^ ((v / 4) & 7) of
    // the tile row, so both the row-wise copies and the per-thread reads (eight lanes
    // of a quarter-warp read eight rows 4 apart) are free of bank conflicts.
    // s[8 i + e] = S[row 8 rg + e][column 4 cq + i].
    float s[32];
    const size_t slice = state_base + (size_t)(vs * VS) * DK;   // first element of the slice
    auto tile_chunk = [&](int row, int q) -> float4 * {
        return reinterpret_cast<float4 *>(&tile[row * DK + 4 * (q ^ ((row >> 2) & 7))]);
    };
    if (p.init) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int row = warp * 8 + r;   // this warp's rows, lane = 16-byte chunk
            float4 x;
            if (p.state_type == kStateBF16) {
                const uint2 w = reinterpret_cast<const uint2 *>(
                    reinterpret_cast<const __nv_bfloat16 *>(p.init) + slice + (size_t)row * DK)[lane];
                x = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                                __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
            } else {
                x = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p.init) + slice +
                                                     (size_t)row * DK)[lane];
            }
            *tile_chunk(row, lane) = x;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int hq = 0; hq < 2; ++hq) {
                const float4 x = *tile_chunk(4 * cq + i, 2 * rg + hq);
                s[8 * i + 4 * hq] = x.x; s[8 * i + 4 * hq + 1] = x.y;
                s[8 * i + 4 * hq + 2] = x.z; s[8 * i + 4 * hq + 3] = x.w;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = 0.f;
    }

    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    // Activations of every token of the call, once: decay factors (thread = channel),
    // L2 norms (warp = token), then the normalised k and q over the dead state tile.
    for (int t = 0; t < (int)len; ++t) {
        const float gc = __bfloat162float(tin[(2 * Tm + t) * DK + tid]);
        alf[t * DK + tid] = exp2f(lb2 * __fdividef(1.f, 1.f + exp2f(fmaf(gc, a2, b2))));
    }
    for (int t = warp; t < (int)len; t += 4) {
        const uint2 qw = *reinterpret_cast<const uint2 *>(&tin[t * DK + 4 * lane]);
        const uint2 kw = *reinterpret_cast<const uint2 *>(&tin[(Tm + t) * DK + 4 * lane]);
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
            rnq[t] = rsqrtf(sq + 1e-6f);
            rnk[t] = rsqrtf(sk + 1e-6f);
        }
    }
    __syncthreads();   // norms ready; every thread is done with the initial-state tile
    for (int t = 0; t < (int)len; ++t) {
        knt[t * DK + tid] = __bfloat162float(tin[(Tm + t) * DK + tid]) * rnk[t];
        qnt[t * DK + tid] = __bfloat162float(tin[t * DK + tid]) * rnq[t];
    }
    if (tid < len) tb[tid] = 1.f / (1.f + exp2f(-tb[tid] * kLog2e));
    __syncthreads();

    for (int64_t t = 0; t < len; ++t) {
        const int64_t tok = ((row_base + t) * p.H + h) * DK;
        const float4 *alpha4 = reinterpret_cast<const float4 *>(alf + t * DK) + 2 * rg;
        const float4 *kn4 = reinterpret_cast<const float4 *>(knt + t * DK) + 2 * rg;
        const float4 *qn4 = reinterpret_cast<const float4 *>(qnt + t * DK) + 2 * rg;
        const float4 a0 = alpha4[0], a1 = alpha4[1], k0 = kn4[0], k1 = kn4[1];
        const float2 al[4] = {make_float2(a0.x, a0.y), make_float2(a0.z, a0.w), make_float2(a1.x, a1.y),
                              make_float2(a1.z, a1.w)};
        const float2 kk[4] = {make_float2(k0.x, k0.y), make_float2(k0.z, k0.w), make_float2(k1.x, k1.y),
                              make_float2(k1.z, k1.w)};

        // decay, then this thread's part of S^T k_hat for its four columns
        float ks[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x = mul2(make_float2(s[8 * i + 2 * e], s[8 * i + 2 * e + 1]), al[e]);
                acc = fma2(kk[e], x, acc);
                s[8 * i + 2 * e] = x.x; s[8 * i + 2 * e + 1] = x.y;
            }
            ks[i] = acc.x + acc.y;
        }
        // the warp's four row groups (lanes 8 and 16 apart), then the four warps
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ks[i] += __shfl_xor_sync(0xffffffffu, ks[i], 8);
            ks[i] += __shfl_xor_sync(0xffffffffu, ks[i], 16);
        }
        if (lane < 8) *reinterpret_cast<float4 *>(&red[0][warp][4 * cq]) = make_float4(ks[0], ks[1], ks[2], ks[3]);
        __syncthreads();
        float u[4];
        {
            const float4 r0 = *reinterpret_cast<const float4 *>(&red[0][0][4 * cq]);
            const float4 r1 = *reinterpret_cast<const float4 *>(&red[0][1][4 * cq]);
            const float4 r2 = *reinterpret_cast<const float4 *>(&red[0][2][4 * cq]);
            const float4 r3 = *reinterpret_cast<const float4 *>(&red[0][3][4 * cq]);
            const uint2 vw = *reinterpret_cast<const uint2 *>(&tv[t * VS + 4 * cq]);
            const float beta = tb[t];
            u[0] = beta * (__uint_as_float(vw.x << 16) - (r0.x + r1.x + r2.x + r3.x));
            u[1] = beta * (__uint_as_float(vw.x & 0xFFFF0000u) - (r0.y + r1.y + r2.y + r3.y));
            u[2] = beta * (__uint_as_float(vw.y << 16) - (r0.z + r1.z + r2.z + r3.z));
            u[3] = beta * (__uint_as_float(vw.y & 0xFFFF0000u) - (r0.w + r1.w + r2.w + r3.w));
        }
        // rank-1 update and this thread's part of S^T q_hat
        const float4 q0 = qn4[0], q1 = qn4[1];
        const float2 qq[4] = {make_float2(q0.x, q0.y), make_float2(q0.z, q0.w), make_float2(q1.x, q1.y),
                              make_float2(q1.z, q1.w)};
        float os[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 u2 = make_float2(u[i], u[i]);
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x = fma2(kk[e], u2, make_float2(s[8 * i + 2 * e], s[8 * i + 2 * e + 1]));
                acc = fma2(qq[e], x, acc);
                s[8 * i + 2 * e] = x.x; s[8 * i + 2 * e + 1] = x.y;
            }
            os[i] = acc.x + acc.y;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            os[i] += __shfl_xor_sync(0xffffffffu, os[i], 8);
            os[i] += __shfl_xor_sync(0xffffffffu, os[i], 16);
        }
        if (lane < 8) *reinterpret_cast<float4 *>(&red[1][warp][4 * cq]) = make_float4(os[0], os[1], os[2], os[3]);
        __syncthreads();
        if (warp == 0 && lane < 8) {
            const float4 r0 = *reinterpret_cast<const float4 *>(&red[1][0][4 * cq]);
            const float4 r1 = *reinterpret_cast<const float4 *>(&red[1][1][4 * cq]);
            const float4 r2 = *reinterpret_cast<const float4 *>(&red[1][2][4 * cq]);
            const float4 r3 = *reinterpret_cast<const float4 *>(&red[1][3][4 * cq]);
            const float sc = p.scale;
            const __nv_bfloat162 o01 = __floats2bfloat162_rn(sc * (r0.x + r1.x + r2.x + r3.x),
                                                             sc * (r0.y + r1.y + r2.y + r3.y));
            const __nv_bfloat162 o23 = __floats2bfloat162_rn(sc * (r0.z + r1.z + r2.z + r3.z),
                                                             sc * (r0.w + r1.w + r2.w + r3.w));
            *reinterpret_cast<uint2 *>(p.out + tok + vs * VS + 4 * cq) =
                make_uint2(*reinterpret_cast<const uint32_t *>(&o01), *reinterpret_cast<const uint32_t *>(&o23));
        }
    }

    if (p.fin) {
        __syncthreads();   // the tile may still hold the initial state being read
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int hq = 0; hq < 2; ++hq)
                *tile_chunk(4 * cq + i, 2 * rg + hq) = make_float4(s[8 * i + 4 * hq], s[8 * i + 4 * hq + 1],
                                                                   s[8 * i + 4 * hq + 2], s[8 * i + 4 * hq + 3]);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int row = warp * 8 + r;
            const float4 x = *tile_chunk(row, lane);
            if (p.state_type == kStateBF16) {
                const __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), b = __floats2bfloat162_rn(x.z, x.w);
                reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.fin) + slice + (size_t)row * DK)[lane] =
                    make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
            } else {
                reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.fin) + slice + (size_t)row * DK)[lane] = x;
            }
        }
    }
}

}  // namespace

cudaError_t launch_decode(const Params &p, cudaStream_t stream) {
    const int64_t units = p.n_seqs * p.H;
    if (units == 0) return cudaSuccess;
    kda_decode_kernel<<<(unsigned)(units * (DK / VS)), NTD, decode_smem_bytes((int)p.T), stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
