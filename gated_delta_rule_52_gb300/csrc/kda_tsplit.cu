// Sequence-parallel (T-split) prefill for calls with few (sequence, head) units.
//
// The chunk map of the KDA recurrence is affine in the entering state:
//   S_out = P S_in + R,  P = prod over the chunks of (Diag(Gamma_C) - Kbar^T W),
// with R the state reached from S_in = 0 (the chunk equations of the tensor-core
// path: U = T'V - W S_in, S_out = Diag(Gamma_C) S_in + Kbar^T U).  So a sequence
// cut into segments runs as:
//   1. every segment from S = 0 (segment 0 from the call's initial state): R_s; and
//   2. beside it, over the same chunk packets, every segment with v = 0 from S = I:
//      the transition P_s (the pool kernel's second state, one run for both);
//   3. a scan over the segments: S_in(0) = S_0, S_in(s) = P_{s-1} S_in(s-1) + R_{s-1};
//   4. every segment from S_in(s), writing the outputs (and, for the last segment,
//      the final state).
// Steps 1-2 and 4 are the persistent pool kernel over the segments as independent
// packed sequences (segment boundaries as cu_seqlens, so each run plans its units
// first); 1-2 writes no outputs.  With P segments per sequence each of those runs has
// P times the parallelism of the plain call; the chunk work (the fronts) is done twice.
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int DK = kHeadDim;
constexpr int64_t kState = (int64_t)DK * DK;             // elements of one state
constexpr int64_t kStateBytes = kState * 4;               // fp32 segment states

// cu_seqlens of the segments over the flattened [B*T] token rows: segment i = b P + s
// covers rows b T + s Ls .. min(b T + (s + 1) Ls, (b + 1) T); entry N P is N T.
__global__ void seg_bounds_kernel(int64_t *cu, int64_t N, int64_t P, int64_t T, int64_t Ls) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i > N * P) return;
    const int64_t b = i / P, s = i % P;
    cu[i] = b * T + (s * Ls < T ? s * Ls : T);
}

// Initial states of steps 1 and 2: r0[b P + s, h] = the call's initial state for s = 0
// (zero if none), zero otherwise; id[b P + s, h] = I.  Grid (segment states, 16):
// block y covers rows 8 y .. 8 y + 7 of one state, four channels per thread.
__global__ void seg_init_kernel(float *r0, float *id, const void *init, int state_type, int64_t P,
                                int64_t H) {
    const int64_t idx = blockIdx.x, h = idx % H, seg = idx / H, b = seg / P, s = seg % P;
    const int i = (int)blockIdx.y * 1024 + 4 * threadIdx.x;   // 256 threads x 4 = 8 rows
    const int row = i / DK, col = i % DK;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (s == 0 && init) {
        const int64_t off = (b * H + h) * kState + i;
        if (state_type == kStateBF16) {
            const uint2 w = *reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(init) + off);
            x = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                            __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
        } else {
            x = *reinterpret_cast<const float4 *>(static_cast<const float *>(init) + off);
        }
    }
    *reinterpret_cast<float4 *>(r0 + idx * kState + i) = x;
    *reinterpret_cast<float4 *>(id + idx * kState + i) =
        make_float4(row == col, row == col + 1, row == col + 2, row == col + 3);
}

// The scan of step 3: sin[s] = sin[s-1] x Pst[s-1] + R[s-1] in the stored (transposed)
// layout, sin[0] given; fp32 on paired FMAs.  The rows of the product are independent,
// so grid (sequence states, 32): block y carries rows 4 y .. 4 y + 3 through every step,
// reading each transition (L2-resident) whole into shared memory.  256 threads, thread
// (tr, tc) = row 4 y + tr, columns 2 tc and 2 tc + 1.  The block's rows sit in shared
// memory padded to 129 floats (a warp shares its row: reads are broadcasts), the
// transition unpadded (a warp reads 32 consecutive float pairs).
constexpr int kZs = DK + 1;
constexpr int kScanRows = 4;
__global__ void __launch_bounds__(256) seg_scan_kernel(float *sin, const float *R, const float *Pst,
                                                       int64_t P, int64_t H) {
    extern __shared__ __align__(16) float scan_sm[];
    float *pm = scan_sm;                 // [j][k]: stored transition of the previous segment
    float *zs = scan_sm + kState;        // [tr][j]: this block's rows of the entering state
    const int64_t b = blockIdx.x / H, h = blockIdx.x % H;
    const int rb = (int)blockIdx.y * kScanRows;
    const int tid = threadIdx.x, tr = tid >> 6, tc = tid & 63;
    auto slot = [&](int64_t s) { return ((b * P + s) * H + h) * kState; };
    const float *z0 = sin + slot(0) + (int64_t)rb * DK;
    for (int i = tid; i < kScanRows * DK; i += 256) zs[(i / DK) * kZs + i % DK] = z0[i];
    for (int64_t s = 1; s < P; ++s) {
        const float *ps = Pst + slot(s - 1);
        for (int i = tid * 4; i < kState; i += 1024)
            *reinterpret_cast<float4 *>(pm + i) = *reinterpret_cast<const float4 *>(ps + i);
        __syncthreads();
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll 16
        for (int j = 0; j < DK; ++j) {
            const float z = zs[tr * kZs + j];
            acc = sm103::fma2(make_float2(z, z), *reinterpret_cast<const float2 *>(pm + j * DK + 2 * tc), acc);
        }
        __syncthreads();   // every thread is done with zs and pm
        const int v = rb + tr, k = 2 * tc;
        const float2 x = sm103::add2(acc, *reinterpret_cast<const float2 *>(R + slot(s - 1) + (int64_t)v * DK + k));
        *reinterpret_cast<float2 *>(sin + slot(s) + (int64_t)v * DK + k) = x;
        zs[tr * kZs + k] = x.x;
        zs[tr * kZs + k + 1] = x.y;
    }
}

// Step 4's final states -> the call's final state: fin[b, h] = fin3[b P + P - 1, h].
// Grid (sequence states, 16), four channels per thread.
__global__ void seg_final_kernel(void *fin, int state_type, const float *fin3, int64_t P, int64_t H) {
    const int64_t b = blockIdx.x / H, h = blockIdx.x % H;
    const int i = (int)blockIdx.y * 1024 + 4 * threadIdx.x;
    const float4 x = *reinterpret_cast<const float4 *>(fin3 + ((b * P + P - 1) * H + h) * kState + i);
    const int64_t dst = (b * H + h) * kState + i;
    if (state_type == kStateBF16)
        *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(fin) + dst) =
            make_uint2(sm103::pack_bf16(x.x, x.y), sm103::pack_bf16(x.z, x.w));
    else
        *reinterpret_cast<float4 *>(static_cast<float *>(fin) + dst) = x;
}

int64_t seg_len(int64_t T, int64_t P) {
    const int64_t per = (T + P - 1) / P;
    return (per + kChunk - 1) / kChunk * kChunk;
}

}  // namespace

int64_t tsplit_segments(const Params &p, int sms) {
    if (p.cu_seqlens || p.B <= 0 || p.T < kTsplitMinSeg * 4) return 0;
    const int64_t units = p.n_seqs * p.H;
    if (units <= 0) return 0;
    // Each run is bound by the slower of its chains (T / P chunks in a row, about 6K
    // cycles each) and its fronts (every chunk of every unit, about 9.5K cycles each, over
    // the SMs the chains leave): they balance with the chains on about 3/8 of the SMs.
    // Up to sms / 8 units, 4 segments still beat the plain path.
    int64_t P = (sms * 3 / 8) / units;
    if (P < 4 && (sms / 2) / units >= 4) P = 4;
    if (P > p.T / kTsplitMinSeg) P = p.T / kTsplitMinSeg;
    if (P > kTsplitMaxSeg) P = kTsplitMaxSeg;
    return P >= 4 ? P : 0;
}

size_t tsplit_scratch_bytes(const Params &p, int64_t P, int sms) {
    const int64_t N = p.n_seqs, H = p.H;
    const size_t cu = ((size_t)(N * P + 1) * 8 + 255) / 256 * 256;
    return cu + 4 * (size_t)(N * P * H) * kStateBytes + pool_scratch_bytes_varlen(N * P, H, N * p.T, sms);
}

cudaError_t launch_tsplit(const Params &p, int64_t P, int sms, unsigned char *scratch, cudaStream_t stream) {
    const int64_t N = p.n_seqs, H = p.H, T = p.T, Ls = seg_len(T, P), S = N * P;
    const size_t cu_bytes = ((size_t)(S + 1) * 8 + 255) / 256 * 256, sb = (size_t)(S * H) * kStateBytes;
    int64_t *cu = reinterpret_cast<int64_t *>(scratch);
    float *sin = reinterpret_cast<float *>(scratch + cu_bytes);            // also step 1's initial states
    float *fin3 = reinterpret_cast<float *>(scratch + cu_bytes + sb);      // also step 2's identities
    float *R = reinterpret_cast<float *>(scratch + cu_bytes + 2 * sb);
    float *Pst = reinterpret_cast<float *>(scratch + cu_bytes + 3 * sb);
    unsigned char *ws = scratch + cu_bytes + 4 * sb;

    seg_bounds_kernel<<<(unsigned)((S + 1 + 255) / 256), 256, 0, stream>>>(cu, N, P, T, Ls);
    seg_init_kernel<<<dim3((unsigned)(S * H), 16), 256, 0, stream>>>(sin, fin3, p.init, p.state_type, P, H);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    Params q = p;   // the segments as packed sequences over the flattened rows
    q.cu_seqlens = cu;
    q.n_seqs = S;
    q.B = 1;
    q.T = N * T;
    q.state_type = kStateFP32;
    q.mixed = 0;   // every segment on the pool
    q.ws = ws;
    // 1 and 2 in one state-only run over the same packets: R_s from S = 0 (segment 0
    // from the call's initial state), and beside it the transition P_s from S = I with
    // values of zero
    q.init = sin;
    q.fin = R;
    q.out = nullptr;
    q.init2 = fin3;
    q.fin2 = Pst;
    if ((e = launch_pool(q, sms, stream)) != cudaSuccess) return e;
    q.init2 = nullptr;
    q.fin2 = nullptr;
    // 3. the scan
    const int scan_smem = (int)((kState + (int64_t)kScanRows * kZs) * 4);
    static std::atomic<bool> attr_done[kMaxDevices];
    if ((e = once_per_device(attr_done, [&](int) {
             return cudaFuncSetAttribute(seg_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, scan_smem);
         })) != cudaSuccess)
        return e;
    seg_scan_kernel<<<dim3((unsigned)(N * H), DK / kScanRows), 256, scan_smem, stream>>>(sin, R, Pst, P, H);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 4. every segment from its entering state, with outputs (the same segments, heads
    // and workspace as the first run: its plan stands)
    q.init = sin;
    q.fin = fin3;
    q.out = p.out;
    if ((e = launch_pool(q, sms, stream, true)) != cudaSuccess) return e;
    if (p.fin) {
        seg_final_kernel<<<dim3((unsigned)(N * H), 16), 256, 0, stream>>>(p.fin, p.state_type, fin3, P, H);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace kda
