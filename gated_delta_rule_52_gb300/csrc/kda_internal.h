// Internal launch parameters shared by the host entry points and the kernels of
// libkda.so.  Not part of the public ABI (that is include/kda.h).
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace kda {

constexpr int kHeadDim = 128;   // K = V = 128, the only supported head size
constexpr int kChunk = 64;      // tokens per chunk of the UT/WY form
// Workspace per (sequence, head): two slots of the chain operands of one chunk
// (Kbar, Q_hat*Gamma, K_hat*Gamma as fp16 tiles, 16 KB each, and exp(G_C), 512 B).
constexpr int64_t kWsSlot = 3 * 16384 + 512;
constexpr int64_t kWsBytesPerUnit = 2 * kWsSlot;

enum StateType : int { kStateNone = 0, kStateBF16 = 1, kStateFP32 = 2 };

// Device error word values (kda_status codes of include/kda.h).
constexpr int kErrTimeout = 8;   // a bounded wait gave up
constexpr int kErrRange = 10;    // an fp16 operand (v, state, U, W, T', M) left +-65504

// Problem description after host-side validation.  Tensor layouts are those of
// the FlashKDA README "Kernel API" table: q,k,g [B,T,H,128], v,out [B,T,H,128],
// beta [B,T,H], A_log [H], dt_bias [H,128], states [N,H,V,K].
struct Params {
    const __nv_bfloat16 *q, *k, *v, *g, *beta;   // v may be null inside the library: values of zero
    __nv_bfloat16 *out;                            // null inside the library: outputs not written
    const float *A_log, *dt_bias;
    float scale, lower_bound;
    const void *init;   // nullptr = zero state
    void *fin;          // nullptr = not written
    int state_type;
    const int64_t *cu_seqlens;   // nullptr = fixed-length batch
    int64_t n_seqs;     // N: sequences (B without cu_seqlens)
    int64_t B, T, H;
    int *err;           // device error word (bounded waits that give up set it)
    unsigned char *ws;  // workspace: kWsBytesPerUnit bytes per (sequence, head), 16-byte aligned
    int unbounded;      // the gate without a lower bound (lower_bound unused); pool kernel only
    int mixed;          // varlen call split by length: the short-step kernel takes the
                        // sequences of at most kShortMaxT tokens, the chunked kernel the rest
    // Pool kernel, varlen state-only runs (out == nullptr, bounded gate): a second state
    // carried beside the first over the same packets, with values of zero (U = -W S),
    // from init2 to fin2 (fp32, [N][H][V][K]); fin2 == nullptr: no second state
    const float *init2;
    float *fin2;
};

// Token range of sequence n: packed batch row `b`, first token `t0`, `len` tokens.
__device__ __forceinline__ void seq_range(const Params &p, int64_t n, int64_t &b, int64_t &t0,
                                          int64_t &len) {
    if (p.cu_seqlens) {
        b = 0;
        t0 = p.cu_seqlens[n];
        len = p.cu_seqlens[n + 1] - t0;
    } else {
        b = n;
        t0 = 0;
        len = p.T;
    }
}

// Calls with at most kShortMaxT token rows (T of the packed batch) run a kernel with
// no workspace instead of the chunked cluster kernel: the token recurrence for one row
// (decode), blocks of 16 rows on warp-level tensor-core MMAs otherwise.
constexpr int64_t kShortMaxT = 64;
// Varlen calls with more rows but at most this many per sequence on average run both
// kernels, each on its own sequences (Params::mixed).
constexpr int64_t kMixedMaxAvg = 256;

// Per-device values that a launcher sets up once (a kernel's shared-memory limit, the SM
// count): `f(device)` runs until it succeeds on that device; two threads racing both run
// it, which is harmless.  Devices beyond kMaxDevices run it every time.
constexpr int kMaxDevices = 64;
template <typename F>
cudaError_t once_per_device(std::atomic<bool> (&done)[kMaxDevices], F &&f) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = f(dev);
    if (e == cudaSuccess && dev < kMaxDevices) done[dev].store(true, std::memory_order_release);
    return e;
}
// The SM count of the current device (cached).
cudaError_t sm_count(int &sms);

// Launchers (each returns the cudaError_t of its launch).
cudaError_t launch_cluster(const Params &p, cudaStream_t stream);   // chunked, needs p.ws
cudaError_t launch_decode(const Params &p, cudaStream_t stream);    // token recurrence, T = 1 only
cudaError_t launch_short(const Params &p, cudaStream_t stream);     // 16-row blocks, 2 <= T <= 64

// Persistent pool kernel for calls of more than kShortMaxT rows: chain CTAs run the state
// recurrence, front CTAs the chunk-parallel work, handing each chunk over through a ring
// in p.ws (pool_scratch_bytes long).  Varlen calls (up to kPoolMaxSeqs sequences; with
// p.mixed set, only the sequences of more than kShortMaxT tokens) first run a one-CTA plan
// that orders the units longest first and spreads them over the chains.
constexpr int64_t kPoolMaxSeqs = 4096;
int64_t pool_chains(int64_t units, int sms);
bool pool_takes(const Params &p, int sms);   // the pool path accepts this call
size_t pool_scratch_bytes(const Params &p, int sms);
size_t pool_scratch_bytes_varlen(int64_t N, int64_t H, int64_t T, int sms);   // N sequences, T packed rows
// plan_ready: a varlen call whose plan an earlier launch on the same stream wrote into the
// same workspace for the same cu_seqlens, H and sms (the plan kernel is skipped)
cudaError_t launch_pool(const Params &p, int sms, cudaStream_t stream, bool plan_ready = false);

// Sequence-parallel prefill (fixed-length calls with few (sequence, head) units): each
// sequence cut into P segments of at least kTsplitMinSeg tokens, P in [4, kTsplitMaxSeg].
constexpr int64_t kTsplitMinSeg = 2048;
constexpr int64_t kTsplitMaxSeg = 32;
int64_t tsplit_segments(const Params &p, int sms);   // P, or 0: run the plain path
size_t tsplit_scratch_bytes(const Params &p, int64_t P, int sms);
cudaError_t launch_tsplit(const Params &p, int64_t P, int sms, unsigned char *scratch, cudaStream_t stream);

// Backward (kda_bwd): the gradients of L = sum(dout * out) + sum(dfinal * final) with
// respect to the forward's inputs, fp32, on p's forward inputs.
struct BwdGrads {
    const __nv_bfloat16 *dout;   // [B,T,H,V]
    const float *dfinal;         // [N,H,V,K] or null
    float *dq, *dk, *dv, *dg, *dbeta, *dA_log, *ddt_bias, *dinit;   // dinit may be null
};
size_t bwd_scratch_bytes(const Params &p, int sms);
cudaError_t launch_bwd(const Params &p, const BwdGrads &g, int unbounded, unsigned char *ws, int sms,
                       cudaStream_t stream);

}  // namespace kda
