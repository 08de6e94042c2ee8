// Host side of the C ABI declared in include/kda.h: argument validation, the
// device error word, and dispatch to the kernels.
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/kda.h"
#include "kda_internal.h"

static_assert(KDA_WORKSPACE_BYTES_PER_UNIT == kda::kWsBytesPerUnit, "workspace size in kda.h");
static_assert(KDA_ERR_TIMEOUT == kda::kErrTimeout && KDA_ERR_RANGE == kda::kErrRange, "device error codes");

// Scratch of kda_fwd_static, for callers that cannot allocate: a fixed array in the
// library's own device memory, present on every device that loads the library.  Host
// code must not pass its name to a kernel (on the host it names a host-side stand-in);
// the device address comes from cudaGetSymbolAddress (static_workspace below).
static __device__ __align__(256) unsigned char
    g_kda_static_ws[(size_t)KDA_STATIC_MAX_UNITS * KDA_WORKSPACE_BYTES_PER_UNIT];

namespace {

// Set by kernels whose bounded waits give up; read and cleared by
// kda_get_device_status().  One word per device (module-scope __device__).
__device__ int g_kda_error = 0;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Most (sequence, head) units one call may hold: the widest launch (the sequence-parallel
// path's per-segment kernels, up to 32 segments per unit) must stay within 2^31 - 1 CTAs.
constexpr int64_t kMaxUnits = ((int64_t(1) << 31) - 1) / 32;

// Validates the arguments of kda_fwd and fills `p`.  Touches no device state.
kda_status validate(const void *q, const void *k, const void *v, const void *g, const void *beta,
                    float scale, void *out, const float *A_log, const float *dt_bias,
                    float lower_bound, const void *initial_state, void *final_state,
                    int state_dtype, const int64_t *cu_seqlens, int64_t num_seqs, int64_t B,
                    int64_t T, int64_t H, int64_t K, int64_t V, kda::Params &p) {
    if (K != kda::kHeadDim || V != kda::kHeadDim) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || T < 0 || H < 0) return KDA_ERR_SHAPE;
    // Token tensors may be NULL only when they hold no element (B*T*H == 0).
    const bool has_tokens = B > 0 && T > 0 && H > 0;
    if (has_tokens && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_NULL;
    if (H > 0 && (!A_log || !dt_bias)) return KDA_ERR_NULL;
    if (cu_seqlens) {
        if (B != 1 || num_seqs < 1) return KDA_ERR_SHAPE;
    }
    const int64_t N = cu_seqlens ? num_seqs : B;
    if (H == 0 && N > 0 && T > 0) return KDA_ERR_SHAPE;
    if (N > 0 && H > 0 && N > kMaxUnits / H) return KDA_ERR_SHAPE;
    if (initial_state || final_state) {
        if (state_dtype != KDA_STATE_BF16 && state_dtype != KDA_STATE_FP32) return KDA_ERR_DTYPE;
    } else if (state_dtype != KDA_STATE_NONE && state_dtype != KDA_STATE_BF16 &&
               state_dtype != KDA_STATE_FP32) {
        return KDA_ERR_DTYPE;
    }
    if (!(lower_bound >= -5.0f && lower_bound <= 0.0f)) return KDA_ERR_VALUE;
    if (!std::isfinite(scale)) return KDA_ERR_VALUE;
    const void *ptrs[] = {q, k, v, g, beta, out, A_log, dt_bias, initial_state, final_state};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return KDA_ERR_ALIGN;

    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.g = static_cast<const __nv_bfloat16 *>(g);
    p.beta = static_cast<const __nv_bfloat16 *>(beta);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    p.scale = scale;
    p.lower_bound = lower_bound;
    p.init = initial_state;
    p.fin = final_state;
    p.state_type = state_dtype;
    p.cu_seqlens = cu_seqlens;
    p.n_seqs = N;
    p.B = B;
    p.T = T;
    p.H = H;
    p.err = nullptr;
    p.ws = nullptr;
    return KDA_OK;
}

// Memory pool for kda_fwd's workspaces, one per device, created on first use and
// kept for the life of the process.  Its release threshold keeps freed blocks
// mapped, so the stream-ordered allocation of a call after the first is cheap;
// the device's default pool is left untouched.
cudaMemPool_t workspace_pool(int device) {
    static std::mutex mu;
    static std::vector<cudaMemPool_t> pools;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)pools.size() <= device) pools.resize(device + 1, nullptr);
    if (!pools[device]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = device;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
        uint64_t keep = UINT64_MAX;
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        pools[device] = pool;
    }
    return pools[device];
}

}  // namespace

namespace kda {
// The token recurrence with the gate that has no lower bound (csrc/kda_recur.cu).
cudaError_t launch_recur(const Params &p, cudaStream_t stream);

cudaError_t sm_count(int &sms) {
    static std::atomic<bool> done[kMaxDevices];
    static int count[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= kMaxDevices) return cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    e = once_per_device(done, [&](int d) { return cudaDeviceGetAttribute(&count[d], cudaDevAttrMultiProcessorCount, d); });
    sms = count[dev];
    return e;
}
}  // namespace kda

namespace {

// tsplit > 0: the sequence-parallel path with that many segments per sequence (p.ws is
// then its scratch, tsplit_scratch_bytes long); pool_sms > 0: the persistent pool kernel
// on that many SMs (p.ws its ring, pool_scratch_bytes long).
kda_status launch(kda::Params &p, void *stream, int64_t tsplit = 0, int pool_sms = 0) {
    // the device error word's address, looked up once per device
    static std::atomic<bool> done[kda::kMaxDevices];
    static int *err_of[kda::kMaxDevices];
    int *err = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::once_per_device(done, [&](int d) {
            return cudaGetSymbolAddress(reinterpret_cast<void **>(&err_of[d < kda::kMaxDevices ? d : 0]),
                                        g_kda_error);
        }) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (dev < kda::kMaxDevices) {
        err = err_of[dev];
    } else if (cudaGetSymbolAddress(reinterpret_cast<void **>(&err), g_kda_error) != cudaSuccess) {
        return KDA_ERR_CUDA;
    }
    p.err = err;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (tsplit > 0) {
        e = kda::launch_tsplit(p, tsplit, pool_sms, p.ws, cs);
    } else if (pool_sms > 0) {
        e = cudaSuccess;
        if (p.cu_seqlens && p.T <= kda::kMixedMaxAvg * p.n_seqs && !p.unbounded) {
            // mostly short sequences: those of at most kShortMaxT tokens on the short-step
            // kernel, the rest on the pool, one launch after the other
            p.mixed = 1;
            e = kda::launch_short(p, cs);
        }
        if (e == cudaSuccess) e = kda::launch_pool(p, pool_sms, cs);
    } else if (p.T == 1) {
        e = kda::launch_decode(p, cs);
    } else if (p.T <= kda::kShortMaxT) {
        e = kda::launch_short(p, cs);
    } else if (p.cu_seqlens && p.T <= kda::kMixedMaxAvg * p.n_seqs) {
        // mostly short sequences: each kernel on its own sequences, one after the other
        p.mixed = 1;
        e = kda::launch_short(p, cs);
        if (e == cudaSuccess) e = kda::launch_cluster(p, cs);
    } else {
        e = kda::launch_cluster(p, cs);
    }
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// Device address of g_kda_static_ws on the current device, looked up once per device
// (with that device current) and cached.
cudaError_t static_workspace(unsigned char *&ws) {
    static std::atomic<bool> done[kda::kMaxDevices];
    static unsigned char *addr_of[kda::kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= kda::kMaxDevices) return cudaGetSymbolAddress(reinterpret_cast<void **>(&ws), g_kda_static_ws);
    e = kda::once_per_device(done, [&](int d) {
        return cudaGetSymbolAddress(reinterpret_cast<void **>(&addr_of[d]), g_kda_static_ws);
    });
    if (e != cudaSuccess) return e;
    ws = addr_of[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

kda_status kda_fwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                   float scale, void *out, const float *A_log, const float *dt_bias,
                   float lower_bound, const void *initial_state, void *final_state,
                   int state_dtype, const int64_t *cu_seqlens, int64_t num_seqs, int64_t B,
                   int64_t T, int64_t H, int64_t K, int64_t V, void *stream) {
    kda::Params p{};   // every field zero until validate() fills it
    kda_status st = validate(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                             initial_state, final_state, state_dtype, cu_seqlens, num_seqs, B, T,
                             H, K, V, p);
    if (st != KDA_OK) return st;
    if (p.n_seqs == 0 || p.H == 0) return KDA_OK;
    if (p.T <= kda::kShortMaxT) return launch(p, stream);   // the short-step kernels need no workspace
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return KDA_ERR_CUDA;
    cudaMemPool_t pool = workspace_pool(device);
    if (!pool) return KDA_ERR_CUDA;
    // Few (sequence, head) units on a long fixed-length call: the sequence-parallel path
    int sms = 0;
    if (kda::sm_count(sms) != cudaSuccess) return KDA_ERR_CUDA;
    const int64_t tsplit = kda::tsplit_segments(p, sms);
    // other calls run the persistent pool kernel (varlen calls of up to kPoolMaxSeqs
    // sequences), the rest the cluster kernel
    const int pool_sms = (tsplit > 0 || kda::pool_takes(p, sms)) ? sms : 0;
    const size_t bytes = tsplit > 0     ? kda::tsplit_scratch_bytes(p, tsplit, sms)
                         : pool_sms > 0 ? kda::pool_scratch_bytes(p, pool_sms)
                                        : (size_t)(p.n_seqs * p.H) * kda::kWsBytesPerUnit;
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, bytes, pool, cs) != cudaSuccess) return KDA_ERR_CUDA;
    p.ws = static_cast<unsigned char *>(ws);
    st = launch(p, stream, tsplit, pool_sms);
    if (cudaFreeAsync(ws, cs) != cudaSuccess) st = KDA_ERR_CUDA;
    return st;
}

kda_status kda_fwd_ws(const void *q, const void *k, const void *v, const void *g, const void *beta,
                      float scale, void *out, const float *A_log, const float *dt_bias,
                      float lower_bound, const void *initial_state, void *final_state,
                      int state_dtype, const int64_t *cu_seqlens, int64_t num_seqs, int64_t B,
                      int64_t T, int64_t H, int64_t K, int64_t V, void *workspace,
                      size_t workspace_bytes, void *stream) {
    kda::Params p{};   // every field zero until validate() fills it
    kda_status st = validate(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                             initial_state, final_state, state_dtype, cu_seqlens, num_seqs, B, T,
                             H, K, V, p);
    if (st != KDA_OK) return st;
    const int64_t units = p.n_seqs * p.H;
    if (units > 0 && !workspace) return KDA_ERR_NULL;
    if (workspace && !aligned16(workspace)) return KDA_ERR_ALIGN;
    if ((uint64_t)workspace_bytes < (uint64_t)units * kda::kWsBytesPerUnit) return KDA_ERR_VALUE;
    if (units == 0) return KDA_OK;
    p.ws = static_cast<unsigned char *>(workspace);
    // a fixed-length call of more than 64 rows with room for the pool kernel's ring
    // (kda_workspace_size_pool) runs the pool kernel; otherwise the cluster kernel
    if (!p.cu_seqlens && p.T > kda::kShortMaxT) {
        int sms = 0;
        if (kda::sm_count(sms) != cudaSuccess) return KDA_ERR_CUDA;
        if (workspace_bytes >= kda::pool_scratch_bytes(p, sms)) return launch(p, stream, 0, sms);
    }
    return launch(p, stream);
}

kda_status kda_fwd_unbounded(const void *q, const void *k, const void *v, const void *g,
                             const void *beta, float scale, void *out, const float *A_log,
                             const float *dt_bias, const void *initial_state, void *final_state,
                             int state_dtype, const int64_t *cu_seqlens, int64_t num_seqs,
                             int64_t B, int64_t T, int64_t H, int64_t K, int64_t V, void *stream) {
    kda::Params p{};   // every field zero until validate() fills it
    // the lower bound is not an argument here; 0 passes its range check
    kda_status st = validate(q, k, v, g, beta, scale, out, A_log, dt_bias, 0.f, initial_state,
                             final_state, state_dtype, cu_seqlens, num_seqs, B, T, H, K, V, p);
    if (st != KDA_OK) return st;
    if (p.n_seqs == 0 || p.H == 0) return KDA_OK;
    p.unbounded = 1;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int sms = 0;
    if (kda::sm_count(sms) != cudaSuccess) return KDA_ERR_CUDA;
    // Calls of at most 64 rows, and varlen batches beyond the pool's plan, run the token
    // recurrence; the rest the pool kernel's chunked form (every sequence on it), long
    // fixed-length calls with few units sequence-parallel as in kda_fwd.
    const int64_t tsplit = p.T > kda::kShortMaxT ? kda::tsplit_segments(p, sms) : 0;
    if (tsplit == 0 && (p.T <= kda::kShortMaxT || !kda::pool_takes(p, sms)))
        return kda::launch_recur(p, cs) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return KDA_ERR_CUDA;
    cudaMemPool_t pool = workspace_pool(device);
    if (!pool) return KDA_ERR_CUDA;
    const size_t bytes = tsplit > 0 ? kda::tsplit_scratch_bytes(p, tsplit, sms) : kda::pool_scratch_bytes(p, sms);
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, bytes, pool, cs) != cudaSuccess) return KDA_ERR_CUDA;
    p.ws = static_cast<unsigned char *>(ws);
    st = launch(p, stream, tsplit, sms);
    if (cudaFreeAsync(ws, cs) != cudaSuccess) st = KDA_ERR_CUDA;
    return st;
}

kda_status kda_bwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                   float scale, const float *A_log, const float *dt_bias, float lower_bound,
                   int unbounded, const void *initial_state, int state_dtype, const void *dout,
                   const float *dfinal, const int64_t *cu_seqlens, int64_t num_seqs, int64_t B,
                   int64_t T, int64_t H, int64_t K, int64_t V, float *dq, float *dk, float *dv,
                   float *dg, float *dbeta, float *dA_log, float *ddt_bias,
                   float *dinitial_state, void *stream) {
    kda::Params p{};   // every field zero until validate() fills it
    // dout stands where out stands in kda_fwd (same shape); no final state is an input
    kda_status st = validate(q, k, v, g, beta, scale, const_cast<void *>(dout), A_log, dt_bias,
                             unbounded ? 0.f : lower_bound, initial_state, nullptr,
                             initial_state ? state_dtype : KDA_STATE_NONE, cu_seqlens, num_seqs, B,
                             T, H, K, V, p);
    if (st != KDA_OK) return st;
    const bool has_tokens = B > 0 && T > 0 && H > 0;
    if (has_tokens && (!dq || !dk || !dv || !dg || !dbeta)) return KDA_ERR_NULL;
    if (H > 0 && (!dA_log || !ddt_bias)) return KDA_ERR_NULL;
    const void *ptrs[] = {dfinal, dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dinitial_state};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return KDA_ERR_ALIGN;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int sms = 0;
    if (kda::sm_count(sms) != cudaSuccess) return KDA_ERR_CUDA;
    kda::BwdGrads gr{static_cast<const __nv_bfloat16 *>(dout), dfinal, dq, dk, dv, dg, dbeta,
                     dA_log, ddt_bias, dinitial_state};
    void *ws = nullptr;
    const size_t bytes = kda::bwd_scratch_bytes(p, sms);
    if (p.n_seqs * p.H > 0) {
        int device = 0;
        if (cudaGetDevice(&device) != cudaSuccess) return KDA_ERR_CUDA;
        cudaMemPool_t pool = workspace_pool(device);
        if (!pool) return KDA_ERR_CUDA;
        if (cudaMallocFromPoolAsync(&ws, bytes, pool, cs) != cudaSuccess) return KDA_ERR_CUDA;
    }
    st = kda::launch_bwd(p, gr, unbounded ? 1 : 0, static_cast<unsigned char *>(ws), sms, cs) == cudaSuccess
             ? KDA_OK
             : KDA_ERR_CUDA;
    if (ws && cudaFreeAsync(ws, cs) != cudaSuccess) st = KDA_ERR_CUDA;
    return st;
}

kda_status kda_fwd_static(const void *q, const void *k, const void *v, const void *g,
                          const void *beta, float scale, void *out, const float *A_log,
                          const float *dt_bias, float lower_bound, const void *initial_state,
                          void *final_state, int state_dtype, const int64_t *cu_seqlens,
                          int64_t num_seqs, int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                          void *stream) {
    kda::Params p{};   // every field zero until validate() fills it
    kda_status st = validate(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                             initial_state, final_state, state_dtype, cu_seqlens, num_seqs, B, T,
                             H, K, V, p);
    if (st != KDA_OK) return st;
    const int64_t units = p.n_seqs * p.H;
    if (units > KDA_STATIC_MAX_UNITS) return KDA_ERR_LIMIT;
    if (units == 0) return KDA_OK;
    unsigned char *ws = nullptr;
    if (static_workspace(ws) != cudaSuccess) return KDA_ERR_CUDA;
    p.ws = ws;
    return launch(p, stream);
}

size_t kda_workspace_size_pool(int64_t num_seqs, int64_t H) {
    if (num_seqs <= 0 || H <= 0 || num_seqs > (int64_t(1) << 30) || H > (int64_t(1) << 22)) return 0;
    int sms = 0;
    if (kda::sm_count(sms) != cudaSuccess) return 0;
    kda::Params p{};
    p.n_seqs = num_seqs;
    p.H = H;
    p.B = num_seqs;
    const size_t pool = kda::pool_scratch_bytes(p, sms);
    const size_t cluster = kda_workspace_size(num_seqs, H);
    return pool > cluster ? pool : cluster;
}

size_t kda_workspace_size(int64_t num_seqs, int64_t H) {
    if (num_seqs < 0 || H < 0) return 0;
    if (num_seqs == 0 || H == 0) return 0;
    const uint64_t per = (uint64_t)KDA_WORKSPACE_BYTES_PER_UNIT;
    const uint64_t n = (uint64_t)num_seqs, h = (uint64_t)H;
    if (n > SIZE_MAX / h || n * h > SIZE_MAX / per) return 0;
    return (size_t)(n * h * per);
}

const char *kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_NULL: return "KDA_ERR_NULL: a required pointer is NULL";
        case KDA_ERR_DTYPE: return "KDA_ERR_DTYPE: bad state dtype";
        case KDA_ERR_SHAPE: return "KDA_ERR_SHAPE: inconsistent sizes";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: only K = V = 128 is supported";
        case KDA_ERR_ALIGN: return "KDA_ERR_ALIGN: tensor pointer not 16-byte aligned";
        case KDA_ERR_VALUE: return "KDA_ERR_VALUE: lower_bound outside [-5, 0], non-finite scale or workspace too small";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA call or launch failed";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a bounded device wait expired";
        case KDA_ERR_RANGE: return "KDA_ERR_RANGE: an fp16 operand (v, state, U, W, T', M; q, k on short steps) exceeded 65504";
        case KDA_ERR_LIMIT: return "KDA_ERR_LIMIT: kda_fwd_static takes at most KDA_STATIC_MAX_UNITS (sequence, head) units";
        default: return "KDA: unknown status";
    }
}

kda_status kda_get_device_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KDA_ERR_CUDA;
    int h = 0;
    if (cudaMemcpyFromSymbol(&h, g_kda_error, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_kda_error, &zero, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    return h == 0 ? KDA_OK : static_cast<kda_status>(h);
}

int kda_version(void) { return 101; }

}  // extern "C"
