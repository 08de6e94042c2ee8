/*
 * kda.h — C ABI of the GB300 (sm_103a) Kimi Delta Attention forward library
 * (libkda.so).
 *
 * The operation is the one the FlashKDA README documents under "Kernel API"
 * (flash_kda.fwd and its parameter table): the forward pass of KDA, the
 * channel-wise gated delta rule (agents-report.net "FlashKDA" article,
 * background section).  Per (sequence, head), with S a K x V state:
 *
 *   q_hat, k_hat = L2-normalised q, k        beta_t = sigmoid(beta_logit_t)
 *   gk_t[c]      = lower_bound * sigmoid(exp(A_log[h]) * (g_t[c] + dt_bias[h][c]))
 *   S_t          = (I - beta_t k_t k_t^T) Diag(exp(gk_t)) S_{t-1} + beta_t k_t v_t^T
 *   out_t        = scale * S_t^T q_t
 *
 * The pages name the gate inputs (A_log "log-gate parameter", dt_bias "gate
 * bias", lower_bound "gate lower bound, -5.0 to 0") but print no formula; the
 * gate above is this library's reading.  kda_fwd_unbounded takes the gate with no
 * lower bound instead, -exp(A_log[h]) * softplus(g_t[c] + dt_bias[h][c]).  The L2
 * norm uses eps = 1e-6 inside the square root.
 *
 * Everything here is plain C: device pointers, host scalars, a stream handle.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  Argument errors are detected on the host before any work is
 * enqueued; nothing is launched and no output is touched when one is returned. */
typedef enum {
    KDA_OK = 0,
    KDA_ERR_NULL = 1,        /* a required pointer is NULL (token tensors may be NULL
                                only when B*T*H == 0; A_log, dt_bias when H == 0)       */
    KDA_ERR_DTYPE = 2,       /* state pointer given with state_dtype KDA_STATE_NONE,
                                or an unknown state_dtype code                          */
    KDA_ERR_SHAPE = 3,       /* negative size, H == 0 with work to do, B != 1 with
                                cu_seqlens, num_seqs < 1 with cu_seqlens, or more than
                                2^26 - 1 (sequence, head) units (N * H) in one call    */
    KDA_ERR_UNSUPPORTED = 4, /* K != 128 or V != 128 (the only head size supported)    */
    KDA_ERR_ALIGN = 5,       /* a tensor pointer is not 16-byte aligned                 */
    KDA_ERR_VALUE = 6,       /* lower_bound outside [-5, 0], non-finite scale, or (for
                                kda_fwd_ws) a workspace smaller than required          */
    KDA_ERR_CUDA = 7,        /* a CUDA runtime call or kernel launch failed             */
    KDA_ERR_TIMEOUT = 8,     /* a bounded on-device wait expired (kda_get_device_status) */
    KDA_ERR_LIMIT = 9,       /* kda_fwd_static: N * H above KDA_STATIC_MAX_UNITS          */
    KDA_ERR_RANGE = 10       /* an fp16 operand left +-65504 (kda_get_device_status; see
                                "Value range" at kda_fwd)                              */
} kda_status;

/* Element type of initial_state / final_state (both, when both are given). */
typedef enum {
    KDA_STATE_NONE = 0,
    KDA_STATE_BF16 = 1,
    KDA_STATE_FP32 = 2
} kda_state_dtype;

/*
 * kda_fwd — KDA forward pass, written in place into `out` (and `final_state`).
 * Follows the FlashKDA README "Kernel API" table (flash_kda.fwd) and the 2kiu.com
 * article on its `out` parameter (section 一, "what is the out parameter": the
 * caller allocates `out`, the call returns nothing and writes it in place).
 *
 * Arguments (all tensors contiguous, row-major, on the current CUDA device):
 *   q, k, g        bf16 [B, T, H, K]   query, key, gate before activation
 *   v              bf16 [B, T, H, V]   value
 *   beta           bf16 [B, T, H]      beta logits (sigmoid applied inside)
 *   scale          host float          output scale
 *   out            bf16 [B, T, H, V]   output, fully overwritten (never read)
 *   A_log          fp32 [H]            log-gate parameter
 *   dt_bias        fp32 [H, K]         gate bias
 *   lower_bound    host float in [-5, 0]
 *   initial_state  [N, H, V, K] or NULL (NULL = zero state); state[n][h][v][c]
 *                  holds S[c][v] (V before K)
 *   final_state    [N, H, V, K] or NULL (NULL = not written)
 *   state_dtype    kda_state_dtype of both states; KDA_STATE_NONE only when both
 *                  state pointers are NULL
 *   cu_seqlens     device int64 [num_seqs + 1] or NULL.  With it, B must be 1,
 *                  sequence n is tokens [cu_seqlens[n], cu_seqlens[n+1]) of the
 *                  packed T, and N = num_seqs.  Without it, each batch row is a
 *                  sequence and N = B.  Its contents are not validated on the host
 *                  (that would need a device sync): they must start at 0, be
 *                  non-decreasing and end at T.
 *   B, T, H, K, V  sizes; K = V = 128 is required
 *   stream         cudaStream_t to enqueue on (NULL = legacy default stream)
 *
 * Ownership: the caller owns every buffer and the call keeps no pointer after it
 * returns.  The only memory the call allocates is its workspace, taken
 * stream-ordered on `stream` from a memory pool that libkda.so creates once per
 * device and keeps mapped, and released on `stream` after the kernel:
 *   - fixed-length calls of more than 64 rows run one persistent kernel, one CTA
 *     per SM launched cooperatively (it starts once every CTA can be resident):
 *     "front" CTAs form the chunk-parallel operands of every chunk and hand them
 *     to "chain" CTAs, one per (sequence, head) in flight, through a ring of
 *     packets in L2; the ring takes 8 or more slots of 66 KB per chain (33.8 MB
 *     for 64 units on 152 SMs);
 *   - varlen calls of up to 4096 sequences run the same kernel after a one-CTA
 *     plan (longest sequences first), with the ring and the plan's packet list in
 *     the workspace; varlen calls of more sequences take
 *     KDA_WORKSPACE_BYTES_PER_UNIT bytes per (sequence, head), the per-chunk
 *     operands that move between the two CTAs of a cluster;
 *   - calls of at most 64 token rows need no workspace.
 * A fixed-length call
 * (cu_seqlens == NULL) whose N * H (sequence, head) units would leave most of the
 * GPU idle, with T >= 8192, runs the sequence-parallel path: each sequence is cut
 * into P >= 4 segments of at least 2048 tokens, whose affine state maps are joined
 * by a scan (same results within the stated tolerances, twice the chunk work on P
 * times the parallelism); its scratch, also from the pool, is about
 * N * H * P * (4 * 64 KB + KDA_WORKSPACE_BYTES_PER_UNIT) bytes.
 * kda_fwd_ws is the same call with a caller-provided workspace; for more than 64
 * rows it runs the two-CTA cluster kernel, whose workspace kda_workspace_size gives,
 * or, for fixed-length calls whose workspace holds kda_workspace_size_pool bytes, the
 * persistent pool kernel (never the sequence-parallel path).  Both are asynchronous: they return once the work is enqueued,
 * without synchronising.
 * q/k/v/g/beta/out/A_log/dt_bias/states must be 16-byte aligned.  `out` must not
 * alias an input.
 *
 * Value range: the tensor-core paths (every call of more than one token row) hold v,
 * the recurrent state and the intermediate products U, W, T' and M as fp16 MMA
 * operands (fp32 accumulation), and calls of 2-64 rows also q and k scaled by their
 * decay.  Those values must stay within +-65504.  A call that meets a larger value (or
 * a NaN) sets KDA_ERR_RANGE in the device status word that kda_get_device_status
 * returns, and its outputs are then undefined; the call itself still returns KDA_OK
 * (the check runs on the device).  Calls of one token row (the fp32 token recurrence)
 * have no such limit, nor have kda_fwd_unbounded calls that run its token recurrence
 * (below); its chunked form has the same limit.
 *
 * Returns KDA_OK, or an argument error (nothing enqueued), or KDA_ERR_CUDA if
 * the workspace allocation or the launch failed.
 */
kda_status kda_fwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                   float scale, void *out, const float *A_log, const float *dt_bias,
                   float lower_bound, const void *initial_state, void *final_state,
                   int state_dtype, const int64_t *cu_seqlens, int64_t num_seqs, int64_t B,
                   int64_t T, int64_t H, int64_t K, int64_t V, void *stream);

/* Workspace bytes per (sequence, head): N * H * KDA_WORKSPACE_BYTES_PER_UNIT in
 * total (N = num_seqs with cu_seqlens, else B). */
#define KDA_WORKSPACE_BYTES_PER_UNIT 99328

/* Bytes of the workspace kda_fwd_ws needs for N sequences of H heads (N = num_seqs with
 * cu_seqlens, else B): N * H * KDA_WORKSPACE_BYTES_PER_UNIT.  Returns 0 for negative
 * sizes or a product that does not fit in size_t.  Pure host arithmetic. */
size_t kda_workspace_size(int64_t num_seqs, int64_t H);

/* Bytes of a kda_fwd_ws workspace with which fixed-length calls of more than 64 rows
 * run the persistent pool kernel (its ring of chain packets and their flags) instead
 * of the cluster kernel, on the current device: at least kda_workspace_size, and
 * independent of T.  Varlen calls through kda_fwd_ws keep the cluster kernel.  Queries
 * the current device's SM count; returns 0 for sizes out of range or if that query
 * fails.  A workspace sized on one device is valid on devices with as many SMs. */
size_t kda_workspace_size_pool(int64_t num_seqs, int64_t H);

/*
 * kda_fwd_ws — kda_fwd without any allocation: the caller passes the workspace.
 * Same arguments and semantics as kda_fwd, plus
 *   workspace        device buffer of at least N * H * KDA_WORKSPACE_BYTES_PER_UNIT
 *                    bytes, 16-byte aligned; owned by the caller, read and written
 *                    by the kernel of this call only (its contents on entry do not
 *                    matter and are undefined on exit).  It must not be used by
 *                    another call that can run concurrently (another stream)
 *                    until this call's work on `stream` has completed.  May be
 *                    NULL when the call has no work (N * H == 0).
 *   workspace_bytes  its size in bytes
 * Additional argument errors: KDA_ERR_NULL (NULL workspace with work to do),
 * KDA_ERR_VALUE (workspace_bytes too small), KDA_ERR_ALIGN (misaligned workspace).
 */
kda_status kda_fwd_ws(const void *q, const void *k, const void *v, const void *g, const void *beta,
                      float scale, void *out, const float *A_log, const float *dt_bias,
                      float lower_bound, const void *initial_state, void *final_state,
                      int state_dtype, const int64_t *cu_seqlens, int64_t num_seqs, int64_t B,
                      int64_t T, int64_t H, int64_t K, int64_t V, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * kda_fwd_unbounded — KDA forward with the gate that has no lower bound (the
 * FlashKDA usage notes' safe_gate switched off; the pages give no formula for this
 * gate, the one below is this library's reading):
 *
 *   gk_t[c] = -exp(A_log[h]) * softplus(g_t[c] + dt_bias[h][c]),
 *   softplus(x) = log(1 + exp(x)),
 *
 * a per-token log decay in (-inf, 0) with no floor.  Everything else (norms, beta,
 * the recurrence, scale, states, cu_seqlens) is as for kda_fwd, whose argument list
 * this is without lower_bound.
 * Calls of more than 64 token rows (up to 4096 sequences when varlen) run the chunked
 * tensor-core form of kda_fwd's persistent kernel, with each token's decay factor
 * floored at 2^-14 (about 6.1e-5) per key channel: where the exact factor is smaller,
 * the state that crosses that token keeps at most 6.1e-5 of itself instead of less.
 * Long fixed-length calls with few (sequence, head) units run sequence-parallel as in
 * kda_fwd.  They take a workspace from the same pool as kda_fwd.  Calls of at most 64 rows and
 * larger varlen batches apply the recurrence token by token, exact for any decay,
 * without workspace.  The chunked form holds the same values as fp16 MMA operands as
 * kda_fwd's and reports values beyond +-65504 the same way (KDA_ERR_RANGE in the
 * device status word).  Asynchronous like kda_fwd.  Same argument errors as kda_fwd
 * (no lower_bound check), KDA_ERR_CUDA if the workspace or a launch failed.
 */
kda_status kda_fwd_unbounded(const void *q, const void *k, const void *v, const void *g,
                             const void *beta, float scale, void *out, const float *A_log,
                             const float *dt_bias, const void *initial_state, void *final_state,
                             int state_dtype, const int64_t *cu_seqlens, int64_t num_seqs,
                             int64_t B, int64_t T, int64_t H, int64_t K, int64_t V, void *stream);

/*
 * kda_bwd — gradients of the KDA forward.  The pages ship the forward only (the
 * FlashKDA Q&A, its notes on training); this is the derivative of kda_fwd (or, with
 * `unbounded` nonzero, of kda_fwd_unbounded's exact recurrence) for the scalar loss
 *
 *   L = sum(dout * out) + sum(dfinal * final_state),
 *
 * taken in reverse token order on the fp32 recurrence (states recomputed from
 * checkpoints every 16 tokens), then through the norms, the beta sigmoid and the gate.
 *
 * Inputs: q, k, v, g, beta, scale, A_log, dt_bias, lower_bound (ignored when
 * `unbounded`), initial_state, state_dtype, cu_seqlens, num_seqs, B, T, H, K, V as for
 * kda_fwd (final_state is not an input here); dout bf16 [B,T,H,V], the gradient of
 * out; dfinal fp32 [N,H,V,K] or NULL (zero), the gradient of the final state.
 * Outputs (fp32, contiguous, caller-allocated, every element written):
 *   dq, dk, dg [B,T,H,K]   gradients of q, k and g
 *   dv [B,T,H,V]           gradient of v
 *   dbeta [B,T,H]          gradient of the beta logits
 *   dA_log [H], ddt_bias [H,K]   gradients of A_log and dt_bias (summed over tokens)
 *   dinitial_state [N,H,V,K]     gradient of the initial state, or NULL (not written)
 * Rows of cu_seqlens-packed calls all belong to some sequence, so dq..dbeta are fully
 * written.  Takes a workspace from kda_fwd's pool: the state at the start of every
 * 64-token chunk (64 KB each) plus 4 MB per SM in use.  Asynchronous.  Returns the
 * argument errors of kda_fwd, KDA_ERR_NULL for a missing gradient buffer,
 * KDA_ERR_ALIGN for one not 16-byte aligned, KDA_ERR_CUDA if the workspace or a launch
 * failed.
 */
kda_status kda_bwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                   float scale, const float *A_log, const float *dt_bias, float lower_bound,
                   int unbounded, const void *initial_state, int state_dtype, const void *dout,
                   const float *dfinal, const int64_t *cu_seqlens, int64_t num_seqs, int64_t B,
                   int64_t T, int64_t H, int64_t K, int64_t V, float *dq, float *dk, float *dv,
                   float *dg, float *dbeta, float *dA_log, float *ddt_bias,
                   float *dinitial_state, void *stream);

/* Most (sequence, head) units, N * H, that one kda_fwd_static call may hold. */
#define KDA_STATIC_MAX_UNITS 128

/*
 * kda_fwd_static — kda_fwd for a caller that cannot allocate device memory.
 * The pages describe nothing like it: it exists for callers such as a serving
 * engine that reserves all device memory for its own pool up front (a library's
 * cudaMalloc there fails, or breaks the engine's budget), a plug-in host whose
 * interface hands a plug-in only its input and output buffers, or a request path
 * that must not allocate because an allocation can block or synchronise the device.
 *
 * Same arguments, results and asynchrony as kda_fwd.  The caller passes the inputs
 * and outputs only; the call allocates nothing (no cudaMalloc, cudaMallocAsync or
 * cudaFree, no allocating library routine).  Its scratch is one array of
 * KDA_STATIC_MAX_UNITS * KDA_WORKSPACE_BYTES_PER_UNIT bytes (12,713,984 bytes) in
 * libkda.so's own device memory: every GPU that loads the library holds it until
 * the process exits.  Consequences:
 *   - calls with N * H > KDA_STATIC_MAX_UNITS return KDA_ERR_LIMIT (nothing enqueued);
 *   - every call on a device shares that one array, and calls that can overlap on
 *     the GPU (different streams, without an ordering between them) race on it and
 *     give wrong results: order them, for instance on one stream;
 *   - the array keeps what the last call left in it; the kernels write every part of
 *     it they read within a call before reading it, so nothing needs clearing;
 *   - the first call on a device looks up the array's device address (with that
 *     device current) and caches it: make that first call before any stream capture.
 * It always takes the plain path (no sequence-parallel split), like kda_fwd_ws.
 * Returns what kda_fwd returns, plus KDA_ERR_LIMIT, and KDA_ERR_CUDA when the address
 * lookup fails.
 */
kda_status kda_fwd_static(const void *q, const void *k, const void *v, const void *g,
                          const void *beta, float scale, void *out, const float *A_log,
                          const float *dt_bias, float lower_bound, const void *initial_state,
                          void *final_state, int state_dtype, const int64_t *cu_seqlens,
                          int64_t num_seqs, int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                          void *stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char *kda_status_string(int status);

/*
 * kda_get_device_status — synchronises `stream`, then reads and clears the
 * device-side error word that kernels set when a bounded wait gives up
 * (KDA_ERR_TIMEOUT) or an fp16 operand leaves its range (KDA_ERR_RANGE).  Returns
 * KDA_OK when no kernel reported a problem, the reported code, or KDA_ERR_CUDA if the
 * synchronisation itself failed.
 */
kda_status kda_get_device_status(void *stream);

/* Library ABI version (major * 100 + minor). */
int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
