/*
 * kda.h -- C ABI of libkda.so: Kimi Delta Attention (KDA) on one GB300 (sm_103a).
 *
 * The operation (sources cited by page title and section):
 *   [blog]  "Kimi k3 技术报告详解（1）——架构再升华" (stevenstage.github.io/posts/blog7)
 *     section "Kimi Delta Attention" -- the KDA recurrence, per sequence and head:
 *         S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *         o_t = S_t^T q_t                      (S is d_k x d_v, no scale on q)
 *     section "Chunkwise parallel form" -- the same result computed chunk by chunk
 *         (chunk length 64, 16-token sub-tiles) and the lower-bounded gate
 *         g_t = g_min * Sigmoid(e^{A_h} z_t)  in (g_min, 0),   alpha_t = exp(g_t),
 *         which replaces g_t = -e^{A_h} Softplus(z_t)  (kda_fwd_chunked_softplus);
 *     section "Gated MLA" -- the layer output W_o [Sigmoid(W_g x_t) (.) RMSNorm(o~_t)]
 *         (kda_output_norm_gate, kda_decode_step_gated: the part between W_g and W_o);
 *     load-balancing section "Quantile Balancing (QB)" -- the expert-bias update
 *         (kda_quantile_balance).
 *   [guide] "A Look at Kimi K3: Three Core Innovations and Engineering Tuning Guide",
 *     section 2.2 -- the same gate (per head A_h, per channel z), g_min in [-6, -3];
 *     section 4.2 -- quantile-based expert thresholds.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; every pointer must be
 *     16-byte aligned.  No entry point allocates device memory.  Every entry point that
 *     needs scratch takes a caller-provided workspace, except kda_fwd_chunked_noalloc,
 *     whose scratch is a 64 MiB static device buffer inside the library: it occupies
 *     memory on every GPU the library's module is loaded on, from that moment until the
 *     process exits.
 *   - The first call on a device looks up and caches, for that device ordinal, the device
 *     addresses of the library's static device variables (the error word below and the
 *     no-alloc scratch).  Do not reset a device (cudaDeviceReset) after calling into the
 *     library on it: the cached addresses would then be stale.
 *   - Layouts are contiguous row-major with the feature dimension innermost:
 *         q, k, z : [T, H, dk]     v, o : [T, H, dv]     beta : [T, H]
 *         A_log   : [H] fp32       state S : [N, H, dk, dv] fp32 (row = key channel)
 *     where T is the number of tokens (packed over sequences).
 *   - io_dt selects the element type of q, k, v, beta, z and o: KDA_F32 or KDA_BF16.
 *     The recurrent state and all accumulation are fp32.
 *   - dk, dv must be 64 or 128 (KDA_ERR_UNSUPPORTED otherwise); g_min must be < 0.
 *   - Work is enqueued on `stream` (NULL = the legacy default stream) and the call
 *     returns without synchronising.  Argument errors are detected on the host
 *     before anything is enqueued and return KDA_ERR_INVALID_ARG / _UNSUPPORTED;
 *     launch failures return KDA_ERR_CUDA.  Problems only visible on the device
 *     (e.g. malformed cu_seqlens) set a device error word that kda_device_status()
 *     reports.  kda_last_error() gives a readable message for the calling thread.
 *   - Results are deterministic: the same inputs give bitwise identical outputs.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA header. */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, g_min >= 0, ... */
    KDA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. dk = 96)          */
    KDA_ERR_CUDA = 3,         /* a CUDA launch or runtime call failed               */
    KDA_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up                 */
    KDA_ERR_DEVICE = 5        /* the device reported malformed input (cu_seqlens)   */
} kda_status_t;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype_t;

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int kda_version(void);

/* Static name of a status code. */
const char *kda_status_string(kda_status_t status);

/* Message describing the most recent failing call made by this thread ("" if none). */
const char *kda_last_error(void);

/*
 * kda_gate -- the lower-bounded decay gate alone ([blog] "Chunkwise parallel form",
 * [guide] 2.2):  g_out[t,h,c] = g_min * Sigmoid(exp(A_log[h]) * z[t,h,c]).
 *   z      : [n_tokens, H, dk] of z_dt        A_log : [H] fp32
 *   g_out  : [n_tokens, H, dk] fp32 (written)
 * dk may be any positive multiple of 4 here.  n_tokens = 0 is a no-op.
 */
kda_status_t kda_gate(const void *z, kda_dtype_t z_dt, const float *A_log, float g_min,
                      float *g_out, int64_t n_tokens, int H, int dk, kda_stream_t stream);

/*
 * Bytes of device workspace kda_fwd_chunked needs for this problem shape (0 when the
 * selected kernels need none: fp32 I/O).  T_total is the packed token count, N the number of
 * sequences.  Safe to call without a GPU.
 */
size_t kda_fwd_workspace_size(int64_t T_total, int N, int H, int dk, int dv,
                              kda_dtype_t io_dt);

/*
 * kda_fwd_chunked -- KDA forward over N packed sequences in the chunkwise-parallel form
 * ([blog] "Chunkwise parallel form"; chunk length 64).
 *   q, k, z     : [T_total, H, dk]   io_dt
 *   v           : [T_total, H, dv]   io_dt
 *   beta        : [T_total, H]       io_dt
 *   A_log       : [H] fp32, g_min < 0
 *   S0          : [N, H, dk, dv] fp32 initial state, or NULL for zeros
 *   S_out       : [N, H, dk, dv] fp32 final state (written), or NULL; may alias S0
 *   cu_seqlens  : device int32 [N + 1] token offsets (cu[0] = 0, nondecreasing,
 *                 cu[N] = T_total), or NULL for N equal sequences of T_total / N tokens
 *   o           : [T_total, H, dv] io_dt output (written)
 *   workspace   : device scratch of at least kda_fwd_workspace_size(...) bytes
 *                 (may be NULL when that size is 0); its contents are not preserved.
 * A sequence may be empty; chunks never cross a sequence boundary.  With cu_seqlens
 * malformed on the device the affected sequences are skipped and kda_device_status()
 * returns KDA_ERR_DEVICE.
 */
kda_status_t kda_fwd_chunked(const void *q, const void *k, const void *v, const void *beta,
                             const void *z, const float *A_log, float g_min, const float *S0,
                             float *S_out, const int32_t *cu_seqlens, int N, int64_t T_total,
                             int H, int dk, int dv, kda_dtype_t io_dt, void *o,
                             void *workspace, size_t ws_bytes, kda_stream_t stream);

/*
 * kda_fwd_chunked_softplus -- the same chunked forward with the gate the bound replaces
 * ([blog] "Chunkwise parallel form"): g = -e^{A_log[h]} Softplus(z), unbounded below, so a
 * sub-tile's decay can leave the exponent range and no decay factor of a diagonal sub-tile
 * splits into a bounded row factor and column factor.  A comparison variant: it measures
 * what the bound buys.  bf16 runs the mixed path the page describes: the off-diagonal
 * 16-token sub-tile pairs on the tensor cores with sub-tile-start references (every factor
 * <= 1), the diagonal 16 x 16 blocks per pair on CUDA cores (e^{G_r - G_i}, exponent <= 0,
 * in fp32).  fp32 runs the explicit per-pair path (every pair on CUDA cores).  Arguments as kda_fwd_chunked without g_min; the workspace is sized
 * by kda_fwd_workspace_size (0 bytes, and workspace may be NULL, on the explicit path).
 * z must be finite or -inf.
 */
kda_status_t kda_fwd_chunked_softplus(const void *q, const void *k, const void *v,
                                      const void *beta, const void *z, const float *A_log,
                                      const float *S0, float *S_out, const int32_t *cu_seqlens,
                                      int N, int64_t T_total, int H, int dk, int dv,
                                      kda_dtype_t io_dt, void *o, void *workspace,
                                      size_t ws_bytes, kda_stream_t stream);

/*
 * kda_bwd -- gradients of kda_fwd_chunked's outputs ([blog] "Kimi Delta Attention": the
 * derivatives of the recurrence the page defines; the pages print no backward).  For a loss
 * with gradient dout [T_total, H, dv] io_dt on o and dS_out [N, H, dk, dv] fp32 (or NULL) on
 * S_out, writes
 *   dq, dk, dz : [T_total, H, dk] io_dt     dv : [T_total, H, dv] io_dt
 *   dbeta      : [T_total, H] io_dt         dA_log : [H] fp32 (summed over sequences)
 *   dS0        : [N, H, dk, dv] fp32, or NULL when not wanted
 * Other arguments as kda_fwd_chunked (same inputs, S0 may be NULL).
 * bf16 problems (dk, dv in {64, 128}) take the chunk form on the tcgen05 tensor cores: the
 * tensor-core forward (its chunk packages kept) and a reversed chain give the state and its
 * gradient at every chunk boundary as bf16 operand images, then two per-chunk kernels form
 * every gradient.  fp32 problems run on CUDA cores in fp32, parallel over chunks: every
 * chunk's forward and backward maps on the state are formed at once, two short chains give
 * the state and its gradient at every chunk boundary, and every (chunk, head) applies the
 * reverse rules token by token.  The workspace (kda_bwd_workspace_size bytes, the larger of
 * the two layouts) holds those per-(chunk, head) blocks.  Correct for every shape
 * kda_fwd_chunked takes.  Deterministic.
 */
size_t kda_bwd_workspace_size(int64_t T_total, int N, int H, int dk, int dv);
kda_status_t kda_bwd(const void *q, const void *k, const void *v, const void *beta,
                     const void *z, const float *A_log, float g_min, const float *S0,
                     const int32_t *cu_seqlens, int N, int64_t T_total, int H, int dk, int dv,
                     kda_dtype_t io_dt, const void *dout, const float *dS_out, void *dq,
                     void *dk_out, void *dv_out, void *dbeta, void *dz, float *dA_log,
                     float *dS0, void *workspace, size_t ws_bytes, kda_stream_t stream);

/*
 * kda_decode_step -- one token of the KDA recurrence ([blog] "Kimi Delta Attention")
 * for N independent sequences, updating the state in place:
 *   alpha = exp(g_min * Sigmoid(exp(A_log[h]) z));  S <- Diag(alpha) S;
 *   u = beta (v - S^T k);  S <- S + k u^T;  o = S^T q.
 *   q, k, z : [N, H, dk] io_dt    v : [N, H, dv] io_dt    beta : [N, H] io_dt
 *   S       : [N, H, dk, dv] fp32, read and overwritten
 *   o       : [N, H, dv] io_dt (written)
 */
kda_status_t kda_decode_step(const void *q, const void *k, const void *v, const void *beta,
                             const void *z, const float *A_log, float g_min, float *S, int N,
                             int H, int dk, int dv, kda_dtype_t io_dt, void *o,
                             kda_stream_t stream);

/*
 * kda_output_norm_gate -- the gated output step of [blog] section "Gated MLA", whose layer
 * output is y_t = W_o [Sigmoid(W_g x_t) (.) RMSNorm(o~_t)]: the part between the two
 * projections (which need trained weights), per (token, head) row of dv channels:
 *     y[t,h,j] = Sigmoid(gate[t,h,j]) * norm_w[j] * o[t,h,j] / sqrt(mean_j o[t,h,j]^2 + eps)
 *   o, gate : [n_tokens, H, dv] io_dt; gate is W_g x_t, computed by the caller
 *   norm_w  : [dv] fp32 weight of the norm, or NULL for ones
 *   eps     : finite and >= 0, added to the mean square
 *   y       : [n_tokens, H, dv] io_dt (written); may be the same buffer as o
 * dv must be 64 or 128.  n_tokens = 0 is a no-op.
 */
kda_status_t kda_output_norm_gate(const void *o, const void *gate, const float *norm_w,
                                  float eps, void *y, int64_t n_tokens, int H, int dv,
                                  kda_dtype_t io_dt, kda_stream_t stream);

/*
 * kda_decode_step_gated -- kda_decode_step with the gated output step fused into it: the
 * state update is the same, and in place of o the call writes, per (sequence, head),
 *     y = Sigmoid(gate) * norm_w * o / sqrt(mean(o^2) + eps)        (as kda_output_norm_gate)
 * so o never reaches memory.
 *   gate   : [N, H, dv] io_dt        norm_w : [dv] fp32 or NULL        eps : finite, >= 0
 *   y      : [N, H, dv] io_dt (written)
 * Other arguments and rules as kda_decode_step.
 */
kda_status_t kda_decode_step_gated(const void *q, const void *k, const void *v,
                                   const void *beta, const void *z, const float *A_log,
                                   float g_min, float *S, const void *gate, const float *norm_w,
                                   float eps, int N, int H, int dk, int dv, kda_dtype_t io_dt,
                                   void *y, kda_stream_t stream);

/*
 * kda_quantile_balance -- quantile-balancing update of a mixture-of-experts router's expert
 * biases ([blog] section "Quantile Balancing (QB)"; [guide] section 4.2):
 *     alpha_i   = the (k+1)-th largest of scores[i,:] + bias          (token threshold)
 *     margin_ij = scores[i,j] - alpha_i
 *     bhat_j    = -(the (q+1)-th largest of margin[:,j]),  q = floor(m k / n)
 *                 (expert j would then receive exactly q tokens)
 *     bias_new  = bhat - mean(bhat)
 * s + bias and the margins are formed in fp32 and the selections are exact, so alpha and
 * bhat are bitwise reproducible; equal values count separately ("(q+1)-th largest" of the
 * sorted list).
 *   scores    : [m, n] fp32 device, row-major (token-major)       bias : [n] fp32
 *   k         : experts per token, 0 <= k < n;   1 <= n <= 1024;   1 <= m < 2^31
 *   bias_new  : [n] fp32 (written)
 *   bhat, alpha : [n] and [m] fp32 outputs, or NULL when not wanted
 *   workspace : device scratch of kda_quantile_balance_workspace_size(m, n) bytes
 */
size_t kda_quantile_balance_workspace_size(int64_t m, int n);
kda_status_t kda_quantile_balance(const float *scores, const float *bias, int64_t m, int n,
                                  int k, float *bias_new, float *bhat, float *alpha,
                                  void *workspace, size_t ws_bytes, kda_stream_t stream);

/*
 * kda_selftest_timeout -- the failure path of the bounded device waits, without a fault:
 * enqueues a kernel that waits on an mbarrier nothing ever arrives on, gives up after
 * limit_us microseconds (1 .. 2e6), sets the timeout bit of the device error word and
 * returns, exactly as the library's kernels do when a wait runs out.  The next
 * kda_device_status() on the stream then returns KDA_ERR_TIMEOUT (and clears the word).
 * Not part of the method; a diagnostic of the error reporting.
 */
kda_status_t kda_selftest_timeout(unsigned limit_us, kda_stream_t stream);

/*
 * Waits for `stream`, then reads and clears the device error word that kernels set
 * when they meet malformed device-side input or give up a bounded wait.  Returns
 * KDA_OK, KDA_ERR_DEVICE or KDA_ERR_TIMEOUT (or KDA_ERR_CUDA if the wait failed).
 */
kda_status_t kda_device_status(kda_stream_t stream);

/*
 * kda_fwd_chunked_noalloc -- the same forward as kda_fwd_chunked for callers that must not
 * allocate device memory (a runtime that owns every byte of GPU memory, a plugin that may
 * not call the CUDA allocator, code where an allocation would synchronise the device).  The
 * pages have no counterpart: this is an interface convenience.
 * Arguments are those of kda_fwd_chunked without the workspace.  Scratch comes from a 64 MiB
 * buffer compiled into the library, which every GPU that loads the library holds until the
 * process exits; problems whose kda_fwd_workspace_size() exceeds 64 MiB are rejected with
 * KDA_ERR_INVALID_ARG (nothing is launched).  No call allocates memory.
 *  - The first call on a device looks up the buffer's device address (cudaGetSymbolAddress);
 *    make that first call before any stream capture.
 *  - All calls share the one buffer, which keeps the last call's contents; nothing in it
 *    has to start at zero (every byte a call reads it has first written).  Calls whose
 *    execution overlaps on the GPU (other streams, other threads) race on the buffer:
 *    serialise them.
 */
kda_status_t kda_fwd_chunked_noalloc(const void *q, const void *k, const void *v,
                                     const void *beta, const void *z, const float *A_log,
                                     float g_min, const float *S0, float *S_out,
                                     const int32_t *cu_seqlens, int N, int64_t T_total, int H,
                                     int dk, int dv, kda_dtype_t io_dt, void *o,
                                     kda_stream_t stream);

/*
 * Per-kernel timing (tracing aid; not part of the method).  After kda_profile_begin(),
 * every kernel the library launches is bracketed by two CUDA events recorded on the
 * launching stream.  kda_profile_end() waits for those events, stops recording and fills
 * `entries` with one record per kernel name (number of launches, summed device time in
 * ms); it returns the number of records written, or -1 if a CUDA event call failed.
 * Host-side state is process-wide; calls from several threads are serialised.
 */
typedef struct {
    char name[32];
    int launches;
    double total_ms;
} kda_profile_entry_t;

kda_status_t kda_profile_begin(void);
int kda_profile_end(kda_profile_entry_t *entries, int max_entries);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
