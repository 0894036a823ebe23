// kda_internal.h -- host-side launchers shared between the C ABI (api.cu) and the
// kernel translation units.  Not part of the public interface (that is include/kda.h).
#pragma once

#include <cuda_runtime.h>

#include "kda.h"
#include <stddef.h>
#include <stdint.h>

namespace kda {

struct FwdArgs {
    const void *q, *k, *v, *beta, *z;
    const float* A_log;
    float g_min;
    const float* S0;
    float* S_out;
    const int32_t* cu_seqlens;
    int N;
    int64_t T_total;
    int H, dk, dv;
    int io_bf16;  // 1: bf16 I/O, 0: fp32 I/O
    int gate_kind;  // 0: g_min Sigmoid(e^A z); 1: -e^A Softplus(z)
    void* o;              // may be nullptr on the tensor-core path (no output stored)
    void* workspace;
    size_t ws_bytes;
    unsigned* dev_err;
    cudaStream_t stream;
    // tensor-core path only, for a backward pass (nullptr otherwise; o must then be nullptr):
    // the backward's image blocks [chunks][H] in the order of the chunk offsets
    // (bwd_tc_layout.cuh), which receive S_0, Vt and N of every chunk; selects the two-launch
    // form, which also leaves every (chunk, head) package in the workspace
    void* bimg;
    // two-launch form, optional: recorded on `stream` once the intra stage is enqueued (the
    // backward starts its gradient chain on a second stream from there)
    cudaEvent_t after_intra;
};

struct BwdArgs {
    const void *q, *k, *v, *beta, *z, *dout;
    const float* A_log;
    float g_min;
    const float* S0;
    const float* dS_out;
    const int32_t* cu_seqlens;
    int N;
    int64_t T_total;
    int H, dk, dv;
    int io_bf16;
    void *dq, *dk_, *dv_, *dbeta, *dz;
    float* dA_log;
    float* dS0;
    void* workspace;
    unsigned* dev_err;
    cudaStream_t stream;
};

// Gradients of the forward (bwd.cu): token-level reverse mode on CUDA cores.
size_t bwd_workspace_size_public(int64_t T_total, int N, int H, int dk, int dv);
cudaError_t launch_bwd(const BwdArgs& a);

// A bounded wait that runs out (selftest.cu): sets the timeout bit of the error word.
cudaError_t launch_selftest_timeout(uint64_t limit_ns, unsigned* err, cudaStream_t stream);

// K1: elementwise gate.
cudaError_t launch_gate(const void* z, int z_bf16, const float* A_log, float g_min, float* g_out,
                        int64_t n_tokens, int H, int dk, cudaStream_t stream);

// K4: one decode token per sequence, state updated in place.
cudaError_t launch_decode(const void* q, const void* k, const void* v, const void* beta,
                          const void* z, const float* A_log, float g_min, float* S, int N, int H,
                          int dk, int dv, int io_bf16, void* o, cudaStream_t stream);

// K4 with the gated output step of "Gated MLA" fused: writes y instead of o.
cudaError_t launch_decode_gated(const void* q, const void* k, const void* v, const void* beta,
                                const void* z, const float* A_log, float g_min, float* S, int N,
                                int H, int dk, int dv, int io_bf16, const void* gate,
                                const float* norm_w, float eps, void* y, cudaStream_t stream);

// The gated output step alone: rows of dv channels (one per token and head).
cudaError_t launch_output_gate(const void* o, const void* gate, const float* norm_w, float eps,
                               void* y, int64_t n_rows, int dv, int io_bf16,
                               cudaStream_t stream);

// Quantile-balancing bias update of the expert router (qb.cu).
size_t qb_workspace_size(int64_t m, int n);
cudaError_t launch_quantile_balance(const float* s, const float* b, int64_t m, int n, int k,
                                    float* b_new, float* bhat, float* alpha, void* workspace,
                                    cudaStream_t stream);

// Chunked forward on CUDA cores in fp32 (any dtype, dk/dv in {64,128}).
cudaError_t launch_fwd_generic(const FwdArgs& a);

// Chunked forward on tcgen05 tensor cores (bf16 I/O, dk = dv = 128); needs a workspace of
// fwd_tc_workspace_size() bytes.
size_t fwd_tc_workspace_size(int64_t T_total, int N, int H);
cudaError_t launch_fwd_tc(const FwdArgs& a);

// The backward's gradient chain on tcgen05 tensor cores (bwd_chain_tc.cu), bf16 problems:
// from the packages that launch_fwd_tc with bimg set left in `fwd_ws`, the state's gradient
// at every chunk end and dVt into the image blocks `bimg`, and a.dS0.
cudaError_t launch_bwd_chain_tc(const BwdArgs& a, void* fwd_ws, void* bimg, cudaStream_t stream);

// The backward's per-chunk kernels on tcgen05 tensor cores (bwd_item_tc.cu), bf16 problems:
// from the image blocks, every gradient but dS0, plus the [chunks][H] dA_log partials; `mid`
// holds the mid blocks between its two kernels.
cudaError_t launch_bwd_items_tc(const BwdArgs& a, void* fwd_ws, const void* bimg, void* mid,
                                float* dA_item, cudaStream_t stream);

// The argument checks of kda_fwd_chunked except those of the workspace (api.cu): KDA_OK, or
// the failing status with the calling thread's last error set.
kda_status_t check_fwd_args(const void* q, const void* k, const void* v, const void* beta,
                            const void* z, const float* A_log, float g_min, const float* S0,
                            float* S_out, const int32_t* cu_seqlens, int N, int64_t T_total,
                            int H, int dk, int dv, kda_dtype_t io_dt, void* o);

// Records `msg` as the calling thread's last error (see kda_last_error) and returns `s`.
kda_status_t set_last_error(kda_status_t s, const char* msg);

// Kernel timing hooks (profile.cu): no-ops unless kda_profile_begin() is active.
int prof_kernel_begin(const char* name, cudaStream_t s);
void prof_kernel_end(int ev, cudaStream_t s);

struct ProfScope {
    int ev;
    cudaStream_t s;
    ProfScope(const char* name, cudaStream_t stream) : ev(prof_kernel_begin(name, stream)), s(stream) {}
    ~ProfScope() { prof_kernel_end(ev, s); }
    ProfScope(const ProfScope&) = delete;
    ProfScope& operator=(const ProfScope&) = delete;
};

}  // namespace kda
