// api.cu -- the C ABI of libkda.so (declared in include/kda.h): argument checks,
// kernel selection and the device error word.  No entry point allocates device memory.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "kda.h"
#include "kda_common.cuh"
#include "kda_internal.h"

namespace {

__device__ unsigned g_device_error = 0u;

thread_local std::string t_last_error;

kda_status_t fail(kda_status_t s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
kda_status_t fail(kda_status_t s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

kda_status_t cuda_fail(cudaError_t e, const char* where) {
    return fail(KDA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define KDA_REQUIRE(cond, ...)                                   \
    do {                                                         \
        if (!(cond)) return fail(KDA_ERR_INVALID_ARG, __VA_ARGS__); \
    } while (0)

#define KDA_REQUIRE_PTR(p, name)                                                   \
    do {                                                                           \
        if ((p) == nullptr) return fail(KDA_ERR_INVALID_ARG, "%s is NULL", name);  \
        if (!aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name); \
    } while (0)

#define KDA_OPTIONAL_PTR(p, name)                                                  \
    do {                                                                           \
        if ((p) != nullptr && !aligned16(p))                                       \
            return fail(KDA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);   \
    } while (0)

// Device address of the error word on the current device (looked up once per device).
unsigned* device_error_ptr() {
    static std::mutex mu;
    static unsigned* cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<unsigned*>(p);
    }
    return cache[dev];
}

kda_status_t check_dims(int dk, int dv) {
    if (dk <= 0 || dv <= 0) return fail(KDA_ERR_INVALID_ARG, "dk=%d dv=%d must be positive", dk, dv);
    if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128))
        return fail(KDA_ERR_UNSUPPORTED, "dk=%d dv=%d: only 64 and 128 are supported", dk, dv);
    return KDA_OK;
}

kda_status_t check_gmin(float g_min) {
    if (!(g_min < 0.f) || !std::isfinite(g_min))
        return fail(KDA_ERR_INVALID_ARG, "g_min=%g must be finite and negative", (double)g_min);
    return KDA_OK;
}

}  // namespace

namespace kda {
kda_status_t set_last_error(kda_status_t s, const char* msg) {
    t_last_error = msg;
    return s;
}
}  // namespace kda

extern "C" {

int kda_version(void) { return 200; /* 0.2.0: backward, softplus variant, output step, quantile balancing */ }

const char* kda_status_string(kda_status_t s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        case KDA_ERR_DEVICE: return "KDA_ERR_DEVICE";
    }
    return "KDA_ERR_UNKNOWN";
}

const char* kda_last_error(void) { return t_last_error.c_str(); }

kda_status_t kda_gate(const void* z, kda_dtype_t z_dt, const float* A_log, float g_min,
                      float* g_out, int64_t n_tokens, int H, int dk, kda_stream_t stream) {
    t_last_error.clear();
    KDA_REQUIRE(z_dt == KDA_F32 || z_dt == KDA_BF16, "z_dt=%d is not a kda_dtype_t", (int)z_dt);
    KDA_REQUIRE(n_tokens >= 0, "n_tokens=%lld must be >= 0", (long long)n_tokens);
    KDA_REQUIRE(H > 0, "H=%d must be positive", H);
    KDA_REQUIRE(dk > 0 && dk % 4 == 0, "dk=%d must be a positive multiple of 4", dk);
    if (kda_status_t s = check_gmin(g_min)) return s;
    if (n_tokens == 0) return KDA_OK;
    KDA_REQUIRE_PTR(z, "z");
    KDA_REQUIRE_PTR(A_log, "A_log");
    KDA_REQUIRE_PTR(g_out, "g_out");
    cudaError_t e = kda::launch_gate(z, z_dt == KDA_BF16, A_log, g_min, g_out, n_tokens, H, dk,
                                     reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kda_gate launch");
    return KDA_OK;
}

// Which forward kernels a problem takes: bf16 I/O the tensor-core path at every head size
// (a 64 runs zero-padded to 128), fp32 I/O the fp32 CUDA-core path.  KDA_FWD_PATH=generic
// in the environment forces the CUDA-core path (the tests use it to cross-check the two).
static bool use_tc_path(int dk, int dv, kda_dtype_t io_dt) {
    if (io_dt != KDA_BF16 || (dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return false;
    const char* env = getenv("KDA_FWD_PATH");
    return !(env && strcmp(env, "generic") == 0);
}

size_t kda_fwd_workspace_size(int64_t T_total, int N, int H, int dk, int dv, kda_dtype_t io_dt) {
    if (T_total < 0 || N < 0 || H <= 0) return 0;
    if (!use_tc_path(dk, dv, io_dt)) return 0;
    return kda::fwd_tc_workspace_size(T_total, N, H);
}

}  // extern "C"

namespace kda {
// The argument checks of kda_fwd_chunked other than the workspace ones (shared with
// kda_fwd_chunked_noalloc, which must report a malformed call before anything else).
kda_status_t check_fwd_args(const void* q, const void* k, const void* v, const void* beta,
                            const void* z, const float* A_log, float g_min, const float* S0,
                            float* S_out, const int32_t* cu_seqlens, int N, int64_t T_total,
                            int H, int dk, int dv, kda_dtype_t io_dt, void* o) {
    KDA_REQUIRE(io_dt == KDA_F32 || io_dt == KDA_BF16, "io_dt=%d is not a kda_dtype_t", (int)io_dt);
    KDA_REQUIRE(N >= 0, "N=%d must be >= 0", N);
    KDA_REQUIRE(H > 0, "H=%d must be positive", H);
    KDA_REQUIRE(T_total >= 0, "T_total=%lld must be >= 0", (long long)T_total);
    if (kda_status_t s = check_dims(dk, dv)) return s;
    if (kda_status_t s = check_gmin(g_min)) return s;
    if (cu_seqlens == nullptr) {
        KDA_REQUIRE(N > 0 || T_total == 0, "N=0 requires T_total=0");
        KDA_REQUIRE(N == 0 || T_total % N == 0,
                    "without cu_seqlens T_total=%lld must be a multiple of N=%d",
                    (long long)T_total, N);
    }
    KDA_REQUIRE((int64_t)N * H * 4 < (int64_t)1 << 31, "N*H=%lld is too large",
                (long long)N * H);
    if (N == 0) return KDA_OK;
    if (T_total > 0) {
        KDA_REQUIRE_PTR(q, "q");
        KDA_REQUIRE_PTR(k, "k");
        KDA_REQUIRE_PTR(v, "v");
        KDA_REQUIRE_PTR(z, "z");
        KDA_REQUIRE_PTR(o, "o");
        KDA_REQUIRE(beta != nullptr, "beta is NULL");
    }
    KDA_REQUIRE_PTR(A_log, "A_log");
    KDA_OPTIONAL_PTR(S0, "S0");
    KDA_OPTIONAL_PTR(S_out, "S_out");
    KDA_OPTIONAL_PTR(cu_seqlens, "cu_seqlens");
    return KDA_OK;
}
}  // namespace kda

extern "C" {

kda_status_t kda_fwd_chunked(const void* q, const void* k, const void* v, const void* beta,
                             const void* z, const float* A_log, float g_min, const float* S0,
                             float* S_out, const int32_t* cu_seqlens, int N, int64_t T_total,
                             int H, int dk, int dv, kda_dtype_t io_dt, void* o, void* workspace,
                             size_t ws_bytes, kda_stream_t stream) {
    t_last_error.clear();
    if (kda_status_t s = kda::check_fwd_args(q, k, v, beta, z, A_log, g_min, S0, S_out,
                                             cu_seqlens, N, T_total, H, dk, dv, io_dt, o))
        return s;
    if (N == 0) return KDA_OK;
    const size_t need = kda_fwd_workspace_size(T_total, N, H, dk, dv, io_dt);
    if (need > 0) {
        KDA_REQUIRE_PTR(workspace, "workspace");
        KDA_REQUIRE(ws_bytes >= need, "workspace of %zu bytes is smaller than the %zu needed",
                    ws_bytes, need);
    }

    kda::FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.z = z;
    a.A_log = A_log; a.g_min = g_min; a.S0 = S0; a.S_out = S_out;
    a.cu_seqlens = cu_seqlens; a.N = N; a.T_total = T_total; a.H = H; a.dk = dk; a.dv = dv;
    a.io_bf16 = (io_dt == KDA_BF16); a.o = o; a.workspace = workspace; a.ws_bytes = ws_bytes;
    a.dev_err = device_error_ptr();
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    if (a.dev_err == nullptr) return fail(KDA_ERR_CUDA, "no CUDA device is usable");
    cudaError_t e =
        use_tc_path(dk, dv, io_dt) ? kda::launch_fwd_tc(a) : kda::launch_fwd_generic(a);
    if (e != cudaSuccess) return cuda_fail(e, "kda_fwd_chunked launch");
    return KDA_OK;
}

kda_status_t kda_fwd_chunked_softplus(const void* q, const void* k, const void* v,
                                      const void* beta, const void* z, const float* A_log,
                                      const float* S0, float* S_out, const int32_t* cu_seqlens,
                                      int N, int64_t T_total, int H, int dk, int dv,
                                      kda_dtype_t io_dt, void* o, void* workspace,
                                      size_t ws_bytes, kda_stream_t stream) {
    t_last_error.clear();
    KDA_REQUIRE(io_dt == KDA_F32 || io_dt == KDA_BF16, "io_dt=%d is not a kda_dtype_t", (int)io_dt);
    KDA_REQUIRE(N >= 0, "N=%d must be >= 0", N);
    KDA_REQUIRE(H > 0, "H=%d must be positive", H);
    KDA_REQUIRE(T_total >= 0, "T_total=%lld must be >= 0", (long long)T_total);
    if (kda_status_t s = check_dims(dk, dv)) return s;
    if (cu_seqlens == nullptr) {
        KDA_REQUIRE(N > 0 || T_total == 0, "N=0 requires T_total=0");
        KDA_REQUIRE(N == 0 || T_total % N == 0,
                    "without cu_seqlens T_total=%lld must be a multiple of N=%d",
                    (long long)T_total, N);
    }
    KDA_REQUIRE((int64_t)N * H * 4 < (int64_t)1 << 31, "N*H=%lld is too large",
                (long long)N * H);
    if (N == 0) return KDA_OK;
    if (T_total > 0) {
        KDA_REQUIRE_PTR(q, "q");
        KDA_REQUIRE_PTR(k, "k");
        KDA_REQUIRE_PTR(v, "v");
        KDA_REQUIRE_PTR(z, "z");
        KDA_REQUIRE_PTR(o, "o");
        KDA_REQUIRE(beta != nullptr, "beta is NULL");
    }
    KDA_REQUIRE_PTR(A_log, "A_log");
    KDA_OPTIONAL_PTR(S0, "S0");
    KDA_OPTIONAL_PTR(S_out, "S_out");
    KDA_OPTIONAL_PTR(cu_seqlens, "cu_seqlens");
    const size_t need = kda_fwd_workspace_size(T_total, N, H, dk, dv, io_dt);
    if (need > 0) {
        KDA_REQUIRE_PTR(workspace, "workspace");
        KDA_REQUIRE(ws_bytes >= need, "workspace of %zu bytes is smaller than the %zu needed",
                    ws_bytes, need);
    }
    kda::FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.z = z;
    a.A_log = A_log; a.g_min = -1.f; a.S0 = S0; a.S_out = S_out;
    a.cu_seqlens = cu_seqlens; a.N = N; a.T_total = T_total; a.H = H; a.dk = dk; a.dv = dv;
    a.io_bf16 = (io_dt == KDA_BF16); a.gate_kind = 1; a.o = o;
    a.workspace = workspace; a.ws_bytes = ws_bytes;
    a.dev_err = device_error_ptr();
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    if (a.dev_err == nullptr) return fail(KDA_ERR_CUDA, "no CUDA device is usable");
    // bf16: the mixed path (tensor cores off the diagonal sub-tiles); fp32: the explicit
    // per-pair path
    cudaError_t e =
        use_tc_path(dk, dv, io_dt) ? kda::launch_fwd_tc(a) : kda::launch_fwd_generic(a);
    if (e != cudaSuccess) return cuda_fail(e, "kda_fwd_chunked_softplus launch");
    return KDA_OK;
}

size_t kda_bwd_workspace_size(int64_t T_total, int N, int H, int dk, int dv) {
    if (T_total < 0 || N <= 0 || H <= 0 || check_dims(dk, dv) != KDA_OK) return 0;
    return kda::bwd_workspace_size_public(T_total, N, H, dk, dv);
}

kda_status_t kda_bwd(const void* q, const void* k, const void* v, const void* beta,
                     const void* z, const float* A_log, float g_min, const float* S0,
                     const int32_t* cu_seqlens, int N, int64_t T_total, int H, int dk, int dv,
                     kda_dtype_t io_dt, const void* dout, const float* dS_out, void* dq,
                     void* dk_out, void* dv_out, void* dbeta, void* dz, float* dA_log,
                     float* dS0, void* workspace, size_t ws_bytes, kda_stream_t stream) {
    t_last_error.clear();
    KDA_REQUIRE(io_dt == KDA_F32 || io_dt == KDA_BF16, "io_dt=%d is not a kda_dtype_t", (int)io_dt);
    KDA_REQUIRE(N > 0, "N=%d must be positive", N);
    KDA_REQUIRE(H > 0, "H=%d must be positive", H);
    KDA_REQUIRE(T_total >= 0, "T_total=%lld must be >= 0", (long long)T_total);
    if (kda_status_t s = check_dims(dk, dv)) return s;
    if (kda_status_t s = check_gmin(g_min)) return s;
    if (cu_seqlens == nullptr)
        KDA_REQUIRE(T_total % N == 0, "without cu_seqlens T_total=%lld must be a multiple of N=%d",
                    (long long)T_total, N);
    KDA_REQUIRE((int64_t)N * H < (int64_t)1 << 31, "N*H=%lld is too large", (long long)N * H);
    if (T_total > 0) {
        KDA_REQUIRE_PTR(q, "q");
        KDA_REQUIRE_PTR(k, "k");
        KDA_REQUIRE_PTR(v, "v");
        KDA_REQUIRE_PTR(z, "z");
        KDA_REQUIRE_PTR(dout, "dout");
        KDA_REQUIRE_PTR(dq, "dq");
        KDA_REQUIRE_PTR(dk_out, "dk");
        KDA_REQUIRE_PTR(dv_out, "dv");
        KDA_REQUIRE_PTR(dz, "dz");
        KDA_REQUIRE(beta != nullptr, "beta is NULL");
        KDA_REQUIRE(dbeta != nullptr, "dbeta is NULL");
    }
    KDA_REQUIRE_PTR(A_log, "A_log");
    KDA_REQUIRE_PTR(dA_log, "dA_log");
    KDA_OPTIONAL_PTR(S0, "S0");
    KDA_OPTIONAL_PTR(dS_out, "dS_out");
    KDA_OPTIONAL_PTR(dS0, "dS0");
    KDA_OPTIONAL_PTR(cu_seqlens, "cu_seqlens");
    const size_t need = kda::bwd_workspace_size_public(T_total, N, H, dk, dv);
    KDA_REQUIRE_PTR(workspace, "workspace");
    KDA_REQUIRE(ws_bytes >= need, "workspace of %zu bytes is smaller than the %zu needed",
                ws_bytes, need);
    kda::BwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.z = z; a.dout = dout;
    a.A_log = A_log; a.g_min = g_min; a.S0 = S0; a.dS_out = dS_out; a.cu_seqlens = cu_seqlens;
    a.N = N; a.T_total = T_total; a.H = H; a.dk = dk; a.dv = dv; a.io_bf16 = io_dt == KDA_BF16;
    a.dq = dq; a.dk_ = dk_out; a.dv_ = dv_out; a.dbeta = dbeta; a.dz = dz; a.dA_log = dA_log;
    a.dS0 = dS0; a.workspace = workspace; a.dev_err = device_error_ptr();
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    if (a.dev_err == nullptr) return fail(KDA_ERR_CUDA, "no CUDA device is usable");
    cudaError_t e = kda::launch_bwd(a);
    if (e != cudaSuccess) return cuda_fail(e, "kda_bwd launch");
    return KDA_OK;
}

kda_status_t kda_decode_step(const void* q, const void* k, const void* v, const void* beta,
                             const void* z, const float* A_log, float g_min, float* S, int N,
                             int H, int dk, int dv, kda_dtype_t io_dt, void* o,
                             kda_stream_t stream) {
    t_last_error.clear();
    KDA_REQUIRE(io_dt == KDA_F32 || io_dt == KDA_BF16, "io_dt=%d is not a kda_dtype_t", (int)io_dt);
    KDA_REQUIRE(N >= 0, "N=%d must be >= 0", N);
    KDA_REQUIRE(H > 0, "H=%d must be positive", H);
    if (kda_status_t s = check_dims(dk, dv)) return s;
    if (kda_status_t s = check_gmin(g_min)) return s;
    KDA_REQUIRE((int64_t)N * H < (int64_t)1 << 31, "N*H=%lld is too large", (long long)N * H);
    if (N == 0) return KDA_OK;
    KDA_REQUIRE_PTR(q, "q");
    KDA_REQUIRE_PTR(k, "k");
    KDA_REQUIRE_PTR(v, "v");
    KDA_REQUIRE_PTR(z, "z");
    KDA_REQUIRE_PTR(o, "o");
    KDA_REQUIRE_PTR(S, "S");
    KDA_REQUIRE_PTR(A_log, "A_log");
    KDA_REQUIRE(beta != nullptr, "beta is NULL");
    cudaError_t e = kda::launch_decode(q, k, v, beta, z, A_log, g_min, S, N, H, dk, dv,
                                       io_dt == KDA_BF16, o,
                                       reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kda_decode_step launch");
    return KDA_OK;
}

kda_status_t kda_output_norm_gate(const void* o, const void* gate, const float* norm_w,
                                  float eps, void* y, int64_t n_tokens, int H, int dv,
                                  kda_dtype_t io_dt, kda_stream_t stream) {
    t_last_error.clear();
    KDA_REQUIRE(io_dt == KDA_F32 || io_dt == KDA_BF16, "io_dt=%d is not a kda_dtype_t", (int)io_dt);
    KDA_REQUIRE(n_tokens >= 0, "n_tokens=%lld must be >= 0", (long long)n_tokens);
    KDA_REQUIRE(H > 0, "H=%d must be positive", H);
    KDA_REQUIRE(dv > 0, "dv=%d must be positive", dv);
    if (dv != 64 && dv != 128) return fail(KDA_ERR_UNSUPPORTED, "dv=%d: only 64 and 128 are supported", dv);
    KDA_REQUIRE(eps >= 0.f && std::isfinite(eps), "eps=%g must be finite and >= 0", (double)eps);
    if (n_tokens == 0) return KDA_OK;
    KDA_REQUIRE_PTR(o, "o");
    KDA_REQUIRE_PTR(gate, "gate");
    KDA_REQUIRE_PTR(y, "y");
    KDA_OPTIONAL_PTR(norm_w, "norm_w");
    cudaError_t e = kda::launch_output_gate(o, gate, norm_w, eps, y, n_tokens * H, dv,
                                            io_dt == KDA_BF16,
                                            reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kda_output_norm_gate launch");
    return KDA_OK;
}

kda_status_t kda_decode_step_gated(const void* q, const void* k, const void* v,
                                   const void* beta, const void* z, const float* A_log,
                                   float g_min, float* S, const void* gate, const float* norm_w,
                                   float eps, int N, int H, int dk, int dv, kda_dtype_t io_dt,
                                   void* y, kda_stream_t stream) {
    t_last_error.clear();
    KDA_REQUIRE(io_dt == KDA_F32 || io_dt == KDA_BF16, "io_dt=%d is not a kda_dtype_t", (int)io_dt);
    KDA_REQUIRE(N >= 0, "N=%d must be >= 0", N);
    KDA_REQUIRE(H > 0, "H=%d must be positive", H);
    if (kda_status_t s = check_dims(dk, dv)) return s;
    if (kda_status_t s = check_gmin(g_min)) return s;
    KDA_REQUIRE(eps >= 0.f && std::isfinite(eps), "eps=%g must be finite and >= 0", (double)eps);
    KDA_REQUIRE((int64_t)N * H < (int64_t)1 << 31, "N*H=%lld is too large", (long long)N * H);
    if (N == 0) return KDA_OK;
    KDA_REQUIRE_PTR(q, "q");
    KDA_REQUIRE_PTR(k, "k");
    KDA_REQUIRE_PTR(v, "v");
    KDA_REQUIRE_PTR(z, "z");
    KDA_REQUIRE_PTR(gate, "gate");
    KDA_REQUIRE_PTR(y, "y");
    KDA_REQUIRE_PTR(S, "S");
    KDA_REQUIRE_PTR(A_log, "A_log");
    KDA_OPTIONAL_PTR(norm_w, "norm_w");
    KDA_REQUIRE(beta != nullptr, "beta is NULL");
    cudaError_t e = kda::launch_decode_gated(q, k, v, beta, z, A_log, g_min, S, N, H, dk, dv,
                                             io_dt == KDA_BF16, gate, norm_w, eps, y,
                                             reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kda_decode_step_gated launch");
    return KDA_OK;
}

size_t kda_quantile_balance_workspace_size(int64_t m, int n) {
    if (m <= 0 || n <= 0) return 0;
    return kda::qb_workspace_size(m, n);
}

kda_status_t kda_quantile_balance(const float* scores, const float* bias, int64_t m, int n,
                                  int k, float* bias_new, float* bhat, float* alpha,
                                  void* workspace, size_t ws_bytes, kda_stream_t stream) {
    t_last_error.clear();
    KDA_REQUIRE(m >= 1 && m < ((int64_t)1 << 31), "m=%lld must be in [1, 2^31)", (long long)m);
    KDA_REQUIRE(n >= 1 && n <= 1024, "n=%d must be in [1, 1024]", n);
    KDA_REQUIRE(k >= 0 && k < n, "k=%d must satisfy 0 <= k < n=%d", k, n);
    KDA_REQUIRE_PTR(scores, "scores");
    KDA_REQUIRE_PTR(bias, "bias");
    KDA_REQUIRE_PTR(bias_new, "bias_new");
    KDA_OPTIONAL_PTR(bhat, "bhat");
    KDA_OPTIONAL_PTR(alpha, "alpha");
    const size_t need = kda::qb_workspace_size(m, n);
    KDA_REQUIRE_PTR(workspace, "workspace");
    KDA_REQUIRE(ws_bytes >= need, "workspace of %zu bytes is smaller than the %zu needed",
                ws_bytes, need);
    cudaError_t e = kda::launch_quantile_balance(scores, bias, m, n, k, bias_new, bhat, alpha,
                                                 workspace,
                                                 reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kda_quantile_balance launch");
    return KDA_OK;
}

kda_status_t kda_selftest_timeout(unsigned limit_us, kda_stream_t stream) {
    t_last_error.clear();
    KDA_REQUIRE(limit_us >= 1 && limit_us <= 2000000u, "limit_us=%u must be in [1, 2e6]",
                limit_us);
    unsigned* err = device_error_ptr();
    if (err == nullptr) return fail(KDA_ERR_CUDA, "no CUDA device is usable");
    cudaError_t e = kda::launch_selftest_timeout((uint64_t)limit_us * 1000u, err,
                                                 reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kda_selftest_timeout launch");
    return KDA_OK;
}

kda_status_t kda_device_status(kda_stream_t stream) {
    t_last_error.clear();
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kda_device_status wait");
    unsigned word = 0u;
    e = cudaMemcpyFromSymbol(&word, g_device_error, sizeof word);
    if (e != cudaSuccess) return cuda_fail(e, "kda_device_status read");
    const unsigned zero = 0u;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "kda_device_status clear");
    if (word & kda::kDevErrTimeout)
        return fail(KDA_ERR_TIMEOUT, "a device-side wait gave up (error word 0x%x)", word);
    if (word & kda::kDevErrBadSeqlens)
        return fail(KDA_ERR_DEVICE, "malformed cu_seqlens met on the device (error word 0x%x)",
                    word);
    return KDA_OK;
}

}  // extern "C"
