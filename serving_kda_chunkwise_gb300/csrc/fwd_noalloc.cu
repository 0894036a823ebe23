// fwd_noalloc.cu -- kda_fwd_chunked_noalloc: the chunked forward for callers that must not
// allocate device memory at all.  A host framework that owns every byte of GPU memory
// (a serving runtime with a fixed memory budget, a plugin that may not call the CUDA
// allocator, code running where an allocation would synchronise the device) cannot supply
// the workspace kda_fwd_chunked asks for.  This entry point takes its scratch from a fixed
// buffer compiled into the library instead.
#include <cstdio>
#include <mutex>

#include "kda.h"
#include "kda_internal.h"

namespace {

// Fixed scratch for the tensor-core path.  It lives in every GPU's memory from the moment
// the library is loaded on that GPU until the process exits.
constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[64] = {};  // device address of g_scratch, per device ordinal

// Device address of g_scratch on the current device (looked up on the first call there).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" kda_status_t kda_fwd_chunked_noalloc(
    const void* q, const void* k, const void* v, const void* beta, const void* z,
    const float* A_log, float g_min, const float* S0, float* S_out, const int32_t* cu_seqlens,
    int N, int64_t T_total, int H, int dk, int dv, kda_dtype_t io_dt, void* o,
    kda_stream_t stream) {
    // a malformed call is reported as such before the scratch size is looked at
    if (kda_status_t s = kda::check_fwd_args(q, k, v, beta, z, A_log, g_min, S0, S_out,
                                             cu_seqlens, N, T_total, H, dk, dv, io_dt, o))
        return s;
    const size_t need = kda_fwd_workspace_size(T_total, N, H, dk, dv, io_dt);
    if (need == 0)  // the selected kernels need no scratch
        return kda_fwd_chunked(q, k, v, beta, z, A_log, g_min, S0, S_out, cu_seqlens, N, T_total,
                               H, dk, dv, io_dt, o, nullptr, 0, stream);
    if (need > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "kda_fwd_chunked_noalloc: this problem needs %zu bytes of scratch, more than "
                 "the %zu built into the library; use kda_fwd_chunked with a workspace",
                 need, kScratchBytes);
        return kda::set_last_error(KDA_ERR_INVALID_ARG, msg);
    }
    void* scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "kda_fwd_chunked_noalloc: scratch address lookup failed: %s",
                 cudaGetErrorString(e));
        return kda::set_last_error(KDA_ERR_CUDA, msg);
    }
    return kda_fwd_chunked(q, k, v, beta, z, A_log, g_min, S0, S_out, cu_seqlens, N, T_total, H,
                           dk, dv, io_dt, o, scratch, kScratchBytes, stream);
}
