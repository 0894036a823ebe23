// gate.cu -- K1, the lower-bounded decay gate on its own:
//   g[t,h,c] = g_min * Sigmoid(exp(A_log[h]) * z[t,h,c])
// ("Kimi k3 技术报告详解（1）", section "Chunkwise parallel form", gate equation;
//  "A Look at Kimi K3 ... Tuning Guide", section 2.2 and its pseudocode.)
// Pure streaming work: 4 elements per thread per step (dk is a multiple of 4), grid
// sized to a multiple of the SM count, grid-stride loop.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

struct alignas(8) bf16x4 { __nv_bfloat162 a, b; };

template <typename IO>
__device__ __forceinline__ float4 load4(const IO* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(p));
    bf16x4 v;
    v.a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    v.b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    const float2 lo = __bfloat1622float2(v.a), hi = __bfloat1622float2(v.b);
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

template <typename IO>
__global__ void __launch_bounds__(256) gate_kernel(const IO* __restrict__ z,
                                                   const float* __restrict__ A_log, float g_min,
                                                   float* __restrict__ g, int64_t n_vec, int H,
                                                   int dk4) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec; i += stride) {
        const int h = (int)((i / dk4) % H);
        const float scale = expf(__ldg(A_log + h));
        const float4 zz = load4<IO>(z + i * 4);
        float4 out;
        out.x = gate_precise(zz.x, scale, g_min);
        out.y = gate_precise(zz.y, scale, g_min);
        out.z = gate_precise(zz.z, scale, g_min);
        out.w = gate_precise(zz.w, scale, g_min);
        __stcs(reinterpret_cast<float4*>(g) + i, out);
    }
}

}  // namespace

cudaError_t launch_gate(const void* z, int z_bf16, const float* A_log, float g_min, float* g_out,
                        int64_t n_tokens, int H, int dk, cudaStream_t stream) {
    const int64_t n_vec = n_tokens * H * (dk / 4);
    if (n_vec == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (n_vec + 255) / 256;
    const int64_t cap = (int64_t)sms * 8;  // 8 resident CTAs of 256 threads per SM
    const int grid = (int)(want < cap ? want : cap);
    ProfScope prof("gate_kernel", stream);
    if (z_bf16)
        gate_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(z), A_log, g_min, g_out, n_vec, H, dk / 4);
    else
        gate_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(z), A_log, g_min,
                                                     g_out, n_vec, H, dk / 4);
    return cudaGetLastError();
}

}  // namespace kda
