// kda_common.cuh -- device helpers shared by the KDA kernels of libkda.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// Bits of the device error word (see kda_device_status in kda.h).
enum : unsigned { kDevErrBadSeqlens = 1u, kDevErrTimeout = 2u };

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Lower-bounded gate ("Kimi k3 技术报告详解（1）", section "Chunkwise parallel form";
// "A Look at Kimi K3 ... Tuning Guide", section 2.2):
//   g = g_min * Sigmoid(e^{A_h} z),  with scale = e^{A_h} precomputed per head.
// Written as g_min / (1 + e^{-scale z}); z = -inf gives -0 (alpha = 1), z = +inf gives g_min.
__device__ __forceinline__ float gate_precise(float z, float scale, float g_min) {
    return g_min / (1.0f + expf(-scale * z));
}

// The gate the bound replaces (same page and section): g = -e^{A_h} Softplus(z), in
// (-inf, 0), Softplus(z) = ln(1 + e^z) written so that e^z never overflows.  z = -inf gives
// -0 (alpha = 1); z must be finite otherwise (z = +inf would give g = -inf).
__device__ __forceinline__ float gate_softplus(float z, float scale) {
    const float sp = z > 0.f ? z + log1pf(expf(-z)) : log1pf(expf(z));
    return -scale * sp;
}

// Token range [begin, end) of sequence n.  cu == nullptr means N equal sequences of
// T_total / N tokens.  A malformed range raises kDevErrBadSeqlens and reads as empty.
__device__ __forceinline__ void seq_range(const int32_t* cu, int n, int N, int64_t T_total,
                                          unsigned* err, int64_t& begin, int64_t& end) {
    if (cu == nullptr) {
        const int64_t len = T_total / N;
        begin = (int64_t)n * len;
        end = begin + len;
        return;
    }
    const int64_t a = cu[n], b = cu[n + 1];
    if (a < 0 || b < a || b > T_total || (n == 0 && a != 0) || (n == N - 1 && b != T_total)) {
        if (err) atomicOr(err, kDevErrBadSeqlens);
        begin = end = 0;
        return;
    }
    begin = a;
    end = b;
}

}  // namespace kda
