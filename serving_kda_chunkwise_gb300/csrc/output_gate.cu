// output_gate.cu -- the gated, RMS-normalised output step on its own:
//   y[t,h,j] = Sigmoid(gate[t,h,j]) * w[j] * o[t,h,j] / sqrt(mean_j o[t,h,j]^2 + eps)
// ("Kimi k3 技术报告详解（1）", section "Gated MLA": the layer output is
//  W_o [Sigmoid(W_g x_t) (.) RMSNorm(o~_t)]; this is the part between the two projections,
//  with the norm taken per head over its d_v channels and gate = W_g x_t given.)
//
// Pure streaming work, 3 x 2 bytes per element for bf16 I/O.  A row (one token and head) of
// dv channels is covered by dv / 8 lanes, 8 channels each (16 bytes of bf16 per load), so a
// warp reads 2 (dv = 128) or 4 (dv = 64) whole rows per row group; the row's sum of squares
// is a shuffle reduction over its lanes.  Every lane keeps its 8 norm weights in registers.
// Each step of the grid-stride loop takes two row groups and issues all four loads first;
// the sigmoid's division is the fast reciprocal form (the step was issue-bound with the
// IEEE division: 349 us against 288 us on 65536 x 32 rows of 128).  o and gate go through
// the read-only path, y is written with the streaming hint.  y may alias o: then o is read
// with ordinary (coherent) evict-first loads; each lane reads its 8 values of o before the
// row's reduction and writes them after it.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

template <typename IO>
struct Vec8;
// kNc: the read-only (non-coherent) load path, for tensors this kernel never writes
template <>
struct Vec8<__nv_bfloat16> {
    template <bool kNc>
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[8]) {
        const uint4* q = reinterpret_cast<const uint4*>(p);
        const uint4 u = kNc ? __ldg(q) : __ldcs(q);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
            v[2 * e] = f.x;
            v[2 * e + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
            w[e] = *reinterpret_cast<const uint32_t*>(&b);
        }
        __stcs(reinterpret_cast<uint4*>(p), make_uint4(w[0], w[1], w[2], w[3]));
    }
};
template <>
struct Vec8<float> {
    template <bool kNc>
    static __device__ __forceinline__ void load(const float* p, float (&v)[8]) {
        const float4* q = reinterpret_cast<const float4*>(p);
        const float4 a = kNc ? __ldg(q) : __ldcs(q);
        const float4 b = kNc ? __ldg(q + 1) : __ldcs(q + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    static __device__ __forceinline__ void store(float* p, const float (&v)[8]) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
        __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(v[4], v[5], v[6], v[7]));
    }
};

template <typename IO, int DV, bool kInPlace>
__global__ void __launch_bounds__(256) output_gate_kernel(const IO* o,  // y when kInPlace
                                                          const IO* __restrict__ gate,
                                                          const float* __restrict__ w,
                                                          float eps, IO* y, int64_t n_rows) {
    constexpr int kLanes = DV / 8;               // lanes per row
    constexpr int kRowsPerWarp = 32 / kLanes;
    const int lane = threadIdx.x & 31;
    const int sub = lane / kLanes, c8 = lane % kLanes;
    float wv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) wv[e] = w ? __ldg(w + 8 * c8 + e) : 1.f;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    // r0 is the same in every lane of a warp, so the shuffles below see full warps; each
    // step handles kU row groups, all loads issued before any arithmetic
    constexpr int kU = 2;
    for (int64_t r0 = wid * kU * kRowsPerWarp; r0 < n_rows; r0 += warps * kU * kRowsPerWarp) {
        float ov[kU][8], gv[kU][8];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t row = r0 + u * kRowsPerWarp + sub;
#pragma unroll
            for (int e = 0; e < 8; ++e) ov[u][e] = gv[u][e] = 0.f;
            if (row < n_rows) {
                const size_t off = (size_t)row * DV + 8 * c8;
                Vec8<IO>::template load<!kInPlace>(o + off, ov[u]);
                Vec8<IO>::template load<true>(gate + off, gv[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t row = r0 + u * kRowsPerWarp + sub;
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(ov[u][e], ov[u][e], ss);
#pragma unroll
            for (int s = kLanes / 2; s > 0; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
            const float inv_rms = rsqrtf(ss * (1.f / DV) + eps);
            if (row < n_rows) {
                float yv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    yv[e] = __fdividef(ov[u][e] * inv_rms * wv[e], 1.f + __expf(-gv[u][e]));
                Vec8<IO>::store(y + (size_t)row * DV + 8 * c8, yv);
            }
        }
    }
}

template <typename IO, int DV>
cudaError_t launch_t(const void* o, const void* gate, const float* w, float eps, void* y,
                     int64_t n_rows, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    constexpr int kRowsPerCta = 8 * (32 / (DV / 8)) * 2;
    const int64_t want = (n_rows + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t cap = (int64_t)sms * 8;
    const int grid = (int)(want < cap ? want : cap);
    ProfScope prof("output_gate_kernel", stream);
    if (o == y)
        output_gate_kernel<IO, DV, true><<<grid, 256, 0, stream>>>(
            static_cast<const IO*>(o), static_cast<const IO*>(gate), w, eps, static_cast<IO*>(y),
            n_rows);
    else
        output_gate_kernel<IO, DV, false><<<grid, 256, 0, stream>>>(
            static_cast<const IO*>(o), static_cast<const IO*>(gate), w, eps, static_cast<IO*>(y),
            n_rows);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_output_gate(const void* o, const void* gate, const float* norm_w, float eps,
                               void* y, int64_t n_rows, int dv, int io_bf16,
                               cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    if (io_bf16)
        return dv == 128 ? launch_t<__nv_bfloat16, 128>(o, gate, norm_w, eps, y, n_rows, stream)
                         : launch_t<__nv_bfloat16, 64>(o, gate, norm_w, eps, y, n_rows, stream);
    return dv == 128 ? launch_t<float, 128>(o, gate, norm_w, eps, y, n_rows, stream)
                     : launch_t<float, 64>(o, gate, norm_w, eps, y, n_rows, stream);
}

}  // namespace kda
