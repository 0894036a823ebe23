// decode.cu -- K4, one token of the KDA recurrence per sequence, state in place.
//
// "Kimi k3 技术报告详解（1）", section "Kimi Delta Attention":
//   S_t = (I - beta k k^T) Diag(alpha) S_{t-1} + beta k v^T,   o_t = S_t^T q_t.
// Rewritten for one pass over the state (S is d_k x d_v, row i = key channel):
//   a_j = sum_i alpha_i k_i S_ij,   b_j = sum_i alpha_i q_i S_ij
//   u_j = beta (v_j - a_j)                      (= beta (v - (Diag(alpha) S)^T k))
//   S_ij <- alpha_i S_ij + k_i u_j             (= Diag(alpha) S + k u^T)
//   o_j  = b_j + u_j (k . q)                    (= S_new^T q)
// so each state element is read once and written once: the kernel is a pure HBM
// stream of 2 * 4 * dk * dv bytes per (sequence, head).
//
// Layout: one CTA of 256 threads per (sequence, head).  A state row of dv fp32 is
// covered by dv/4 lanes with one float4 each (a warp reads 512 contiguous bytes for
// dv = 128); the dk rows are spread over the 8 warps, so every thread holds
// dk*dv/1024 floats.  The state is read twice: once for the two reductions (half of a
// thread's rows in flight while the gate is evaluated, the other half issued before the
// first is used) and again, from L2, for the update, so that no thread holds the whole
// state in registers and four CTAs fit on an SM.  HBM sees one read and one write; the
// second read and the write carry the streaming hint.
//
// The gated variant fuses the output step of section "Gated MLA" of the same page (between
// its two projections): instead of o it writes
//   y_j = Sigmoid(gate_j) * w_j * o_j / sqrt(mean_j o_j^2 + eps),
// the mean over the dv outputs of the (sequence, head), which one CTA holds, so o never
// reaches memory.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

template <int DK, int DV, typename IO, bool kGated>
__global__ void __launch_bounds__(256) decode_kernel(const IO* __restrict__ q,
                                                     const IO* __restrict__ k,
                                                     const IO* __restrict__ v,
                                                     const IO* __restrict__ beta,
                                                     const IO* __restrict__ z,
                                                     const float* __restrict__ A_log, float g_min,
                                                     float* __restrict__ S, int H,
                                                     const IO* __restrict__ gate,
                                                     const float* __restrict__ norm_w, float eps,
                                                     IO* __restrict__ o) {
    constexpr int kWarps = 8;
    constexpr int kLanesPerRow = DV / 4;
    constexpr int kRowsPerWarp = 32 / kLanesPerRow;
    constexpr int kRowsPerPass = kRowsPerWarp * kWarps;
    constexpr int kRowsPerThread = DK / kRowsPerPass;
    static_assert(DK % kRowsPerPass == 0, "dk must be a multiple of the rows per pass");

    __shared__ float s_alpha[DK], s_k[DK], s_q[DK], s_u[DV];
    __shared__ float s_red[2][kWarps][DV];
    __shared__ float s_kq;
    __shared__ float s_ss[DV / 32];  // gated variant: partial sums of o^2

    const int nh = blockIdx.x;
    const int h = nh % H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int col4 = lane % kLanesPerRow;
    const int sub = lane / kLanesPerRow;
    float* Sp = S + (size_t)nh * DK * DV;

    // first half of this thread's rows in flight while the gate is evaluated
    constexpr int kHalf = (kRowsPerThread + 1) / 2;
    float4 s[kHalf];
#pragma unroll
    for (int m = 0; m < kHalf; ++m) {
        const int row = m * kRowsPerPass + warp * kRowsPerWarp + sub;
        s[m] = __ldcg(reinterpret_cast<const float4*>(Sp + (size_t)row * DV) + col4);
    }

    const float scale = expf(__ldg(A_log + h));
    for (int c = tid; c < DK; c += blockDim.x) {
        const size_t idx = (size_t)nh * DK + c;
        s_alpha[c] = expf(gate_precise(to_f32(z[idx]), scale, g_min));
        s_k[c] = to_f32(k[idx]);
        s_q[c] = to_f32(q[idx]);
    }
    __syncthreads();

    float pa[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
    auto accumulate = [&](int m, const float4& sv) {
        const int row = m * kRowsPerPass + warp * kRowsPerWarp + sub;
        const float ak = s_alpha[row] * s_k[row], aq = s_alpha[row] * s_q[row];
        pa[0] = fmaf(ak, sv.x, pa[0]); pa[1] = fmaf(ak, sv.y, pa[1]);
        pa[2] = fmaf(ak, sv.z, pa[2]); pa[3] = fmaf(ak, sv.w, pa[3]);
        pb[0] = fmaf(aq, sv.x, pb[0]); pb[1] = fmaf(aq, sv.y, pb[1]);
        pb[2] = fmaf(aq, sv.z, pb[2]); pb[3] = fmaf(aq, sv.w, pb[3]);
    };
    {
        float4 s2[kRowsPerThread - kHalf];  // second half, issued before the first is used
#pragma unroll
        for (int m = kHalf; m < kRowsPerThread; ++m) {
            const int row = m * kRowsPerPass + warp * kRowsPerWarp + sub;
            s2[m - kHalf] = __ldcg(reinterpret_cast<const float4*>(Sp + (size_t)row * DV) + col4);
        }
#pragma unroll
        for (int m = 0; m < kHalf; ++m) accumulate(m, s[m]);
#pragma unroll
        for (int m = kHalf; m < kRowsPerThread; ++m) accumulate(m, s2[m - kHalf]);
    }
#pragma unroll
    for (int off = kLanesPerRow; off < 32; off <<= 1)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            pa[e] += __shfl_xor_sync(0xffffffffu, pa[e], off);
            pb[e] += __shfl_xor_sync(0xffffffffu, pb[e], off);
        }
    if (sub == 0)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            s_red[0][warp][col4 * 4 + e] = pa[e];
            s_red[1][warp][col4 * 4 + e] = pb[e];
        }
    if (warp == 0) {
        float t = 0.f;
        for (int c = lane; c < DK; c += 32) t = fmaf(s_k[c], s_q[c], t);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        if (lane == 0) s_kq = t;
    }
    __syncthreads();

    float o_j = 0.f;  // output channel tid (tid < DV)
    if (tid < DV) {
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            a += s_red[0][w][tid];
            b += s_red[1][w][tid];
        }
        const float u = to_f32(beta[nh]) * (to_f32(v[(size_t)nh * DV + tid]) - a);
        s_u[tid] = u;
        o_j = fmaf(u, s_kq, b);
        if (!kGated) o[(size_t)nh * DV + tid] = from_f32<IO>(o_j);
    }
    if (kGated && warp < DV / 32) {  // the DV outputs are warps 0 .. DV/32 - 1
        float sq = o_j * o_j;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
        if (lane == 0) s_ss[warp] = sq;
    }
    __syncthreads();
    if (kGated && tid < DV) {
        float ms = 0.f;
#pragma unroll
        for (int w = 0; w < DV / 32; ++w) ms += s_ss[w];
        const float inv_rms = rsqrtf(ms * (1.f / DV) + eps);
        const float wj = norm_w ? __ldg(norm_w + tid) : 1.f;
        const float gj = to_f32(gate[(size_t)nh * DV + tid]);
        o[(size_t)nh * DV + tid] = from_f32<IO>(o_j * inv_rms * wj / (1.f + __expf(-gj)));
    }

    const float4 u4 = reinterpret_cast<const float4*>(s_u)[col4];
#pragma unroll
    for (int m = 0; m < kRowsPerThread; ++m) {
        const int row = m * kRowsPerPass + warp * kRowsPerWarp + sub;
        float4* sp = reinterpret_cast<float4*>(Sp + (size_t)row * DV) + col4;
        const float4 sv = __ldcs(sp);  // second read, from L2
        const float al = s_alpha[row], kr = s_k[row];
        float4 r;
        r.x = fmaf(al, sv.x, kr * u4.x);
        r.y = fmaf(al, sv.y, kr * u4.y);
        r.z = fmaf(al, sv.z, kr * u4.z);
        r.w = fmaf(al, sv.w, kr * u4.w);
        __stcs(sp, r);
    }
}

struct DecodeOut {
    const void* gate;     // gated variant: [N, H, dv] io_dt, or nullptr for plain o
    const float* norm_w;  // [dv] or nullptr (ones)
    float eps;
    void* out;            // o, or y for the gated variant
};

template <int DK, int DV, typename IO>
cudaError_t launch_t(const void* q, const void* k, const void* v, const void* beta, const void* z,
                     const float* A_log, float g_min, float* S, int N, int H, const DecodeOut& d,
                     cudaStream_t stream) {
    const int grid = N * H;
    const IO* gate = static_cast<const IO*>(d.gate);
    if (gate) {
        ProfScope prof("decode_gated_kernel", stream);
        decode_kernel<DK, DV, IO, true><<<grid, 256, 0, stream>>>(
            static_cast<const IO*>(q), static_cast<const IO*>(k), static_cast<const IO*>(v),
            static_cast<const IO*>(beta), static_cast<const IO*>(z), A_log, g_min, S, H, gate,
            d.norm_w, d.eps, static_cast<IO*>(d.out));
    } else {
        ProfScope prof("decode_kernel", stream);
        decode_kernel<DK, DV, IO, false><<<grid, 256, 0, stream>>>(
            static_cast<const IO*>(q), static_cast<const IO*>(k), static_cast<const IO*>(v),
            static_cast<const IO*>(beta), static_cast<const IO*>(z), A_log, g_min, S, H, nullptr,
            nullptr, 0.f, static_cast<IO*>(d.out));
    }
    return cudaGetLastError();
}

template <typename IO>
cudaError_t dispatch_dims(const void* q, const void* k, const void* v, const void* beta,
                          const void* z, const float* A_log, float g_min, float* S, int N, int H,
                          int dk, int dv, const DecodeOut& d, cudaStream_t stream) {
    if (dk == 128 && dv == 128)
        return launch_t<128, 128, IO>(q, k, v, beta, z, A_log, g_min, S, N, H, d, stream);
    if (dk == 128 && dv == 64)
        return launch_t<128, 64, IO>(q, k, v, beta, z, A_log, g_min, S, N, H, d, stream);
    if (dk == 64 && dv == 128)
        return launch_t<64, 128, IO>(q, k, v, beta, z, A_log, g_min, S, N, H, d, stream);
    return launch_t<64, 64, IO>(q, k, v, beta, z, A_log, g_min, S, N, H, d, stream);
}

cudaError_t decode_any(const void* q, const void* k, const void* v, const void* beta,
                       const void* z, const float* A_log, float g_min, float* S, int N, int H,
                       int dk, int dv, int io_bf16, const DecodeOut& d, cudaStream_t stream) {
    if ((int64_t)N * H == 0) return cudaSuccess;
    if (io_bf16)
        return dispatch_dims<__nv_bfloat16>(q, k, v, beta, z, A_log, g_min, S, N, H, dk, dv, d,
                                            stream);
    return dispatch_dims<float>(q, k, v, beta, z, A_log, g_min, S, N, H, dk, dv, d, stream);
}

}  // namespace

cudaError_t launch_decode(const void* q, const void* k, const void* v, const void* beta,
                          const void* z, const float* A_log, float g_min, float* S, int N, int H,
                          int dk, int dv, int io_bf16, void* o, cudaStream_t stream) {
    return decode_any(q, k, v, beta, z, A_log, g_min, S, N, H, dk, dv, io_bf16,
                      DecodeOut{nullptr, nullptr, 0.f, o}, stream);
}

cudaError_t launch_decode_gated(const void* q, const void* k, const void* v, const void* beta,
                                const void* z, const float* A_log, float g_min, float* S, int N,
                                int H, int dk, int dv, int io_bf16, const void* gate,
                                const float* norm_w, float eps, void* y, cudaStream_t stream) {
    return decode_any(q, k, v, beta, z, A_log, g_min, S, N, H, dk, dv, io_bf16,
                      DecodeOut{gate, norm_w, eps, y}, stream);
}

}  // namespace kda
