// qb.cu -- quantile-balancing update of the router's expert biases.
//
// "Kimi k3 技术报告详解（1）——架构再升华", section on load balancing, "Quantile Balancing
// (QB)" (and "A Look at Kimi K3 ...", section 4.2): with router scores s [m, n], k experts
// per token and the current biases b [n],
//   alpha_i  = the (k+1)-th largest of s_i + b          (token i's threshold)
//   margin_ij = s_ij - alpha_i
//   bhat_j   = -(the (q+1)-th largest margin of expert j),  q = floor(m k / n)
//              (so that expert j would receive exactly q tokens under bhat_j)
//   b_new    = bhat - mean(bhat).
// s + b and the margins are formed in fp32; the selections are exact (no arithmetic).
//
// Kernels, all on the caller's stream:
//   qb_alpha_kernel   one warp per token: the row's n values in registers (n <= 1024,
//                     ceil(n/32) per lane), the (k+1)-th largest by k+1 rounds of warp
//                     maximum and removal of one occurrence (or the (n-k)-th smallest, by
//                     rounds of minimum, when that takes fewer rounds).
//   qb_hist_kernel    radix select over the margins of every expert at once, 8 bits per pass
//                     (4 passes, most significant digit first) on an order-preserving
//                     uint32 key, inverted so that ascending keys are descending margins:
//                     a CTA takes 32 experts (a lane per expert, so a warp reads 128
//                     contiguous bytes of a score row) and a range of tokens, counts the
//                     digits of the keys that still match the expert's prefix in shared
//                     memory and adds its counts to a global [n][256] histogram.  The
//                     scores (m n 4 bytes) are re-read every pass; at 64 MB they stay in L2.
//   qb_select_kernel  one warp per expert: the digit holding rank q (prefix scan over the
//                     256 counts), appended to the expert's prefix; the histogram is cleared
//                     for the next pass.  After the last pass the key is the (q+1)-th
//                     largest margin itself.
//   qb_mean_kernel    one CTA: bhat and bhat - mean(bhat).
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

// order-preserving map of fp32 to uint32 (ascending floats -> ascending keys), inverted so
// that ascending keys are descending floats
__device__ __forceinline__ uint32_t desc_key(float x) {
    const uint32_t u = __float_as_uint(x);
    const uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ~asc;
}
__device__ __forceinline__ float key_value(uint32_t key) {
    const uint32_t asc = ~key;
    const uint32_t u = (asc & 0x80000000u) ? (asc & 0x7fffffffu) : ~asc;
    return __uint_as_float(u);
}

// kP values per lane (n <= 32 kP).  The (k+1)-th largest is found by k+1 rounds of "take the
// warp maximum, remove one occurrence", or, when that is shorter, as the (n-k)-th smallest by
// rounds of minimum.
template <int kP>
__global__ void __launch_bounds__(256) qb_alpha_kernel(const float* __restrict__ s,
                                                       const float* __restrict__ b, int64_t m,
                                                       int n, int k, float* __restrict__ alpha) {
    const int lane = threadIdx.x & 31;
    const bool from_top = k + 1 <= n - k;
    const int rounds = from_top ? k + 1 : n - k;
    const float pad = from_top ? -INFINITY : INFINITY;  // never selected
    float bj[kP];
#pragma unroll
    for (int e = 0; e < kP; ++e) {
        const int j = lane + 32 * e;
        bj[e] = (j < n) ? __ldg(b + j) : 0.f;
    }
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t i = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); i < m;
         i += warps) {
        float v[kP];
#pragma unroll
        for (int e = 0; e < kP; ++e) {
            const int j = lane + 32 * e;
            // s + b in fp32; the top-down search works on -v, so both are "largest first"
            const float x = (j < n) ? s[i * n + j] + bj[e] : pad;
            v[e] = from_top ? x : -x;
        }
        float a = 0.f;
        for (int r = 0; r < rounds; ++r) {
            float mx = v[0];
#pragma unroll
            for (int e = 1; e < kP; ++e) mx = fmaxf(mx, v[e]);
            float wm = mx;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, off));
            a = wm;
            if (r + 1 == rounds) break;
            // remove one occurrence of the maximum: in the lowest lane holding it, its first
            const unsigned holders = __ballot_sync(0xffffffffu, mx == wm);
            if (lane == __ffs(holders) - 1) {
                bool done = false;
#pragma unroll
                for (int e = 0; e < kP; ++e)
                    if (!done && v[e] == wm) {
                        v[e] = -INFINITY;
                        done = true;
                    }
            }
        }
        if (lane == 0) alpha[i] = from_top ? a : -a;
    }
}

struct QbColumn {
    uint32_t prefix;  // key bits fixed so far (the passes before this one)
    uint32_t rank;    // rank of the wanted key among the keys with that prefix (0-based)
};

__global__ void __launch_bounds__(256) qb_hist_kernel(const float* __restrict__ s,
                                                      const float* __restrict__ alpha, int64_t m,
                                                      int n, int rows_per_cta, int shift,
                                                      const QbColumn* __restrict__ col_state,
                                                      unsigned* __restrict__ hist) {
    __shared__ unsigned sh[32][257];  // padded: lane + bin spreads over the banks
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 32 * 257; i += blockDim.x) (&sh[0][0])[i] = 0u;
    __syncthreads();
    const int col = blockIdx.y * 32 + lane;
    const bool live = col < n;
    uint32_t prefix = 0u;
    if (live && shift < 24) prefix = col_state[col].prefix >> (shift + 8);
    const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
    const int64_t r1 = min(m, r0 + rows_per_cta);
    if (live) {
        auto count = [&](float x, float al) {
            const uint32_t key = desc_key(x - al);
            if (shift == 24 || (key >> (shift + 8)) == prefix)
                atomicAdd(&sh[lane][(key >> shift) & 255u], 1u);
        };
        int64_t i = r0 + warp;
        for (; i + 24 < r1; i += 32) {  // four rows per step, loads first
            float x[4], al[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                x[u] = s[(i + 8 * u) * n + col];
                al[u] = __ldg(alpha + i + 8 * u);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) count(x[u], al[u]);
        }
        for (; i < r1; i += 8) count(s[i * n + col], __ldg(alpha + i));
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < 32 * 256; idx += blockDim.x) {
        const int c = idx >> 8, bin = idx & 255;
        const unsigned cnt = sh[c][bin];
        if (cnt && blockIdx.y * 32 + c < n) atomicAdd(&hist[(size_t)(blockIdx.y * 32 + c) * 256 + bin], cnt);
    }
}

__global__ void __launch_bounds__(256) qb_select_kernel(int n, int shift, uint32_t q,
                                                        QbColumn* __restrict__ col_state,
                                                        unsigned* __restrict__ hist,
                                                        float* __restrict__ bhat) {
    const int lane = threadIdx.x & 31;
    const int col = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (col >= n) return;
    QbColumn st = (shift == 24) ? QbColumn{0u, q} : col_state[col];
    unsigned* h = hist + (size_t)col * 256;
    unsigned c[8];
    unsigned tot = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {  // lane holds bins 8 lane .. 8 lane + 7
        c[e] = h[8 * lane + e];
        tot += c[e];
    }
    unsigned incl = tot;  // inclusive prefix over the lanes
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
    }
    const unsigned excl = incl - tot;
    // the lane whose bins contain rank st.rank
    const unsigned mine = __ballot_sync(0xffffffffu, excl <= st.rank && st.rank < incl);
    const int owner = __ffs(mine) - 1;  // exactly one lane (the counts cover the rank)
    if (lane == owner) {
        unsigned before = excl;
        int digit = 8 * lane;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (st.rank < before + c[e]) {
                digit = 8 * lane + e;
                break;
            }
            before += c[e];
        }
        st.prefix |= (uint32_t)digit << shift;
        st.rank -= before;
        col_state[col] = st;
        if (shift == 0) bhat[col] = -key_value(st.prefix);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) h[8 * lane + e] = 0u;  // ready for the next pass
}

__global__ void __launch_bounds__(1024) qb_mean_kernel(const float* __restrict__ bhat, int n,
                                                       float* __restrict__ b_new) {
    __shared__ double part[32];
    double acc = 0.0;
    for (int j = threadIdx.x; j < n; j += blockDim.x) acc += (double)bhat[j];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x < 32) {
        double t = (threadIdx.x < blockDim.x / 32) ? part[threadIdx.x] : 0.0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        if (threadIdx.x == 0) part[0] = t;
    }
    __syncthreads();
    const double mean = part[0] / n;
    for (int j = threadIdx.x; j < n; j += blockDim.x) b_new[j] = (float)((double)bhat[j] - mean);
}

}  // namespace

size_t qb_workspace_size(int64_t m, int n) {
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    return al((size_t)m * 4) + al((size_t)n * 256 * 4) + al((size_t)n * sizeof(QbColumn)) +
           al((size_t)n * 4);
}

cudaError_t launch_quantile_balance(const float* s, const float* b, int64_t m, int n, int k,
                                    float* b_new, float* bhat_out, float* alpha_out,
                                    void* workspace, cudaStream_t stream) {
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    uint8_t* w = static_cast<uint8_t*>(workspace);
    float* alpha = reinterpret_cast<float*>(w);
    unsigned* hist = reinterpret_cast<unsigned*>(w + al((size_t)m * 4));
    QbColumn* cols = reinterpret_cast<QbColumn*>(w + al((size_t)m * 4) + al((size_t)n * 1024));
    float* bhat = reinterpret_cast<float*>(w + al((size_t)m * 4) + al((size_t)n * 1024) +
                                           al((size_t)n * sizeof(QbColumn)));
    if (alpha_out) alpha = alpha_out;
    if (bhat_out) bhat = bhat_out;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t e = cudaMemsetAsync(hist, 0, (size_t)n * 1024, stream);
    if (e != cudaSuccess) return e;
    {
        const int64_t want = (m + 7) / 8;
        const int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
        ProfScope prof("qb_alpha_kernel", stream);
        const int per_lane = (n + 31) / 32;
        if (per_lane <= 1)
            qb_alpha_kernel<1><<<grid, 256, 0, stream>>>(s, b, m, n, k, alpha);
        else if (per_lane <= 2)
            qb_alpha_kernel<2><<<grid, 256, 0, stream>>>(s, b, m, n, k, alpha);
        else if (per_lane <= 4)
            qb_alpha_kernel<4><<<grid, 256, 0, stream>>>(s, b, m, n, k, alpha);
        else if (per_lane <= 8)
            qb_alpha_kernel<8><<<grid, 256, 0, stream>>>(s, b, m, n, k, alpha);
        else if (per_lane <= 16)
            qb_alpha_kernel<16><<<grid, 256, 0, stream>>>(s, b, m, n, k, alpha);
        else
            qb_alpha_kernel<32><<<grid, 256, 0, stream>>>(s, b, m, n, k, alpha);
    }
    const uint32_t q = (uint32_t)((m * k) / n);
    const int col_blocks = (n + 31) / 32;
    // about four CTAs per SM in total, at least 256 tokens each
    int64_t row_blocks = ((int64_t)sms * 4 + col_blocks - 1) / col_blocks;
    if (row_blocks > (m + 255) / 256) row_blocks = (m + 255) / 256;
    if (row_blocks < 1) row_blocks = 1;
    const int rows_per_cta = (int)((m + row_blocks - 1) / row_blocks);
    row_blocks = (m + rows_per_cta - 1) / rows_per_cta;
    for (int shift = 24; shift >= 0; shift -= 8) {
        {
            ProfScope prof("qb_hist_kernel", stream);
            qb_hist_kernel<<<dim3((unsigned)row_blocks, (unsigned)col_blocks), 256, 0, stream>>>(
                s, alpha, m, n, rows_per_cta, shift, cols, hist);
        }
        ProfScope prof("qb_select_kernel", stream);
        qb_select_kernel<<<(n + 7) / 8, 256, 0, stream>>>(n, shift, q, cols, hist, bhat);
    }
    {
        ProfScope prof("qb_mean_kernel", stream);
        qb_mean_kernel<<<1, 1024, 0, stream>>>(bhat, n, b_new);
    }
    return cudaGetLastError();
}

}  // namespace kda
