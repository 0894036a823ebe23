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
//                     ceil(n/32) per lane, sorted within the lane), the (k+1)-th largest by
//                     k+1 rounds of warp maximum over the lanes' first values and removal of
//                     that value from the lowest lane holding it (or the (n-k)-th smallest,
//                     by rounds of minimum, when that takes fewer rounds).
//   qb_hist_kernel    radix select over the margins of every expert at once, 8 bits per pass
//                     (4 passes, most significant digit first) on an order-preserving
//                     uint32 key, inverted so that ascending keys are descending margins:
//                     a CTA takes 32 experts (a lane per expert, so a warp reads 128
//                     contiguous bytes of a score row) and a range of tokens, counts the
//                     digits of the keys that still match the expert's prefix in shared
//                     memory and adds its counts to a global [n][256] histogram.  The
//                     scores (m n 4 bytes) are re-read every pass; at 64 MB they stay in L2.
//                     The last CTA of each column of experts to finish a pass selects
//                     their digits (the digit holding rank q, by a prefix scan over the 256
//                     counts, appended to the expert's prefix) and clears their counts; after
//                     the last pass the key is the (q+1)-th largest margin itself, and the last
//                     column to finish forms bhat - mean(bhat).
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

// order-preserving map of fp32 to uint32 (ascending floats -> ascending keys) and back
__device__ __forceinline__ uint32_t asc_key(float x) {
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float asc_value(uint32_t asc) {
    return __uint_as_float((asc & 0x80000000u) ? (asc & 0x7fffffffu) : ~asc);
}

// Sort kP keys descending (odd-even transposition network, unrolled).
template <int kP>
__device__ __forceinline__ void sort_desc(uint32_t (&v)[kP]) {
#pragma unroll
    for (int rnd = 0; rnd < kP; ++rnd)
#pragma unroll
        for (int e = rnd & 1; e + 1 < kP; e += 2) {
            const uint32_t a = v[e], b2 = v[e + 1];
            v[e] = max(a, b2);
            v[e + 1] = min(a, b2);
        }
}

// kP values per lane (n <= 32 kP) as order-preserving keys, kept sorted (largest first), so a
// lane's candidate is its first key.  The (k+1)-th largest is found by k+1 rounds of "take
// the warp maximum of the lanes' first keys (one warp reduction), and the lowest lane holding
// it drops that key", or, when that is shorter, as the (n-k)-th smallest by the same rounds
// on negated values.  Zeros are made +0 first, so that the two zeros are one key.
template <int kP>
__global__ void __launch_bounds__(256) qb_alpha_kernel(const float* __restrict__ s,
                                                       const float* __restrict__ b, int64_t m,
                                                       int n, int k, float* __restrict__ alpha) {
    const int lane = threadIdx.x & 31;
    const bool from_top = k + 1 <= n - k;
    const int rounds = from_top ? k + 1 : n - k;
    const float pad = from_top ? -INFINITY : INFINITY;  // never selected
    constexpr uint32_t kGone = 0u;                       // below every value's key
    float bj[kP];
#pragma unroll
    for (int e = 0; e < kP; ++e) {
        const int j = lane + 32 * e;
        bj[e] = (j < n) ? __ldg(b + j) : 0.f;
    }
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    // the scores of the warp's next token are loaded while it selects in the current one
    auto load_row = [&](int64_t i, float (&x)[kP]) {
#pragma unroll
        for (int e = 0; e < kP; ++e) {
            const int j = lane + 32 * e;
            x[e] = (i < m && j < n) ? __ldg(s + i * n + j) : 0.f;
        }
    };
    int64_t i = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    float xn[kP];
    load_row(i, xn);
    for (; i < m; i += warps) {
        uint32_t v[kP];
#pragma unroll
        for (int e = 0; e < kP; ++e) {
            const int j = lane + 32 * e;
            // s + b in fp32; the top-down search works on -v, so both are "largest first"
            const float x = (j < n) ? xn[e] + bj[e] : pad;
            v[e] = asc_key((from_top ? x : -x) + 0.f);
        }
        load_row(i + warps, xn);
        sort_desc(v);
        uint32_t a = 0u;
        for (int r = 0; r < rounds; ++r) {
            const uint32_t wm = __reduce_max_sync(0xffffffffu, v[0]);
            a = wm;
            if (r + 1 == rounds) break;
            // the lowest lane holding the maximum drops it (its list moves up by one)
            const unsigned holders = __ballot_sync(0xffffffffu, v[0] == wm);
            const bool pop = lane == __ffs(holders) - 1;
#pragma unroll
            for (int e = 0; e + 1 < kP; ++e) v[e] = pop ? v[e + 1] : v[e];
            v[kP - 1] = pop ? kGone : v[kP - 1];
        }
        if (lane == 0) {
            const float av = asc_value(a);
            alpha[i] = from_top ? av : -av;
        }
    }
}

struct QbColumn {
    uint32_t prefix;  // key bits fixed so far (the passes before this one)
    uint32_t rank;    // rank of the wanted key among the keys with that prefix (0-based)
};

// The digit of expert `col` holding its rank (prefix scan over the 256 counts of `h`, one
// warp), appended to the expert's prefix; the counts are cleared for the next pass.  After
// the last pass (shift 0) the key is the (q+1)-th largest margin and bhat = -(its value).
__device__ __forceinline__ void select_digit(int col, int shift, uint32_t q,
                                             QbColumn* __restrict__ col_state,
                                             unsigned* __restrict__ h, float* __restrict__ bhat) {
    const int lane = threadIdx.x & 31;
    QbColumn st = (shift == 24) ? QbColumn{0u, q} : col_state[col];
    unsigned c[8];
    unsigned tot = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {  // lane holds bins 8 lane .. 8 lane + 7
        c[e] = __ldcg(h + 8 * lane + e);
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

// The end of a radix pass, after a CTA has counted its keys into `sh`: its counts go into the
// global histogram; the last CTA of its column of experts to finish selects their digits, and
// after the last pass the last column to finish forms bias_new = bhat - mean(bhat).
__device__ __forceinline__ void finish_pass(unsigned (&sh)[32][257], double (&part)[8], int& last,
                                            int n, int shift, uint32_t q,
                                            QbColumn* __restrict__ col_state,
                                            unsigned* __restrict__ hist,
                                            unsigned* __restrict__ done,
                                            float* __restrict__ bhat,
                                            float* __restrict__ b_new) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    for (int idx = threadIdx.x; idx < 32 * 256; idx += blockDim.x) {
        const int c = idx >> 8, bin = idx & 255;
        const unsigned cnt = sh[c][bin];
        if (cnt && blockIdx.y * 32 + c < n) atomicAdd(&hist[(size_t)(blockIdx.y * 32 + c) * 256 + bin], cnt);
    }
    // the last CTA of this column of experts selects their digits
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(&done[blockIdx.y], 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    for (int c = warp; c < 32; c += blockDim.x / 32) {
        const int cc = blockIdx.y * 32 + c;
        if (cc < n) select_digit(cc, shift, q, col_state, hist + (size_t)cc * 256, bhat);
    }
    if (threadIdx.x == 0) done[blockIdx.y] = 0u;  // ready for the next pass
    if (shift != 0) return;
    // after the last pass: the last column to finish forms bias_new
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(&done[gridDim.y], 1u) == gridDim.y - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    double acc = 0.0;
    for (int j = threadIdx.x; j < n; j += blockDim.x) acc += (double)__ldcg(bhat + j);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) part[warp] = acc;
    __syncthreads();
    double tot = 0.0;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += part[w];
    const double mean = tot / n;
    for (int j = threadIdx.x; j < n; j += blockDim.x)
        b_new[j] = (float)((double)__ldcg(bhat + j) - mean);
    if (threadIdx.x == 0) done[gridDim.y] = 0u;
}

// One radix pass: a CTA counts the digits of 32 experts' margins over its token range and
// adds them to the global histogram (then finish_pass).  A lane takes one expert, so a warp
// load reads 128 contiguous bytes of a score row.
template <int kU>
__global__ void __launch_bounds__(256) qb_hist_kernel(const float* __restrict__ s,
                                                      const float* __restrict__ alpha, int64_t m,
                                                      int n, int rows_per_cta, int shift,
                                                      uint32_t q, QbColumn* __restrict__ col_state,
                                                      unsigned* __restrict__ hist,
                                                      unsigned* __restrict__ done,
                                                      float* __restrict__ bhat,
                                                      float* __restrict__ b_new) {
    __shared__ unsigned sh[32][257];  // padded: lane + bin spreads over the banks
    __shared__ double part[8];
    __shared__ int last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 32 * 257; i += blockDim.x) (&sh[0][0])[i] = 0u;
    __syncthreads();
    const int col = blockIdx.y * 32 + lane;
    const bool live = col < n;
    uint32_t prefix = 0u;
    if (live && shift < 24) prefix = __ldcg(&col_state[col].prefix) >> (shift + 8);
    const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
    const int64_t r1 = min(m, r0 + rows_per_cta);
    if (live) {
        auto count = [&](float x, float al) {
            const uint32_t key = desc_key(x - al);
            if (shift == 24 || (key >> (shift + 8)) == prefix)
                atomicAdd(&sh[lane][(key >> shift) & 255u], 1u);
        };
        int64_t i = r0 + warp;
        for (; i + 8 * (kU - 1) < r1; i += 8 * kU) {  // kU rows per step, loads first
            float x[kU], al[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                x[u] = __ldg(s + (i + 8 * u) * n + col);
                al[u] = __ldg(alpha + i + 8 * u);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) count(x[u], al[u]);
        }
        for (; i < r1; i += 8) count(__ldg(s + i * n + col), __ldg(alpha + i));
    }
    finish_pass(sh, part, last, n, shift, q, col_state, hist, done, bhat, b_new);
}

// The same pass for n a multiple of 4 (and 16-byte aligned scores): a lane takes four
// consecutive experts of one row (lane = 8 x row of 4 + quad), so that a warp load reads 4
// rows x 128 bytes, four times the bytes per load instruction and in flight.
template <int kU>
__global__ void __launch_bounds__(256) qb_hist4_kernel(const float* __restrict__ s,
                                                       const float* __restrict__ alpha, int64_t m,
                                                       int n, int rows_per_cta, int shift,
                                                       uint32_t q, QbColumn* __restrict__ col_state,
                                                       unsigned* __restrict__ hist,
                                                       unsigned* __restrict__ done,
                                                       float* __restrict__ bhat,
                                                       float* __restrict__ b_new) {
    __shared__ unsigned sh[32][257];
    __shared__ double part[8];
    __shared__ int last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 32 * 257; i += blockDim.x) (&sh[0][0])[i] = 0u;
    __syncthreads();
    const int r4 = lane >> 3, eq = lane & 7;
    const int c0 = blockIdx.y * 32 + 4 * eq;  // this lane's experts c0 .. c0 + 3 (all live or none)
    const bool live = c0 < n;
    uint32_t prefix[4] = {0u, 0u, 0u, 0u};
    if (live && shift < 24) {
#pragma unroll
        for (int e = 0; e < 4; ++e) prefix[e] = __ldcg(&col_state[c0 + e].prefix) >> (shift + 8);
    }
    const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
    const int64_t r1 = min(m, r0 + rows_per_cta);
    if (live) {
        // a step: rows b + 32 u + r4 for u < kU, b = r0 + 4 warp + 32 kU (step); the next
        // step's loads are issued before this step's keys are counted
        auto load_step = [&](int64_t b, float4 (&x)[kU], float (&al)[kU]) {
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t i = b + 32 * u + r4;
                if (i < r1) {
                    x[u] = __ldg(reinterpret_cast<const float4*>(s + i * n + c0));
                    al[u] = __ldg(alpha + i);
                }
            }
        };
        float4 xn[kU];
        float aln[kU];
        load_step(r0 + 4 * warp, xn, aln);
        for (int64_t b = r0 + 4 * warp; b < r1; b += 32 * kU) {
            float4 x[kU];
            float al[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                x[u] = xn[u];
                al[u] = aln[u];
            }
            load_step(b + 32 * kU, xn, aln);
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (b + 32 * u + r4 < r1) {
                    const float xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t key = desc_key(xv[e] - al[u]);
                        if (shift == 24 || (key >> (shift + 8)) == prefix[e])
                            atomicAdd(&sh[4 * eq + e][(key >> shift) & 255u], 1u);
                    }
                }
            }
        }
    }
    finish_pass(sh, part, last, n, shift, q, col_state, hist, done, bhat, b_new);
}

}  // namespace

// workspace: alpha [m], hist [n][256], pass counters [column blocks + 1], column states [n],
// bhat [n]
struct QbWs {
    size_t alpha, hist, done, cols, bhat, total;
};
static QbWs qb_ws(int64_t m, int n) {
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    QbWs w;
    w.alpha = 0;
    w.hist = al((size_t)m * 4);
    w.done = w.hist + al((size_t)n * 256 * 4);
    w.cols = w.done + al((size_t)((n + 31) / 32 + 1) * 4);
    w.bhat = w.cols + al((size_t)n * sizeof(QbColumn));
    w.total = w.bhat + al((size_t)n * 4);
    return w;
}

size_t qb_workspace_size(int64_t m, int n) { return qb_ws(m, n).total; }

cudaError_t launch_quantile_balance(const float* s, const float* b, int64_t m, int n, int k,
                                    float* b_new, float* bhat_out, float* alpha_out,
                                    void* workspace, cudaStream_t stream) {
    const QbWs L = qb_ws(m, n);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    float* alpha = reinterpret_cast<float*>(w + L.alpha);
    unsigned* hist = reinterpret_cast<unsigned*>(w + L.hist);
    unsigned* done = reinterpret_cast<unsigned*>(w + L.done);
    QbColumn* cols = reinterpret_cast<QbColumn*>(w + L.cols);
    float* bhat = reinterpret_cast<float*>(w + L.bhat);
    if (alpha_out) alpha = alpha_out;
    if (bhat_out) bhat = bhat_out;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // histogram and pass counters cleared (contiguous); every pass leaves them cleared
    cudaError_t e = cudaMemsetAsync(w + L.hist, 0, L.cols - L.hist, stream);
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
    // about two CTAs per SM in total (each warp with a step of loads in flight while it
    // counts the previous one), at least 256 tokens each
    int64_t row_blocks = ((int64_t)sms * 2 + col_blocks - 1) / col_blocks;
    if (row_blocks > (m + 255) / 256) row_blocks = (m + 255) / 256;
    if (row_blocks < 1) row_blocks = 1;
    const int rows_per_cta = (int)((m + row_blocks - 1) / row_blocks);
    row_blocks = (m + rows_per_cta - 1) / rows_per_cta;
    // four experts a lane when the rows allow 16-byte loads
    const bool quad = n % 4 == 0 && (reinterpret_cast<uintptr_t>(s) & 15) == 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
        ProfScope prof("qb_hist_kernel", stream);
        const dim3 grid((unsigned)row_blocks, (unsigned)col_blocks);
        if (quad)
            qb_hist4_kernel<8><<<grid, 256, 0, stream>>>(s, alpha, m, n, rows_per_cta, shift, q, cols,
                                                         hist, done, bhat, b_new);
        else
            qb_hist_kernel<16><<<grid, 256, 0, stream>>>(s, alpha, m, n, rows_per_cta, shift, q, cols,
                                                         hist, done, bhat, b_new);
    }
    return cudaGetLastError();
}

}  // namespace kda
