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
// Then, for n a multiple of 4 and 8192 <= m <= 2^18 (the sampled-bracket path):
//   qb_bracket_kernel a CTA per expert gathers the margins of every 2^sshift-th token (2048
//                     to 4095 of them) and takes, to 16 bits of the key, the sample margins a
//                     few binomial standard deviations either side of the wanted quantile as
//                     the expert's bracket [lo, hi].
//   qb_count_kernel   one pass over all margins: per expert the number above hi, and the
//                     margins in [lo, hi] (a few thousand) copied to the expert's candidate
//                     list.
//   qb_select_kernel  a CTA per expert: when the bracket holds the wanted margin (at most q
//                     margins above hi, at least q + 1 at or above lo) and the list did not
//                     overflow, radix select among the candidates; otherwise among all m
//                     margins of the expert.  The selection is exact either way; the sample
//                     only decides how much work it takes.  The last CTA forms bhat - mean.
// Otherwise (the radix path):
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
// Scores are taken to be finite (a NaN margin has no place in the order).
#include <cmath>

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

__device__ __forceinline__ void cx_desc(uint32_t& a, uint32_t& b) {
    const uint32_t hi = max(a, b), lo = min(a, b);
    a = hi;
    b = lo;
}

// Sort kP keys descending: eight by Batcher's odd-even merge network (19 comparators), other
// counts by odd-even transposition (unrolled).
template <int kP>
__device__ __forceinline__ void sort_desc(uint32_t (&v)[kP]) {
    if constexpr (kP == 8) {
        cx_desc(v[0], v[1]); cx_desc(v[2], v[3]); cx_desc(v[4], v[5]); cx_desc(v[6], v[7]);
        cx_desc(v[0], v[2]); cx_desc(v[1], v[3]); cx_desc(v[4], v[6]); cx_desc(v[5], v[7]);
        cx_desc(v[1], v[2]); cx_desc(v[5], v[6]);
        cx_desc(v[0], v[4]); cx_desc(v[1], v[5]); cx_desc(v[2], v[6]); cx_desc(v[3], v[7]);
        cx_desc(v[2], v[4]); cx_desc(v[3], v[5]);
        cx_desc(v[1], v[2]); cx_desc(v[3], v[4]); cx_desc(v[5], v[6]);
    } else {
#pragma unroll
        for (int rnd = 0; rnd < kP; ++rnd)
#pragma unroll
            for (int e = rnd & 1; e + 1 < kP; e += 2) cx_desc(v[e], v[e + 1]);
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

// bias_new = bhat - mean(bhat), by the last of `total` CTAs to arrive on the counter *ctr
// (which it clears again); the mean in fp64.  part holds a partial sum per warp.
template <int kW>
__device__ __forceinline__ void form_bias(int n, const float* __restrict__ bhat,
                                          float* __restrict__ b_new, unsigned* __restrict__ ctr,
                                          unsigned total, double (&part)[kW], int& last) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(ctr, 1u) == total - 1;
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
    for (int w = 0; w < (int)(blockDim.x / 32); ++w) tot += part[w];
    const double mean = tot / n;
    for (int j = threadIdx.x; j < n; j += blockDim.x)
        b_new[j] = (float)((double)__ldcg(bhat + j) - mean);
    if (threadIdx.x == 0) *ctr = 0u;
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
    const int warp = threadIdx.x >> 5;
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
    form_bias(n, bhat, b_new, done + gridDim.y, gridDim.y, part, last);
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


// ---- the sampled-bracket path ----

// The three kernels after the thresholds are launched as programmatic dependents of the one
// before (their launch and setup overlap its tail); each waits here for that grid to complete
// and its writes to be visible before it reads them.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// One warp: the digit whose bin of the 256 counts h holds position `rank` (a prefix scan over
// the counts, eight bins a lane), and the count of the bins before it.  True on the one lane
// that found it.
__device__ __forceinline__ bool pick_digit(const unsigned* h, uint32_t rank, uint32_t& digit,
                                           uint32_t& before) {
    const int lane = threadIdx.x & 31;
    unsigned c[8];
    unsigned tot = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        c[e] = h[8 * lane + e];
        tot += c[e];
    }
    unsigned incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
    }
    const unsigned excl = incl - tot;
    const unsigned mine = __ballot_sync(0xffffffffu, excl <= rank && rank < incl);
    if (lane != __ffs(mine) - 1) return false;
    before = excl;
    digit = 8 * lane;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        if (rank < before + c[e]) {
            digit = 8 * lane + e;
            break;
        }
        before += c[e];
    }
    return true;
}

// Radix select among the cnt keys key_at(0 .. cnt - 1): the key at 0-based position `rank`
// (rank < cnt) in ascending order, 8-bit digits from bit shift0 + 8 down.  The bits above
// were fixed by the caller in `prefix` (every key shares them); with npass < the remaining
// digits it stops early and returns the prefix of the bin holding the rank (low bits zero).
// kMatch: the keys of a warp step that share a digit add to the count with one
// shared-memory atomic (match_any) -- for key sets whose leading digits are concentrated --
// else one atomic per key.  Every thread of the CTA calls it; hist is shared [256], st shared
// [2].  (hist and st are written by other threads between the barriers, so they must not be
// declared __restrict__: with it the compiler kept the counts and the selected digit of an
// earlier read.)
template <bool kMatch, class KeyAt>
__device__ uint32_t block_select(KeyAt key_at, int64_t cnt, uint32_t rank, uint32_t prefix,
                                 int shift0, int npass, unsigned* hist, uint32_t* st) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int shift = shift0, pass = 0; shift >= 0 && pass < npass; shift -= 8, ++pass) {
        for (int d = threadIdx.x; d < 256; d += blockDim.x) hist[d] = 0u;
        __syncthreads();
        const uint32_t fixed = shift == 24 ? 0u : (0xffffffffu << (shift + 8));
        for (int64_t base = (int64_t)warp * 32; base < cnt; base += (int64_t)nw * 32) {
            const int64_t idx = base + lane;
            unsigned digit = 256u;  // none
            if (idx < cnt) {
                const uint32_t key = key_at(idx);
                if (((key ^ prefix) & fixed) == 0u) digit = (key >> shift) & 255u;
            }
            if (kMatch) {
                const unsigned peers = __match_any_sync(0xffffffffu, digit);
                if (digit < 256u && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], (unsigned)__popc(peers));
            } else if (digit < 256u) {
                atomicAdd(&hist[digit], 1u);
            }
        }
        __syncthreads();
        if (warp == 0) {  // the digit holding the rank
            uint32_t digit, before;
            if (pick_digit(hist, rank, digit, before)) {
                st[0] = prefix | (digit << shift);
                st[1] = rank - before;
            }
        }
        __syncthreads();
        prefix = st[0];
        rank = st[1];
    }
    return prefix;
}

// The bracket of every expert from a sample of the tokens: a CTA per expert gathers the
// margins of every 2^sshift-th token (S of them) and finds, to 16 bits of the key (two
// histogram passes shared by both), the bins holding the sample margins at descending
// positions r_hi and r_lo; hi = the largest value of
// the first bin (+inf when r_hi < 0), lo = the smallest of the second (-inf when r_lo >= S).
// At most r_hi sample margins lie above hi and at least r_lo + 1 at or above lo.  The bracket
// only steers the counting pass; the selection checks afterwards that the wanted margin
// lies inside it, so its precision matters for speed alone.
__global__ void __launch_bounds__(256) qb_bracket_kernel(const float* __restrict__ s,
                                                         const float* __restrict__ alpha, int n,
                                                         int sshift, int S, int r_hi, int r_lo,
                                                         float2* __restrict__ brk) {
    extern __shared__ uint32_t keys[];  // [S]
    __shared__ unsigned hist[512];
    __shared__ uint32_t st[4];
    const int j = blockIdx.x;
    grid_dependency_wait();
    constexpr int kG = 8;  // gathers in flight per thread
    for (int t0 = threadIdx.x; t0 < S; t0 += kG * blockDim.x) {
        float x[kG], a[kG];
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            const int t = t0 + g * blockDim.x;
            const int64_t i = (int64_t)min(t, S - 1) << sshift;
            x[g] = __ldg(s + i * n + j);
            a[g] = __ldg(alpha + i);
        }
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            const int t = t0 + g * blockDim.x;
            if (t < S) keys[t] = desc_key((x[g] - a[g]) + 0.f);
        }
    }
    __syncthreads();
    // both positions at once: one histogram of the top byte, then one of the second byte
    // for each of the two bins found (warp 0 picks for hi, warp 1 for lo)
    const int warp = threadIdx.x >> 5;
    const uint32_t rank[2] = {(uint32_t)max(r_hi, 0), (uint32_t)min(r_lo, S - 1)};
    for (int d = threadIdx.x; d < 512; d += blockDim.x) hist[d] = 0u;
    __syncthreads();
    for (int t = threadIdx.x; t < S; t += blockDim.x) atomicAdd(&hist[keys[t] >> 24], 1u);
    __syncthreads();
    if (warp < 2) {
        uint32_t digit, before;
        if (pick_digit(hist, rank[warp], digit, before)) {
            st[2 * warp] = digit;
            st[2 * warp + 1] = rank[warp] - before;
        }
    }
    __syncthreads();
    const uint32_t top0 = st[0], top1 = st[2], rest0 = st[1], rest1 = st[3];
    for (int d = threadIdx.x; d < 512; d += blockDim.x) hist[d] = 0u;
    __syncthreads();
    for (int t = threadIdx.x; t < S; t += blockDim.x) {
        const uint32_t key = keys[t], d2 = (key >> 16) & 255u;
        if ((key >> 24) == top0) atomicAdd(&hist[d2], 1u);
        if ((key >> 24) == top1) atomicAdd(&hist[256 + d2], 1u);
    }
    __syncthreads();
    if (warp < 2) {
        uint32_t digit, before;
        if (pick_digit(hist + 256 * warp, warp ? rest1 : rest0, digit, before))
            st[2 * warp] = ((warp ? top1 : top0) << 24) | (digit << 16);
    }
    __syncthreads();
    float hi = INFINITY, lo = -INFINITY;
    if (r_hi >= 0) hi = key_value(st[0]);
    if (r_lo < S) lo = key_value(st[2] | 0xffffu);
    // +0 for a zero bound, as for the margins, so that the candidates' keys lie between the
    // bounds' keys
    if (threadIdx.x == 0) brk[j] = make_float2(lo + 0.f, hi + 0.f);
}

constexpr int kCountSlots = 8;          // candidates a thread stages per expert
constexpr int kCountStride = 4 * kCountSlots + 1;  // words per thread (padded against conflicts)
constexpr int kSelKeys = 8192;          // candidates the selection stages in shared memory

// The counting pass over all margins (n a multiple of 4, 16-byte aligned scores): per expert,
// the number of margins above hi, and the margins in [lo, hi] appended to the expert's
// candidate list of `cap` entries (the count keeps growing past cap, which
// tells the selection that the list overflowed).  A CTA takes 256 experts (64 quads of four
// consecutive experts, a lane per quad, so that a warp load reads 512 contiguous bytes of a
// row) and four interleaved token streams over its range; the next step's loads are issued
// before the current step is compared.  A thread keeps its experts' counts in registers and
// its candidates in its own shared-memory slots (kCountSlots per expert, past which it appends
// to the global list directly); at the end the CTA reserves each expert's place in the list
// with one global atomic and copies the staged candidates there.
template <int kU>
__global__ void __launch_bounds__(256, 3) qb_count_kernel(const float* __restrict__ s,
                                                          const float* __restrict__ alpha,
                                                          int64_t m, int n, int rows_per_cta,
                                                          const float2* __restrict__ brk,
                                                          unsigned* __restrict__ cnt_hi,
                                                          unsigned* __restrict__ cand_cnt,
                                                          float* __restrict__ cand, int cap) {
    __shared__ unsigned sh[256];     // margins above hi, per expert
    __shared__ unsigned scnt[256];   // staged candidates, per expert; then the CTA's base
    __shared__ float sbuf[256 * kCountStride];
    const int qd = threadIdx.x & 63, rl = threadIdx.x >> 6;
    const int c0 = blockIdx.y * 256 + 4 * qd;
    const bool live = c0 < n;
    grid_dependency_wait();
    sh[threadIdx.x] = 0u;
    scnt[threadIdx.x] = 0u;
    __syncthreads();
    float* mine = sbuf + threadIdx.x * kCountStride;
    unsigned nc[4] = {0u, 0u, 0u, 0u};
    const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
    const int64_t r1 = min(m, r0 + rows_per_cta);
    if (live) {
        float lo[4], hi[4];
        unsigned ch[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 b2 = __ldcg(brk + c0 + e);
            lo[e] = b2.x;
            hi[e] = b2.y;
        }
        // a step: rows b + 4 u for u < kU; b = r0 + rl + 4 kU (step)
        auto load_step = [&](int64_t b, float4 (&x)[kU], float (&al)[kU]) {
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t i = b + 4 * u;
                if (i < r1) {
                    x[u] = __ldg(reinterpret_cast<const float4*>(s + i * n + c0));
                    al[u] = __ldg(alpha + i);
                }
            }
        };
        float4 xn[kU];
        float aln[kU];
        load_step(r0 + rl, xn, aln);
        for (int64_t b = r0 + rl; b < r1; b += 4 * kU) {
            float4 x[kU];
            float al[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                x[u] = xn[u];
                al[u] = aln[u];
            }
            load_step(b + 4 * kU, xn, aln);
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (b + 4 * u < r1) {
                    const float xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
                    // the row's four comparisons first, then one branch into the candidates
                    float mg[4];
                    unsigned cm = 0u;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        mg[e] = xv[e] - al[u];
                        const bool above = mg[e] > hi[e];
                        ch[e] += above ? 1u : 0u;
                        cm |= (!above && mg[e] >= lo[e]) ? (1u << e) : 0u;
                    }
                    if (cm) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if ((cm >> e) & 1u) {
                                if (nc[e] < (unsigned)kCountSlots) {
                                    mine[e * kCountSlots + nc[e]] = mg[e];
                                } else {  // this thread's slots are full: straight to the list
                                    const unsigned g = atomicAdd(cand_cnt + c0 + e, 1u);
                                    if (g < (unsigned)cap) cand[(int64_t)(c0 + e) * cap + g] = mg[e];
                                }
                                ++nc[e];
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (ch[e]) atomicAdd(&sh[4 * qd + e], ch[e]);
    }
    // each thread's place among the CTA's staged candidates of its experts
    unsigned off[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        nc[e] = min(nc[e], (unsigned)kCountSlots);
        off[e] = nc[e] ? atomicAdd(&scnt[4 * qd + e], nc[e]) : 0u;
    }
    __syncthreads();
    // one global atomic per expert for the count above, one to reserve the CTA's candidates
    const int col = blockIdx.y * 256 + threadIdx.x;
    if (col < n) {
        if (sh[threadIdx.x]) atomicAdd(cnt_hi + col, sh[threadIdx.x]);
        const unsigned c = scnt[threadIdx.x];
        sh[threadIdx.x] = c ? atomicAdd(cand_cnt + col, c) : 0u;  // the CTA's base in the list
    }
    __syncthreads();
    if (live) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const unsigned base = sh[4 * qd + e] + off[e];
            for (unsigned t = 0; t < nc[e]; ++t)
                if (base + t < (unsigned)cap)
                    cand[(int64_t)(c0 + e) * cap + base + t] = mine[e * kCountSlots + t];
        }
    }
}

// The selection, a CTA per expert: when the wanted margin (descending position q) lies in
// the bracket -- at most q margins above hi, at least q + 1 at or above lo -- and the list
// did not overflow, it is the candidate at descending position q - (count above hi), selected
// in shared memory when the list fits kSelKeys;
// otherwise the CTA selects position q among all m margins of the expert, recomputed from
// the scores and thresholds.  bhat = -(that margin); the last CTA forms bias_new.
__global__ void __launch_bounds__(512) qb_select_kernel(const float* __restrict__ s,
                                                        const float* __restrict__ alpha, int64_t m,
                                                        int n, uint32_t q,
                                                        const float2* __restrict__ brk,
                                                        const unsigned* __restrict__ cnt_hi,
                                                        const unsigned* __restrict__ cand_cnt,
                                                        const float* __restrict__ cand, int cap,
                                                        float* __restrict__ bhat,
                                                        float* __restrict__ b_new,
                                                        unsigned* __restrict__ done) {
    extern __shared__ uint32_t skeys[];  // [kSelKeys]
    __shared__ unsigned hist[256];
    __shared__ uint32_t st[2];
    __shared__ double part[16];
    __shared__ int last;
    const int j = blockIdx.x;
    grid_dependency_wait();
    const unsigned above = __ldcg(cnt_hi + j), mid = __ldcg(cand_cnt + j);
    const float2 b2 = __ldcg(brk + j);
    uint32_t key;
    if (above <= q && (uint64_t)above + mid >= (uint64_t)q + 1u && mid <= (unsigned)cap) {
        // every candidate lies in [lo, hi], so its key shares the leading bits of the keys of
        // hi and lo: the whole bytes of those are fixed, the digits start below them
        const uint32_t k0 = desc_key(b2.y), k1 = desc_key(b2.x);
        const int same = (k0 == k1) ? 32 : __clz(k0 ^ k1);
        const int bytes = same >= 32 ? 3 : same / 8;  // whole leading bytes fixed (at most 3)
        const uint32_t prefix = bytes == 0 ? 0u : (k0 & (0xffffffffu << (32 - 8 * bytes)));
        const int shift0 = 24 - 8 * bytes;
        const float* cj = cand + (int64_t)j * cap;
        if (mid <= (unsigned)kSelKeys) {  // the list staged in shared memory (one read) as keys
            for (unsigned t0 = threadIdx.x; t0 < mid; t0 += 8 * blockDim.x) {
                float v[8];
#pragma unroll
                for (int g = 0; g < 8; ++g) v[g] = __ldcg(cj + min(t0 + g * blockDim.x, mid - 1));
#pragma unroll
                for (int g = 0; g < 8; ++g)
                    if (t0 + g * blockDim.x < mid) skeys[t0 + g * blockDim.x] = desc_key(v[g] + 0.f);
            }
            __syncthreads();
            key = block_select<false>([&](int64_t idx) { return skeys[idx]; }, (int64_t)mid,
                                      q - above, prefix, shift0, 4, hist, st);
        } else {
            key = block_select<false>([&](int64_t idx) { return desc_key(__ldcg(cj + idx) + 0.f); },
                                      (int64_t)mid, q - above, prefix, shift0, 4, hist, st);
        }
    } else {
        key = block_select<true>([&](int64_t i) { return desc_key((__ldg(s + i * n + j) - __ldcg(alpha + i)) + 0.f); },
                                 m, q, 0u, 24, 4, hist, st);
    }
    if (threadIdx.x == 0) bhat[j] = -key_value(key);
    form_bias(n, bhat, b_new, done, gridDim.x, part, last);
}

}  // namespace

// workspace of the radix path: alpha [m], hist [n][256], pass counters [column blocks + 1],
// column states [n], bhat [n]
struct QbWs {
    size_t alpha, hist, done, cols, bhat, total;
};
static size_t al256(size_t x) { return (x + 255) & ~size_t(255); }
static QbWs qb_ws(int64_t m, int n) {
    QbWs w;
    w.alpha = 0;
    w.hist = al256((size_t)m * 4);
    w.done = w.hist + al256((size_t)n * 256 * 4);
    w.cols = w.done + al256((size_t)((n + 31) / 32 + 1) * 4);
    w.bhat = w.cols + al256((size_t)n * sizeof(QbColumn));
    w.total = w.bhat + al256((size_t)n * 4);
    return w;
}

// The sampled-bracket path: for n a multiple of 4 and 8192 <= m <= 2^18, every 2^sshift-th
// token (S = ceil(m / 2^sshift) in [2048, 4096) of them) is sampled, and every expert's
// candidate list holds `cap` margins: three times the number a bracket of
// 6 sqrt(S p (1 - p)) + 4 sample positions either side of the wanted one takes in
// expectation, at p (1 - p) <= 1/4, so the size does not depend on k.  Workspace: alpha [m],
// brackets [n], counts above [n], candidate counts [n], the done counter, bhat [n],
// candidates [n][cap]; at most 64 MiB of candidates, else the radix path.
struct QbFast {
    bool ok;
    int sshift, S, cap;
    size_t alpha, brk, cnt_hi, cand_cnt, done, bhat, cand, total;
};
static QbFast qb_fast(int64_t m, int n) {
    QbFast f{};
    f.ok = false;
    if (n % 4 != 0 || m < 8192 || m > (int64_t(1) << 18)) return f;
    f.sshift = 0;
    while ((m >> (f.sshift + 1)) >= 2048) ++f.sshift;
    f.S = (int)((m + (int64_t(1) << f.sshift) - 1) >> f.sshift);
    const double dmax = 3.0 * std::sqrt((double)f.S) + 4.0;
    const double expect = 2.0 * dmax * (double)(int64_t(1) << f.sshift) + 64.0;
    int64_t cap = 1024;
    while ((double)cap < 3.0 * expect) cap *= 2;
    if ((double)n * (double)cap * 4.0 > 64.0 * 1024 * 1024) return f;
    f.cap = (int)cap;
    f.alpha = 0;
    f.brk = al256((size_t)m * 4);
    f.cnt_hi = f.brk + al256((size_t)n * 8);
    f.cand_cnt = f.cnt_hi + al256((size_t)n * 4);
    f.done = f.cand_cnt + al256((size_t)n * 4);
    f.bhat = f.done + 256;
    f.cand = f.bhat + al256((size_t)n * 4);
    f.total = f.cand + al256((size_t)n * cap * 4);
    f.ok = true;
    return f;
}

size_t qb_workspace_size(int64_t m, int n) {
    const QbFast f = qb_fast(m, n);
    return f.ok ? f.total : qb_ws(m, n).total;
}

static cudaError_t launch_alpha(const float* s, const float* b, int64_t m, int n, int k,
                                float* alpha, int sms, cudaStream_t stream) {
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
    return cudaGetLastError();
}

// a launch that may begin while the previous kernel on the stream finishes (the kernel waits
// for it with griddepcontrol.wait)
template <typename... KArgs, typename... Args>
static cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

static cudaError_t launch_fast(const QbFast& f, const float* s, const float* b, int64_t m,
                               int n, int k, float* b_new, float* bhat_out, float* alpha_out,
                               uint8_t* w, int sms, cudaStream_t stream) {
    float* alpha = alpha_out ? alpha_out : reinterpret_cast<float*>(w + f.alpha);
    float2* brk = reinterpret_cast<float2*>(w + f.brk);
    unsigned* cnt_hi = reinterpret_cast<unsigned*>(w + f.cnt_hi);
    unsigned* cand_cnt = reinterpret_cast<unsigned*>(w + f.cand_cnt);
    unsigned* done = reinterpret_cast<unsigned*>(w + f.done);
    float* bhat = bhat_out ? bhat_out : reinterpret_cast<float*>(w + f.bhat);
    float* cand = reinterpret_cast<float*>(w + f.cand);
    const uint32_t q = (uint32_t)((m * k) / n);
    // the sample positions of the bracket: the wanted margin is the (q+1)-th largest, so
    // about q S / m sample margins lie above it; delta = 6 binomial standard deviations + 4
    const double p = (double)(q + 1) / (double)m;
    const double delta = 6.0 * std::sqrt((double)f.S * p * (1.0 - p)) + 4.0;
    const double r_hi_d = std::floor((double)q * f.S / (double)m - delta);
    const double r_lo_d = std::ceil((double)(q + 1) * f.S / (double)m + delta);
    const int r_hi = r_hi_d < 0.0 ? -1 : (int)r_hi_d;
    const int r_lo = r_lo_d >= (double)f.S ? f.S : (int)r_lo_d;
    // counts and the done counter cleared (contiguous)
    cudaError_t e = cudaMemsetAsync(w + f.cnt_hi, 0, f.bhat - f.cnt_hi, stream);
    if (e == cudaSuccess) e = launch_alpha(s, b, m, n, k, alpha, sms, stream);
    if (e != cudaSuccess) return e;
    {
        const int smem = f.S * 4;
        e = cudaFuncSetAttribute(qb_bracket_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        ProfScope prof("qb_bracket_kernel", stream);
        e = launch_dependent(qb_bracket_kernel, dim3(n), dim3(256), smem, stream, s,
                             (const float*)alpha, n, f.sshift, f.S, r_hi, r_lo, brk);
        if (e != cudaSuccess) return e;
    }
    {
        const int col_blocks = (n + 255) / 256;
        int64_t row_blocks = ((int64_t)sms * 3 + col_blocks - 1) / col_blocks;
        const int rows_per_cta = (int)((m + row_blocks - 1) / row_blocks);
        row_blocks = (m + rows_per_cta - 1) / rows_per_cta;
        ProfScope prof("qb_count_kernel", stream);
        e = launch_dependent(qb_count_kernel<4>, dim3((unsigned)row_blocks, (unsigned)col_blocks),
                             dim3(256), 0, stream, s, (const float*)alpha, m, n, rows_per_cta,
                             (const float2*)brk, cnt_hi, cand_cnt, cand, f.cap);
        if (e != cudaSuccess) return e;
    }
    {
        const int smem = kSelKeys * 4;
        e = cudaFuncSetAttribute(qb_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        ProfScope prof("qb_select_kernel", stream);
        e = launch_dependent(qb_select_kernel, dim3(n), dim3(512), smem, stream, s,
                             (const float*)alpha, m, n, q, (const float2*)brk,
                             (const unsigned*)cnt_hi, (const unsigned*)cand_cnt,
                             (const float*)cand, f.cap, bhat, b_new, done);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_quantile_balance(const float* s, const float* b, int64_t m, int n, int k,
                                    float* b_new, float* bhat_out, float* alpha_out,
                                    void* workspace, cudaStream_t stream) {
    uint8_t* w = static_cast<uint8_t*>(workspace);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const QbFast f = qb_fast(m, n);
    if (f.ok && (reinterpret_cast<uintptr_t>(s) & 15) == 0)
        return launch_fast(f, s, b, m, n, k, b_new, bhat_out, alpha_out, w, sms, stream);
    const QbWs L = qb_ws(m, n);
    float* alpha = reinterpret_cast<float*>(w + L.alpha);
    unsigned* hist = reinterpret_cast<unsigned*>(w + L.hist);
    unsigned* done = reinterpret_cast<unsigned*>(w + L.done);
    QbColumn* cols = reinterpret_cast<QbColumn*>(w + L.cols);
    float* bhat = reinterpret_cast<float*>(w + L.bhat);
    if (alpha_out) alpha = alpha_out;
    if (bhat_out) bhat = bhat_out;
    // histogram and pass counters cleared (contiguous); every pass leaves them cleared
    cudaError_t e = cudaMemsetAsync(w + L.hist, 0, L.cols - L.hist, stream);
    if (e == cudaSuccess) e = launch_alpha(s, b, m, n, k, alpha, sms, stream);
    if (e != cudaSuccess) return e;
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
