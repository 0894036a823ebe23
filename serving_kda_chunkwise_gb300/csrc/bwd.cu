// bwd.cu -- gradients of the KDA forward with respect to q, k, v, beta, z, A_log and S0.
//
// "Kimi k3 技术报告详解（1）——架构再升华", section "Kimi Delta Attention": per token
//   alpha = exp(g),  g = g_min Sigmoid(x),  x = e^{A_h} z       (section "Chunkwise parallel form")
//   S' = Diag(alpha) S_{t-1};   w = v - S'^T k;   u = beta w;   S_t = S' + k u^T;   o = S_t^T q
// and, for a loss with gradients do_t (and dS_out for the final state), reverse mode gives,
// with dS the gradient of S_t:
//   dS += q do^T;   dq = S_t do;   du = dS^T k;   dv = beta du;   dbeta = du . w;
//   dk = dS u - S' (beta du);   dS' = dS - k (beta du)^T;   dalpha_i = sum_j dS'_ij S_{t-1,ij};
//   dS <- Diag(alpha) dS';   dx = dalpha alpha g_min s (1 - s), s = Sigmoid(x);
//   dz = dx e^{A_h};   dA_h += sum dx x.
// The pages print no backward; these are the derivatives of the forward they define.
//
// Parallel over chunks.  For bf16 problems the states at the chunk starts come from the
// tensor-core forward (its chain stage writes them, no output); otherwise, and for the rest,
// on CUDA cores in fp32.  The state and its gradient are the only
// serial quantities, and over one 64-token chunk both are affine.  Forward, S_t =
// (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T, so S_(chunk end) =
// A S_(chunk start) + B.  Backward, going back through token t maps dS_t to
// B_t (dS_t + q_t do_t^T) with B_t = Diag(alpha_t) (I - beta_t k_t k_t^T), so
//   dS_(chunk start) = Phi dS_(chunk end) + Psi,  Phi = B_t0 .. B_t1-1,
//   Psi = sum_t B_t0 .. B_t (q_t do_t^T).
// Kernels (512 threads; in the per-chunk kernels warp w owns rows [w dk/16, (w+1) dk/16) of a
// state-shaped matrix and lane l its columns l, l + 32, ..; matrices live in registers, and
// each chunk's token inputs are staged in shared memory once):
//   bwd_plan_kernel   chunk offsets of every sequence and a table entry per chunk
//   (bf16)            the tensor-core forward (fwd_tc.cu, two-launch form) with its chain
//                     stage writing the state at every chunk start, the checkpoints, then
//                     the gradient chain on the tensor cores (bwd_chain_tc.cu) reading its
//                     chunk packages: dS at every chunk end and dS0.  They replace the next
//                     four kernels.
//   bwd_fwdtrans_kernel  per (chunk, head), all in parallel: the chunk's forward map on the
//                     state, S_end = A S_start + B
//   bwd_chain_kernel<fwd>  per (sequence, head, 32-column slice): S at every chunk start
//                     (S <- A S + B, first chunk first), the checkpoints
//   bwd_phi_kernel    per (chunk, head), all in parallel: Phi and Psi of the chunk
//   bwd_chain_kernel  per (sequence, head, 32-column slice): dS at every chunk end, last
//                     chunk first (dS <- Phi dS + Psi), and dS0
//   bwd_item_kernel   per (chunk, head), all in parallel: the reverse rules above token by
//                     token from the chunk's dS, the state before each token recomputed from
//                     the chunk's checkpoint by 8-token sub-blocks (per-CTA scratch)
//   bwd_dA_kernel     dA_log[h] = the per-(chunk, head) partial sums in chunk order
//                     (deterministic)
#include <map>
#include <mutex>

#include "bwd_tc_layout.cuh"
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kBwdThreads = 512;
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int kBwdC = 64;


template <int DK, int DV>
struct BwdLayout {
    static constexpr int RPW = DK / kBwdWarps;  // rows per warp
    static constexpr int CPL = DV / 32;         // columns per lane
};

struct BwdParams {
    const void *q, *k, *v, *beta, *z, *dout;
    const float* A_log;
    float g_min;
    const float* S0;
    const float* dS_out;
    const int32_t* cu;
    int N, H;
    int64_t T_total;
    void *dq, *dk, *dv, *dbeta, *dz;
    float* dS0;
    int32_t* chunk_off;  // [N + 1]: first global chunk of each sequence, then the total
    int4* chunk_tab;     // [chunks]: {first token (low, high), sequence, rows}
    float* ckpt;         // [chunks][H][DK][DV]: the state at each chunk start
    float* phi;          // [chunks][H][DK][DK]
    float* psi;          // [chunks][H][DK][DV]
    float* dsend;        // [chunks][H][DK][DV]: the state's gradient at each chunk end
    float* snap;         // [grid][16][DK][DV]: per-CTA scratch (sub-block starts, token states)
    float* dA_item;      // [chunks][H]
    unsigned* err;
};

// chunk offsets (serial scan by one thread: N is small next to the work) and the chunk table
__global__ void __launch_bounds__(1024) bwd_plan_kernel(const int32_t* __restrict__ cu, int N,
                                                        int64_t T_total, int32_t* chunk_off,
                                                        int4* chunk_tab, unsigned* err) {
    if (threadIdx.x == 0) {
        int32_t acc = 0;
        for (int n = 0; n < N; ++n) {
            int64_t b, e;
            seq_range(cu, n, N, T_total, err, b, e);
            chunk_off[n] = acc;
            acc += (int32_t)((e - b + kBwdC - 1) / kBwdC);
        }
        chunk_off[N] = acc;
    }
    __syncthreads();
    const int32_t total = chunk_off[N];
    for (int32_t c = threadIdx.x; c < total; c += blockDim.x) {
        int lo = 0, hi = N - 1;  // the last sequence whose first chunk is <= c
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (chunk_off[mid] <= c) lo = mid;
            else hi = mid - 1;
        }
        int64_t b, e;
        seq_range(cu, lo, N, T_total, nullptr, b, e);
        const int64_t t0 = b + (int64_t)(c - chunk_off[lo]) * kBwdC;
        const int64_t rows = e - t0 < kBwdC ? e - t0 : kBwdC;
        chunk_tab[c] = make_int4((int)(t0 & 0xffffffff), (int)(t0 >> 32), lo, (int)rows);
    }
}

// One chunk's token inputs, staged in (dynamic) shared memory as fp32 by the whole CTA at the
// start of an item, so that the per-token steps read no global memory: k, q [64][DK], the
// gate's x = e^{A_h} z and alpha = exp(g) [64][DK], v, do [64][DV], beta [64].  Arrays a
// kernel does not use are given no space (nullptr).
template <int DK, int DV>
struct Stage {
    float *k, *q, *x, *a, *v, *dout, *beta;
};

// the floats a Stage with these arrays occupies (k and alpha always, beta always)
template <int DK, int DV>
__host__ __device__ constexpr int stage_floats(bool q, bool x, bool v, bool dout) {
    return kBwdC * DK * (2 + (q ? 1 : 0) + (x ? 1 : 0)) +
           kBwdC * DV * ((v ? 1 : 0) + (dout ? 1 : 0)) + kBwdC;
}

// carve the arrays out of `base` in a fixed order (the layout stage_floats counts)
template <int DK, int DV>
__device__ __forceinline__ Stage<DK, DV> stage_carve(float* base, bool q, bool x, bool v,
                                                     bool dout) {
    Stage<DK, DV> st{};
    st.k = base;            base += kBwdC * DK;
    st.a = base;            base += kBwdC * DK;
    if (q) { st.q = base;   base += kBwdC * DK; }
    if (x) { st.x = base;   base += kBwdC * DK; }
    if (v) { st.v = base;   base += kBwdC * DV; }
    if (dout) { st.dout = base; base += kBwdC * DV; }
    st.beta = base;
    return st;
}

template <typename IO, int DK, int DV>
__device__ __forceinline__ void stage_chunk(const Stage<DK, DV>& st, const BwdParams& p,
                                            int64_t t0, int rows, int h, float scale) {
    const IO* k = static_cast<const IO*>(p.k);
    const IO* q = static_cast<const IO*>(p.q);
    const IO* z = static_cast<const IO*>(p.z);
    const IO* v = static_cast<const IO*>(p.v);
    const IO* dout = static_cast<const IO*>(p.dout);
    const IO* beta = static_cast<const IO*>(p.beta);
    const size_t kb = ((size_t)t0 * p.H + h) * DK, vb = ((size_t)t0 * p.H + h) * DV;
    for (int idx = threadIdx.x; idx < rows * DK; idx += kBwdThreads) {
        const int tt = idx / DK, i = idx % DK;
        const size_t o = kb + (size_t)tt * p.H * DK + i;
        st.k[idx] = to_f32(k[o]);
        if (st.q) st.q[idx] = to_f32(q[o]);
        const float xv = scale * to_f32(z[o]);
        if (st.x) st.x[idx] = xv;
        st.a[idx] = expf(p.g_min / (1.0f + expf(-xv)));
    }
    if (st.v || st.dout) {
        for (int idx = threadIdx.x; idx < rows * DV; idx += kBwdThreads) {
            const int tt = idx / DV, j = idx % DV;
            const size_t o = vb + (size_t)tt * p.H * DV + j;
            if (st.v) st.v[idx] = to_f32(v[o]);
            if (st.dout) st.dout[idx] = to_f32(dout[o]);
        }
    }
    for (int tt = threadIdx.x; tt < rows; tt += kBwdThreads)
        st.beta[tt] = to_f32(beta[(size_t)(t0 + tt) * p.H + h]);
}

// the item (chunk, head) `it`: head, first token, rows
__device__ __forceinline__ void item_of(const BwdParams& p, int64_t it, int& h, int64_t& t0,
                                        int& rows) {
    h = (int)(it % p.H);
    const int4 e = p.chunk_tab[it / p.H];
    t0 = (static_cast<int64_t>(e.y) << 32) | static_cast<uint32_t>(e.x);
    rows = e.w;
}

// a warp's RPW consecutive rows of a staged [DK] vector, as 16-byte shared-memory loads
template <int RPW>
__device__ __forceinline__ void load_rows(const float* v, int warp, float (&out)[RPW]) {
    static_assert(RPW % 4 == 0, "rows per warp");
    const float4* v4 = reinterpret_cast<const float4*>(v + warp * RPW);
#pragma unroll
    for (int x = 0; x < RPW / 4; ++x) {
        const float4 f = v4[x];
        out[4 * x] = f.x;
        out[4 * x + 1] = f.y;
        out[4 * x + 2] = f.z;
        out[4 * x + 3] = f.w;
    }
}

// Phi and Psi of every (chunk, head) in parallel, tokens in reverse from Phi = I, Psi = 0:
// X <- Diag(alpha) (I - beta k k^T) X per token, and Psi += q do^T before its step.
template <typename IO, int DK, int DV>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_phi_kernel(const BwdParams p) {
    using L = BwdLayout<DK, DV>;
    constexpr int CK = DK / 32;  // Phi columns per lane
    extern __shared__ __align__(16) float stage_smem[];
    const Stage<DK, DV> st = stage_carve<DK, DV>(stage_smem, true, false, false, true);
    // per-warp column sums and their totals, in buffers alternating with the token's parity
    __shared__ float partA[2][kBwdWarps][DK];
    __shared__ float partB[2][kBwdWarps][DV];
    __shared__ float duA[2][DK], duB[2][DV];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t items = (int64_t)p.chunk_off[p.N] * p.H;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        int h, rows;
        int64_t t0;
        item_of(p, it, h, t0, rows);
        __syncthreads();  // the previous item's staged inputs are consumed
        stage_chunk<IO, DK, DV>(st, p, t0, rows, h, expf(p.A_log[h]));
        float Phi[L::RPW][CK], Psi[L::RPW][L::CPL];
#pragma unroll
        for (int r = 0; r < L::RPW; ++r) {
#pragma unroll
            for (int c = 0; c < CK; ++c) Phi[r][c] = (warp * L::RPW + r == lane + 32 * c) ? 1.f : 0.f;
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) Psi[r][c] = 0.f;
        }
        __syncthreads();
        for (int tt = rows - 1; tt >= 0; --tt) {
            const int b = tt & 1;
            const float* kt = st.k + tt * DK;
            const float* qt = st.q + tt * DK;
            const float* at = st.a + tt * DK;
            const float* dot = st.dout + tt * DV;
            // Psi += q do^T; column sums of Phi^T k and Psi^T k
            float pa[CK], pb[L::CPL], doj[L::CPL];
#pragma unroll
            for (int c = 0; c < CK; ++c) pa[c] = 0.f;
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) {
                pb[c] = 0.f;
                doj[c] = dot[lane + 32 * c];
            }
            float kr[L::RPW], qr[L::RPW];
            load_rows<L::RPW>(kt, warp, kr);
            load_rows<L::RPW>(qt, warp, qr);
#pragma unroll
            for (int r = 0; r < L::RPW; ++r) {
                const float kk = kr[r], qq = qr[r];
#pragma unroll
                for (int c = 0; c < CK; ++c) pa[c] = fmaf(Phi[r][c], kk, pa[c]);
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) {
                    Psi[r][c] = fmaf(qq, doj[c], Psi[r][c]);
                    pb[c] = fmaf(Psi[r][c], kk, pb[c]);
                }
            }
#pragma unroll
            for (int c = 0; c < CK; ++c) partA[b][warp][lane + 32 * c] = pa[c];
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) partB[b][warp][lane + 32 * c] = pb[c];
            __syncthreads();
            if (tid < DK) {
                float sa = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kBwdWarps; ++w2) sa += partA[b][w2][tid];
                duA[b][tid] = sa;
            } else if (tid >= 256 && tid < 256 + DV) {
                float sb = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kBwdWarps; ++w2) sb += partB[b][w2][tid - 256];
                duB[b][tid - 256] = sb;
            }
            __syncthreads();
            // X <- Diag(alpha) (X - beta k du^T) for X = Phi and Psi
            const float bt = st.beta[tt];
            float ar[L::RPW];
            load_rows<L::RPW>(at, warp, ar);
#pragma unroll
            for (int r = 0; r < L::RPW; ++r) {
                const float a = ar[r], bk = bt * kr[r];
#pragma unroll
                for (int c = 0; c < CK; ++c) Phi[r][c] = a * fmaf(-bk, duA[b][lane + 32 * c], Phi[r][c]);
#pragma unroll
                for (int c = 0; c < L::CPL; ++c)
                    Psi[r][c] = a * fmaf(-bk, duB[b][lane + 32 * c], Psi[r][c]);
            }
        }
        float* ph = p.phi + (size_t)it * DK * DK;
        float* ps = p.psi + (size_t)it * DK * DV;
#pragma unroll
        for (int r = 0; r < L::RPW; ++r) {
            const int i = warp * L::RPW + r;
#pragma unroll
            for (int c = 0; c < CK; ++c) ph[i * DK + lane + 32 * c] = Phi[r][c];
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) ps[i * DV + lane + 32 * c] = Psi[r][c];
        }
    }
}

// The forward map of one chunk on the state, S_end = A S_start + B, for every (chunk, head) in
// parallel: A and B follow the token recurrence from A = I, B = 0 (per token X <- Diag(alpha)X,
// then X <- X - beta k (k^T X)^T, and for B also + beta k v^T).  Stored in the Phi / Psi
// buffers, which the backward stages reuse afterwards.
template <typename IO, int DK, int DV>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_fwdtrans_kernel(const BwdParams p) {
    using L = BwdLayout<DK, DV>;
    constexpr int CK = DK / 32;
    extern __shared__ __align__(16) float stage_smem[];
    const Stage<DK, DV> st = stage_carve<DK, DV>(stage_smem, false, false, true, false);
    __shared__ float partA[2][kBwdWarps][DK];
    __shared__ float partB[2][kBwdWarps][DV];
    __shared__ float wA[2][DK], wB[2][DV];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t items = (int64_t)p.chunk_off[p.N] * p.H;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        int h, rows;
        int64_t t0;
        item_of(p, it, h, t0, rows);
        __syncthreads();  // the previous item's staged inputs are consumed
        stage_chunk<IO, DK, DV>(st, p, t0, rows, h, expf(p.A_log[h]));
        float A[L::RPW][CK], B[L::RPW][L::CPL];
#pragma unroll
        for (int r = 0; r < L::RPW; ++r) {
#pragma unroll
            for (int c = 0; c < CK; ++c) A[r][c] = (warp * L::RPW + r == lane + 32 * c) ? 1.f : 0.f;
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) B[r][c] = 0.f;
        }
        __syncthreads();
        for (int tt = 0; tt < rows; ++tt) {
            const int b = tt & 1;
            const float* kt = st.k + tt * DK;
            const float* at = st.a + tt * DK;
            float pa[CK], pb[L::CPL];
#pragma unroll
            for (int c = 0; c < CK; ++c) pa[c] = 0.f;
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) pb[c] = 0.f;
            float kr[L::RPW], ar[L::RPW];
            load_rows<L::RPW>(kt, warp, kr);
            load_rows<L::RPW>(at, warp, ar);
#pragma unroll
            for (int r = 0; r < L::RPW; ++r) {
                const float a = ar[r], kk = kr[r];
#pragma unroll
                for (int c = 0; c < CK; ++c) {
                    A[r][c] *= a;
                    pa[c] = fmaf(A[r][c], kk, pa[c]);
                }
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) {
                    B[r][c] *= a;
                    pb[c] = fmaf(B[r][c], kk, pb[c]);
                }
            }
#pragma unroll
            for (int c = 0; c < CK; ++c) partA[b][warp][lane + 32 * c] = pa[c];
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) partB[b][warp][lane + 32 * c] = pb[c];
            __syncthreads();
            if (tid < DK) {
                float sa = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kBwdWarps; ++w2) sa += partA[b][w2][tid];
                wA[b][tid] = sa;
            } else if (tid >= 256 && tid < 256 + DV) {
                float sb = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kBwdWarps; ++w2) sb += partB[b][w2][tid - 256];
                wB[b][tid - 256] = sb - st.v[tt * DV + tid - 256];  // (k^T B') - v
            }
            __syncthreads();
            const float bt = st.beta[tt];
#pragma unroll
            for (int r = 0; r < L::RPW; ++r) {
                const float bk = bt * kr[r];
#pragma unroll
                for (int c = 0; c < CK; ++c) A[r][c] = fmaf(-bk, wA[b][lane + 32 * c], A[r][c]);
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) B[r][c] = fmaf(-bk, wB[b][lane + 32 * c], B[r][c]);
            }
        }
        float* pa_out = p.phi + (size_t)it * DK * DK;
        float* pb_out = p.psi + (size_t)it * DK * DV;
#pragma unroll
        for (int r = 0; r < L::RPW; ++r) {
            const int i = warp * L::RPW + r;
#pragma unroll
            for (int c = 0; c < CK; ++c) pa_out[i * DK + lane + 32 * c] = A[r][c];
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) pb_out[i * DV + lane + 32 * c] = B[r][c];
        }
    }
}

// The chain over a sequence's chunks, column slice by column slice (X <- Phi X + Psi acts on
// each column of X alone): CTA (nh, slice) carries columns [32 slice, 32 slice + 32) of X.
// kFwd: the states at the chunk starts (X = S, Phi/Psi holding the chunk's forward map A/B,
// first chunk first, each start stored in the checkpoints); otherwise the state's gradient
// at the chunk ends (X = dS, last chunk first, each end stored) and finally dS0.
// Warp w owns rows [RPW w, RPW (w + 1)), lane l column 32 slice + l.  Dynamic shared memory:
// the slice of X [DK][32] and the chunk's Phi [DK][DK], fetched by the whole CTA into
// registers one chunk ahead (coalesced float4s) and stored to shared memory per chunk.
constexpr int kChainCols = 32;

template <int DK, int DV, bool kFwd>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_chain_kernel(const BwdParams p) {
    constexpr int RPW = DK / kBwdWarps;
    constexpr int NS = DV / kChainCols;
    extern __shared__ __align__(16) float chain_smem[];
    float* xs = chain_smem;                  // [DK][32]
    float* phs = chain_smem + DK * kChainCols;  // [DK][DK]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int blk = blockIdx.x; blk < p.N * p.H * NS; blk += gridDim.x) {
        const int nh = blk / NS, col = (blk % NS) * kChainCols + lane;
        const int h = nh % p.H, n = nh / p.H;
        const float* init = kFwd ? p.S0 : p.dS_out;
        float X[RPW];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
            X[r] = init ? init[((size_t)nh * DK + warp * RPW + r) * DV + col] : 0.f;
        const int32_t g0 = p.chunk_off[n], g1 = p.chunk_off[n + 1];
        // the next chunk's Phi (this thread's float4s of it) and Psi column, fetched one chunk
        // ahead so that the loads overlap the product
        constexpr int kPf = DK * DK / 4 / kBwdThreads;
        float4 pf[kPf];
        float psv[RPW];
        auto fetch = [&](int32_t step) {
            const int32_t g = kFwd ? g0 + step : g1 - 1 - step;
            const size_t it = (size_t)g * p.H + h;
            const float4* ph4 = reinterpret_cast<const float4*>(p.phi + it * DK * DK);
#pragma unroll
            for (int x = 0; x < kPf; ++x) pf[x] = __ldg(ph4 + tid + x * kBwdThreads);
#pragma unroll
            for (int r = 0; r < RPW; ++r) psv[r] = p.psi[it * DK * DV + (warp * RPW + r) * DV + col];
        };
        if (g1 > g0) fetch(0);
        for (int32_t step = 0; step < g1 - g0; ++step) {
            const int32_t g = kFwd ? g0 + step : g1 - 1 - step;
            const size_t it = (size_t)g * p.H + h;
            float* de = (kFwd ? p.ckpt : p.dsend) + it * DK * DV;
#pragma unroll
            for (int x = 0; x < kPf; ++x) reinterpret_cast<float4*>(phs)[tid + x * kBwdThreads] = pf[x];
            float acc[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const int i = warp * RPW + r;
                de[i * DV + col] = X[r];
                xs[i * kChainCols + lane] = X[r];
                acc[r] = psv[r];
            }
            if (step + 1 < g1 - g0) fetch(step + 1);
            __syncthreads();
            // X <- Phi X + Psi, four Phi columns per shared-memory load
            for (int l = 0; l < DK; l += 4) {
                const float x0 = xs[(l + 0) * kChainCols + lane];
                const float x1 = xs[(l + 1) * kChainCols + lane];
                const float x2 = xs[(l + 2) * kChainCols + lane];
                const float x3 = xs[(l + 3) * kChainCols + lane];
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    const float4 f = *reinterpret_cast<const float4*>(phs + (warp * RPW + r) * DK + l);
                    acc[r] = fmaf(f.x, x0, acc[r]);
                    acc[r] = fmaf(f.y, x1, acc[r]);
                    acc[r] = fmaf(f.z, x2, acc[r]);
                    acc[r] = fmaf(f.w, x3, acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < RPW; ++r) X[r] = acc[r];
            __syncthreads();  // xs and phs are rewritten for the next chunk
        }
        if (!kFwd && p.dS0) {
#pragma unroll
            for (int r = 0; r < RPW; ++r)
                p.dS0[((size_t)nh * DK + warp * RPW + r) * DV + col] = X[r];
        }
    }
}

// Per (chunk, head): the reverse rules token by token from the chunk's dS, with the state
// before each token recomputed from the chunk's checkpoint by sub-blocks of kSB tokens: one
// forward pass keeps the state at every sub-block start (and the states of the last
// sub-block); each earlier sub-block is re-run from its start just before it is reversed.
// Per-CTA scratch: kNB sub-block starts and kSB token states, thread-private float4s laid out
// [slot][float4][thread] so that every store and load is coalesced; the kSB states that are
// written and read back within a sub-block stay in L2.  Two barriers per forward token and
// three per reverse token.
constexpr int kSB = 8;
constexpr int kNB = kBwdC / kSB;

template <typename IO, int DK, int DV>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_item_kernel(const BwdParams p) {
    using L = BwdLayout<DK, DV>;
    constexpr int NE = L::RPW * L::CPL;  // state elements per thread
    constexpr int NV4 = NE / 4;
    static_assert(NE % 4 == 0, "state elements per thread");
    extern __shared__ __align__(16) float stage_smem[];
    const Stage<DK, DV> st = stage_carve<DK, DV>(stage_smem, true, true, true, true);
    __shared__ float part[kBwdWarps][DV];
    __shared__ float part2[kBwdWarps][DV];
    __shared__ float w_s[DV], u_s[DV], du_s[DV];
    __shared__ float rowv[3][DK];  // dq, dk, dalpha
    __shared__ float red[kBwdWarps];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float4* bnd = reinterpret_cast<float4*>(p.snap) +
                  (size_t)blockIdx.x * (kNB + kSB) * NV4 * kBwdThreads + tid;
    float4* snp = bnd + (size_t)kNB * NV4 * kBwdThreads;
    auto put = [&](float4* base, int slot, const float (&X)[L::RPW][L::CPL]) {
#pragma unroll
        for (int x = 0; x < NV4; ++x) {
            const int e = 4 * x;
            base[((size_t)slot * NV4 + x) * kBwdThreads] =
                make_float4(X[e / L::CPL][e % L::CPL], X[(e + 1) / L::CPL][(e + 1) % L::CPL],
                            X[(e + 2) / L::CPL][(e + 2) % L::CPL],
                            X[(e + 3) / L::CPL][(e + 3) % L::CPL]);
        }
    };
    auto get = [&](const float4* base, int slot, float (&X)[L::RPW][L::CPL]) {
#pragma unroll
        for (int x = 0; x < NV4; ++x) {
            const float4 f = base[((size_t)slot * NV4 + x) * kBwdThreads];
            const int e = 4 * x;
            X[e / L::CPL][e % L::CPL] = f.x;
            X[(e + 1) / L::CPL][(e + 1) % L::CPL] = f.y;
            X[(e + 2) / L::CPL][(e + 2) % L::CPL] = f.z;
            X[(e + 3) / L::CPL][(e + 3) % L::CPL] = f.w;
        }
    };
    const int64_t items = (int64_t)p.chunk_off[p.N] * p.H;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        int h, rows;
        int64_t t0;
        item_of(p, it, h, t0, rows);
        const float scale = expf(p.A_log[h]);
        __syncthreads();  // the previous item's staged inputs and sums are consumed
        stage_chunk<IO, DK, DV>(st, p, t0, rows, h, scale);
        float dA_acc = 0.f;
        float dS[L::RPW][L::CPL];  // the state's gradient at the chunk end
        float S[L::RPW][L::CPL];   // the state at the chunk start
        const float* de = p.dsend + (size_t)it * DK * DV;
        const float* src = p.ckpt + (size_t)it * DK * DV;
#pragma unroll
        for (int r = 0; r < L::RPW; ++r)
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) {
                const int o = (warp * L::RPW + r) * DV + lane + 32 * c;
                dS[r][c] = de[o];
                S[r][c] = src[o];
            }
        __syncthreads();
        // one forward token on S (S <- Diag(alpha) S + k u^T, u = beta (v - S'^T k))
        auto fwd_step = [&](int tt) {
            float kr[L::RPW], ar[L::RPW];
            load_rows<L::RPW>(st.k + tt * DK, warp, kr);
            load_rows<L::RPW>(st.a + tt * DK, warp, ar);
            float pc[L::CPL];
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) pc[c] = 0.f;
#pragma unroll
            for (int r = 0; r < L::RPW; ++r) {
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) {
                    S[r][c] *= ar[r];
                    pc[c] = fmaf(S[r][c], kr[r], pc[c]);
                }
            }
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) part[warp][lane + 32 * c] = pc[c];
            __syncthreads();
            if (tid < DV) {
                float s = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kBwdWarps; ++w2) s += part[w2][tid];
                u_s[tid] = st.beta[tt] * (st.v[tt * DV + tid] - s);
            }
            __syncthreads();
            float uc[L::CPL];
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) uc[c] = u_s[lane + 32 * c];
#pragma unroll
            for (int r = 0; r < L::RPW; ++r)
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) S[r][c] = fmaf(kr[r], uc[c], S[r][c]);
        };
        // ---- first forward pass: the sub-block starts, and the last sub-block's states
        const int nb = (rows + kSB - 1) / kSB;
        for (int tt = 0; tt < rows; ++tt) {
            if (tt % kSB == 0 && tt / kSB < nb - 1) put(bnd, tt / kSB, S);
            if (tt >= (nb - 1) * kSB) put(snp, tt % kSB, S);
            if (tt + 1 == rows) break;  // the last token's state is not needed
            fwd_step(tt);
        }
        // ---- back through the chunk's tokens, sub-block by sub-block from the last
        float P[L::RPW][L::CPL];  // S_{t-1}, this thread's part
        for (int b = nb - 1; b >= 0; --b) {
            const int lo = b * kSB, hi = min(lo + kSB, rows);
            if (b < nb - 1) {  // re-run the sub-block from its start, keeping its states
                get(bnd, b, S);
                for (int tt = lo; tt < hi; ++tt) {
                    put(snp, tt - lo, S);
                    if (tt + 1 == hi) break;
                    fwd_step(tt);
                }
            }
            get(snp, hi - 1 - lo, P);
            for (int tt = hi - 1; tt >= lo; --tt) {
                const int64_t t = t0 + tt;
                const float* kt = st.k + tt * DK;
                const float* qt = st.q + tt * DK;
                const float* at = st.a + tt * DK;
                const float bt = st.beta[tt];
                // B1: dS += q do^T; column sums of S' k = P (alpha k) (for w) and of dS k (for du)
                float doj[L::CPL];
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) doj[c] = st.dout[tt * DV + lane + 32 * c];
                float pw[L::CPL], pdu[L::CPL];
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) pw[c] = pdu[c] = 0.f;
                {
                    float kr[L::RPW], qr[L::RPW], ar[L::RPW];
                    load_rows<L::RPW>(kt, warp, kr);
                    load_rows<L::RPW>(qt, warp, qr);
                    load_rows<L::RPW>(at, warp, ar);
#pragma unroll
                    for (int r = 0; r < L::RPW; ++r) {
                        const float ak = ar[r] * kr[r];
#pragma unroll
                        for (int c = 0; c < L::CPL; ++c) {
                            dS[r][c] = fmaf(qr[r], doj[c], dS[r][c]);
                            pw[c] = fmaf(P[r][c], ak, pw[c]);
                            pdu[c] = fmaf(dS[r][c], kr[r], pdu[c]);
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) {
                    part[warp][lane + 32 * c] = pw[c];
                    part2[warp][lane + 32 * c] = pdu[c];
                }
                __syncthreads();
                // B2: w, u per column (first warps), du and dv per column (middle warps)
                if (tid < DV) {
                    float s = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < kBwdWarps; ++w2) s += part[w2][tid];
                    const float wj = st.v[tt * DV + tid] - s;
                    w_s[tid] = wj;
                    u_s[tid] = bt * wj;
                } else if (tid >= 256 && tid < 256 + DV) {
                    const int j = tid - 256;
                    float d = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < kBwdWarps; ++w2) d += part2[w2][j];
                    du_s[j] = d;
                    const size_t vo = ((size_t)t * p.H + h) * DV + j;
                    static_cast<IO*>(p.dv)[vo] = from_f32<IO>(bt * d);
                }
                __syncthreads();
                // B3: per element.  With S' = Diag(alpha) P and S_t = S' + k u^T the row sums are
                //   dq_i     = alpha_i sum_j P_ij do_j + k_i (u . do)
                //   dk_i     = sum_j dS_ij u_j - alpha_i sum_j P_ij beta du_j
                //   dalpha_i = sum_j (dS_ij - k_i beta du_j) P_ij
                // the per-row factors are applied to each lane's partial before the lanes are summed.
                float uj[L::CPL], bduj[L::CPL];
                float ud = 0.f;
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) {
                    uj[c] = u_s[lane + 32 * c];
                    bduj[c] = bt * du_s[lane + 32 * c];
                    ud = fmaf(uj[c], doj[c], ud);
                }
                float vals[32];  // [quantity][row]: 3 x RPW used, the rest zero
#pragma unroll
                for (int x = 0; x < 32; ++x) vals[x] = 0.f;
                float kr[L::RPW], ar[L::RPW];
                load_rows<L::RPW>(kt, warp, kr);
                load_rows<L::RPW>(at, warp, ar);
#pragma unroll
                for (int r = 0; r < L::RPW; ++r) {
                    const float a = ar[r], kk = kr[r];
                    float s1 = 0.f, s2 = 0.f, s3 = 0.f, s4 = 0.f;
#pragma unroll
                    for (int c = 0; c < L::CPL; ++c) {
                        s1 = fmaf(P[r][c], doj[c], s1);
                        s2 = fmaf(dS[r][c], uj[c], s2);
                        s3 = fmaf(P[r][c], bduj[c], s3);
                        const float dsp = fmaf(-kk, bduj[c], dS[r][c]);
                        s4 = fmaf(dsp, P[r][c], s4);
                        dS[r][c] = a * dsp;
                    }
                    vals[r] = a * s1;
                    vals[8 + r] = fmaf(-a, s3, s2);
                    vals[16 + r] = s4;
                }
                if (tt > lo) get(snp, tt - 1 - lo, P);  // P is dead from here on: fetch the next one
                // sum over the 32 lanes, halving the values each step: lane l ends with value l
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) {
                    const bool up = (lane & m) != 0;
#pragma unroll
                    for (int x = 0; x < m; ++x) {
                        const float send = up ? vals[x] : vals[x + m];
                        const float keep = up ? vals[x + m] : vals[x];
                        vals[x] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ud += __shfl_xor_sync(0xffffffffu, ud, off);
                {
                    const int qn = lane >> 3, r = lane & 7;
                    if (qn < 3 && r < L::RPW) {
                        const int i = warp * L::RPW + r;
                        rowv[qn][i] = qn == 0 ? fmaf(kt[i], ud, vals[0]) : vals[0];
                    }
                }
                if (warp == kBwdWarps - 1) {  // dbeta = du . w
                    float wdu = 0.f;
#pragma unroll
                    for (int c = 0; c < L::CPL; ++c) wdu = fmaf(du_s[lane + 32 * c], w_s[lane + 32 * c], wdu);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) wdu += __shfl_xor_sync(0xffffffffu, wdu, off);
                    if (lane == 0) static_cast<IO*>(p.dbeta)[(size_t)t * p.H + h] = from_f32<IO>(wdu);
                }
                __syncthreads();
                // B4: per key channel: dq, dk, dz and the dA_log partial
                if (tid < DK) {
                    const size_t ko = ((size_t)t * p.H + h) * DK + tid;
                    const float x = st.x[tt * DK + tid];
                    const float s = 1.0f / (1.0f + expf(-x));
                    const float dx = rowv[2][tid] * at[tid] * p.g_min * s * (1.0f - s);
                    static_cast<IO*>(p.dq)[ko] = from_f32<IO>(rowv[0][tid]);
                    static_cast<IO*>(p.dk)[ko] = from_f32<IO>(rowv[1][tid]);
                    static_cast<IO*>(p.dz)[ko] = from_f32<IO>(dx * scale);
                    dA_acc = fmaf(dx, x, dA_acc);
                }
            }
        }
        // this (chunk, head)'s dA_log partial
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dA_acc += __shfl_xor_sync(0xffffffffu, dA_acc, off);
        __syncthreads();
        if (lane == 0) red[warp] = dA_acc;
        __syncthreads();
        if (tid == 0) {
            float s2 = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < DK / 32; ++w2) s2 += red[w2];
            p.dA_item[it] = s2;
        }
    }
}

__global__ void bwd_dA_kernel(const float* __restrict__ part, const int32_t* __restrict__ chunk_off,
                              int N, int H, float* __restrict__ dA_log) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H) return;
    const int32_t nc = chunk_off[N];
    float s = 0.f;
    for (int32_t g = 0; g < nc; ++g) s += part[(size_t)g * H + h];
    dA_log[h] = s;
}

template <typename IO, int DK, int DV>
cudaError_t launch_t(const BwdParams& p, int grid_nh, int grid_items, cudaStream_t stream) {
    constexpr int chain_smem = (DK * kChainCols + DK * DK) * 4;
    cudaError_t e = cudaFuncSetAttribute(bwd_chain_kernel<DK, DV, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, chain_smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_chain_kernel<DK, DV, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, chain_smem);
    constexpr int smem_fwdtrans = stage_floats<DK, DV>(false, false, true, false) * 4;
    constexpr int smem_phi = stage_floats<DK, DV>(true, false, false, true) * 4;
    constexpr int smem_item = stage_floats<DK, DV>(true, true, true, true) * 4;
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_fwdtrans_kernel<IO, DK, DV>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem_fwdtrans);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_phi_kernel<IO, DK, DV>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem_phi);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_item_kernel<IO, DK, DV>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem_item);
    if (e != cudaSuccess) return e;
    {
        ProfScope prof("bwd_fwdtrans_kernel", stream);
        bwd_fwdtrans_kernel<IO, DK, DV><<<grid_items, kBwdThreads, smem_fwdtrans, stream>>>(p);
    }
    {
        ProfScope prof("bwd_fchain_kernel", stream);
        bwd_chain_kernel<DK, DV, true><<<grid_nh, kBwdThreads, chain_smem, stream>>>(p);
    }
    {
        ProfScope prof("bwd_phi_kernel", stream);
        bwd_phi_kernel<IO, DK, DV><<<grid_items, kBwdThreads, smem_phi, stream>>>(p);
    }
    {
        ProfScope prof("bwd_chain_kernel", stream);
        bwd_chain_kernel<DK, DV, false><<<grid_nh, kBwdThreads, chain_smem, stream>>>(p);
    }
    {
        ProfScope prof("bwd_item_kernel", stream);
        bwd_item_kernel<IO, DK, DV><<<grid_items, kBwdThreads, smem_item, stream>>>(p);
    }
    return cudaGetLastError();
}

// A second stream (and its fork and join events) per device, created on first use.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    cudaError_t ok = cudaErrorNotReady;
    std::mutex mu;
};
SideStream& side_stream() {
    static std::mutex mu;
    static std::map<int, SideStream*> streams;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    SideStream*& ss = streams[dev];
    if (!ss) {
        ss = new SideStream;
        ss->ok = cudaStreamCreateWithFlags(&ss->s, cudaStreamNonBlocking);
        if (ss->ok == cudaSuccess) ss->ok = cudaEventCreateWithFlags(&ss->fork, cudaEventDisableTiming);
        if (ss->ok == cudaSuccess) ss->ok = cudaEventCreateWithFlags(&ss->join, cudaEventDisableTiming);
    }
    return *ss;
}

int sm_count() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

}  // namespace

// Workspace, for at most C = T/64 + N chunks.  fp32 problems: chunk offsets [N + 1] and table
// [C]; the state at each chunk start, Psi and the state's gradient at each chunk end
// [C][H][dk][dv] fp32; Phi [C][H][dk][dk] fp32; kNB + kSB = 16 states of scratch per CTA of
// the per-chunk kernel; [C][H] dA_log partials.  bf16 problems: the chunk offsets and table,
// the dA_log partials, the workspace of the tensor-core forward (plan and chunk packages),
// then the image and mid blocks of the tensor-core per-chunk kernels, [C][H] each
// (bwd_tc_layout.cuh).  The public size is the larger of the two.
struct BwdLayoutWs {
    size_t off, tab, ckpt, phi, psi, dsend, snap, dA, fwd, bimg, mid, total;
};

BwdLayoutWs bwd_ws_layout(int64_t T_total, int N, int H, int dk, int dv, int grid_items,
                          bool bf16) {
    auto al = [](size_t x) { return (x + 1023) & ~size_t(1023); };
    const size_t C = (size_t)(T_total / kBwdC + N);
    BwdLayoutWs w{};
    size_t o = 0;
    w.off = o;   o += al((size_t)(N + 1) * 4);
    w.tab = o;   o += al(C * 16);
    w.dA = o;    o += al(C * H * 4);
    if (bf16) {
        w.fwd = o;   o += al(fwd_tc_workspace_size(T_total, N, H));
        w.bimg = o;  o += al(C * H * (size_t)bwdtc::kBiBytes);
        w.mid = o;   o += al(C * H * (size_t)bwdtc::kMdBytes);
    } else {
        w.ckpt = o;  o += al(C * H * dk * dv * 4);
        w.phi = o;   o += al(C * H * dk * dk * 4);
        w.psi = o;   o += al(C * H * dk * dv * 4);
        w.dsend = o; o += al(C * H * dk * dv * 4);
        w.snap = o;  o += al((size_t)grid_items * (kNB + kSB) * dk * dv * 4);
    }
    w.total = o;
    return w;
}

int bwd_grid_items(int64_t T_total, int N, int H) {
    const int64_t items = (T_total / kBwdC + N) * (int64_t)H;
    const int64_t cap = (int64_t)sm_count() * 2;
    return (int)(items < cap ? (items > 0 ? items : 1) : cap);
}

size_t bwd_workspace_size_public(int64_t T_total, int N, int H, int dk, int dv) {
    const int gi = bwd_grid_items(T_total, N, H);
    const size_t a = bwd_ws_layout(T_total, N, H, dk, dv, gi, false).total;
    const size_t b = bwd_ws_layout(T_total, N, H, dk, dv, gi, true).total;
    return a > b ? a : b;
}

cudaError_t launch_bwd(const BwdArgs& a) {
    if ((int64_t)a.N * a.H == 0) return cudaSuccess;
    const int grid_items = bwd_grid_items(a.T_total, a.N, a.H);
    const int64_t nh = (int64_t)a.N * a.H * (a.dv / kChainCols);  // chain CTAs: column slices
    const int cap_nh = sm_count() * 2;
    const int grid_nh = (int)(nh < cap_nh ? nh : cap_nh);
    const BwdLayoutWs w = bwd_ws_layout(a.T_total, a.N, a.H, a.dk, a.dv, grid_items, a.io_bf16 != 0);
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    BwdParams p{};
    p.q = a.q; p.k = a.k; p.v = a.v; p.beta = a.beta; p.z = a.z; p.dout = a.dout;
    p.A_log = a.A_log; p.g_min = a.g_min; p.S0 = a.S0; p.dS_out = a.dS_out; p.cu = a.cu_seqlens;
    p.N = a.N; p.H = a.H; p.T_total = a.T_total;
    p.dq = a.dq; p.dk = a.dk_; p.dv = a.dv_; p.dbeta = a.dbeta; p.dz = a.dz; p.dS0 = a.dS0;
    p.chunk_off = reinterpret_cast<int32_t*>(ws + w.off);
    p.chunk_tab = reinterpret_cast<int4*>(ws + w.tab);
    p.ckpt = reinterpret_cast<float*>(ws + w.ckpt);
    p.phi = reinterpret_cast<float*>(ws + w.phi);
    p.psi = reinterpret_cast<float*>(ws + w.psi);
    p.dsend = reinterpret_cast<float*>(ws + w.dsend);
    p.snap = reinterpret_cast<float*>(ws + w.snap);
    p.dA_item = reinterpret_cast<float*>(ws + w.dA);
    p.err = a.dev_err;
    {
        ProfScope prof("bwd_plan_kernel", a.stream);
        bwd_plan_kernel<<<1, 1024, 0, a.stream>>>(a.cu_seqlens, a.N, a.T_total, p.chunk_off,
                                                  p.chunk_tab, a.dev_err);
    }
    cudaError_t e;
    if (a.io_bf16) {
        // bf16: the tensor-core forward in its two-launch form (its packages stay in the
        // workspace; its intra stage writes N and its chain S_0 and Vt into the image
        // blocks), the gradient chain (dS_C, dVt and dS0), then the per-chunk kernels
        FwdArgs f{};
        f.q = a.q; f.k = a.k; f.v = a.v; f.beta = a.beta; f.z = a.z;
        f.A_log = a.A_log; f.g_min = a.g_min; f.S0 = a.S0; f.S_out = nullptr;
        f.cu_seqlens = a.cu_seqlens; f.N = a.N; f.T_total = a.T_total; f.H = a.H;
        f.dk = a.dk; f.dv = a.dv; f.io_bf16 = 1; f.gate_kind = 0; f.o = nullptr;
        f.workspace = ws + w.fwd;
        f.ws_bytes = fwd_tc_workspace_size(a.T_total, a.N, a.H);
        f.dev_err = a.dev_err;
        f.stream = a.stream;
        f.bimg = ws + w.bimg;
        // The gradient chain needs the packages and dout but nothing of the forward's chain,
        // so it runs on a second stream next to it (each holds one CTA per chain; together
        // 2 C of the SMs), forked once the intra stage is enqueued and joined before the
        // per-chunk kernels.  The enqueue is serialised, so concurrent calls do not mix up
        // the fork and join events.
        SideStream& ss = side_stream();
        std::lock_guard<std::mutex> lock(ss.mu);
        e = ss.ok;
        if (e == cudaSuccess) {
            f.after_intra = ss.fork;
            e = launch_fwd_tc(f);
        }
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ss.s, ss.fork, 0);
        if (e == cudaSuccess) e = launch_bwd_chain_tc(a, ws + w.fwd, ws + w.bimg, ss.s);
        if (e == cudaSuccess) e = cudaEventRecord(ss.join, ss.s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(a.stream, ss.join, 0);
        if (e == cudaSuccess)
            e = launch_bwd_items_tc(a, ws + w.fwd, ws + w.bimg, ws + w.mid, p.dA_item, a.stream);
    } else {
        if (a.dk == 128 && a.dv == 128) e = launch_t<float, 128, 128>(p, grid_nh, grid_items, a.stream);
        else if (a.dk == 128 && a.dv == 64) e = launch_t<float, 128, 64>(p, grid_nh, grid_items, a.stream);
        else if (a.dk == 64 && a.dv == 128) e = launch_t<float, 64, 128>(p, grid_nh, grid_items, a.stream);
        else e = launch_t<float, 64, 64>(p, grid_nh, grid_items, a.stream);
    }
    if (e != cudaSuccess) return e;
    ProfScope prof("bwd_dA_kernel", a.stream);
    bwd_dA_kernel<<<(a.H + 127) / 128, 128, 0, a.stream>>>(p.dA_item, p.chunk_off, a.N, a.H,
                                                           a.dA_log);
    return cudaGetLastError();
}

}  // namespace kda
