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
// On CUDA cores in fp32, parallel over chunks.  The gradient of the state is the only serial
// quantity, and over one 64-token chunk it is affine: going back through token t maps
// dS_t to B_t (dS_t + q_t do_t^T) with B_t = Diag(alpha_t) (I - beta_t k_t k_t^T), so
//   dS_(chunk start) = Phi dS_(chunk end) + Psi,  Phi = B_t0 .. B_t1-1,
//   Psi = sum_t B_t0 .. B_t (q_t do_t^T).
// Kernels (512 threads; warp w owns rows [w dk/16, (w+1) dk/16) of a state-shaped matrix and
// lane l its columns l, l + 32, ..; matrices live in registers):
//   bwd_plan_kernel   chunk offsets of every sequence and a table entry per chunk
//   bwd_fwdtrans_kernel  per (chunk, head), all in parallel: the chunk's forward map on the
//                     state, S_end = A S_start + B
//   bwd_chain_kernel<fwd>  per (sequence, head, 32-column slice): S at every chunk start
//                     (S <- A S + B, first chunk first), the checkpoints
//   bwd_phi_kernel    per (chunk, head), all in parallel: Phi and Psi of the chunk
//   bwd_chain_kernel  per (sequence, head, 32-column slice): dS at every chunk end, last
//                     chunk first (dS <- Phi dS + Psi), and dS0
//   bwd_item_kernel   per (chunk, head), all in parallel: the chunk's forward from its
//                     checkpoint (the state before every token kept in per-CTA scratch), then
//                     the reverse rules above token by token from the chunk's dS
//   bwd_dA_kernel     dA_log[h] = the per-(chunk, head) partial sums in chunk order
//                     (deterministic)
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

// the per-token vectors in shared memory
template <int DK, int DV>
struct TokVec {
    float k[DK], q[DK], alpha[DK], x[DK];
    float v[DV], dout[DV], w[DV], u[DV], du[DV];
    float beta;
};

template <typename IO, int DK, int DV>
__device__ __forceinline__ void load_token(TokVec<DK, DV>& tv, const IO* q, const IO* k,
                                           const IO* v, const IO* beta, const IO* z,
                                           const IO* dout, int64_t t, int H, int h, float scale,
                                           float g_min, int tid) {
    const size_t kofs = ((size_t)t * H + h) * DK, vofs = ((size_t)t * H + h) * DV;
    if (tid < DK) {
        tv.k[tid] = to_f32(k[kofs + tid]);
        tv.q[tid] = to_f32(q[kofs + tid]);
        const float x = scale * to_f32(z[kofs + tid]);
        tv.x[tid] = x;
        tv.alpha[tid] = expf(g_min / (1.0f + expf(-x)));
    } else if (tid >= 256 && tid < 256 + DV) {
        const int j = tid - 256;
        tv.v[j] = to_f32(v[vofs + j]);
        if (dout) tv.dout[j] = to_f32(dout[vofs + j]);
    }
    if (tid == 511) tv.beta = to_f32(beta[(size_t)t * H + h]);
}

// one forward token on the register-resident state (S <- S' + k u^T); uses tv.w, tv.u and
// `part` ([warps][DV]) as scratch; two barriers
template <int DK, int DV>
__device__ __forceinline__ void fwd_token(float (&S)[BwdLayout<DK, DV>::RPW][BwdLayout<DK, DV>::CPL],
                                          TokVec<DK, DV>& tv, float (*part)[DV], int warp,
                                          int lane, int tid) {
    using L = BwdLayout<DK, DV>;
    float pc[L::CPL];
#pragma unroll
    for (int c = 0; c < L::CPL; ++c) pc[c] = 0.f;
#pragma unroll
    for (int r = 0; r < L::RPW; ++r) {
        const int i = warp * L::RPW + r;
        const float a = tv.alpha[i], kk = tv.k[i];
#pragma unroll
        for (int c = 0; c < L::CPL; ++c) {
            S[r][c] *= a;
            pc[c] = fmaf(S[r][c], kk, pc[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < L::CPL; ++c) part[warp][lane + 32 * c] = pc[c];
    __syncthreads();
    if (tid < DV) {
        float s = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kBwdWarps; ++w2) s += part[w2][tid];
        const float wj = tv.v[tid] - s;
        tv.w[tid] = wj;
        tv.u[tid] = tv.beta * wj;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < L::RPW; ++r) {
        const float kk = tv.k[warp * L::RPW + r];
#pragma unroll
        for (int c = 0; c < L::CPL; ++c) S[r][c] = fmaf(kk, tv.u[lane + 32 * c], S[r][c]);
    }
}

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
    float* snap;         // [grid][64][DK][DV]: per-CTA scratch
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

template <typename IO, int DK, int DV>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_phi_kernel(const BwdParams p) {
    using L = BwdLayout<DK, DV>;
    constexpr int CK = DK / 32;  // Phi columns per lane
    __shared__ TokVec<DK, DV> tv;
    __shared__ float partA[kBwdWarps][DK];
    __shared__ float partB[kBwdWarps][DV];
    __shared__ float duA[DK];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const IO* q = static_cast<const IO*>(p.q);
    const IO* k = static_cast<const IO*>(p.k);
    const IO* v = static_cast<const IO*>(p.v);
    const IO* beta = static_cast<const IO*>(p.beta);
    const IO* z = static_cast<const IO*>(p.z);
    const IO* dout = static_cast<const IO*>(p.dout);
    const int64_t items = (int64_t)p.chunk_off[p.N] * p.H;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int h = (int)(it % p.H);
        const int4 e = p.chunk_tab[it / p.H];
        const int64_t t0 = (static_cast<int64_t>(e.y) << 32) | static_cast<uint32_t>(e.x);
        const int64_t t1 = t0 + e.w;
        const float scale = expf(p.A_log[h]);
        float Phi[L::RPW][CK], Psi[L::RPW][L::CPL];
#pragma unroll
        for (int r = 0; r < L::RPW; ++r) {
#pragma unroll
            for (int c = 0; c < CK; ++c) Phi[r][c] = (warp * L::RPW + r == lane + 32 * c) ? 1.f : 0.f;
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) Psi[r][c] = 0.f;
        }
        for (int64_t t = t1 - 1; t >= t0; --t) {
            __syncthreads();  // the previous token's vectors and sums are consumed
            load_token<IO, DK, DV>(tv, q, k, v, beta, z, dout, t, p.H, h, scale, p.g_min, tid);
            __syncthreads();
            // Psi += q do^T; column sums of Phi^T k and Psi^T k
            float pa[CK], pb[L::CPL];
#pragma unroll
            for (int c = 0; c < CK; ++c) pa[c] = 0.f;
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) pb[c] = 0.f;
#pragma unroll
            for (int r = 0; r < L::RPW; ++r) {
                const int i = warp * L::RPW + r;
                const float kk = tv.k[i], qq = tv.q[i];
#pragma unroll
                for (int c = 0; c < CK; ++c) pa[c] = fmaf(Phi[r][c], kk, pa[c]);
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) {
                    Psi[r][c] = fmaf(qq, tv.dout[lane + 32 * c], Psi[r][c]);
                    pb[c] = fmaf(Psi[r][c], kk, pb[c]);
                }
            }
#pragma unroll
            for (int c = 0; c < CK; ++c) partA[warp][lane + 32 * c] = pa[c];
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) partB[warp][lane + 32 * c] = pb[c];
            __syncthreads();
            if (tid < DK) {
                float sa = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kBwdWarps; ++w2) sa += partA[w2][tid];
                duA[tid] = sa;
            } else if (tid >= 256 && tid < 256 + DV) {
                float sb = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kBwdWarps; ++w2) sb += partB[w2][tid - 256];
                tv.du[tid - 256] = sb;
            }
            __syncthreads();
            // X <- Diag(alpha) (X - beta k du^T) for X = Phi and Psi
#pragma unroll
            for (int r = 0; r < L::RPW; ++r) {
                const int i = warp * L::RPW + r;
                const float a = tv.alpha[i], bk = tv.beta * tv.k[i];
#pragma unroll
                for (int c = 0; c < CK; ++c) Phi[r][c] = a * fmaf(-bk, duA[lane + 32 * c], Phi[r][c]);
#pragma unroll
                for (int c = 0; c < L::CPL; ++c)
                    Psi[r][c] = a * fmaf(-bk, tv.du[lane + 32 * c], Psi[r][c]);
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
    __shared__ TokVec<DK, DV> tv;
    __shared__ float partA[kBwdWarps][DK];
    __shared__ float partB[kBwdWarps][DV];
    __shared__ float wA[DK];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const IO* q = static_cast<const IO*>(p.q);
    const IO* k = static_cast<const IO*>(p.k);
    const IO* v = static_cast<const IO*>(p.v);
    const IO* beta = static_cast<const IO*>(p.beta);
    const IO* z = static_cast<const IO*>(p.z);
    const int64_t items = (int64_t)p.chunk_off[p.N] * p.H;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int h = (int)(it % p.H);
        const int4 e = p.chunk_tab[it / p.H];
        const int64_t t0 = (static_cast<int64_t>(e.y) << 32) | static_cast<uint32_t>(e.x);
        const int64_t t1 = t0 + e.w;
        const float scale = expf(p.A_log[h]);
        float A[L::RPW][CK], B[L::RPW][L::CPL];
#pragma unroll
        for (int r = 0; r < L::RPW; ++r) {
#pragma unroll
            for (int c = 0; c < CK; ++c) A[r][c] = (warp * L::RPW + r == lane + 32 * c) ? 1.f : 0.f;
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) B[r][c] = 0.f;
        }
        for (int64_t t = t0; t < t1; ++t) {
            __syncthreads();
            load_token<IO, DK, DV>(tv, q, k, v, beta, z, nullptr, t, p.H, h, scale, p.g_min, tid);
            __syncthreads();
            float pa[CK], pb[L::CPL];
#pragma unroll
            for (int c = 0; c < CK; ++c) pa[c] = 0.f;
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) pb[c] = 0.f;
#pragma unroll
            for (int r = 0; r < L::RPW; ++r) {
                const int i = warp * L::RPW + r;
                const float a = tv.alpha[i], kk = tv.k[i];
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
            for (int c = 0; c < CK; ++c) partA[warp][lane + 32 * c] = pa[c];
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) partB[warp][lane + 32 * c] = pb[c];
            __syncthreads();
            if (tid < DK) {
                float sa = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kBwdWarps; ++w2) sa += partA[w2][tid];
                wA[tid] = sa;
            } else if (tid >= 256 && tid < 256 + DV) {
                float sb = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kBwdWarps; ++w2) sb += partB[w2][tid - 256];
                tv.w[tid - 256] = sb - tv.v[tid - 256];  // (k^T B') - v
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < L::RPW; ++r) {
                const float bk = tv.beta * tv.k[warp * L::RPW + r];
#pragma unroll
                for (int c = 0; c < CK; ++c) A[r][c] = fmaf(-bk, wA[lane + 32 * c], A[r][c]);
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) B[r][c] = fmaf(-bk, tv.w[lane + 32 * c], B[r][c]);
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
// the slice of X [DK][32] and the chunk's Phi [DK][DK], loaded by the whole CTA in one
// coalesced pass per chunk.
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
        for (int32_t step = 0; step < g1 - g0; ++step) {
            const int32_t g = kFwd ? g0 + step : g1 - 1 - step;
            const size_t it = (size_t)g * p.H + h;
            float* de = (kFwd ? p.ckpt : p.dsend) + it * DK * DV;
            const float4* ph4 = reinterpret_cast<const float4*>(p.phi + it * DK * DK);
            const float* ps = p.psi + it * DK * DV;
            for (int i4 = tid; i4 < DK * DK / 4; i4 += kBwdThreads)
                reinterpret_cast<float4*>(phs)[i4] = __ldg(ph4 + i4);
            float acc[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const int i = warp * RPW + r;
                de[i * DV + col] = X[r];
                xs[i * kChainCols + lane] = X[r];
                acc[r] = ps[i * DV + col];
            }
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

template <typename IO, int DK, int DV>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_item_kernel(const BwdParams p) {
    using L = BwdLayout<DK, DV>;
    __shared__ TokVec<DK, DV> tv;
    __shared__ float part[kBwdWarps][DV];
    __shared__ float part2[kBwdWarps][DV];
    __shared__ float rowv[3][DK];  // dq, dk, dalpha
    __shared__ float red[kBwdWarps];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float* snap = p.snap + (size_t)blockIdx.x * kBwdC * DK * DV;
    const IO* q = static_cast<const IO*>(p.q);
    const IO* k = static_cast<const IO*>(p.k);
    const IO* v = static_cast<const IO*>(p.v);
    const IO* beta = static_cast<const IO*>(p.beta);
    const IO* z = static_cast<const IO*>(p.z);
    const IO* dout = static_cast<const IO*>(p.dout);
    const int64_t items = (int64_t)p.chunk_off[p.N] * p.H;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int h = (int)(it % p.H);
        const int4 e = p.chunk_tab[it / p.H];
        const int64_t t0 = (static_cast<int64_t>(e.y) << 32) | static_cast<uint32_t>(e.x);
        const int64_t t1 = t0 + e.w;
        const float scale = expf(p.A_log[h]);
        float dA_acc = 0.f;
        float dS[L::RPW][L::CPL];  // the state's gradient at the chunk end
        const float* de = p.dsend + (size_t)it * DK * DV;
#pragma unroll
        for (int r = 0; r < L::RPW; ++r)
#pragma unroll
            for (int c = 0; c < L::CPL; ++c)
                dS[r][c] = de[(warp * L::RPW + r) * DV + lane + 32 * c];
        // ---- the chunk's forward from its checkpoint, keeping the state before each token
        float S[L::RPW][L::CPL];
        const float* src = p.ckpt + (size_t)it * DK * DV;
#pragma unroll
        for (int r = 0; r < L::RPW; ++r)
#pragma unroll
            for (int c = 0; c < L::CPL; ++c)
                S[r][c] = src[(warp * L::RPW + r) * DV + lane + 32 * c];
        for (int64_t t = t0; t < t1; ++t) {
            float* dst = snap + (size_t)(t - t0) * DK * DV;
#pragma unroll
            for (int r = 0; r < L::RPW; ++r)
#pragma unroll
                for (int c = 0; c < L::CPL; ++c)
                    dst[(warp * L::RPW + r) * DV + lane + 32 * c] = S[r][c];
            __syncthreads();
            load_token<IO, DK, DV>(tv, q, k, v, beta, z, nullptr, t, p.H, h, scale, p.g_min,
                                   tid);
            __syncthreads();
            if (t + 1 < t1) fwd_token<DK, DV>(S, tv, part, warp, lane, tid);
        }
        // ---- back through the chunk's tokens
        for (int64_t t = t1 - 1; t >= t0; --t) {
            __syncthreads();  // previous token's vectors and partial sums are consumed
            load_token<IO, DK, DV>(tv, q, k, v, beta, z, dout, t, p.H, h, scale, p.g_min,
                                   tid);
            float P[L::RPW][L::CPL];  // S_{t-1}, this thread's part
            const float* ps = snap + (size_t)(t - t0) * DK * DV;
#pragma unroll
            for (int r = 0; r < L::RPW; ++r)
#pragma unroll
                for (int c = 0; c < L::CPL; ++c)
                    P[r][c] = ps[(warp * L::RPW + r) * DV + lane + 32 * c];
            __syncthreads();
            // B1: dS += q do^T; column sums of S' k = P (alpha k) (for w) and of dS k (for du)
            float doj[L::CPL];
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) doj[c] = tv.dout[lane + 32 * c];
            float pw[L::CPL], pdu[L::CPL];
#pragma unroll
            for (int c = 0; c < L::CPL; ++c) pw[c] = pdu[c] = 0.f;
#pragma unroll
            for (int r = 0; r < L::RPW; ++r) {
                const int i = warp * L::RPW + r;
                const float kk = tv.k[i], qq = tv.q[i], ak = tv.alpha[i] * kk;
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) {
                    dS[r][c] = fmaf(qq, doj[c], dS[r][c]);
                    pw[c] = fmaf(P[r][c], ak, pw[c]);
                    pdu[c] = fmaf(dS[r][c], kk, pdu[c]);
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
                const float wj = tv.v[tid] - s;
                tv.w[tid] = wj;
                tv.u[tid] = tv.beta * wj;
            } else if (tid >= 256 && tid < 256 + DV) {
                const int j = tid - 256;
                float d = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kBwdWarps; ++w2) d += part2[w2][j];
                tv.du[j] = d;
                const size_t vo = ((size_t)t * p.H + h) * DV + j;
                static_cast<IO*>(p.dv)[vo] = from_f32<IO>(tv.beta * d);
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
                uj[c] = tv.u[lane + 32 * c];
                bduj[c] = tv.beta * tv.du[lane + 32 * c];
                ud = fmaf(uj[c], doj[c], ud);
            }
            float vals[32];  // [quantity][row]: 3 x RPW used, the rest zero
#pragma unroll
            for (int x = 0; x < 32; ++x) vals[x] = 0.f;
#pragma unroll
            for (int r = 0; r < L::RPW; ++r) {
                const int i = warp * L::RPW + r;
                const float a = tv.alpha[i], kk = tv.k[i];
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
                    rowv[qn][i] = qn == 0 ? fmaf(tv.k[i], ud, vals[0]) : vals[0];
                }
            }
            if (warp == kBwdWarps - 1) {  // dbeta = du . w
                float wdu = 0.f;
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) wdu = fmaf(tv.du[lane + 32 * c], tv.w[lane + 32 * c], wdu);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) wdu += __shfl_xor_sync(0xffffffffu, wdu, off);
                if (lane == 0) static_cast<IO*>(p.dbeta)[(size_t)t * p.H + h] = from_f32<IO>(wdu);
            }
            __syncthreads();
            // B4: per key channel: dq, dk, dz and the dA_log partial
            if (tid < DK) {
                const size_t ko = ((size_t)t * p.H + h) * DK + tid;
                const float x = tv.x[tid];
                const float s = 1.0f / (1.0f + expf(-x));
                const float dx = rowv[2][tid] * tv.alpha[tid] * p.g_min * s * (1.0f - s);
                static_cast<IO*>(p.dq)[ko] = from_f32<IO>(rowv[0][tid]);
                static_cast<IO*>(p.dk)[ko] = from_f32<IO>(rowv[1][tid]);
                static_cast<IO*>(p.dz)[ko] = from_f32<IO>(dx * scale);
                dA_acc = fmaf(dx, x, dA_acc);
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
        __syncthreads();
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
    if (e != cudaSuccess) return e;
    {
        ProfScope prof("bwd_fwdtrans_kernel", stream);
        bwd_fwdtrans_kernel<IO, DK, DV><<<grid_items, kBwdThreads, 0, stream>>>(p);
    }
    {
        ProfScope prof("bwd_fchain_kernel", stream);
        bwd_chain_kernel<DK, DV, true><<<grid_nh, kBwdThreads, chain_smem, stream>>>(p);
    }
    {
        ProfScope prof("bwd_phi_kernel", stream);
        bwd_phi_kernel<IO, DK, DV><<<grid_items, kBwdThreads, 0, stream>>>(p);
    }
    {
        ProfScope prof("bwd_chain_kernel", stream);
        bwd_chain_kernel<DK, DV, false><<<grid_nh, kBwdThreads, chain_smem, stream>>>(p);
    }
    {
        ProfScope prof("bwd_item_kernel", stream);
        bwd_item_kernel<IO, DK, DV><<<grid_items, kBwdThreads, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

int sm_count() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

}  // namespace

// Workspace, for at most C = T/64 + N chunks: chunk offsets [N + 1] and table [C]; the state
// at each chunk start, Psi and the state's gradient at each chunk end [C][H][dk][dv] fp32;
// Phi [C][H][dk][dk] fp32; 64 states of scratch per CTA of the per-chunk kernel; [C][H]
// dA_log partials.
struct BwdLayoutWs {
    size_t off, tab, ckpt, phi, psi, dsend, snap, dA, total;
};

BwdLayoutWs bwd_ws_layout(int64_t T_total, int N, int H, int dk, int dv, int grid_items) {
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t C = (size_t)(T_total / kBwdC + N);
    BwdLayoutWs w{};
    size_t o = 0;
    w.off = o;   o += al((size_t)(N + 1) * 4);
    w.tab = o;   o += al(C * 16);
    w.ckpt = o;  o += al(C * H * dk * dv * 4);
    w.phi = o;   o += al(C * H * dk * dk * 4);
    w.psi = o;   o += al(C * H * dk * dv * 4);
    w.dsend = o; o += al(C * H * dk * dv * 4);
    w.snap = o;  o += al((size_t)grid_items * kBwdC * dk * dv * 4);
    w.dA = o;    o += al(C * H * 4);
    w.total = o;
    return w;
}

int bwd_grid_items(int64_t T_total, int N, int H) {
    const int64_t items = (T_total / kBwdC + N) * (int64_t)H;
    const int64_t cap = (int64_t)sm_count() * 2;
    return (int)(items < cap ? (items > 0 ? items : 1) : cap);
}

size_t bwd_workspace_size_public(int64_t T_total, int N, int H, int dk, int dv) {
    return bwd_ws_layout(T_total, N, H, dk, dv, bwd_grid_items(T_total, N, H)).total;
}

cudaError_t launch_bwd(const BwdArgs& a) {
    if ((int64_t)a.N * a.H == 0) return cudaSuccess;
    const int grid_items = bwd_grid_items(a.T_total, a.N, a.H);
    const int64_t nh = (int64_t)a.N * a.H * (a.dv / kChainCols);  // chain CTAs: column slices
    const int cap_nh = sm_count() * 2;
    const int grid_nh = (int)(nh < cap_nh ? nh : cap_nh);
    const BwdLayoutWs w = bwd_ws_layout(a.T_total, a.N, a.H, a.dk, a.dv, grid_items);
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
        if (a.dk == 128 && a.dv == 128) e = launch_t<__nv_bfloat16, 128, 128>(p, grid_nh, grid_items, a.stream);
        else if (a.dk == 128 && a.dv == 64) e = launch_t<__nv_bfloat16, 128, 64>(p, grid_nh, grid_items, a.stream);
        else if (a.dk == 64 && a.dv == 128) e = launch_t<__nv_bfloat16, 64, 128>(p, grid_nh, grid_items, a.stream);
        else e = launch_t<__nv_bfloat16, 64, 64>(p, grid_nh, grid_items, a.stream);
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
