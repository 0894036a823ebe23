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
// This is the token-level form on CUDA cores in fp32 (a first backward: serial over tokens,
// latency-bound; the chunked tensor-core backward is not built).  One CTA of 512 threads per
// (sequence, head): warp w owns rows [w dk/16, (w+1) dk/16) of the d_k x d_v state and lane
// l owns columns l, l + 32, ..; S and dS live in registers.
//   bwd_ckpt_kernel   the forward, storing S at the start of every 64-token chunk
//   bwd_kernel        per chunk, last to first: re-run the chunk's forward from its checkpoint
//                     storing the state before every token (scratch), then step back through
//                     the tokens with the rules above
//   bwd_dA_kernel     dA_log[h] = the per-(sequence, head) partial sums, added in sequence
//                     order (deterministic)
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kBwdThreads = 512;
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int kBwdC = 64;

// checkpoint slot of the chunk that starts at token t0 of sequence n (injective: see the
// workspace description in bwd_workspace_size)
__device__ __forceinline__ int64_t ckpt_slot(int64_t t0, int n) { return t0 / kBwdC + n; }

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
    float* ckpt;       // [slots][H][DK][DV]
    float* snap;       // [grid][64][DK][DV]
    float* dA_part;    // [N][H]
    unsigned* err;
};

template <typename IO, int DK, int DV>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_ckpt_kernel(const BwdParams p) {
    using L = BwdLayout<DK, DV>;
    __shared__ TokVec<DK, DV> tv;
    __shared__ float part[kBwdWarps][DV];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int nh = blockIdx.x; nh < p.N * p.H; nh += gridDim.x) {
        const int h = nh % p.H, n = nh / p.H;
        int64_t tb, te;
        seq_range(p.cu, n, p.N, p.T_total, p.err, tb, te);
        const float scale = expf(p.A_log[h]);
        float S[L::RPW][L::CPL];
#pragma unroll
        for (int r = 0; r < L::RPW; ++r)
#pragma unroll
            for (int c = 0; c < L::CPL; ++c)
                S[r][c] = p.S0 ? p.S0[((size_t)nh * DK + warp * L::RPW + r) * DV + lane + 32 * c]
                               : 0.f;
        for (int64_t t = tb; t < te; ++t) {
            if ((t - tb) % kBwdC == 0) {  // the state before this chunk
                float* dst = p.ckpt + ((size_t)ckpt_slot(t, n) * p.H + h) * DK * DV;
#pragma unroll
                for (int r = 0; r < L::RPW; ++r)
#pragma unroll
                    for (int c = 0; c < L::CPL; ++c)
                        dst[(warp * L::RPW + r) * DV + lane + 32 * c] = S[r][c];
            }
            __syncthreads();  // the previous token's vectors are no longer read
            load_token<IO, DK, DV>(tv, static_cast<const IO*>(p.q), static_cast<const IO*>(p.k),
                                   static_cast<const IO*>(p.v), static_cast<const IO*>(p.beta),
                                   static_cast<const IO*>(p.z), nullptr, t, p.H, h, scale,
                                   p.g_min, tid);
            __syncthreads();
            fwd_token<DK, DV>(S, tv, part, warp, lane, tid);
        }
        __syncthreads();
    }
}

template <typename IO, int DK, int DV>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_kernel(const BwdParams p) {
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
    for (int nh = blockIdx.x; nh < p.N * p.H; nh += gridDim.x) {
        const int h = nh % p.H, n = nh / p.H;
        int64_t tb, te;
        seq_range(p.cu, n, p.N, p.T_total, p.err, tb, te);
        const float scale = expf(p.A_log[h]);
        float dA_acc = 0.f;
        float dS[L::RPW][L::CPL];
#pragma unroll
        for (int r = 0; r < L::RPW; ++r)
#pragma unroll
            for (int c = 0; c < L::CPL; ++c)
                dS[r][c] = p.dS_out
                               ? p.dS_out[((size_t)nh * DK + warp * L::RPW + r) * DV + lane + 32 * c]
                               : 0.f;
        const int64_t nchunks = (te - tb + kBwdC - 1) / kBwdC;
        for (int64_t ci = nchunks - 1; ci >= 0; --ci) {
            const int64_t t0 = tb + ci * kBwdC;
            const int64_t t1 = (t0 + kBwdC < te) ? t0 + kBwdC : te;
            // ---- the chunk's forward from its checkpoint, keeping the state before each token
            float S[L::RPW][L::CPL];
            const float* src = p.ckpt + ((size_t)ckpt_slot(t0, n) * p.H + h) * DK * DV;
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
                // B1: S' = alpha P; column sums of S' k (for w) and of (dS + q do^T) k (for du)
                float pw[L::CPL], pdu[L::CPL];
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) pw[c] = pdu[c] = 0.f;
#pragma unroll
                for (int r = 0; r < L::RPW; ++r) {
                    const int i = warp * L::RPW + r;
                    const float a = tv.alpha[i], kk = tv.k[i], qq = tv.q[i];
#pragma unroll
                    for (int c = 0; c < L::CPL; ++c) {
                        const int j = lane + 32 * c;
                        dS[r][c] = fmaf(qq, tv.dout[j], dS[r][c]);
                        pw[c] = fmaf(a * P[r][c], kk, pw[c]);
                        pdu[c] = fmaf(dS[r][c], kk, pdu[c]);
                    }
                }
#pragma unroll
                for (int c = 0; c < L::CPL; ++c) {
                    part[warp][lane + 32 * c] = pw[c];
                    part2[warp][lane + 32 * c] = pdu[c];
                }
                __syncthreads();
                // B2: w, u, du per column; dv and the dbeta partial
                float wdu = 0.f;
                if (tid < DV) {
                    float s = 0.f, d = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < kBwdWarps; ++w2) {
                        s += part[w2][tid];
                        d += part2[w2][tid];
                    }
                    const float wj = tv.v[tid] - s;
                    tv.w[tid] = wj;
                    tv.u[tid] = tv.beta * wj;
                    tv.du[tid] = d;
                    wdu = d * wj;
                    const size_t vo = ((size_t)t * p.H + h) * DV + tid;
                    static_cast<IO*>(p.dv)[vo] = from_f32<IO>(tv.beta * d);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) wdu += __shfl_xor_sync(0xffffffffu, wdu, off);
                if (lane == 0) red[warp] = wdu;
                __syncthreads();
                if (tid == 0) {
                    float b = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < DV / 32; ++w2) b += red[w2];
                    static_cast<IO*>(p.dbeta)[(size_t)t * p.H + h] = from_f32<IO>(b);
                }
                // B3: per element; row sums of S_t do (dq), dS u - S' beta du (dk), dS' P (dalpha)
#pragma unroll
                for (int r = 0; r < L::RPW; ++r) {
                    const int i = warp * L::RPW + r;
                    const float a = tv.alpha[i], kk = tv.k[i];
                    float sq = 0.f, sk = 0.f, sa = 0.f;
#pragma unroll
                    for (int c = 0; c < L::CPL; ++c) {
                        const int j = lane + 32 * c;
                        const float sp = a * P[r][c];
                        const float bdu = tv.beta * tv.du[j];
                        sq = fmaf(sp + kk * tv.u[j], tv.dout[j], sq);
                        sk = fmaf(dS[r][c], tv.u[j], sk);
                        sk = fmaf(-sp, bdu, sk);
                        const float dsp = fmaf(-kk, bdu, dS[r][c]);
                        sa = fmaf(dsp, P[r][c], sa);
                        dS[r][c] = a * dsp;
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        sq += __shfl_xor_sync(0xffffffffu, sq, off);
                        sk += __shfl_xor_sync(0xffffffffu, sk, off);
                        sa += __shfl_xor_sync(0xffffffffu, sa, off);
                    }
                    if (lane == 0) {
                        rowv[0][i] = sq;
                        rowv[1][i] = sk;
                        rowv[2][i] = sa;
                    }
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
        }
        // dS0 and this (sequence, head)'s dA_log partial
        if (p.dS0) {
#pragma unroll
            for (int r = 0; r < L::RPW; ++r)
#pragma unroll
                for (int c = 0; c < L::CPL; ++c)
                    p.dS0[((size_t)nh * DK + warp * L::RPW + r) * DV + lane + 32 * c] = dS[r][c];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dA_acc += __shfl_xor_sync(0xffffffffu, dA_acc, off);
        __syncthreads();
        if (lane == 0) red[warp] = dA_acc;
        __syncthreads();
        if (tid == 0) {
            float s = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < DK / 32; ++w2) s += red[w2];
            p.dA_part[nh] = s;
        }
        __syncthreads();
    }
}

__global__ void bwd_dA_kernel(const float* __restrict__ part, int N, int H,
                              float* __restrict__ dA_log) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H) return;
    float s = 0.f;
    for (int n = 0; n < N; ++n) s += part[(size_t)n * H + h];
    dA_log[h] = s;
}

template <typename IO, int DK, int DV>
cudaError_t launch_t(const BwdParams& p, int grid, cudaStream_t stream) {
    {
        ProfScope prof("bwd_ckpt_kernel", stream);
        bwd_ckpt_kernel<IO, DK, DV><<<grid, kBwdThreads, 0, stream>>>(p);
    }
    {
        ProfScope prof("bwd_kernel", stream);
        bwd_kernel<IO, DK, DV><<<grid, kBwdThreads, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

int bwd_grid(int N, int H) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t units = (int64_t)N * H;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 2;
    return (int)(units < cap ? units : cap);
}

}  // namespace

// Workspace: checkpoint slots floor(t0 / 64) + n over every chunk start t0 of sequence n --
// distinct for distinct chunks (a sequence's chunks advance the first term by one each, and
// the next sequence starts at least one slot further on), fewer than T/64 + N + 1 -- each
// d_k x d_v fp32 per head; 64 states of scratch per CTA; N x H dA_log partials.
size_t bwd_workspace_size(int64_t T_total, int N, int H, int dk, int dv, int grid) {
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t slots = (size_t)(T_total / kBwdC + N + 1);
    return al(slots * H * dk * dv * 4) + al((size_t)grid * kBwdC * dk * dv * 4) +
           al((size_t)N * H * 4);
}

size_t bwd_workspace_size_public(int64_t T_total, int N, int H, int dk, int dv) {
    return bwd_workspace_size(T_total, N, H, dk, dv, bwd_grid(N, H));
}

cudaError_t launch_bwd(const BwdArgs& a) {
    if ((int64_t)a.N * a.H == 0) return cudaSuccess;
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    const int grid = bwd_grid(a.N, a.H);
    const size_t slots = (size_t)(a.T_total / kBwdC + a.N + 1);
    uint8_t* w = static_cast<uint8_t*>(a.workspace);
    BwdParams p{};
    p.q = a.q; p.k = a.k; p.v = a.v; p.beta = a.beta; p.z = a.z; p.dout = a.dout;
    p.A_log = a.A_log; p.g_min = a.g_min; p.S0 = a.S0; p.dS_out = a.dS_out; p.cu = a.cu_seqlens;
    p.N = a.N; p.H = a.H; p.T_total = a.T_total;
    p.dq = a.dq; p.dk = a.dk_; p.dv = a.dv_; p.dbeta = a.dbeta; p.dz = a.dz; p.dS0 = a.dS0;
    p.ckpt = reinterpret_cast<float*>(w);
    p.snap = reinterpret_cast<float*>(w + al(slots * a.H * a.dk * a.dv * 4));
    p.dA_part = reinterpret_cast<float*>(w + al(slots * a.H * a.dk * a.dv * 4) +
                                         al((size_t)grid * kBwdC * a.dk * a.dv * 4));
    p.err = a.dev_err;
    cudaError_t e;
    if (a.io_bf16) {
        if (a.dk == 128 && a.dv == 128) e = launch_t<__nv_bfloat16, 128, 128>(p, grid, a.stream);
        else if (a.dk == 128 && a.dv == 64) e = launch_t<__nv_bfloat16, 128, 64>(p, grid, a.stream);
        else if (a.dk == 64 && a.dv == 128) e = launch_t<__nv_bfloat16, 64, 128>(p, grid, a.stream);
        else e = launch_t<__nv_bfloat16, 64, 64>(p, grid, a.stream);
    } else {
        if (a.dk == 128 && a.dv == 128) e = launch_t<float, 128, 128>(p, grid, a.stream);
        else if (a.dk == 128 && a.dv == 64) e = launch_t<float, 128, 64>(p, grid, a.stream);
        else if (a.dk == 64 && a.dv == 128) e = launch_t<float, 64, 128>(p, grid, a.stream);
        else e = launch_t<float, 64, 64>(p, grid, a.stream);
    }
    if (e != cudaSuccess) return e;
    ProfScope prof("bwd_dA_kernel", a.stream);
    bwd_dA_kernel<<<(a.H + 127) / 128, 128, 0, a.stream>>>(p.dA_part, a.N, a.H, a.dA_log);
    return cudaGetLastError();
}

}  // namespace kda
