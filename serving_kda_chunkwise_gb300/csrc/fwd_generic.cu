// fwd_generic.cu -- chunked KDA forward on CUDA cores, fp32 arithmetic throughout.
//
// This is the path for fp32 I/O (where bf16 tensor-core operands would miss a 1e-4
// relative tolerance) and for the (dk, dv) shapes the tensor-core path does not take.
// It follows "Kimi k3 技术报告详解（1）", section "Chunkwise parallel form", chunk by
// chunk (C = 64 rows; the last chunk of a sequence may be short and is zero-padded
// with g = 0, beta = 0, k = q = v = 0, which leaves the state untouched):
//   G[r]   = sum_{s<=r} g_s              (log of gamma^{1->r}, per key channel)
//   L[r,i] = beta_r sum_c k_rc k_ic e^{G_rc - G_ic}        i <  r
//   A[r,i] =        sum_c q_rc k_ic e^{G_rc - G_ic}        i <= r  (inclusive Tril)
//   [W | U] = (I + L)^{-1} Diag(beta) [Gamma*K | V]        (forward substitution)
//   Vt = U - W S
//   O  = (Gamma*Q) S + A Vt
//   S <- Diag(gamma^C) S + (K * gamma^C / Gamma)^T Vt
// Every decay factor is formed as e^{(difference of log-decays)} with a non-positive
// exponent, so nothing can overflow for any g_min -- nor for the unbounded gate the bound
// replaces, g = -e^{A_h} Softplus(z), which this kernel also takes (gate_kind = 1): it is the
// explicit per-pair path that such a gate needs.
//
// Parallelism: one CTA per (sequence, head, 32-column slice of d_v).  The columns of S
// evolve independently (each column obeys the recurrence with its own v_j), so the
// slices need no communication; each recomputes the state-independent part.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kC = 64;      // chunk length
constexpr int kThreads = 512;
constexpr int kDvs = 32;    // d_v columns per CTA

template <int DK>
struct GenericSmem {
    static constexpr int PK = DK + 1;              // padded row stride of [C][DK] tiles
    static constexpr int PX = DK + kDvs + 1;       // padded row stride of [W | U]
    static constexpr int PA = kC + 1;              // padded row stride of [C][C]
    static constexpr size_t floats = 3 * kC * PK + kC * PX + 2 * kC * PA + kC * kDvs +
                                     DK * kDvs + kC + DK;
    static constexpr size_t bytes = floats * sizeof(float);
};

template <int DK, int DV, typename IO>
__global__ void __launch_bounds__(kThreads) fwd_generic_kernel(FwdArgs a) {
    using SM = GenericSmem<DK>;
    constexpr int PK = SM::PK, PX = SM::PX, PA = SM::PA;
    constexpr int kSlices = DV / kDvs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slice = blockIdx.x % kSlices;
    const int nh = blockIdx.x / kSlices;
    const int h = nh % a.H, n = nh / a.H;
    const int H = a.H;
    const int j0 = slice * kDvs;

    extern __shared__ float smem[];
    float* sQ = smem;                 // [C][PK]  q, later Gamma*q
    float* sK = sQ + kC * PK;         // [C][PK]  k, later k*gamma^C/Gamma
    float* sG = sK + kC * PK;         // [C][PK]  g, then cumulative log-decay G
    float* sX = sG + kC * PK;         // [C][PX]  W | U
    float* sL = sX + kC * PX;         // [C][PA]  L (strict lower, beta folded in)
    float* sA = sL + kC * PA;         // [C][PA]  A (inclusive lower)
    float* sV = sA + kC * PA;         // [C][Dvs] v slice, later Vt
    float* sS = sV + kC * kDvs;       // [DK][Dvs] state slice
    float* sB = sS + DK * kDvs;       // [C] beta
    float* sGl = sB + kC;             // [DK] G of the chunk's last row

    const IO* q = static_cast<const IO*>(a.q);
    const IO* k = static_cast<const IO*>(a.k);
    const IO* v = static_cast<const IO*>(a.v);
    const IO* bt = static_cast<const IO*>(a.beta);
    const IO* z = static_cast<const IO*>(a.z);
    IO* o = static_cast<IO*>(a.o);

    int64_t t_begin, t_end;
    seq_range(a.cu_seqlens, n, a.N, a.T_total, a.dev_err, t_begin, t_end);
    const float scale = expf(a.A_log[h]);
    const size_t state_base = (size_t)nh * DK * DV;

    for (int idx = tid; idx < DK * kDvs; idx += kThreads) {
        const int c = idx / kDvs, j = idx % kDvs;
        sS[idx] = a.S0 ? a.S0[state_base + (size_t)c * DV + j0 + j] : 0.f;
    }

    const int j = tid % kDvs;     // column owned in the state phases
    const int rg = tid / kDvs;    // row group (0 .. kThreads / 32 - 1)

    for (int64_t t0 = t_begin; t0 < t_end; t0 += kC) {
        const int L = (int)((t_end - t0) < kC ? (t_end - t0) : kC);
        __syncthreads();  // previous chunk finished with every buffer
        for (int idx = tid; idx < kC * DK; idx += kThreads) {
            const int r = idx / DK, c = idx % DK;
            float qq = 0.f, kk = 0.f, gg = 0.f;
            if (r < L) {
                const size_t off = ((size_t)(t0 + r) * H + h) * DK + c;
                qq = to_f32(q[off]);
                kk = to_f32(k[off]);
                gg = a.gate_kind ? gate_softplus(to_f32(z[off]), scale)
                                 : gate_precise(to_f32(z[off]), scale, a.g_min);
            }
            sQ[r * PK + c] = qq;
            sK[r * PK + c] = kk;
            sG[r * PK + c] = gg;
        }
        for (int idx = tid; idx < kC * kDvs; idx += kThreads) {
            const int r = idx / kDvs, jj = idx % kDvs;
            sV[idx] = (r < L) ? to_f32(v[((size_t)(t0 + r) * H + h) * DV + j0 + jj]) : 0.f;
        }
        if (tid < kC) sB[tid] = (tid < L) ? to_f32(bt[(size_t)(t0 + tid) * H + h]) : 0.f;
        __syncthreads();

        // G = cumulative sum of g within the chunk (one channel per thread).
        if (tid < DK) {
            float acc = 0.f;
            for (int r = 0; r < kC; ++r) {
                acc += sG[r * PK + tid];
                sG[r * PK + tid] = acc;
            }
            sGl[tid] = acc;
        }
        __syncthreads();

        // L and A: one warp per (r, i) pair with i <= r, lanes over channels.
        constexpr int kPairs = kC * (kC + 1) / 2;
        for (int p = warp; p < kPairs; p += kThreads / 32) {
            int r = (int)((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
            while ((r + 1) * (r + 2) / 2 <= p) ++r;
            while (r * (r + 1) / 2 > p) --r;
            const int i = p - r * (r + 1) / 2;
            float kk = 0.f, qk = 0.f;
            for (int c = lane; c < DK; c += 32) {
                const float e = expf(sG[r * PK + c] - sG[i * PK + c]);
                const float ki = sK[i * PK + c] * e;
                kk = fmaf(sK[r * PK + c], ki, kk);
                qk = fmaf(sQ[r * PK + c], ki, qk);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                kk += __shfl_xor_sync(0xffffffffu, kk, off);
                qk += __shfl_xor_sync(0xffffffffu, qk, off);
            }
            if (lane == 0) {
                sA[r * PA + i] = qk;
                sL[r * PA + i] = (i < r) ? sB[r] * kk : 0.f;
            }
        }
        __syncthreads();

        // [W | U] = (I + L)^{-1} Diag(beta) [Gamma*K | V]: one column per thread, rows in
        // order; a column only depends on its own earlier rows, so no barrier is needed.
        if (tid < DK + kDvs) {
            const int col = tid;
            for (int r = 0; r < kC; ++r) {
                const float y = (col < DK) ? sK[r * PK + col] * expf(sG[r * PK + col])
                                           : sV[r * kDvs + (col - DK)];
                float x0 = sB[r] * y, x1 = 0.f, x2 = 0.f, x3 = 0.f;
                int i = 0;
                for (; i + 3 < r; i += 4) {
                    x0 = fmaf(-sL[r * PA + i], sX[i * PX + col], x0);
                    x1 = fmaf(-sL[r * PA + i + 1], sX[(i + 1) * PX + col], x1);
                    x2 = fmaf(-sL[r * PA + i + 2], sX[(i + 2) * PX + col], x2);
                    x3 = fmaf(-sL[r * PA + i + 3], sX[(i + 3) * PX + col], x3);
                }
                for (; i < r; ++i) x0 = fmaf(-sL[r * PA + i], sX[i * PX + col], x0);
                sX[r * PX + col] = (x0 + x1) + (x2 + x3);
            }
        }
        __syncthreads();

        // Q <- Gamma*Q, K <- K * gamma^C / Gamma (both factors <= 1).
        for (int idx = tid; idx < kC * DK; idx += kThreads) {
            const int r = idx / DK, c = idx % DK;
            const float G = sG[r * PK + c];
            sQ[r * PK + c] *= expf(G);
            sK[r * PK + c] *= expf(sGl[c] - G);
        }
        // Vt = U - W S  (into sV; V itself is no longer needed)
        for (int r = rg; r < kC; r += kThreads / kDvs) {
            float acc = sX[r * PX + DK + j];
            for (int c = 0; c < DK; ++c) acc = fmaf(-sX[r * PX + c], sS[c * kDvs + j], acc);
            sV[r * kDvs + j] = acc;
        }
        __syncthreads();

        // O = (Gamma*Q) S + A Vt  for the valid rows.
        for (int r = rg; r < L; r += kThreads / kDvs) {
            float inter = 0.f, intra = 0.f;
            for (int c = 0; c < DK; ++c) inter = fmaf(sQ[r * PK + c], sS[c * kDvs + j], inter);
            for (int i = 0; i <= r; ++i) intra = fmaf(sA[r * PA + i], sV[i * kDvs + j], intra);
            o[((size_t)(t0 + r) * H + h) * DV + j0 + j] = from_f32<IO>(inter + intra);
        }
        __syncthreads();

        // S <- Diag(gamma^C) S + (K * gamma^C / Gamma)^T Vt
        for (int c = rg; c < DK; c += kThreads / kDvs) {
            float acc = expf(sGl[c]) * sS[c * kDvs + j];
            for (int r = 0; r < kC; ++r) acc = fmaf(sK[r * PK + c], sV[r * kDvs + j], acc);
            sS[c * kDvs + j] = acc;
        }
    }
    __syncthreads();
    if (a.S_out)
        for (int idx = tid; idx < DK * kDvs; idx += kThreads) {
            const int c = idx / kDvs, jj = idx % kDvs;
            a.S_out[state_base + (size_t)c * DV + j0 + jj] = sS[idx];
        }
}

template <int DK, int DV, typename IO>
cudaError_t launch_t(const FwdArgs& a) {
    constexpr size_t bytes = GenericSmem<DK>::bytes;
    auto kern = fwd_generic_kernel<DK, DV, IO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
    if (e != cudaSuccess) return e;
    const int64_t grid = (int64_t)a.N * a.H * (DV / kDvs);
    ProfScope prof("fwd_generic_kernel", a.stream);
    kern<<<(unsigned)grid, kThreads, bytes, a.stream>>>(a);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t dispatch_dims(const FwdArgs& a) {
    if (a.dk == 128 && a.dv == 128) return launch_t<128, 128, IO>(a);
    if (a.dk == 128 && a.dv == 64) return launch_t<128, 64, IO>(a);
    if (a.dk == 64 && a.dv == 128) return launch_t<64, 128, IO>(a);
    return launch_t<64, 64, IO>(a);
}

}  // namespace

cudaError_t launch_fwd_generic(const FwdArgs& a) {
    if ((int64_t)a.N * a.H == 0) return cudaSuccess;
    return a.io_bf16 ? dispatch_dims<__nv_bfloat16>(a) : dispatch_dims<float>(a);
}

}  // namespace kda
