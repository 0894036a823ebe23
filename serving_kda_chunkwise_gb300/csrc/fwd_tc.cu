// fwd_tc.cu -- chunked KDA forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA),
// bf16 I/O, heads of 64 or 128 channels (a 64 runs zero-padded to 128), chunk C = 64 with
// 16-token sub-tiles, fp32 state.
//
// Method ("Kimi k3 技术报告详解（1）——架构再升华", section "Chunkwise parallel form"):
// per chunk, with G[r] = sum_{s<=r} g_s (per key channel) and gamma = e^G,
//   L = StrictTril(Diag(beta)(Gamma*K)(K/Gamma)^T),  A = Tril((Gamma*Q)(K/Gamma)^T)
//   M = (I + L)^{-1} Diag(beta),  W = M (Gamma*K),  U = M V                      (UT form)
//   Vt = U - W S,  O = (Gamma*Q) S + A Vt,  S <- Diag(gamma^C) S + (K*gamma^C/Gamma)^T Vt
// The last line (chunk-to-chunk update) is the recurrence unrolled over one chunk.
//
// Two stages (fwd_intra.cuh, fwd_chain.cuh) joined by a per-(head, chunk) "package" of
// S-independent operands (fwd_tc_layout.cuh):
//   intra stage   every (chunk, head) in parallel: gate + in-chunk cumsum, both sub-tiled
//                 Gram matrices in one tcgen05 MMA, the UT solve, W and U by tcgen05; writes
//                 the chunk's package, whose bytes are the chain stage's shared-memory tiles.
//   chain stage   per (sequence, head), serial over chunks, the state transposed in TMEM:
//                 [W; Gamma Q] S, K~^T Vt and A Vt on tcgen05, fp32 state in registers.
// Launch forms, on the caller's stream, after plan_kernel (chunk offsets of every sequence,
// a table entry per chunk, the sequences longest first):
//   fwd_fused_kernel  one cooperative launch: CTAs [0, C) run the C chains, the others the
//                     intra stage, the packages handed over through a ring of slots that
//                     stays in L2 (equal-length sequences without cu_seqlens, C <= 64);
//   intra_kernel, then chain_kernel  the packages through the workspace in HBM (otherwise).
// The intra stage also has the mixed-path instantiation for the softplus gate (see
// fwd_intra.cuh).
//
// Sub-tiling ("16-token tiles" of the same section; the bounded gate g > g_min is what
// keeps these factors finite): the Gram entry for rows r >= i needs e^{G_r - G_i} per
// channel.  With rho_s = G at the 8th row of sub-tile s (its middle), every row r of
// sub-tile s uses ONE row factor e^{G_r - rho_s} (|exponent| <= 8|g_min| <= 48) and the
// column operand for that sub-tile is k_i e^{rho_s - G_i}: for i in the same sub-tile the
// exponent is again bounded by 48, for earlier i it is <= 0 (underflow there only drops
// terms below e^{-39}).  So the column operand comes in four versions (sub-tile s uses
// columns i < 16(s+1)); stacking them gives one B operand of 16+32+48+64 = 160 rows, and
// stacking the q-side and (beta-scaled) k-side row operands gives A with M = 128: a single
// M=128, N=160, K=128 MMA yields both Grams for every sub-tile pair.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fwd_chain.cuh"
#include "fwd_intra.cuh"
#include "fwd_tc_layout.cuh"
#include "kda_common.cuh"
#include "kda_internal.h"
#include "tc_util.cuh"

namespace kda {
namespace fwdtc {
namespace {

using namespace tc;

// ================================================================= plan ====

// Sequence n holding global chunk `chunk` (largest n with chunk_off[n] <= chunk).
__device__ __forceinline__ int find_seq(const int32_t* chunk_off, int N, int chunk) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= chunk) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Chunk offsets of every sequence (exclusive scan of ceil(len / 64)), then one table entry
// per global chunk: {t0 low, t0 high, sequence, rows}, so that a consumer decodes a chunk
// with one 16-byte load.
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ cu, int N,
                                                    int64_t T_total, int32_t* chunk_off,
                                                    int4* chunk_tab, int32_t* order,
                                                    uint32_t* flags, int n_flags, unsigned* err) {
    __shared__ int32_t s_warp[32];
    __shared__ int32_t s_carry;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    for (int i = tid; i < n_flags; i += blockDim.x) flags[i] = 0u;  // the fused kernel's ring flags
    if (tid == 0) s_carry = 0;
    __syncthreads();
    for (int base = 0; base < N; base += blockDim.x) {
        const int n = base + tid;
        int32_t cnt = 0;
        if (n < N) {
            int64_t b, e;
            seq_range(cu, n, N, T_total, err, b, e);
            cnt = static_cast<int32_t>((e - b + kC - 1) / kC);
        }
        int32_t x = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_warp[w] = x;
        __syncthreads();
        if (w == 0) {
            int32_t v = (lane < (int)(blockDim.x >> 5)) ? s_warp[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += y;
            }
            s_warp[lane] = v;
        }
        __syncthreads();
        const int32_t incl = x + (w > 0 ? s_warp[w - 1] : 0);
        if (n < N) chunk_off[n] = s_carry + incl - cnt;
        __syncthreads();
        if (tid == (int)blockDim.x - 1) s_carry += incl;
        __syncthreads();
    }
    if (tid == 0) chunk_off[N] = s_carry;
    __syncthreads();
    const int total = s_carry;
    for (int c = tid; c < total; c += blockDim.x) {
        const int n = find_seq(chunk_off, N, c);
        int64_t b, e;
        seq_range(cu, n, N, T_total, nullptr, b, e);
        const int64_t t0 = b + (int64_t)(c - chunk_off[n]) * kC;
        const int64_t rem = e - t0;
        chunk_tab[c] = make_int4(static_cast<int>(t0 & 0xffffffff), static_cast<int>(t0 >> 32), n,
                                 static_cast<int>(rem < kC ? rem : kC));
    }
    // Sequences by decreasing chunk count (ties by index) for the chain stage, whose work
    // per sequence is serial: the longest chains start first.  Beyond kOrderMax sequences
    // the O(N^2) ranking is skipped and the index order kept.
    constexpr int kOrderMax = 4096;
    for (int n = tid; n < N; n += blockDim.x) {
        if (N > kOrderMax) {
            order[n] = n;
            continue;
        }
        const int32_t cn = chunk_off[n + 1] - chunk_off[n];
        int rank = 0;
        for (int m = 0; m < N; ++m) {
            const int32_t cm = chunk_off[m + 1] - chunk_off[m];
            rank += (cm > cn) || (cm == cn && m < n);
        }
        order[rank] = n;
    }
}

// ============================================================== kernels ====

template <int kGate>
__global__ void __launch_bounds__(kIntraThreads, 1) intra_kernel(const __grid_constant__ IntraParams p) {
    extern __shared__ uint8_t smem_raw[];
    intra_body<kGate>(p, smem_raw, blockIdx.x, gridDim.x);
}

template <bool kImg>
__global__ void __launch_bounds__(kChainThreads, 1) chain_kernel(const __grid_constant__ ChainParams p) {
    extern __shared__ uint8_t smem_raw[];
    chain_body<kImg>(p, smem_raw, blockIdx.x, gridDim.x);
}

// The two stages in one cooperative launch: CTAs [0, C) run the chain of (sequence, head)
// c = blockIdx.x, the others run the intra stage over all (chunk, head) items in chunk-major
// order, handing each package to its chain through a ring of slots in global memory (small
// enough to stay in L2), so that packages do not make an HBM round trip and both stages run
// at once.  Every CTA is resident (cooperative launch), and every wait is bounded.
constexpr int kFusedThreads = 384;
constexpr uint32_t kFusedSmem = kIntraSmem > kChainSmem ? kIntraSmem : kChainSmem;
// Ring slots per chain: enough to cover the intra stage's latency from taking a slot to
// publishing it (about two item periods of a CTA, several chunks of a chain), capped so
// that the ring stays well inside L2.
constexpr int kRingSlotsMax = 12, kRingSlotsMin = 8;
constexpr size_t kRingBytesMax = size_t(64) << 20;
constexpr int kFusedMaxChains = 64;

struct FusedParams {
    IntraParams ip;
    ChainParams cp;
    int C;
};

// Registers: the launch gives every thread 168 (384 x 168 = 64,512).  In an intra CTA of the
// bounded gate the third warpgroup has no work: it returns its registers (24 each) and the
// two working warpgroups take 240 each, 2 x 128 x 240 + 128 x 24 = 64,512, the launch's
// total.  (The softplus instantiation measured faster at 168: 4.77 against 5.0 ms at
// T = 65536, H = 32, so it keeps the launch's registers.)
constexpr int kFusedRegs = 168, kIntraRegs = 240, kIdleRegs = 24;
static_assert(kFusedThreads == kIntraThreads + 128, "one idle warpgroup in an intra CTA");
static_assert(kIntraThreads * kIntraRegs + 128 * kIdleRegs <= kFusedThreads * kFusedRegs,
              "the intra CTA's register split exceeds the launch's registers");

template <int kGate>
__global__ void __launch_bounds__(kFusedThreads, 1) fwd_fused_kernel(const __grid_constant__ FusedParams p) {
    extern __shared__ uint8_t smem_raw[];
    if ((int)blockIdx.x < p.C) {
        if (threadIdx.x < kChainThreads) chain_body<false>(p.cp, smem_raw, blockIdx.x, p.C);
    } else if (threadIdx.x >= kIntraThreads) {
        if constexpr (kGate == kGateBounded) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kIdleRegs));
    } else {
        if constexpr (kGate == kGateBounded) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kIntraRegs));
        intra_body<kGate>(p.ip, smem_raw, blockIdx.x - p.C, gridDim.x - p.C);
    }
}

// ================================================================= host ====

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

}  // namespace

#ifdef KDA_PHASE_TIMING
int debug_chain_cycles(unsigned long long* out, int n) {
    if (n > 16) n = 16;
    if (cudaMemcpyFromSymbol(out, g_chain_phase, n * sizeof(unsigned long long)) != cudaSuccess)
        return -1;
    static const unsigned long long zeros[16] = {};
    return cudaMemcpyToSymbol(g_chain_phase, zeros, sizeof zeros) == cudaSuccess ? n : -1;
}
int debug_phase_cycles(unsigned long long* out, int n) {
    if (n > 32) n = 32;
    if (cudaMemcpyFromSymbol(out, g_phase, n * sizeof(unsigned long long)) != cudaSuccess) return -1;
    static const unsigned long long zeros[32] = {};
    return cudaMemcpyToSymbol(g_phase, zeros, sizeof zeros) == cudaSuccess ? n : -1;
}
#endif

// [T_total, H, d] bf16 tensor (d = 64 or 128), boxes of `box_cols` columns x 1 head x 64
// rows; 64-column boxes use the 128-byte swizzle, 32-column boxes the 64-byte swizzle,
// 128-column boxes none.  With d = 64 a box at column 64 lies wholly outside the tensor and
// reads zeros: the kernels then see the head zero-padded to 128 channels.
bool make_map(CUtensorMap* m, const void* base, int64_t T_total, int H, int d, int box_cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T_total};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    const cuuint32_t box[3] = {(cuuint32_t)box_cols, 1, kC};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapSwizzle sw = box_cols == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                   : CU_TENSOR_MAP_SWIZZLE_NONE;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fwdtc

#ifdef KDA_PHASE_TIMING
extern "C" int kda_debug_phase_cycles(unsigned long long* out, int n) {
    return fwdtc::debug_phase_cycles(out, n);
}
extern "C" int kda_debug_chain_cycles(unsigned long long* out, int n) {
    return fwdtc::debug_chain_cycles(out, n);
}
#endif

size_t fwd_tc_workspace_size(int64_t T_total, int N, int H) {
    return fwdtc::ws_layout(T_total, N, H).total;
}

cudaError_t launch_fwd_tc(const FwdArgs& a) {
    using namespace fwdtc;
    if ((int64_t)a.N * a.H == 0) return cudaSuccess;
    if (a.bimg && a.o) return cudaErrorInvalidValue;  // the image stores take the output's place
    const bool mixed = a.gate_kind == 1;  // the softplus gate on the mixed path
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    const WsLayout L = ws_layout(a.T_total, a.N, a.H);
    const int maxchunks = (int)(a.T_total / kC + a.N);
    int32_t* chunk_off = reinterpret_cast<int32_t*>(ws + L.off_chunk_off);
    int4* chunk_tab = reinterpret_cast<int4*>(ws + L.off_tab);
    int32_t* order = reinterpret_cast<int32_t*>(ws + L.off_order);
    uint8_t* pkg = ws + L.off_pkg;

    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // The fused form needs equal sequence lengths (no cu_seqlens: the chunk-major item order
    // then follows every chain in step), at most kFusedMaxChains chains, and SMs left over
    // for the intra stage, and no backward image blocks wanted.  KDA_FWD_FUSED=0 in the environment
    // selects the two-launch form.
    // The ring and its flags live in the workspace's package region, which holds
    // H * maxchunks >= C * nct packages: nct > ring_slots leaves room for both.
    const int C = a.N * a.H;
    const int64_t nct_all = a.N > 0 ? (a.T_total / a.N + kC - 1) / kC : 0;
    int ring_slots = C > 0 ? (int)(kRingBytesMax / ((size_t)C * kPkgBytes)) : 0;
    ring_slots = ring_slots > kRingSlotsMax ? kRingSlotsMax : ring_slots;
    const char* fenv = getenv("KDA_FWD_FUSED");
    const bool fused = !a.bimg && a.cu_seqlens == nullptr && a.T_total > 0 &&
                       C <= kFusedMaxChains && sms - C >= 16 && ring_slots >= kRingSlotsMin && nct_all > ring_slots &&
                       !(fenv && strcmp(fenv, "0") == 0);
    // fused: the ring [C][ring_slots] packages, then ready flags [C][ring_slots], consumed
    // counters [C] and the item counter, inside the package region of the workspace
    uint8_t* ring = pkg;
    uint32_t* flags = reinterpret_cast<uint32_t*>(pkg + (size_t)C * ring_slots * kPkgBytes);
    const int n_flags = fused ? C * (ring_slots + 1) + 1 : 0;  // + the item counter

    {
        ProfScope prof("plan_kernel", a.stream);
        plan_kernel<<<1, 1024, 0, a.stream>>>(a.cu_seqlens, a.N, a.T_total, chunk_off, chunk_tab,
                                              order, flags, n_flags, a.dev_err);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    IntraParams ip{};
    ChainParams cp{};
    if (a.T_total > 0) {
        if (!make_map(&ip.tq, a.q, a.T_total, a.H, a.dk, 64) ||
            !make_map(&ip.tk, a.k, a.T_total, a.H, a.dk, 64) ||
            !make_map(&ip.tv, a.v, a.T_total, a.H, a.dv, 64) ||
            !make_map(&ip.tz, a.z, a.T_total, a.H, a.dk, 64))
            return cudaErrorInvalidValue;
    }
    ip.beta = static_cast<const __nv_bfloat16*>(a.beta);
    ip.A_log = a.A_log;
    ip.cu = a.cu_seqlens;
    ip.chunk_off = chunk_off;
    ip.chunk_tab = chunk_tab;
    ip.pkg = fused ? ring : pkg;
    ip.err = a.dev_err;
    ip.T_total = a.T_total;
    ip.g_min = a.g_min;
    ip.N = a.N;
    ip.H = a.H;
    ip.maxchunks = maxchunks;
    ip.bimg = static_cast<uint8_t*>(a.bimg);
    cp.pkg = pkg;
    cp.cu = a.cu_seqlens;
    cp.chunk_off = chunk_off;
    cp.order = order;
    cp.S0 = a.S0;
    cp.S_out = a.S_out;
    cp.o = static_cast<__nv_bfloat16*>(a.o);
    cp.err = a.dev_err;
    cp.T_total = a.T_total;
    cp.N = a.N;
    cp.H = a.H;
    cp.dk = a.dk;
    cp.dv = a.dv;
    cp.bimg = static_cast<uint8_t*>(a.bimg);
    cp.maxchunks = maxchunks;

    if (fused) {
        const int64_t len = a.T_total / a.N;
        ip.fused_C = C;
        ip.nct = (int)((len + kC - 1) / kC);
        ip.ring_slots = ring_slots;
        ip.ready = flags;
        ip.consumed = flags + (size_t)C * ring_slots;
        ip.item_ctr = reinterpret_cast<int*>(flags + (size_t)C * (ring_slots + 1));
        cp.fused = 1;
        cp.ring_slots = ring_slots;
        cp.ring = ring;
        cp.ready = ip.ready;
        cp.consumed = ip.consumed;
        FusedParams fp;
        fp.ip = ip;
        fp.cp = cp;
        fp.C = C;
        const void* fn = mixed ? reinterpret_cast<const void*>(fwd_fused_kernel<kGateSoftplus>)
                               : reinterpret_cast<const void*>(fwd_fused_kernel<kGateBounded>);
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFusedSmem);
        if (e != cudaSuccess) return e;
        void* args[] = {&fp};
        ProfScope prof(mixed ? "fwd_fused_mixed_kernel" : "fwd_fused_kernel", a.stream);
        e = cudaLaunchCooperativeKernel(fn, dim3(sms), dim3(kFusedThreads), args, kFusedSmem,
                                        a.stream);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }

    if (a.T_total > 0) {
        const void* fn = mixed ? reinterpret_cast<const void*>(intra_kernel<kGateSoftplus>)
                               : reinterpret_cast<const void*>(intra_kernel<kGateBounded>);
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kIntraSmem);
        if (e != cudaSuccess) return e;
        ProfScope prof(mixed ? "intra_mixed_kernel" : "intra_kernel", a.stream);
        if (mixed)
            intra_kernel<kGateSoftplus><<<sms, kIntraThreads, kIntraSmem, a.stream>>>(ip);
        else
            intra_kernel<kGateBounded><<<sms, kIntraThreads, kIntraSmem, a.stream>>>(ip);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (a.after_intra) {
        e = cudaEventRecord(a.after_intra, a.stream);
        if (e != cudaSuccess) return e;
    }
    const void* cfn = a.bimg ? reinterpret_cast<const void*>(chain_kernel<true>)
                             : reinterpret_cast<const void*>(chain_kernel<false>);
    e = cudaFuncSetAttribute(cfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kChainSmem);
    if (e != cudaSuccess) return e;
    const int grid = (int)(C < sms ? C : sms);
    ProfScope prof("chain_kernel", a.stream);
    if (a.bimg)
        chain_kernel<true><<<grid, kChainThreads, kChainSmem, a.stream>>>(cp);
    else
        chain_kernel<false><<<grid, kChainThreads, kChainSmem, a.stream>>>(cp);
    return cudaGetLastError();
}

}  // namespace kda
