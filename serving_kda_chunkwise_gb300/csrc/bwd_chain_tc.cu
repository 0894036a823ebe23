// bwd_chain_tc.cu -- the backward's serial step on the sm_103a tensor cores: the gradient of
// the state at every chunk end, last chunk first, for bf16 problems.
//
// Reverse of the chunk form ("Kimi k3 技术报告详解（1）——架构再升华", section "Chunkwise
// parallel form": the derivatives of Vt = U - W S, O = (Gamma*Q) S + A Vt,
// S' = Diag(gamma^C) S + K~^T Vt with respect to S, the pages print no backward): with dS'
// the gradient at a chunk's end and dO its output gradient,
//   Z  = K~ dS' + A^T dO                          (the gradient of Vt)
//   dS = Diag(gamma^C) dS' + (Gamma*Q)^T dO - W^T Z   (the gradient at the chunk's start).
// Every operand except dS' and dO is the chunk's package from the forward's intra stage
// (fwd_tc_layout.cuh), kept in the workspace; dO is read by TMA.
//
// One CTA per (sequence, head) at a time, the gradient transposed in TMEM (lane j holds
// column j of dS, i.e. row j of dS^T), as in the forward's chain stage (fwd_chain.cuh):
//   MMA1  Z^T  = dS'^T_hi [K~_hi; K~_lo]^T + dS'^T_lo K~_hi^T + dO^T [A_hi; A_lo]
//                                                            (M = 128 value columns, N = 64)
//   E1    -Z^T -> bf16 hi + lo into TMEM
//   MMA2  D2   = dO^T (Gamma*Q) + (-Z)^T_hi W + (-Z)^T_lo W       (N = 128 key channels)
//   E2    dS^T <- dS'^T Diag(gamma^C) + D2 in fp32 registers; bf16 hi + lo copy into TMEM
// For the per-chunk kernels, each chunk's image block (bwd_tc_layout.cuh) receives dS_C^T (the
// gradient at the chunk's end) and dVt^T as bf16 operand images; after a sequence's first
// chunk the gradient of the initial state is written out in fp32.
#include <cuda.h>

#include "bwd_tc_layout.cuh"
#include "fwd_tc_layout.cuh"
#include "kda_common.cuh"
#include "kda_internal.h"
#include "tc_util.cuh"

namespace kda {
namespace bwdtc {
namespace {

using namespace tc;
using fwdtc::kC;
using fwdtc::kD;

// Optional per-phase cycle counters (debug builds with -DKDA_PHASE_TIMING only): the MMA
// thread and thread 0 of CTA 0 accumulate clock64() deltas.
#ifdef KDA_PHASE_TIMING
__device__ unsigned long long g_gchain_phase[16];
#define GC_T0() long long gc_t = clock64()
#define GC_MARK(i)                                                                         \
    do {                                                                                   \
        const long long gc_n = clock64();                                                  \
        if (cta == 0) atomicAdd(&g_gchain_phase[(i)], (unsigned long long)(gc_n - gc_t)); \
        gc_t = gc_n;                                                                       \
    } while (0)
#else
#define GC_T0() \
    do {        \
    } while (0)
#define GC_MARK(i) \
    do {           \
    } while (0)
#endif

constexpr int kThreads = 320;  // 8 epilogue warps, an MMA thread (warp 8), copy lanes (warp 9)
constexpr int kMmaT = 256;
constexpr int kCopyW = 9;

// shared memory (1024-aligned offsets)
constexpr uint32_t kPA = 0;         // part A [W; Gamma*Q], two stages of 32 KB
constexpr uint32_t kKC = 65536;     // K~ hi + lo, two stages of 32 KB
constexpr uint32_t kAT = 131072;    // A hi + lo, two stages of 16 KB
constexpr uint32_t kDO = 163840;    // dO [2 blk][64 r][128 B], two stages of 16 KB
constexpr uint32_t kGm = 196608;    // gamma^C, four stages of 512 B
constexpr uint32_t kBars = 198656;
constexpr uint32_t kSmem = kBars + 256 + 1024;
static_assert(kSmem <= 232448, "gradient chain exceeds the shared-memory limit");

// TMEM columns: dS^T bf16 hi [0, 64); -Z^T bf16 hi [64, 96), lo [96, 128); D1 and D1b (Z^T in
// two parts, added in E1) [128, 192) and [384, 448); dS^T bf16 lo [192, 256); D2 [256, 384)
constexpr uint32_t kTS = 0, kTZ = 64, kTZlo = 96, kTD1 = 128, kTSlo = 192, kTD2 = 256, kTD1b = 384, kTCols = 512;

struct Params {
    CUtensorMap tdo;  // dO [T_total, H, dv] bf16, boxes of 64 columns x 1 head x 64 rows
    const uint8_t* pkg;       // packages [H][maxchunks]
    const int32_t* cu;
    const int32_t* chunk_off;
    const int32_t* order;     // sequences, longest first
    const float* dS_out;      // [N][H][dk][dv] or nullptr
    uint8_t* bimg;            // image blocks [chunks][H]
    float* dS0;               // [N][H][dk][dv] or nullptr
    unsigned* err;
    int64_t T_total;
    int N, H, maxchunks, dk, dv;
};

__device__ __forceinline__ int chain_of(int k, int b, int G) {
    return k * G + ((k & 1) ? (G - 1 - b) : b);
}

struct Chain {
    int n, h, nch, c0;
    int64_t t_begin, t_end;
};

__device__ __forceinline__ Chain decode_chain(const Params& p, int ci) {
    Chain c;
    c.n = __ldg(p.order + ci / p.H);
    c.h = ci % p.H;
    seq_range(p.cu, c.n, p.N, p.T_total, nullptr, c.t_begin, c.t_end);
    c.c0 = __ldg(p.chunk_off + c.n);
    c.nch = __ldg(p.chunk_off + c.n + 1) - c.c0;
    return c;
}

__device__ __forceinline__ void sync_all() { asm volatile("bar.sync 1, 320;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads, 1) bwd_chain_tc_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(sm);
    uint64_t* fullPA = reinterpret_cast<uint64_t*>(sm + kBars);  // [2]
    uint64_t* fullKC = fullPA + 2;                                // [2] K~ and gamma^C
    uint64_t* fullAT = fullPA + 4;                                // [2]
    uint64_t* fullDO = fullPA + 6;                                // [2]
    uint64_t* mma1 = fullPA + 8;                                  // [2]
    uint64_t* mma2 = fullPA + 10;                                 // [2]
    uint64_t* z_ready = fullPA + 12;                              // [2], 8 arrivals
    uint64_t* s_ready = fullPA + 14;                              // 8 arrivals
    uint64_t* drain = fullPA + 15;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fullPA + 16);
    __shared__ int s_abort;
    volatile int* abort = &s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x, G = gridDim.x;
    if (tid == 0) {
        for (int i = 0; i < 16; ++i) mbar_init(&fullPA[i], 1);
        mbar_init(&z_ready[0], 8);
        mbar_init(&z_ready[1], 8);
        mbar_init(s_ready, 8);
        fence_mbar_init();
        s_abort = 0;
    }
    if (warp == 0) tmem_alloc(tmem_slot, kTCols);
    tc_fence_before();
    sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n_chains = p.N * p.H;

    if (tid == kMmaT) {
        // ------------------------------------------------------------ MMA thread
        constexpr uint32_t id1s = idesc_bf16(128, 64, false, false);  // A in TMEM, B K-major
        constexpr uint32_t id1d = idesc_bf16(128, 64, true, true);    // dO^T x A, both MN-major
        constexpr uint32_t id2d = idesc_bf16(128, 128, true, true);   // dO^T x (Gamma Q)
        constexpr uint32_t id2z = idesc_bf16(128, 128, false, true);  // (-Z)^T x W
        uint32_t g = 0;
        bool ok = true;
        GC_T0();
        for (int k = 0; ok; ++k) {
            const int ci = chain_of(k, cta, G);
            if (ci >= n_chains) break;
            const Chain c = decode_chain(p, ci);
            for (int t = c.nch - 1; t >= 0; --t, ++g) {
                const uint32_t st = g & 1, ph = (g >> 1) & 1;
                // Z^T = dO^T [A_hi; A_lo]      (K = 64 query tokens, A rows as MN-major B)
                //     + dS'^T [K~_hi; K~_lo]^T (K = 128 key channels, K~ rows as K-major B).
                // The dO part needs no dS': it is issued first, while E2 of the previous chunk
                // still runs (D1 is free: E1 of the previous chunk, its reader, preceded the
                // previous MMA2).
                if (!mbar_wait_ab(&fullAT[st], ph, p.err, abort)) { ok = false; break; }
                GC_MARK(1);
                if (!mbar_wait_ab(&fullDO[st], ph, p.err, abort)) { ok = false; break; }
                GC_MARK(2);
                tc_fence_after();
                const uint32_t d1 = tmem + kTD1;
                const uint64_t dDO = sdesc_sw128(sbase + kDO + st * 16384, 8192, 1024);
                const uint64_t dAT = sdesc_sw128(sbase + kAT + st * 16384, 8192, 1024);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int part = ks >> 2, kk = ks & 3;  // part 0: A hi, 1: A lo
                    mma_bf16(d1, dDO + ((kk * 2048) >> 4), dAT + ((part * 8192 + kk * 2048) >> 4),
                             id1d, ks > 0);
                }
                if (!mbar_wait_ab(&fullKC[st], ph, p.err, abort)) { ok = false; break; }
                GC_MARK(0);
                if (!mbar_wait_ab(s_ready, g & 1, p.err, abort)) { ok = false; break; }
                GC_MARK(3);
                tc_fence_after();
                const uint64_t dKC = sdesc_sw128(sbase + kKC + st * 32768, 0, 1024);
                // two independent accumulators, issued alternately: D1 takes dS hi x K~ hi and
                // dS lo x K~ hi over key steps 0..3, D1b dS hi x K~ lo and dS lo x K~ hi over
                // steps 4..7 (E1 adds them)
#pragma unroll
                for (int i = 0; i < 12; ++i) {
                    const int kka = i < 8 ? i : i - 8;           // D1: hi x hi (8), lo x hi (kk 0..3)
                    const bool loa = i >= 8;
                    mma_bf16_ts(d1, tmem + (loa ? kTSlo : kTS) + 8 * kka,
                                dKC + (((kka >> 2) * 8192 + (kka & 3) * 32) >> 4), id1s, 1);
                    const int kkb = i < 8 ? i : i - 4;           // D1b: hi x lo (8), lo x hi (kk 4..7)
                    const bool lob = i >= 8;
                    mma_bf16_ts(tmem + kTD1b, tmem + (lob ? kTSlo : kTS) + 8 * kkb,
                                dKC + (((lob ? 0 : 16384) + (kkb >> 2) * 8192 + (kkb & 3) * 32) >> 4), id1s,
                                i > 0);
                }
                mma_commit(&mma1[st]);
                GC_MARK(4);
                if (!mbar_wait_ab(&fullPA[st], ph, p.err, abort)) { ok = false; break; }
                GC_MARK(5);
                // D2 = dO^T (Gamma*Q) + (-Z)^T_hi W + (-Z)^T_lo W  (K = 64 tokens).  The dO part
                // needs no Z: it goes in before E1 ends (D2 is free: E2 of the previous chunk,
                // its reader, preceded this chunk's dS' products).
                const uint64_t dQ = sdesc_sw128(sbase + kPA + st * 32768 + fwdtc::kPkgStkQ,
                                                fwdtc::kPkgStkBlk, 1024);
                const uint64_t dW = sdesc_sw128(sbase + kPA + st * 32768, fwdtc::kPkgStkBlk, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + kTD2, dDO + ((kk * 2048) >> 4), dQ + ((kk * 2048) >> 4), id2d,
                             kk > 0);
                if (!mbar_wait_ab(&z_ready[st], ph, p.err, abort)) { ok = false; break; }
                GC_MARK(6);
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int part = ks >> 2, kk = ks & 3;  // part 0: -Z hi, 1: -Z lo
                    mma_bf16_ts(tmem + kTD2, tmem + (part ? kTZlo : kTZ) + 8 * kk,
                                dW + ((kk * 2048) >> 4), id2z, 1);
                }
                mma_commit(&mma2[st]);
                GC_MARK(7);
            }
        }
    }

    // Copy lanes of warp 9, one per part, each refilling its stage as soon as it is free:
    //   lane 0: part A (W; Gamma*Q), free once MMA2 of chunk g - 2 completed;
    //   lane 1: K~ hi + lo and gamma^C (four stages), free once MMA1 of chunk g - 2 completed;
    //   lane 2: A hi + lo, free once MMA1 of chunk g - 2 completed;
    //   lane 3: dO by TMA, free once MMA2 of chunk g - 2 completed.
    int last_ph[2] = {-1, -1};
    const int cpart = (warp == kCopyW && lane < 4) ? lane : -1;
    if (cpart >= 0) {
        uint32_t g = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int ci = chain_of(k, cta, G);
            if (ci >= n_chains) break;
            const Chain c = decode_chain(p, ci);
            for (int t = c.nch - 1; t >= 0; --t, ++g) {
                const uint32_t st = g & 1;
                const uint8_t* src = p.pkg + ((size_t)c.h * p.maxchunks + c.c0 + t) * fwdtc::kPkgBytes;
                uint64_t* freed = (cpart == 0 || cpart == 3) ? &mma2[st] : &mma1[st];
                if (g >= 2 && !mbar_wait_ab(freed, ((g - 2) >> 1) & 1, p.err, abort)) { ok = false; break; }
                if (cpart == 0) {
                    mbar_expect_tx(&fullPA[st], fwdtc::kPkgPartA);
                    bulk_g2s(sm + kPA + st * 32768, src + fwdtc::kPkgStk, fwdtc::kPkgPartA, &fullPA[st]);
                } else if (cpart == 1) {
                    mbar_expect_tx(&fullKC[st], fwdtc::kPkgKTBytes + fwdtc::kPkgGBytes);
                    bulk_g2s(sm + kKC + st * 32768, src + fwdtc::kPkgKT, fwdtc::kPkgKTBytes, &fullKC[st]);
                    bulk_g2s(sm + kGm + (g & 3) * fwdtc::kPkgGBytes, src + fwdtc::kPkgG,
                             fwdtc::kPkgGBytes, &fullKC[st]);
                } else if (cpart == 2) {
                    mbar_expect_tx(&fullAT[st], fwdtc::kPkgAQKBytes);
                    bulk_g2s(sm + kAT + st * 16384, src + fwdtc::kPkgAQK, fwdtc::kPkgAQKBytes, &fullAT[st]);
                } else {
                    const int t0 = (int)(c.t_begin + (int64_t)t * kC);
                    mbar_expect_tx(&fullDO[st], 16384);
                    tma_load_3d(sm + kDO + st * 16384, &p.tdo, 0, c.h, t0, &fullDO[st]);
                    tma_load_3d(sm + kDO + st * 16384 + 8192, &p.tdo, 64, c.h, t0, &fullDO[st]);
                }
                last_ph[st] = (int)((g >> 1) & 1);
            }
        }
    }

    if (warp < 8) {
        // ------------------------------------------------------- epilogue warps
        const int q = warp & 3, wg = warp >> 2;
        const int j = 32 * q + lane;  // value column = TMEM lane
        const uint32_t lb = static_cast<uint32_t>(32 * q) << 16;
        uint32_t g = 0;
        bool ok = true;
        const bool rec = (tid == 0);
        GC_T0();
        for (int k = 0; ok; ++k) {
            const int ci = chain_of(k, cta, G);
            if (ci >= n_chains) break;
            const Chain c = decode_chain(p, ci);
            // dS[e] = dS[i = 64 wg + e][j] (fp32, registers); padding rows and columns are zero
            float dS[64];
            const bool sv = j < p.dv && 64 * wg < p.dk;
            const size_t sbase_el = ((size_t)(c.n * p.H + c.h) * p.dk + 64 * wg) * p.dv + j;
#pragma unroll
            for (int e = 0; e < 64; ++e) dS[e] = (p.dS_out && sv) ? p.dS_out[sbase_el + (size_t)e * p.dv] : 0.f;
            if (c.nch > 0) {
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    uint32_t ph8[8], pl8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float a0 = dS[16 * x + 2 * e], a1 = dS[16 * x + 2 * e + 1];
                        ph8[e] = pack_bf16x2(a0, a1);
                        pl8[e] = pack_bf16x2(a0 - __uint_as_float(ph8[e] << 16),
                                             a1 - __uint_as_float(ph8[e] & 0xffff0000u));
                    }
                    tmem_st8(tmem + lb + kTS + 32 * wg + 8 * x, ph8);
                    tmem_st8(tmem + lb + kTSlo + 32 * wg + 8 * x, pl8);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_ready);
            }
            for (int t = c.nch - 1; t >= 0; --t, ++g) {
                const uint32_t st = g & 1, ph = (g >> 1) & 1;
                // the gradient at this chunk's end: row j of key-channel block wg of the dS_C^T
                // image (bf16 hi + lo), the 64 channels in eight 16-byte chunks
                uint8_t* blk = p.bimg + ((size_t)(c.c0 + t) * p.H + c.h) * kBiBytes;
                {
                    uint8_t* dst = blk + kBiDS + wg * 16384 + j * 128;
#pragma unroll
                    for (int c8 = 0; c8 < 8; c8 += 2) {
                        float v0[8], v1[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            v0[e] = dS[8 * c8 + e];
                            v1[e] = dS[8 * c8 + 8 + e];
                        }
                        uint4 h0, l0, h1, l1;
                        pk8_hilo(v0, h0, l0);
                        pk8_hilo(v1, h1, l1);
                        st_swz_pair(dst, c8, j, h0, h1);
                        st_swz_pair(dst + 32768, c8, j, l0, l1);
                    }
                }
                if (rec) GC_MARK(8);
                // ---- E1: -Z^T as bf16 hi + lo for tokens r = 32 wg + e
                bool okc = mbar_wait_ab(&mma1[st], ph, p.err, abort);
                if (rec) GC_MARK(9);
                if (okc) {
                    tc_fence_after();
                    float z0[16], z1[16], y0[16], y1[16];
                    tmem_ld16(tmem + lb + kTD1 + 32 * wg, z0);
                    tmem_ld16(tmem + lb + kTD1 + 32 * wg + 16, z1);
                    tmem_ld16(tmem + lb + kTD1b + 32 * wg, y0);
                    tmem_ld16(tmem + lb + kTD1b + 32 * wg + 16, y1);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        z0[e] += y0[e];
                        z1[e] += y1[e];
                    }
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        uint32_t hi[8], lo[8];
#pragma unroll
                        for (int e2 = 0; e2 < 8; ++e2) {
                            const float a0 = -(hf ? z1[2 * e2] : z0[2 * e2]);
                            const float a1 = -(hf ? z1[2 * e2 + 1] : z0[2 * e2 + 1]);
                            hi[e2] = pack_bf16x2(a0, a1);
                            lo[e2] = pack_bf16x2(a0 - __uint_as_float(hi[e2] << 16),
                                                 a1 - __uint_as_float(hi[e2] & 0xffff0000u));
                        }
                        tmem_st8(tmem + lb + kTZ + 16 * wg + 8 * hf, hi);
                        tmem_st8(tmem + lb + kTZlo + 16 * wg + 8 * hf, lo);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&z_ready[st]);
                if (rec) GC_MARK(10);
                // dVt^T row j into the image block, read back from TMEM while MMA2 runs: tokens
                // 32 wg + 8 x are chunk 4 wg + x of the row; TMEM holds -Z, so the words are
                // negated
                if (okc) {
                    float fh[16], fl[16];
                    tmem_ld16(tmem + lb + kTZ + 16 * wg, fh);
                    tmem_ld16(tmem + lb + kTZlo + 16 * wg, fl);
                    tmem_ld_wait();
                    constexpr uint32_t kSign = 0x80008000u;
                    uint32_t wh[16], wl[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        wh[e] = __float_as_uint(fh[e]) ^ kSign;
                        wl[e] = __float_as_uint(fl[e]) ^ kSign;
                    }
                    uint8_t* zimg = blk + kBiDV + j * 128;
#pragma unroll
                    for (int pr = 0; pr < 2; ++pr) {
                        st_swz_pair(zimg, 4 * wg + 2 * pr, j,
                                    make_uint4(wh[8 * pr], wh[8 * pr + 1], wh[8 * pr + 2], wh[8 * pr + 3]),
                                    make_uint4(wh[8 * pr + 4], wh[8 * pr + 5], wh[8 * pr + 6], wh[8 * pr + 7]));
                        st_swz_pair(zimg + 16384, 4 * wg + 2 * pr, j,
                                    make_uint4(wl[8 * pr], wl[8 * pr + 1], wl[8 * pr + 2], wl[8 * pr + 3]),
                                    make_uint4(wl[8 * pr + 4], wl[8 * pr + 5], wl[8 * pr + 6], wl[8 * pr + 7]));
                    }
                }
                if (rec) GC_MARK(11);
                // ---- E2: dS^T <- dS'^T Diag(gamma^C) + D2; bf16 copy for the next MMA1
                okc = okc && mbar_wait_ab(&mma2[st], ph, p.err, abort);
                if (rec) GC_MARK(12);
                if (okc) {
                    tc_fence_after();
                    const float* gam = reinterpret_cast<const float*>(sm + kGm + (g & 3) * fwdtc::kPkgGBytes) + 64 * wg;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        float d0[16], d1v[16];
                        tmem_ld16(tmem + lb + kTD2 + 64 * wg + 32 * hf, d0);
                        tmem_ld16(tmem + lb + kTD2 + 64 * wg + 32 * hf + 16, d1v);
                        float4 gv[8];
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4)
                            gv[e4] = *reinterpret_cast<const float4*>(gam + 32 * hf + 4 * e4);
                        tmem_ld_wait();
#pragma unroll
                        for (int qt = 0; qt < 2; ++qt) {
                            uint32_t pk[8], pl[8];
#pragma unroll
                            for (int e4 = 0; e4 < 4; ++e4) {
                                const float4 g4 = gv[4 * qt + e4];
                                const int e = 32 * hf + 16 * qt + 4 * e4;
                                const float* dd = qt ? d1v : d0;
                                dS[e] = fmaf(g4.x, dS[e], dd[4 * e4]);
                                dS[e + 1] = fmaf(g4.y, dS[e + 1], dd[4 * e4 + 1]);
                                dS[e + 2] = fmaf(g4.z, dS[e + 2], dd[4 * e4 + 2]);
                                dS[e + 3] = fmaf(g4.w, dS[e + 3], dd[4 * e4 + 3]);
#pragma unroll
                                for (int y = 0; y < 2; ++y) {
                                    const float a0 = dS[e + 2 * y], a1 = dS[e + 2 * y + 1];
                                    const uint32_t h = pack_bf16x2(a0, a1);
                                    pk[2 * e4 + y] = h;
                                    pl[2 * e4 + y] = pack_bf16x2(a0 - __uint_as_float(h << 16),
                                                                 a1 - __uint_as_float(h & 0xffff0000u));
                                }
                            }
                            tmem_st8(tmem + lb + kTS + 32 * wg + 16 * hf + 8 * qt, pk);
                            tmem_st8(tmem + lb + kTSlo + 32 * wg + 16 * hf + 8 * qt, pl);
                        }
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (!okc) { ok = false; break; }
                if (lane == 0 && t > 0) mbar_arrive(s_ready);
                if (rec) GC_MARK(13);
            }
            if (!ok) break;
            if (p.dS0 && sv) {
#pragma unroll
                for (int e = 0; e < 64; ++e) p.dS0[sbase_el + (size_t)e * p.dv] = dS[e];
            }
        }
    }

    sync_all();
    const bool aborted = s_abort != 0;
    // on an abort, let copies and MMAs still in flight land before leaving
    if (aborted && cpart >= 0) {
        uint64_t* bar = cpart == 0 ? fullPA : cpart == 1 ? fullKC : cpart == 2 ? fullAT : fullDO;
        for (int s2 = 0; s2 < 2; ++s2)
            if (last_ph[s2] >= 0) mbar_wait(&bar[s2], last_ph[s2], nullptr);
    }
    if (aborted && tid == kMmaT) {
        mma_commit(drain);
        mbar_wait(drain, 0, nullptr);
    }
    tc_fence_before();
    sync_all();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTCols);
    }
}

}  // namespace
}  // namespace bwdtc

#ifdef KDA_PHASE_TIMING
extern "C" int kda_debug_gchain_cycles(unsigned long long* out, int n) {
    if (n > 16) n = 16;
    if (cudaMemcpyFromSymbol(out, bwdtc::g_gchain_phase, n * sizeof(unsigned long long)) != cudaSuccess)
        return -1;
    static const unsigned long long zeros[16] = {};
    return cudaMemcpyToSymbol(bwdtc::g_gchain_phase, zeros, sizeof zeros) == cudaSuccess ? n : -1;
}
#endif

// The gradient chain on the tensor cores: reads the packages the forward's two-launch form
// left in its workspace (fwd_ws), writes dS_C and dVt into the image blocks and dS0.
cudaError_t launch_bwd_chain_tc(const BwdArgs& a, void* fwd_ws, void* bimg, cudaStream_t stream) {
    using namespace bwdtc;
    if ((int64_t)a.N * a.H == 0) return cudaSuccess;
    const fwdtc::WsLayout L = fwdtc::ws_layout(a.T_total, a.N, a.H);
    uint8_t* ws = static_cast<uint8_t*>(fwd_ws);
    Params p{};
    if (a.T_total > 0 && !fwdtc::make_map(&p.tdo, a.dout, a.T_total, a.H, a.dv, 64))
        return cudaErrorInvalidValue;
    p.pkg = ws + L.off_pkg;
    p.cu = a.cu_seqlens;
    p.chunk_off = reinterpret_cast<const int32_t*>(ws + L.off_chunk_off);
    p.order = reinterpret_cast<const int32_t*>(ws + L.off_order);
    p.dS_out = a.dS_out;
    p.bimg = static_cast<uint8_t*>(bimg);
    p.dS0 = a.dS0;
    p.err = a.dev_err;
    p.T_total = a.T_total;
    p.N = a.N;
    p.H = a.H;
    p.maxchunks = (int)(a.T_total / kC + a.N);
    p.dk = a.dk;
    p.dv = a.dv;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int C = a.N * a.H;
    cudaError_t e = cudaFuncSetAttribute(bwd_chain_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmem);
    if (e != cudaSuccess) return e;
    ProfScope prof("bwd_chain_tc_kernel", stream);
    bwd_chain_tc_kernel<<<(C < sms ? C : sms), kThreads, kSmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
