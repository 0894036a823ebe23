// fwd_chain.cuh -- the serial stage of the tensor-core chunked forward: for every (sequence,
// head), chunk after chunk, the pseudo-values, the output and the state update
// ("Kimi k3 技术报告详解（1）——架构再升华", section "Chunkwise parallel form"):
//   Vt = U - W S,   O = (Gamma*Q) S + A Vt,   S <- Diag(gamma^C) S + K~^T Vt.
//
// One CTA per (sequence, head) at a time, all 128 value columns, with the state kept
// transposed in tensor memory: lane j of TMEM holds column j of S (row j of S^T).  Then
// every product of the chain has S^T or Vt^T as its A operand, read straight from TMEM,
// and the package tiles (bf16, in shared memory) as B operands:
//   MMA1  D1  = S^T [W; Gamma*Q]^T        (M = 128 value columns, N = 128, K = 128 keys)
//             -> lanes j, columns r < 64: X^T = (W S)^T;  columns 64 + r: ((Gamma*Q) S)^T
//   E1    Vt^T = U^T - X^T, rounded to bf16 hi + lo and stored back into TMEM
//   MMA2  dS^T = [Vt_hi | Vt_lo | Vt_hi]^T [K~_hi; K~_hi; K~_lo]   (K = 3 x 64 tokens)
//   E2    S^T <- S^T Diag(gamma^C) + dS^T in fp32 registers; bf16 copy of S^T into TMEM
//   MMA3  O^T += [Vt_hi | Vt_lo | Vt_hi]^T [A_hi; A_hi; A_lo]^T  (into D1's columns 64..127)
//   E3    O^T -> bf16 -> o (for each token, the 32 lanes of a warp store 64 contiguous bytes)
// With no output wanted (the forward of a backward pass), neither the A tile, MMA3 nor E3 runs,
// and MMA1 takes the W rows alone (N = 64).  The backward's instantiation (kImg) also writes
// S_0^T and Vt^T of every chunk as operand images, each warp's 4 KB parts through shared-memory
// stages and bulk copies.
// The state update takes three bf16 products (hi x hi, lo x hi, hi x lo) so that the fp32
// state is not limited by bf16 rounding of K~ or Vt; the output takes the same three.
// No intermediate of the chain goes through shared memory, so a chain step is
// MMA1 -> E1 -> MMA2 -> E2 with one TMEM round trip per epilogue.
//
// Threads: 8 epilogue warps (warp w reaches TMEM lanes 32 (w % 4) .. + 31, i.e. value columns
// j; warps w and w + 4 split the other index), one thread issuing every MMA, one issuing
// every bulk copy.  They meet only on mbarriers.  Each CTA walks a fixed list of (sequence,
// head) chains: sequences sorted longest first, dealt to the CTAs in a snake order.
#pragma once

#include <cuda.h>

#include "bwd_tc_layout.cuh"
#include "fwd_tc_layout.cuh"
#include "kda_common.cuh"
#include "tc_util.cuh"

namespace kda {
namespace fwdtc {
namespace {

using namespace tc;

// Optional per-phase cycle counters (debug builds with -DKDA_PHASE_TIMING only): the MMA
// thread and lane 0 of epilogue warp 0 of CTA 0 accumulate clock64() deltas.
#ifdef KDA_PHASE_TIMING
__device__ unsigned long long g_chain_phase[16];
#define CH_T0() long long ch_t = clock64()
#define CH_MARK(i)                                                       \
    do {                                                                 \
        const long long ch_n = clock64();                                \
        if (cta == 0) atomicAdd(&g_chain_phase[(i)], (unsigned long long)(ch_n - ch_t)); \
        ch_t = ch_n;                                                     \
    } while (0)
#else
#define CH_T0() \
    do {        \
    } while (0)
#define CH_MARK(i) \
    do {           \
    } while (0)
#endif

constexpr int kChainThreads = 320;
// Barrier over the chain stage's 320 threads (the fused kernel's CTAs have more threads; the
// rest leave at once).
__device__ __forceinline__ void chain_sync() { asm volatile("bar.sync 1, 320;" ::: "memory"); }
constexpr int kMmaT = 256;   // lane 0 of warp 8
constexpr int kCopyT = 288;  // lane 0 of warp 9

// shared memory (1024-aligned offsets)
constexpr uint32_t kChPA = 0;          // part A, two stages of 32 KB
// no output wanted (a backward pass): part A holds W alone (two stages of 16 KB) and the
// image stores have two 4 KB stages per epilogue warp: the first set in the rest of part A's
// place, the second in the A tile's place (warps 0..3) and at kChStageB (warps 4..7)
constexpr uint32_t kChWOnly = 16384, kChStage = 32768;
constexpr uint32_t kChKC = 65536;      // K~ hi + lo, two stages of 32 KB
constexpr uint32_t kChAT = 131072;     // A hi + lo (16 KB)
constexpr uint32_t kChU = 147456;      // U, two stages of 32 KB
constexpr uint32_t kChG = 212992;      // gamma^C, three stages of 512 B
constexpr uint32_t kChBars = 214528;
constexpr uint32_t kChStageB = 214784;
constexpr uint32_t kChainSmem = kChStageB + 16384 + 1024;
static_assert(kChainSmem <= 232448, "chain kernel exceeds the shared-memory limit");

// TMEM columns: S^T bf16 [0, 64); Vt^T bf16 hi [64, 96), lo [96, 128); D1 for chunk g in
// [128 + 128 (g & 1), +128); dS^T [384, 512)
constexpr uint32_t kTS = 0, kTV = 64, kTVlo = 96, kTD1 = 128, kTDS = 384, kTCols = 512;

struct ChainParams {
    const uint8_t* pkg;
    const int32_t* cu;
    const int32_t* chunk_off;
    const int32_t* order;
    const float* S0;
    float* S_out;
    __nv_bfloat16* o;
    unsigned* err;
    int64_t T_total;
    int N, H, maxchunks;
    // head sizes of q, k (dk) and v, o, S (dv), 64 or 128: a 64 is zero-padded to 128 inside
    // (the tensor maps read zeros past it), so only the state and output addresses use them
    int dk, dv;
    // optional (nullptr otherwise), for a backward pass, which wants no output (o == nullptr):
    // the image blocks [chunks][H] (bwd_tc_layout.cuh), chunk = chunk_off[n] + t, receive
    // S_0^T (the state at the chunk start) and Vt^T as bf16 hi + lo operand images
    uint8_t* bimg;
    // fused kernel only (fused = 0 otherwise): CTA c serves chain c and reads chunk t from
    // ring slot c * ring_slots + t % ring_slots once ready[slot] >= t + 1; it raises
    // consumed[c] to t + 1 once every part of chunk t is in shared memory
    int fused, ring_slots;
    const uint8_t* ring;
    const uint32_t* ready;
    uint32_t* consumed;
};

// The k-th chain of CTA b out of G: snake order over the longest-first list.
__device__ __forceinline__ int chain_of(int k, int b, int G) {
    return k * G + ((k & 1) ? (G - 1 - b) : b);
}

struct Chain {
    int ci, n, h, nch;
    int64_t t_begin, t_end;
    const uint8_t* pkg0;
};

__device__ __forceinline__ Chain decode_chain(const ChainParams& p, int ci) {
    Chain c;
    c.ci = ci;
    c.n = __ldg(p.order + ci / p.H);
    c.h = ci % p.H;
    seq_range(p.cu, c.n, p.N, p.T_total, nullptr, c.t_begin, c.t_end);
    const int c0 = __ldg(p.chunk_off + c.n);
    c.nch = __ldg(p.chunk_off + c.n + 1) - c0;
    c.pkg0 = p.pkg + ((size_t)c.h * p.maxchunks + c0) * kPkgBytes;
    return c;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) { return pack_bf16x2(lo, hi); }

// kImg: the backward's instantiation, which writes the operand images (p.bimg) and no output.
template <bool kImg>
__device__ __forceinline__ void chain_body(const ChainParams& p, uint8_t* smem_raw, int cta, int ncta) {
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(sm);
    uint64_t* fullPA = reinterpret_cast<uint64_t*>(sm + kChBars);  // [2] part A
    uint64_t* fullU = fullPA + 2;                                  // [2] U + gamma^C
    uint64_t* fullKC = fullPA + 4;                                 // [2]
    uint64_t* fullAT = fullPA + 6;
    uint64_t* mma1 = fullPA + 7;                                   // [2]
    uint64_t* mma2 = fullPA + 9;                                   // [2]
    uint64_t* mma3 = fullPA + 11;                                  // [2]
    uint64_t* vt_ready = fullPA + 13;                              // [2], 8 arrivals
    uint64_t* s_ready = fullPA + 15;                               // 8 arrivals
    uint64_t* drain = fullPA + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fullPA + 17);
    __shared__ int s_abort;
    __shared__ uint32_t s_landed_v;  // fused: chunks (counted over the CTA's chains) in smem
    volatile uint32_t* s_landed = &s_landed_v;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort = &s_abort;
    if (tid == 0) {
        for (int i = 0; i < 17; ++i) mbar_init(&fullPA[i], 1);
        mbar_init(&vt_ready[0], 8);
        mbar_init(&vt_ready[1], 8);
        mbar_init(s_ready, 8);
        fence_mbar_init();
        s_abort = 0;
        s_landed_v = 0;
    }
    if (warp == 0) tmem_alloc(tmem_slot, kTCols);
    tc_fence_before();
    chain_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n_chains = p.N * p.H;
    const int G = ncta;
    const bool want_o = !kImg && p.o != nullptr;

    if (tid == kMmaT) {
        // ------------------------------------------------------------ MMA thread
        constexpr uint32_t id1 = idesc_bf16(128, 128, false, false);
        constexpr uint32_t id1w = idesc_bf16(128, 64, false, false);  // no output: W rows alone
        constexpr uint32_t id2 = idesc_bf16(128, 128, false, true);
        constexpr uint32_t id3 = idesc_bf16(128, 64, false, false);
        const uint64_t dPA = sdesc_sw128(sbase + kChPA, 0, 1024);
        const uint64_t dKC = sdesc_sw128(sbase + kChKC, 8192, 1024);
        const uint64_t dAT = sdesc_sw128(sbase + kChAT, 0, 1024);
        uint32_t g = 0;
        bool ok = true;
        CH_T0();
        for (int k = 0; ok; ++k) {
            const int ci = chain_of(k, cta, G);
            if (ci >= n_chains) break;
            const Chain c = decode_chain(p, ci);
            for (int t = 0; t < c.nch; ++t, ++g) {
                const uint32_t st = g & 1, ph = (g >> 1) & 1;
                if (!mbar_wait_ab(&fullPA[st], ph, p.err, abort)) { ok = false; break; }
                CH_MARK(0);
                if (!mbar_wait_ab(s_ready, g & 1, p.err, abort)) { ok = false; break; }
                CH_MARK(1);
                tc_fence_after();
                const uint32_t d1 = tmem + kTD1 + 128 * st;
                if (want_o) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16_ts(d1, tmem + kTS + 8 * ks,
                                    dPA + ((st * kPkgPartA + (ks >> 2) * kPkgStkBlk + (ks & 3) * 32) >> 4),
                                    id1, ks > 0);
                } else {  // X^T = S^T W^T only (N = 64): the W rows of each key block, 8 KB apart
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16_ts(d1, tmem + kTS + 8 * ks,
                                    dPA + ((st * kChWOnly + (ks >> 2) * 8192 + (ks & 3) * 32) >> 4),
                                    id1w, ks > 0);
                }
                mma_commit(&mma1[st]);
                CH_MARK(2);
                if (!mbar_wait_ab(&fullKC[st], ph, p.err, abort)) { ok = false; break; }
                CH_MARK(3);
                if (!mbar_wait_ab(&vt_ready[st], ph, p.err, abort)) { ok = false; break; }
                CH_MARK(4);
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 12; ++ks) {
                    const int seg = ks >> 2, kk = ks & 3;
                    mma_bf16_ts(tmem + kTDS, tmem + (seg == 1 ? kTVlo : kTV) + 8 * kk,
                                dKC + ((st * kPkgKTBytes + (seg == 2 ? 16384u : 0u) + kk * 2048) >> 4),
                                id2, ks > 0);
                }
                mma_commit(&mma2[st]);
                CH_MARK(5);
                if (!want_o) {  // no output: neither the A tile nor MMA3
                    if (p.fused) *s_landed = g + 1;
                    continue;
                }
                if (!mbar_wait_ab(fullAT, g & 1, p.err, abort)) { ok = false; break; }
                CH_MARK(6);
                if (p.fused) *s_landed = g + 1;  // every part of chunk g is in shared memory
#pragma unroll
                for (int ks = 0; ks < 12; ++ks) {
                    const int seg = ks >> 2, kk = ks & 3;
                    mma_bf16_ts(d1 + 64, tmem + (seg == 1 ? kTVlo : kTV) + 8 * kk,
                                dAT + (((seg == 2 ? 8192u : 0u) + kk * 32) >> 4), id3, 1);
                }
                mma_commit(&mma3[st]);
                CH_MARK(7);
            }
        }
    }

    // Copy lanes: lanes 0..3 of warp 9 each stream one part of the packages, so that a part
    // is fetched as soon as its buffer is free, independently of the others.
    //   lane 0: part A ([W; Gamma*Q]), two stages, free once MMA1 of chunk g - 2 completed;
    //   lane 1: U and gamma^C, two stages of U (free once E1 of chunk g - 2 is done) and three
    //           of gamma (E2 of chunk g - 3 precedes E1 of chunk g - 2 on the same warps);
    //   lane 2: K~ hi + lo, two stages, free once MMA2 of chunk g - 2 completed;
    //   lane 3: A hi + lo, one stage, free once MMA3 of chunk g - 1 completed.
    int last_ph[2] = {-1, -1};  // the phase parity a drain must let land, per stage
    const int cpart = (warp == kCopyT / 32 && lane < (want_o ? 4 : 3)) ? lane : -1;
    if (cpart >= 0) {
        uint32_t g = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int ci = chain_of(k, cta, G);
            if (ci >= n_chains) break;
            const Chain c = decode_chain(p, ci);
            for (int t = 0; t < c.nch; ++t, ++g) {
                const uint32_t st = g & 1;
                const uint8_t* src;
                if (p.fused) {
                    const size_t slot = (size_t)c.ci * p.ring_slots + t % p.ring_slots;
                    src = p.ring + slot * kPkgBytes;
                    if (!wait_flag_ge(p.ready + slot, (uint32_t)t + 1, p.err, abort)) { ok = false; break; }
                    fence_proxy_async_global();
                } else {
                    src = c.pkg0 + (size_t)t * kPkgBytes;
                }
                if (cpart == 0) {
                    if (g >= 2 && !mbar_wait_ab(&mma1[st], ((g - 2) >> 1) & 1, p.err, abort)) { ok = false; break; }
                    if (want_o) {
                        mbar_expect_tx(&fullPA[st], kPkgPartA);
                        bulk_g2s(sm + kChPA + st * kPkgPartA, src + kPkgStk, kPkgPartA, &fullPA[st]);
                    } else {  // the W rows (the first 8 KB) of the two key blocks
                        mbar_expect_tx(&fullPA[st], kChWOnly);
                        bulk_g2s(sm + kChPA + st * kChWOnly, src + kPkgStk, 8192, &fullPA[st]);
                        bulk_g2s(sm + kChPA + st * kChWOnly + 8192, src + kPkgStk + kPkgStkBlk, 8192, &fullPA[st]);
                    }
                    last_ph[st] = (int)((g >> 1) & 1);
                } else if (cpart == 1) {
                    if (g >= 2 && !mbar_wait_ab(&vt_ready[st], ((g - 2) >> 1) & 1, p.err, abort)) { ok = false; break; }
                    mbar_expect_tx(&fullU[st], kPkgUBytes + kPkgGBytes);
                    bulk_g2s(sm + kChU + st * kPkgUBytes, src + kPkgU, kPkgUBytes, &fullU[st]);
                    bulk_g2s(sm + kChG + (g % 3) * kPkgGBytes, src + kPkgG, kPkgGBytes, &fullU[st]);
                    last_ph[st] = (int)((g >> 1) & 1);
                } else if (cpart == 2) {
                    if (g >= 2 && !mbar_wait_ab(&mma2[st], ((g - 2) >> 1) & 1, p.err, abort)) { ok = false; break; }
                    mbar_expect_tx(&fullKC[st], kPkgKTBytes);
                    bulk_g2s(sm + kChKC + st * kPkgKTBytes, src + kPkgKT, kPkgKTBytes, &fullKC[st]);
                    last_ph[st] = (int)((g >> 1) & 1);
                } else {
                    if (g >= 1 && !mbar_wait_ab(&mma3[(g - 1) & 1], ((g - 1) >> 1) & 1, p.err, abort)) { ok = false; break; }
                    mbar_expect_tx(fullAT, kPkgAQKBytes);
                    bulk_g2s(sm + kChAT, src + kPkgAQK, kPkgAQKBytes, fullAT);
                    last_ph[0] = (int)(g & 1);
                }
            }
        }
    }

    if (p.fused && warp == kCopyT / 32 && lane == 4) {
        // ------------------------------------------------ ring-slot releaser (fused)
        // Once the MMA thread has seen every part of chunk g land in shared memory, hand
        // the chunk's ring slot back to the intra stage (a gpu-scope release, kept off the
        // MMA thread).
        uint32_t g = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int ci = chain_of(k, cta, G);
            if (ci >= n_chains) break;
            const Chain c = decode_chain(p, ci);
            for (int t = 0; t < c.nch; ++t, ++g) {
                if (*s_landed < g + 1) {
                    const uint64_t t0 = globaltimer();
                    while (*s_landed < g + 1) {
                        if (*abort) { ok = false; break; }
                        if (globaltimer() - t0 > kWaitLimitNs) {
                            atomicOr(p.err, kDevErrTimeout);
                            *abort = 1;
                            ok = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                    if (!ok) break;
                }
                st_release_gpu(p.consumed + c.ci, (uint32_t)t + 1);
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
        CH_T0();
        const bool rec = (tid == 0);
        // E3 of chunk gg (first token t0): O^T -> bf16 -> o, straight from the lanes (for each
        // token the 32 lanes of a warp write 64 contiguous bytes); rows past the sequence end
        // belong to the next sequence and are skipped
        auto store_out = [&](uint32_t gg, int64_t t0, const Chain& c) -> bool {
            if (!want_o) return true;
            if (!mbar_wait_ab(&mma3[gg & 1], (gg >> 1) & 1, p.err, abort)) return false;
            tc_fence_after();
            float o0[16], o1[16];
            const uint32_t col = tmem + lb + kTD1 + 128 * (gg & 1) + 64 + 32 * wg;
            tmem_ld16(col, o0);
            tmem_ld16(col + 16, o1);
            tmem_ld_wait();
            const int64_t r0 = t0 + 32 * wg;
            if (j >= p.dv || p.o == nullptr) {  // a padding column, or no output wanted
                tc_fence_before();
                return true;
            }
            __nv_bfloat16* orow = p.o + ((size_t)r0 * p.H + c.h) * p.dv + j;
            const size_t rstride = (size_t)p.H * p.dv;
            if (r0 + 32 <= c.t_end) {
#pragma unroll
                for (int e = 0; e < 16; ++e) orow[e * rstride] = __float2bfloat16_rn(o0[e]);
#pragma unroll
                for (int e = 0; e < 16; ++e) orow[(16 + e) * rstride] = __float2bfloat16_rn(o1[e]);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (r0 + e < c.t_end) orow[e * rstride] = __float2bfloat16_rn(o0[e]);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (r0 + 16 + e < c.t_end) orow[(16 + e) * rstride] = __float2bfloat16_rn(o1[e]);
            }
            tc_fence_before();
            return true;
        };
        for (int k = 0; ok; ++k) {
            const int ci = chain_of(k, cta, G);
            if (ci >= n_chains) break;
            const Chain c = decode_chain(p, ci);
            // S[e] = S[i = 64 wg + e][j] (fp32, registers); padding rows (i >= dk) and
            // columns (j >= dv) hold zeros and are neither read nor written
            float S[64];
            const bool sv = j < p.dv && 64 * wg < p.dk;
            const size_t sbase_el = ((size_t)(c.n * p.H + c.h) * p.dk + 64 * wg) * p.dv + j;
#pragma unroll
            for (int e = 0; e < 64; ++e) S[e] = (p.S0 && sv) ? p.S0[sbase_el + (size_t)e * p.dv] : 0.f;
            // the image block of chunk t (backward pass only)
            auto bimg_of = [&](int t) -> uint8_t* {
                return p.bimg + ((size_t)(__ldg(p.chunk_off + c.n) + t) * p.H + c.h) * bwdtc::kBiBytes;
            };
            // Image stores (no output wanted): the warp's 32 rows of an image part go into one
            // of its two 4 KB stages in the image's own order, and lane 0 hands the 4 KB to a
            // bulk copy, so that no epilogue warp waits for its stores to leave the SM.  Per
            // chunk the parts are S_0 hi (first stage), S_0 lo (second) and Vt (first); a stage
            // is rewritten once lane 0's bulk copies have read it (all but the newest for the
            // second stage and for Vt, all for S_0 hi).
            uint8_t* stg0 = sm + kChStage + warp * 4096;
            uint8_t* stg1 = warp < 4 ? sm + kChAT + warp * 4096 : sm + kChStageB + (warp - 4) * 4096;
            auto stage_free = [&](bool all) {
                if (lane == 0) {
                    if (all) bulk_wait_read0();
                    else bulk_wait_read1();
                }
                __syncwarp();
            };
            auto stage_out = [&](uint8_t* dst, const uint8_t* stg) {
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    bulk_s2g(dst, stg, 4096);
                    bulk_commit();
                }
            };
            // S_0^T of chunk t as bf16 hi + lo: row j of key-channel block wg, the 64 channels
            // in eight 16-byte chunks (padding rows and columns are zeros)
            auto store_ckpt = [&](int t) {
                if constexpr (!kImg) return;
                uint8_t* dst = bimg_of(t) + bwdtc::kBiS + wg * 16384 + (32 * q) * 128;
#pragma unroll
                for (int part = 0; part < 2; ++part) {  // hi, lo
                    uint8_t* stg = part ? stg1 : stg0;
                    stage_free(part == 0);
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        float v8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v8[e] = S[8 * c8 + e];
                        uint4 hi, lo;
                        pk8_hilo(v8, hi, lo);
                        stage_chunk(stg, lane, c8, part ? lo : hi);
                    }
                    stage_out(dst + part * 32768, stg);
                }
            };
            if (c.nch > 0) {
                store_ckpt(0);
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) pk[e] = pack2(S[2 * e], S[2 * e + 1]);
                tmem_st32(tmem + lb + kTS + 32 * wg, pk);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_ready);
            }
            for (int t = 0; t < c.nch; ++t, ++g) {
                const uint32_t st = g & 1, ph = (g >> 1) & 1;
                const int64_t t0 = c.t_begin + (int64_t)t * kC;
                // ---- E1: Vt^T = U^T - X^T for tokens r = 32 wg + e.  U is read from shared
                //      memory while MMA1 runs.
                bool okc = mbar_wait_ab(&fullU[st], ph, p.err, abort);
                if (rec) CH_MARK(8);
                float uu[32];
                if (okc) {
                    const uint8_t* ub = sm + kChU + st * kPkgUBytes + q * kPkgUQ + (lane & 3) * 4;
                    const uint32_t cpos = lane >> 2;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int r = 32 * wg + e;
                        uu[e] = *reinterpret_cast<const float*>(ub + r * 128 + ((cpos ^ (uint32_t)(r & 7)) << 4));
                    }
                }
                okc = okc && mbar_wait_ab(&mma1[st], ph, p.err, abort);
                if (rec) CH_MARK(9);
                if (okc) {
                    tc_fence_after();
                    float x0[16], x1[16];
                    tmem_ld16(tmem + lb + kTD1 + 128 * st + 32 * wg, x0);
                    tmem_ld16(tmem + lb + kTD1 + 128 * st + 32 * wg + 16, x1);
                    tmem_ld_wait();
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        uint32_t hi[8], lo[8];
#pragma unroll
                        for (int e2 = 0; e2 < 8; ++e2) {
                            const float a0 = uu[16 * hf + 2 * e2] - (hf ? x1[2 * e2] : x0[2 * e2]);
                            const float a1 = uu[16 * hf + 2 * e2 + 1] - (hf ? x1[2 * e2 + 1] : x0[2 * e2 + 1]);
                            hi[e2] = pack2(a0, a1);
                            lo[e2] = pack2(a0 - __uint_as_float(hi[e2] << 16),
                                           a1 - __uint_as_float(hi[e2] & 0xffff0000u));
                        }
                        tmem_st8(tmem + lb + kTV + 16 * wg + 8 * hf, hi);
                        tmem_st8(tmem + lb + kTVlo + 16 * wg + 8 * hf, lo);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&vt_ready[st]);
                // backward pass: Vt^T row j into the image block, read back from TMEM while MMA2
                // runs, once every warp's half of the row is there: warps of the first group
                // store the hi rows, the second group the lo rows (64 tokens each, chunk x =
                // tokens 8x .. 8x + 7)
                if constexpr (kImg) {
                    okc = __all_sync(0xffffffffu, okc && mbar_wait_ab(&vt_ready[st], ph, p.err, abort));
                    if (okc) {
                        tc_fence_after();
                        stage_free(false);
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            float f16[16];
                            tmem_ld16(tmem + lb + (wg ? kTVlo : kTV) + 16 * hf, f16);
                            tmem_ld_wait();
#pragma unroll
                            for (int x = 0; x < 4; ++x)
                                stage_chunk(stg0, lane, 4 * hf + x,
                                            make_uint4(__float_as_uint(f16[4 * x]), __float_as_uint(f16[4 * x + 1]),
                                                       __float_as_uint(f16[4 * x + 2]), __float_as_uint(f16[4 * x + 3])));
                        }
                        stage_out(bimg_of(t) + bwdtc::kBiV + wg * 16384 + (32 * q) * 128, stg0);
                    }
                }
                if (rec) CH_MARK(10);
                // ---- E3 of the previous chunk, while MMA2 of this one runs
                if (t > 0 && !store_out(g - 1, t0 - kC, c)) { ok = false; break; }
                if (rec) CH_MARK(13);
                // ---- E2: S^T <- S^T Diag(gamma^C) + dS^T; bf16 copy for the next MMA1
                okc = okc && mbar_wait_ab(&mma2[st], ph, p.err, abort);
                if (rec) CH_MARK(11);
                if (okc) {
                    tc_fence_after();
                    const float* gam = reinterpret_cast<const float*>(sm + kChG + (g % 3) * kPkgGBytes) + 64 * wg;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {  // 32 key channels at a time
                        float d0[16], d1v[16];
                        tmem_ld16(tmem + lb + kTDS + 64 * wg + 32 * hf, d0);
                        tmem_ld16(tmem + lb + kTDS + 64 * wg + 32 * hf + 16, d1v);
                        float4 gv[8];
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4)
                            gv[e4] = *reinterpret_cast<const float4*>(gam + 32 * hf + 4 * e4);
                        tmem_ld_wait();
#pragma unroll
                        for (int qt = 0; qt < 2; ++qt) {
                            uint32_t pk[8];
#pragma unroll
                            for (int e4 = 0; e4 < 4; ++e4) {
                                const float4 g4 = gv[4 * qt + e4];
                                const int e = 32 * hf + 16 * qt + 4 * e4;
                                const float* dd = qt ? d1v : d0;
                                S[e] = fmaf(g4.x, S[e], dd[4 * e4]);
                                S[e + 1] = fmaf(g4.y, S[e + 1], dd[4 * e4 + 1]);
                                S[e + 2] = fmaf(g4.z, S[e + 2], dd[4 * e4 + 2]);
                                S[e + 3] = fmaf(g4.w, S[e + 3], dd[4 * e4 + 3]);
                                pk[2 * e4] = pack2(S[e], S[e + 1]);
                                pk[2 * e4 + 1] = pack2(S[e + 2], S[e + 3]);
                            }
                            tmem_st8(tmem + lb + kTS + 32 * wg + 16 * hf + 8 * qt, pk);
                        }
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && t + 1 < c.nch) mbar_arrive(s_ready);
                if (t + 1 < c.nch) store_ckpt(t + 1);
                if (rec) CH_MARK(12);
                if (t + 1 == c.nch && !store_out(g, t0, c)) { ok = false; break; }
                tc_fence_before();
                if (rec) CH_MARK(14);
            }
            if (!ok) break;
            if (p.S_out && sv) {
#pragma unroll
                for (int e = 0; e < 64; ++e) p.S_out[sbase_el + (size_t)e * p.dv] = S[e];
            }
        }
        if (kImg && lane == 0) bulk_wait0();  // the stages are read and the images written
    }

    chain_sync();
    const bool aborted = s_abort != 0;
    // on an abort, let copies and MMAs still in flight land before leaving
    if (aborted && cpart >= 0) {
        uint64_t* bar = cpart == 0 ? fullPA : cpart == 1 ? fullU : cpart == 2 ? fullKC : fullAT;
        for (int s2 = 0; s2 < 2; ++s2)
            if (last_ph[s2] >= 0) mbar_wait(&bar[s2], last_ph[s2], nullptr);
    }
    if (aborted && tid == kMmaT) {
        mma_commit(drain);  // arrives once every MMA issued so far has completed
        mbar_wait(drain, 0, nullptr);
    }
    tc_fence_before();
    chain_sync();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTCols);
    }
}

}  // namespace
}  // namespace fwdtc
}  // namespace kda
