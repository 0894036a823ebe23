// bwd_item_tc.cu -- the backward's per-chunk work on the sm_103a tensor cores, bf16 problems:
// every (chunk, head) item in parallel, once the chains have written the chunk's start state,
// end gradient, Vt and dVt as operand images (bwd_tc_layout.cuh lists the equations).
//
//   bwd_state_kernel  the products with the chunk's d x d matrices S_0 and dS_C, plus dV, dA,
//                     dM and the solve's reverse (X0 = N^T dM, dbeta1 = diag X0,
//                     dL = -StrictTril(X0 M^T), fp32 on CUDA cores); writes dv and the mid
//                     block
//   bwd_decay_kernel  the decayed intra-chunk products D(dA, K), D(dL, K), D^T(dA, Q) +
//                     D^T(Diag(beta) dL, K) and every remaining gradient (dq, dk, dbeta, dz and
//                     the dA_log partial)
//
// Every product runs transposed, with the 128 key (or value) channels as M = 128 TMEM lanes, so
// that one thread owns one channel over 32 tokens: the gate's cumulative sum and the final
// reverse cumulative sum run in registers.  The decayed products keep every factor finite
// with the sub-tile references of the forward's intra stage (rho_S = G at the middle row of
// 16-token block S): D(X, Y)_ri = sum_S e^{G_r - rho_S} sum_{s in S} X_rs Y_s e^{rho_S - G_s}
// takes one column operand Y e^{rho_{S(s)} - G_s} and one accumulator per block S (only
// blocks S <= R(r) reach token r); D^T likewise with row blocks R and the operand
// Y e^{G_r - rho_{R(r)}}.  Operands that the cancellation in dz is sensitive to are bf16
// hi + lo (three products per contraction).
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

// Optional per-phase cycle counters (debug builds with -DKDA_PHASE_TIMING only): thread 0 and
// the issuing thread of CTA 0 accumulate clock64() deltas between marked points.
#ifdef KDA_PHASE_TIMING
__device__ unsigned long long g_bwd_phase[32];
#define BP_T0() long long bp_t = clock64()
#define BP_MARK(i)                                                                          \
    do {                                                                                    \
        const long long bp_n = clock64();                                                   \
        if (blockIdx.x == 0 && tid == 0)                                                    \
            atomicAdd(&g_bwd_phase[(i)], (unsigned long long)(bp_n - bp_t));                 \
        bp_t = bp_n;                                                                        \
    } while (0)
#else
#define BP_T0() \
    do {        \
    } while (0)
#define BP_MARK(i) \
    do {           \
    } while (0)
#endif

constexpr int kThreads = 256;  // 8 warps; thread 0 also issues every copy and MMA
constexpr float kLog2e = 1.4426950408889634f;

struct ItemParams {
    CUtensorMap tq, tk, tv, tz, tdo;  // [T_total, H, d] bf16, boxes of 64 columns x 1 x 64 rows
    CUtensorMap tdq, tdk, tdz, tdv;   // the outputs, same boxes (TMA stores of full chunks)
    const __nv_bfloat16* beta;
    const __nv_bfloat16* v;           // raw v (the state kernel's Y = V - K+ S_0)
    const float* A_log;
    const int32_t* chunk_off;         // [N + 1] (the forward's plan)
    const int4* chunk_tab;            // per chunk: t0 (lo, hi), sequence, length
    const uint8_t* bimg;              // image blocks [chunks][H]
    uint8_t* mid;                     // mid blocks [chunks][H]
    __nv_bfloat16 *dq, *dkg, *dvg, *dbeta, *dz;
    float* dA_item;                   // [chunks][H]
    unsigned* err;
    float g_min;
    int N, H, dk, dv;
};

__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// barrier over the compute warps that also ANDs a flag over them (so that every compute thread
// takes the same branch afterwards)
__device__ __forceinline__ bool csync_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// element (row, col) of a [rows][128 B] 128-byte-swizzled bf16 tile (col < 64)
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return static_cast<uint32_t>(row * 128 + ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1)));
}
// element (row, ch) of a [2 blocks of 64 channels][rows][128 B] tile
__device__ __forceinline__ uint32_t swz2(int row, int ch, int rows) {
    return static_cast<uint32_t>((ch >> 6) * rows * 128) + swz(row, ch & 63);
}
// Global loads issued where they are written (a plain load may be sunk to its first use,
// which would expose its latency there).
__device__ __forceinline__ float ld_early(const float* q) {
    float r;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(r) : "l"(q));
    return r;
}
__device__ __forceinline__ float4 ld_early4(const float* q) {
    float4 r;
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(q));
    return r;
}
// Sum of v[u] over the 32 lanes of the warp for 16 values at once (transposing halving
// exchange: 16 shuffles); lanes 2u and 2u + 1 end with the sum of value u, returned.
__device__ __forceinline__ float warp_sum16(float (&v)[16], int lane) {
#pragma unroll
    for (int w = 8, o = 16; w >= 1; w >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < w; ++k) {
            const float keep = up ? v[k + w] : v[k], send = up ? v[k] : v[k + w];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

__device__ __forceinline__ float ldbf(const uint8_t* p) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
}
__device__ __forceinline__ uint16_t bfbits(float x) {
    return static_cast<uint16_t>(pack_bf16x2(x, 0.f) & 0xffffu);
}
__device__ __forceinline__ void st_hilo(uint8_t* hi, uint8_t* lo, float x) {
    const uint16_t h = bfbits(x);
    *reinterpret_cast<uint16_t*>(hi) = h;
    *reinterpret_cast<uint16_t*>(lo) = bfbits(x - __uint_as_float(static_cast<uint32_t>(h) << 16));
}

struct Item {
    int chunk, h, L;
    int64_t t0;
};
__device__ __forceinline__ Item decode(const ItemParams& p, int item) {
    Item it;
    it.chunk = item / p.H;
    it.h = item - it.chunk * p.H;
    const int4 e = __ldg(p.chunk_tab + it.chunk);
    it.t0 = (static_cast<int64_t>(e.y) << 32) | static_cast<uint32_t>(e.x);
    it.L = e.w;
    return it;
}

// TMA of a [64 rows][128] bf16 tile (two 64-column blocks) of one tensor at the item's rows
__device__ __forceinline__ void load_tile(const CUtensorMap* m, uint8_t* dst, const Item& it,
                                          uint64_t* bar) {
    tma_load_3d(dst, m, 0, it.h, (int)it.t0, bar);
    tma_load_3d(dst + 8192, m, 64, it.h, (int)it.t0, bar);
}

// Rows [0, L) of a staged [2 blocks][64 rows][128 B] bf16 tile into out [T_total, H, d]: a full
// chunk by two TMA stores from thread 0 (which must later wait for their reads before the tile
// is rewritten), a short one by 16-byte copies of the valid rows (rows past L belong to the
// next sequence).  The tile's writers have fenced and synchronised before.
__device__ __forceinline__ void store_tile(const CUtensorMap* m, const uint8_t* tile,
                                           __nv_bfloat16* out, const Item& it, int H, int d,
                                           int tid) {
    if (it.L == 64) {
        if (tid == 0) {
            tma_store_3d(m, tile, 0, it.h, (int)it.t0);
            tma_store_3d(m, tile + 8192, 64, it.h, (int)it.t0);
            bulk_commit();
        }
        return;
    }
    for (int q = tid; q < it.L * 16; q += 256) {
        const int r = q >> 4, blk = (q >> 3) & 1, c = q & 7;
        if (64 * blk + 8 * c >= d) continue;
        const uint4 v = *reinterpret_cast<const uint4*>(tile + blk * 8192 + r * 128 + ((c ^ (r & 7)) << 4));
        *reinterpret_cast<uint4*>(out + ((size_t)(it.t0 + r) * H + it.h) * d + 64 * blk + 8 * c) = v;
    }
}

// The cumulative gate of channel i over rows [32 wh, 32 wh + 32) in log2 units (rows past L
// add nothing), in G2; tot (smem [128]) carries the first half's total to the second.
__device__ __forceinline__ void gate_scan(const uint8_t* zt, int i, int wh, int L, float scale2,
                                          float gmin2, float* tot, float (&G2)[32]) {
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const int r = 32 * wh + e;
        const float z = ldbf(zt + swz2(r, i, 64));
        const float g = __fdividef(gmin2, 1.f + ex2f(-scale2 * z));
        acc += r < L ? g : 0.f;
        G2[e] = acc;
    }
    if (wh == 0) tot[i] = acc;
    csync();
    if (wh == 1) {
        const float t = tot[i];
#pragma unroll
        for (int e = 0; e < 32; ++e) G2[e] += t;
    }
}

// ======================================================= state kernel ====

// shared memory (1024-aligned offsets)
constexpr uint32_t kSI = 0;          // S_0^T hi, lo (bulk)
constexpr uint32_t kDVI = 65536;     // dVt^T hi, lo (bulk); batch 3: dS_C^T hi
constexpr uint32_t kVI = 98304;      // Vt^T hi, lo (bulk)
constexpr uint32_t kYI = 131072;     // z tile, then Y^T hi (rows j); batch 3: dS_C^T lo
constexpr uint32_t kDVO = 147456;    // k tile, then Y^T lo (rows j); batch 3: dS_C^T lo
constexpr uint32_t kDOt = 163840;    // dO tile; after batch 2: dM fp32 [64][64]
constexpr uint32_t kRX = 180224;     // K+ (K-major rows s) + M (rows r); after batch 1: dV^T
                                     // (one bf16, rows j); after batch 2: X0^T, N^T fp32
constexpr uint32_t kVt = 212992;     // v tile
constexpr uint32_t kMisc = 229376;   // beta [64], tot [128], glast [128], dbeta1 halves [2][64]
constexpr uint32_t kSBars = kMisc + 1792;
constexpr uint32_t kStateSmem = kSBars + 128 + 1024;
static_assert(kStateSmem <= 232448, "state kernel exceeds the shared-memory limit");
// TMEM columns: dV^T [0, 64), (K+ S_0)^T [64, 128), S_0 dO^T [128, 192), S_0 dV^T [192, 256),
// dA^T (lanes 0..63) [256, 320), dM^T (lanes 64..127) [320, 384), dS_C Vt^T [384, 448), in
// batch 3 dS_C S_0^T [0, 128) (only its diagonal is read), then the solve's reverse:
// Z1^T [128, 192), Z1^T bf16 hi [192, 224), lo [224, 256), dL^T [256, 320)
constexpr uint32_t kTCols = 512;

// The state kernel: one CTA of 256 threads per SM walks items (chunk, head); thread 0 also
// issues every copy and MMA, each right after the barrier that makes its operands ready.
__global__ void __launch_bounds__(kThreads, 1) bwd_state_kernel(const __grid_constant__ ItemParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kSBars);
    uint64_t* fullIn = bars + 0;  // z, k, v tiles
    uint64_t* fullS = bars + 1;
    uint64_t* fullV = bars + 2;
    uint64_t* fullDO = bars + 3;
    uint64_t* fullDS = bars + 4;
    uint64_t* mma1 = bars + 5;
    uint64_t* mma2 = bars + 6;
    uint64_t* mma3 = bars + 7;
    uint64_t* mma4 = bars + 8;  // Z1^T = M dM^T
    uint64_t* mma5 = bars + 9;  // dL^T = (N^T Z1)^T
    uint64_t* drain = bars + 10;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 11);
    float* sBeta = reinterpret_cast<float*>(sm + kMisc);
    float* sTot = sBeta + 64;
    float* sGlast = sTot + 128;
    float* sDb1 = sGlast + 128;  // [2][64]: dbeta1 halves
    __shared__ int s_abort;
    volatile int* abort = &s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool iss = tid == 0;
    if (tid == 0) {
        for (int i = 0; i < 11; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        s_abort = 0;
    }
    if (warp == 0) tmem_alloc(tmem_slot, kTCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n_items = __ldg(p.chunk_off + p.N) * p.H;

    constexpr uint32_t idZ = idesc_bf16(128, 64, false, true);    // M x dM^T, Z1^T x N
    constexpr uint32_t idV = idesc_bf16(128, 64, false, true);    // dVt^T x M
    constexpr uint32_t idY = idesc_bf16(128, 64, false, false);   // S_0^T x K+^T
    constexpr uint32_t idMN = idesc_bf16(128, 64, true, false);   // S_0 x dO^T, [Vt; Y] x dO^T
    constexpr uint32_t idMM = idesc_bf16(128, 64, true, true);    // MN-major A and B, N = 64
    constexpr uint32_t idD = idesc_bf16(128, 128, true, true);    // dS_C x S_0^T

    const int wq = warp & 3, wh = warp >> 2;
    const int ch = 32 * wq + lane;  // TMEM lane: a key or value channel (or a token s)
    const uint32_t lb = static_cast<uint32_t>(32 * wq) << 16;
    // thread 0: the phase each copy barrier (fullIn, fullS, fullV, fullDO, fullDS) has in
    // flight, or -1
    int pend[5] = {-1, -1, -1, -1, -1};
    // z, k, dVt and Vt of an item: issued while the previous item finishes (its batch 3 has
    // read their places), or at the item's start for a CTA's first item
    auto issue_early = [&](const Item& e, const uint8_t* eblk, uint32_t eph) {
        pend[0] = (int)eph;
        mbar_expect_tx(fullIn, 32768);
        load_tile(&p.tz, sm + kYI, e, fullIn);
        load_tile(&p.tk, sm + kDVO, e, fullIn);
        pend[2] = (int)eph;
        mbar_expect_tx(fullV, 65536);
        bulk_g2s(sm + kDVI, eblk + kBiDV, 32768, fullV);
        bulk_g2s(sm + kVI, eblk + kBiV, 32768, fullV);
    };
    bool early_done = false;  // thread 0: this item's early copies are issued
    bool ok = true;
    uint32_t iter = 0;
    BP_T0();
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++iter) {
        const Item it = decode(p, item);
        const uint32_t ph = iter & 1;
        const uint8_t* blk = p.bimg + (size_t)item * kBiBytes;
        if (iss) {
            if (!early_done) issue_early(it, blk, ph);
            early_done = false;
            bulk_wait_read0();  // the previous item's dv store has read the v tile's place
            pend[1] = (int)ph;  // S_0 (read by batch 1) and v (epilogue 1)
            mbar_expect_tx(fullS, 65536 + 16384);
            bulk_g2s(sm + kSI, blk + kBiS, 65536, fullS);
            load_tile(&p.tv, sm + kVt, it, fullS);
            pend[3] = (int)ph;
            mbar_expect_tx(fullDO, 16384);
            load_tile(&p.tdo, sm + kDOt, it, fullDO);
            const int nx = item + gridDim.x;  // the next item's inputs into L2
            if (nx < n_items) {
                const Item in = decode(p, nx);
                l2_prefetch(p.bimg + (size_t)nx * kBiBytes, kBiBytes);
                for (int b = 0; b < 2; ++b) {
                    tma_prefetch_3d(&p.tz, 64 * b, in.h, (int)in.t0);
                    tma_prefetch_3d(&p.tk, 64 * b, in.h, (int)in.t0);
                    tma_prefetch_3d(&p.tv, 64 * b, in.h, (int)in.t0);
                    tma_prefetch_3d(&p.tdo, 64 * b, in.h, (int)in.t0);
                }
            }
        }
        const float eA = expf(__ldg(p.A_log + it.h));
        const float scale2 = eA * kLog2e, gmin2 = p.g_min * kLog2e;
        uint8_t* mid = p.mid + (size_t)item * kMdBytes;
        const float* Ng = reinterpret_cast<const float*>(blk + kBiN);
        if (tid < 64)
            sBeta[tid] = tid < it.L ? __bfloat162float(p.beta[(size_t)(it.t0 + tid) * p.H + it.h]) : 0.f;
        // this thread's 16 entries of N (row tid / 4) for the M image, in flight during the gate
        float4 nrow[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) nrow[x] = ld_early4(Ng + (tid >> 2) * 64 + 16 * (tid & 3) + 4 * x);
        ok = ok && mbar_wait_ab(fullIn, ph, p.err, abort);
        if (iss && ok) pend[0] = -1;
        BP_MARK(0);
        float G2[32];
        if (ok) {
            gate_scan(sm + kYI, ch, wh, it.L, scale2, gmin2, sTot, G2);
            if (wh == 1) sGlast[ch] = G2[31];
            // K+ = Gamma*K, rows s of this half (K-major [2 blocks][64 rows][128 B]); every k
            // is read before the first store
            float kk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e)
                kk[e] = 32 * wh + e < it.L ? ldbf(sm + kDVO + swz2(32 * wh + e, ch, 64)) : 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e)
                *reinterpret_cast<uint16_t*>(sm + kRX + swz2(32 * wh + e, ch, 64)) = bfbits(ex2f(G2[e]) * kk[e]);
            // M = N Diag(beta): row r, 16 columns per thread (MN-major rows r)
            const int r = tid >> 2, cq = tid & 3;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const float4 n0 = nrow[2 * hf], n1 = nrow[2 * hf + 1];
                const float* b = sBeta + 16 * cq + 8 * hf;
                const float v8[8] = {n0.x * b[0], n0.y * b[1], n0.z * b[2], n0.w * b[3],
                                     n1.x * b[4], n1.y * b[5], n1.z * b[6], n1.w * b[7]};
                *reinterpret_cast<uint4*>(sm + kRX + 16384 + r * 128 + (((2 * cq + hf) ^ (r & 7)) << 4)) = pk8(v8);
            }
        } else {
            csync();  // the gate scan's barrier
        }
        fence_async_smem();
        ok = csync_and(ok);
        BP_MARK(1);
        if (iss && ok) {
            ok = mbar_wait_ab(fullS, ph, p.err, abort) && mbar_wait_ab(fullV, ph, p.err, abort) &&
                 mbar_wait_ab(fullDO, ph, p.err, abort);
            if (ok) {
                pend[1] = pend[2] = pend[3] = -1;
                tc_fence_after();
                // batch 1 -----------------------------------------------------------
                // dV^T = dVt^T M: A = dVt^T rows j hi, lo (K = 64 tokens, K-major), B = M rows r
                // (MN-major)
                const uint64_t dMd = sdesc_sw128(sb + kRX + 16384, 8192, 1024);
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const uint64_t dA = sdesc_sw128(sb + kDVI + 16384 * x, 0, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + 0, dA + ((kk * 32) >> 4), dMd + ((kk * 2048) >> 4), idV,
                                 (x | kk) != 0);
                }
                // (K+ S_0)^T = S_0^T K+^T: A = S_0^T hi rows j (K = 128 key channels, K-major),
                // B = K+ rows s (K-major)
                {
                    const uint64_t dA = sdesc_sw128(sb + kSI, 0, 1024);
                    const uint64_t dB = sdesc_sw128(sb + kRX, 0, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tmem + 64, dA + ((((kk >> 2) * 16384) + (kk & 3) * 32) >> 4),
                                 dB + ((((kk >> 2) * 8192) + (kk & 3) * 32) >> 4), idY, kk > 0);
                }
                // S_0 dO^T: A = S_0 hi, lo (M = key channels, MN-major rows j), B = dO rows r
                // (K-major; K = 128 value channels)
                {
                    const uint64_t dB = sdesc_sw128(sb + kDOt, 0, 1024);
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        const uint64_t dA = sdesc_sw128(sb + kSI + 32768 * x, 16384, 1024);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_bf16(tmem + 128, dA + ((kk * 2048) >> 4),
                                     dB + ((((kk >> 2) * 8192) + (kk & 3) * 32) >> 4), idMN,
                                     (x | kk) != 0);
                    }
                }
                mma_commit(mma1);
            }
        }
        // ---- epilogue 1
        ok = ok && mbar_wait_ab(mma1, ph, p.err, abort);
        BP_MARK(2);
        if (ok) {
            tc_fence_after();
            // dV^T and Y^T: lane = value channel j, columns s of this half
            const int j = ch;
            float a0[16], a1[16], y0[16], y1[16];
            tmem_ld16(tmem + lb + 0 + 32 * wh, a0);
            tmem_ld16(tmem + lb + 16 + 32 * wh, a1);
            tmem_ld16(tmem + lb + 64 + 32 * wh, y0);
            tmem_ld16(tmem + lb + 80 + 32 * wh, y1);
            // v of this lane's value channel for the tokens of this half, all before the stores
            // below (a load after a shared-memory store may not be hoisted above it)
            float vv[32];
#pragma unroll
            for (int u = 0; u < 32; ++u)
                vv[u] = 32 * wh + u < it.L ? ldbf(sm + kVt + swz2(32 * wh + u, j, 64)) : 0.f;
            tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                float dv8[8], y8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int u = 8 * x + e;  // token s = 32 wh + u
                    const int s = 32 * wh + u;
                    dv8[e] = u < 16 ? a0[u] : a1[u - 16];
                    y8[e] = vv[u] - (u < 16 ? y0[u] : y1[u - 16]);
                    // dv replaces v (staged for the output store)
                    *reinterpret_cast<uint16_t*>(sm + kVt + swz2(s, j, 64)) = bfbits(dv8[e]);
                }
                const uint32_t off = (uint32_t)(j * 128 + (((4 * wh + x) ^ (j & 7)) << 4));
                *reinterpret_cast<uint4*>(sm + kRX + off) = pk8(dv8);
                uint4 yh, yl;
                pk8_hilo(y8, yh, yl);
                *reinterpret_cast<uint4*>(sm + kYI + off) = yh;
                *reinterpret_cast<uint4*>(sm + kDVO + off) = yl;
            }
            // pQ = Gamma*(S_0 dO^T): lane = key channel i, columns r of this half
            float q0[16], q1[16];
            tmem_ld16(tmem + lb + 128 + 32 * wh, q0);
            tmem_ld16(tmem + lb + 144 + 32 * wh, q1);
            tmem_ld_wait();
            float* pq = reinterpret_cast<float*>(mid + kMdQ) + ch;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                pq[(32 * wh + u) * 128] = ex2f(G2[u]) * (u < 16 ? q0[u] : q1[u - 16]);
        }
        tc_fence_before();
        fence_async_smem();
        ok = csync_and(ok);
        BP_MARK(3);
        if (iss && ok) {
            tc_fence_after();
            // batch 2 ---------------------------------------------------------------
            // S_0 dV^T: A = S_0 hi, lo (MN-major), B = dV^T rows j (MN-major, N = 64 tokens)
            {
                const uint64_t dB = sdesc_sw128(sb + kRX, 8192, 1024);
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const uint64_t dA = sdesc_sw128(sb + kSI + 32768 * x, 16384, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tmem + 192, dA + ((kk * 2048) >> 4), dB + ((kk * 2048) >> 4), idMM,
                                 (x | kk) != 0);
                }
            }
            // [Vt; Y] dO^T: A = [Vt^T rows j | Y^T rows j] as an MN-major M = 128 operand (M
            // blocks 32 KB apart: [Vt_hi; Y_hi] and [Vt_lo; Y_lo]); the lanes 0..63 hold
            // dA^T = Vt dO^T (lanes 64..127 are not read)
            {
                const uint64_t dB = sdesc_sw128(sb + kDOt, 0, 1024);
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const uint64_t dA = sdesc_sw128(sb + kVI + 16384 * x, 32768, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tmem + 256, dA + ((kk * 2048) >> 4),
                                 dB + ((((kk >> 2) * 8192) + (kk & 3) * 32) >> 4), idMN,
                                 (x | kk) != 0);
                }
            }
            // [Vt; Y] dVt^T, hi x hi + hi x lo + lo x hi: lanes 64..127 hold dM^T = Y dVt^T
#pragma unroll
            for (int x = 0; x < 3; ++x) {
                const uint64_t dA = sdesc_sw128(sb + kVI + (x == 2 ? 16384 : 0), 32768, 1024);
                const uint64_t dB = sdesc_sw128(sb + kDVI + (x == 1 ? 16384 : 0), 8192, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + 320, dA + ((kk * 2048) >> 4), dB + ((kk * 2048) >> 4), idMM,
                             (x | kk) != 0);
            }
            mma_commit(mma2);
            if (it.L == 64) store_tile(&p.tdv, sm + kVt, p.dvg, it, p.H, p.dv, tid);
        }
        // ---- epilogue 2
        float nc[32];  // lanes 64 + s: N[r][s] for r of this half (dbeta1 = sum_r N[r][s] dM[r][s])
        if (wq >= 2) {
#pragma unroll
            for (int u = 0; u < 32; ++u) nc[u] = ld_early(Ng + (32 * wh + u) * 64 + (ch - 64));
        }
        ok = ok && mbar_wait_ab(mma2, ph, p.err, abort);
        BP_MARK(4);
        if (iss && ok) {
            // dVt and Y are consumed: dS_C^T hi, lo into their place
            pend[4] = (int)ph;
            mbar_expect_tx(fullDS, 65536);
            bulk_g2s(sm + kDVI, blk + kBiDS, 32768, fullDS);
            bulk_g2s(sm + kYI, blk + kBiDS + 32768, 32768, fullDS);
        }
        if (ok) {
            tc_fence_after();
            // pP = -Gamma*(S_0 dV^T): lane = key channel
            float* pp = reinterpret_cast<float*>(mid + kMdP) + ch;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float b16[16];
                tmem_ld16(tmem + lb + 192 + 32 * wh + 16 * hf, b16);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int u = 16 * hf + e;
                    pp[(32 * wh + u) * 128] = -ex2f(G2[u]) * b16[e];
                }
            }
            if (wq < 2) {
                // dA^T (lane s): row s of the dA image, columns c = 63 - r (hi, lo)
                const int s = ch;
                float d0[16], d1[16];
                tmem_ld16(tmem + lb + 256 + 32 * wh, d0);
                tmem_ld16(tmem + lb + 272 + 32 * wh, d1);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float v8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int u = 31 - 8 * k - e;  // r = 32 wh + u
                        const int r = 32 * wh + u;
                        const float d = u < 16 ? d0[u] : d1[u - 16];
                        v8[e] = (r >= s && r < it.L) ? d : 0.f;
                    }
                    uint4 hi, lo;
                    pk8_hilo(v8, hi, lo);
                    const uint32_t off = (uint32_t)(s * 128 + (((4 - 4 * wh + k) ^ (s & 7)) << 4));
                    *reinterpret_cast<uint4*>(mid + kMdA + off) = hi;
                    *reinterpret_cast<uint4*>(mid + kMdA + 8192 + off) = lo;
                }
            } else {
                // dM^T (lane 64 + s): row s of the dM^T image (r contiguous, hi and lo) and this
                // half's part of dbeta1_s = sum_r N[r][s] dM[r][s]
                const int s = ch - 64;
                float d0[16], d1[16];
                tmem_ld16(tmem + lb + 320 + 32 * wh, d0);
                tmem_ld16(tmem + lb + 336 + 32 * wh, d1);
                tmem_ld_wait();
                float db = 0.f;
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    float v8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int u = 8 * x + e;
                        v8[e] = u < 16 ? d0[u] : d1[u - 16];
                        db = fmaf(nc[u], v8[e], db);
                    }
                    uint4 hi, lo;
                    pk8_hilo(v8, hi, lo);
                    const uint32_t off = (uint32_t)(s * 128 + (((4 * wh + x) ^ (s & 7)) << 4));
                    *reinterpret_cast<uint4*>(sm + kDOt + off) = hi;
                    *reinterpret_cast<uint4*>(sm + kDOt + 8192 + off) = lo;
                }
                sDb1[64 * wh + s] = db;
            }
        }
        tc_fence_before();
        ok = csync_and(ok);
        BP_MARK(5);
        if (iss && ok) {
            ok = mbar_wait_ab(fullDS, ph, p.err, abort);
            if (ok) {
                pend[4] = -1;
                tc_fence_after();
                // batch 3 -----------------------------------------------------------
                // dS_C Vt^T: A = dS_C (MN-major rows j), B = Vt^T rows j (MN-major); hi x hi,
                // hi x lo, lo x hi
#pragma unroll
                for (int x = 0; x < 3; ++x) {
                    const uint64_t dA = sdesc_sw128(sb + (x == 2 ? kYI : kDVI), 16384, 1024);
                    const uint64_t dB = sdesc_sw128(sb + kVI + (x == 1 ? 16384 : 0), 8192, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tmem + 384, dA + ((kk * 2048) >> 4), dB + ((kk * 2048) >> 4), idMM,
                                 (x | kk) != 0);
                }
                // dS_C S_0^T (N = 128 key channels; its diagonal is rs): B = S_0^T rows j, MN-major
#pragma unroll
                for (int x = 0; x < 3; ++x) {
                    const uint64_t dA = sdesc_sw128(sb + (x == 2 ? kYI : kDVI), 16384, 1024);
                    const uint64_t dB = sdesc_sw128(sb + kSI + (x == 1 ? 32768 : 0), 16384, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tmem + 0, dA + ((kk * 2048) >> 4), dB + ((kk * 2048) >> 4), idD,
                                 (x | kk) != 0);
                }
                mma_commit(mma3);
            }
        }
        if (tid < 64 && ok) reinterpret_cast<float*>(mid + kMdB)[tid] = sDb1[tid] + sDb1[64 + tid];
        // this thread's 16 entries of N (row tid / 4) for the solve's operand images
#pragma unroll
        for (int x = 0; x < 4; ++x) nrow[x] = ld_early4(Ng + (tid >> 2) * 64 + 16 * (tid & 3) + 4 * x);
        BP_MARK(6);
        // ---- epilogue 3: pE = (gamma^C/Gamma)*(dS_C Vt^T) and rs = diag(dS_C S_0^T)
        ok = ok && mbar_wait_ab(mma3, ph, p.err, abort);
        BP_MARK(7);
        // batch 3 has read the dS_C, Vt and Y places: the next item's z, k, dVt and Vt go in
        // now, so that they land during this item's last phases
        if (iss && ok) {
            const int nx = item + (int)gridDim.x;
            if (nx < n_items) {
                issue_early(decode(p, nx), p.bimg + (size_t)nx * kBiBytes, ph ^ 1u);
                early_done = true;
            }
        }
        if (ok) {
            tc_fence_after();
            const float gl = sGlast[ch];
            float* pe = reinterpret_cast<float*>(mid + kMdE) + ch;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float c16[16];
                tmem_ld16(tmem + lb + 384 + 32 * wh + 16 * hf, c16);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int u = 16 * hf + e;
                    pe[(32 * wh + u) * 128] = ex2f(gl - G2[u]) * c16[e];
                }
            }
            if (wh == 0) {  // lane i reads column i of its warp's 32 columns
                float d0[16], d1[16];
                tmem_ld16(tmem + lb + 32 * wq, d0);
                tmem_ld16(tmem + lb + 32 * wq + 16, d1);
                tmem_ld_wait();
                float rs = 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    rs = (lane == e) ? d0[e] : rs;
                    rs = (lane == 16 + e) ? d1[e] : rs;
                }
                reinterpret_cast<float*>(mid + kMdRs)[ch] = rs;
            }
        }
        // ---- the solve's reverse on the tensor cores: Z1 = dM M^T, dL = -StrictTril(N^T Z1)
        //      (= -StrictTril(X0 M^T) with X0 = N^T dM), both hi x hi + hi x lo + lo x hi.
        //      Operand images in the S_0 region (batch 3 has read it): M rows i hi, lo
        //      [0, 16 KB), N rows r hi, lo [16, 32 KB), both with the 64 columns contiguous
        if (ok) {
            const int r = tid >> 2, cq = tid & 3;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const float4 n0 = nrow[2 * hf], n1 = nrow[2 * hf + 1];
                const float* b = sBeta + 16 * cq + 8 * hf;
                const float nv[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
                float mv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mv[e] = nv[e] * b[e];
                uint4 nh, nl, mh, ml;
                pk8_hilo(nv, nh, nl);
                pk8_hilo(mv, mh, ml);
                const uint32_t off = (uint32_t)(r * 128 + (((2 * cq + hf) ^ (r & 7)) << 4));
                *reinterpret_cast<uint4*>(sm + kSI + off) = mh;
                *reinterpret_cast<uint4*>(sm + kSI + 8192 + off) = ml;
                *reinterpret_cast<uint4*>(sm + kSI + 16384 + off) = nh;
                *reinterpret_cast<uint4*>(sm + kSI + 24576 + off) = nl;
            }
        }
        fence_async_smem();
        tc_fence_before();
        ok = csync_and(ok);
        if (iss && ok) {
            tc_fence_after();
            // Z1^T = M dM^T: A = M rows i (K-major; rows 64..127 are not read back),
            // B = dM^T rows s (MN-major, N = 64 tokens r)
#pragma unroll
            for (int x = 0; x < 3; ++x) {
                const uint64_t dA = sdesc_sw128(sb + kSI + (x == 2 ? 8192 : 0), 0, 1024);
                const uint64_t dB = sdesc_sw128(sb + kDOt + (x == 1 ? 8192 : 0), 8192, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + 128, dA + ((kk * 32) >> 4), dB + ((kk * 2048) >> 4), idZ,
                             (x | kk) != 0);
            }
            mma_commit(mma4);
        }
        ok = ok && mbar_wait_ab(mma4, ph, p.err, abort);
        if (ok && wq < 2) {  // lanes i < 64: Z1^T -> bf16 hi + lo into TMEM (tokens in pairs)
            tc_fence_after();
            float z0[16], z1[16];
            tmem_ld16(tmem + lb + 128 + 32 * wh, z0);
            tmem_ld16(tmem + lb + 144 + 32 * wh, z1);
            tmem_ld_wait();
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float a0 = e < 8 ? z0[2 * e] : z1[2 * e - 16];
                const float a1 = e < 8 ? z0[2 * e + 1] : z1[2 * e - 15];
                hi[e] = pack_bf16x2(a0, a1);
                lo[e] = pack_bf16x2(a0 - __uint_as_float(hi[e] << 16), a1 - __uint_as_float(hi[e] & 0xffff0000u));
            }
            tmem_st16(tmem + lb + 192 + 16 * wh, hi);
            tmem_st16(tmem + lb + 224 + 16 * wh, lo);
            tmem_st_wait();
        }
        tc_fence_before();
        ok = csync_and(ok);
        if (iss && ok) {
            tc_fence_after();
            // dL^T = Z1^T N: A = Z1^T from TMEM (K = 64 tokens r), B = N rows r (MN-major)
#pragma unroll
            for (int x = 0; x < 3; ++x) {
                const uint64_t dB = sdesc_sw128(sb + kSI + 16384 + (x == 1 ? 8192 : 0), 8192, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ts(tmem + 256, tmem + (x == 2 ? 224 : 192) + 8 * kk, dB + ((kk * 2048) >> 4),
                                idZ, (x | kk) != 0);
            }
            mma_commit(mma5);
        }
        ok = ok && mbar_wait_ab(mma5, ph, p.err, abort);
        if (ok && wq < 2) {
            // lane i: row i of the dL image, columns c = 63 - r' (hi, lo): dL[r'][i] = -D[i][r']
            // for i < r' < L
            tc_fence_after();
            const int i = ch;
            float d0[16], d1[16];
            tmem_ld16(tmem + lb + 256 + 32 * wh, d0);
            tmem_ld16(tmem + lb + 272 + 32 * wh, d1);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float v8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int u = 31 - 8 * k - e;  // r' = 32 wh + u
                    const int rr = 32 * wh + u;
                    const float d = u < 16 ? d0[u] : d1[u - 16];
                    v8[e] = (i < rr && rr < it.L) ? -d : 0.f;
                }
                uint4 hi, lo;
                pk8_hilo(v8, hi, lo);
                const uint32_t off = (uint32_t)(i * 128 + (((4 - 4 * wh + k) ^ (i & 7)) << 4));
                *reinterpret_cast<uint4*>(mid + kMdL + off) = hi;
                *reinterpret_cast<uint4*>(mid + kMdL + 8192 + off) = lo;
            }
        }
        if (ok && it.L < 64) store_tile(&p.tdv, sm + kVt, p.dvg, it, p.H, p.dv, tid);
        tc_fence_before();
        fence_async_smem();  // the next item's copies overwrite what was written here
        ok = csync_and(ok);
        BP_MARK(8);
        if (!ok) break;
    }

    __syncthreads();
    if (s_abort && iss) {
        // let the copies and MMAs still in flight land before the CTA leaves
        for (int b = 0; b < 5; ++b)
            if (pend[b] >= 0) mbar_wait(&bars[b], (uint32_t)pend[b], nullptr);
        mma_commit(drain);
        mbar_wait(drain, 0, nullptr);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTCols);
    }
}

// ======================================================= decay kernel ====

constexpr uint32_t kQt = 0, kKt = 16384, kZt = 32768;
constexpr uint32_t kKT = 49152;   // K~ = K e^{rho_S(s) - G_s}, rows s: hi, lo (+16384)
constexpr uint32_t kQH = 81920;   // Q^ = Q e^{G_r - rho_R(r)}, rows 63 - r: hi, lo
constexpr uint32_t kKB = 114688;  // K^b = beta K e^{G_r - rho_R(r)}, rows 63 - r: hi, lo
constexpr uint32_t kDAi = 147456; // dA image hi, lo (+8192)
constexpr uint32_t kDLi = 163840; // dL image hi, lo (+8192)
constexpr uint32_t kDMisc = 180224;  // beta [64], tot [128], glast [128], rho [4][128],
                                     // last [2][128], dbeta [4][64], red [8]
constexpr uint32_t kDG = kDMisc + 6144;  // G (log2 units) fp32 [64 rows][128 channels]
constexpr uint32_t kDBars = kDG + 32768;
constexpr uint32_t kDecaySmem = kDBars + 128 + 1024;
static_assert(kDecaySmem <= 232448, "decay kernel exceeds the shared-memory limit");
// TMEM: D(dA, K) per block S at [kOffS[S], + 64 - 16 S), D(dL, K) at 160 + the same, and
// D^T per row block R at [320 + kOffR[R], + 16 (R + 1))
__device__ __constant__ int kOffS[4] = {0, 64, 112, 144};
__device__ __constant__ int kOffR[4] = {0, 16, 48, 96};

__global__ void __launch_bounds__(kThreads, 1) bwd_decay_kernel(const __grid_constant__ ItemParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kDBars);
    uint64_t* fullIn = bars + 0;
    uint64_t* fullX = bars + 1;
    uint64_t* mma1 = bars + 2;
    uint64_t* drain = bars + 3;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4);
    float* sBeta = reinterpret_cast<float*>(sm + kDMisc);
    float* sTot = sBeta + 64;
    float* sGlast = sTot + 128;
    float* sRho = sGlast + 128;   // [4][128]
    float* sLast = sRho + 512;    // [2][128]
    float* sDb = sLast + 256;     // [4][64]
    float* sRed = sDb + 256;      // [8]
    __shared__ int s_abort;
    volatile int* abort = &s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool iss = tid == 0;
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        s_abort = 0;
    }
    if (warp == 0) tmem_alloc(tmem_slot, kTCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n_items = __ldg(p.chunk_off + p.N) * p.H;

    const int wq = warp & 3, wh = warp >> 2;
    const int ch = 32 * wq + lane;  // key channel i = TMEM lane
    const uint32_t lb = static_cast<uint32_t>(32 * wq) << 16;
    uint32_t inflight = 0, inflight_ph = 0;
    bool ok = true;
    uint32_t iter = 0;
    BP_T0();
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++iter) {
        const Item it = decode(p, item);
        const uint32_t ph = iter & 1;
        const uint8_t* mid = p.mid + (size_t)item * kMdBytes;
        if (iss) {
            bulk_wait_read0();  // the previous item's output stores have read the stack region
            inflight = 0x3u;
            inflight_ph = ph;
            mbar_expect_tx(fullIn, 49152);
            load_tile(&p.tq, sm + kQt, it, fullIn);
            load_tile(&p.tk, sm + kKt, it, fullIn);
            load_tile(&p.tz, sm + kZt, it, fullIn);
            mbar_expect_tx(fullX, 32768);
            bulk_g2s(sm + kDAi, mid + kMdA, 32768, fullX);  // dA then dL images (adjacent)
            const int nx = item + gridDim.x;  // the next item's inputs into L2
            if (nx < n_items) {
                const Item in = decode(p, nx);
                l2_prefetch(p.mid + (size_t)nx * kMdBytes, kMdBytes);
                for (int b = 0; b < 2; ++b) {
                    tma_prefetch_3d(&p.tq, 64 * b, in.h, (int)in.t0);
                    tma_prefetch_3d(&p.tk, 64 * b, in.h, (int)in.t0);
                    tma_prefetch_3d(&p.tz, 64 * b, in.h, (int)in.t0);
                }
            }
        }
        const float eA = expf(__ldg(p.A_log + it.h));
        const float scale2 = eA * kLog2e, gmin2 = p.g_min * kLog2e;
        if (tid < 64)
            sBeta[tid] = tid < it.L ? __bfloat162float(p.beta[(size_t)(it.t0 + tid) * p.H + it.h]) : 0.f;
        ok = ok && mbar_wait_ab(fullIn, ph, p.err, abort);
        BP_MARK(10);
        float G2[32];
        if (ok) {
            gate_scan(sm + kZt, ch, wh, it.L, scale2, gmin2, sTot, G2);
            if (wh == 1) sGlast[ch] = G2[31];
            sRho[(2 * wh) * 128 + ch] = G2[8];
            sRho[(2 * wh + 1) * 128 + ch] = G2[24];
            float* gs = reinterpret_cast<float*>(sm + kDG) + 32 * wh * 128 + ch;
#pragma unroll
            for (int e = 0; e < 32; ++e) gs[e * 128] = G2[e];
        } else {
            csync();
        }
        csync();
        BP_MARK(11);
        if (ok) {
            // K~ (rows s), Q^ and K^b (rows 63 - r): thread = (row, 8 channels), four of them,
            // 16-byte chunks in and out
            const float* gs = reinterpret_cast<const float*>(sm + kDG);
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int u = tid + 256 * x, r = u >> 4, c = u & 15, blk = c >> 3, cc = c & 7;
                const int c0 = 8 * c;
                const uint32_t oin = blk * 8192 + r * 128 + ((cc ^ (r & 7)) << 4);
                const int rv = 63 - r;
                const uint32_t orv = blk * 8192 + rv * 128 + ((cc ^ (rv & 7)) << 4);
                float kv[8], qv[8];
                if (r < it.L) {
                    ld8(sm + kKt + oin, kv);
                    ld8(sm + kQt + oin, qv);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) { kv[e] = 0.f; qv[e] = 0.f; }
                }
                const float4 g0 = *reinterpret_cast<const float4*>(gs + r * 128 + c0);
                const float4 g1 = *reinterpret_cast<const float4*>(gs + r * 128 + c0 + 4);
                const float* rh = sRho + (r >> 4) * 128 + c0;
                const float4 h0 = *reinterpret_cast<const float4*>(rh);
                const float4 h1 = *reinterpret_cast<const float4*>(rh + 4);
                const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
                const float b = sBeta[r];
                float kt[8], qh[8], kb[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float up = ex2f(gv[e] - hv[e]), dn = ex2f(hv[e] - gv[e]);
                    kt[e] = kv[e] * dn;
                    qh[e] = qv[e] * up;
                    kb[e] = b * kv[e] * up;
                }
                uint4 hi, lo;
                pk8_hilo(kt, hi, lo);
                *reinterpret_cast<uint4*>(sm + kKT + oin) = hi;
                *reinterpret_cast<uint4*>(sm + kKT + 16384 + oin) = lo;
                pk8_hilo(qh, hi, lo);
                *reinterpret_cast<uint4*>(sm + kQH + orv) = hi;
                *reinterpret_cast<uint4*>(sm + kQH + 16384 + orv) = lo;
                pk8_hilo(kb, hi, lo);
                *reinterpret_cast<uint4*>(sm + kKB + orv) = hi;
                *reinterpret_cast<uint4*>(sm + kKB + 16384 + orv) = lo;
            }
        }
        fence_async_smem();
        ok = csync_and(ok);
        BP_MARK(12);
        if (iss && ok) {
            ok = mbar_wait_ab(fullX, ph, p.err, abort);
            if (ok) {
                tc_fence_after();
                // D(X, K) per block S: A = K~^T rows s in S (MN-major, M = 128 key channels),
                // B = X^T rows s in S with columns c = 63 - r < 64 - 16 S (MN-major,
                // N = 64 - 16 S); hi x hi + hi x lo + lo x hi
#pragma unroll
                for (int S = 0; S < 4; ++S) {
                    const uint32_t idS = idesc_bf16(128, 64 - 16 * S, true, true);
                    const uint64_t kh = sdesc_sw128(sb + kKT + 2048 * S, 8192, 1024);
                    const uint64_t kl = sdesc_sw128(sb + kKT + 16384 + 2048 * S, 8192, 1024);
#pragma unroll
                    for (int xs = 0; xs < 2; ++xs) {  // 0: dA, 1: dL
                        const uint32_t xb = sb + (xs ? kDLi : kDAi) + 2048 * S;
                        const uint64_t xh = sdesc_sw128(xb, 8192, 1024);
                        const uint64_t xl = sdesc_sw128(xb + 8192, 8192, 1024);
                        const uint32_t d = tmem + 160 * xs + kOffS[S];
                        mma_bf16(d, kh, xh, idS, 0);
                        mma_bf16(d, kh, xl, idS, 1);
                        mma_bf16(d, kl, xh, idS, 1);
                    }
                }
                // D^T per row block R: A = Q^^T (then K^b^T) rows 63 - r for r in R (MN-major),
                // B = dA (then dL) rows s < 16 (R + 1), K = the columns 63 - r of block R
                // (K-major)
#pragma unroll
                for (int R = 0; R < 4; ++R) {
                    const uint32_t idR = idesc_bf16(128, 16 * (R + 1), true, false);
                    const uint32_t arow = (48 - 16 * R) * 128, bcol = (48 - 16 * R) * 2;
                    const uint32_t d = tmem + 320 + kOffR[R];
#pragma unroll
                    for (int xs = 0; xs < 2; ++xs) {
                        const uint32_t ab = sb + (xs ? kKB : kQH) + arow;
                        const uint64_t ah = sdesc_sw128(ab, 8192, 1024);
                        const uint64_t al = sdesc_sw128(ab + 16384, 8192, 1024);
                        const uint32_t xb = sb + (xs ? kDLi : kDAi) + bcol;
                        const uint64_t xh = sdesc_sw128(xb, 0, 1024);
                        const uint64_t xl = sdesc_sw128(xb + 8192, 0, 1024);
                        mma_bf16(d, ah, xh, idR, xs);
                        mma_bf16(d, ah, xl, idR, 1);
                        mma_bf16(d, al, xh, idR, 1);
                    }
                }
                mma_commit(mma1);
            }
        }
        ok = ok && mbar_wait_ab(mma1, ph, p.err, abort);
        BP_MARK(13);
        float dG[32];
        float lastp = 0.f;
        const float rs_i = ld_early(reinterpret_cast<const float*>(mid + kMdRs) + ch);
        const float db1 = ld_early(reinterpret_cast<const float*>(mid + kMdB) + (tid & 63));
        if (ok) {
            tc_fence_after();
            const float* pQ = reinterpret_cast<const float*>(mid + kMdQ) + ch;
            const float* pP = reinterpret_cast<const float*>(mid + kMdP) + ch;
            const float* pE = reinterpret_cast<const float*>(mid + kMdE) + ch;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const int r0 = 32 * wh + 16 * g, R0 = 2 * wh + g;
                float pq16[16], pp16[16], pe16[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) pq16[u] = ld_early(pQ + (r0 + u) * 128);
#pragma unroll
                for (int u = 0; u < 16; ++u) pp16[u] = ld_early(pP + (r0 + u) * 128);
#pragma unroll
                for (int u = 0; u < 16; ++u) pe16[u] = ld_early(pE + (r0 + u) * 128);
                BP_MARK(16);
                float dqd[16], ee[16], ff[16], t16[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) { dqd[u] = 0.f; ee[u] = 0.f; ff[u] = 0.f; }
                // D(., K): element e of columns 48 - r0 .. is token r0 + 15 - e
                for (int S = 0; S <= R0; ++S) {
                    const float rho = sRho[S * 128 + ch];
                    float a16[16];
                    tmem_ld16(tmem + lb + kOffS[S] + 48 - r0, a16);
                    tmem_ld16(tmem + lb + 160 + kOffS[S] + 48 - r0, t16);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int u = 15 - e;
                        const float f = ex2f(G2[16 * g + u] - rho);
                        dqd[u] = fmaf(f, a16[e], dqd[u]);
                        ee[u] = fmaf(f, t16[e], ee[u]);
                    }
                }
                BP_MARK(17);
                // D^T: element e of columns r0 .. of block R is token r0 + e
                for (int R = R0; R < 4; ++R) {
                    const float rho = sRho[R * 128 + ch];
                    tmem_ld16(tmem + lb + 320 + kOffR[R] + r0, t16);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) ff[e] = fmaf(ex2f(rho - G2[16 * g + e]), t16[e], ff[e]);
                }
                BP_MARK(18);
                // this group's k, q and beta first (loads after the staging stores below may
                // not be hoisted above them)
                float k16[16], q16[16], b16[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int r = r0 + u;
                    const bool live = r < it.L;
                    k16[u] = live ? ldbf(sm + kKt + swz2(r, ch, 64)) : 0.f;
                    q16[u] = live ? ldbf(sm + kQt + swz2(r, ch, 64)) : 0.f;
                    b16[u] = sBeta[r];
                }
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int r = r0 + u;
                    const bool live = r < it.L;
                    const float kv = k16[u], qv = q16[u], b = b16[u];
                    const float pq = pq16[u], pp = pp16[u], pe = pe16[u];
                    const float dq = pq + dqd[u];
                    const float dkv = pp + b * ee[u] + ff[u] + pe;
                    dG[16 * g + u] = live ? kv * (pp + b * ee[u] - ff[u] - pe) + qv * dq : 0.f;
                    lastp = fmaf(kv, pe, lastp);
                    t16[u] = kv * ee[u];  // dbeta's E term, summed over channels below
                    const uint32_t o = swz2(r, ch, 64);  // dq, dk staged (the stacks are consumed)
                    *reinterpret_cast<uint16_t*>(sm + kKT + o) = bfbits(dq);
                    *reinterpret_cast<uint16_t*>(sm + kKT + 16384 + o) = bfbits(dkv);
                }
                BP_MARK(19);
                // sum over the 32 channels of this warp, then over the four warps
                {
                    const float v = warp_sum16(t16, lane);
                    if ((lane & 1) == 0) sDb[wq * 64 + r0 + (lane >> 1)] = v;
                }
                BP_MARK(20);
            }
            sLast[wh * 128 + ch] = lastp;
        }
        BP_MARK(14);
        csync();
        BP_MARK(21);
        float dAp = 0.f;
        if (ok) {
            // dG of the chunk's last row L - 1 also takes sum_r K pE + gamma^C rs
            const float last = sLast[ch] + sLast[128 + ch] + ex2f(sGlast[ch]) * rs_i;
            const int ul = it.L - 1 - 32 * wh;
            // reverse cumulative sum over this half, then the second half's total
            float acc = 0.f;
#pragma unroll
            for (int u = 31; u >= 0; --u) {
                if (u == ul) dG[u] += last;
                acc += dG[u];
                dG[u] = acc;
            }
            if (wh == 1) sTot[ch] = acc;
        }
        csync();
        BP_MARK(22);
        if (ok) {
            const float add = wh == 0 ? sTot[ch] : 0.f;
            // every z first: a load after a shared-memory store may not be hoisted above it
            float zz[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) zz[u] = ldbf(sm + kZt + swz2(32 * wh + u, ch, 64));
            const float gm = p.g_min;
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int r = 32 * wh + u;
                const float x = eA * zz[u];
                const float sg = __fdividef(1.f, 1.f + __expf(-x));
                const float dx = r < it.L ? (dG[u] + add) * gm * sg * (1.f - sg) : 0.f;
                dAp = fmaf(dx, x, dAp);
                *reinterpret_cast<uint16_t*>(sm + kQH + swz2(r, ch, 64)) = bfbits(dx * eA);
            }
            BP_MARK(24);
            if (tid < 64 && tid < it.L) {
                const float db = db1 + sDb[tid] + sDb[64 + tid] + sDb[128 + tid] + sDb[192 + tid];
                p.dbeta[(size_t)(it.t0 + tid) * p.H + it.h] = __float2bfloat16_rn(db);
            }
            BP_MARK(25);
        }
        // dA_log partial of the item: channels past dk have zero z and contribute x = 0
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dAp += __shfl_xor_sync(0xffffffffu, dAp, o);
        if (lane == 0) sRed[warp] = dAp;
        BP_MARK(23);
        tc_fence_before();
        fence_async_smem();
        ok = csync_and(ok);
        if (tid == 0 && ok) {
            float s = 0.f;
            for (int w = 0; w < 8; ++w) s += sRed[w];
            p.dA_item[item] = s;
        }
        if (ok) {
            store_tile(&p.tdq, sm + kKT, p.dq, it, p.H, p.dk, tid);
            store_tile(&p.tdk, sm + kKT + 16384, p.dkg, it, p.H, p.dk, tid);
            store_tile(&p.tdz, sm + kQH, p.dz, it, p.H, p.dk, tid);
        }
        csync();  // a short chunk's copies have read the staged tiles
        BP_MARK(15);
        if (!ok) break;
    }

    __syncthreads();
    if (s_abort && iss) {
        for (int b = 0; b < 2; ++b)
            if (inflight & (1u << b)) mbar_wait(&bars[b], inflight_ph, nullptr);
        mma_commit(drain);
        mbar_wait(drain, 0, nullptr);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTCols);
    }
}

}  // namespace
}  // namespace bwdtc

// The per-chunk backward on the tensor cores (see the top of this file): fwd_ws holds the
// forward's plan (chunk offsets and table), bimg the image blocks, mid the mid blocks.
#ifdef KDA_PHASE_TIMING
extern "C" int kda_debug_bwd_cycles(unsigned long long* out, int n) {
    if (n > 32) n = 32;
    if (cudaMemcpyFromSymbol(out, bwdtc::g_bwd_phase, n * sizeof(unsigned long long)) != cudaSuccess)
        return -1;
    static const unsigned long long zeros[32] = {};
    return cudaMemcpyToSymbol(bwdtc::g_bwd_phase, zeros, sizeof zeros) == cudaSuccess ? n : -1;
}
#endif

cudaError_t launch_bwd_items_tc(const BwdArgs& a, void* fwd_ws, const void* bimg, void* mid,
                                float* dA_item, cudaStream_t stream) {
    using namespace bwdtc;
    if ((int64_t)a.N * a.H == 0 || a.T_total == 0) return cudaSuccess;
    const fwdtc::WsLayout L = fwdtc::ws_layout(a.T_total, a.N, a.H);
    uint8_t* ws = static_cast<uint8_t*>(fwd_ws);
    ItemParams p{};
    if (!fwdtc::make_map(&p.tq, a.q, a.T_total, a.H, a.dk, 64) ||
        !fwdtc::make_map(&p.tk, a.k, a.T_total, a.H, a.dk, 64) ||
        !fwdtc::make_map(&p.tv, a.v, a.T_total, a.H, a.dv, 64) ||
        !fwdtc::make_map(&p.tz, a.z, a.T_total, a.H, a.dk, 64) ||
        !fwdtc::make_map(&p.tdo, a.dout, a.T_total, a.H, a.dv, 64) ||
        !fwdtc::make_map(&p.tdq, a.dq, a.T_total, a.H, a.dk, 64) ||
        !fwdtc::make_map(&p.tdk, a.dk_, a.T_total, a.H, a.dk, 64) ||
        !fwdtc::make_map(&p.tdz, a.dz, a.T_total, a.H, a.dk, 64) ||
        !fwdtc::make_map(&p.tdv, a.dv_, a.T_total, a.H, a.dv, 64))
        return cudaErrorInvalidValue;
    p.beta = static_cast<const __nv_bfloat16*>(a.beta);
    p.v = static_cast<const __nv_bfloat16*>(a.v);
    p.A_log = a.A_log;
    p.chunk_off = reinterpret_cast<const int32_t*>(ws + L.off_chunk_off);
    p.chunk_tab = reinterpret_cast<const int4*>(ws + L.off_tab);
    p.bimg = static_cast<const uint8_t*>(bimg);
    p.mid = static_cast<uint8_t*>(mid);
    p.dq = static_cast<__nv_bfloat16*>(a.dq);
    p.dkg = static_cast<__nv_bfloat16*>(a.dk_);
    p.dvg = static_cast<__nv_bfloat16*>(a.dv_);
    p.dbeta = static_cast<__nv_bfloat16*>(a.dbeta);
    p.dz = static_cast<__nv_bfloat16*>(a.dz);
    p.dA_item = dA_item;
    p.err = a.dev_err;
    p.g_min = a.g_min;
    p.N = a.N;
    p.H = a.H;
    p.dk = a.dk;
    p.dv = a.dv;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t items = (a.T_total / fwdtc::kC + a.N) * (int64_t)a.H;  // an upper bound
    const int grid = (int)(items < sms ? items : sms);
    cudaError_t e = cudaFuncSetAttribute(bwd_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kStateSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_decay_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kDecaySmem);
    if (e != cudaSuccess) return e;
    {
        ProfScope prof("bwd_state_kernel", stream);
        bwd_state_kernel<<<grid, kThreads, kStateSmem, stream>>>(p);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ProfScope prof("bwd_decay_kernel", stream);
    bwd_decay_kernel<<<grid, kThreads, kDecaySmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
