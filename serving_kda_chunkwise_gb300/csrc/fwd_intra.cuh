// fwd_intra.cuh -- the parallel stage of the tensor-core chunked forward: every (chunk,
// head) item builds the chunk's UT form and writes its package (see fwd_tc_layout.cuh).
// Included by fwd_tc.cu, which launches it alone (intra_kernel) or as one role of the fused
// forward kernel (fwd_fused_kernel).
//
// Sub-tiling ("Kimi k3 技术报告详解（1）——架构再升华", section "Chunkwise parallel form",
// 16-token tiles; the bounded gate g > g_min is what keeps these factors finite): the Gram
// entry for rows r >= i needs e^{G_r - G_i} per channel.  With rho_s = G at the 8th row of
// sub-tile s (its middle), every row r of sub-tile s uses ONE row factor e^{G_r - rho_s}
// (|exponent| <= 8|g_min| <= 48) and the column operand for that sub-tile is
// k_i e^{rho_s - G_i}: for i in the same sub-tile the exponent is again bounded by 48, for
// earlier i it is <= 0 (underflow there only drops terms below e^{-39}).  So the column
// operand comes in four versions (sub-tile s uses columns i < 16(s+1)); stacking them gives
// one B operand of 16+32+48+64 = 160 rows, and stacking the q-side and (beta-scaled) k-side
// row operands gives A with M = 128: a single M=128, N=160, K=128 MMA yields both Grams for
// every sub-tile pair.
#pragma once

#include "fwd_tc_layout.cuh"
#include "kda_common.cuh"
#include "tc_util.cuh"

namespace kda {
namespace fwdtc {
namespace {

using namespace tc;

// 8 warps (two per SM sub-partition); lane 0 of warp 6, whose row work is among the
// lightest, also issues every copy and MMA
constexpr int kIntraThreads = 256;
constexpr int kIss = 192;

// Barrier over the intra stage's 256 threads (the fused kernel's CTAs have more threads;
// the rest leave at once).
__device__ __forceinline__ void intra_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Optional phase timers (debug builds with -DKDA_PHASE_TIMING only): thread 0 of CTA 0
// accumulates clock64() deltas between marked points of each kernel's loop.
#ifdef KDA_PHASE_TIMING
__device__ unsigned long long g_phase[32];
#define KDA_PHASE_INIT()              \
    long long kda_t_last = clock64(); \
    unsigned long long kda_acc[32] = {}
#define KDA_PHASE(i)                                                \
    do {                                                            \
        const long long kda_t = clock64();                          \
        kda_acc[(i)] += (unsigned long long)(kda_t - kda_t_last);   \
        kda_t_last = kda_t;                                         \
    } while (0)
#define KDA_PHASE_FLUSH()                                                     \
    do {                                                                      \
        if (cta == 0 && threadIdx.x == 0)                                     \
            for (int kda_i = 0; kda_i < 32; ++kda_i)                          \
                if (kda_acc[kda_i]) atomicAdd(&g_phase[kda_i], kda_acc[kda_i]); \
    } while (0)
#else
#define KDA_PHASE_INIT() \
    do {                 \
    } while (0)
#define KDA_PHASE(i) \
    do {             \
    } while (0)
#define KDA_PHASE_FLUSH() \
    do {                  \
    } while (0)
#endif

// ================================================================ intra ====

struct IntraParams {
    CUtensorMap tq, tk, tv, tz;  // [T_total, H, 128] bf16, box 64 x 1 x 64, 128-byte swizzle
    const __nv_bfloat16* beta;
    const float* A_log;
    const int32_t* cu;
    const int32_t* chunk_off;
    const int4* chunk_tab;
    uint8_t* pkg;  // packages [H][maxchunks], or the ring [C][ring_slots] in the fused kernel
    unsigned* err;
    int64_t T_total;
    float g_min;
    int N, H, maxchunks;
    // fused kernel only (fused_C = 0 otherwise): C = N * H chains of nct chunks each (equal
    // sequence lengths), items in chunk-major order (item = t * C + chain, chain = n * H + h);
    // the package of chunk t of chain c goes to ring slot c * ring_slots + t % ring_slots
    int fused_C, nct, ring_slots;
    uint32_t* ready;     // [C][ring_slots]: t + 1 once the slot holds chunk t
    uint32_t* consumed;  // [C]: chunks of the chain whose slots the chain stage has released
    // fused kernel: items are taken from this counter in order (a CTA whose item waits for a
    // slot holds up no other chain's items); otherwise CTA b takes items b, b + ncta, ...
    int* item_ctr;
};

// Shared-memory map of the intra kernel (offsets from a 1024-aligned base).  q and k are
// double buffered (the next item's are fetched by TMA once this item's operands are built);
// v and z have one buffer each, refilled as soon as the current item has consumed them.
constexpr uint32_t kQKBuf = 32768;            // per q/k buffer: q, k (16 KB each)
constexpr uint32_t kOffQ = 0, kOffK = 16384;
constexpr uint32_t kVBuf = 2 * kQKBuf;        //  65536: v   [2 blk][64 rows][128 B]
constexpr uint32_t kZBuf = kVBuf + 16384;     //  81920: z
constexpr uint32_t kKbar = kZBuf + 16384;     //  98304: Gam*K (A of W = M Gam K, MN-major);
                                              //         earlier: per-warp cumsum totals fp32[8][128]
constexpr uint32_t kAStk = kKbar + 16384;     // 114688: A hi [2 blk][128 rows][128 B]
constexpr uint32_t kALo = kAStk + 32768;      // 147456: q-side A lo [2 blk][64 rows][128 B]
constexpr uint32_t kBStk = kALo + 16384;      // 163840: B hi [2 blk][160 rows][128 B]
constexpr uint32_t kBLo = kBStk + 40960;      // 204800: diagonal-column lo [2 blk][64][128 B]
constexpr uint32_t kXch = kBLo + 16384;       // 221184: rho fp32[4][128], glast fp32[128]
constexpr uint32_t kBeta = kXch + 2560;       // 223744: beta [2][64] fp32
constexpr uint32_t kBars = kBeta + 512;       // 224256: mbarriers
constexpr uint32_t kIntraSmem = kBars + 64 + 1024;  // + alignment slack
static_assert(kIntraSmem <= 232448, "intra kernel exceeds the shared-memory limit");
// reuse after the Gram MMAs: A hi -> A tile hi, lo (8 KB each) + M tile (8 KB);
// B hi -> L, T, Y (fp32).
// The M tile is stored twice (rows 0..63 and 64..127 of a 128-row operand).
constexpr uint32_t kAqkTile = kAStk, kAqkLoTile = kAStk + 8192, kMTile = kAStk + 16384;
constexpr int kLd = 68;                       // padded fp32 row stride of L and T (fewer
                                              // bank conflicts in the 16x16 tile fragments)
constexpr uint32_t kSL = kBStk, kST = kBStk + 64 * kLd * 4;
static_assert(kST + 64 * kLd * 4 <= kBStk + 40960, "L and T must fit the B stack");
// the solve's scratch (9 tiles of 16 x 20 floats) reuses the A-lo region
constexpr uint32_t kSolveScr = kALo;
static_assert(9 * 16 * 20 * 4 <= 16384, "solve scratch must fit the A-lo region");
// TMEM columns: main Gram accumulator [0, 160), diagonal-column lo correction [160, 224),
// q-side lo correction [256, 416);
// later W [0, 128) and U [128, 256).
constexpr uint32_t kTmemCols = 512, kTLo = 256, kTDiag = 160;

__device__ __constant__ int kStkOff[4] = {0, 16, 48, 96};  // B-stack row offset per version

struct ItemInfo {
    int item;  // item index (>= the item count: no further item)
    int h, n, L;
    int64_t t0;
    size_t pkg;  // package index (ring slot in the fused kernel)
    int fc, ft;  // fused kernel: chain and chunk within the chain
};

// Loads that are issued well ahead of their use.  The asm keeps each load where it is
// written: a plain load may be sunk to its first use, which would expose its latency there.
__device__ __forceinline__ int4 ld_ahead(const int4* q) {
    int4 r;
    asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(q));
    return r;
}
__device__ __forceinline__ float ld_ahead(const float* q) {
    float r;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(r) : "l"(q));
    return r;
}
__device__ __forceinline__ unsigned short ld_ahead(const __nv_bfloat16* q) {
    unsigned short r;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(q));
    return r;
}

// Item = chunk * H + head (fused kernel: item = t * C + n * H + h).  The table entry is
// fetched ahead and decoded when needed.
__device__ __forceinline__ int fused_chunk_index(const IntraParams& p, int item) {
    const int t = item / p.fused_C, c = item - t * p.fused_C;
    return (c / p.H) * p.nct + t;
}
__device__ __forceinline__ int4 fetch_item(const IntraParams& p, int item) {
    return ld_ahead(p.chunk_tab + (p.fused_C ? fused_chunk_index(p, item) : item / p.H));
}
__device__ __forceinline__ ItemInfo decode_item(const IntraParams& p, int item, int4 e) {
    ItemInfo it;
    it.item = item;
    it.n = e.z;
    it.t0 = (static_cast<int64_t>(e.y) << 32) | static_cast<uint32_t>(e.x);
    it.L = e.w;
    if (p.fused_C) {
        const int t = item / p.fused_C, c = item - t * p.fused_C;
        it.h = c - (c / p.H) * p.H;
        it.fc = c;
        it.ft = t;
        it.pkg = (size_t)c * p.ring_slots + t % p.ring_slots;
    } else {
        const int chunk = item / p.H;
        it.h = item - chunk * p.H;
        it.fc = 0;
        it.ft = 0;
        it.pkg = (size_t)it.h * p.maxchunks + chunk;
    }
    return it;
}
// The item a CTA takes after `cur` (the first one: cur = -1).
__device__ __forceinline__ int take_item(const IntraParams& p, int cur, int cta, int ncta) {
    if (p.item_ctr) return atomicAdd(p.item_ctr, 1);
    return cur < 0 ? cta : cur + ncta;
}

// TMA: [64 rows][128] bf16 tiles of one or two tensors for this item (two 64-column
// blocks each), completing on `bar`.
__device__ __forceinline__ void load_tiles(const CUtensorMap* m0, uint8_t* d0,
                                           const CUtensorMap* m1, uint8_t* d1,
                                           const ItemInfo& it, uint64_t* bar) {
    mbar_expect_tx(bar, m1 ? 32768 : 16384);
#pragma unroll
    for (int cb = 0; cb < 2; ++cb) {
        tma_load_3d(d0 + cb * 8192, m0, cb * 64, it.h, (int)it.t0, bar);
        if (m1) tma_load_3d(d1 + cb * 8192, m1, cb * 64, it.h, (int)it.t0, bar);
    }
}

__device__ __forceinline__ void load_beta(const IntraParams& p, const ItemInfo& it, float* dst,
                                          int tid) {
    if (tid < kC)
        dst[tid] = (tid < it.L) ? __bfloat162float(p.beta[(size_t)(it.t0 + tid) * p.H + it.h]) : 0.f;
}

// 2^x (the hardware approximation; results below 2^-126 flush to zero)
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 8 consecutive bf16 of a swizzled tile <-> fp32 registers
__device__ __forceinline__ void ld8(const uint8_t* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
        v[2 * e] = f.x;
        v[2 * e + 1] = f.y;
    }
}
__device__ __forceinline__ uint4 pk8(const float (&v)[8]) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
}
// hi = bf16(v), lo = bf16(v - hi)  (the fp32 value of a packed bf16 is its bits shifted up)
__device__ __forceinline__ void pk8_hilo(const float (&v)[8], uint4& hi, uint4& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        h[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
        l[e] = pack_bf16x2(v[2 * e] - __uint_as_float(h[e] << 16),
                           v[2 * e + 1] - __uint_as_float(h[e] & 0xffff0000u));
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// ---- 16x16 fp32 tiles on the legacy warp-level tensor-core path (mma.sync, tf32 inputs,
//      fp32 accumulation), used for the small triangular solve.  A tile is held by a warp
//      as two m16n8 accumulators: element (row, col) of accumulator nn, slot q sits in lane
//      4*(row % 8) + (col % 8) / 2 with row = g + 8*(q >> 1), col = 8*nn + 2*t + (q & 1).
struct Tile16 {
    float c[2][4];
};

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void tile_zero(Tile16& f) {
#pragma unroll
    for (int nn = 0; nn < 2; ++nn)
#pragma unroll
        for (int q = 0; q < 4; ++q) f.c[nn][q] = 0.f;
}

// f = scale * X
__device__ __forceinline__ void tile_load(Tile16& f, const float* X, int ld, float scale) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nn = 0; nn < 2; ++nn)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int row = g + 8 * (q >> 1), col = 8 * nn + 2 * t + (q & 1);
            f.c[nn][q] = scale * X[row * ld + col];
        }
}

// X = scale * f + diag * I
__device__ __forceinline__ void tile_store(const Tile16& f, float* X, int ld, float scale,
                                           float diag) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nn = 0; nn < 2; ++nn)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int row = g + 8 * (q >> 1), col = 8 * nn + 2 * t + (q & 1);
            X[row * ld + col] = scale * f.c[nn][q] + (row == col ? diag : 0.f);
        }
}

// f += A B  (A, B: 16x16 fp32 tiles in shared memory, row-major with strides lda, ldb)
__device__ __forceinline__ void tile_mma(Tile16& f, const float* A, int lda, const float* B,
                                         int ldb) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        const uint32_t a0 = to_tf32(A[g * lda + 8 * kk + t]);
        const uint32_t a1 = to_tf32(A[(g + 8) * lda + 8 * kk + t]);
        const uint32_t a2 = to_tf32(A[g * lda + 8 * kk + t + 4]);
        const uint32_t a3 = to_tf32(A[(g + 8) * lda + 8 * kk + t + 4]);
#pragma unroll
        for (int nn = 0; nn < 2; ++nn) {
            const uint32_t b0 = to_tf32(B[(8 * kk + t) * ldb + 8 * nn + g]);
            const uint32_t b1 = to_tf32(B[(8 * kk + t + 4) * ldb + 8 * nn + g]);
            asm volatile(
                "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
                "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                : "+f"(f.c[nn][0]), "+f"(f.c[nn][1]), "+f"(f.c[nn][2]), "+f"(f.c[nn][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
        }
    }
}

// T = (I + L)^{-1} for the 64x64 strictly lower L (16x16 blocks).  Warp w < 4 first inverts
// diagonal block w by forward substitution in fp32 (lane j holds column j:
// T_ij = delta_ij - sum_{k<i} L_ik T_kj); the off-diagonal blocks follow from the expansion
// below.  `scr_all` holds 9 scratch tiles of 16 x kScrLd floats.
constexpr int kScrLd = 20;
constexpr int kScrTile = 16 * kScrLd;

__device__ __forceinline__ int lane16() { return threadIdx.x & 15; }

__device__ __forceinline__ void solve_tril64(const float* sL, float* sT, float* scr_all,
                                             int warp, int iter_for_trace) {
    if (warp < 4) {
        const float* Lb = sL + (16 * warp) * kLd + 16 * warp;
        const int j = lane16();
        float tc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float Lr[16];  // row i of the block (only k < i is used)
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                if (4 * k4 < i) {
                    const float4 v = *reinterpret_cast<const float4*>(Lb + i * kLd + 4 * k4);
                    Lr[4 * k4] = v.x; Lr[4 * k4 + 1] = v.y; Lr[4 * k4 + 2] = v.z; Lr[4 * k4 + 3] = v.w;
                }
            }
            float acc = (i == j) ? 1.f : 0.f;
#pragma unroll
            for (int k = 0; k < i; ++k) acc = fmaf(-Lr[k], tc[k], acc);
            tc[i] = acc;
        }
        if ((threadIdx.x & 31) < 16)
#pragma unroll
            for (int i = 0; i < 16; ++i) sT[(16 * warp + i) * kLd + 16 * warp + j] = tc[i];
    }
    intra_sync();
    // Off-diagonal blocks: with Delta the inverted diagonal blocks and F_ij = Delta_i L_ij
    // (i > j, nilpotent), T = (I + F)^{-1} Delta = (I - F + F^2 - F^3) Delta, so
    //   T_{i+1,i} = -F_{i+1,i} Delta_i,
    //   T_20 = G20 Delta_0, G20 = -F20 + F21 F10;   T_31 = G31 Delta_1, G31 = -F31 + F32 F21;
    //   T_30 = G30 Delta_0, G30 = -F30 + F31 F10 - F32 G20:
    // four levels of independent 16x16 products instead of a chain by distance.
    auto Lb = [&](int i, int j) { return sL + (16 * i) * kLd + 16 * j; };
    auto Tb = [&](int i, int j) { return sT + (16 * i) * kLd + 16 * j; };
    auto Sc = [&](int k) { return scr_all + k * kScrTile; };  // F10 F21 F32 F20 F31 F30 G20 G31 H30
    // level 1: F_ij = Delta_i L_ij for the six off-diagonal blocks
    if (warp < 6) {
        // (i, j) = (1,0) (2,1) (3,2) (2,0) (3,1) (3,0), packed in nibbles
        const int i = (0x332321 >> (4 * warp)) & 15, j = (0x010210 >> (4 * warp)) & 15;
        Tile16 f;
        tile_zero(f);
        tile_mma(f, Tb(i, i), kLd, Lb(i, j), kLd);
        tile_store(f, Sc(warp), kScrLd, 1.f, 0.f);
    }
    intra_sync();
    // level 2: G20, G31, H30 = -F30 + F31 F10; T10, T21, T32
    if (warp < 3) {
        // G20 = -F20 + F21 F10, G31 = -F31 + F32 F21, H30 = -F30 + F31 F10
        const int fa = (0x421 >> (4 * warp)) & 15, fb = (0x010 >> (4 * warp)) & 15;
        Tile16 f;
        tile_load(f, Sc(3 + warp), kScrLd, -1.f);
        tile_mma(f, Sc(fa), kScrLd, Sc(fb), kScrLd);
        tile_store(f, Sc(6 + warp), kScrLd, 1.f, 0.f);
    } else if (warp < 6) {
        const int k = warp - 3;  // T_{k+1,k} = -F_{k+1,k} Delta_k
        Tile16 f;
        tile_zero(f);
        tile_mma(f, Sc(k), kScrLd, Tb(k, k), kLd);
        tile_store(f, Tb(k + 1, k), kLd, -1.f, 0.f);
    }
    intra_sync();
    // levels 3 and 4: G30 then T30 (warp 0); T20, T31 (warps 1, 2)
    if (warp == 0) {
        Tile16 f, q;
        tile_load(f, Sc(8), kScrLd, 1.f);  // H30
        tile_zero(q);
        tile_mma(q, Sc(2), kScrLd, Sc(6), kScrLd);  // F32 G20
#pragma unroll
        for (int nn = 0; nn < 2; ++nn)
#pragma unroll
            for (int e = 0; e < 4; ++e) f.c[nn][e] -= q.c[nn][e];
        tile_store(f, Sc(8), kScrLd, 1.f, 0.f);  // G30
        __syncwarp();
        tile_zero(q);
        tile_mma(q, Sc(8), kScrLd, Tb(0, 0), kLd);
        tile_store(q, Tb(3, 0), kLd, 1.f, 0.f);
    } else if (warp < 3) {
        const int k = warp - 1;  // T_{k+2,k} = G_{k+2,k} Delta_k
        Tile16 f;
        tile_zero(f);
        tile_mma(f, Sc(6 + k), kScrLd, Tb(k, k), kLd);
        tile_store(f, Tb(k + 2, k), kLd, 1.f, 0.f);
    }
    intra_sync();
}

__device__ __forceinline__ void intra_body(const IntraParams& p, uint8_t* smem_raw, int cta, int ncta) {
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(sm);
    float* tot = reinterpret_cast<float*>(sm + kKbar);   // [8 warps][128] cumsum totals
    float* xrho = reinterpret_cast<float*>(sm + kXch);   // [4][128]
    uint64_t* qk_bar = reinterpret_cast<uint64_t*>(sm + kBars);  // [2]
    uint64_t* v_bar = qk_bar + 2;
    uint64_t* z_bar = qk_bar + 3;
    uint64_t* mma_bar = qk_bar + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qk_bar + 5);
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // operand passes: 8 channels [8 cg, 8 cg + 8) of rows [4 rg, 4 rg + 4)
    const int cg = tid & 15, rg = tid >> 4, sub = rg >> 2;
    const uint32_t cofs = (cg >> 3) * 8192;  // 64-column block of the channel group
    const int ch0 = 8 * cg;
    if (tid == 0) {
        mbar_init(&qk_bar[0], 1);
        mbar_init(&qk_bar[1], 1);
        mbar_init(v_bar, 1);
        mbar_init(z_bar, 1);
        mbar_init(mma_bar, 1);
        fence_mbar_init();
        s_abort = 0;
    }
    if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    intra_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n_items = p.fused_C ? p.nct * p.fused_C : __ldg(p.chunk_off + p.N) * p.H;
    int pub_slot = -1;      // issuing thread, fused kernel: the finished package not yet
    uint32_t pub_val = 0;   // published (ring slot, ready value)
    uint32_t mma_phase = 0;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;

    // parity of the phase a load in flight will complete, or -1 (issuing thread; for a clean
    // abort)
    int pend_q[2] = {-1, -1}, pend_v = -1, pend_z = -1;
    // The issuing thread walks the item table and publishes each item's description and
    // A_log in s_item / s_alog (two slots by item parity) one item before its use, so the
    // row warps start an item without global loads.
    // The issuing thread also takes the items: it keeps the index of the item after the one
    // it publishes (taken one item early, so that a counter's latency is never waited for).
    __shared__ ItemInfo s_item[2];
    __shared__ float s_alog[2];
    int lead_next = n_items;
    if (tid == kIss) {
        const int first_item = take_item(p, -1, cta, ncta);
        s_item[0].item = first_item;
        if (first_item < n_items) lead_next = take_item(p, first_item, cta, ncta);
    }
    if (tid == kIss && s_item[0].item < n_items) {
        const ItemInfo first = decode_item(p, s_item[0].item, fetch_item(p, s_item[0].item));
        load_tiles(&p.tq, sm + kOffQ, &p.tk, sm + kOffK, first, &qk_bar[0]);
        load_tiles(&p.tv, sm + kVBuf, nullptr, nullptr, first, v_bar);
        load_tiles(&p.tz, sm + kZBuf, nullptr, nullptr, first, z_bar);
        pend_q[0] = 0;
        pend_v = 0;
        pend_z = 0;
        s_item[0] = first;
        s_alog[0] = __ldg(p.A_log + first.h);
    }
    intra_sync();
    if (s_item[0].item < n_items) load_beta(p, s_item[0], reinterpret_cast<float*>(sm + kBeta), tid);

    int iter = 0;
    KDA_PHASE_INIT();
    for (;; ++iter) {
        KDA_PHASE(7);
        const int b = iter & 1;
        // published before the previous item's last barrier (or the first one's)
        if (s_item[b].item >= n_items) break;
        uint8_t* qk = sm + b * kQKBuf;
        float* sBeta = reinterpret_cast<float*>(sm + kBeta) + 64 * b;
        const int itL = s_item[b].L;  // rows of this item (< 64 for a sequence's last chunk)
        const float alog = s_alog[b];
        // the next item, known to the issuing thread (which took it one item ago) and
        // needed by its warp only (that warp loads the next item's beta); the item after it
        // is taken now
        const int next = warp == (kIss >> 5) ? __shfl_sync(0xffffffffu, lead_next, kIss & 31) : n_items;
        const bool has_next = next < n_items;
        int next2 = n_items;
        if (tid == kIss && has_next) next2 = take_item(p, next, cta, ncta);
        unsigned short beta_nx[2] = {0, 0};  // issuing thread's warp: the next item's beta (bf16)
        float alog_nx = 0.f;                 // issuing thread: the next item's A_log
        // issuing thread: the next item's table entry, decoded once the scan is done
        int4 raw_next;
        if (tid == kIss && has_next) raw_next = fetch_item(p, next);
        // this item's package (re-read where used: nothing held in registers across phases)
        auto item_pkg = [&]() { return p.pkg + s_item[b].pkg * kPkgBytes; };

        // ---- gate and in-chunk cumsum
        if (mbar_wait(z_bar, iter & 1, p.err)) {
            if (tid == kIss) pend_z = -1;
        } else {
            s_abort = 1;
        }
        KDA_PHASE(0);
        // G[i][e]: cumulative gate of row 4 rg + i, channel ch0 + e; gl: G of the last row.
        // Cumulative gate in log2 units (G2 = G log2 e, so every decay factor is one ex2).
        // Scan: in-thread over 4 rows, in-warp over its two row groups (shuffle), then over
        // the 8 warps' totals (one thread per channel).
        float G[4][8], gl[8], pre[8];
        float* xtot = xrho + 512;  // [128]: G2 of the chunk's last row
        {
            const float scale2 = expf(alog) * 1.4426950408889634f;  // e^{A_log} log2 e
            const float gmin2 = p.g_min * 1.4426950408889634f;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * rg + i;
                const bool live = r < itL;
                float zz[8];
                ld8(sm + kZBuf + cofs + sw128_chunk(r, cg & 7), zz);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    // evaluated for every row and masked after (a conditional evaluation
                    // serialises the special-function work)
                    const float g = __fdividef(gmin2, 1.f + ex2f(-scale2 * zz[e]));
                    acc[e] += live ? g : 0.f;
                    G[i][e] = acc[e];
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float lo = __shfl_up_sync(0xffffffffu, acc[e], 16);  // row group 2 warp
                pre[e] = (lane >= 16) ? lo : 0.f;
            }
            if (lane >= 16) {  // this warp's total over its 8 rows
                float4* tw = reinterpret_cast<float4*>(tot + warp * 128 + ch0);
                tw[0] = make_float4(acc[0] + pre[0], acc[1] + pre[1], acc[2] + pre[2], acc[3] + pre[3]);
                tw[1] = make_float4(acc[4] + pre[4], acc[5] + pre[5], acc[6] + pre[6], acc[7] + pre[7]);
            }
        }
        intra_sync();
        KDA_PHASE(9);
        if (tid < kD) {  // exclusive scan over the warps, in place, one channel per thread
            float v[8];
#pragma unroll
            for (int w2 = 0; w2 < 8; ++w2) v[w2] = tot[w2 * 128 + tid];
            float a = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < 8; ++w2) {
                tot[w2 * 128 + tid] = a;
                a += v[w2];
            }
            xtot[tid] = a;
        }
        intra_sync();
        // z is consumed: the issuing thread publishes the next item and fetches its z
        // (issued here, where a long phase follows, so that a slow issue never holds up a
        // barrier)
        if (tid == kIss && !has_next) s_item[b ^ 1].item = n_items;  // no further item
        if (warp == (kIss >> 5) && has_next) {
            if (tid == kIss) {
                const ItemInfo nx = decode_item(p, next, raw_next);
                s_item[b ^ 1] = nx;  // read after the next CTA barrier
                alog_nx = ld_ahead(p.A_log + nx.h);
                load_tiles(&p.tz, sm + kZBuf, nullptr, nullptr, nx, z_bar);
                pend_z = (iter + 1) & 1;
            }
            __syncwarp();
            // the next item's beta (rows lane, lane + 32), stored into its slot during the
            // operand pass, where this warp has no other work
            const ItemInfo& nxs = s_item[b ^ 1];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int r = lane + 32 * h2;
                if (r < nxs.L)
                    beta_nx[h2] = ld_ahead(p.beta + (size_t)(nxs.t0 + r) * p.H + nxs.h);
            }
        }
        {
            const float4 pa = *reinterpret_cast<const float4*>(tot + warp * 128 + ch0);
            const float4 pb = *reinterpret_cast<const float4*>(tot + warp * 128 + ch0 + 4);
            const float4 ga = *reinterpret_cast<const float4*>(xtot + ch0);
            const float4 gb = *reinterpret_cast<const float4*>(xtot + ch0 + 4);
            const float p8[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
            const float g8[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                gl[e] = g8[e];
                pre[e] += p8[e];
#pragma unroll
                for (int i = 0; i < 4; ++i) G[i][e] += pre[e];
            }
        }
        KDA_PHASE(10);
        if ((rg & 3) == 1)  // rows 4 rg + 3 = 16 s + 7: the reference of sub-tile s
#pragma unroll
            for (int e = 0; e < 8; ++e) xrho[sub * 128 + ch0 + e] = G[3][e];
        if (mbar_wait(&qk_bar[b], (iter >> 1) & 1, p.err)) {
            if (tid == kIss) pend_q[b] = -1;
        } else {
            s_abort = 1;
        }
        // the previous item's package stores read the A tiles, the B-stack region and
        // the other q/k buffer: all are rewritten from here on.  In the fused kernel the
        // previous item is published first (its stores complete, then its ready flag), and
        // only then does this item wait for its ring slot: a CTA never waits for a slot
        // while holding a finished but unpublished package.
        if (tid == kIss) {
            if (p.fused_C) {
                if (pub_slot >= 0) {
                    bulk_wait0();
                    fence_proxy_async_global();
                    st_release_gpu(p.ready + pub_slot, pub_val);
                    pub_slot = -1;
                }
                const ItemInfo& cur = s_item[b];
                if (cur.ft >= p.ring_slots &&
                    !wait_flag_ge(p.consumed + cur.fc, (uint32_t)(cur.ft - p.ring_slots + 1), p.err,
                                  reinterpret_cast<volatile int*>(&s_abort)))
                    s_abort = 1;
            } else {
                bulk_wait_read0();
            }
        }
        intra_sync();
        KDA_PHASE(1);
        if (s_abort) break;
        if (rg == 15)
#pragma unroll
            for (int e = 0; e < 8; ++e) reinterpret_cast<float*>(item_pkg() + kPkgG)[ch0 + e] = ex2f(gl[e]);

        if (warp == (kIss >> 5)) {
            float* dst = reinterpret_cast<float*>(sm + kBeta) + 64 * (b ^ 1);
            dst[lane] = __bfloat162float(__ushort_as_bfloat16(beta_nx[0]));
            dst[lane + 32] = __bfloat162float(__ushort_as_bfloat16(beta_nx[1]));
            if (lane == 0) s_alog[b ^ 1] = alog_nx;
        }

        // ---- decay-scaled operands.  Row r of sub-tile s uses e1 = e^{G_r - rho_s}; the
        //      column operand of version s2 >= s is k_r e^{rho_s2 - G_r}.
        {
            // Ev[v][e] = e^{rho_{s2} - rho_s} for the later sub-tiles s2 = sub + 1 + v (<= 1;
            // may underflow to 0, which drops Gram terms below e^-13 of their neighbours):
            // the column operand of version s2 is then k e^{rho_s - G} Ev.
            float rho[8], Ev[3][8];
#pragma unroll
            for (int e = 0; e < 8; ++e) rho[e] = xrho[sub * 128 + ch0 + e];  // (log2 units, as G)
#pragma unroll
            for (int v = 0; v < 3; ++v) {
                const int s2 = min(sub + 1 + v, 3);  // entries past sub-tile 3 are unused
#pragma unroll
                for (int e = 0; e < 8; ++e) Ev[v][e] = ex2f(xrho[s2 * 128 + ch0 + e] - rho[e]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * rg + i;
                const bool ok = r < itL;
                const uint32_t o64 = cofs + sw128_chunk(r, cg & 7);
                const uint32_t o128 = (cg >> 3) * 16384 + sw128_chunk(r, cg & 7);
                float qv[8], kv[8], e1[8], dc[8], t[8];
                ld8(qk + kOffQ + o64, qv);
                ld8(qk + kOffK + o64, kv);
                const float br = sBeta[r];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (!ok) { qv[e] = 0.f; kv[e] = 0.f; }
                    e1[e] = ex2f(G[i][e] - rho[e]);
                    dc[e] = ex2f(rho[e] - G[i][e]);
                }
                uint4 hi, lo;
#pragma unroll
                for (int e = 0; e < 8; ++e) t[e] = qv[e] * e1[e];
                pk8_hilo(t, hi, lo);
                *reinterpret_cast<uint4*>(sm + kAStk + o128) = hi;
                *reinterpret_cast<uint4*>(sm + kALo + o64) = lo;
#pragma unroll
                for (int e = 0; e < 8; ++e) t[e] = br * kv[e] * e1[e];
                *reinterpret_cast<uint4*>(sm + kAStk + o128 + 64 * 128) = pk8(t);
#pragma unroll
                for (int e = 0; e < 8; ++e) t[e] = kv[e] * dc[e];
                pk8_hilo(t, hi, lo);
                *reinterpret_cast<uint4*>(
                    sm + kBStk + (cg >> 3) * 20480 + sw128_chunk(kStkOff[sub] + r, cg & 7)) = hi;
                *reinterpret_cast<uint4*>(sm + kBLo + o64) = lo;
#pragma unroll
                for (int v = 0; v < 3; ++v) {
                    const int s2 = sub + 1 + v;
                    if (s2 < 4) {  // uniform within a warp
#pragma unroll
                        for (int e = 0; e < 8; ++e) t[e] = kv[e] * dc[e] * Ev[v][e];
                        *reinterpret_cast<uint4*>(sm + kBStk + (cg >> 3) * 20480 +
                                                  sw128_chunk(kStkOff[s2] + r, cg & 7)) = pk8(t);
                    }
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        intra_sync();
        KDA_PHASE(2);
        if (tid == kIss) {
            if (has_next) {
                fence_async_smem();
                load_tiles(&p.tq, sm + (b ^ 1) * kQKBuf + kOffQ, &p.tk,
                           sm + (b ^ 1) * kQKBuf + kOffK, s_item[b ^ 1], &qk_bar[b ^ 1]);
                pend_q[b ^ 1] = ((iter + 1) >> 1) & 1;
            }
        }

        // ---- Grams: D = [Q'; beta K']_hi Bstack_hi^T (+ diagonal-column lo terms),
        //      D_lo = Q'_lo Bstack_hi^T (its k-side lanes are unused)
        if (tid == kIss) {
            tc_fence_after();
            constexpr uint32_t id160 = idesc_bf16(128, 160, false, false);
            constexpr uint32_t id64 = idesc_bf16(128, 64, false, false);
            // descriptors differ only in the start-address field (address / 16)
            const uint64_t dA = sdesc_sw128(sbase + kAStk, 0, 1024);
            const uint64_t dB = sdesc_sw128(sbase + kBStk, 0, 1024);
            const uint64_t dAl = sdesc_sw128(sbase + kALo, 0, 1024);
            const uint64_t dBl = sdesc_sw128(sbase + kBLo, 0, 1024);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kofs = (ks & 3) * 32;
                const uint64_t ah = dA + (((ks >> 2) * 16384 + kofs) >> 4);
                const uint64_t bh = dB + (((ks >> 2) * 20480 + kofs) >> 4);
                mma_bf16(tmem, ah, bh, id160, ks > 0);
                mma_bf16(tmem + kTLo, dAl + (((ks >> 2) * 8192 + kofs) >> 4), bh, id160, ks > 0);
            }
            // diagonal-column lo parts of all four versions at once: D' = A_hi Blo^T
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kofs = (ks & 3) * 32;
                mma_bf16(tmem + kTDiag, dA + (((ks >> 2) * 16384 + kofs) >> 4),
                         dBl + (((ks >> 2) * 8192 + kofs) >> 4), id64, ks > 0);
            }
            mma_commit(mma_bar);
        }

        // ---- while the Gram MMAs run: the globally scaled operands of the later products,
        //      Gam*Q and K*gamma^C/Gam (package, for the state kernel) and Gam*K (W = M Gam K)
        {
        uint8_t* pkg = item_pkg();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 4 * rg + i;
            const bool ok = r < itL;
            const uint32_t o64 = cofs + sw128_chunk(r, cg & 7);
            float qv[8], kv[8], eg[8], ek[8], t[8];
            ld8(qk + kOffQ + o64, qv);
            ld8(qk + kOffK + o64, kv);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (!ok) { qv[e] = 0.f; kv[e] = 0.f; }
                eg[e] = ex2f(G[i][e]);           // e^{G_r}
                ek[e] = ex2f(gl[e] - G[i][e]);   // e^{G_last - G_r}
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) t[e] = qv[e] * eg[e];
            *reinterpret_cast<uint4*>(pkg + kPkgStk + (cg >> 3) * kPkgStkBlk + kPkgStkQ +
                                      sw128_chunk(r, cg & 7)) = pk8(t);     // Gam*Q
#pragma unroll
            for (int e = 0; e < 8; ++e) t[e] = kv[e] * ek[e];
            {
                uint4 hi, lo;
                pk8_hilo(t, hi, lo);
                *reinterpret_cast<uint4*>(pkg + kPkgKT + o64) = hi;        // K*gamma^C/Gam
                *reinterpret_cast<uint4*>(pkg + kPkgKTLo + o64) = lo;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) t[e] = kv[e] * eg[e];
            *reinterpret_cast<uint4*>(sm + kKbar + o64) = pk8(t);         // Gam*K
        }
        }

        if (!mbar_wait(mma_bar, mma_phase & 1, p.err)) s_abort = 1;
        ++mma_phase;
        tc_fence_after();
        KDA_PHASE(3);

        // ---- Gram epilogue: q-side rows -> A tile (bf16 hi + lo), k-side rows -> L (fp32).
        //      TMEM lane m = 32 (warp % 4) + lane; the groups of 16 columns a lane quadrant
        //      needs are split between the two warpgroups.
        {
            const int quad = warp & 3, wg = warp >> 2;
            const int m = 32 * quad + lane;
            const int side = m >> 6, r = m & 63, s = r >> 4;
            float* sL = reinterpret_cast<float*>(sm + kSL);
            uint8_t* aq = sm + kAqkTile;
            // rows 0..31 of a side need groups 0..2 (versions 0, 1); rows 32..63 groups 3..9
            const int g_lo = (quad & 1) ? (wg ? 7 : 3) : (wg ? 2 : 0);
            const int g_hi = (quad & 1) ? (wg ? 10 : 7) : (wg ? 3 : 2);
            for (int g = g_lo; g < g_hi; ++g) {
                float v[16], vl[16], vd[16];
                const int sg = (g == 0) ? 0 : (g < 3) ? 1 : (g < 6) ? 2 : 3;
                const int ib = 16 * g - kStkOff[sg];
                const bool diag = (ib == 16 * sg);  // this group holds version sg's own sub-tile
                tmem_ld16(tmem + lane_base + 16 * g, v);
                tmem_ld16(tmem + lane_base + kTLo + 16 * g, vl);
                if (diag) tmem_ld16(tmem + lane_base + kTDiag + 16 * sg, vd);
                tmem_ld_wait();
                if (diag)
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] += vd[e];
                if (sg == s) {
                    if (side == 0) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            float a8[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int j0 = 8 * hf + e;
                                a8[e] = (ib + j0 <= r) ? v[j0] + vl[j0] : 0.f;
                            }
                            uint4 hi, lo;
                            pk8_hilo(a8, hi, lo);
                            *reinterpret_cast<uint4*>(aq + sw128_chunk(r, (ib >> 3) + hf)) = hi;
                            *reinterpret_cast<uint4*>(sm + kAqkLoTile +
                                                      sw128_chunk(r, (ib >> 3) + hf)) = lo;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            sL[r * kLd + ib + e] = (ib + e < r) ? v[e] : 0.f;
                    }
                }
            }
            if (side == 0 && wg == 0)  // columns past this sub-tile's version are zero
                for (int ch = 2 * (s + 1); ch < 8; ++ch) {
                    *reinterpret_cast<uint4*>(aq + sw128_chunk(r, ch)) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4*>(sm + kAqkLoTile + sw128_chunk(r, ch)) =
                        make_uint4(0, 0, 0, 0);
                }
        }
        tc_fence_before();
        intra_sync();
        KDA_PHASE(4);
        if (s_abort) break;

        // ---- T = (I + L)^{-1}: 16x16 diagonal blocks by forward substitution, then the
        //      off-diagonal blocks by distance: T_ss' = -T_ss * sum_{t=s'}^{s-1} L_st T_ts'
        {
            const float* sL = reinterpret_cast<const float*>(sm + kSL);
            float* sT = reinterpret_cast<float*>(sm + kST);
            float* sScr = reinterpret_cast<float*>(sm + kSolveScr);
            solve_tril64(sL, sT, sScr, warp, iter);
            KDA_PHASE(8);
            // M = T Diag(beta) (lower triangle) as a bf16 K-major tile, written twice: the
            // 128-row operand [M; M] of the W / U MMA
            {
                const int r = tid >> 2, cq = tid & 3;
                uint8_t* mt = sm + kMTile;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t pw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i0 = 16 * cq + 8 * hf + 2 * e;
                        const float m0 = (i0 <= r) ? sT[r * kLd + i0] * sBeta[i0] : 0.f;
                        const float m1 =
                            (i0 + 1 <= r) ? sT[r * kLd + i0 + 1] * sBeta[i0 + 1] : 0.f;
                        pw[e] = pack_bf16x2(m0, m1);
                    }
                    const uint4 pk = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                    *reinterpret_cast<uint4*>(mt + sw128_chunk(r, 2 * cq + hf)) = pk;
                    *reinterpret_cast<uint4*>(mt + 8192 + sw128_chunk(r, 2 * cq + hf)) = pk;
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        intra_sync();
        KDA_PHASE(5);

        // ---- W = M (Gam K) and U = M V: A = [M; M] (rows 64..127 repeat rows 0..63, so
        //      every TMEM lane quadrant holds a copy of the 64 rows), N = 128 channels each
        if (mbar_wait(v_bar, iter & 1, p.err)) {
            if (tid == kIss) pend_v = -1;
        } else {
            s_abort = 1;
        }
        if (tid == kIss) {
            tc_fence_after();
            constexpr uint32_t idesc = idesc_bf16(128, 128, false, true);
            const uint64_t dM = sdesc_sw128(sbase + kMTile, 0, 1024);
            const uint64_t dK = sdesc_sw128(sbase + kKbar, 8192, 1024);
            const uint64_t dV = sdesc_sw128(sbase + kVBuf, 8192, 1024);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t am = dM + ((ks * 32) >> 4);
                mma_bf16(tmem, am, dK + ((ks * 2048) >> 4), idesc, ks > 0);
                mma_bf16(tmem + 128, am, dV + ((ks * 2048) >> 4), idesc, ks > 0);
            }
            mma_commit(mma_bar);
        }
        if (!mbar_wait(mma_bar, mma_phase & 1, p.err)) s_abort = 1;
        ++mma_phase;
        tc_fence_after();
        {
            // lane quadrants 0, 1: W rows (bf16), quadrants 2, 3: U rows (fp32); the
            // warpgroup picks the 64-column half.  Both are staged in shared memory in
            // their package layout (W in this item's q slot, U in the B-stack region) and
            // leave by bulk copies.
            const int quad = warp & 3, wg = warp >> 2;
            const int r = 32 * (quad & 1) + lane;
            float v[4][16];
            const uint32_t col = (quad < 2 ? 0u : 128u) + 64 * wg;
#pragma unroll
            for (int g = 0; g < 4; ++g) tmem_ld16(tmem + lane_base + col + 16 * g, v[g]);
            tmem_ld_wait();
            if (quad < 2) {
                uint8_t* dst = qk + kOffQ + wg * 8192;
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        float v8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v8[e] = v[g][8 * hf + e];
                        *reinterpret_cast<uint4*>(dst + sw128_chunk(r, 2 * g + hf)) = pk8(v8);
                    }
            } else {
                // columns [64 wg + 4 cidx, +4): quarter 2 wg + (cidx >> 3), chunk cidx & 7
                uint8_t* urow = sm + kBStk + 2 * wg * kPkgUQ + r * 128;
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int cidx = 4 * g + q;
                        *reinterpret_cast<float4*>(urow + (cidx >> 3) * kPkgUQ +
                                                   (((cidx & 7) ^ (r & 7)) << 4)) =
                            make_float4(v[g][4 * q], v[g][4 * q + 1], v[g][4 * q + 2],
                                        v[g][4 * q + 3]);
                    }
            }
        }
        fence_async_smem();
        tc_fence_before();
        intra_sync();
        KDA_PHASE(6);
        if (s_abort) break;
        if (tid == kIss && has_next) {  // v is consumed: fetch the next item's
            load_tiles(&p.tv, sm + kVBuf, nullptr, nullptr, s_item[b ^ 1], v_bar);
            pend_v = (iter + 1) & 1;
        }
        if (tid == kIss) {
            uint8_t* pkg = item_pkg();
            bulk_s2g(pkg + kPkgStk, qk + kOffQ, 8192);                     // W, channels 0..63
            bulk_s2g(pkg + kPkgStk + kPkgStkBlk, qk + kOffQ + 8192, 8192);  // W, channels 64..127
            bulk_s2g(pkg + kPkgU, sm + kBStk, kPkgUBytes);                  // U
            bulk_s2g(pkg + kPkgAQK, sm + kAqkTile, 16384);                  // A hi and lo
            bulk_commit();
            if (p.fused_C) {
                pub_slot = (int)s_item[b].pkg;
                pub_val = (uint32_t)s_item[b].ft + 1;
            }
            lead_next = next2;
        }
    }
    KDA_PHASE_FLUSH();
    // teardown: stores complete (the last package published), no load in flight, TMEM
    // released
    if (tid == kIss) {
        bulk_wait0();
        if (p.fused_C && pub_slot >= 0 && !s_abort) {
            fence_proxy_async_global();
            st_release_gpu(p.ready + pub_slot, pub_val);
        }
        if (s_abort) {
            for (int q = 0; q < 2; ++q)
                if (pend_q[q] >= 0) mbar_wait(&qk_bar[q], pend_q[q], nullptr);
            if (pend_v >= 0) mbar_wait(v_bar, pend_v, nullptr);
            if (pend_z >= 0) mbar_wait(z_bar, pend_z, nullptr);
            mma_commit(mma_bar);  // arrives once every MMA issued so far has completed
            mbar_wait(mma_bar, mma_phase & 1, nullptr);
        }
    }
    tc_fence_before();
    intra_sync();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}


}  // namespace
}  // namespace fwdtc
}  // namespace kda
