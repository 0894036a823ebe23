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

#include "bwd_tc_layout.cuh"
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
    // two-launch form, optional (nullptr otherwise): the backward's image blocks
    // [chunks][H] (bwd_tc_layout.cuh); item = chunk * H + h writes N = (I + L)^{-1} there
    uint8_t* bimg;
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

// Gate kinds.  kGateBounded: g = g_min Sigmoid(e^{A_h} z).  kGateSoftplus: the gate the bound
// replaces, g = -e^{A_h} Softplus(z), on the mixed path of the same page and section: with
// no bound, a sub-tile's decay can exceed the exponent range, so every factor must stay
// <= 1.  The reference of sub-tile s is then G at its start (rho_s = G_{16 s - 1}, rho_0 = 0):
// the row factor e^{G_r - rho_s} (r in sub-tile s) and the column operand
// k_i e^{rho_s - G_i} (i < 16 s) are both <= 1, so the off-diagonal sub-tile pairs stay on
// the tensor cores (three column versions, s = 1..3, 96 stack rows), while the diagonal
// 16 x 16 blocks, where no such split exists, are formed per pair on CUDA cores as
// sum_c q_rc k_ic e^{G_rc - G_ic} (exponent <= 0), during the Gram MMAs.
constexpr int kGateBounded = 0, kGateSoftplus = 1;
// B-stack block stride (two 64-channel blocks): 160 rows, or 96 on the mixed path
template <int kGate>
__device__ __forceinline__ constexpr uint32_t stk_blk() { return kGate == kGateBounded ? 20480u : 12288u; }
// mixed path: the stack row offset of version s = 1..3 (0, 16, 48)
__device__ __forceinline__ int stk_off_sp(int s) { return 8 * s * (s - 1); }
// mixed path: G (fp32 [64 rows][128]) during the Gram MMAs, then the diagonal blocks
// A_d, L_d (fp32 [4 sub-tiles][16][16] each); the 32 KB after the 96-row stack
constexpr uint32_t kSpXch = kBStk + 24576;
static_assert(kSpXch + 32768 <= kXch, "the mixed path's exchange must fit before rho");

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

// The gate in log2 units (G2 = G log2 e, so that every decay factor is one ex2).
//   bounded:  g_min Sigmoid(e^{A_h} z) log2 e = gmin2 / (1 + 2^{-scale2 z}),
//             scale2 = e^{A_h} log2 e, gmin2 = g_min log2 e;
//   softplus: -e^{A_h} Softplus(z) log2 e = -eA (max(z, 0) log2 e + log2(1 + 2^{-|z| log2 e})),
//             eA = e^{A_h}; z = -inf gives -0 (alpha = 1), z must be finite otherwise.
template <int kGate>
__device__ __forceinline__ float gate2(float z, float scale2, float gmin2, float eA) {
    if constexpr (kGate == kGateBounded) {
        return __fdividef(gmin2, 1.f + ex2f(-scale2 * z));
    } else {
        constexpr float kLog2e = 1.4426950408889634f;
        return -eA * fmaf(fmaxf(z, 0.f), kLog2e, lg2f(1.f + ex2f(-fabsf(z) * kLog2e)));
    }
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

// Mixed path: the diagonal 16 x 16 blocks of both Grams, per pair on CUDA cores.  Thread
// (sub-tile ds, row pair dp, channel slice dsl) takes rows ra = 16 ds + dp and
// rb = 16 ds + 15 - dp (17 pairs together, the same for every thread) over the 16 channels
// [16 dsl, 16 dsl + 16); the 8 slices of a row pair are adjacent lanes and are summed by a
// reduce-scatter (each lane ends with 6 of the pair sums).  G comes from `xg` (fp32 [64][128],
// written by every thread); the blocks go to the same region afterwards: A_d at xg, L_d at
// xg + 1024 (fp32 [4][16][16], row-local index then column-local index; entries above the
// diagonal are not written).  Rows and columns at or past L read as zero.
__device__ __forceinline__ void diag_blocks(const uint8_t* qk, float* xg, const float* sBeta,
                                            int itL, int tid) {
    const int ds = tid >> 6, dp = (tid >> 3) & 7, dsl = tid & 7;
    const int ra = 16 * ds + dp, rb = 16 * ds + 15 - dp;
    float aA[8], aL[8], bA[16], bL[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        bA[j] = 0.f;
        bL[j] = 0.f;
        if (j < 8) {
            aA[j] = 0.f;
            aL[j] = 0.f;
        }
    }
#pragma unroll 1
    for (int hc = 0; hc < 2; ++hc) {
        const int c0 = 16 * dsl + 8 * hc;  // 8 channels: one 16-byte chunk of a tile row
        const uint32_t blk = (c0 >> 6) * 8192;
        const int chk = (c0 & 63) >> 3;
        float qa[8], ka[8], qb[8], kb[8], Ga[8], Gb[8];
        ld8(qk + kOffQ + blk + sw128_chunk(ra, chk), qa);
        ld8(qk + kOffK + blk + sw128_chunk(ra, chk), ka);
        ld8(qk + kOffQ + blk + sw128_chunk(rb, chk), qb);
        ld8(qk + kOffK + blk + sw128_chunk(rb, chk), kb);
        {
            const float4* pa = reinterpret_cast<const float4*>(xg + ra * 128 + c0);
            const float4* pb = reinterpret_cast<const float4*>(xg + rb * 128 + c0);
            const float4 a0 = pa[0], a1 = pa[1], b0 = pb[0], b1 = pb[1];
            Ga[0] = a0.x; Ga[1] = a0.y; Ga[2] = a0.z; Ga[3] = a0.w;
            Ga[4] = a1.x; Ga[5] = a1.y; Ga[6] = a1.z; Ga[7] = a1.w;
            Gb[0] = b0.x; Gb[1] = b0.y; Gb[2] = b0.z; Gb[3] = b0.w;
            Gb[4] = b1.x; Gb[5] = b1.y; Gb[6] = b1.z; Gb[7] = b1.w;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (ra >= itL) { qa[e] = 0.f; ka[e] = 0.f; }
            if (rb >= itL) { qb[e] = 0.f; kb[e] = 0.f; }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int i = 16 * ds + j;
            float ki[8], Gi[8];
            ld8(qk + kOffK + blk + sw128_chunk(i, chk), ki);
            {
                const float4* pi = reinterpret_cast<const float4*>(xg + i * 128 + c0);
                const float4 i0 = pi[0], i1 = pi[1];
                Gi[0] = i0.x; Gi[1] = i0.y; Gi[2] = i0.z; Gi[3] = i0.w;
                Gi[4] = i1.x; Gi[5] = i1.y; Gi[6] = i1.z; Gi[7] = i1.w;
            }
            const bool live = i < itL;
            if (j <= 15 - dp) {  // i <= rb
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float kf = live ? ki[e] * ex2f(Gb[e] - Gi[e]) : 0.f;
                    bA[j] = fmaf(qb[e], kf, bA[j]);
                    bL[j] = fmaf(kb[e], kf, bL[j]);
                }
            }
            if (j < 8) {
                if (j <= dp) {  // i <= ra
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float kf = live ? ki[e] * ex2f(Ga[e] - Gi[e]) : 0.f;
                        aA[j] = fmaf(qa[e], kf, aA[j]);
                        aL[j] = fmaf(ka[e], kf, aL[j]);
                    }
                }
            }
        }
    }
    // reduce-scatter over the 8 slices: values [bA 16 | bL 16 | aA 8 | aL 8]; after the
    // rounds with lane masks 4, 2, 1 the lane with slice bits (b2 b1 b0) holds the sums of
    // values 24 b2 + 12 b1 + 6 b0 + u, u < 6
    float V[48];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        V[j] = bA[j];
        V[16 + j] = bL[j];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        V[32 + j] = aA[j];
        V[40 + j] = aL[j];
    }
    const bool b2 = (dsl >> 2) & 1, b1 = (dsl >> 1) & 1, b0 = dsl & 1;
    float W1[24], W2[12], W3[6];
#pragma unroll
    for (int t = 0; t < 24; ++t)
        W1[t] = (b2 ? V[24 + t] : V[t]) + __shfl_xor_sync(0xffffffffu, b2 ? V[t] : V[24 + t], 4);
#pragma unroll
    for (int t = 0; t < 12; ++t)
        W2[t] = (b1 ? W1[12 + t] : W1[t]) + __shfl_xor_sync(0xffffffffu, b1 ? W1[t] : W1[12 + t], 2);
#pragma unroll
    for (int t = 0; t < 6; ++t)
        W3[t] = (b0 ? W2[6 + t] : W2[t]) + __shfl_xor_sync(0xffffffffu, b0 ? W2[t] : W2[6 + t], 1);
    intra_sync();  // every thread has read G: the region takes the blocks
    float* dA = xg;
    float* dL = xg + 1024;
#pragma unroll
    for (int u = 0; u < 6; ++u) {
        const int idx = 24 * b2 + 12 * b1 + 6 * b0 + u;
        const bool rowb = idx < 32;
        const bool isL = rowb ? idx >= 16 : idx >= 40;
        const int j = rowb ? (idx & 15) : (idx - 32) & 7;
        const int rl = rowb ? 15 - dp : dp;
        const int o = (16 * ds + rl) * 16 + j;
        if (isL)
            dL[o] = (j < rl) ? W3[u] * sBeta[16 * ds + rl] : 0.f;
        else
            dA[o] = W3[u];
    }
    intra_sync();  // the blocks are complete
}

template <int kGate>
__device__ __forceinline__ void intra_body(const IntraParams& p, uint8_t* smem_raw, int cta, int ncta) {
    constexpr uint32_t kStkBlk = stk_blk<kGate>();
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
    int4 raw_lead;  // issuing thread: lead_next's chunk-table entry, fetched when it is taken
    if (tid == kIss) {
        const int first_item = take_item(p, -1, cta, ncta);
        s_item[0].item = first_item;
        if (first_item < n_items) lead_next = take_item(p, first_item, cta, ncta);
        if (lead_next < n_items) raw_lead = fetch_item(p, lead_next);
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
        // the next item, known to the issuing thread (which took it and fetched its table
        // entry one item ago) and needed by its warp only: the issuing thread publishes it
        // now (read after the next CTA barrier) and the warp loads its beta, a whole gate
        // phase ahead of the store into its slot.  The item after it is taken and its
        // entry fetched now.
        const int next = warp == (kIss >> 5) ? __shfl_sync(0xffffffffu, lead_next, kIss & 31) : n_items;
        const bool has_next = next < n_items;
        int next2 = n_items;
        unsigned short beta_nx[2] = {0, 0};  // issuing thread's warp: the next item's beta (bf16)
        float alog_nx = 0.f;                 // issuing thread: the next item's A_log
        if (warp == (kIss >> 5)) {
            if (tid == kIss) {
                if (has_next) {
                    const ItemInfo nx = decode_item(p, next, raw_lead);
                    s_item[b ^ 1] = nx;
                    alog_nx = ld_ahead(p.A_log + nx.h);
                    next2 = take_item(p, next, cta, ncta);
                    if (next2 < n_items) raw_lead = fetch_item(p, next2);
                } else {
                    s_item[b ^ 1].item = n_items;  // no further item
                }
            }
            __syncwarp();
            if (has_next) {
                const ItemInfo& nxs = s_item[b ^ 1];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int r = lane + 32 * h2;
                    if (r < nxs.L)
                        beta_nx[h2] = ld_ahead(p.beta + (size_t)(nxs.t0 + r) * p.H + nxs.h);
                }
            }
        }
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
            const float eA = expf(alog);
            const float scale2 = eA * 1.4426950408889634f;  // e^{A_log} log2 e
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
                    const float g = gate2<kGate>(zz[e], scale2, gmin2, eA);
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
        // z is consumed: the issuing thread fetches the next item's z (issued here, where a
        // long phase follows, so that a slow issue never holds up a barrier)
        if (tid == kIss && has_next) {
            load_tiles(&p.tz, sm + kZBuf, nullptr, nullptr, s_item[b ^ 1], z_bar);
            pend_z = (iter + 1) & 1;
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
        if constexpr (kGate == kGateBounded) {
            if ((rg & 3) == 1)  // rows 4 rg + 3 = 16 s + 7: the reference of sub-tile s
#pragma unroll
                for (int e = 0; e < 8; ++e) xrho[sub * 128 + ch0 + e] = G[3][e];
        } else {
            if ((rg & 3) == 3 && sub < 3)  // row 16 (s + 1) - 1: the reference of sub-tile s + 1
#pragma unroll
                for (int e = 0; e < 8; ++e) xrho[(sub + 1) * 128 + ch0 + e] = G[3][e];
            if (rg == 0)  // sub-tile 0 starts at the chunk start
#pragma unroll
                for (int e = 0; e < 8; ++e) xrho[ch0 + e] = 0.f;
        }
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

        // ---- decay-scaled operands.  Row r of sub-tile s uses e1 = e^{G_r - rho_s}.
        //      Bounded gate: the column operand of version s2 >= s is k_r e^{rho_s2 - G_r},
        //      own version hi + lo.  Mixed path: versions s2 > s only, k_r e^{rho_s2 - G_r}
        //      formed as e^{rho_{s+1} - G_r} e^{rho_s2 - rho_{s+1}} (both factors <= 1).
        {
            // Ev[v][e] = e^{rho_{s2} - rho_b} for the later sub-tiles s2 = sub + 1 + v, with
            // rho_b = rho_s (bounded) or rho_{s+1} (mixed); <= 1 and may underflow to 0,
            // which drops Gram terms below e^-13 of their neighbours (bounded gate) or terms
            // whose true factor underflows too (mixed path)
            float rho[8], rhob[8], Ev[3][8];
            const int sb = kGate == kGateBounded ? sub : min(sub + 1, 3);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                rho[e] = xrho[sub * 128 + ch0 + e];  // (log2 units, as G)
                rhob[e] = kGate == kGateBounded ? rho[e] : xrho[sb * 128 + ch0 + e];
            }
#pragma unroll
            for (int v = 0; v < 3; ++v) {
                const int s2 = min(sub + 1 + v, 3);  // entries past sub-tile 3 are unused
#pragma unroll
                for (int e = 0; e < 8; ++e) Ev[v][e] = ex2f(xrho[s2 * 128 + ch0 + e] - rhob[e]);
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
                    dc[e] = ex2f(rhob[e] - G[i][e]);
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
                if constexpr (kGate == kGateBounded) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) t[e] = kv[e] * dc[e];
                    pk8_hilo(t, hi, lo);
                    *reinterpret_cast<uint4*>(sm + kBStk + (cg >> 3) * kStkBlk +
                                              sw128_chunk(kStkOff[sub] + r, cg & 7)) = hi;
                    *reinterpret_cast<uint4*>(sm + kBLo + o64) = lo;
                }
#pragma unroll
                for (int v = 0; v < 3; ++v) {
                    const int s2 = sub + 1 + v;
                    if (s2 < 4) {  // uniform within a warp
#pragma unroll
                        for (int e = 0; e < 8; ++e) t[e] = kv[e] * dc[e] * Ev[v][e];
                        const int srow = kGate == kGateBounded ? kStkOff[s2] : stk_off_sp(s2);
                        *reinterpret_cast<uint4*>(sm + kBStk + (cg >> 3) * kStkBlk +
                                                  sw128_chunk(srow + r, cg & 7)) = pk8(t);
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
            // N = the stack's rows: 160 (four versions) or 96 (mixed path: three)
            constexpr uint32_t idN = idesc_bf16(128, kGate == kGateBounded ? 160 : 96, false, false);
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
                const uint64_t bh = dB + (((ks >> 2) * kStkBlk + kofs) >> 4);
                mma_bf16(tmem, ah, bh, idN, ks > 0);
                mma_bf16(tmem + kTLo, dAl + (((ks >> 2) * 8192 + kofs) >> 4), bh, idN, ks > 0);
            }
            if constexpr (kGate == kGateBounded) {
                // diagonal-column lo parts of all four versions at once: D' = A_hi Blo^T
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kofs = (ks & 3) * 32;
                    mma_bf16(tmem + kTDiag, dA + (((ks >> 2) * 16384 + kofs) >> 4),
                             dBl + (((ks >> 2) * 8192 + kofs) >> 4), id64, ks > 0);
                }
            }
            mma_commit(mma_bar);
        }

        // ---- while the Gram MMAs run: the globally scaled operands of the later products,
        //      Gam*Q and K*gamma^C/Gam (package, for the chain stage) and Gam*K (W = M Gam K)
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

        // the next item's beta and A_log into their slots (loaded at the top of the loop;
        // stored here, where a late load holds up no barrier)
        if (warp == (kIss >> 5)) {
            float* dst = reinterpret_cast<float*>(sm + kBeta) + 64 * (b ^ 1);
            dst[lane] = __bfloat162float(__ushort_as_bfloat16(beta_nx[0]));
            dst[lane + 32] = __bfloat162float(__ushort_as_bfloat16(beta_nx[1]));
            if (lane == 0) s_alog[b ^ 1] = alog_nx;
        }

        // ---- mixed path, while the Gram MMAs run: the diagonal 16 x 16 blocks per pair,
        //      A_d[r][i] = sum_c q_rc k_ic 2^{G_rc - G_ic} (i <= r) and
        //      L_d[r][i] = beta_r sum_c k_rc k_ic 2^{G_rc - G_ic} (i < r), r, i in one sub-tile
        if constexpr (kGate == kGateSoftplus) {
            float* xg = reinterpret_cast<float*>(sm + kSpXch);  // G [64][128]
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float4* d = reinterpret_cast<float4*>(xg + (4 * rg + i) * 128 + ch0);
                d[0] = make_float4(G[i][0], G[i][1], G[i][2], G[i][3]);
                d[1] = make_float4(G[i][4], G[i][5], G[i][6], G[i][7]);
            }
            intra_sync();
            diag_blocks(qk, xg, sBeta, itL, tid);
        }

        if (!mbar_wait(mma_bar, mma_phase & 1, p.err)) s_abort = 1;
        ++mma_phase;
        tc_fence_after();
        KDA_PHASE(3);

        // ---- Gram epilogue: q-side rows -> A tile (bf16 hi + lo), k-side rows -> L (fp32).
        //      TMEM lane m = 32 (warp % 4) + lane; the groups of 16 columns a lane quadrant
        //      needs are split between the two warpgroups.
        if constexpr (kGate == kGateBounded) {
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
        } else {
            // mixed path: version s (of rows in sub-tile s = 1..3) holds columns i < 16 s in
            // TMEM groups gbase(s) + i / 16 (gbase = 0, 1, 3); the diagonal block comes from
            // the per-pair pass.  Groups by warp: lane quadrants 0 / 2 (rows 0..31 of a side)
            // need group 0, quadrants 1 / 3 (rows 32..63) groups 1..5; warpgroup 0 takes
            // groups 0..3, warpgroup 1 groups 4, 5 and the diagonal blocks.
            const int quad = warp & 3, wg = warp >> 2;
            const int m = 32 * quad + lane;
            const int side = m >> 6, r = m & 63, s = r >> 4, rl = r & 15;
            float* sL = reinterpret_cast<float*>(sm + kSL);
            uint8_t* aq = sm + kAqkTile;
            const int g_lo = (quad & 1) ? (wg ? 4 : 1) : 0;
            const int g_hi = (quad & 1) ? (wg ? 6 : 4) : (wg ? 0 : 1);
            for (int g = g_lo; g < g_hi; ++g) {
                float v[16], vl[16];
                const int sg = (g == 0) ? 1 : (g < 3) ? 2 : 3;
                const int ib = 16 * (g - stk_off_sp(sg) / 16);
                tmem_ld16(tmem + lane_base + 16 * g, v);
                tmem_ld16(tmem + lane_base + kTLo + 16 * g, vl);
                tmem_ld_wait();
                if (sg == s) {
                    if (side == 0) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            float a8[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) a8[e] = v[8 * hf + e] + vl[8 * hf + e];
                            uint4 hi, lo;
                            pk8_hilo(a8, hi, lo);
                            *reinterpret_cast<uint4*>(aq + sw128_chunk(r, (ib >> 3) + hf)) = hi;
                            *reinterpret_cast<uint4*>(sm + kAqkLoTile +
                                                      sw128_chunk(r, (ib >> 3) + hf)) = lo;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) sL[r * kLd + ib + e] = v[e];
                    }
                }
            }
            if (wg == 1) {  // the diagonal block of this row (masked and beta-scaled already
                            // for L; A masked here)
                const float* dA = reinterpret_cast<const float*>(sm + kSpXch) + (16 * s + rl) * 16;
                const float* dL = reinterpret_cast<const float*>(sm + kSpXch) + 1024 + (16 * s + rl) * 16;
                if (side == 0) {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        float a8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) a8[e] = (8 * hf + e <= rl) ? dA[8 * hf + e] : 0.f;
                        uint4 hi, lo;
                        pk8_hilo(a8, hi, lo);
                        *reinterpret_cast<uint4*>(aq + sw128_chunk(r, 2 * s + hf)) = hi;
                        *reinterpret_cast<uint4*>(sm + kAqkLoTile + sw128_chunk(r, 2 * s + hf)) = lo;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) sL[r * kLd + 16 * s + e] = (e < rl) ? dL[e] : 0.f;
                }
            }
            if (side == 0 && wg == 0)  // columns past the diagonal block are zero
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
                if (p.bimg) {  // N = T (lower triangle) in fp32 for the backward
                    float4* nd = reinterpret_cast<float4*>(
                        p.bimg + (size_t)s_item[b].item * bwdtc::kBiBytes + bwdtc::kBiN + r * 256 + 64 * cq);
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) {
                        const int c0 = 16 * cq + 4 * e4;
                        const float* tr = sT + r * kLd + c0;
                        nd[e4] = make_float4(c0 <= r ? tr[0] : 0.f, c0 + 1 <= r ? tr[1] : 0.f,
                                             c0 + 2 <= r ? tr[2] : 0.f, c0 + 3 <= r ? tr[3] : 0.f);
                    }
                }
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
