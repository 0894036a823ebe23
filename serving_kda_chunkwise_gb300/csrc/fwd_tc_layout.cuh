// fwd_tc_layout.cuh -- what the two stages of the tensor-core chunked forward share: the
// per-(head, chunk) "package" the intra-chunk stage writes and the state-chain stage reads,
// the workspace layout, and the chain stage's launcher.
//
// Method ("Kimi k3 技术报告详解（1）——架构再升华", section "Chunkwise parallel form"): per
// chunk of C = 64 tokens, with G[r] = sum_{s<=r} g_s per key channel and gamma = e^G,
//   M = (I + StrictTril(Diag(beta)(Gamma*K)(K/Gamma)^T))^{-1} Diag(beta),
//   W = M (Gamma*K),  U = M V,  A = Tril((Gamma*Q)(K/Gamma)^T),
//   Vt = U - W S,  O = (Gamma*Q) S + A Vt,  S <- Diag(gamma^C) S + (K*gamma^C/Gamma)^T Vt.
// The package holds everything of one chunk that the chain needs and that does not depend
// on S: [W; Gamma*Q], K~ = K*gamma^C/Gamma (bf16 hi + lo), A (bf16 hi + lo), gamma^C and
// U (fp32).  Its bytes are the images of the chain kernel's shared-memory operand tiles, so
// the chain stage moves them with plain bulk copies.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {
namespace fwdtc {

constexpr int kC = 64;    // chunk length
constexpr int kD = 128;   // head dim (dk = dv)

// ---- package (per head and chunk) ----
// part A: the row stack [W; Gamma*Q] (B operand of the chain's first product), K-major
// 128-byte swizzle, two 64-channel blocks of 16 KB, each W rows 0..63 then Gamma*Q rows
// 0..63 (128 B per row)
constexpr uint32_t kPkgStk = 0;
constexpr uint32_t kPkgStkBlk = 16384;
constexpr uint32_t kPkgStkQ = 8192;   // Gamma*Q rows within a block
constexpr uint32_t kPkgPartA = 32768;
// K~ = K*gamma^C/Gamma as bf16 hi then lo, each [2 channel blocks][64 r][128 B] (MN-major
// with channels contiguous)
constexpr uint32_t kPkgKT = 32768;
constexpr uint32_t kPkgKTLo = 49152;
constexpr uint32_t kPkgKTBytes = 32768;
// A = Tril((Gamma*Q)(K/Gamma)^T) as bf16 hi then lo, each [64 r][64 i] K-major 128-byte swizzle
constexpr uint32_t kPkgAQK = 65536;
constexpr uint32_t kPkgAQKLo = 73728;
constexpr uint32_t kPkgAQKBytes = 16384;
constexpr uint32_t kPkgG = 81920;     // gamma^C [128] fp32
constexpr uint32_t kPkgGBytes = 512;
// U = M V in fp32: four quarters of 32 value columns, each [64 r][32 j] with the 16-byte
// chunk c of row r at chunk position c ^ (r & 7)
constexpr uint32_t kPkgU = 82432;
constexpr uint32_t kPkgUQ = 8192;
constexpr uint32_t kPkgUBytes = 4 * kPkgUQ;
constexpr uint32_t kPkgBytes = kPkgU + kPkgUBytes;  // 115200
static_assert(kPkgBytes % 16 == 0 && kPkgU % 16 == 0, "bulk copies need 16-byte alignment");

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---- workspace: chunk offsets [N + 1], chunk table [maxchunks] (int4), sequence order
// [N] (longest first), then the packages [H][maxchunks] ----
struct WsLayout {
    size_t off_chunk_off, off_tab, off_order, off_pkg, total;
};
inline WsLayout ws_layout(int64_t T_total, int N, int H) {
    const size_t maxchunks = (size_t)(T_total / kC + N);
    WsLayout l;
    l.off_chunk_off = 0;
    l.off_tab = align_up((size_t)(N + 1) * sizeof(int32_t), 1024);
    l.off_order = l.off_tab + align_up(maxchunks * 16, 1024);
    l.off_pkg = l.off_order + align_up((size_t)N * sizeof(int32_t), 1024);
    l.total = l.off_pkg + (size_t)H * maxchunks * kPkgBytes;
    return l;
}

// [T_total, H, d] bf16 tensor map (d = 64 or 128) with boxes of `box_cols` columns x 1 head
// x 64 rows: 64-column boxes use the 128-byte swizzle, 32-column boxes the 64-byte swizzle,
// 128-column boxes none (fwd_tc.cu).  Columns past d read as zero.
bool make_map(CUtensorMap* m, const void* base, int64_t T_total, int H, int d, int box_cols);

}  // namespace fwdtc
}  // namespace kda
