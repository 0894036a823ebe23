// bwd_tc_layout.cuh -- the per-(chunk, head) blocks the tensor-core backward hands between its
// stages (bf16 problems).
//
// The reverse of the chunk form ("Kimi k3 技术报告详解（1）——架构再升华", section "Chunkwise
// parallel form"; the pages print no backward, these are the derivatives of the forward they
// define), per chunk with start state S_0, end gradient dS_C, output gradient dO and
// Gamma = e^G, K+ = Gamma*K, M = N Diag(beta), N = (I + L)^{-1}:
//   dVt = A^T dO + K~ dS_C            (serial, in the gradient chain)
//   dA  = Tril(dO Vt^T),  dV = M^T dVt,  Y = V - K+ S_0,  dM = dVt Y^T,
//   X0  = N^T dM,  dbeta_s = X0_ss + sum_i K_si E_si,  dL = -StrictTril(X0 M^T),
//   dQ  = Gamma*(dO S_0^T) + D(dA, K),   E = D(dL, K),   F = D^T(dA, Q) + D^T(Diag(beta) dL, K),
//   dK  = -Gamma*(dV S_0^T) + Diag(beta) E + F + (gamma^C/Gamma)*(Vt dS_C^T),
// with the decayed products D(X, Y)_ri = sum_{s<=r} X_rs Y_si e^{G_ri - G_si} and
// D^T(X, Y)_si = sum_{r>=s} X_rs Y_ri e^{G_ri - G_si}; then dG, its reverse cumulative sum
// and the gate's derivative.
//
// Stage blocks (all bf16 images are 128-byte-swizzled tiles of 128-byte rows: the 16-byte
// chunk c of row x sits at chunk position c ^ (x & 7)):
//  * the "image" block, written by the forward's chain (S_0, Vt), the gradient chain (dS_C,
//    dVt) and the intra stage (N), read by the state kernel:
//      S_0^T hi, lo   [2 blocks of 64 key channels][128 value rows j][128 B]   (i contiguous)
//      Vt^T hi, lo    [128 value rows j][128 B]                                (r contiguous)
//      dS_C^T hi, lo  [2 blocks of 64 key channels][128 value rows j][128 B]
//      dVt^T hi, lo   [128 value rows j][128 B]                                (r contiguous)
//      N              fp32 [64][64] row-major, lower triangle with unit diagonal
//  * the "mid" block, written by the state kernel, read by the decay kernel:
//      pQ  = Gamma*(dO S_0^T),  pP = -Gamma*(dV S_0^T),  pE = (gamma^C/Gamma)*(Vt dS_C^T):
//            fp32 [64 tokens][128 key channels] each
//      dA, dL images (hi, lo): [64 rows s][128 B], entry (s, 63 - r) = X_rs (columns in
//            reversed token order)
//      dbeta1 fp32 [64]: X0_ss;   rs fp32 [128]: sum_j dS_C_ij S_0_ij
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace kda {
namespace bwdtc {

// image block
constexpr uint32_t kBiS = 0;            // S_0^T hi, lo at + 32768
constexpr uint32_t kBiV = 65536;        // Vt^T hi, lo at + 16384
constexpr uint32_t kBiDS = 98304;       // dS_C^T hi, lo at + 32768
constexpr uint32_t kBiDV = 163840;      // dVt^T hi, lo at + 16384
constexpr uint32_t kBiN = 196608;       // N fp32
constexpr uint32_t kBiBytes = 212992;

// mid block
constexpr uint32_t kMdQ = 0;
constexpr uint32_t kMdP = 32768;
constexpr uint32_t kMdE = 65536;
constexpr uint32_t kMdA = 98304;        // dA hi, lo at + 8192
constexpr uint32_t kMdL = 114688;       // dL hi, lo at + 8192
constexpr uint32_t kMdB = 131072;       // dbeta1
constexpr uint32_t kMdRs = 131328;      // rs
constexpr uint32_t kMdBytes = 131840;
static_assert(kMdBytes % 16 == 0 && kBiBytes % 1024 == 0, "stage blocks must stay aligned");

}  // namespace bwdtc
}  // namespace kda
