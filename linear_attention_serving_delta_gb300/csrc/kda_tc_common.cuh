// kda_tc_common.cuh -- record layout and helpers shared by the tensor-core
// intra-chunk (K2) and inter-chunk (K3) prefill kernels (bf16, dk = dv = 128,
// chunk 64).
//
// Chunked form of the recurrence (delta rule with a diagonal gate, "From KV
// Cache to Depth Attention", Technical Details; FlashKDA's unrolling in
// chunks, "Kimi K3: The Manos, The Mythos, The Legendos", bullet list).  For
// a chunk of L <= 64 tokens with start state S0, G_i = sum_{m<=i} log alpha_m
// per key channel and Gamma = exp(G):
//
//   Kp = K^ o Gamma,  Kn = K^ o Gamma^{-1},  Qp = Q^ o Gamma,  Kr = K^ o Gamma_L/Gamma
//   [A_kk ; A_qk] = [Kp ; Qp] Kn^T            (K2, tensor cores)
//   A_kk <- diag(beta) strict-lower(A_kk),   A_qk <- lower(A_qk)
//   Tb = (I + A_kk)^{-1} diag(beta)           (K2, CUDA cores)
//   [W | U~] = Tb [Kp | V]                    (K2, tensor cores)
//   per chunk, in order (K3):  U = U~ - W S0
//                              O = scale (Qp S0 + A_qk U)
//                              S_end = Diag(Gamma_L) S0 + Kr^T U
//
// Exponent range.  A_kk and A_qk need exp(G_i - G_j) for j <= i, formed by
// the tensor cores as the product of a row factor and a column factor.  K2
// keeps G in log2 units.  While a channel's total decay over the chunk G_L
// stays above 2^-120 the factors are referred to the chunk start: row
// factors 2^G_i <= 1 and column factors 2^-G_j <= 2^120.  Past that the
// channel takes a power-of-two reference s = round(G_L / 2) (half the
// chunk's decay): row factors 2^(G_i - s), column factors 2^(s - G_j), both
// inside 2^-126 .. 2^126 while G_L stays above 2^-250 (about e^-173).  Only
// MMA 1 sees these factors; the record keeps Qp, Kp and Kr referred to the
// chunk start (Gamma <= 1, so they can only underflow, which is harmless).
// A chunk past that range raises status flag 16 (its results are not
// reliable); the fp32 CUDA-core path (kda_simt.cu) has no such limit.
#pragma once

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace tcp {

constexpr uint32_t kD = 128;  // dk = dv on this path

// Record written by K2 for every (chunk, head) and read by K3, bytes.  The
// tiles are in the tcgen05 no-swizzle K-major operand layout (kda_tc.cuh), so
// K3 moves them into shared memory with single bulk copies.
//   AW  [128][128] bf16, R=128: rows 0-63 W, rows 64-127 Qp (K = key channel)
//   AK  [128][64]  bf16, MN-major (M = key channel, K = token): Kr^T
//   AQ  [64][64]   bf16, K-major, R=64: A_qk (row i, K = j).  K3 multiplies it
//       as rows 64-127 of an M=128 tile whose descriptor starts 1 KB early, so
//       the product lands in the accumulator lanes of the Qp S0 rows; rows
//       0-63 of that tile are whatever precedes it in shared memory and feed
//       accumulator lanes that are dead by then
//   UT  fp32, element (i, e) at ((e/4)*64 + i)*4 + e%4   (U~)
//   GL  [128] fp32: Gamma_L
struct Rec {
  static constexpr uint32_t AW = 0;
  static constexpr uint32_t AK = AW + 128 * 128 * 2;
  static constexpr uint32_t AQ = AK + 128 * 64 * 2;
  static constexpr uint32_t UT = AQ + 64 * 64 * 2;
  static constexpr uint32_t GL = UT + 64 * 128 * 4;
  static constexpr uint32_t BYTES = GL + 128 * 4;
  static constexpr uint32_t kAkSbo = 8 * 128;  // AK: 8 K-groups (64 tokens) per MN-group
};
static_assert(Rec::BYTES % 256 == 0, "records stay 256-byte aligned");

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t bf16_bits(float x) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// element j (0..7) of 8 bf16 packed in a uint4
__device__ __forceinline__ float bf16_at(const uint4& v, int j) {
  const uint32_t w = j < 2 ? v.x : j < 4 ? v.y : j < 6 ? v.z : v.w;
  return (j & 1) ? bf16_hi(w) : bf16_lo(w);
}

__device__ __forceinline__ void flag(int32_t* status, int32_t f) { atomicOr(status, f); }

// 2^x with the hardware approximation (ex2.approx: relative error about
// 2^-22), results below 2^-126 flushed to zero (every use keeps x >= -126 or
// needs no more than that)
__device__ __forceinline__ float exp2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;  // 1 / ln 2
// A chunk whose total decay in some channel is below 2^-kMaxChunkDecayLog2
// is past the range of the tensor-core operands (status flag 16)
constexpr float kMaxChunkDecayLog2 = 250.f;
// Below a total decay of 2^-kScaleFromLog2 in a channel, its factors are
// referred to half the chunk's decay instead of the chunk start
constexpr float kScaleFromLog2 = 120.f;

// log2 alpha = -softplus(g) / ln 2, softplus(g) = max(g, 0) + ln(1 + e^-|g|),
// with the fast base-2 exponential and logarithm (absolute error a few 1e-7
// per token; the operands it feeds are rounded to bf16).  g = -inf gives 0
// (alpha = 1), a large g gives -g / ln 2 without overflow.
__device__ __forceinline__ float log2_alpha_fast(float g) {
  return -fmaf(fmaxf(g, 0.f), kLog2e, __log2f(1.f + exp2_fast(-fabsf(g) * kLog2e)));
}

// y sigmoid(y) = y / (1 + e^-y), the activation after the short convolution,
// with the same intrinsics (its output is rounded to bf16 right after); a
// very negative y gives -0.
__device__ __forceinline__ float silu_fast(float y) { return __fdividef(y, 1.f + __expf(-y)); }

// sigmoid(r), the output gate's factor, from t = e / (1 + e), e = e^-|r|:
// t for r < 0 and 1 - t for r >= 0 (no cancellation on either side; a
// saturated logit gives exactly 1 since t < 2^-25 rounds away).  Fast
// exponential and division: o is rounded to bf16 right after.
__device__ __forceinline__ float gate_fast(float r) {
  const float e = __expf(-fabsf(r));
  const float t = __fdividef(e, 1.f + e);
  return r >= 0.f ? 1.f - t : t;
}

// dependent: launched as the programmatic dependent of the planning kernel
cudaError_t launch_intra(const ChunkParams& p, cudaStream_t stream, bool dependent = false);

}  // namespace tcp
}  // namespace kda
