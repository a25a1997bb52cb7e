// kda_common.cuh -- types and small device helpers shared by the libkda kernels.
//
// Layout conventions: token-major packed tensors, q/k/g [T, H, dk],
// v/o [T, H, dv], b [T, H]; states [.., H, dk, dv] fp32 row-major (row = key
// channel, column = value channel).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int kChunk = KDA_CHUNK;  // tokens per chunk of the chunked prefill

// Bits of the device status word (first int32 of the prefill workspace).
enum : int32_t {
  kFlagBadSeqlens = 1,
  kFlagBadBoundaries = 2,
  kFlagChunkOverflow = 4,
  kFlagTimeout = 8,
  kFlagDecayRange = 16,  // tensor-core path: a chunk decayed past its operands' range
};

// One entry of the chunk table: a run of <= kChunk tokens of one sequence
// that ends at a chunk edge, at a snapshot position or at the sequence end.
struct Chunk {
  int64_t tok0;      // packed index of its first token
  int32_t seq;       // sequence index
  int32_t len;       // 1..kChunk tokens
  int32_t snap_slot; // snapshot slot written after this chunk, or -1
  int32_t flags;     // kChunkFirst | kChunkLast
  int64_t pos;       // its first token's index within its sequence
};
static_assert(sizeof(Chunk) == 32, "chunk table entry is 32 bytes");
enum : int32_t { kChunkFirst = 1, kChunkLast = 2 };

// Scalars the planning kernels publish for the later kernels.
struct PlanMeta {
  int64_t total_chunks;
  int64_t pad[3];
};

// Programmatic dependent launch (griddepcontrol, sm_90 and later).  A
// kernel launched as the programmatic dependent of the kernel before it on
// the stream may start once every CTA of that kernel has signalled
// (pdl_launch_dependents) or exited; at pdl_wait it waits until that kernel
// has completed and its memory operations are visible.  Both are no-ops for
// a kernel launched the ordinary way or without such a dependent.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ input access
template <typename T>
__device__ __forceinline__ float ld_in(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ld_in<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld_in<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}

template <typename T>
__device__ __forceinline__ void st_out(T* p, int64_t i, float x);
template <>
__device__ __forceinline__ void st_out<float>(float* p, int64_t i, float x) { p[i] = x; }
template <>
__device__ __forceinline__ void st_out<__nv_bfloat16>(__nv_bfloat16* p, int64_t i, float x) {
  p[i] = __float2bfloat16_rn(x);
}

// ------------------------------------------------------------ gates
// log alpha = -softplus(g); softplus(x) = log(1 + e^x), = x above 20.
__device__ __forceinline__ float log_alpha_of(float g) {
  return g > 20.f ? -g : -log1pf(expf(g));
}
// beta = sigmoid(b)
__device__ __forceinline__ float beta_of(float b) { return 1.f / (1.f + expf(-b)); }
// y sigmoid(y), the activation after the short convolution
__device__ __forceinline__ float silu_of(float y) { return y / (1.f + expf(-y)); }
// the output gate's factor sigmoid(r)
__device__ __forceinline__ float out_gate_of(float r) { return 1.f / (1.f + expf(-r)); }
// x rounded to the input dtype (the precision the convolution's output is kept in)
template <typename T>
__device__ __forceinline__ float round_in(float x);
template <>
__device__ __forceinline__ float round_in<float>(float x) { return x; }
template <>
__device__ __forceinline__ float round_in<__nv_bfloat16>(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}
// 1 / max(sqrt(ss), 1e-6)
__device__ __forceinline__ float inv_norm_of(float ss) {
  return 1.f / fmaxf(sqrtf(ss), 1e-6f);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Index of the sequence holding packed token t: largest s with cu[s] <= t.
__device__ __forceinline__ int32_t seq_of_token(const int64_t* cu, int32_t n, int64_t t) {
  int32_t lo = 0, hi = n - 1;
  while (lo < hi) {
    int32_t mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ------------------------------------------------------------ workspace layout
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Per (chunk, head) intermediate record of the fp32 CUDA-core path:
//   W, QG, KR : [kChunk][dk] fp32   (W = T diag(beta) (K^ o Gamma),
//                                    QG = Q^ o Gamma, KR = K^ o Gamma_L / Gamma)
//   AQK       : [kChunk][kChunk] fp32 (masked j <= i)
//   UT        : [kChunk][dv] fp32   (U~ = T diag(beta) V)
//   GL        : [dk] fp32           (Gamma_L = exp(G_L))
struct SimtRec {
  static __host__ __device__ size_t w(int) { return 0; }
  static __host__ __device__ size_t qg(int dk) { return (size_t)kChunk * dk; }
  static __host__ __device__ size_t kr(int dk) { return 2 * (size_t)kChunk * dk; }
  static __host__ __device__ size_t aqk(int dk) { return 3 * (size_t)kChunk * dk; }
  static __host__ __device__ size_t ut(int dk) { return aqk(dk) + (size_t)kChunk * kChunk; }
  static __host__ __device__ size_t gl(int dk, int dv) { return ut(dk) + (size_t)kChunk * dv; }
  // floats per record, rounded up to 64 floats (256 bytes)
  static __host__ __device__ size_t floats(int dk, int dv) {
    return ((gl(dk, dv) + dk) + 63) / 64 * 64;
  }
};

struct WsLayout {
  size_t status = 0, meta = 0, seq_len = 0, seq_chunk_begin = 0, seq_seg_begin = 0,
         bnd_nonaligned = 0, bnd_nonmult = 0, seq_aux = 0, chunks = 0, inter = 0, total = 0;
  int64_t max_chunks = 0;
  size_t rec_bytes = 0;  // bytes of one (chunk, head) intermediate record
  // segment scan: segment count (1 = off) and its buffers
  int32_t scan_P = 1;
  size_t scan_cu = 0, scan_A = 0, scan_B = 0, scan_inits = 0, scan_finals = 0;
  // fused and overlapped tensor-core prefill: a flag per record (where the
  // arguments can take it); (overlapped) its counters, right before the
  // flags, and the words of both, which the planning kernel clears
  size_t rec_ready = 0;
  size_t seq_order = 0;
  size_t ovl = 0;
  int64_t ovl_words = 0;
};

}  // namespace kda
