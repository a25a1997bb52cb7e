// kda_layer.cu -- the windows of the short convolution after a prefill.
//
// The convolution on q, k and v ("Kimi K3: The Manos, The Mythos, The
// Legendos", bullet on the stability details; formula and window layout in
// include/kda.h) is causal along each sequence, so the next call on the same
// sequence (a later prefill piece or a decode step) needs the raw inputs of
// its last conv_width - 1 positions.  Those are the last rows of window ++
// sequence: tokens of the sequence where it is long enough, older window
// entries otherwise.  The convolution itself runs inside the prefill and
// decode kernels.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxD = 256;   // widest head
constexpr int kMaxPer = (KDA_CONV_MAX - 1) * kMaxD / kThreads;  // elements per thread

// One CTA per (sequence, tensor, head).  Every read comes before the first
// write, so `out` may be the same buffer as `in`.
template <typename E>
__global__ void __launch_bounds__(kThreads)
conv_windows(const int64_t* __restrict__ cu, int64_t T, int32_t H, int32_t dk, int32_t dv, int32_t R, const void* x0,
             const void* x1, const void* x2, const void* in0, const void* in1, const void* in2, void* out0,
             void* out1, void* out2) {
  const int s = blockIdx.x, t = blockIdx.y, h = blockIdx.z;
  const int d = t == 2 ? dv : dk;
  const E* x = static_cast<const E*>(t == 0 ? x0 : t == 1 ? x1 : x2);
  const E* in = static_cast<const E*>(t == 0 ? in0 : t == 1 ? in1 : in2);
  E* out = static_cast<E*>(t == 0 ? out0 : t == 1 ? out1 : out2);
  if (!out) return;
  const int64_t start = cu[s], len = cu[s + 1] - start;
  // a malformed cu_seqlens (flagged by the planner) leaves the window as it is
  if (start < 0 || len < 0 || start + len > T) return;
  const int n = R * d;  // <= (KDA_CONV_MAX - 1) * kMaxD
  E val[kMaxPer];
#pragma unroll
  for (int u = 0; u < kMaxPer; ++u) {
    const int e = threadIdx.x + u * kThreads;
    val[u] = E(0.f);
    if (e < n) {
      const int m = e / d, c = e - m * d;
      const int64_t pos = len + m;  // index in window ++ sequence
      if (pos >= R)
        val[u] = x[((start + pos - R) * H + h) * (int64_t)d + c];
      else if (in)
        val[u] = in[(((int64_t)s * R + pos) * H + h) * d + c];
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kMaxPer; ++u) {
    const int e = threadIdx.x + u * kThreads;
    if (e < n) {
      const int m = e / d, c = e - m * d;
      out[(((int64_t)s * R + m) * H + h) * d + c] = val[u];
    }
  }
}

}  // namespace

cudaError_t launch_conv_windows(const kda_layer_args& l, int32_t num_seqs, int32_t H, int32_t dk,
                                int32_t dv, const int64_t* cu_seqlens, int64_t total_tokens, kda_dtype_t dt,
                                const void* const x[3], cudaStream_t stream) {
  const int32_t R = l.conv_width - 1;
  if (R <= 0 || !(l.conv_out[0] || l.conv_out[1] || l.conv_out[2])) return cudaSuccess;
  static_assert((KDA_CONV_MAX - 1) * kMaxD <= kMaxPer * kThreads, "one pass covers a window");
  dim3 grid((unsigned)num_seqs, 3, (unsigned)H);
  if (dt == KDA_BF16)
    conv_windows<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(
        cu_seqlens, total_tokens, H, dk, dv, R, x[0], x[1], x[2], l.conv_in[0], l.conv_in[1], l.conv_in[2], l.conv_out[0],
        l.conv_out[1], l.conv_out[2]);
  else
    conv_windows<float><<<grid, kThreads, 0, stream>>>(cu_seqlens, total_tokens, H, dk, dv, R, x[0], x[1], x[2],
                                                       l.conv_in[0], l.conv_in[1], l.conv_in[2],
                                                       l.conv_out[0], l.conv_out[1], l.conv_out[2]);
  return cudaGetLastError();
}

}  // namespace kda
