// kda_prep.cu -- the preparation step of the KDA recurrence as its own kernel.
//
// Per (token, head): q^ = q / max(|q|, 1e-6), k^ likewise (queries and keys
// are L2-normalised, "Kimi K3: The Manos, The Mythos, The Legendos", bullet
// on stability details); beta = sigmoid(b) (update strength); and G, the
// running sum of log alpha = -softplus(g) (per-channel retention, "From KV
// Cache to Depth Attention", Technical Details) restarted at the first token
// of every chunk of KDA_CHUNK tokens counted from the sequence start -- the
// log of the cumulative decay Gamma used by the chunked form.
//
// One CTA per (64-token tile of the packed index, head).  A tile may hold
// the tail of one sequence and the head of the next, and its first chunk
// may have started in the previous tile; each channel thread first sums the
// log-decays from that chunk start up to the tile (at most 63 tokens).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kPrepThreads = 128;

template <typename TIn>
__global__ void __launch_bounds__(kPrepThreads)
prep_kernel(kda_prep_args a) {
  __shared__ float inv_q[kChunk], inv_k[kChunk];
  const int64_t t0 = (int64_t)blockIdx.x * kChunk;
  const int h = blockIdx.y, H = a.num_heads, dk = a.dk;
  const int64_t T = a.total_tokens;
  const int64_t t1 = t0 + kChunk < T ? t0 + kChunk : T;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const TIn* q = static_cast<const TIn*>(a.q);
  const TIn* k = static_cast<const TIn*>(a.k);
  const TIn* g = static_cast<const TIn*>(a.g);
  const TIn* b = static_cast<const TIn*>(a.b);

  for (int i = warp; i < kChunk; i += kPrepThreads / 32) {
    const int64_t t = t0 + i;
    if (t >= t1) break;
    const int64_t base = (t * H + h) * dk;
    float sq = 0.f, sk = 0.f;
    for (int c = lane; c < dk; c += 32) {
      const float xq = ld_in(q, base + c), xk = ld_in(k, base + c);
      sq += xq * xq;
      sk += xk * xk;
    }
    sq = inv_norm_of(warp_sum(sq));
    sk = inv_norm_of(warp_sum(sk));
    if (lane == 0) {
      inv_q[i] = sq;
      inv_k[i] = sk;
      a.beta[t * H + h] = beta_of(ld_in(b, t * H + h));
    }
  }
  __syncthreads();

  for (int c = tid; c < dk; c += kPrepThreads) {
    int32_t s = seq_of_token(a.cu_seqlens, a.num_seqs, t0);
    int64_t seq0 = a.cu_seqlens[s];
    // warm-up: the chunk holding t0 may have started before the tile
    int64_t cs = seq0 + ((t0 - seq0) / kChunk) * kChunk;
    const int64_t lo = t0 - (kChunk - 1) > 0 ? t0 - (kChunk - 1) : 0;
    if (cs < lo) cs = lo;  // only reachable with malformed cu_seqlens
    if (cs > t0) cs = t0;
    float run = 0.f;
    for (int64_t t = cs; t < t0; ++t) run += log_alpha_of(ld_in(g, (t * H + h) * dk + c));
    for (int64_t t = t0; t < t1; ++t) {
      while (s + 1 < a.num_seqs && a.cu_seqlens[s + 1] <= t) {
        ++s;
        seq0 = a.cu_seqlens[s];
      }
      if ((t - seq0) % kChunk == 0) run = 0.f;
      const int64_t e = (t * H + h) * dk + c;
      run += log_alpha_of(ld_in(g, e));
      a.G[e] = run;
      a.qhat[e] = ld_in(q, e) * inv_q[t - t0];
      a.khat[e] = ld_in(k, e) * inv_k[t - t0];
    }
  }
}

}  // namespace

cudaError_t launch_prep(const kda_prep_args& a, cudaStream_t stream) {
  if (a.total_tokens == 0) return cudaSuccess;
  dim3 grid((unsigned)((a.total_tokens + kChunk - 1) / kChunk), (unsigned)a.num_heads);
  if (a.in_dtype == KDA_BF16)
    prep_kernel<__nv_bfloat16><<<grid, kPrepThreads, 0, stream>>>(a);
  else
    prep_kernel<float><<<grid, kPrepThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kda
