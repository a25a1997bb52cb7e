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

// Input x (q or k: tensor t) of token tok (sequence s starting at packed
// index seq0), head h, channel c, after the short convolution when there is
// one (formula and windows in include/kda.h): inputs before the sequence
// start from its window, or zeros.
template <typename TIn>
__device__ float prep_input(const kda_prep_args& a, const kda_layer_args& l, int t, const TIn* x, int64_t tok,
                            int32_t s, int64_t seq0, int h, int c) {
  const int H = a.num_heads, dk = a.dk, W = l.conv_width;
  const int64_t e = (tok * H + h) * dk + c;
  if (W == 0) return ld_in(x, e);
  const TIn* win = static_cast<const TIn*>(l.conv_in[t]);
  float acc = 0.f;
  for (int j = 0; j < W; ++j) {
    const int64_t src = tok - j;
    float xv = 0.f;
    if (src >= seq0)
      xv = ld_in(x, e - (int64_t)j * H * dk);
    else if (win && seq0 - src <= W - 1)  // window row W - 1 - (seq0 - src) (further back:
                                          // only with malformed cu_seqlens)
      xv = ld_in(win, (((int64_t)s * (W - 1) + (W - 1) - (seq0 - src)) * H + h) * dk + c);
    acc += l.conv_w[t][((int64_t)j * H + h) * dk + c] * xv;
  }
  if (l.conv_silu) acc = silu_of(acc);
  return round_in<TIn>(acc);
}

template <typename TIn>
__global__ void __launch_bounds__(kPrepThreads)
prep_kernel(kda_prep_args a, const kda_layer_args l) {
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
    const int32_t st = l.conv_width > 0 ? seq_of_token(a.cu_seqlens, a.num_seqs, t) : 0;
    const int64_t s0 = l.conv_width > 0 ? a.cu_seqlens[st] : 0;
    float sq = 0.f, sk = 0.f;
    for (int c = lane; c < dk; c += 32) {
      const float xq = prep_input(a, l, 0, q, t, st, s0, h, c), xk = prep_input(a, l, 1, k, t, st, s0, h, c);
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
    const bool ph = a.gate_per_head != 0;  // g [T, H]: one logit per token and head
    for (int64_t t = cs; t < t0; ++t) run += log_alpha_of(ld_in(g, ph ? t * H + h : (t * H + h) * dk + c));
    for (int64_t t = t0; t < t1; ++t) {
      while (s + 1 < a.num_seqs && a.cu_seqlens[s + 1] <= t) {
        ++s;
        seq0 = a.cu_seqlens[s];
      }
      if ((t - seq0) % kChunk == 0) run = 0.f;
      const int64_t e = (t * H + h) * dk + c;
      run += log_alpha_of(ld_in(g, ph ? t * H + h : e));
      a.G[e] = run;
      a.qhat[e] = prep_input(a, l, 0, q, t, s, seq0, h, c) * inv_q[t - t0];
      a.khat[e] = prep_input(a, l, 1, k, t, s, seq0, h, c) * inv_k[t - t0];
    }
  }
}

// bf16 inputs with dk = 128 and 16-byte aligned buffers: the same step with
// 16-byte loads and 32-byte stores, so that each thread keeps a dozen loads
// in flight.  Thread (cg = lane % 16, tb = 2 warp + lane / 16) owns channels
// 8 cg .. 8 cg + 7 of the tile's tokens 8 tb .. 8 tb + 7.  The norms reduce
// over the 16 lanes of a token; G is a segmented scan (restarting at chunk
// starts): inside a thread's 8 tokens, then across the 8 token blocks
// through shared memory, then the log-decays of the tile's first chunk
// before t0 (only when the tile does not start a chunk).
constexpr int kVecThreads = 128;

__device__ __forceinline__ void bf16x8(const uint4& v, float* x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// (5 CTAs per SM: at most 102 registers a thread, a few spilled; it is
// bound by memory latency, and 20 warps an SM instead of 12 hide more of it:
// 168 -> 138 us on the 8192-token, 32-head inputs)
__global__ void __launch_bounds__(kVecThreads, 5) prep_vec(kda_prep_args a) {
  __shared__ float blk_tot[8][128];  // per token block: log-decay sum since its last chunk start
  __shared__ int blk_reset[8];       // the block holds a chunk start
  __shared__ int starts[kChunk];     // token i of the tile starts a chunk
  __shared__ float warm[128];        // log-decays from the tile's first chunk start to t0
  const int64_t t0 = (int64_t)blockIdx.x * kChunk;
  const int h = blockIdx.y, H = a.num_heads;
  const int64_t T = a.total_tokens;
  const int64_t t1 = t0 + kChunk < T ? t0 + kChunk : T;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cg = lane & 15, tb = 2 * warp + (lane >> 4), c0 = 8 * cg;
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(a.g);
  const __nv_bfloat16* b = static_cast<const __nv_bfloat16*>(a.b);
  auto row16 = [&](const __nv_bfloat16* base, int64_t t) {
    return __ldg(reinterpret_cast<const uint4*>(base + (t * H + h) * 128 + c0));
  };

  // the first 4 rows of this thread are in flight while the chunk starts
  // of the tile are found
  uint4 qr[4], kr[4], gr[4];
  auto load4 = [&](int pass) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int64_t t = t0 + 8 * tb + 4 * pass + r;
      const uint4 z = make_uint4(0, 0, 0, 0);
      qr[r] = t < t1 ? row16(q, t) : z;
      kr[r] = t < t1 ? row16(k, t) : z;
      gr[r] = t < t1 ? row16(g, t) : z;
    }
  };
  load4(0);
  if (tid < kChunk) {
    const int64_t t = t0 + tid;
    int flag = 0;
    if (t < t1) {
      const int32_t sq = seq_of_token(a.cu_seqlens, a.num_seqs, t);
      flag = (t - a.cu_seqlens[sq]) % kChunk == 0;
    }
    starts[tid] = flag;
  }
  if (tid < 16) {  // warp 0, lanes 0-15: the chunk holding t0 may have started before the tile
    const int32_t sq = seq_of_token(a.cu_seqlens, a.num_seqs, t0);
    const int64_t seq0 = a.cu_seqlens[sq];
    int64_t cs = seq0 + ((t0 - seq0) / kChunk) * kChunk;
    const int64_t lo = t0 - (kChunk - 1) > 0 ? t0 - (kChunk - 1) : 0;
    if (cs < lo) cs = lo;  // only reachable with malformed cu_seqlens
    if (cs > t0) cs = t0;
    float w[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int64_t t = cs; t < t0; ++t) {
      float x[8];
      bf16x8(row16(g, t), x);
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] += log_alpha_of(x[j]);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) warm[c0 + j] = w[j];
  }
  __syncthreads();

  float la[8][8];  // log alpha of this thread's 8 tokens x 8 channels, then their prefix sums
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    if (pass == 1) load4(1);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int64_t t = t0 + 8 * tb + 4 * pass + r;
      float xq[8], xk[8], xg[8];
      bf16x8(qr[r], xq);
      bf16x8(kr[r], xk);
      bf16x8(gr[r], xg);
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        sq += xq[j] * xq[j];
        sk += xk[j] * xk[j];
        la[4 * pass + r][j] = log_alpha_of(xg[j]);
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
      }
      if (t < t1) {
        const float iq = inv_norm_of(sq), ik = inv_norm_of(sk);
        const int64_t e = (t * H + h) * 128 + c0;
        float4* oq = reinterpret_cast<float4*>(a.qhat + e);
        float4* ok = reinterpret_cast<float4*>(a.khat + e);
        oq[0] = make_float4(xq[0] * iq, xq[1] * iq, xq[2] * iq, xq[3] * iq);
        oq[1] = make_float4(xq[4] * iq, xq[5] * iq, xq[6] * iq, xq[7] * iq);
        ok[0] = make_float4(xk[0] * ik, xk[1] * ik, xk[2] * ik, xk[3] * ik);
        ok[1] = make_float4(xk[4] * ik, xk[5] * ik, xk[6] * ik, xk[7] * ik);
        if (cg == 0) a.beta[t * H + h] = beta_of(__bfloat162float(b[t * H + h]));
      }
    }
  }
  // segmented prefix sums inside the block of 8 tokens
  bool reset_seen = false;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const bool st = starts[8 * tb + r] != 0;
    reset_seen = reset_seen || st;
#pragma unroll
    for (int j = 0; j < 8; ++j) la[r][j] += (r > 0 && !st) ? la[r - 1][j] : 0.f;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) blk_tot[tb][c0 + j] = la[7][j];
  if (cg == 0) blk_reset[tb] = reset_seen;
  __syncthreads();
  // carry into this block: the blocks before it back to the last chunk start,
  // and the warm-up sum when no chunk starts inside the tile before it
  float carry[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  bool closed = false;
  for (int bb = tb - 1; bb >= 0 && !closed; --bb) {
#pragma unroll
    for (int j = 0; j < 8; ++j) carry[j] += blk_tot[bb][c0 + j];
    closed = blk_reset[bb] != 0;
  }
  if (!closed)
#pragma unroll
    for (int j = 0; j < 8; ++j) carry[j] += warm[c0 + j];
  bool after_start = false;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int64_t t = t0 + 8 * tb + r;
    after_start = after_start || starts[8 * tb + r] != 0;
    if (t < t1) {
      float x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = la[r][j] + (after_start ? 0.f : carry[j]);
      float4* og = reinterpret_cast<float4*>(a.G + (t * H + h) * 128 + c0);
      og[0] = make_float4(x[0], x[1], x[2], x[3]);
      og[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
  }
}

bool aligned16p(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

cudaError_t launch_prep(const kda_prep_args& a, cudaStream_t stream) {
  if (a.total_tokens == 0) return cudaSuccess;
  dim3 grid((unsigned)((a.total_tokens + kChunk - 1) / kChunk), (unsigned)a.num_heads);
  kda_layer_args l{};  // by value: the kernel cannot read the caller's host struct
  if (a.layer && a.layer->conv_width > 0) {
    l.conv_width = a.layer->conv_width;
    l.conv_silu = a.layer->conv_silu != 0;
    for (int t = 0; t < 2; ++t) {
      l.conv_w[t] = a.layer->conv_w[t];
      l.conv_in[t] = l.conv_width > 1 ? a.layer->conv_in[t] : nullptr;
    }
  }
  if (l.conv_width == 0 && a.in_dtype == KDA_BF16 && a.dk == 128 && !a.gate_per_head && aligned16p(a.q) &&
      aligned16p(a.k) && aligned16p(a.g) && aligned16p(a.qhat) && aligned16p(a.khat) && aligned16p(a.G))
    prep_vec<<<grid, kVecThreads, 0, stream>>>(a);
  else if (a.in_dtype == KDA_BF16)
    prep_kernel<__nv_bfloat16><<<grid, kPrepThreads, 0, stream>>>(a, l);
  else
    prep_kernel<float><<<grid, kPrepThreads, 0, stream>>>(a, l);
  return cudaGetLastError();
}

}  // namespace kda
