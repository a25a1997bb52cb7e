// kda_simt.cu -- fp32 CUDA-core chunked prefill (any supported head size).
//
// The chunked form of the recurrence (FlashKDA's "unrolling the recurrence in
// chunks", "Kimi K3: The Manos, The Mythos, The Legendos", bullet list).
// For a chunk of L <= 64 tokens with start state S0, log-decay running sums
// G_i = sum_{m<=i} log alpha_m (per key channel) and Gamma = exp(G):
//
//   A_kk[i,j] = beta_i sum_c k_ic k_jc exp(G_ic - G_jc)      (j < i)
//   T         = (I + A_kk)^{-1}
//   W         = T diag(beta) (K o Gamma)      U~ = T diag(beta) V
//   A_qk[i,j] = sum_c q_ic k_jc exp(G_ic - G_jc)            (j <= i)
//   U         = U~ - W S0
//   O         = scale ((Q o Gamma) S0 + A_qk U)
//   S_end     = Diag(Gamma_L) S0 + (K o Gamma_L / Gamma)^T U
//
// obtained by expanding the token recurrence (delta rule with a diagonal
// gate, "From KV Cache to Depth Attention", Technical Details) inside the
// chunk.  This path keeps everything in fp32; it serves fp32 inputs and head
// sizes other than 128.  A_kk and A_qk are products of factors with a
// per-channel reference s (an integer number of nats, so G - s is exact):
// Kp = k^ e^(G - s), Qp = q^ e^(G - s), Kn = k^ e^(s - G), so that
// exp(G_i - G_j) = e^(G_i - s) e^(s - G_j) with both factors in fp32 range.
// s = 0 while a channel's chunk decay G_L stays above -kRefNats, else
// round(G_L / 2); a chunk (or block of channels) whose G_L falls below
// -kMaxNats in some channel forms exp(G_i - G_j) directly instead, so the
// path has no exponent-range limit.
//
// K2 (intra) runs one CTA per (chunk, head) and writes a SimtRec per pair;
// K3 (inter) runs one CTA per (sequence, head, value-column slice) and walks
// the sequence's chunks in order, carrying its slice of S in shared memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
// 16-byte asynchronous copy global -> shared (both 16-byte aligned), and
// its groups
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr float kRefNats = 80.f;   // e^-80 and e^80 are inside the fp32 range
constexpr float kMaxNats = 170.f;  // e^(+-85) are too

// The per-channel references of a block of nb channels from its running
// log-decay G ([64][ld], rows past the chunk carrying G_{L-1}): s[c], and
// whether some channel is past kMaxNats (the direct form is then taken).
// Every thread of the CTA calls it; the result is the same for all.
__device__ __forceinline__ bool channel_refs(const float* G, int ld, int nb, float* sref) {
  bool direct = false;
  for (int c = threadIdx.x; c < nb; c += kThreads) {
    const float gl = G[(kChunk - 1) * ld + c];
    sref[c] = gl >= -kRefNats ? 0.f : rintf(0.5f * gl);
    direct |= gl < -kMaxNats;
  }
  return __syncthreads_or(direct);
}

// In place over a block of nb channels: X (q^) <- Qp, Kb (k^) <- Kp and
// G <- Kn, with the references sref.
__device__ __forceinline__ void factor_block(float* X, float* Kb, float* G, int ld, int nb, const float* sref) {
  for (int idx = threadIdx.x; idx < kChunk * nb; idx += kThreads) {
    const int i = idx / nb, c = idx - i * nb;
    const float e = G[i * ld + c] - sref[c];
    const float ep = expf(e), en = expf(-e), k = Kb[i * ld + c];
    X[i * ld + c] *= ep;
    Kb[i * ld + c] = k * ep;
    G[i * ld + c] = k * en;
  }
}

// T = (I + A)^{-1} for strictly lower-triangular A (64 x 64, row-major),
// by blocks (all 256 threads): the four 16 x 16 diagonal blocks by forward
// substitution (a thread per column, 16 steps), then within each 32 x 32
// half T10 = -T11 A10 T00, then T[32:64, 0:32] = -T_hi A T_lo, each product
// as fp32 dot products.  X: scratch of 1024 floats.
__device__ __noinline__ void simt_inverse(const float* __restrict__ A, float* __restrict__ T,
                                          float* __restrict__ X) {
  const int tid = threadIdx.x;
  if (tid < kChunk) {
    const int d = tid >> 4, jj = tid & 15, j = 16 * d + jj;
    float col[16];
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) {
      const float* ar = A + (16 * d + ii) * kChunk + 16 * d;
      float acc = ii == jj ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < ii; ++m) acc -= ar[m] * col[m];
      col[ii] = acc;
    }
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) T[(16 * d + ii) * kChunk + j] = col[ii];
  } else {
    // the blocks above the diagonal are zero
    for (int idx = tid - kChunk; idx < 6 * 256; idx += kThreads - kChunk) {
      const int t = idx >> 8, e = idx & 255;
      const int bi = t < 3 ? 0 : (t < 5 ? 1 : 2);
      const int bj = t < 3 ? t + 1 : (t < 5 ? t - 1 : 3);
      T[(16 * bi + (e >> 4)) * kChunk + 16 * bj + (e & 15)] = 0.f;
    }
  }
  __syncthreads();
  // level 1: half P = e / 256; X1 = A10 T00, then T10 = -T11 X1
  for (int e = tid; e < 512; e += kThreads) {
    const int P = e >> 8, r = (e >> 4) & 15, c = e & 15, r0 = 32 * P + 16, c0 = 32 * P;
    float acc = 0.f;
    for (int m = 0; m < 16; ++m) acc += A[(r0 + r) * kChunk + c0 + m] * T[(c0 + m) * kChunk + c0 + c];
    X[e] = acc;
  }
  __syncthreads();
  for (int e = tid; e < 512; e += kThreads) {
    const int P = e >> 8, r = (e >> 4) & 15, c = e & 15, r0 = 32 * P + 16, c0 = 32 * P;
    float acc = 0.f;
    for (int m = 0; m <= r; ++m) acc += T[(r0 + r) * kChunk + r0 + m] * X[(P << 8) + (m << 4) + c];
    T[(r0 + r) * kChunk + c0 + c] = -acc;
  }
  __syncthreads();
  // level 2: X = A[32:64, 0:32] T[0:32, 0:32], then T[32:64, 0:32] = -T[32:64, 32:64] X
  for (int e = tid; e < 1024; e += kThreads) {
    const int r = e >> 5, c = e & 31;
    float acc = 0.f;
    for (int m = c & ~15; m < 32; ++m) acc += A[(32 + r) * kChunk + m] * T[m * kChunk + c];
    X[e] = acc;
  }
  __syncthreads();
  for (int e = tid; e < 1024; e += kThreads) {
    const int r = e >> 5, c = e & 31;
    float acc = 0.f;
    for (int m = 0; m <= r; ++m) acc += T[(32 + r) * kChunk + 32 + m] * X[(m << 5) + c];
    T[(32 + r) * kChunk + c] = -acc;
  }
  __syncthreads();
}

// A[i][j] += beta_i (Kp Kn^T)[i][j] for j < i and AQ[i][j] += (Qp Kn^T)[i][j]
// for j <= i, rows i < len, over nb channels; thread t takes rows
// 4 (t / 16) .. +3 and columns 4 (t % 16) .. +3 (tiles above the diagonal
// are zero and skipped).
__device__ __forceinline__ void accumulate_products(const float* Qp, const float* Kp, const float* Kn, int ld,
                                                    int nb, int len, const float* beta, float* A, float* AQ) {
  const int I = threadIdx.x >> 4, J = threadIdx.x & 15;
  if (J > I) return;
  float akk[4][4], aqk[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int t = 0; t < 4; ++t) akk[r][t] = aqk[r][t] = 0.f;
  const float* kp = Kp + 4 * I * ld;
  const float* qp = Qp + 4 * I * ld;
  const float* kn = Kn + 4 * J * ld;
  for (int c = 0; c < nb; ++c) {
    float a[4], q[4], b[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      a[r] = kp[r * ld + c];
      q[r] = qp[r * ld + c];
      b[r] = kn[r * ld + c];
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        akk[r][t] += a[r] * b[t];
        aqk[r][t] += q[r] * b[t];
      }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = 4 * I + r;
    if (i >= len) continue;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int j = 4 * J + t;
      if (j < i) A[i * kChunk + j] += beta[i] * akk[r][t];
      if (j <= i) AQ[i * kChunk + j] += aqk[r][t];
    }
  }
}

// Tensor t (0 q, 1 k, 2 v; head size d) at token i of chunk ch, channel col,
// after the short convolution when there is one:
//   y = sum_{j < W} w[j][h][col] x_{i-j}   (x before the sequence start from
//   its window, or 0), SiLU if asked, rounded to the input dtype.
template <typename TIn>
__device__ float conv_input(const ChunkParams& p, int t, const TIn* x, int d, const Chunk& ch, int i, int h,
                            int col) {
  const int H = p.H, W = p.conv_width;
  const int64_t e = ((ch.tok0 + i) * H + h) * (int64_t)d + col;
  if (W == 0) return ld_in(x, e);
  const int64_t pos = (p.conv_one_seq ? ch.tok0 : ch.pos) + i;  // index in the sequence
  const int seq = p.conv_one_seq ? 0 : ch.seq;
  const TIn* win = static_cast<const TIn*>(p.conv_in[t]);
  const float* w = p.conv_w[t];
  float acc = 0.f;
  for (int j = 0; j < W; ++j) {
    float xv = 0.f;
    if (pos - j >= 0)
      xv = ld_in(x, e - (int64_t)j * H * d);
    else if (win)  // window row W - 1 + (pos - j): the input (j - pos) tokens before the start
      xv = ld_in(win, (((int64_t)seq * (W - 1) + (W - 1) + (pos - j)) * H + h) * d + col);
    acc += w[((int64_t)j * H + h) * d + col] * xv;
  }
  if (p.conv_silu) acc = silu_of(acc);
  return round_in<TIn>(acc);
}

// 8 consecutive elements x[e .. e+7] as floats, one 16-byte load (bf16) or
// two (fp32); e a multiple of 8, x 16-byte aligned
__device__ __forceinline__ void ld8(const __nv_bfloat16* x, int64_t e, float* out) {
  const uint4 u = *reinterpret_cast<const uint4*>(x + e);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    out[2 * t] = __uint_as_float(w[t] << 16);
    out[2 * t + 1] = __uint_as_float(w[t] & 0xffff0000u);
  }
}
__device__ __forceinline__ void ld8(const float* x, int64_t e, float* out) {
  const float4 a = *reinterpret_cast<const float4*>(x + e), b = *reinterpret_cast<const float4*>(x + e + 4);
  out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
  out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
}
__device__ __forceinline__ bool aligned16_dev(const void* x) {
  return (reinterpret_cast<uintptr_t>(x) & 15) == 0;
}
// The rows of q, k, v, g can be read 8 channels at a time: no convolution
// (it reads other rows), 16-byte aligned tensors (head sizes are multiples
// of 8)
template <typename TIn>
__device__ __forceinline__ bool vector_rows(const ChunkParams& p) {
  return p.conv_width == 0 && aligned16_dev(p.q) && aligned16_dev(p.k) && aligned16_dev(p.v) &&
         (p.gate_per_head || aligned16_dev(p.g));
}

template <typename TIn>
__global__ void __launch_bounds__(kThreads)
simt_intra(ChunkParams p) {
  extern __shared__ float sm[];
  const int64_t c = blockIdx.x;
  const Chunk ch = p.chunks[c];  // entries past the table's end have len 0
  if (ch.len == 0) return;
  const int h = blockIdx.y, H = p.H, dk = p.dk, dv = p.dv;
  const int len = ch.len;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // rows of q^, k^, G and e^G padded to dk + 1 floats: the A loop's lanes
  // read 32 different rows of one column, which then fall in distinct banks
  const int ld = dk + 1;
  float* qh = sm;                   // [64][ld]
  float* kh = qh + kChunk * ld;     // [64][ld]
  float* G = kh + kChunk * ld;      // [64][ld]
  float* EG = G + kChunk * ld;      // [64][ld] e^G
  float* V = EG + kChunk * ld;      // [64][dv]
  float* A = V + kChunk * dv;       // [64][64]
  float* Tm = A + kChunk * kChunk;  // [64][64]
  float* beta = Tm + kChunk * kChunk;  // [64]
  float* sref = beta + kChunk;          // [dk] per-channel references

  const TIn* q = static_cast<const TIn*>(p.q);
  const TIn* k = static_cast<const TIn*>(p.k);
  const TIn* v = static_cast<const TIn*>(p.v);
  const TIn* g = static_cast<const TIn*>(p.g);
  const TIn* b = static_cast<const TIn*>(p.b);

  if (vector_rows<TIn>(p)) {
    // 8 channels a thread and load
    const int dk8 = dk / 8, dv8 = dv / 8;
#pragma unroll 2
    for (int idx = tid; idx < kChunk * dk8; idx += kThreads) {
      const int i = idx / dk8, c0 = 8 * (idx - i * dk8);
      float xq[8], xk[8], la[8];
      if (i < len) {
        const int64_t e = ((ch.tok0 + i) * H + h) * dk + c0;
        ld8(q, e, xq);
        ld8(k, e, xk);
        if (p.gate_per_head) {
          const float l = log_alpha_of(ld_in(g, (ch.tok0 + i) * H + h));
#pragma unroll
          for (int t = 0; t < 8; ++t) la[t] = l;
        } else {
          ld8(g, e, la);
#pragma unroll
          for (int t = 0; t < 8; ++t) la[t] = log_alpha_of(la[t]);
        }
      } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) xq[t] = xk[t] = la[t] = 0.f;
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        qh[i * ld + c0 + t] = xq[t];
        kh[i * ld + c0 + t] = xk[t];
        G[i * ld + c0 + t] = la[t];
      }
    }
#pragma unroll 2
    for (int idx = tid; idx < kChunk * dv8; idx += kThreads) {
      const int i = idx / dv8, c0 = 8 * (idx - i * dv8);
      float xv[8];
      if (i < len) {
        ld8(v, ((ch.tok0 + i) * H + h) * dv + c0, xv);
      } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) xv[t] = 0.f;
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) V[i * dv + c0 + t] = xv[t];
    }
  } else {
#pragma unroll 4
    for (int idx = tid; idx < kChunk * dk; idx += kThreads) {
      const int i = idx / dk, col = idx - i * dk;
      float xq = 0.f, xk = 0.f, la = 0.f;
      if (i < len) {
        const int64_t e = ((ch.tok0 + i) * H + h) * dk + col;
        xq = conv_input(p, 0, q, dk, ch, i, h, col);
        xk = conv_input(p, 1, k, dk, ch, i, h, col);
        la = log_alpha_of(ld_in(g, p.gate_per_head ? (ch.tok0 + i) * H + h : e));
      }
      qh[i * ld + col] = xq;
      kh[i * ld + col] = xk;
      G[i * ld + col] = la;
    }
#pragma unroll 4
    for (int idx = tid; idx < kChunk * dv; idx += kThreads) {
      const int i = idx / dv, col = idx - i * dv;
      V[idx] = i < len ? conv_input(p, 2, v, dv, ch, i, h, col) : 0.f;
    }
  }
  if (tid < kChunk) beta[tid] = tid < len ? beta_of(ld_in(b, (ch.tok0 + tid) * H + h)) : 0.f;
  __syncthreads();

  // L2 normalisation of each token's q and k (one warp per token)
  for (int i = warp; i < kChunk; i += kThreads / 32) {
    float sq = 0.f, sk = 0.f;
    for (int col = lane; col < dk; col += 32) {
      sq += qh[i * ld + col] * qh[i * ld + col];
      sk += kh[i * ld + col] * kh[i * ld + col];
    }
    sq = inv_norm_of(warp_sum(sq));
    sk = inv_norm_of(warp_sum(sk));
    for (int col = lane; col < dk; col += 32) {
      qh[i * ld + col] *= sq;
      kh[i * ld + col] *= sk;
    }
  }
  // running sum of log alpha down the chunk, one thread per key channel
  for (int col = tid; col < dk; col += kThreads) {
    float run = 0.f;
    for (int i = 0; i < kChunk; ++i) {
      run += G[i * ld + col];
      G[i * ld + col] = run;
      EG[i * ld + col] = expf(run);
    }
  }
  __syncthreads();

  float* rec = p.inter + ((size_t)c * H + h) * p.rec_floats;
  // the record's Q^ o Gamma, K^ o Gamma_L / Gamma and Gamma_L, and
  // K^ o Gamma (into EG) for W
  const float* GLrow = G + (kChunk - 1) * ld;  // padded rows carry G_{L-1} forward
  for (int idx = tid; idx < kChunk * dk; idx += kThreads) {
    const int i = idx / dk, col = idx - i * dk;
    const float eg = EG[i * ld + col], kv = kh[i * ld + col];
    rec[SimtRec::qg(dk) + idx] = qh[i * ld + col] * eg;
    rec[SimtRec::kr(dk) + idx] = kv * expf(GLrow[col] - G[i * ld + col]);
    EG[i * ld + col] = kv * eg;
  }
  for (int col = tid; col < dk; col += kThreads) rec[SimtRec::gl(dk, dv) + col] = expf(GLrow[col]);
  // A_kk (into A) and A_qk (into the record, by way of Tm)
  if (!channel_refs(G, ld, dk, sref)) {
    factor_block(qh, kh, G, ld, dk, sref);  // qh, kh, G <- Qp, Kp, Kn
    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) A[idx] = Tm[idx] = 0.f;
    __syncthreads();
    accumulate_products(qh, kh, G, ld, dk, len, beta, A, Tm);
    __syncthreads();
    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) rec[SimtRec::aqk(dk) + idx] = Tm[idx];
  } else {
    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
      const int i = idx >> 6, j = idx & 63;
      float akk = 0.f, aqk = 0.f;
      if (j <= i && i < len) {
        for (int col = 0; col < dk; ++col) {
          const float d = expf(G[i * ld + col] - G[j * ld + col]);
          const float kj = kh[j * ld + col] * d;
          akk += kh[i * ld + col] * kj;
          aqk += qh[i * ld + col] * kj;
        }
        akk = j < i ? beta[i] * akk : 0.f;
      }
      A[idx] = akk;
      rec[SimtRec::aqk(dk) + idx] = aqk;
    }
  }
  __syncthreads();

  // T = (I + A_kk)^{-1}, unit lower triangular (q^ rows are free: scratch)
  simt_inverse(A, Tm, qh);
  // fold beta into the columns: Tb = T diag(beta)
  for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) Tm[idx] *= beta[idx & 63];
  __syncthreads();

  // W = T diag(beta) (K^ o Gamma), K^ o Gamma held in EG
  for (int idx = tid; idx < kChunk * dk; idx += kThreads) {
    const int i = idx / dk, col = idx - i * dk;
    float w = 0.f;
    for (int m = 0; m <= i; ++m) w += Tm[i * kChunk + m] * EG[m * ld + col];
    rec[SimtRec::w(dk) + idx] = w;
  }
  for (int idx = tid; idx < kChunk * dv; idx += kThreads) {
    const int i = idx / dv, col = idx - i * dv;
    float u = 0.f;
    for (int m = 0; m <= i; ++m) u += Tm[i * kChunk + m] * V[m * dv + col];
    rec[SimtRec::ut(dk) + idx] = u;
  }
}

// Heads wider than 128 channels (dk or dv = 256): the same chunk algebra with
// the channels taken in blocks of kCB, so that shared memory holds one block
// of q^, k^ and G (or of V) at a time.  Pass 1 forms the inverse norms of the
// rows; pass 2 sums A_kk and A_qk over the key blocks (each block's G is its
// channels' running sum, channels being independent); then T; pass 3 forms
// W, Q^ o Gamma, K^ o Gamma_L / Gamma and Gamma_L block by block, and U~ over
// the value blocks.  q, k, g are read twice (the second time mostly from L2).
constexpr int kCB = 128;

template <typename TIn>
__global__ void __launch_bounds__(kThreads)
simt_intra_blocked(ChunkParams p) {
  extern __shared__ float sm[];
  const int64_t c = blockIdx.x;
  const Chunk ch = p.chunks[c];  // entries past the table's end have len 0
  if (ch.len == 0) return;
  const int h = blockIdx.y, H = p.H, dk = p.dk, dv = p.dv;
  const int len = ch.len;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // block rows padded to kCB + 1 floats (the A loop's lanes read 32 rows of
  // one column)
  constexpr int kLd = kCB + 1;
  float* X = sm;                     // [64][kLd]: q^ block, then V block
  float* Kb = X + kChunk * kLd;      // [64][kLd]: k^ block
  float* G = Kb + kChunk * kLd;      // [64][kLd]: running log-decay block
  float* A = G + kChunk * kLd;       // [64][64] A_kk
  float* AQ = A + kChunk * kChunk;   // [64][64] A_qk
  float* Tm = AQ + kChunk * kChunk;  // [64][64] T, then T diag(beta)
  float* beta = Tm + kChunk * kChunk;  // [64]
  float* invq = beta + kChunk;       // [64]
  float* invk = invq + kChunk;       // [64]
  float* sref = invk + kChunk;       // [kCB] per-channel references of a block

  const TIn* q = static_cast<const TIn*>(p.q);
  const TIn* k = static_cast<const TIn*>(p.k);
  const TIn* v = static_cast<const TIn*>(p.v);
  const TIn* g = static_cast<const TIn*>(p.g);
  const TIn* b = static_cast<const TIn*>(p.b);

  // pass 1: inverse norms of the (convolved) q and k rows, one warp per token
  const bool vec = vector_rows<TIn>(p);
  for (int i = warp; i < kChunk; i += kThreads / 32) {
    float sq = 0.f, sk = 0.f;
    if (i < len && vec) {
      for (int c0 = 8 * lane; c0 < dk; c0 += 256) {
        float xq[8], xk[8];
        const int64_t e = ((ch.tok0 + i) * H + h) * dk + c0;
        ld8(q, e, xq);
        ld8(k, e, xk);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          sq += xq[t] * xq[t];
          sk += xk[t] * xk[t];
        }
      }
    } else if (i < len)
#pragma unroll 4
      for (int col = lane; col < dk; col += 32) {
        const float xq = conv_input(p, 0, q, dk, ch, i, h, col), xk = conv_input(p, 1, k, dk, ch, i, h, col);
        sq += xq * xq;
        sk += xk * xk;
      }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    if (lane == 0) {
      invq[i] = inv_norm_of(sq);
      invk[i] = inv_norm_of(sk);
    }
  }
  if (tid < kChunk) beta[tid] = tid < len ? beta_of(ld_in(b, (ch.tok0 + tid) * H + h)) : 0.f;
  for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) A[idx] = AQ[idx] = 0.f;
  __syncthreads();

  // one key block [c0, c0 + nb) of q^, k^ and the running log-decay G
  auto load_key_block = [&](int c0, int nb) {
    if (vec) {
      const int nb8 = nb / 8;
#pragma unroll 2
      for (int idx = tid; idx < kChunk * nb8; idx += kThreads) {
        const int i = idx / nb8, cc = 8 * (idx - i * nb8);
        float xq[8], xk[8], la[8];
        if (i < len) {
          const int64_t e = ((ch.tok0 + i) * H + h) * dk + c0 + cc;
          ld8(q, e, xq);
          ld8(k, e, xk);
          if (p.gate_per_head) {
            const float l = log_alpha_of(ld_in(g, (ch.tok0 + i) * H + h));
#pragma unroll
            for (int t = 0; t < 8; ++t) la[t] = l;
          } else {
            ld8(g, e, la);
#pragma unroll
            for (int t = 0; t < 8; ++t) la[t] = log_alpha_of(la[t]);
          }
        } else {
#pragma unroll
          for (int t = 0; t < 8; ++t) xq[t] = xk[t] = la[t] = 0.f;
        }
        const float iq = i < len ? invq[i] : 0.f, ik = i < len ? invk[i] : 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          X[i * kLd + cc + t] = xq[t] * iq;
          Kb[i * kLd + cc + t] = xk[t] * ik;
          G[i * kLd + cc + t] = la[t];
        }
      }
    } else {
#pragma unroll 4
      for (int idx = tid; idx < kChunk * nb; idx += kThreads) {
        const int i = idx / nb, col = idx - i * nb;
        float xq = 0.f, xk = 0.f, la = 0.f;
        if (i < len) {
          xq = conv_input(p, 0, q, dk, ch, i, h, c0 + col) * invq[i];
          xk = conv_input(p, 1, k, dk, ch, i, h, c0 + col) * invk[i];
          const int64_t e = ((ch.tok0 + i) * H + h) * dk + c0 + col;
          la = log_alpha_of(ld_in(g, p.gate_per_head ? (ch.tok0 + i) * H + h : e));
        }
        X[i * kLd + col] = xq;
        Kb[i * kLd + col] = xk;
        G[i * kLd + col] = la;
      }
    }
    __syncthreads();
    for (int col = tid; col < nb; col += kThreads) {  // rows past len carry G_{L-1}
      float run = 0.f;
      for (int i = 0; i < kChunk; ++i) {
        run += G[i * kLd + col];
        G[i * kLd + col] = run;
      }
    }
    __syncthreads();
  };

  // pass 2: A_kk and A_qk, summed over the key blocks (each block takes the
  // factored products, or the direct form if its decay is past the range)
  for (int c0 = 0; c0 < dk; c0 += kCB) {
    const int nb = dk - c0 < kCB ? dk - c0 : kCB;
    load_key_block(c0, nb);
    if (!channel_refs(G, kLd, nb, sref)) {
      factor_block(X, Kb, G, kLd, nb, sref);  // X, Kb, G <- Qp, Kp, Kn
      __syncthreads();
      accumulate_products(X, Kb, G, kLd, nb, len, beta, A, AQ);
      __syncthreads();
      continue;
    }
    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
      const int i = idx >> 6, j = idx & 63;
      if (j <= i && i < len) {
        float akk = 0.f, aqk = 0.f;
        for (int col = 0; col < nb; ++col) {
          const float d = expf(G[i * kLd + col] - G[j * kLd + col]);
          const float kj = Kb[j * kLd + col] * d;
          akk += Kb[i * kLd + col] * kj;
          aqk += X[i * kLd + col] * kj;
        }
        if (j < i) A[idx] += beta[i] * akk;
        AQ[idx] += aqk;
      }
    }
    __syncthreads();
  }
  float* rec = p.inter + ((size_t)c * H + h) * p.rec_floats;
  for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) rec[SimtRec::aqk(dk) + idx] = AQ[idx];

  // T = (I + A_kk)^{-1} (A_qk is in the record: its tile is scratch), then
  // T diag(beta)
  __syncthreads();
  simt_inverse(A, Tm, AQ);
  for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) Tm[idx] *= beta[idx & 63];
  __syncthreads();

  // pass 3: W, Q^ o Gamma, K^ o Gamma_L / Gamma and Gamma_L per key block
  for (int c0 = 0; c0 < dk; c0 += kCB) {
    const int nb = dk - c0 < kCB ? dk - c0 : kCB;
    load_key_block(c0, nb);
    const float* GL = G + (kChunk - 1) * kLd;
    // Q^ o Gamma and K^ o Gamma_L / Gamma to the record, K^ o Gamma into X
    for (int idx = tid; idx < kChunk * nb; idx += kThreads) {
      const int i = idx / nb, col = idx - i * nb;
      const float eg = expf(G[i * kLd + col]), kv = Kb[i * kLd + col];
      const size_t o = (size_t)i * dk + c0 + col;
      rec[SimtRec::qg(dk) + o] = X[i * kLd + col] * eg;
      rec[SimtRec::kr(dk) + o] = kv * expf(GL[col] - G[i * kLd + col]);
      X[i * kLd + col] = kv * eg;
    }
    for (int col = tid; col < nb; col += kThreads) rec[SimtRec::gl(dk, dv) + c0 + col] = expf(GL[col]);
    __syncthreads();
    for (int idx = tid; idx < kChunk * nb; idx += kThreads) {
      const int i = idx / nb, col = idx - i * nb;
      float w = 0.f;
      for (int m = 0; m <= i; ++m) w += Tm[i * kChunk + m] * X[m * kLd + col];
      rec[SimtRec::w(dk) + (size_t)i * dk + c0 + col] = w;
    }
    __syncthreads();
  }
  // U~ = T diag(beta) V per value block
  for (int v0 = 0; v0 < dv; v0 += kCB) {
    const int nb = dv - v0 < kCB ? dv - v0 : kCB;
    if (vec) {
      const int nb8 = nb / 8;
#pragma unroll 2
      for (int idx = tid; idx < kChunk * nb8; idx += kThreads) {
        const int i = idx / nb8, cc = 8 * (idx - i * nb8);
        float xv[8];
        if (i < len) {
          ld8(v, ((ch.tok0 + i) * H + h) * dv + v0 + cc, xv);
        } else {
#pragma unroll
          for (int t = 0; t < 8; ++t) xv[t] = 0.f;
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) X[i * kLd + cc + t] = xv[t];
      }
    } else {
#pragma unroll 4
      for (int idx = tid; idx < kChunk * nb; idx += kThreads) {
        const int i = idx / nb, col = idx - i * nb;
        X[i * kLd + col] = i < len ? conv_input(p, 2, v, dv, ch, i, h, v0 + col) : 0.f;
      }
    }
    __syncthreads();
    for (int idx = tid; idx < kChunk * nb; idx += kThreads) {
      const int i = idx / nb, col = idx - i * nb;
      float u = 0.f;
      for (int m = 0; m <= i; ++m) u += Tm[i * kChunk + m] * X[m * kLd + col];
      rec[SimtRec::ut(dk) + (size_t)i * dv + v0 + col] = u;
    }
    __syncthreads();
  }
}

// K3 on CUDA cores: one CTA per (sequence, head, NS-column slice of S),
// walking the sequence's chunks with its slice of S in shared memory.  Per
// chunk the record's W, Q^ o Gamma and K^ o Gamma_L / Gamma are staged in
// shared memory by asynchronous 16-byte copies, each one stage ahead of its
// use, in two alternating buffers (rows padded by 4 floats), and each thread
// works on a register tile: token rows i0 .. i0 + RPT - 1 of
// a column pair for U = U~ - W S and O = scale ((Q^ o Gamma) S + A_qk U),
// and key rows r0 .. r0 + SR - 1 of the same column pair for
// S <- Diag(Gamma_L) S + KR^T U (written in place: each thread reads and
// writes only its own elements of S there).
template <typename TIn, int NS>
__global__ void __launch_bounds__(kThreads)
simt_inter(ChunkParams p) {
  extern __shared__ float sm[];
  constexpr int NO = NS / 8;          // column octets
  constexpr int kMaxRB = 4;           // key rows per thread (dk <= 256)
  // CTAs start in the order of their linear index: with seq_order, the
  // sequences longest first, each with all its heads and column slices
  int s = blockIdx.x, h = blockIdx.y, zs = blockIdx.z;
  if (p.seq_order) {
    const unsigned lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    const unsigned per = gridDim.y * gridDim.z, r = lin % per;
    s = p.seq_order[lin / per];
    h = (int)(r / gridDim.z);
    zs = (int)(r % gridDim.z);
  }
  const int n0 = zs * NS;
  const int H = p.H, dk = p.dk, dv = p.dv, tid = threadIdx.x;
  const int64_t c_begin = p.seq_chunk_begin[s], c_end = p.seq_chunk_begin[s + 1];
  if (c_end > c_begin && p.meta->total_chunks == 0) return;  // chunk table overflowed

  const int xs = dk + 4;                  // padded row stride of the staged rows
  float* S = sm;                          // [dk][NS]
  float* U = S + dk * NS;                 // [64][NS]
  float* Xb = U + kChunk * NS;            // two [64][dk + 4]: W / Q^ o Gamma / KR, in turn
  float* AQb = Xb + 2 * kChunk * xs;      // two [64][64]: A_qk
  float* GLb = AQb + 2 * kChunk * kChunk; // two [dk]: Gamma_L
  // U and O: token row ti, columns c0 .. c0 + 7 (threads past 64 NO idle);
  // the state update: key rows r0 .. r0 + RB - 1, the same columns
  const int cg = tid % NO, c0 = 8 * cg;
  const int ti = tid / NO;
  const bool row_thread = ti < kChunk;
  const int RB = dk * NO >= kThreads ? dk * NO / kThreads : 1;
  const int r0 = (tid / NO) * RB;
  const bool key_thread = r0 < dk;

  const size_t sbase = ((size_t)s * H + h) * dk * dv;
  for (int idx = tid; idx < dk * NS; idx += kThreads) {
    const int r = idx / NS, n = idx - r * NS;
    S[idx] = p.initial_state ? p.initial_state[sbase + (size_t)r * dv + n0 + n] : 0.f;
  }
  // The record's rows go to shared memory by asynchronous 16-byte copies,
  // one stage ahead: W (with A_qk and Gamma_L) of chunk c+1 while chunk c
  // forms O, Q^ o Gamma while it forms U, KR while it forms O.  The two row
  // buffers alternate: chunk c's W and KR in buffer c % 2, its Q^ o Gamma
  // and the next chunk's W in the other.
  auto rec_of = [&](int64_t c) { return p.inter + ((size_t)c * H + h) * p.rec_floats; };
  auto issue_rows = [&](float* dst, const float* src) {
    const int q4 = dk / 4;
    for (int idx = tid; idx < kChunk * q4; idx += kThreads) {
      const int i = idx / q4, c4 = idx - i * q4;
      cp_async16(dst + i * xs + 4 * c4, src + (size_t)i * dk + 4 * c4);
    }
  };
  auto issue_w = [&](int64_t c, int buf) {
    const float* rec = rec_of(c);
    issue_rows(Xb + buf * kChunk * xs, rec + SimtRec::w(dk));
    for (int idx = tid; idx < kChunk * kChunk / 4; idx += kThreads)
      cp_async16(AQb + buf * kChunk * kChunk + 4 * idx, rec + SimtRec::aqk(dk) + 4 * idx);
    for (int idx = tid; idx < dk / 4; idx += kThreads)
      cp_async16(GLb + buf * dk + 4 * idx, rec + SimtRec::gl(dk, dv) + 4 * idx);
    cp_async_commit();
  };
  // acc[t] += X[ti] . S[:, c0 + t]
  auto row_times_state = [&](const float* X, float* acc) {
    const float* xr = X + ti * xs;
    for (int r = 0; r < dk; ++r) {
      const float4 sa = *reinterpret_cast<const float4*>(S + r * NS + c0);
      const float4 sb = *reinterpret_cast<const float4*>(S + r * NS + c0 + 4);
      const float x = xr[r];
      acc[0] += x * sa.x; acc[1] += x * sa.y; acc[2] += x * sa.z; acc[3] += x * sa.w;
      acc[4] += x * sb.x; acc[5] += x * sb.y; acc[6] += x * sb.z; acc[7] += x * sb.w;
    }
  };
  TIn* o = static_cast<TIn*>(p.o);
  const TIn* og = static_cast<const TIn*>(p.out_gate);
  if (c_end > c_begin) issue_w(c_begin, 0);
  for (int64_t c = c_begin; c < c_end; ++c) {
    const int par = (int)((c - c_begin) & 1);
    float* Xw = Xb + par * kChunk * xs;        // W, then KR
    float* Xq = Xb + (1 - par) * kChunk * xs;  // Q^ o Gamma, then the next W
    const float* AQ = AQb + par * kChunk * kChunk;
    const float* GLs = GLb + par * dk;
    const Chunk ch = p.chunks[c];
    const float* rec = rec_of(c);
    issue_rows(Xq, rec + SimtRec::qg(dk));
    cp_async_commit();
    float4 uta = make_float4(0.f, 0.f, 0.f, 0.f), utb = uta;
    if (row_thread) {
      const float* ut = rec + SimtRec::ut(dk) + (size_t)ti * dv + n0 + c0;
      uta = *reinterpret_cast<const float4*>(ut);
      utb = *reinterpret_cast<const float4*>(ut + 4);
    }
    cp_async_wait<1>();  // W, A_qk, Gamma_L
    __syncthreads();
    // U = U~ - W S
    if (row_thread) {
      float a[8] = {};
      row_times_state(Xw, a);
      *reinterpret_cast<float4*>(U + ti * NS + c0) =
          make_float4(uta.x - a[0], uta.y - a[1], uta.z - a[2], uta.w - a[3]);
      *reinterpret_cast<float4*>(U + ti * NS + c0 + 4) =
          make_float4(utb.x - a[4], utb.y - a[5], utb.z - a[6], utb.w - a[7]);
    }
    __syncthreads();  // U complete, W read
    issue_rows(Xw, rec + SimtRec::kr(dk));
    cp_async_commit();
    cp_async_wait<1>();  // Q^ o Gamma
    __syncthreads();
    // O = scale ((Q^ o Gamma) S + A_qk U), A_qk masked j <= i
    if (row_thread) {
      float a[8] = {};
      row_times_state(Xq, a);
      const int i = ti;
      for (int j = 0; j <= i; ++j) {
        const float aq = AQ[i * kChunk + j];
        const float4 ua = *reinterpret_cast<const float4*>(U + j * NS + c0);
        const float4 ub = *reinterpret_cast<const float4*>(U + j * NS + c0 + 4);
        a[0] += aq * ua.x; a[1] += aq * ua.y; a[2] += aq * ua.z; a[3] += aq * ua.w;
        a[4] += aq * ub.x; a[5] += aq * ub.y; a[6] += aq * ub.z; a[7] += aq * ub.w;
      }
      if (i < ch.len) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int64_t oi = ((ch.tok0 + i) * H + h) * dv + n0 + c0 + t;
          float val = p.scale * a[t];
          if (og) val *= out_gate_of(ld_in(og, p.out_gate_per_head ? (ch.tok0 + i) * H + h : oi));
          st_out(o, oi, val);
        }
      }
    }
    __syncthreads();  // Q^ o Gamma and S read
    if (c + 1 < c_end) {
      issue_w(c + 1, 1 - par);
      cp_async_wait<1>();  // KR
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    // S <- Diag(Gamma_L) S + KR^T U on this thread's key rows
    if (key_thread) {
      float b[kMaxRB][8];
#pragma unroll
      for (int rr = 0; rr < kMaxRB; ++rr) {
        const int r = r0 + rr;
        const bool live = rr < RB;
#pragma unroll
        for (int t = 0; t < 8; ++t) b[rr][t] = live ? GLs[r] * S[r * NS + c0 + t] : 0.f;
      }
      for (int i = 0; i < kChunk; ++i) {
        const float4 ua = *reinterpret_cast<const float4*>(U + i * NS + c0);
        const float4 ub = *reinterpret_cast<const float4*>(U + i * NS + c0 + 4);
        const float u[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
        float x[kMaxRB];
        if (RB == 4) {
          const float4 xv = *reinterpret_cast<const float4*>(Xw + i * xs + r0);
          x[0] = xv.x; x[1] = xv.y; x[2] = xv.z; x[3] = xv.w;
        } else {
#pragma unroll
          for (int rr = 0; rr < kMaxRB; ++rr) x[rr] = rr < RB ? Xw[i * xs + r0 + rr] : 0.f;
        }
#pragma unroll
        for (int rr = 0; rr < kMaxRB; ++rr)
#pragma unroll
          for (int t = 0; t < 8; ++t) b[rr][t] += x[rr] * u[t];
      }
#pragma unroll
      for (int rr = 0; rr < kMaxRB; ++rr)
        if (rr < RB) {
          *reinterpret_cast<float4*>(S + (r0 + rr) * NS + c0) = make_float4(b[rr][0], b[rr][1], b[rr][2], b[rr][3]);
          *reinterpret_cast<float4*>(S + (r0 + rr) * NS + c0 + 4) =
              make_float4(b[rr][4], b[rr][5], b[rr][6], b[rr][7]);
        }
    }
    __syncthreads();
    if (ch.snap_slot >= 0 && p.snapshots) {
      const size_t base = ((size_t)ch.snap_slot * H + h) * dk * dv;
      for (int idx = tid; idx < dk * NS; idx += kThreads) {
        const int r = idx / NS, n = idx - r * NS;
        p.snapshots[base + (size_t)r * dv + n0 + n] = S[idx];
      }
    }
  }
  __syncthreads();
  if (p.final_state) {
    for (int idx = tid; idx < dk * NS; idx += kThreads) {
      const int r = idx / NS, n = idx - r * NS;
      p.final_state[sbase + (size_t)r * dv + n0 + n] = S[idx];
    }
  }
}

template <typename TIn>
cudaError_t launch_simt_t(const ChunkParams& p, cudaStream_t stream, cudaEvent_t mid) {
  // heads up to 128 channels keep a whole chunk in shared memory; wider ones
  // take the blocked kernel
  const bool blocked = p.dk > kCB || p.dv > kCB;
  const size_t smem_intra =
      blocked ? sizeof(float) * (3 * (size_t)kChunk * (kCB + 1) + 3 * kChunk * kChunk + 3 * kChunk + kCB)
              : sizeof(float) * (4 * (size_t)kChunk * (p.dk + 1) + (size_t)kChunk * p.dv + 2 * kChunk * kChunk + kChunk +
                                 p.dk);
  auto intra = blocked ? simt_intra_blocked<TIn> : simt_intra<TIn>;
  cudaError_t e = cudaFuncSetAttribute(intra, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_intra);
  if (e != cudaSuccess) return e;
  if (p.max_chunks > 0) {
    dim3 grid((unsigned)p.max_chunks, (unsigned)p.H);
    intra<<<grid, kThreads, smem_intra, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (mid) {
    e = cudaEventRecord(mid, stream);
    if (e != cudaSuccess) return e;
  }
  const int ns = p.dv < 32 ? p.dv : 32;  // 16 or 32 value columns per CTA
  const size_t smem_inter = sizeof(float) * ((size_t)p.dk * ns + (size_t)kChunk * ns +
                                             2 * (size_t)kChunk * (p.dk + 4) + 2 * kChunk * kChunk + 2 * (size_t)p.dk);
  auto inter = ns == 32 ? simt_inter<TIn, 32> : simt_inter<TIn, 16>;
  e = cudaFuncSetAttribute(inter, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_inter);
  if (e != cudaSuccess) return e;
  dim3 grid2((unsigned)p.num_seqs, (unsigned)p.H, (unsigned)(p.dv / ns));
  inter<<<grid2, kThreads, smem_inter, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_prefill(const ChunkParams& p, kda_dtype_t dt, cudaStream_t stream,
                                cudaEvent_t mid) {
  return dt == KDA_BF16 ? launch_simt_t<__nv_bfloat16>(p, stream, mid)
                        : launch_simt_t<float>(p, stream, mid);
}

}  // namespace kda
